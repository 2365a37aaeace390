"""dv_sparse_mlp_noalloc: the sparse MLP block for callers that cannot allocate
device memory (a plugin inside a serving engine that owns all device memory,
code that must not allocate after start-up). Its partial sums live in a fixed
array inside the library instead of a caller workspace.

Called through the C ABI, it must give the same block output as dv_sparse_mlp
(which uses a caller workspace) and as the CPU oracle's gathered MLP, on two
calls in a row, since every call reuses the same array. The cases include one
where the array holds fewer partial sums than one per SM (d 12288, batch 4),
so the launch uses fewer CTAs that each stream more rows. The host-side
rejections (packed 4-bit rows, sizes beyond the array) are checked without a
GPU in tests/test_abi.py. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, host, npf, rel_err, setup_lib

pytestmark = pytest.mark.gpu


def _fn():
    L = setup_lib()
    f = L.dv_sparse_mlp_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(dv.Dims),
                  ctypes.POINTER(dv.LayerWeights), ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


@pytest.mark.parametrize("wl,over,B,keep", [
    ("tiny", {}, 1, 0.25),
    ("opt-6.7b", {}, 1, 0.1),
    ("tiny", dict(d=512, F=2048), 4, 0.1),
    # 4 x 12288 fp32 partial sums per CTA: the 8 MiB array holds 42 of them,
    # so 6000 rows run on 42 CTAs of up to 143 rows instead of one per SM
    ("tiny", dict(d=12288, F=6400), 4, 0.9375),
])
def test_noalloc_matches_workspace_entry_point_and_oracle(wl, over, B, keep):
    f = _fn()
    dv.set_tuning()
    w = synth.workload(wl, **over)
    W = synth.layer_weights(w, 0, seed=21, full_bias=True, device="cuda")
    x = synth.hidden(w, B=B, seed=22).cuda()
    k = oracle.k_from_keep(keep, w.F)
    idx_h = np.sort(np.random.default_rng(3).choice(w.F, k, replace=False)).astype(np.int32)
    idx = torch.from_numpy(idx_h).cuda()
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    ws = dv.workspace(D, B)
    ref = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
    dv.sparse_mlp(x, D, W, idx, k, ref, ws, flags=dv.DV_NO_RESIDUAL)
    lw = dv.layer_weights(W)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    Wh = host({n: W[n] for n in ("fc1", "b1", "fc2T", "b2", "ln2_g", "ln2_b")})
    xh = x.cpu().numpy()
    want = [oracle.mlp_gather(xh[b], Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], idx_h,
                              ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"]) for b in range(B)]
    for _ in range(2):   # the array keeps the previous call's contents
        out = torch.full((B, w.d), float("nan"), dtype=torch.float16, device="cuda")
        rc = f(x.data_ptr(), B, ctypes.byref(D), ctypes.byref(lw), idx.data_ptr(), k, None,
               dv.DV_NO_RESIDUAL, out.data_ptr(), st.data_ptr(), s)
        assert rc == dv.DV_OK, dv.status_string(rc)
        torch.cuda.synchronize()
        assert st.item() == 0
        for b in range(B):
            assert rel_err(npf(out[b]), npf(ref[b])) < TOL
            assert rel_err(npf(out[b]), want[b]) < TOL
