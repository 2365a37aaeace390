"""dv_sparse_mlp_noalloc: the sparse MLP block for callers that cannot allocate
device memory (its partial sums live in a fixed array inside the library).

Called through the C ABI, it must give the same block output as dv_sparse_mlp
(which uses a caller workspace), on two calls in a row since every call reuses
the same array. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, npf, rel_err, setup_lib, to_dev

pytestmark = pytest.mark.gpu


def _fn():
    L = setup_lib()
    f = L.dv_sparse_mlp_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(dv.Dims),
                  ctypes.POINTER(dv.LayerWeights), ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f


@pytest.mark.parametrize("wl,over,B,keep", [("tiny", {}, 1, 0.25), ("opt-6.7b", {}, 1, 0.1),
                                            ("tiny", dict(d=512, F=2048), 4, 0.1)])
def test_noalloc_matches_workspace_entry_point(wl, over, B, keep):
    f = _fn()
    dv.set_tuning()
    w = synth.workload(wl, **over)
    W = to_dev(synth.layer_weights(w, 0, seed=21, full_bias=True))
    x = synth.hidden(w, B=B, seed=22).cuda()
    k = oracle.k_from_keep(keep, w.F)
    idx = torch.from_numpy(np.sort(np.random.default_rng(3).choice(w.F, k, replace=False))
                           .astype(np.int32)).cuda()
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    ws = dv.workspace(D, B)
    ref = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
    dv.sparse_mlp(x, D, W, idx, k, ref, ws, flags=dv.DV_NO_RESIDUAL)
    lw = dv.layer_weights(W)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):   # the array keeps the previous call's contents
        out = torch.full((B, w.d), float("nan"), dtype=torch.float16, device="cuda")
        rc = f(x.data_ptr(), B, ctypes.byref(D), ctypes.byref(lw), idx.data_ptr(), k, None,
               dv.DV_NO_RESIDUAL, out.data_ptr(), st.data_ptr(), s)
        assert rc == dv.DV_OK, dv.status_string(rc)
        torch.cuda.synchronize()
        assert st.item() == 0
        for b in range(B):
            assert rel_err(npf(out[b]), npf(ref[b])) < TOL


def test_noalloc_rejects_problems_beyond_its_array():
    f = _fn()
    D = dv.dims(16384, 128, 128, 128, 262144, 8, 8)
    lw = dv.LayerWeights(*([None] * 12 + [0x100000, None, 0x100000, None, None, None]))
    # 4 rows of 16384 fp32 partial sums need 256 KiB per CTA and at least 1024
    # CTAs for 262144 rows: beyond 8 MiB; rejected before anything is launched.
    rc = f(0x200000, 4, ctypes.byref(D), ctypes.byref(lw), None, 0, None, 0, 0x300000, None, None)
    assert rc == dv.DV_ERR_WORKSPACE
