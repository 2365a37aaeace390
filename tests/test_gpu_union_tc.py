"""The batched union MLP on the tensor cores ("Deja Vu" §5.2, App. C.1: a batch
computes every row over the union of its sequences' sets) against the oracle's
gather MLP of each sequence over that union, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, host, np16, npf, rel_err, setup_lib, to_dev

pytestmark = pytest.mark.gpu


def _union(F, k, B, rng):
    return np.unique(np.concatenate([rng.choice(F, k, replace=False) for _ in range(B)])).astype(np.int32)


@pytest.mark.parametrize("wl,over,B,keep", [
    ("opt-6.7b", dict(d=512, F=1024), 8, 0.1),
    ("opt-6.7b", dict(d=512, F=1024), 16, 0.05),
    ("opt-6.7b", dict(d=1024, F=2048), 32, 0.02),
    ("opt-6.7b", dict(d=512, F=4096), 64, 0.01),
    ("opt-175b", dict(F=8192), 8, 0.1),                  # d 12288
    ("opt-66b", {}, 8, 0.1),                              # d 9216, F 36864: ~21000 union rows
])
def test_union_mlp_parity(wl, over, B, keep):
    setup_lib()
    w = synth.workload(wl, **over)
    rng = np.random.default_rng(B)
    W = synth.layer_weights(w, 0, seed=41, full_bias=True)
    U = _union(w.F, max(1, int(keep * w.F)), B, rng)
    x = synth.hidden(w, B=B, seed=42)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    out = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dv.union_mlp(x.cuda(), D, to_dev(W), torch.from_numpy(U).cuda(), len(U), out, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Wh = host(W)
    for b in range(B):
        ref = oracle.mlp_gather(np16(x[b]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh.get("b2"), U,
                                ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
        want = np16(x[b]).astype(np.float64) + ref
        assert rel_err(npf(out[b]), want) < TOL, b


def test_union_mlp_device_count_and_shapes():
    setup_lib()
    w = synth.workload("opt-6.7b", d=512, F=1024)
    rng = np.random.default_rng(3)
    W = synth.layer_weights(w, 0, seed=43, full_bias=True)
    U = _union(w.F, 60, 8, rng)
    cnt = torch.tensor([len(U) - 17], dtype=torch.int32, device="cuda")    # only the first ones
    x = synth.hidden(w, B=8, seed=44)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    out = torch.empty(8, w.d, dtype=torch.float16, device="cuda")
    dv.union_mlp(x.cuda(), D, to_dev(W), torch.from_numpy(U).cuda(), len(U), out, dev_count=cnt,
                 flags=dv.DV_NO_RESIDUAL)
    torch.cuda.synchronize()
    Wh = host(W)
    for b in range(8):
        ref = oracle.mlp_gather(np16(x[b]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh.get("b2"),
                                U[: len(U) - 17], ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
        assert rel_err(npf(out[b]), ref) < TOL, b
    assert dv.lib().dv_union_mlp_ws_size(12, 512, 10) == 0          # B not 8, 16, 32 or 64
    assert dv.lib().dv_union_mlp_ws_size(8, 496, 10) == 0           # d not a multiple of 64
