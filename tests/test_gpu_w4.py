"""W4A16 sparse MLP ("Deja Vu" §5.2, Table 7: 4-bit weights, fp16
activations) through the C ABI: the GPU quantizer against the oracle's
(bit-exact packed rows), and the 4-bit gather MLP against the oracle's MLP on
the dequantized weights."""
import numpy as np
import pytest
import torch

from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, host, np16, npf, rel_err, setup_lib, to_dev
from oracle import w4 as ow4

pytestmark = pytest.mark.gpu


def _tricky_rows(rows, d, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((rows, d)) * rng.uniform(1e-3, 4.0, (rows, 1))).astype(np.float16)
    W[0, :128] = 0                                   # a zero group
    if rows > 1:                                     # exact ties w / s = k + 1/2 (s = 1)
        W[1, :128] = 0
        W[1, :8] = [7.0, -3.5, 2.5, 0.5, -1.5, -7.0, 4.5, 6.5]
    if rows > 2:
        W[2, -128:] = np.float16(6e-5) * rng.integers(-7, 8, 128)     # subnormal scale
    return W


@pytest.mark.parametrize("rows,d", [(3, 128), (40, 256), (257, 4096), (64, 12288), (9, 16384)])
def test_quantizer_matches_the_oracle_bit_for_bit(rows, d):
    setup_lib()
    W = _tricky_rows(rows, d, rows + d)
    got = dv.quantize_w4(torch.from_numpy(W).cuda()).cpu().numpy()
    want = ow4.pack(*ow4.quantize(W))
    assert got.shape == want.shape == (rows, dv.w4_row_bytes(d))
    assert np.array_equal(got, want)


def _mlp_case(wl, over, n_sel, B, seed):
    w = synth.workload(wl, **over)
    W = synth.layer_weights(w, 0, seed=seed, full_bias=True)
    fc1q = dv.quantize_w4(W["fc1"].cuda())
    fc2q = dv.quantize_w4(W["fc2T"].cuda())
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    idx = np.sort(rng.choice(w.F, n_sel, replace=False)).astype(np.int32)
    x = synth.hidden(w, B=B, seed=seed + 7)
    return w, W, fc1q, fc2q, idx, x


@pytest.mark.parametrize("wl,over,n_sel,B,flags", [
    ("tiny", {}, 100, 1, 0),
    ("opt-6.7b", dict(F=2048), 300, 1, 0),
    ("opt-6.7b", dict(F=2048), 300, 1, dv.DV_SKIP_INACTIVE),
    ("opt-175b", {}, 512, 1, 0),                       # full width 49152, d 12288
    ("opt-66b", dict(F=4096), 700, 4, 0),              # batch 4 over one (union) set
    ("opt-6.7b", dict(d=16384, h=8, h_kv=8, F=512), 200, 1, 0),   # largest d
])
def test_w4_mlp_parity(wl, over, n_sel, B, flags):
    setup_lib()
    w, W, fc1q, fc2q, idx, x = _mlp_case(wl, over, n_sel, B, seed=11)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    ws = dv.workspace(D, B)
    out = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dv.sparse_mlp_w4(x.cuda(), D, to_dev(W), fc1q, fc2q, torch.from_numpy(idx).cuda(), len(idx),
                     out, ws, flags=flags | dv.DV_NO_RESIDUAL, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    Wh = host(W)
    q1, s1 = ow4.unpack(fc1q.cpu().numpy(), w.d)
    q2, s2 = ow4.unpack(fc2q.cpu().numpy(), w.d)
    for b in range(B):
        ref = ow4.mlp(np16(x[b]), q1, s1, Wh["b1"], q2, s2, Wh.get("b2"), idx,
                      ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
        assert rel_err(npf(out[b]), ref) < TOL, b


def test_w4_mlp_residual_and_dense_index_list():
    setup_lib()
    w, W, fc1q, fc2q, _, x = _mlp_case("tiny", {}, 10, 1, seed=3)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 8)
    ws = dv.workspace(D, 1)
    out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
    dv.sparse_mlp_w4(x.cuda(), D, to_dev(W), fc1q, fc2q, None, w.F, out, ws)
    torch.cuda.synchronize()
    Wh = host(W)
    q1, s1 = ow4.unpack(fc1q.cpu().numpy(), w.d)
    q2, s2 = ow4.unpack(fc2q.cpu().numpy(), w.d)
    ref = ow4.mlp(np16(x[0]), q1, s1, Wh["b1"], q2, s2, Wh.get("b2"), np.arange(w.F),
                  ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
    want = np16(x[0]).astype(np.float64) + ref
    assert rel_err(npf(out[0]), want) < TOL
