"""W4A16 sparse MLP ("Deja Vu" §5.2, Table 7: 4-bit weights, fp16
activations) through the C ABI: the GPU quantizer against the oracle's
(bit-exact packed rows), and the 4-bit gather MLP against the oracle's MLP on
the dequantized weights."""
import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, check_sets, host, np16, npf, rel_err, setup_lib, to_dev
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
    ("opt-175b", {}, 49152, 1, 0),                     # every row: > 256 rows per CTA
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


W4_NAMES = ("Wq", "Wk", "Wv", "WoT", "fc1", "fc2T")


def _w4_layer(w, seed):
    """Device weights of one layer with the six projection matrices as packed
    4-bit rows (GPU quantizer), and the oracle's view of them."""
    W = synth.layer_weights(w, 0, seed=seed, full_bias=True)
    Wd = to_dev(W)
    Wq = dict(Wd)
    for k in W4_NAMES:
        Wq[k] = dv.quantize_w4(Wd[k])
    torch.cuda.synchronize()
    Wo = host(W)
    for k in W4_NAMES:
        Wo[k] = ow4.unpack(Wq[k].cpu().numpy(), w.d)
    return Wq, Wo


@pytest.mark.parametrize("wl,over,n,sel", [
    ("tiny", {}, 64, [1, 3]),
    ("opt-6.7b", dict(F=64), 200, [0, 5, 31]),
    ("compose", dict(d=512, h=8, h_kv=2, F=64), 300, [1]),        # GQA, 4 query heads per unit
    # batch-1 4-bit launches give each thread V consecutive code words: V = 2
    # with full stages at d 12288, V = 3 (per-word scales, a partial last
    # thread) at d 16384
    ("opt-175b", dict(F=64), 100, [0, 7, 95]),
    ("opt-6.7b", dict(d=16384, h=8, h_kv=8, F=64), 100, [0, 5]),
])
def test_w4_attention_block_parity(wl, over, n, sel):
    setup_lib()
    w = synth.workload(wl, **over)
    Wq, Wo = _w4_layer(w, seed=21)
    n_max = n + 5
    K, V = synth.kv_cache(w, 0, n_max, B=1, seed=21)
    x = synth.hidden(w, B=1, seed=22)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws = dv.workspace(D, 1)
    Kd, Vd = K.cuda(), V.cuda()
    kv = dv.kv_cache(Kd, Vd)
    out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    sd = torch.tensor(sel, dtype=torch.int32, device="cuda")
    dv.sparse_attn(x.cuda(), D, Wq, sd, len(sel), kv, n, out, ws,
                   flags=dv.DV_NO_RESIDUAL | dv.DV_W4, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    delta, knew, vnew = ow4.attn(np16(x[0]), Wo, np16(K[0]), np16(V[0]), n, sel)
    assert rel_err(npf(out[0]), delta) < TOL
    for u in sel:
        assert rel_err(npf(Kd[0, u, n]), knew[u].astype(float)) < TOL
        assert rel_err(npf(Vd[0, u, n]), vnew[u].astype(float)) < TOL


@pytest.mark.parametrize("wl,over,B", [("tiny", {}, 1), ("opt-6.7b", dict(F=2048), 1),
                                       ("opt-6.7b", dict(F=2048), 4)])
def test_w4_decode_layer_parity(wl, over, B):
    # one layer through the driver with 4-bit projection and MLP rows (its own
    # fp16 predictor chooses the sets); teacher-forced against the oracle layer
    setup_lib()
    w = synth.workload(wl, **over)
    Wq, Wo = _w4_layer(w, seed=31)
    n_max = w.n + 4
    K, V = synth.kv_cache(w, 0, n_max, B=B, seed=31)
    x = synth.hidden(w, B=B, seed=32).cuda()
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws = dv.workspace(D, B)
    kN = oracle.k_from_keep(w.keep_N, w.F)
    kH = oracle.k_from_keep(w.keep_H, w.h_kv)
    cur, cur_t = dv.sets(B, w.F, w.h_kv, kN, kH)
    kv = dv.kv_cache(K.cuda(), V.cuda())
    y = torch.empty_like(x)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dv.decode_layer(D, dv.Keep(w.keep_N, w.keep_H, 1.0), Wq, None, kv, w.n, cur, None, x, y, ws,
                    dv.DV_SYNC_PREDICT | dv.DV_W4, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() == 0
    if B == 1:
        selH, selN = cur_t["idx_H"][0].cpu().numpy(), cur_t["idx_N"][0].cpu().numpy()
    else:
        c = cur_t["ucnt"].cpu().numpy()
        selH, selN = cur_t["uH"][: c[1]].cpu().numpy(), cur_t["uN"][: c[0]].cpu().numpy()
    for b in range(B):
        ref = oracle.predict(np16(x[b]), Wo["P1"], Wo["P2"])
        if B == 1:
            check_sets(selN, ref[: w.F], kN)
            check_sets(selH, ref[w.F:], kH)
        y_ref, _ = ow4.layer(np16(x[b]), Wo, np16(K[b]), np16(V[b]), w.n, selH, selN)
        assert rel_err(npf(y[b]), y_ref.astype(np.float64)) < TOL, b


@pytest.mark.parametrize("wl,over,n0,T", [
    ("tiny", {}, 30, 8),
    ("opt-6.7b", dict(F=64), 100, 5),                                   # d 4096, 32 units
    ("compose", dict(d=512, h=8, h_kv=2, F=64), 60, 6),                 # GQA
])
def test_w4_multistep_missing_kv_recompute(wl, over, n0, T):
    # head-sparse decode steps with 4-bit W^K, W^V: the missing k, v of a unit
    # are recomputed from the kept inputs with the 4-bit rows ("Deja Vu" §4.2
    # with §5.2's W4A16), against the oracle's W4 attention where every past
    # token's k, v come from that token's own input
    setup_lib()
    w = synth.workload(wl, **over)
    Wq, Wo = _w4_layer(w, seed=41)
    rng = np.random.default_rng(n0)
    n_max = n0 + T + 3
    K, V = synth.kv_cache(w, 0, n_max, B=1, seed=41)
    ys = [synth.hidden(w, B=1, seed=800 + t) for t in range(T)]
    k = max(1, w.h_kv // 2)
    sels = [sorted(rng.choice(w.h_kv, k, replace=False).tolist()) for _ in range(T)]
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws = dv.workspace(D, 1)
    Kd, Vd = K.cuda(), V.cuda()
    y_side = torch.zeros(1, n_max, w.d, dtype=torch.float16, device="cuda")
    miss = torch.zeros(1, n_max, (w.h_kv + 31) // 32, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(Kd, Vd, y_side=y_side, kv_missing=miss)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for t in range(T):
        out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
        sd = torch.tensor(sels[t], dtype=torch.int32, device="cuda")
        dv.sparse_attn(ys[t].cuda(), D, Wq, sd, len(sels[t]), kv, n0 + t, out, ws,
                       flags=dv.DV_NO_RESIDUAL | dv.DV_KV_FILL | dv.DV_W4, dev_status=st)
        outs.append(out)
    torch.cuda.synchronize()
    assert st.item() == 0
    Kc, Vc = np16(K[0]).copy(), np16(V[0]).copy()
    for t in range(T):
        y = np16(ys[t][0])
        delta, _, _ = ow4.attn(y, Wo, Kc, Vc, n0 + t, sels[t])
        assert rel_err(npf(outs[t][0]), delta) < TOL, t
        _, kn, vn = ow4.attn(y, Wo, Kc, Vc, n0 + t, range(w.h_kv))   # every unit's k, v
        Kc[:, n0 + t], Vc[:, n0 + t] = kn, vn
