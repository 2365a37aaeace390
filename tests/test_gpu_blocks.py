"""GPU parity of each block against the fp64 oracle (through the C ABI).

Sizes are chosen so the oracle finishes in seconds while the kernels still
span several CTAs, stages and a ragged tail; edge cases cover k = 1, k = N,
dense (idx = NULL), n = 0, ragged d, GQA, batch > 1 with unions, and the
kernels' own bounds checks.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import (TOL, check_kv_kept, check_sets, host, np16, npf, rel_err,
                         setup_lib, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    setup_lib()
    dv.set_tuning()


def _dims(w: synth.Workload, n_max):
    return dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)


# ---------------------------------------------------------------------------
# a2 predictor + a3 top-k
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("wl,B", [("tiny", 1), ("tiny", 4), ("opt-175b", 1)])
def test_predict_scores_and_sets(wl, B):
    w = synth.workload(wl)
    W = synth.layer_weights(w, 0, seed=1)
    y = synth.hidden(w, B=B, seed=1)
    P1, P2 = W["P1"], W["P2"]
    D = _dims(w, w.n + 1)
    ws = dv.workspace(D, B)
    scores = torch.zeros(B, P2.shape[0], device="cuda")
    dv.predict(y.cuda(), P1.cuda(), P2.cuda(), scores, ws)
    torch.cuda.synchronize()
    got = npf(scores)
    kN = oracle.k_from_keep(w.keep_N, w.F)
    for b in range(B):
        ref = oracle.predict(np16(y[b]), np16(P1), np16(P2))
        assert rel_err(got[b], ref) < 1e-5
        # GPU top-k of the GPU scores equals the oracle's top-k of the same scores
        idx = torch.zeros(1, kN, dtype=torch.int32, device="cuda")
        dv.select_topk(scores[b:b + 1, : w.F].contiguous(), w.F, kN, idx)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy()[0], oracle.topk(got[b, : w.F], kN))
        # end to end: swaps only within 1e-6 of the k-th reference score
        check_sets(idx.cpu().numpy()[0], ref[: w.F], kN)


@pytest.mark.parametrize("N,B", [(1, 1), (5, 3), (96, 1), (1000, 3), (49152, 1), (49152, 3),
                                 (131072, 2), (140000, 1)])
def test_topk_bit_exact_with_ties(N, B):
    g = torch.Generator().manual_seed(N * 7 + B)
    s = torch.randint(-20, 20, (B, N), generator=g).float() / 4.0   # many ties
    s[:, ::7] = -0.0
    s[:, ::11] = 0.0
    sd = s.cuda()
    for k in sorted({1, max(1, N // 10), max(1, N // 2), N}):
        idx = torch.zeros(B, k, dtype=torch.int32, device="cuda")
        uni = torch.zeros(N, dtype=torch.int32, device="cuda")
        cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        dv.select_topk(sd, N, k, idx, union_idx=uni, union_count=cnt)
        torch.cuda.synchronize()
        ref = np.stack([oracle.topk(s[b].double().numpy(), k) for b in range(B)])
        assert np.array_equal(idx.cpu().numpy(), ref)
        u = oracle.union(ref, N)
        assert int(cnt.item()) == len(u)
        assert np.array_equal(uni.cpu().numpy()[: len(u)], u)


@pytest.mark.parametrize("N,B", [(96, 2), (2047, 1), (49152, 2), (65536, 1), (65537, 1)])
def test_topk_bit_exact_continuous(N, B):
    # distinct scores: the threshold bin's keys fit in shared memory
    g = torch.Generator().manual_seed(N + B)
    s = torch.randn(B, N, generator=g) * 3.0
    sd = s.cuda()
    for k in sorted({1, 2, max(1, N // 10), N - 1, N} - {0}):
        idx = torch.zeros(B, k, dtype=torch.int32, device="cuda")
        dv.select_topk(sd, N, k, idx)
        torch.cuda.synchronize()
        ref = np.stack([oracle.topk(s[b].double().numpy(), k) for b in range(B)])
        assert np.array_equal(idx.cpu().numpy(), ref), k


def test_topk_flags_nan_without_faulting():
    s = torch.randn(1, 100)
    s[0, 17] = float("nan")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.zeros(1, 10, dtype=torch.int32, device="cuda")
    dv.select_topk(s.cuda(), 100, 10, idx, dev_status=st)
    torch.cuda.synchronize()
    assert st.item() & dv.DV_DEV_NONFINITE
    assert 17 not in idx.cpu().numpy()


# ---------------------------------------------------------------------------
# a4 sparse MLP
# ---------------------------------------------------------------------------
def _mlp_case(wl, d=None, F=None, seed=0, full_bias=True):
    w = synth.workload(wl)
    if d is not None:
        w = synth.workload(wl, d=d, F=F or w.F)
    W = synth.layer_weights(w, 0, seed=seed, full_bias=full_bias)
    return w, W


@pytest.mark.parametrize("wl,d,F,keep", [("tiny", None, None, 0.25), ("tiny", 264, 520, 0.1),
                                         ("opt-6.7b", None, None, 0.1),
                                         ("opt-6.7b", None, None, 1.0),
                                         ("opt-6.7b", 16384, 512, 0.25),      # largest d
                                         # 49152 rows per phase: more than 256 per CTA at
                                         # one CTA per SM
                                         ("opt-175b", None, None, 1.0)])
@pytest.mark.parametrize("flags", [0, dv.DV_SKIP_INACTIVE])
def test_mlp_parity(wl, d, F, keep, flags):
    w, W = _mlp_case(wl, d, F)
    x = synth.hidden(w, B=1, seed=3, name="h")
    rng = np.random.default_rng(0)
    k = oracle.k_from_keep(keep, w.F)
    idx = np.sort(rng.choice(w.F, k, replace=False)).astype(np.int32)
    Wd = to_dev(W)
    D = _dims(w, 8)
    ws = dv.workspace(D)
    out = torch.empty_like(x, device="cuda")
    xd = x.cuda()
    Wh = host(W)
    ref = oracle.mlp_gather(np16(x[0]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], idx,
                            ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
    idx_d = None if keep == 1.0 else torch.from_numpy(idx).cuda()
    dv.sparse_mlp(xd, D, Wd, idx_d, k, out, ws, flags=flags | dv.DV_NO_RESIDUAL)
    torch.cuda.synchronize()
    assert rel_err(npf(out[0]), ref) < TOL
    dv.sparse_mlp(xd, D, Wd, idx_d, k, out, ws, flags=flags)
    torch.cuda.synchronize()
    y_ref = oracle.round_fp16(npf(x[0]) + ref)
    assert rel_err(npf(out[0]), y_ref) < TOL


@pytest.mark.parametrize("wl,d,F,keep", [("tiny", None, None, 0.25), ("opt-175b", 12288, 4096, 0.5)])
def test_mlp_skip_inactive_counts_active_rows(wl, d, F, keep):
    # with DV_SKIP_INACTIVE the MLP streams the fc2T rows of the selected
    # neurons whose activation is above zero (Eq. 1: a ReLU zero adds nothing);
    # dv_count_active counts them: the oracle's positive activations, up to
    # activations the fp32 and fp64 sums could put on either side of zero
    w, W = _mlp_case(wl, d, F)
    x = synth.hidden(w, B=1, seed=11, name="h")
    k = oracle.k_from_keep(keep, w.F)
    idx = np.sort(np.random.default_rng(1).choice(w.F, k, replace=False)).astype(np.int32)
    D = _dims(w, 8)
    ws = dv.workspace(D)
    out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    dv.count_active(cnt)
    try:
        dv.sparse_mlp(x.cuda(), D, to_dev(W), torch.from_numpy(idx).cuda(), k, out, ws,
                      flags=dv.DV_SKIP_INACTIVE | dv.DV_NO_RESIDUAL)
        torch.cuda.synchronize()
    finally:
        dv.count_active(None)
    Wh = host(W)
    ref, act = oracle.mlp_gather(np16(x[0]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], idx,
                                 ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"], return_act=True)
    assert rel_err(npf(out[0]), ref) < TOL
    near = int(np.sum(np.abs(act) < 1e-4 * max(1.0, np.abs(act).max())))
    assert abs(cnt.item() - int(np.sum(act > 0))) <= near
    assert 0 < cnt.item() < k


def test_mlp_k1_and_masked_form():
    w, W = _mlp_case("tiny")
    x = synth.hidden(w, B=1, seed=5)
    Wd, Wh = to_dev(W), host(W)
    D = _dims(w, 8)
    ws = dv.workspace(D)
    out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
    for idx in ([0], [w.F - 1], [3, 4, 900]):
        i = np.array(idx, np.int32)
        dv.sparse_mlp(x.cuda(), D, Wd, torch.from_numpy(i).cuda(), len(i), out, ws,
                      flags=dv.DV_NO_RESIDUAL)
        torch.cuda.synchronize()
        mask = np.zeros(w.F, np.uint8)
        mask[i] = 1
        ref = oracle.mlp_masked(np16(x[0]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], mask,
                                ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
        assert rel_err(npf(out[0]), ref) < TOL


@pytest.mark.parametrize("B,d", [(2, 512), (4, 512), (4, 12288)])   # 12288: largest d at B = 4
def test_mlp_batch_union(B, d):
    w, W = _mlp_case("tiny", d=d, F=2048)
    x = synth.hidden(w, B=B, seed=7)
    rng = np.random.default_rng(B)
    k = 200
    sets = np.stack([np.sort(rng.choice(w.F, k, replace=False)) for _ in range(B)]).astype(np.int32)
    u = oracle.union(sets, w.F)
    ud = torch.zeros(w.F, dtype=torch.int32, device="cuda")
    ud[: len(u)] = torch.from_numpy(u).cuda()
    cnt = torch.tensor([len(u)], dtype=torch.int32, device="cuda")
    Wd, Wh = to_dev(W), host(W)
    D = _dims(w, 8)
    ws = dv.workspace(D, B)
    out = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
    dv.sparse_mlp(x.cuda(), D, Wd, ud, min(w.F, B * k), out, ws, dev_count=cnt,
                  flags=dv.DV_NO_RESIDUAL)
    torch.cuda.synchronize()
    for b in range(B):
        ref = oracle.mlp_gather(np16(x[b]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], u,
                                ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
        assert rel_err(npf(out[b]), ref) < TOL


def test_mlp_out_of_range_index_is_flagged_and_skipped():
    w, W = _mlp_case("tiny")
    x = synth.hidden(w, B=1, seed=9)
    Wd, Wh = to_dev(W), host(W)
    D = _dims(w, 8)
    ws = dv.workspace(D)
    out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.tensor([5, 70000, 10], dtype=torch.int32, device="cuda")
    dv.sparse_mlp(x.cuda(), D, Wd, idx, 3, out, ws, dev_status=st, flags=dv.DV_NO_RESIDUAL)
    torch.cuda.synchronize()
    assert st.item() & dv.DV_DEV_BAD_INDEX
    ref = oracle.mlp_gather(np16(x[0]), Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], [5, 10],
                            ln_g=Wh["ln2_g"], ln_b=Wh["ln2_b"])
    assert rel_err(npf(out[0]), ref) < TOL


# ---------------------------------------------------------------------------
# a5-a7 head-sparse attention
# ---------------------------------------------------------------------------
def _attn_setup(w, n, B=1, seed=0):
    W = synth.layer_weights(w, 0, seed=seed, full_bias=True)
    n_max = n + 5
    K, V = synth.kv_cache(w, 0, n_max, B=B, seed=seed)
    x = synth.hidden(w, B=B, seed=seed + 1)
    return W, K, V, x, n_max


def _run_attn(w, W, K, V, x, n, n_max, sel, flags=dv.DV_NO_RESIDUAL, dev_count=None, kk=None):
    B = x.shape[0]
    D = _dims(w, n_max)
    ws = dv.workspace(D, B)
    Kd, Vd = K.cuda(), V.cuda()
    ys = torch.zeros(B, n_max, w.d, dtype=torch.float16, device="cuda")
    words = (w.h_kv + 31) // 32
    miss = torch.zeros(B, n_max, words, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(Kd, Vd, y_side=ys, kv_missing=miss)
    out = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
    sd = None if sel is None else torch.as_tensor(np.asarray(sel, np.int32)).cuda()
    k = w.h_kv if sel is None else (kk or len(sel))
    dv.sparse_attn(x.cuda(), D, to_dev(W), sd, k, kv, n, out, ws, flags=flags, dev_count=dev_count)
    torch.cuda.synchronize()
    return out, Kd, Vd, ys, miss


@pytest.mark.parametrize("wl,over,n,sel", [
    ("tiny", {}, 64, [1, 3]),
    ("tiny", {}, 0, [0, 2]),                               # only the new token
    ("tiny", {}, 64, None),                                # all heads
    ("compose", dict(d=512, h=8, h_kv=2, F=64), 300, [1]),  # GQA, 4 query heads per KV head
    ("opt-6.7b", dict(F=64), 200, [0, 5, 31]),
    ("opt-6.7b", dict(d=16384, h=8, h_kv=8, F=64), 100, [2, 5]),       # largest d
    ("compose", dict(d=512, h=8, h_kv=4, F=64), 300, [1, 3]),         # 2 query heads per KV head
    ("compose", dict(d=512, h=16, h_kv=2, F=64), 300, [0, 1]),        # 8 query heads per KV head
    ("opt-6.7b", dict(d=512, h=4, h_kv=4, F=64), 20000, [2]),         # long range: 3-stage splits
])
def test_attn_parity(wl, over, n, sel):
    w = synth.workload(wl, **over)
    W, K, V, x, n_max = _attn_setup(w, n)
    out, Kd, Vd, ys, miss = _run_attn(w, W, K, V, x, n, n_max, sel)
    Wh = host(W)
    units = list(range(w.h_kv)) if sel is None else sel
    ref = oracle.attn_gather(np16(x[0]), Wh, np16(K[0]), np16(V[0]), n, units)
    assert rel_err(npf(out[0]), ref.delta) < TOL
    Kn, Vn = Kd[0, :, n].cpu().numpy(), Vd[0, :, n].cpu().numpy()
    for u in range(w.h_kv):
        if u in units:
            assert rel_err(Kn[u].astype(float), ref.knew[u].astype(float)) < TOL
            assert rel_err(Vn[u].astype(float), ref.vnew[u].astype(float)) < TOL
        else:   # missing KV: slot n untouched, bit set, y kept
            assert np.array_equal(Kn[u].view(np.uint16), np16(K[0, u, n]).view(np.uint16))
            assert np.array_equal(Vn[u].view(np.uint16), np16(V[0, u, n]).view(np.uint16))
    bits = int(miss[0, n, 0].item()) & 0xFFFFFFFF
    for u in range(min(32, w.h_kv)):
        assert bool(bits >> u & 1) == (u not in units)
    assert np.array_equal(np16(ys[0, n]).view(np.uint16), np16(x[0]).view(np.uint16))
    # residual form
    out2, *_ = _run_attn(w, W, K, V, x, n, n_max, sel, flags=0)
    assert rel_err(npf(out2[0]), oracle.round_fp16(npf(x[0]) + ref.delta)) < TOL


def test_attn_split_count_invariance():
    w = synth.workload("opt-6.7b", F=64)
    W, K, V, x, n_max = _attn_setup(w, 1500, seed=4)
    outs = []
    for ctas in (1, 7, 64, 5000):
        dv.set_tuning(attn_ctas=ctas)
        out, *_ = _run_attn(w, W, K, V, x, 1500, n_max, [2, 9])
        outs.append(npf(out[0]))
    dv.set_tuning()
    for o in outs[1:]:
        assert rel_err(o, outs[0]) < 1e-3


@pytest.mark.parametrize("B", [2, 4])
def test_attn_batch_union(B):
    w = synth.workload("tiny")
    W, K, V, x, n_max = _attn_setup(w, 40, B=B, seed=2)
    u = np.array([0, 1, 3], np.int32)
    ud = torch.zeros(8, dtype=torch.int32, device="cuda")
    ud[:3] = torch.from_numpy(u).cuda()
    cnt = torch.tensor([3], dtype=torch.int32, device="cuda")
    out, *_ = _run_attn(w, W, K, V, x, 40, n_max, ud.cpu().numpy()[:4], dev_count=cnt, kk=4)
    Wh = host(W)
    for b in range(B):
        ref = oracle.attn_gather(np16(x[b]), Wh, np16(K[b]), np16(V[b]), 40, u)
        assert rel_err(npf(out[b]), ref.delta) < TOL


# ---------------------------------------------------------------------------
# a8-a9 KV selection + split-K over the retained buffer
# ---------------------------------------------------------------------------
def _kvsel_case(over, n, keep, seed=0, plant=None):
    w = synth.workload("compose", **over)
    n_max = n + 4
    K, V = synth.kv_cache(w, 0, n_max, B=1, seed=seed)
    K, V = K[0].clone(), V[0].clone()
    q_obs = synth.obs_queries(w, 0, seed=seed)
    if plant is not None:
        G = w.h // w.h_kv
        for u in range(w.h_kv):
            mq = q_obs[u * G:(u + 1) * G].double().mean((0, 1))
            K[u, plant] = (8.0 * mq / mq.norm() * math.sqrt(w.dh)).half()
    q = torch.randn(w.h, w.dh, generator=torch.Generator().manual_seed(seed)) * w.dh ** -0.5
    return w, n_max, K, V, q_obs, q


@pytest.mark.parametrize("over,n,keep,plant,heads", [
    (dict(h=8, h_kv=2, obs_window=16), 300, 0.125, 150, None),
    (dict(obs_window=64), 2048, 0.125, None, None),        # composition shape (32q/8kv x 128)
    (dict(h=8, h_kv=2, obs_window=16), 100, 1.0, None, None),   # budget covers everything
    (dict(h=8, h_kv=2, obs_window=16), 300, 0.05, None, None),  # budget below sinks + window
    # 4 x 24 window queries per KV head: not a multiple of 64, so the scoring
    # runs on the CUDA-core kernels instead of the tensor cores
    (dict(h=8, h_kv=2, obs_window=24), 300, 0.125, 150, None),
    # the composition's long contexts: the kernels run on every KV head, the
    # fp64 oracle's pooled scores are computed for all 8 heads at 32K and for
    # two of them at 128K (the scoring pass is 34 G multiply-adds per layer)
    (dict(obs_window=64), 32768, 0.125, 20000, None),
    (dict(obs_window=64), 131072, 0.125, None, [0, 5]),
])
def test_kv_select_parity(over, n, keep, plant, heads):
    w, n_max, K, V, q_obs, q = _kvsel_case(over, n, keep, plant=plant)
    W = w.obs_window
    b = oracle.kv_budget(n, keep)
    b_max = max(b, 4 + W) + 8
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws = dv.workspace(D, 1, dv.DV_KV_RESELECT)
    Kd, Vd = K[None].cuda(), V[None].cuda()
    Kr = torch.zeros(w.h_kv, b_max, w.dh, dtype=torch.float16, device="cuda")
    Vr = torch.zeros_like(Kr)
    kp = torch.zeros(w.h_kv, b_max, dtype=torch.int32, device="cuda")
    kc = torch.zeros(w.h_kv, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(Kd, Vd, Kr=Kr, Vr=Vr, kept_pos=kp, kept_count=kc, b_max=b_max)
    H = torch.zeros(w.h, w.dh, device="cuda")
    sel = torch.zeros(w.h_kv, n, device="cuda")
    qd = q.cuda()
    dv.kv_select_attn(qd, D, kv, n, H, ws, q_obs=q_obs.cuda(), obs_window=W, kv_keep=keep,
                      flags=dv.DV_KV_RESELECT, sel_scores=sel)
    torch.cuda.synchronize()
    G = w.h // w.h_kv
    heads = list(range(w.h_kv)) if heads is None else heads
    qo, Kh = np16(q_obs), np16(K)
    ref_sm = np.zeros((w.h_kv, n))
    for u in heads:
        ref_sm[u] = oracle.kv_smooth(oracle.kv_pool(qo[u * G:(u + 1) * G], Kh[u:u + 1], n))[0]
    gs = npf(sel)
    assert rel_err(gs[heads], ref_sm[heads]) < 1e-4
    counts = kc.cpu().numpy()
    scale = w.dh ** -0.5
    for u in heads:
        kept = oracle.kv_choose(gs[u], 4, W, b)           # same decision on the GPU's scores
        assert counts[u] == len(kept)
        assert np.array_equal(kp[u, : len(kept)].cpu().numpy(), kept)
        assert np.array_equal(np16(Kr[u, : len(kept)]).view(np.uint16),
                              np16(K[u, kept]).view(np.uint16))
        if plant is not None:
            assert plant in kept
        ref_kept = oracle.kv_choose(ref_sm[u], 4, W, b)
        forced = [p for p in range(n) if p < 4 or p >= n - W]
        check_kv_kept(kept, ref_kept, ref_sm[u], gs[u], forced)
        # attention of every query head of u over kept + the new token (slot n)
        for g in range(G):
            j = u * G + g
            Hr = oracle.attend(npf(q[j]) / scale, np16(K[u]), np16(V[u]),
                               np16(K[u, n]).astype(float), np16(V[u, n]).astype(float), scale,
                               pos=kept)
            assert rel_err(npf(H[j]), Hr) < TOL
    # dense split-K over the full cache, same kernel
    dv.kv_select_attn(qd, D, kv, n, H, ws, flags=dv.DV_KV_DENSE)
    torch.cuda.synchronize()
    for j in (0, w.h - 1):
        u = j // (w.h // w.h_kv)
        Hr = oracle.attend(npf(q[j]) / scale, np16(K[u, :n]), np16(V[u, :n]),
                           np16(K[u, n]).astype(float), np16(V[u, n]).astype(float), scale)
        assert rel_err(npf(H[j]), Hr) < TOL
