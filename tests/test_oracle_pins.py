"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here compares the oracle with something other than itself:
closed forms worked by hand, special cases that reduce to a library routine
(numpy), brute force on tiny inputs, and invariants that follow from the
definitions in "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference
Time" (§2.3 Eq. 1-2, §4.1) and "Where Activation Sparsity and KV-Cache
Sparsity Cross in LLM Decoding" (App. A). Inputs are chosen so that a dropped
term, a wrong sign or index, or a transposed operand fails one of them.
"""
import itertools
import math

import numpy as np
import pytest

import oracle

F16 = np.float16
TIGHT = 1e-12


def _close(a, b, rtol=0.0, atol=TIGHT):
    """Strict comparison: |a - b| <= atol + rtol |b| elementwise (no hidden default rtol)."""
    return bool(np.all(np.abs(np.asarray(a, float) - np.asarray(b, float))
                       <= atol + rtol * np.abs(np.asarray(b, float))))


def f16(a):
    return np.asarray(a, dtype=np.float64).astype(F16)


# --------------------------------------------------------------------------
# fp16 codec (IEEE 754 binary16) against numpy
# --------------------------------------------------------------------------
def test_fp16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle.h2d(bits)
    ref = bits.view(F16).astype(np.float64)
    fin = ~np.isnan(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.isnan(got[~fin]).all()


def test_fp16_encode_matches_numpy_including_ties():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(100000) * np.exp(rng.uniform(-25, 11.5, 100000))
    # exact midpoints between neighbouring halves: ties go to the even code
    h = rng.integers(0, 0x7BFF, 20000).astype(np.uint16)
    lo = h.view(F16).astype(np.float64)
    hi = (h + 1).view(F16).astype(np.float64)
    x = np.concatenate([x, (lo + hi) / 2, -(lo + hi) / 2, [0.0, -0.0, 65504.0, 65519.99, 65520.0,
                                                          1e6, 2.0**-24, 2.0**-25, 3 * 2.0**-26]])
    with np.errstate(over="ignore"):
        ref = x.astype(F16).view(np.uint16)
    assert np.array_equal(oracle.d2h(x), ref)


# --------------------------------------------------------------------------
# LayerNorm: closed forms
# --------------------------------------------------------------------------
def test_layernorm_closed_form():
    # x = 3 + (+1, -1, ...): mean 3, biased variance 1 -> z = +-1/sqrt(1+eps)
    d = 16
    x = f16(3.0 + np.tile([1.0, -1.0], d // 2))
    z = oracle.layernorm(x, eps=1e-5)
    s = 1.0 / math.sqrt(1.0 + 1e-5)
    assert _close(z, np.tile([s, -s], d // 2), rtol=0, atol=TIGHT)
    # gain and bias: z' = g z + b
    g = f16(np.full(d, 2.0))
    b = f16(np.linspace(-1, 1, d))
    z2 = oracle.layernorm(x, g, b, eps=1e-5)
    assert _close(z2, 2 * z + b.astype(np.float64), rtol=0, atol=TIGHT)


def test_layernorm_moments():
    rng = np.random.default_rng(1)
    x = f16(rng.standard_normal(1000) * 4 + 7)
    z = oracle.layernorm(x, eps=1e-5)
    xd = x.astype(np.float64)
    var = xd.var()  # biased variance, a library routine
    assert abs(z.mean()) < 1e-12
    assert abs((z**2).mean() - var / (var + 1e-5)) < 1e-12


# --------------------------------------------------------------------------
# Predictor (Deja Vu §4.1 "Design"): worked example and the MaxIP reduction
# --------------------------------------------------------------------------
def test_predict_worked_example():
    # u = 1*3 + 2*(-1) = 1 ; s = (2*1, -3*1)
    s = oracle.predict(f16([3.0, -1.0]), f16([[1.0, 2.0]]), f16([[2.0], [-3.0]]))
    assert np.array_equal(s, [2.0, -3.0])
    # ReLU between the layers: u = -1 -> 0 -> s = 0
    s = oracle.predict(f16([3.0, -1.0]), f16([[-1.0, -2.0]]), f16([[2.0], [-3.0]]), relu=True)
    assert np.array_equal(s, [0.0, 0.0])
    s = oracle.predict(f16([3.0, -1.0]), f16([[-1.0, -2.0]]), f16([[2.0], [-3.0]]), relu=False)
    assert np.array_equal(s, [-2.0, 3.0])


def test_predict_maxip_special_case():
    # Definition 4.1 / Remark 4.2: with P1 = I (r = d) and P2 = fc1 the scores
    # are the inner products <y, w_j> and top-1 is the exact MaxIP answer.
    rng = np.random.default_rng(2)
    d, F = 64, 300
    y = f16(rng.standard_normal(d))
    fc1 = f16(rng.standard_normal((F, d)) * 0.02)
    s = oracle.predict(y, f16(np.eye(d)), fc1)
    ref = fc1.astype(np.float64) @ y.astype(np.float64)
    assert _close(s, ref, rtol=1e-13, atol=1e-15)
    assert oracle.topk(s, 1)[0] == int(np.argmax(ref))
    k = 17
    assert set(oracle.topk(s, k)) == set(np.argsort(-ref, kind="stable")[:k])


# --------------------------------------------------------------------------
# Top-k (budget of §2.3): brute force over all subsets
# --------------------------------------------------------------------------
def _brute_topk(s, k):
    best = None
    for sub in itertools.combinations(range(len(s)), k):
        key = (sorted((s[i] for i in sub), reverse=True), [-i for i in sorted(sub)])
        # maximal sorted score vector, then lexicographically smallest indices
        if best is None or key > best[0]:
            best = (key, sub)
    return np.array(sorted(best[1]), dtype=np.int32)


@pytest.mark.parametrize("case", ["random", "ties", "equal", "signed_zero", "ulp"])
def test_topk_brute_force(case):
    rng = np.random.default_rng(3)
    for trial in range(20):
        N = int(rng.integers(1, 11))
        if case == "random":
            s = rng.standard_normal(N)
        elif case == "ties":
            s = rng.integers(-2, 3, N).astype(np.float64)
        elif case == "equal":
            s = np.full(N, 1.5)
        elif case == "signed_zero":
            s = rng.choice([0.0, -0.0, 1.0, -1.0], N)
        else:
            base = np.float32(1.0)
            s = np.array([np.nextafter(base, np.float32(2.0)) if rng.random() < 0.5 else base
                          for _ in range(N)], dtype=np.float32).astype(np.float64)
        for k in range(1, N + 1):
            assert np.array_equal(oracle.topk(s, k), _brute_topk(list(s), k)), (s, k)


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.topk(np.zeros(4), 5)
    with pytest.raises(ValueError):
        oracle.topk(np.array([1.0, np.nan]), 1)


def test_union_brute_force():
    rng = np.random.default_rng(4)
    idx = np.stack([np.sort(rng.choice(50, 10, replace=False)) for _ in range(4)])
    assert np.array_equal(oracle.union(idx, 50), np.array(sorted(set(idx.ravel()))))


def test_k_from_keep():
    assert oracle.k_from_keep(0.10, 49152) == 4915
    assert oracle.k_from_keep(0.25, 1024) == 256
    assert oracle.k_from_keep(0.5, 4) == 2
    assert oracle.k_from_keep(0.29, 100) == 29
    assert oracle.k_from_keep(1e-9, 100) == 1
    assert oracle.k_from_keep(1.0, 96) == 96


# --------------------------------------------------------------------------
# MLP block (Eq. 1): a worked example, then the invariants
# --------------------------------------------------------------------------
def _mlp_example():
    d = 8
    x = f16(3.0 + np.tile([1.0, -1.0], 4))        # z = +-s, s = 1/sqrt(1+eps)
    fc1 = np.zeros((3, d))
    fc1[0, 0] = 1.0                                 # pre-act  s + 0.25
    fc1[1, 1] = 1.0                                 # pre-act -s + 0.5  -> ReLU 0
    fc1[2, :3] = 0.5                                # pre-act 0.5 s - 0.125
    b1 = [0.25, 0.5, -0.125]
    fc2T = np.zeros((3, d))
    fc2T[0, 2] = 2.0
    fc2T[1, :] = 1.0
    fc2T[2, 0], fc2T[2, 7] = 1.0, -1.0
    b2 = np.zeros(d)
    b2[6] = 0.5
    s = 1.0 / math.sqrt(1.0 + 1e-5)
    a0, a2 = s + 0.25, 0.5 * s - 0.125
    expect = np.array([a2, 0, 2 * a0, 0, 0, 0, 0.5, -a2])
    return x, f16(fc1), f16(b1), f16(fc2T), f16(b2), expect, (a0, 0.0, a2)


def test_mlp_worked_example():
    x, fc1, b1, fc2T, b2, expect, acts = _mlp_example()
    out, act = oracle.mlp_gather(x, fc1, b1, fc2T, b2, [0, 1, 2], return_act=True)
    assert _close(out, expect, rtol=0, atol=TIGHT)
    assert _close(act, acts, rtol=0, atol=TIGHT)
    # neuron 1 is inactive (ReLU), so dropping it from the set changes nothing
    assert _close(oracle.mlp_gather(x, fc1, b1, fc2T, b2, [0, 2]), expect, atol=TIGHT)
    # only neuron 1 selected: the block output is b2
    assert _close(oracle.mlp_gather(x, fc1, b1, fc2T, b2, [1]), b2.astype(float), atol=TIGHT)
    # masked-dense form of the same example
    assert _close(oracle.mlp_masked(x, fc1, b1, fc2T, b2), expect, atol=TIGHT)
    assert _close(oracle.mlp_masked(x, fc1, b1, fc2T, b2, mask=[1, 0, 0]),
                       expect - np.array([acts[2], 0, 0, 0, 0, 0, 0, -acts[2]]), atol=TIGHT)


def _rand_mlp(rng, d=48, F=96):
    x = f16(rng.standard_normal(d))
    fc1 = f16(rng.standard_normal((F, d)) * 0.2)
    b1 = f16(rng.normal(-0.2, 0.1, F))
    fc2T = f16(rng.standard_normal((F, d)) * 0.2)
    b2 = f16(rng.standard_normal(d) * 0.1)
    g = f16(rng.normal(1.0, 0.1, d))
    be = f16(rng.normal(0.0, 0.1, d))
    return x, fc1, b1, fc2T, b2, g, be


def test_mlp_gather_equals_masked_dense():
    rng = np.random.default_rng(5)
    x, fc1, b1, fc2T, b2, g, be = _rand_mlp(rng)
    F = fc1.shape[0]
    for k in (1, 7, 40, F):
        idx = np.sort(rng.choice(F, k, replace=False)).astype(np.int32)
        mask = np.zeros(F, np.uint8)
        mask[idx] = 1
        a = oracle.mlp_gather(x, fc1, b1, fc2T, b2, idx, ln_g=g, ln_b=be)
        m = oracle.mlp_masked(x, fc1, b1, fc2T, b2, mask, ln_g=g, ln_b=be)
        assert _close(a, m, rtol=1e-13, atol=1e-13)
    # keep = 1.0: the sparse block is the dense block
    dense = oracle.mlp_masked(x, fc1, b1, fc2T, b2, None, ln_g=g, ln_b=be)
    full = oracle.mlp_gather(x, fc1, b1, fc2T, b2, np.arange(F), ln_g=g, ln_b=be)
    assert _close(dense, full, rtol=1e-13, atol=1e-13)


def test_mlp_neuron_permutation_invariance():
    # A neuron is a pair (row j of fc1 with b1[j], row j of fc2T): renumbering
    # neurons must not change the block output.
    rng = np.random.default_rng(6)
    x, fc1, b1, fc2T, b2, g, be = _rand_mlp(rng)
    F = fc1.shape[0]
    perm = rng.permutation(F)
    idx = np.sort(rng.choice(F, 30, replace=False))
    inv = np.argsort(perm)
    a = oracle.mlp_gather(x, fc1, b1, fc2T, b2, idx)
    b = oracle.mlp_gather(x, fc1[perm], b1[perm], fc2T[perm], b2, np.sort(inv[idx]))
    assert _close(a, b, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# MHA block (Eq. 2): closed forms
# --------------------------------------------------------------------------
def _attn_weights(d, h, hkv, dh, rng=None, scale_w=0.0):
    z = lambda *s: np.zeros(s)
    r = (lambda *s: rng.standard_normal(s) * scale_w) if rng is not None else z
    return {"Wq": f16(r(h * dh, d)), "Wk": f16(r(hkv * dh, d)), "Wv": f16(r(hkv * dh, d)),
            "WoT": f16(r(h * dh, d))}


def test_attn_single_token_is_v_new():
    # n = 0 cached tokens: the softmax has one entry, H = v_new (rounded to fp16)
    d, dh = 4, 2
    x = f16([4.0, 2.0, 4.0, 2.0])                   # LN -> (+s, -s, +s, -s)
    W = _attn_weights(d, 1, 1, dh)
    Wv = np.zeros((dh, d))
    Wv[0, 0], Wv[1, 1] = 1.0, 1.0                   # v = (s, -s) -> fp16 (1, -1)
    W["Wv"] = f16(Wv)
    WoT = np.zeros((dh, d))
    WoT[0] = [1, 2, 0, 0]
    WoT[1] = [0, 0, 3, 0]
    W["WoT"] = f16(WoT)
    W["bo"] = f16([0.5, 0, 0, -0.25])
    K = np.zeros((1, 4, dh), F16)
    out = oracle.attn_gather(x, W, K, K.copy(), 0, [0])
    assert np.array_equal(out.vnew.astype(float), [[1.0, -1.0]])
    assert _close(out.H, [[1.0, -1.0]], atol=TIGHT)
    assert _close(out.delta, [1.5, 2.0, -3.0, -0.25], atol=TIGHT)


def test_attn_output_projection_multi_head():
    # two heads, n = 0: H_j = v_new of head j (set by the bias, Wv = 0); the
    # block output is sum_j sum_c H_j[c] WoT[j dh + c] + bo
    d, h, dh = 4, 2, 2
    x = f16([1.0, -1.0, 0.5, 0.0])
    W = _attn_weights(d, h, h, dh)
    W["bv"] = f16([1.0, -1.0, 2.0, 0.5])
    WoT = np.array([[1, 0, 0, 0], [0, 1, 0, 0], [0, 0, 1, 0], [1, 1, 1, 1]], float)
    W["WoT"] = f16(WoT)
    K = np.zeros((h, 2, dh), F16)
    out = oracle.attn_gather(x, W, K, K.copy(), 0, [0, 1])
    assert _close(out.H, [[1.0, -1.0], [2.0, 0.5]])
    assert _close(out.delta, [1.5, -0.5, 2.5, 0.5])
    out = oracle.attn_gather(x, W, K, K.copy(), 0, [1])
    assert _close(out.delta, [0.5, 0.5, 2.5, 0.5])


def test_attn_uniform_scores_average_values():
    # keys all zero (cache and new) -> equal scores -> H = mean of the n cached
    # values and the new one. Catches off-by-one in n and a missing new token.
    rng = np.random.default_rng(7)
    d, dh, n, n_max = 8, 4, 5, 9
    x = f16(rng.standard_normal(d))
    W = _attn_weights(d, 1, 1, dh)
    W["bv"] = f16([1.0, -2.0, 0.5, 3.0])            # v_new = bv (Wv = 0)
    W["Wq"] = f16(rng.standard_normal((dh, d)))     # scores stay 0 because K = 0
    K = np.zeros((1, n_max, dh), F16)
    V = f16(rng.standard_normal((1, n_max, dh)))
    out = oracle.attn_gather(x, W, K, V, n, [0])
    expect = (V[0, :n].astype(float).sum(0) + np.array([1.0, -2.0, 0.5, 3.0])) / (n + 1)
    assert _close(out.H[0], expect, atol=TIGHT)
    # scale 0 gives the same average whatever the keys are
    K2 = f16(rng.standard_normal((1, n_max, dh)))
    out = oracle.attn_gather(x, W, K2, V, n, [0], scale=0.0)
    assert _close(out.H[0], expect, atol=TIGHT)


def test_attn_two_keys_is_logistic():
    # two keys: the softmax weight of key 0 is the logistic function of the
    # score difference (a textbook identity)
    d, dh = 4, 2
    x = f16([4.0, 2.0, 4.0, 2.0])
    W = _attn_weights(d, 1, 1, dh)
    W["bq"] = f16([1.0, 0.5])                       # q = (1, 0.5)
    W["bk"] = f16([0.25, -1.0])                     # k_new = (0.25, -1)
    W["bv"] = f16([0.0, 1.0])                       # v_new = (0, 1)
    K = np.zeros((1, 2, dh), F16)
    K[0, 0] = [2.0, 1.0]
    V = np.zeros((1, 2, dh), F16)
    V[0, 0] = [1.0, 0.0]
    scale = 0.75
    out = oracle.attn_gather(x, W, K, V, 1, [0], scale=scale)
    s0 = scale * (1 * 2.0 + 0.5 * 1.0)
    s1 = scale * (1 * 0.25 + 0.5 * -1.0)
    p0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
    assert _close(out.H[0], [p0, 1 - p0], atol=TIGHT)


def test_attn_dominant_key():
    rng = np.random.default_rng(8)
    d, dh, n = 8, 4, 6
    x = f16(rng.standard_normal(d))
    W = _attn_weights(d, 1, 1, dh)
    W["bq"] = f16([1.0, 0, 0, 0])
    K = np.zeros((1, n + 1, dh), F16)
    K[0, 3, 0] = 60.0                               # score 30 above all the others
    V = f16(rng.standard_normal((1, n + 1, dh)))
    out = oracle.attn_gather(x, W, K, V, n, [0], scale=0.5)
    assert _close(out.H[0], V[0, 3].astype(float), atol=1e-11)


def test_attn_gqa_mapping():
    # h = 4 query heads over h_kv = 2 KV heads: heads 0,1 read KV head 0 and
    # heads 2,3 read KV head 1. Constant values per KV head reveal the mapping.
    d, dh, n = 8, 2, 3
    rng = np.random.default_rng(9)
    x = f16(rng.standard_normal(d))
    W = _attn_weights(d, 4, 2, dh, rng, 0.3)
    W["Wv"] = f16(np.zeros((2 * dh, d)))
    W["bv"] = f16([1, 1, -1, -1])
    V = np.zeros((2, n + 1, dh), F16)
    V[0], V[1] = 1.0, -1.0
    K = f16(rng.standard_normal((2, n + 1, dh)))
    out = oracle.attn_gather(x, W, K, V, n, [0, 1])
    assert _close(out.H, [[1, 1], [1, 1], [-1, -1], [-1, -1]], atol=TIGHT)
    # selecting only unit 1 leaves heads 0 and 1 out of the output
    out = oracle.attn_gather(x, W, K, V, n, [1])
    assert _close(out.H, [[0, 0], [0, 0], [-1, -1], [-1, -1]], atol=TIGHT)


def test_attn_gather_equals_masked_dense():
    rng = np.random.default_rng(10)
    d, h, dh, n, n_max = 32, 6, 8, 7, 10
    x = f16(rng.standard_normal(d))
    W = _attn_weights(d, h, h, dh, rng, 0.2)
    for k in ("bq", "bk", "bv"):
        W[k] = f16(rng.standard_normal(h * dh) * 0.1)
    W["bo"] = f16(rng.standard_normal(d) * 0.1)
    W["ln1_g"] = f16(rng.normal(1, 0.1, d))
    W["ln1_b"] = f16(rng.normal(0, 0.1, d))
    K = f16(rng.standard_normal((h, n_max, dh)))
    V = f16(rng.standard_normal((h, n_max, dh)))
    sel = np.array([1, 2, 5], np.int32)
    mask = np.zeros(h, np.uint8)
    mask[sel] = 1
    a = oracle.attn_gather(x, W, K, V, n, sel)
    m = oracle.attn_masked(x, W, K, V, n, mask)
    assert _close(a.delta, m.delta, rtol=1e-13, atol=1e-13)
    assert np.array_equal(a.knew[sel], m.knew[sel])
    full = oracle.attn_gather(x, W, K, V, n, np.arange(h))
    dense = oracle.attn_masked(x, W, K, V, n, None)
    assert _close(full.delta, dense.delta, rtol=1e-13, atol=1e-13)


def test_attend_positions_equals_gathered_rows():
    rng = np.random.default_rng(11)
    dh, n = 8, 20
    q = rng.standard_normal(dh)
    K = f16(rng.standard_normal((n, dh)))
    V = f16(rng.standard_normal((n, dh)))
    kn, vn = rng.standard_normal(dh), rng.standard_normal(dh)
    pos = np.array([0, 3, 4, 11, 19])
    a = oracle.attend(q, K, V, kn, vn, 0.3, pos)
    b = oracle.attend(q, K[pos], V[pos], kn, vn, 0.3)
    assert _close(a, b, atol=TIGHT)


# --------------------------------------------------------------------------
# KV selection (ByteCross §4.1, App. A)
# --------------------------------------------------------------------------
def test_kv_pool_uniform_closed_form():
    # all keys equal -> obs query t at position p_t spreads 1/(p_t+1) over
    # positions 0..p_t; the pool sums over the W queries and the G heads.
    h, hkv, dh, n, W = 4, 2, 8, 40, 6
    rng = np.random.default_rng(12)
    q = f16(rng.standard_normal((h, W, dh)))
    K = np.zeros((hkv, n + 3, dh), F16)
    pooled = oracle.kv_pool(q, K, n)
    G = h // hkv
    expect = np.zeros(n)
    for t in range(W):
        pt = n - W + t
        expect[: pt + 1] += 1.0 / (pt + 1)
    assert _close(pooled, G * expect[None, :], atol=1e-12)


def test_kv_pool_mass_and_planted_key():
    h, hkv, dh, n, W = 8, 2, 16, 300, 16
    rng = np.random.default_rng(13)
    q = f16(rng.standard_normal((h, W, dh)))
    K = f16(rng.standard_normal((hkv, n, dh)))
    pooled = oracle.kv_pool(q, K, n)
    G = h // hkv
    assert _close(pooled.sum(1), G * W, atol=1e-9)
    # plant a key aligned with the group's mean query at position 150
    K = K.copy()
    for u in range(hkv):
        mq = q[u * G:(u + 1) * G].astype(float).mean((0, 1))
        K[u, 150] = f16(8.0 * mq / np.linalg.norm(mq) * math.sqrt(dh))
    kept, sm = oracle.kv_select(q, K, n, keep=0.125)
    b = oracle.kv_budget(n, 0.125)
    for u in range(hkv):
        assert 150 in kept[u]
        assert len(kept[u]) == b
        assert all(p in kept[u] for p in range(4))
        assert all(p in kept[u] for p in range(n - W, n))
        assert np.all(np.diff(kept[u]) > 0)


def test_kv_smooth_spike_and_edges():
    n = 20
    x = np.zeros(n)
    x[10] = 7.0
    sm = oracle.kv_smooth(x, 7)
    expect = np.zeros(n)
    expect[7:14] = 1.0
    assert _close(sm, expect, atol=TIGHT)
    x = np.zeros(n)
    x[0] = 7.0                                      # zero padding at the left edge
    expect = np.zeros(n)
    expect[:4] = 1.0
    assert _close(oracle.kv_smooth(x, 7), expect, atol=TIGHT)
    x = np.ones(n)                                  # edges see fewer terms, still / 7
    sm = oracle.kv_smooth(x, 7)
    assert _close(sm[3:-3], 1.0) and np.isclose(sm[0], 4 / 7) and np.isclose(sm[-1], 4 / 7)


def test_kv_choose_rules():
    n, W, S = 50, 8, 4
    flat = np.zeros(n)
    # uniform scores: the extra budget goes to the lowest free positions
    kept = oracle.kv_choose(flat, S, W, 20)
    assert list(kept) == list(range(4)) + list(range(4, 12)) + list(range(n - W, n))
    # budget covering everything keeps everything
    assert list(oracle.kv_choose(np.random.default_rng(0).random(n), S, W, n)) == list(range(n))
    assert list(oracle.kv_choose(flat, S, W, n + 10)) == list(range(n))
    # a budget below the forced set keeps the forced set only
    assert list(oracle.kv_choose(flat, S, W, 5)) == list(range(4)) + list(range(n - W, n))
    # highest scores win, forced positions do not count twice
    sm = np.zeros(n)
    sm[[20, 30, 31, 45]] = [3.0, 2.0, 2.0, 9.0]    # 45 lies in the window
    kept = oracle.kv_choose(sm, S, W, S + W + 2)
    assert list(kept) == list(range(4)) + [20, 30] + list(range(n - W, n))


def test_kv_budget():
    assert oracle.kv_budget(2048, 0.125) == 256
    assert oracle.kv_budget(131072, 0.125) == 16384
    assert oracle.kv_budget(100, 0.3) == 30


# --------------------------------------------------------------------------
# multi-step decode with missing K/V ("Deja Vu" §4.2)
# --------------------------------------------------------------------------
def _np_layernorm(x, eps=1e-5):
    x = np.asarray(x, float)
    mu = x.mean()
    return (x - mu) / np.sqrt(((x - mu) ** 2).mean() + eps)


def test_token_kv_is_the_projection_of_the_normalised_token():
    # k = fp16(LN(y) W^K^T + b_k), v likewise, computed here with numpy's matmul
    rng = np.random.default_rng(5)
    d, hkv, dh = 48, 3, 8
    W = _attn_weights(d, hkv, hkv, dh, rng, 0.3)
    W["bk"] = f16(rng.standard_normal(hkv * dh) * 0.1)
    W["bv"] = f16(rng.standard_normal(hkv * dh) * 0.1)
    y = f16(rng.standard_normal(d) * 2 + 0.5)
    z = _np_layernorm(y.astype(float))
    k_ref = (W["Wk"].astype(float) @ z + W["bk"].astype(float)).astype(F16).reshape(hkv, dh)
    v_ref = (W["Wv"].astype(float) @ z + W["bv"].astype(float)).astype(F16).reshape(hkv, dh)
    k, v = oracle.token_kv(y, W, hkv, dh)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_attn_steps_cache_rows_come_from_their_own_token():
    # however the units were selected, position n0 + t ends up holding the k, v
    # of token t (an off-by-one in the position, a row left at zero or a row
    # taken from another token fails), and the prefilled rows are untouched
    rng = np.random.default_rng(6)
    d, hkv, dh, n0, T = 32, 4, 4, 5, 6
    W = _attn_weights(d, hkv, hkv, dh, rng, 0.4)
    K = f16(rng.standard_normal((hkv, n0 + T + 1, dh)))
    V = f16(rng.standard_normal((hkv, n0 + T + 1, dh)))
    ys = [f16(rng.standard_normal(d)) for _ in range(T)]
    sels = [[0], [1, 2], [0], [3], [0, 1, 2, 3], [2]]
    outs, Kf, Vf = oracle.attn_steps(ys, W, K, V, n0, sels)
    assert np.array_equal(Kf[:, :n0], K[:, :n0]) and np.array_equal(Vf[:, :n0], V[:, :n0])
    for t, y in enumerate(ys):
        z = _np_layernorm(y.astype(float))
        k_ref = (W["Wk"].astype(float) @ z).astype(F16).reshape(hkv, dh)
        assert np.array_equal(Kf[:, n0 + t], k_ref)
    # unit 3 is selected only at step 3: it attends over five filled rows of
    # its own tokens' keys; the same step with every unit selected at every
    # earlier step gives it the same output
    dense = oracle.attn_steps(ys, W, K, V, n0, [[0, 1, 2, 3]] * T)[0]
    assert _close(outs[3].H[3], dense[3].H[3], atol=TIGHT)
    assert not np.allclose(outs[3].H[3], 0.0)


# --------------------------------------------------------------------------
# One decode layer ("Deja Vu" App. C.3: y~ = y + MHA(y), y^ = y~ + MLP(y~)),
# with the fp16 points where the library hands values on: h = fp16(y + MHA)
# and y' = fp16(h + MLP(h))
# --------------------------------------------------------------------------
def _layer_example():
    """d 4, one head of d_h 2, F 2, no cached token, eps 0. Worked by hand:

    * LN1(x), x = (4, 2, 4, 2): mean 3, biased variance 1, so z = (1, -1, 1, -1).
    * W^Q = W^K = 0 and no bias: q = k_new = 0; W^V = 0, b_v = (1, -1): v_new =
      (1, -1), exact in fp16. With n = 0 the only key is the new token, whose
      softmax weight is 1: H = (1, -1).
    * MHA = 1 WoT[0] - 1 WoT[1] + b_o = (1, 0, 0, 2) - (0, -1, 1, -1)
      + (2^-10, 0, 0, 0) = (1 + 2^-10, 1, -1, 3).
    * x + MHA = (5 + 2^-10, 3, 3, 5). fp16 values in [4, 8) are 2^-8 apart, so
      5 + 2^-10 rounds to 5: h = (5, 3, 3, 5).
    * LN2(h): mean 4, biased variance 1, z' = (1, -1, -1, 1). Neuron 0 reads
      z'[3] = 1 (bias 0): a_0 = 1. Neuron 1 reads z'[2] + 0.5 = -0.5: a_1 = 0.
    * MLP = a_0 fc2T[0] + b_2 = (0.25 + 3 2^-11, 0, 0, 0).
    * h + MLP = (5.25 + 3 2^-11, 3, 3, 5); 3 2^-11 is below half the spacing
      (2^-9), so y' = (5.25, 3, 3, 5).

    Had the MLP read x instead of h, LN2 would give (1, -1, 1, -1): a_0 = 0,
    a_1 = 1.5 and y' = (5.0, 3, 3.75, 5). Had y' added the unrounded h, its
    first entry 5.25 + 5 2^-11 would pass the midpoint 5.25 + 2^-9 and round to
    5.25 + 2^-8. Unrounded, it would be 5.25 + 3 2^-11.
    """
    x = f16([4.0, 2.0, 4.0, 2.0])
    W = {"Wq": f16(np.zeros((2, 4))), "Wk": f16(np.zeros((2, 4))), "Wv": f16(np.zeros((2, 4))),
         "bv": f16([1.0, -1.0]),
         "WoT": f16([[1, 0, 0, 2], [0, -1, 1, -1]]), "bo": f16([2.0 ** -10, 0, 0, 0]),
         "fc1": f16([[0, 0, 0, 1], [0, 0, 1, 0]]), "b1": f16([0.0, 0.5]),
         "fc2T": f16([[0.25, 0, 0, 0], [0, 0, 0.5, 0]]), "b2": f16([3 * 2.0 ** -11, 0, 0, 0])}
    K = np.zeros((1, 2, 2), F16)
    return x, W, K


def test_layer_worked_example():
    x, W, K = _layer_example()
    y, hmid, a, m = oracle.layer(x, W, K, K.copy(), 0, [0], [0, 1], eps=0.0)
    assert _close(a.H, [[1.0, -1.0]], atol=TIGHT)
    assert _close(a.delta, [1 + 2.0 ** -10, 1, -1, 3], atol=TIGHT)
    assert hmid.dtype == F16 and np.array_equal(hmid.astype(float), [5, 3, 3, 5])
    assert _close(m, [0.25 + 3 * 2.0 ** -11, 0, 0, 0], atol=TIGHT)
    assert y.dtype == F16 and np.array_equal(y.astype(float), [5.25, 3, 3, 5])
    # neuron 1 is inactive: selecting neuron 0 alone gives the same layer
    y0, *_ = oracle.layer(x, W, K, K.copy(), 0, [0], [0], eps=0.0)
    assert np.array_equal(y0, y)
    # neuron 1 alone: the MLP output is b_2, y' = fp16(h + b_2) = h
    y1, _, _, m1 = oracle.layer(x, W, K, K.copy(), 0, [0], [1], eps=0.0)
    assert _close(m1, [3 * 2.0 ** -11, 0, 0, 0], atol=TIGHT)
    assert np.array_equal(y1.astype(float), [5, 3, 3, 5])


def _np_dense_layer(x, W, K, V, n, scale, eps):
    """The dense OPT layer with numpy's matmul (every head, every neuron): the
    keep = 1 case of Eq. 1-2, with the new k, v and h, y' rounded to fp16."""
    def ln(v, g, b):
        v = np.asarray(v, float)
        mu = v.mean()
        out = (v - mu) / np.sqrt(((v - mu) ** 2).mean() + eps)
        return out * (1.0 if g is None else g.astype(float)) + (0.0 if b is None else b.astype(float))

    get = lambda k: None if W.get(k) is None else W[k].astype(float)
    bias = lambda k, n_: np.zeros(n_) if W.get(k) is None else W[k].astype(float)
    hkv, _, dh = K.shape
    h = W["Wq"].shape[0] // dh
    G = h // hkv
    z = ln(x.astype(float), W.get("ln1_g"), W.get("ln1_b"))
    q = (get("Wq") @ z + bias("bq", h * dh)).reshape(h, dh)
    k = (get("Wk") @ z + bias("bk", hkv * dh)).astype(F16).astype(float).reshape(hkv, dh)
    v = (get("Wv") @ z + bias("bv", hkv * dh)).astype(F16).astype(float).reshape(hkv, dh)
    Hs = np.zeros((h, dh))
    for j in range(h):
        u = j // G
        keys = np.vstack([K[u, :n].astype(float), k[u]])
        vals = np.vstack([V[u, :n].astype(float), v[u]])
        s = keys @ q[j] * scale
        p = np.exp(s - s.max())
        Hs[j] = (p / p.sum()) @ vals
    mha = Hs.reshape(-1) @ get("WoT") + bias("bo", x.size)
    hmid = (x.astype(float) + mha).astype(F16)
    z2 = ln(hmid.astype(float), W.get("ln2_g"), W.get("ln2_b"))
    act = np.maximum(get("fc1") @ z2 + bias("b1", W["fc1"].shape[0]), 0.0)
    mlp = act @ get("fc2T") + bias("b2", x.size)
    return (hmid.astype(float) + mlp).astype(F16), hmid, mha, mlp


def _rand_layer(rng, d=32, h=4, hkv=2, dh=8, F=64, n=6):
    W = _attn_weights(d, h, hkv, dh, rng, 0.25)
    W.update({"bq": f16(rng.standard_normal(h * dh) * 0.1),
              "bk": f16(rng.standard_normal(hkv * dh) * 0.1),
              "bv": f16(rng.standard_normal(hkv * dh) * 0.1),
              "bo": f16(rng.standard_normal(d) * 0.1),
              "ln1_g": f16(rng.normal(1, 0.1, d)), "ln1_b": f16(rng.normal(0, 0.1, d)),
              "ln2_g": f16(rng.normal(1, 0.1, d)), "ln2_b": f16(rng.normal(0, 0.1, d)),
              "fc1": f16(rng.standard_normal((F, d)) * 0.25), "b1": f16(rng.normal(-0.2, 0.1, F)),
              "fc2T": f16(rng.standard_normal((F, d)) * 0.25),
              "b2": f16(rng.standard_normal(d) * 0.1)})
    x = f16(rng.standard_normal(d) * 1.5)
    K = f16(rng.standard_normal((hkv, n + 2, dh)))
    V = f16(rng.standard_normal((hkv, n + 2, dh)))
    return x, W, K, V


def _ulps_apart(a, b):
    """fp16 codes apart, for finite values of one sign."""
    ia = np.asarray(a, F16).view(np.int16).astype(int)
    ib = np.asarray(b, F16).view(np.int16).astype(int)
    return np.abs(ia - ib)


def test_layer_keep_all_equals_dense_layer():
    # keep = 1 (every unit and every neuron) is the dense layer: against the
    # oracle's masked-dense blocks (no index lists) and against numpy's matmul
    for seed in range(3):
        x, W, K, V = _rand_layer(np.random.default_rng(100 + seed))
        hkv, n = K.shape[0], K.shape[1] - 2
        F = W["fc1"].shape[0]
        y, hmid, a, m = oracle.layer(x, W, K, V, n, np.arange(hkv), np.arange(F))
        ad = oracle.attn_masked(x, W, K, V, n, None)
        assert _close(a.delta, ad.delta, rtol=1e-13, atol=1e-13)
        md = oracle.mlp_masked(hmid, W["fc1"], W["b1"], W["fc2T"], W["b2"], None,
                               ln_g=W["ln2_g"], ln_b=W["ln2_b"])
        assert _close(m, md, rtol=1e-13, atol=1e-13)
        yn, hn, mha, mlp = _np_dense_layer(x, W, K, V, n, 1.0 / math.sqrt(K.shape[2]), 1e-5)
        assert _close(a.delta, mha, rtol=1e-12, atol=1e-12)
        # h rounds the same way on both sides (no value of these draws sits on
        # a rounding boundary); y' may differ by one fp16 code at a boundary
        assert np.array_equal(hmid, hn)
        assert _close(m, mlp, rtol=1e-9, atol=1e-9 * np.abs(mlp).max())
        assert (_ulps_apart(y, yn) <= 1).all()


def test_layer_mlp_reads_the_attention_output():
    # the MLP block reads h = fp16(x + MHA), not x: equal to the MLP oracle on h
    x, W, K, V = _rand_layer(np.random.default_rng(7))
    hkv, n = K.shape[0], K.shape[1] - 2
    sel_u, sel_n = np.array([0], np.int32), np.arange(0, 64, 3).astype(np.int32)
    y, hmid, a, m = oracle.layer(x, W, K, V, n, sel_u, sel_n)
    expect_h = (x.astype(float) + a.delta).astype(F16)
    assert np.array_equal(hmid, expect_h)
    m_h = oracle.mlp_gather(expect_h, W["fc1"], W["b1"], W["fc2T"], W["b2"], sel_n,
                            ln_g=W["ln2_g"], ln_b=W["ln2_b"])
    m_x = oracle.mlp_gather(x, W["fc1"], W["b1"], W["fc2T"], W["b2"], sel_n,
                            ln_g=W["ln2_g"], ln_b=W["ln2_b"])
    assert _close(m, m_h, atol=TIGHT) and not _close(m, m_x, atol=1e-3)
    assert np.array_equal(y, (expect_h.astype(float) + m_h).astype(F16))


# --------------------------------------------------------------------------
# Attention over the retained KV positions (ByteCross §3.2, §4.1, App. A)
# --------------------------------------------------------------------------
def _rand_attn(rng, d=24, h=4, hkv=2, dh=8, n=40):
    W = _attn_weights(d, h, hkv, dh, rng, 0.3)
    for k_, n_ in (("bq", h * dh), ("bk", hkv * dh), ("bv", hkv * dh)):
        W[k_] = f16(rng.standard_normal(n_) * 0.1)
    W["bo"] = f16(rng.standard_normal(d) * 0.1)
    W["ln1_g"] = f16(rng.normal(1, 0.1, d))
    W["ln1_b"] = f16(rng.normal(0, 0.1, d))
    x = f16(rng.standard_normal(d))
    K = f16(rng.standard_normal((hkv, n + 3, dh)))
    V = f16(rng.standard_normal((hkv, n + 3, dh)))
    return x, W, K, V


def test_attn_kvsel_budget_covering_the_cache_is_dense():
    # b >= n: the selection keeps every position, and attention over the
    # retained positions is dense attention over the cache
    rng = np.random.default_rng(31)
    x, W, K, V = _rand_attn(rng)
    hkv, n, dh = K.shape[0], 40, K.shape[2]
    q_obs = f16(rng.standard_normal((4, 8, dh)))
    kept, _ = oracle.kv_select(q_obs, K, n, 1.0)
    for u in range(hkv):
        assert np.array_equal(kept[u], np.arange(n))
    ld = n + 5
    table = np.zeros((hkv, ld), np.int32)
    for u in range(hkv):
        table[u, :n] = kept[u]
    r = oracle.attn_kvsel(x, W, K, V, n, table, np.full(hkv, n, np.int32))
    dn = oracle.attn_masked(x, W, K, V, n, None)
    assert _close(r.H, dn.H, rtol=1e-13, atol=1e-13)
    assert _close(r.delta, dn.delta, rtol=1e-13, atol=1e-13)
    assert np.array_equal(r.knew, dn.knew) and np.array_equal(r.vnew, dn.vnew)


def test_attn_kvsel_subset_is_attention_over_those_rows():
    # per KV head u, its query heads attend over kept[u][:cnt[u]] plus the new
    # token: (1) the same as attending over a cache that holds only those rows,
    # (2) the same as the single-query routine given those positions. The
    # table is wider than the counts and the counts differ per head, so a
    # wrong row stride or count in the table lookup fails.
    rng = np.random.default_rng(32)
    x, W, K, V = _rand_attn(rng)
    hkv, n, dh = K.shape[0], 40, K.shape[2]
    h = W["Wq"].shape[0] // dh
    G = h // hkv
    scale = 1.0 / math.sqrt(dh)
    cnt = np.array([5, 11], np.int32)
    ld = 16
    table = np.zeros((hkv, ld), np.int32)          # padding: position 0 (valid, wrong)
    for u in range(hkv):
        table[u, :cnt[u]] = np.sort(rng.choice(np.arange(1, n), cnt[u], replace=False))
    r = oracle.attn_kvsel(x, W, K, V, n, table, cnt)
    z = _np_layernorm(x.astype(float))
    z = z * W["ln1_g"].astype(float) + W["ln1_b"].astype(float)
    q = (W["Wq"].astype(float) @ z + W["bq"].astype(float)).reshape(h, dh)
    for u in range(hkv):
        pos = table[u, :cnt[u]]
        Ks = np.zeros((hkv, cnt[u] + 1, dh), F16)
        Vs = np.zeros_like(Ks)
        Ks[u, :cnt[u]], Vs[u, :cnt[u]] = K[u, pos], V[u, pos]
        g = oracle.attn_gather(x, W, Ks, Vs, int(cnt[u]), [u])
        for j in range(u * G, (u + 1) * G):
            assert _close(r.H[j], g.H[j], rtol=1e-13, atol=1e-13)
            Hj = oracle.attend(q[j], K[u], V[u], r.knew[u].astype(float),
                               r.vnew[u].astype(float), scale, pos=pos)
            assert _close(r.H[j], Hj, rtol=1e-12, atol=1e-12)
    # the output projection sums every head's output: delta - b_o = H WoT
    assert _close(r.delta, r.H.reshape(-1) @ W["WoT"].astype(float) + W["bo"].astype(float),
                  rtol=1e-12, atol=1e-12)
