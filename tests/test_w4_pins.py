"""Pins of the oracle's W4A16 format and MLP ("Deja Vu" §5.2, Table 7: 4-bit
weights, 16-bit activations; the format is this project's own: groups of 128
columns, fp16 scale max|w|/7, codes rint(w/s) in [-8, 7])."""
import numpy as np
import pytest

import oracle
from oracle import w4

F16 = np.float16


def _row(vals, d=128):
    r = np.zeros(d, np.float64)
    r[: len(vals)] = vals
    return r.astype(F16)[None, :]


def test_worked_group_with_unit_scale():
    # max |w| = 7 -> s = 1; -3.5 and 0.5 and 2.5 are ties: to even
    q, s = w4.quantize(_row([7.0, -3.5, 1.75, 0.5, -7.0, 2.5, -1.25, 6.5]))
    assert s.tolist() == [[1.0]]
    assert q[0, :8].tolist() == [7, -4, 2, 0, -7, 2, -1, 6]
    assert not q[0, 8:].any()


def test_worked_group_with_scale_two():
    # max |w| = 14 -> s = 2: 3 -> 1.5 -> 2, 5 -> 2.5 -> 2, -1 -> -0.5 -> 0, -14 -> -7
    q, s = w4.quantize(_row([14.0, 3.0, 5.0, -1.0, -14.0, 9.0]))
    assert s.tolist() == [[2.0]]
    assert q[0, :6].tolist() == [7, 2, 2, 0, -7, 4]


def test_scale_is_rounded_to_fp16():
    # max |w| = 1 -> 1/7 in fp32, then to fp16; the codes divide by that value
    q, s = w4.quantize(_row([1.0, 0.5, -0.25]))
    assert s[0, 0] == F16(np.float32(1.0) / np.float32(7.0))
    sf = np.float32(s[0, 0])
    assert q[0, :3].tolist() == [int(np.rint(np.float32(v) / sf)) for v in (1.0, 0.5, -0.25)]


def test_zero_group_and_error_bound_by_brute_force():
    rng = np.random.default_rng(0)
    W = (rng.standard_normal((6, 512)) * rng.uniform(0.01, 5, (6, 1))).astype(F16)
    W[2, 128:256] = 0
    q, s = w4.quantize(W)
    assert s[2, 1] == 0 and not q[2, 128:256].any()
    codes = np.arange(-8, 8)
    for r in range(6):
        for g in range(4):
            sf = np.float32(s[r, g])
            if sf == 0:
                continue
            x = W[r, g * 128:(g + 1) * 128].astype(np.float32) / sf
            # nearest code by search over all 16 codes, ties to the even one
            dist = np.abs(x[:, None] - codes[None, :].astype(np.float32))
            best = dist.min(axis=1, keepdims=True)
            cand = np.where(dist == best, codes[None, :], 99)
            even = np.where(cand % 2 == 0, cand, 99).min(axis=1)
            want = np.where((cand != 99).sum(axis=1) > 1, even, cand.min(axis=1))
            assert np.array_equal(q[r, g * 128:(g + 1) * 128], want)
            assert np.abs(q[r, g * 128:(g + 1) * 128]).max() == 7
    err = np.abs(w4.dequantize(q, s) - W.astype(np.float64))
    assert np.all(err <= np.repeat(s.astype(np.float64), 128, axis=1) / 2 * (1 + 1e-3) + 1e-12)


def test_pack_layout_and_round_trip():
    q = np.zeros((1, 256), np.int8)
    q[0, 0], q[0, 1], q[0, 2], q[0, 3] = -8, 7, 3, -1
    s = np.array([[0.5, 2.0]], F16)
    p = w4.pack(q, s)
    assert p.shape == (1, 144)                      # 128 + 4 bytes, padded to 16
    assert p[0, 0] == 0xF0 and p[0, 1] == (11 | (7 << 4))
    assert p[0, 128:132].view(F16).tolist() == [0.5, 2.0] and not p[0, 132:].any()
    rng = np.random.default_rng(1)
    q = rng.integers(-8, 8, (3, 384)).astype(np.int8)
    s = rng.uniform(0.001, 3, (3, 3)).astype(F16)
    q2, s2 = w4.unpack(w4.pack(q, s), 384)
    assert np.array_equal(q, q2) and np.array_equal(s, s2)


def test_mlp_equals_the_fp16_mlp_when_the_weights_are_exact():
    # scales that are powers of two make every dequantized weight an exact fp16
    # value: the W4 MLP must then equal the oracle's fp16 gather MLP
    rng = np.random.default_rng(2)
    F, d = 40, 256
    q1 = rng.integers(-8, 8, (F, d)).astype(np.int8)
    q2 = rng.integers(-8, 8, (F, d)).astype(np.int8)
    s1 = (2.0 ** rng.integers(-7, -3, (F, d // 128))).astype(F16)
    s2 = (2.0 ** rng.integers(-7, -3, (F, d // 128))).astype(F16)
    W1, W2 = w4.dequantize(q1, s1).astype(F16), w4.dequantize(q2, s2).astype(F16)
    assert np.array_equal(W1.astype(np.float64), w4.dequantize(q1, s1))
    b1 = (rng.standard_normal(F) * 0.1).astype(F16)
    b2 = (rng.standard_normal(d) * 0.1).astype(F16)
    g = (1 + 0.1 * rng.standard_normal(d)).astype(F16)
    bb = (0.1 * rng.standard_normal(d)).astype(F16)
    x = rng.standard_normal(d).astype(F16)
    idx = np.sort(rng.choice(F, 13, replace=False))
    got = w4.mlp(x, q1, s1, b1, q2, s2, b2, idx, g, bb)
    want = oracle.mlp_gather(x, W1, b1, W2, b2, idx, ln_g=g, ln_b=bb)
    assert np.allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())


def test_rejects_ragged_groups():
    with pytest.raises(AssertionError):
        w4.quantize(np.zeros((1, 100), F16))


def _exact_w4(rng, rows, d):
    """Codes with power-of-two scales: every dequantized weight is an exact fp16."""
    q = rng.integers(-8, 8, (rows, d)).astype(np.int8)
    s = (2.0 ** rng.integers(-7, -4, (rows, d // 128))).astype(F16)
    return q, s


def test_attn_and_layer_equal_the_fp16_oracle_when_the_weights_are_exact():
    rng = np.random.default_rng(9)
    d, h, hkv, dh, F, n = 256, 4, 2, 64, 48, 37
    Wq4 = {k: _exact_w4(rng, r, d) for k, r in (("Wq", h * dh), ("Wk", hkv * dh),
                                                 ("Wv", hkv * dh), ("WoT", h * dh),
                                                 ("fc1", F), ("fc2T", F))}
    W16 = {k: w4.dequantize(*v).astype(F16) for k, v in Wq4.items()}
    for k in W16:
        assert np.array_equal(W16[k].astype(np.float64), w4.dequantize(*Wq4[k]))
    extra = {"bq": (rng.standard_normal(h * dh) * 0.1).astype(F16),
             "bk": (rng.standard_normal(hkv * dh) * 0.1).astype(F16),
             "bv": (rng.standard_normal(hkv * dh) * 0.1).astype(F16),
             "bo": (rng.standard_normal(d) * 0.1).astype(F16),
             "b1": (rng.standard_normal(F) * 0.1).astype(F16),
             "b2": (rng.standard_normal(d) * 0.1).astype(F16),
             "ln1_g": (1 + 0.1 * rng.standard_normal(d)).astype(F16),
             "ln1_b": (0.1 * rng.standard_normal(d)).astype(F16),
             "ln2_g": (1 + 0.1 * rng.standard_normal(d)).astype(F16),
             "ln2_b": (0.1 * rng.standard_normal(d)).astype(F16)}
    K = rng.standard_normal((hkv, n + 3, dh)).astype(F16)
    V = rng.standard_normal((hkv, n + 3, dh)).astype(F16)
    x = rng.standard_normal(d).astype(F16)
    sel, nsel = [1], np.sort(rng.choice(F, 20, replace=False))
    delta, knew, vnew = w4.attn(x, {**Wq4, **extra}, K, V, n, sel)
    ref = oracle.attn_gather(x, {**W16, **extra}, K, V, n, sel)
    assert np.allclose(delta, ref.delta, rtol=0, atol=1e-10 * np.abs(ref.delta).max())
    assert np.array_equal(knew[1], ref.knew[1]) and np.array_equal(vnew[1], ref.vnew[1])
    y, hmid = w4.layer(x, {**Wq4, **extra}, K, V, n, sel, nsel)
    y_ref, hmid_ref, _, _ = oracle.layer(x, {**W16, **extra}, K, V, n, sel, nsel)
    assert np.array_equal(hmid, hmid_ref) and np.array_equal(y, y_ref)
