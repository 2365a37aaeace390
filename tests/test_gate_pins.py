"""The oracle's latency gate pinned to closed forms and brute force.

"Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding" §3.3
and App. D: with no kernel costs the latency crossing is the byte crossover
n* = (1 - r_P) W / ((1 - r_KV) b), whatever the dense times are; a fixed token
budget puts r_KV = b/n into it; a constant cost difference moves the crossing
by cost x bandwidth / ((1 - r_KV) b); a batch reads the union of its sets.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import byte_account as ba
from oracle import gate as g

# Llama-3.1-8B attention dimensions with a two-matrix MLP of width 14336
DIMS = dict(d=4096, h=32, h_kv=8, dh=128, F=14336)
CTX = [1024.0, 4096.0, 16384.0, 65536.0, 262144.0]


def _bytes(r=0, keep_N=0.5, keep_H=1.0, keep_KV=0.3, B=1, **kw):
    def at(m, n):
        return g.mode_bytes(m, DIMS["d"], DIMS["h"], DIMS["h_kv"], DIMS["dh"], DIMS["F"], r, n,
                            keep_N, keep_H, keep_KV, B=B, **kw)
    return at


def _zero(ctx=CTX):
    return [[0.0] * len(ctx) for _ in g.MODES], [0.0] * len(ctx)


KV_TOK = 2 * DIMS["h_kv"] * DIMS["dh"] * 2          # K and V bytes per token per layer
W_FF = 2 * DIMS["F"] * DIMS["d"] * 2
W_ATTN = (2 * DIMS["h"] + 2 * DIMS["h_kv"]) * DIMS["dh"] * DIMS["d"] * 2


@pytest.mark.parametrize("N,k,B", [(6, 2, 3), (5, 3, 2), (7, 1, 4), (4, 4, 2)])
def test_expected_union_brute_force(N, k, B):
    subsets = list(itertools.combinations(range(N), k))
    total = sum(len(set().union(*pick)) for pick in itertools.product(subsets, repeat=B))
    assert math.isclose(total / len(subsets) ** B, g.expected_union(N, k, B), rel_tol=1e-12)


def test_mode_bytes_match_the_byte_account():
    n = 5000
    d, h, hk, dh, F = (DIMS[x] for x in ("d", "h", "h_kv", "dh", "F"))
    at = _bytes(r=1000, keep_N=0.25, keep_H=0.5, keep_KV=0.125)
    assert at(g.DENSE, n) == ba.dense_bytes(d, h, hk, dh, F, n)
    kN, kH = int(0.25 * F), 4
    assert at(g.ACT, n) == (ba.selected_bytes(d, h, hk, dh, F, n, kN, kH)
                            + ba.predictor_bytes(d, 1000, F + hk))
    # KV only: every weight, r_KV n + 1 keys
    assert at(g.KV, n) == W_ATTN + W_FF + hk * 2 * dh * (0.125 * n + 1) * 2
    # dense OPT-175B layer = the Deja Vu Table 2 I/O (4 d^2 + 8 d^2 parameters)
    att, mlp = ba.table2_io_gib(12288)
    dense = g.mode_bytes(g.DENSE, 12288, 96, 96, 128, 49152, 0, 0, 1, 1, 1)
    assert dense - 96 * 2 * 128 * 2 == (att + mlp) * 2**30


@pytest.mark.parametrize("keep_N,keep_KV", [(0.5, 0.3), (0.7, 0.3), (0.5, 0.5), (0.25, 0.125)])
def test_zero_cost_crossing_is_the_byte_crossover(keep_N, keep_KV):
    at = _bytes(keep_N=keep_N, keep_KV=keep_KV)
    cost, sel = _zero()
    rng = np.random.default_rng(1)
    dense = list(np.sort(rng.uniform(50, 400, len(CTX))))   # any positive dense times
    n = g.crossing(g.ACT, g.KV, 16.0, 4e6, CTX, dense, cost, sel, at, steps=1)
    r_P = math.floor(keep_N * DIMS["F"]) / DIMS["F"]        # k = floor(keep F) neurons
    star = ba.crossover(W_FF, KV_TOK, r_P, keep_KV)
    assert math.isclose(n, star, rel_tol=1e-9), (n, star)


def test_zero_cost_crossing_with_head_sparsity():
    # Deja Vu Eq. 2: a head-sparse projection branch also skips the K, V rows
    # of the units it drops, so the KV branch only gains r_H - r_KV of the
    # cache per token: r_P W + r_H b (n + 1) = W + b (r_KV n + 1).
    at = _bytes(keep_N=0.5, keep_H=0.5, keep_KV=0.3)
    cost, sel = _zero()
    n = g.crossing(g.ACT, g.KV, 16.0, 4e6, CTX, [100.0] * len(CTX), cost, sel, at, steps=1)
    W = W_FF + W_ATTN
    assert math.isclose(n, (0.5 * W + 0.5 * KV_TOK) / (0.2 * KV_TOK), rel_tol=1e-9)
    assert at(g.ACT, 2 * n) > at(g.KV, 2 * n) and at(g.ACT, n / 2) < at(g.KV, n / 2)


def test_zero_cost_crossing_of_the_golden_keep_pair():
    # §3.3 table: at r_P 0.5 and r_KV 0.3 the feed-forward crossover of a
    # Llama-3.1-8B layer is 61440 tokens; its FFN has three d x 14336 matrices,
    # so a two-matrix MLP of width 1.5 x 14336 holds the same bytes.
    at = lambda m, n: g.mode_bytes(m, 4096, 32, 8, 128, 21504, 0, n, 0.5, 1.0, 0.3)
    cost, sel = _zero()
    n = g.crossing(g.ACT, g.KV, 16.0, 4e6, CTX, [100.0] * len(CTX), cost, sel, at, steps=1)
    assert round(n) == 61440


def test_fixed_token_budget_substitutes_b_over_n():
    b = 2048
    at = _bytes(kv_budget=b)
    cost, sel = _zero()
    n = g.crossing(g.ACT, g.KV, 16.0, 4e6, CTX, [100.0] * len(CTX), cost, sel, at, steps=1)
    # (1 - r_P) W = (1 - b/n) b_tok n  <=>  n = b + (1 - r_P) W / b_tok
    assert math.isclose(n, b + 0.5 * W_FF / KV_TOK, rel_tol=1e-9)
    assert math.isclose(n, ba.crossover(0.5 * W_FF / (1 - b / n) * (1 - b / n) / 0.5, KV_TOK,
                                        0.5, b / n), rel_tol=1e-9)


def test_cost_difference_moves_the_crossing_by_cost_times_bandwidth():
    # dense time = dense bytes / BW at every knot; the act branch pays dc more
    BW = 1.6e12                                    # bytes / s
    at = _bytes()
    star = ba.crossover(W_FF, KV_TOK, 0.5, 0.3)
    knots = [4096.0, 8192.0, 12288.0, 16384.0, 20480.0, 24576.0, 32768.0, 65536.0]
    target = 16384.0
    dc = (star - target) * 0.7 * KV_TOK / BW * 1e6  # µs per layer
    dense = [at(g.DENSE, c) / BW * 1e6 for c in knots]
    cost = [[0.0] * len(knots) for _ in g.MODES]
    cost[g.ACT] = [dc] * len(knots)
    n = g.crossing(g.ACT, g.KV, 1024.0, 1e6, knots, dense, cost, [0.0] * len(knots), at, 1)
    assert math.isclose(n, target, rel_tol=1e-9)
    # §6: on A100 a 1 ms cost difference moves the crossing by about 17K
    # tokens. Per token per step the KV branch saves (1 - 0.3) x 4096 bytes in
    # each of Llama-3.1-8B's 32 layers; at the public 2.039 TB/s of an
    # A100-SXM4-80GB run at 70-85 % of it, 1 ms is 15.6K-18.9K tokens.
    per_ms = [f * 2.039e12 * 1e-3 / (0.7 * KV_TOK * 32) for f in (0.70, 0.85)]
    assert per_ms[0] < 17000 < per_ms[1]


def test_selection_pass_is_spread_over_the_request():
    at = _bytes(keep_N=1.0, keep_KV=0.125)
    cost, _ = _zero()
    dense = [100.0 * (c / CTX[0]) ** 0.3 for c in CTX]
    sel = [c / 1000.0 for c in CTX]
    t1 = g.latency(g.KV, 8192, CTX, dense, cost, sel, at, steps=1)
    t64 = g.latency(g.KV, 8192, CTX, dense, cost, sel, at, steps=64)
    assert math.isclose(t1 - t64, g.linear(8192, CTX, sel) * (1 - 1 / 64), rel_tol=1e-12)
    # with the scoring pass free, KV-only never loses to dense; charged once
    # per decode step it loses below some context
    assert g.crossing(g.DENSE, g.KV, 16.0, 1e6, CTX, dense, cost, _zero()[1], at, 1) is None
    n = g.crossing(g.DENSE, g.KV, 16.0, 1e6, CTX, dense, cost, [10.0] * len(CTX), at, 1)
    assert n is not None and n > 16.0


def test_batch_union_lowers_the_per_step_crossover():
    B = 4
    at = _bytes(B=B)
    cost, sel = _zero()
    n = g.crossing(g.ACT, g.KV, 1.0, 4e6, CTX, [100.0] * len(CTX), cost, sel, at, steps=1)
    kN = int(0.5 * DIMS["F"])
    r_eff = g.expected_union(DIMS["F"], kN, B) / DIMS["F"]
    assert math.isclose(r_eff, 1 - 0.5**4)
    # (1 - r_eff) W = B (1 - r_KV) b n
    assert math.isclose(n, (1 - r_eff) * W_FF / (B * 0.7 * KV_TOK), rel_tol=1e-9)
    assert n < ba.crossover(W_FF, KV_TOK, 0.5, 0.3)
    # a measured union replaces the expectation
    at2 = _bytes(B=B, union_N=kN + 100)
    n2 = g.crossing(g.ACT, g.KV, 1.0, 4e6, CTX, [100.0] * len(CTX), cost, sel, at2, steps=1)
    assert math.isclose(n2, (DIMS["F"] - kN - 100) * 2 * DIMS["d"] * 2 / (B * 0.7 * KV_TOK),
                        rel_tol=1e-9)


def test_loglog_reproduces_a_power_law_and_linear_clamps():
    xs = [100.0, 1000.0, 5000.0, 80000.0]
    ys = [3.0 * x**0.7 for x in xs]
    for x in (50.0, 100.0, 333.0, 4000.0, 80000.0, 2e5):
        assert math.isclose(g.loglog(x, xs, ys), 3.0 * x**0.7, rel_tol=1e-12)
    ys2 = [1.0, 3.0, 2.0, 7.0]
    assert g.linear(50.0, xs, ys2) == 1.0 and g.linear(1e6, xs, ys2) == 7.0
    assert math.isclose(g.linear(550.0, xs, ys2), 2.0)


def test_calibration_recovers_planted_costs():
    at = _bytes(r=1000, keep_N=0.25, keep_KV=0.125)
    dense = [60.0, 70.0, 95.0, 190.0, 600.0]
    planted = [[0.0] * 5, [30.0, 31.0, 29.5, 33.0, 40.0], [2.0, 2.5, 3.0, 4.0, 9.0],
               [32.0, 33.0, 34.0, 36.0, 50.0]]
    measured = [[dense[i] * at(m, c) / at(g.DENSE, c) + planted[m][i] for i, c in enumerate(CTX)]
                for m in range(4)]
    got = g.calibrate(CTX, measured, at)
    assert np.allclose(got, planted, rtol=0, atol=1e-9)
    # and the calibrated model reproduces the sweep times at the sweep contexts
    for m in range(4):
        for i, c in enumerate(CTX):
            assert math.isclose(g.latency(m, c, CTX, dense, got, [0.0] * 5, at, 1),
                                measured[m][i], rel_tol=1e-12)


def test_choose_respects_admission_and_ties():
    at = _bytes(keep_N=0.5, keep_KV=0.3)
    cost, sel = _zero()
    dense = [100.0] * len(CTX)
    m, ts = g.choose(200000.0, CTX, dense, cost, sel, at, 1)
    assert m == g.COMPOSED and ts[g.COMPOSED] == min(ts)
    m, _ = g.choose(200000.0, CTX, dense, cost, sel, at, 1, admitted=(g.DENSE, g.ACT))
    assert m == g.ACT
    same = lambda mm, n: 1.0
    m, _ = g.choose(5000.0, CTX, dense, cost, sel, same, 1)
    assert m == g.DENSE


def test_measured_crossing_interpolates_between_the_bracketing_contexts():
    ctx = [2048, 4096, 8192, 16384]
    ta = [10.0, 12.0, 16.0, 24.0]
    tb = [13.0, 13.5, 14.0, 14.5]      # a leads at 4096, b from 8192 on
    n = g.measured_crossing(ctx, ta, tb)
    assert math.isclose(n, 4096 + (-1.5 / (-1.5 - 2.0)) * 4096)
    assert g.measured_crossing(ctx, ta, [100.0] * 4) is None
