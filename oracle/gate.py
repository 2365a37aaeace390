"""Latency gate of the decode step: mode bytes, the crossing model, dispatch
(test infrastructure; pure Python, fp64).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources:
* "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding":
  §3.1 (a step reads the projection weights once plus a context-dependent KV
  term), §3.2 (projection keep saves context-independent bytes, KV keep saves
  bytes that grow with n; the branches can switch between steps), §3.3 (a
  latency gate adds fixed kernel costs; a fixed KV token budget b means
  r_KV = b / n; a batch reads the union of the activated channels), §5.4 and
  App. I (per-request dispatch; requests that use selection pay for the
  scoring pass), App. D (crossing model: each branch's time = its byte-scaled
  dense time + its measured kernel cost; dense time interpolated log-log,
  kernel costs linearly, across the sweep contexts; solve for equal latency),
  App. E (a measured crossing interpolates the time difference between the
  last context one branch leads and the first the other leads).
* "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time":
  §2.3 Eq. 1-2 (the rows a sparse layer reads), §4.1 (the low-rank predictor
  P1 [r][d], P2 [rows][r]), App. C.1 (a batch computes over the union).

Modes (one decoder layer, one step of B sequences with n cached tokens each):
  DENSE     every weight row, the full cache;
  ACT       the projection branch: the selected neurons / attention units
            (the B-sequence union) plus the predictor, the full cache;
  KV        every weight row, the retained KV (r_KV n tokens per unit);
  COMPOSED  both.
The new token's K, V row is read in every mode (n + 1, or r_KV n + 1, keys).
"""
from __future__ import annotations

import math

import numpy as np

from .byte_account import ELT

DENSE, ACT, KV, COMPOSED = 0, 1, 2, 3
MODES = ("dense", "act", "kv", "composed")


def expected_union(N: int, k: int, B: int) -> float:
    """E|S_1 u ... u S_B| for B independent uniform k-subsets of N items: an
    item is missed by one subset with probability 1 - k/N."""
    return N * (1.0 - (1.0 - k / N) ** B)


def keep_count(keep: float, N: int) -> int:
    """Deja Vu §2.3: k = max(1, floor(keep N)); keep 1 keeps all."""
    return N if keep >= 1.0 else max(1, int(math.floor(keep * N + 1e-9)))


def mode_bytes(mode, d, h, h_kv, dh, F, r, n, keep_N, keep_H, keep_KV, B=1,
               union_N=0, union_H=0, kv_budget=0):
    """Bytes one layer's step reads in `mode` (fp16 everywhere).

    n is real-valued here: r_KV n retained tokens are not floored, so that the
    crossing is a continuous function of n (the closed-form crossover of §3.3
    is real too). union_N / union_H (B > 1): the union sizes; 0 = the
    independent-draw expectation."""
    G = h // h_kv
    sparse = mode in (ACT, COMPOSED)
    retained = mode in (KV, COMPOSED)
    if sparse:
        kN, kH = keep_count(keep_N, F), keep_count(keep_H, h_kv)
        uN = kN if B == 1 else (union_N or expected_union(F, kN, B))
        uH = kH if B == 1 else (union_H or expected_union(h_kv, kH, B))
        rows = (F if keep_N < 1 else 0) + (h_kv if keep_H < 1 else 0)
        pred = 0 if rows == 0 else ELT * r * (d + rows)
    else:
        uN, uH, pred = F, h_kv, 0
    if retained:
        tokens = min(float(n), kv_budget) if kv_budget > 0 else keep_KV * n
    else:
        tokens = float(n)
    weights = uH * (2 * G * dh + 2 * dh) * d * ELT + uN * 2 * d * ELT
    kv = B * uH * 2 * dh * (tokens + 1) * ELT
    return weights + kv + pred


# --------------------------------------------------------------------------
# interpolation over the sweep contexts (App. D)
# --------------------------------------------------------------------------
def loglog(x, xs, ys):
    """Piecewise-linear in (log x, log y) through the knots; the end segments
    extend past the first and last knot."""
    lx, lxs, lys = math.log(x), [math.log(v) for v in xs], [math.log(v) for v in ys]
    i = 0
    while i < len(xs) - 2 and lx > lxs[i + 1]:
        i += 1
    t = (lx - lxs[i]) / (lxs[i + 1] - lxs[i])
    return math.exp(lys[i] + t * (lys[i + 1] - lys[i]))


def linear(x, xs, ys):
    """Piecewise-linear through the knots, held at the end values outside."""
    return float(np.interp(x, xs, ys))


# --------------------------------------------------------------------------
# cost model and latency
# --------------------------------------------------------------------------
def calibrate(ctx, measured_us, bytes_at):
    """Kernel cost of each mode at each sweep context: measured time minus the
    dense time scaled by the mode's byte fraction (App. D). measured_us[m][i]
    is mode m's layer time at ctx[i]; bytes_at(m, n) its bytes."""
    cost = [[0.0] * len(ctx) for _ in MODES]
    for m in range(len(MODES)):
        for i, c in enumerate(ctx):
            cost[m][i] = measured_us[m][i] - measured_us[DENSE][i] * bytes_at(m, c) / bytes_at(DENSE, c)
    return cost


def latency(mode, n, ctx, dense_us, cost_us, select_us, bytes_at, steps):
    """Per-layer time of one step in `mode` at context n: byte-scaled dense
    time + the mode's kernel cost, plus (modes that select KV) the scoring
    pass spread over the request's `steps` decode steps."""
    t = loglog(n, ctx, dense_us) * bytes_at(mode, n) / bytes_at(DENSE, n)
    t += linear(n, ctx, cost_us[mode])
    if mode in (KV, COMPOSED):
        t += linear(n, ctx, select_us) / steps
    return t


def choose(n, ctx, dense_us, cost_us, select_us, bytes_at, steps, admitted=(0, 1, 2, 3)):
    """The admitted mode with the lowest predicted time (ties: lower mode)."""
    ts = [latency(m, n, ctx, dense_us, cost_us, select_us, bytes_at, steps)
          for m in range(len(MODES))]
    best = min(admitted, key=lambda m: (ts[m], m))
    return best, ts


def crossing(a, b, lo, hi, ctx, dense_us, cost_us, select_us, bytes_at, steps, grid=20000):
    """The first context in [lo, hi] where modes a and b take equal predicted
    time (App. D), or None: a sign change of T_a - T_b is bracketed on a fine
    log-spaced grid, then bisected."""
    def f(x):
        return (latency(a, x, ctx, dense_us, cost_us, select_us, bytes_at, steps)
                - latency(b, x, ctx, dense_us, cost_us, select_us, bytes_at, steps))

    xs = np.exp(np.linspace(math.log(lo), math.log(hi), grid))
    prev_x, prev_f = xs[0], f(xs[0])
    if prev_f == 0.0:
        return float(prev_x)
    for x in xs[1:]:
        fx = f(x)
        if fx == 0.0:
            return float(x)
        if (fx < 0) != (prev_f < 0):
            l, h, fl = prev_x, x, prev_f
            for _ in range(200):
                mid = 0.5 * (l + h)
                fm = f(mid)
                if (fm < 0) == (fl < 0):
                    l, fl = mid, fm
                else:
                    h = mid
            return 0.5 * (l + h)
        prev_x, prev_f = x, fx
    return None


def measured_crossing(ctx, t_a, t_b):
    """App. E: between the last context where a leads (t_a < t_b) and the
    first after it where b leads, interpolate t_a - t_b linearly to zero."""
    diff = [x - y for x, y in zip(t_a, t_b)]
    for i in range(len(ctx) - 1):
        if diff[i] < 0 <= diff[i + 1] or diff[i] > 0 >= diff[i + 1]:
            t = diff[i] / (diff[i] - diff[i + 1])
            return ctx[i] + t * (ctx[i + 1] - ctx[i])
    return None
