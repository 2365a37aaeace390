"""The library's latency gate (host-only C entry points, no GPU) against the
oracle's crossing model ("Where Activation Sparsity and KV-Cache Sparsity
Cross in LLM Decoding" §3.3, App. D) and against the closed-form crossover."""
import math

import numpy as np
import pytest

from contextual_sparsity_gb300 import build, dv
from oracle import byte_account as ba
from oracle import gate as g


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    dv.lib()


def f32(x):
    return float(np.float32(x))


def _case(rng):
    G = int(rng.choice([1, 2, 4, 8]))
    h_kv = int(rng.choice([1, 4, 8, 12, 96]))
    d = int(rng.choice([512, 4096, 12288]))
    dims = dict(d=d, h=h_kv * G, h_kv=h_kv, d_h=int(rng.choice([64, 128])),
                F=int(rng.integers(1, 60000)), r=int(rng.choice([0, 8, 1000, 1024])))
    keep = [f32(rng.choice([1.0, rng.uniform(0.01, 1.0)])) for _ in range(3)]
    B = int(rng.choice([1, 1, 2, 4]))
    req = dict(B=B, steps=int(rng.integers(1, 500)),
               union_N=int(rng.choice([0, rng.integers(1, dims["F"] + 1)])) if B > 1 else 0,
               union_H=int(rng.choice([0, rng.integers(1, h_kv + 1)])) if B > 1 else 0,
               kv_budget=int(rng.choice([0, 0, rng.integers(1, 100000)])))
    return dims, keep, req


def _lib_args(dims, keep, req):
    D = dv.dims(dims["d"], dims["h"], dims["h_kv"], dims["d_h"], dims["F"], dims["r"], 1)
    return D, dv.Keep(*keep), dv.request(**req)


def _oracle_bytes(dims, keep, req):
    def at(m, n):
        return g.mode_bytes(m, dims["d"], dims["h"], dims["h_kv"], dims["d_h"], dims["F"],
                            dims["r"], n, keep[0], keep[1], keep[2], B=req["B"],
                            union_N=req["union_N"], union_H=req["union_H"],
                            kv_budget=req["kv_budget"])
    return at


def _model(rng, nc=None):
    nc = nc or int(rng.integers(2, 17))
    ctx = np.sort(rng.choice(np.arange(256, 300000), nc, replace=False)).astype(float)
    dense = np.sort(rng.uniform(20, 900, nc))
    cost = [[0.0] * nc] + [list(rng.uniform(-5, 60, nc)) for _ in range(3)]
    sel = list(rng.uniform(0, 3000, nc))
    return list(ctx), list(dense), cost, sel


@pytest.mark.parametrize("seed", range(40))
def test_bytes_and_times_match_the_oracle(seed):
    rng = np.random.default_rng(seed)
    dims, keep, req = _case(rng)
    D, K, R = _lib_args(dims, keep, req)
    at = _oracle_bytes(dims, keep, req)
    ctx, dense, cost, sel = _model(rng)
    cm = dv.cost_model(ctx, dense, cost, sel)
    for n in list(rng.uniform(1, 400000, 6)) + [ctx[0], ctx[-1], 0.5 * ctx[0], 2 * ctx[-1]]:
        got = dv.plan_bytes(D, K, R, n)
        want = [at(m, n) for m in range(4)]
        assert np.allclose(got, want, rtol=1e-14, atol=0), (n, got, want)
        p = dv.plan_decode(D, K, R, cm, n)
        admitted = (0, 1, 2, 3) if req["B"] == 1 else (0, 1)
        m, ts = g.choose(n, ctx, dense, cost, sel, at, req["steps"], admitted)
        assert np.allclose(p["us"], ts, rtol=1e-12, atol=1e-9), (n, p["us"], ts)
        if sorted(ts)[0] != sorted(ts)[1]:
            assert p["choice"] == m


@pytest.mark.parametrize("seed", range(12))
def test_calibration_matches_the_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    dims, keep, req = _case(rng)
    D, K, R = _lib_args(dims, keep, req)
    at = _oracle_bytes(dims, keep, req)
    ctx = [2048.0, 8192.0, 32768.0, 131072.0]
    measured = [list(rng.uniform(40, 300, 4)) for _ in range(4)]
    sel = list(rng.uniform(0, 100, 4))
    cm = dv.cost_calibrate(D, K, R, ctx, measured, sel)
    want = g.calibrate(ctx, measured, at)
    for m in range(4):
        assert np.allclose(list(cm.cost_us[m])[:4], want[m], rtol=1e-12, atol=1e-9)
    assert list(cm.dense_us)[:4] == measured[0] and list(cm.select_us)[:4] == sel
    # the calibrated model gives back the measured times at the sweep contexts
    for i, c in enumerate(ctx):
        p = dv.plan_decode(D, K, dv.request(**dict(req, steps=10**9)), cm, c)
        assert np.allclose(p["us"], [measured[m][i] for m in range(4)], rtol=1e-6)


@pytest.mark.parametrize("seed", range(16))
def test_crossing_matches_the_oracle(seed):
    rng = np.random.default_rng(200 + seed)
    dims = dict(d=4096, h=32, h_kv=8, d_h=128, F=int(rng.integers(8000, 30000)), r=1000)
    keep = [f32(rng.uniform(0.05, 0.9)), 1.0, f32(rng.uniform(0.05, 0.6))]
    req = dict(B=1, steps=int(rng.integers(1, 300)), union_N=0, union_H=0, kv_budget=0)
    D, K, R = _lib_args(dims, keep, req)
    at = _oracle_bytes(dims, keep, req)
    nc = 5
    ctx = [1024.0, 4096.0, 16384.0, 65536.0, 262144.0]
    dense = list(np.sort(rng.uniform(40, 80, nc)) * np.array([1, 1.1, 1.5, 2.5, 6]))
    base = rng.uniform(0, 40)
    cost = [[0.0] * nc, list(base + rng.uniform(0, 4, nc)), list(rng.uniform(0, 4, nc)),
            list(base + rng.uniform(0, 4, nc))]
    sel = list(rng.uniform(0, 200, nc))
    cm = dv.cost_model(ctx, dense, cost, sel)
    for a, b in ((g.ACT, g.KV), (g.DENSE, g.KV), (g.DENSE, g.ACT), (g.ACT, g.COMPOSED)):
        want = g.crossing(a, b, 64.0, 1e6, ctx, dense, cost, sel, at, req["steps"])
        got = dv.plan_crossing(D, K, R, cm, a, b, 64.0, 1e6)
        if want is None:
            assert got is None, (a, b, got)
        else:
            assert got is not None and math.isclose(got, want, rel_tol=1e-9), (a, b, got, want)


def test_zero_cost_crossing_is_the_byte_crossover():
    # Llama-3.1-8B attention dimensions, two-matrix MLP of width 14336, no predictor
    D = dv.dims(4096, 32, 8, 128, 14336, 0, 1)
    cm = dv.cost_model([1e3, 1e4, 1e5], [90.0, 120.0, 500.0], [[0.0] * 3] * 4)
    for kn, kkv in ((0.5, 0.3), (0.25, 0.125), (0.7, 0.5)):
        n = dv.plan_crossing(D, dv.Keep(kn, 1.0, kkv), dv.request(), cm, 1, 2, 16.0, 1e7)
        r_P = math.floor(f32(kn) * 14336 + 1e-9) / 14336
        star = ba.crossover(2 * 14336 * 4096 * 2, 4096, r_P, f32(kkv))
        assert math.isclose(n, star, rel_tol=1e-9), (kn, kkv, n, star)


def test_dispatch_prefers_kv_at_long_context_and_respects_admission():
    D = dv.dims(4096, 32, 8, 128, 14336, 1000, 1)
    keep = dv.Keep(0.5, 1.0, 0.125)
    cm = dv.cost_model([2048, 131072], [50.0, 200.0], [[0, 0], [5, 5], [3, 5], [8, 10]],
                       [100.0, 4000.0])
    p = dv.plan_decode(D, keep, dv.request(steps=1000), cm, 131072)
    assert p["choice"] == dv.MODE_COMPOSED
    # an expensive projection branch (a 28 µs kernel cost against an 18 µs
    # byte saving at 128K) leaves KV selection alone in front
    cm2 = dv.cost_model([2048, 131072], [50.0, 200.0], [[0, 0], [25, 25], [3, 5], [28, 30]],
                        [100.0, 4000.0])
    assert dv.plan_decode(D, keep, dv.request(steps=1000), cm2, 131072)["choice"] == dv.MODE_KV
    p = dv.plan_decode(D, keep, dv.request(steps=1000, modes=0b0011), cm, 131072)
    assert p["choice"] in (dv.MODE_DENSE, dv.MODE_ACT)
    # a one-step request cannot pay for the scoring pass at 128K
    p = dv.plan_decode(D, keep, dv.request(steps=1), cm, 131072)
    assert p["choice"] in (dv.MODE_DENSE, dv.MODE_ACT)
    # batches: the retained buffers serve batch 1 only
    p = dv.plan_decode(D, keep, dv.request(B=4, steps=1000), cm, 131072)
    assert p["choice"] in (dv.MODE_DENSE, dv.MODE_ACT)
    with pytest.raises(dv.DvError) as e:
        dv.plan_decode(D, keep, dv.request(B=4, modes=0b1100), cm, 131072)
    assert e.value.code == dv.DV_ERR_UNSUPPORTED


def test_validation():
    D = dv.dims(4096, 32, 8, 128, 14336, 1000, 1)
    keep = dv.Keep(0.5, 1.0, 0.125)
    cm = dv.cost_model([2048, 8192], [50.0, 60.0], [[0, 0]] * 4)
    bad = [
        (lambda: dv.plan_bytes(dv.dims(4096, 30, 8, 128, 14336, 1000, 1), keep, dv.request(), 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_bytes(D, dv.Keep(0.0, 1.0, 1.0), dv.request(), 10), dv.DV_ERR_KEEP),
        (lambda: dv.plan_bytes(D, dv.Keep(0.5, 1.5, 1.0), dv.request(), 10), dv.DV_ERR_KEEP),
        (lambda: dv.plan_bytes(D, keep, dv.request(B=0), 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_bytes(D, keep, dv.request(steps=0), 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_bytes(D, keep, dv.request(B=2, union_N=14337), 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_bytes(D, keep, dv.request(), -1), dv.DV_ERR_DIMS),
        (lambda: dv.plan_bytes(D, keep, dv.request(), float("nan")), dv.DV_ERR_DIMS),
        (lambda: dv.plan_decode(D, keep, dv.request(), cm, 0.0), dv.DV_ERR_DIMS),
        (lambda: dv.plan_decode(D, keep, dv.request(), dv.cost_model([8192, 2048], [1, 1], [[0, 0]] * 4), 10),
         dv.DV_ERR_DIMS),
        (lambda: dv.plan_decode(D, keep, dv.request(), dv.cost_model([2048], [1], [[0]] * 4), 10),
         dv.DV_ERR_DIMS),
        (lambda: dv.plan_decode(D, keep, dv.request(), dv.cost_model([2048, 4096], [1, 0], [[0, 0]] * 4), 10),
         dv.DV_ERR_DIMS),
        (lambda: dv.plan_decode(D, keep, dv.request(), dv.cost_model([1, 2], [1, 1], [[0, 0]] * 4, [0, -1]), 10),
         dv.DV_ERR_DIMS),
        (lambda: dv.plan_crossing(D, keep, dv.request(), cm, 1, 1, 1, 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_crossing(D, keep, dv.request(), cm, 1, 4, 1, 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_crossing(D, keep, dv.request(), cm, 1, 2, 10, 10), dv.DV_ERR_DIMS),
        (lambda: dv.plan_crossing(D, keep, dv.request(), cm, 1, 2, 0, 10), dv.DV_ERR_DIMS),
        (lambda: dv.cost_calibrate(D, keep, dv.request(), [1.0], [[1.0]] * 4), dv.DV_ERR_DIMS),
        (lambda: dv.cost_calibrate(D, keep, dv.request(), [1.0, 2.0], [[1.0, float("inf")]] * 4),
         dv.DV_ERR_DIMS),
    ]
    for i, (call, code) in enumerate(bad):
        with pytest.raises(dv.DvError) as e:
            call()
        assert e.value.code == code, i
    L = dv.lib()
    assert L.dv_plan_bytes(None, None, None, 1.0, None) == dv.DV_ERR_NULL
    assert L.dv_plan_decode(None, None, None, None, 1.0, None) == dv.DV_ERR_NULL
