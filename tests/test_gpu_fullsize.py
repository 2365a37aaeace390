"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times: the whole L-layer stack on the GPU (seeded weights drawn on
the device), one decode step replayed from its captured CUDA graph with the
look-ahead predictor on the side stream. The last layer is then checked
against the oracle, teacher-forced: its input y_{L-1} and its index sets come
from the GPU; the sets are checked against the oracle's predictor scores on
y_{L-2} (the look-ahead input), and the layer output against the oracle layer.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, check_sets, np16, npf, rel_err, setup_lib

pytestmark = pytest.mark.gpu


def _step(w, kv_dense=False):
    setup_lib()
    dv.set_tuning()
    m = bench.Model(w, torch.device("cuda", 0), lookahead=True, kv_dense=kv_dense)
    s = torch.cuda.Stream()
    g, _ = m.capture(s)
    g.replay()
    torch.cuda.synchronize()
    assert m.st.item() == 0, m.st.item()
    return m


def _check_layer(m, l, y_prev, y_in, y_out, sets_t, kv_sel=None):
    """Layer l of a replayed step, teacher-forced: its input y_in and its sets
    come from the GPU. The sets are checked against the oracle's predictor of
    layer l on y_prev (the look-ahead input y_{l-1}; for layer 0, which
    predicts synchronously, its own input), and the output y_out against the
    oracle layer on y_in with those sets."""
    w = m.w
    Wh = {k: np16(v) for k, v in m.W[l].items()}
    for b in range(w.B):
        ref = oracle.predict(np16(y_prev[b]), Wh["P1"], Wh["P2"])
        if w.keep_N < 1:
            check_sets(sets_t["idx_N"][b].cpu().numpy(), ref[: w.F], m.kN)
        if w.keep_H < 1:
            check_sets(sets_t["idx_H"][b].cpu().numpy(), ref[w.F:], m.kH)
    if w.B == 1:
        selN = sets_t["idx_N"][0].cpu().numpy() if w.keep_N < 1 else np.arange(w.F)
        selH = sets_t["idx_H"][0].cpu().numpy() if w.keep_H < 1 else np.arange(w.h_kv)
    else:
        c = sets_t["ucnt"].cpu().numpy()
        selN = sets_t["uN"][: c[0]].cpu().numpy() if w.keep_N < 1 else np.arange(w.F)
        selH = sets_t["uH"][: c[1]].cpu().numpy() if w.keep_H < 1 else np.arange(w.h_kv)
        assert np.array_equal(selN, oracle.union(sets_t["idx_N"].cpu().numpy(), w.F))
    K, V = np16(m.K[l]), np16(m.V[l])
    for b in range(w.B):
        if kv_sel is None:
            y_ref, *_ = oracle.layer(np16(y_in[b]), Wh, K[b], V[b], w.n, selH, selN)
        else:
            kept, counts = kv_sel
            a = oracle.attn_kvsel(np16(y_in[b]), Wh, K[b], V[b], w.n, kept, counts)
            hmid = oracle.round_fp16(npf(y_in[b]) + a.delta)
            mm = oracle.mlp_gather(hmid, Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh.get("b2"), selN)
            y_ref = oracle.round_fp16(hmid.astype(float) + mm)
        assert rel_err(npf(y_out[b]), y_ref) < TOL, (l, b)


def _check_last_layer(m, kv_sel=None):
    L = m.L
    y_prev = m.y_tmp[(L - 3) & 1] if L >= 3 else m.x          # y_{L-2}
    y_in = m.y_tmp[(L - 2) & 1] if L >= 2 else m.x            # y_{L-1}
    _check_layer(m, L - 1, y_prev, y_in, m.y_out, m.sets[(L - 1) & 1][1], kv_sel)


def _check_first_layers(m):
    """Layers 0 and 1 of the same stack, from a step over its first two layers
    in the same launch configuration: layer 0 predicts its sets synchronously
    from its input, layer 1 reads the sets layer 0 looked ahead for it."""
    w = m.w
    step2 = dv.Step(m.D, m.keep, m.W[:2], m.kvs[:2], [s for s, _ in m.sets], m.ws, m.step.flags,
                    m.side, m.evf, m.evj, dev_status=m.st)
    y_tmp = torch.empty(2, w.B, w.d, dtype=torch.float16, device="cuda")
    y_out = torch.empty(w.B, w.d, dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step2(m.x, y_tmp, y_out, m.n, stream=s)
    torch.cuda.synchronize()
    assert m.st.item() == 0, m.st.item()
    _check_layer(m, 0, m.x, m.x, y_tmp[0], m.sets[0][1])
    _check_layer(m, 1, m.x, y_tmp[0], y_out, m.sets[1][1])


def test_opt175b_stack_as_benchmarked():
    # 24 layers, d 12288, 96 heads, FFN 49152, neuron keep 10 %, head keep 50 %
    m = _step(synth.workload("opt-175b"))
    _check_last_layer(m)
    _check_first_layers(m)


def test_opt67b_stack():
    m = _step(synth.workload("opt-6.7b"))
    _check_last_layer(m)
    _check_first_layers(m)


@pytest.mark.parametrize("kn,kh", [(0.1, 0.25), (0.5, 1.0)])
def test_opt175b_keep_sweep_corners(kn, kh):
    # the corners of the benchmarked opt-175b keep sweep, 24 layers
    m = _step(synth.workload("opt-175b", keep_N=kn, keep_H=kh))
    _check_last_layer(m)


@pytest.mark.parametrize("kn,kh", [(0.1, 1.0), (0.5, 0.5)])
def test_opt67b_keep_sweep_full_stack(kn, kh):
    m = _step(synth.workload("opt-6.7b", keep_N=kn, keep_H=kh))
    _check_last_layer(m)


def test_opt66b_batch1_stack():
    # 16 layers, d 9216, 72 heads, FFN 36864, neuron keep 10 %, head keep 50 %
    m = _step(synth.workload("opt-66b"))
    _check_last_layer(m)
    _check_first_layers(m)


@pytest.mark.parametrize("kn,kh", [(0.25, 1.0), (1.0, 0.5), (1.0, 1.0)])
def test_opt67b_keep_variants(kn, kh):
    m = _step(synth.workload("opt-6.7b", keep_N=kn, keep_H=kh, layers=4))
    _check_last_layer(m)


def test_opt66b_batch4_union():
    m = _step(synth.workload("opt-66b", B=4))
    _check_last_layer(m)


@pytest.mark.parametrize("n", [2048, 8192, 32768, 131072])
def test_composition_retained_kv(n):
    # d 4096, 32 query / 8 KV heads x 128, neuron keep 1/2, KV keep 1/8;
    # the full 32 layers, decode through the retained KV buffers
    w = synth.workload("compose", n=n)
    m = _step(w)
    L = m.L
    counts = m.kc[L - 1].cpu().numpy()
    b = int(n * w.keep_KV)
    W = w.obs_window
    kept = np.zeros((w.h_kv, int(counts.max())), np.int32)
    for u in range(w.h_kv):
        k = m.kp[L - 1][u, : counts[u]].cpu().numpy()
        assert counts[u] == b and np.all(np.diff(k) > 0)
        assert set(range(4)) <= set(k) and set(range(n - W, n)) <= set(k)
        # the retained rows are the cache rows at the kept positions
        assert np.array_equal(np16(m.Kr[L - 1][u, : counts[u]]).view(np.uint16),
                              np16(m.K[L - 1][0, u, k]).view(np.uint16))
        kept[u, : counts[u]] = k
    _check_last_layer(m, kv_sel=(kept, counts))


def test_composition_dense_split_k_baseline():
    w = synth.workload("compose", n=8192, layers=4)
    m = _step(w, kv_dense=True)
    _check_last_layer(m)


@pytest.mark.parametrize("B", [1, 4])
def test_opt67b_decode_steps_recompute_missing_kv(B):
    # five decode steps of a 3-layer opt-6.7b stack with a growing context,
    # a new input each step and the look-ahead predictor choosing the sets;
    # the last layer of every step is checked against the oracle's multi-step
    # attention ("Deja Vu" §4.2: every past token's k, v from its own input).
    # At batch 4 the sets are the unions of the four sequences' sets.
    setup_lib()
    dv.set_tuning()
    w = synth.workload("opt-6.7b", layers=3, B=B)
    T, L = 5, 3
    dev = torch.device("cuda", 0)
    m = bench.Model(w, dev, lookahead=True, kept_inputs=True, fill=True, extra_slots=T)
    K0, V0 = np16(m.K[L - 1]).copy(), np16(m.V[L - 1]).copy()
    xs = [synth.hidden(w, seed=500 + t, device=dev) for t in range(T)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    y_in, selH, selN, y_out = [], [], [], []
    for t in range(T):
        with torch.cuda.stream(s):
            m.step(xs[t], m.y_tmp, m.y_out, w.n + t, stream=s)
        torch.cuda.synchronize()
        assert m.st.item() == 0
        sets_t = m.sets[(L - 1) & 1][1]
        y_in.append(np16(m.y_tmp[(L - 2) & 1]).copy())
        if B == 1:
            selH.append(sets_t["idx_H"][0].cpu().numpy().copy())
            selN.append(sets_t["idx_N"][0].cpu().numpy().copy())
        else:
            c = sets_t["ucnt"].cpu().numpy()
            selH.append(sets_t["uH"][: c[1]].cpu().numpy().copy())
            selN.append(sets_t["uN"][: c[0]].cpu().numpy().copy())
        y_out.append(npf(m.y_out))
    # the sets change from step to step, so some units have holes to fill
    assert B > 1 or any(set(selH[t]) - set(selH[t - 1]) for t in range(1, T))
    Wh = {k: np16(v) for k, v in m.W[L - 1].items()}
    for b in range(B):
        ref, _, _ = oracle.attn_steps([y[b] for y in y_in], Wh, K0[b], V0[b], w.n, selH)
        for t in range(T):
            hmid = oracle.round_fp16(y_in[t][b].astype(np.float64) + ref[t].delta)
            mm = oracle.mlp_gather(hmid, Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh.get("b2"), selN[t])
            y_ref = oracle.round_fp16(hmid.astype(float) + mm)
            assert rel_err(y_out[t][b], y_ref) < TOL, (b, t)


def test_opt67b_stack_w4a16():
    # the opt-6.7b stack with 4-bit projection and MLP rows (W4A16, "Deja Vu"
    # §5.2, Table 7), fp16 predictor, look-ahead on the side stream, replayed
    # from its graph; the last layer checked against the oracle's W4 layer
    from oracle import w4 as ow4
    setup_lib()
    dv.set_tuning()
    w = synth.workload("opt-6.7b", layers=4)
    m = bench.Model(w, torch.device("cuda", 0), lookahead=True, w4=True)
    s = torch.cuda.Stream()
    g, _ = m.capture(s)
    g.replay()
    torch.cuda.synchronize()
    assert m.st.item() == 0
    L = m.L
    y_prev, y_in = m.y_tmp[(L - 3) & 1], m.y_tmp[(L - 2) & 1]
    sets_t = m.sets[(L - 1) & 1][1]
    Wl = m.W[L - 1]
    Wo = {k: (ow4.unpack(v.cpu().numpy(), w.d) if v.dtype == torch.uint8 else np16(v))
          for k, v in Wl.items()}
    ref = oracle.predict(np16(y_prev[0]), Wo["P1"], Wo["P2"])
    check_sets(sets_t["idx_N"][0].cpu().numpy(), ref[: w.F], m.kN)
    check_sets(sets_t["idx_H"][0].cpu().numpy(), ref[w.F:], m.kH)
    y_ref, _ = ow4.layer(np16(y_in[0]), Wo, np16(m.K[L - 1][0]), np16(m.V[L - 1][0]), w.n,
                         sets_t["idx_H"][0].cpu().numpy(), sets_t["idx_N"][0].cpu().numpy())
    assert rel_err(npf(m.y_out[0]), y_ref.astype(np.float64)) < TOL
