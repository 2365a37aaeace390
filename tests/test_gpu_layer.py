"""GPU parity of whole decode layers and of the per-step driver.

Parity is teacher-forced per layer ("Deja Vu" §4.3 look-ahead makes index
choices depend on fp16 hidden states): layer l of the oracle takes the GPU's
input y_l and the GPU's index sets, and the sets themselves are checked
against the oracle's predictor scores (same size; swaps only within 1e-6 of
the k-th score). The C driver dv_decode_step must reproduce the layer-by-layer
result bit for bit, also when replayed from a CUDA graph.
"""
import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, check_sets, host, np16, npf, rel_err, setup_lib, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    setup_lib()
    dv.set_tuning()


class Stack:
    def __init__(self, w: synth.Workload, L, B=1, seed=0, full_bias=True):
        self.w, self.L, self.B = w, L, B
        self.n = w.n
        self.n_max = w.n + 4
        self.Wh = [synth.layer_weights(w, l, seed=seed, full_bias=full_bias) for l in range(L)]
        self.W = [to_dev(W) for W in self.Wh]
        self.KV0 = [synth.kv_cache(w, l, self.n_max, B=B, seed=seed) for l in range(L)]
        self.x = synth.hidden(w, B=B, seed=seed + 11)
        self.D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, self.n_max)
        self.keep = dv.Keep(w.keep_N, w.keep_H, 1.0)
        self.kN = w.F if w.keep_N >= 1 else oracle.k_from_keep(w.keep_N, w.F)
        self.kH = w.h_kv if w.keep_H >= 1 else oracle.k_from_keep(w.keep_H, w.h_kv)
        self.ws = dv.workspace(self.D, B)
        self.sets = [dv.sets(B, w.F, w.h_kv, self.kN, self.kH) for _ in range(2)]

    def fresh_kv(self):
        self.K = [k.cuda() for k, _ in self.KV0]
        self.V = [v.cuda() for _, v in self.KV0]
        return [dv.kv_cache(self.K[l], self.V[l]) for l in range(self.L)]


def _layer_by_layer(S: Stack, lookahead=True):
    kvs = S.fresh_kv()
    side = torch.cuda.Stream()
    evf, evj = dv.event(), dv.event()
    ys = [S.x.cuda()]
    used_sets = []
    for l in range(S.L):
        f = 0
        if l == 0 or not lookahead:
            f |= dv.DV_SYNC_PREDICT
        if lookahead and l > 0:
            f |= dv.DV_JOIN
        nxt = None
        if lookahead and l + 1 < S.L:
            f |= dv.DV_LOOKAHEAD
            nxt = (S.W[l + 1]["P1"], S.W[l + 1]["P2"])
        y_out = torch.empty_like(ys[0])
        cur, cur_t = S.sets[l & 1]
        dv.decode_layer(S.D, S.keep, S.W[l], nxt, kvs[l], S.n, cur, S.sets[(l + 1) & 1][0], ys[-1],
                        y_out, S.ws, f, ev_fork=evf, ev_join=evj, side=side)
        torch.cuda.synchronize()
        used_sets.append({k: v.clone() for k, v in cur_t.items()})
        ys.append(y_out)
    return ys, used_sets


def _check_stack(S: Stack, ys, used, lookahead=True):
    w = S.w
    for l in range(S.L):
        src = ys[l] if (l == 0 or not lookahead) else ys[l - 1]   # predictor input
        Wp = S.Wh[l]
        for b in range(S.B):
            if w.keep_N < 1 or w.keep_H < 1:
                ref = oracle.predict(np16(src[b]), np16(Wp["P1"]), np16(Wp["P2"]))
                if w.keep_N < 1:
                    check_sets(used[l]["idx_N"][b].cpu().numpy(), ref[: w.F], S.kN)
                if w.keep_H < 1:
                    check_sets(used[l]["idx_H"][b].cpu().numpy(), ref[w.F:], S.kH)
        # oracle layer on the GPU's input and sets (union for B > 1)
        if S.B == 1:
            selN = used[l]["idx_N"][0].cpu().numpy() if w.keep_N < 1 else np.arange(w.F)
            selH = used[l]["idx_H"][0].cpu().numpy() if w.keep_H < 1 else np.arange(w.h_kv)
            selN, selH = [selN], [selH]
        else:
            c = used[l]["ucnt"].cpu().numpy()
            selN = [used[l]["uN"][: c[0]].cpu().numpy() if w.keep_N < 1 else np.arange(w.F)] * S.B
            selH = [used[l]["uH"][: c[1]].cpu().numpy() if w.keep_H < 1 else np.arange(w.h_kv)] * S.B
            u = oracle.union(used[l]["idx_N"].cpu().numpy(), w.F)
            if w.keep_N < 1:
                assert np.array_equal(selN[0], u)
        K, V = S.KV0[l]
        for b in range(S.B):
            y_ref, h_ref, a, m = oracle.layer(np16(ys[l][b]), S.Wh[l], np16(K[b]), np16(V[b]), S.n,
                                              selH[b], selN[b])
            assert rel_err(npf(ys[l + 1][b]), y_ref) < TOL, (l, b)


@pytest.mark.parametrize("wl,over,L,B", [
    ("tiny", {}, 3, 1),
    ("tiny", dict(d=1024, h=16, h_kv=16, F=4096, r=128, n=128), 3, 1),
    ("tiny", dict(keep_H=1.0), 2, 1),          # dense heads, sparse neurons
    ("tiny", dict(keep_N=1.0), 2, 1),          # dense neurons, sparse heads
    ("tiny", {}, 2, 4),                        # batch-4 union path
])
def test_decode_layers_teacher_forced(wl, over, L, B):
    S = Stack(synth.workload(wl, **over), L, B)
    ys, used = _layer_by_layer(S)
    _check_stack(S, ys, used)


def test_sync_mode_layers():
    S = Stack(synth.workload("tiny"), 2)
    ys, used = _layer_by_layer(S, lookahead=False)
    _check_stack(S, ys, used, lookahead=False)


def test_driver_matches_layers_and_graph_replay():
    S = Stack(synth.workload("tiny", d=512, h=8, h_kv=8, F=2048, r=64, n=96), 4)
    ys, _ = _layer_by_layer(S)
    side = torch.cuda.Stream()
    evf, evj = dv.event(), dv.event()
    y_tmp = torch.empty(2, 1, S.w.d, dtype=torch.float16, device="cuda")
    y_out = torch.empty(1, S.w.d, dtype=torch.float16, device="cuda")
    kvs = S.fresh_kv()
    sets2 = [s for s, _ in S.sets]
    x = S.x.cuda()
    dv.decode_step(S.D, S.keep, S.W, kvs, S.n, sets2, x, y_tmp, y_out, S.ws, dv.DV_LOOKAHEAD,
                   side, evf, evj)
    torch.cuda.synchronize()
    assert torch.equal(y_out, ys[-1])
    # capture the whole step in a CUDA graph and replay it
    kvs = S.fresh_kv()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            dv.decode_step(S.D, S.keep, S.W, kvs, S.n, sets2, x, y_tmp, y_out, S.ws,
                           dv.DV_LOOKAHEAD, side, evf, evj, stream=s)
    y_out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(y_out, ys[-1])


def test_composition_layer_retained_kv():
    # d 1024, 8 query / 2 KV heads x 128, neuron keep 1/2, KV keep 1/8 of n = 512
    w = synth.workload("compose", d=1024, h=8, h_kv=2, F=2048, r=64, n=512, obs_window=16)
    S = Stack(w, 1)
    kvs = S.fresh_kv()
    b = oracle.kv_budget(w.n, w.keep_KV)
    b_max = b + 8
    Kr = torch.zeros(w.h_kv, b_max, w.dh, dtype=torch.float16, device="cuda")
    Vr = torch.zeros_like(Kr)
    kp = torch.zeros(w.h_kv, b_max, dtype=torch.int32, device="cuda")
    kc = torch.zeros(w.h_kv, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(S.K[0], S.V[0], Kr=Kr, Vr=Vr, kept_pos=kp, kept_count=kc, b_max=b_max)
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, S.n_max)
    ws = dv.workspace(D, 1, dv.DV_KV_RESELECT)
    q_obs = synth.obs_queries(w, 0)
    H = torch.zeros(w.h, w.dh, device="cuda")
    q = torch.zeros(w.h, w.dh, device="cuda")
    dv.kv_select_attn(q, D, kv, w.n, H, ws, q_obs=q_obs.cuda(), obs_window=w.obs_window,
                      kv_keep=w.keep_KV, flags=dv.DV_KV_RESELECT)
    torch.cuda.synchronize()
    counts = kc.cpu().numpy().copy()
    kept = [kp[u, : counts[u]].cpu().numpy() for u in range(w.h_kv)]
    y_out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
    cur, cur_t = S.sets[0]
    dv.decode_layer(D, dv.Keep(w.keep_N, 1.0, w.keep_KV), S.W[0], None, kv, w.n, cur, None,
                    S.x.cuda(), y_out, ws, dv.DV_SYNC_PREDICT | dv.DV_KV_RETAINED)
    torch.cuda.synchronize()
    selN = cur_t["idx_N"][0].cpu().numpy()
    K, V = S.KV0[0]
    kept_arr = np.zeros((w.h_kv, max(len(k) for k in kept)), np.int32)
    for u in range(w.h_kv):
        kept_arr[u, : len(kept[u])] = kept[u]
    a = oracle.attn_kvsel(np16(S.x[0]), S.Wh[0], np16(K[0]), np16(V[0]), w.n, kept_arr, counts)
    hmid = oracle.round_fp16(npf(S.x[0]) + a.delta)
    Wh = S.Wh[0]
    m = oracle.mlp_gather(hmid, Wh["fc1"], Wh["b1"], Wh["fc2T"], Wh["b2"], selN, ln_g=Wh["ln2_g"],
                          ln_b=Wh["ln2_b"])
    y_ref = oracle.round_fp16(hmid.astype(float) + m)
    assert rel_err(npf(y_out[0]), y_ref) < TOL
    # the new token was appended to the retained buffer after the kept rows
    for u in range(w.h_kv):
        assert rel_err(npf(Kr[u, counts[u]]), a.knew[u].astype(float)) < TOL
