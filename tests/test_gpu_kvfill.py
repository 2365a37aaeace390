"""Multi-step decode with head sparsity: the missing k, v of skipped units are
recomputed from the kept inputs before a later step reads them ("Deja Vu"
§4.2), through the C ABI (dv_sparse_attn with DV_KV_FILL), against the
oracle's multi-step attention, which computes every past token's k, v from
that token's own input."""
import numpy as np
import pytest
import torch

import oracle
from contextual_sparsity_gb300 import dv, synth
from gpu_helpers import TOL, host, np16, npf, rel_err, setup_lib, to_dev

pytestmark = pytest.mark.gpu


def _schedule(kind, hkv, T, rng):
    """Selected units of every step."""
    if kind == "designed":
        # unit 0 every step; unit 1 only at the last step; unit 2 every other
        # step; unit 3 at steps 0, 5 and 6; the rest at random
        sels = []
        for t in range(T):
            s = {0}
            if t == T - 1:
                s.add(1)
            if t % 2 == 0:
                s.add(2)
            if t in (0, 5, 6):
                s.add(3)
            for u in range(4, hkv):
                if rng.random() < 0.5:
                    s.add(u)
            sels.append(sorted(s))
        return sels
    if kind == "deep":
        # unit 1 at step 0 and then only at the last step (a hole run longer
        # than 32 positions); unit 2 first selected at the last step
        sels = [[0, 1] if t == 0 else [0] for t in range(T)]
        sels[-1] = [0, 1, 2]
        return sels
    k = max(1, hkv // 2)
    return [sorted(rng.choice(hkv, k, replace=False).tolist()) for _ in range(T)]


@pytest.mark.parametrize("wl,over,n0,T,kind", [
    ("tiny", {}, 40, 12, "designed"),
    ("tiny", {}, 10, 45, "deep"),
    ("compose", dict(d=512, h=8, h_kv=2, F=64), 100, 8, "random"),      # GQA, 4 heads per unit
    ("opt-6.7b", dict(F=64), 200, 6, "random"),                          # d 4096, 32 units
    ("opt-6.7b", dict(d=1024, h=40, h_kv=40, dh=64, F=64), 60, 10, "random"),  # two mark words
    ("tiny", {}, 0, 9, "designed"),                                      # no prefill at all
    ("opt-175b", dict(F=64), 100, 4, "random"),       # d 12288, 96 units: three mark words
])
def test_multistep_missing_kv_recompute(wl, over, n0, T, kind):
    setup_lib()
    w = synth.workload(wl, **over)
    rng = np.random.default_rng(n0 + T)
    W = synth.layer_weights(w, 0, seed=3, full_bias=True)
    n_max = n0 + T + 3
    K, V = synth.kv_cache(w, 0, n_max, B=1, seed=3)
    ys = [synth.hidden(w, B=1, seed=100 + t) for t in range(T)]
    sels = _schedule(kind, w.h_kv, T, rng)

    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws = dv.workspace(D, 1)
    Kd, Vd = K.cuda(), V.cuda()
    y_side = torch.zeros(1, n_max, w.d, dtype=torch.float16, device="cuda")
    words = (w.h_kv + 31) // 32
    miss = torch.zeros(1, n_max, words, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(Kd, Vd, y_side=y_side, kv_missing=miss)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wd = to_dev(W)
    outs = []
    for t in range(T):
        out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
        sd = torch.tensor(sels[t], dtype=torch.int32, device="cuda")
        dv.sparse_attn(ys[t].cuda(), D, Wd, sd, len(sels[t]), kv, n0 + t, out, ws,
                       flags=dv.DV_NO_RESIDUAL | dv.DV_KV_FILL, dev_status=st)
        outs.append(out)
    torch.cuda.synchronize()
    assert st.item() == 0

    Wh = host(W)
    ref, Kf, Vf = oracle.attn_steps([np16(y[0]) for y in ys], Wh, np16(K[0]), np16(V[0]), n0,
                                    sels)
    for t in range(T):
        assert rel_err(npf(outs[t][0]), ref[t].delta) < TOL, t

    # marks: after the last step, unit u is marked exactly on the positions
    # after its last selection; everything else holds its own token's k, v
    bits = miss[0].cpu().numpy().view(np.uint32)
    Kg, Vg = Kd[0].cpu().numpy(), Vd[0].cpu().numpy()
    n_end = n0 + T
    for u in range(w.h_kv):
        last = max([t for t in range(T) if u in sels[t]], default=-1)
        marked = [(bits[p, u // 32] >> (u % 32)) & 1 for p in range(n_end)]
        want = [1 if p >= n0 + last + 1 else 0 for p in range(n_end)]
        want[:n0] = [0] * n0
        assert marked == want, u
        filled = list(range(n0 + last + 1)) if last >= 0 else list(range(n0))
        if filled:
            assert rel_err(Kg[u, filled].astype(float), Kf[u, filled].astype(float)) < TOL, u
            assert rel_err(Vg[u, filled].astype(float), Vf[u, filled].astype(float)) < TOL, u


def test_fill_needs_the_kept_inputs_and_the_full_cache():
    setup_lib()
    w = synth.workload("tiny")
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, 16)
    ws = dv.workspace(D, 1)
    K = torch.zeros(1, w.h_kv, 16, w.dh, dtype=torch.float16, device="cuda")
    x = torch.zeros(1, w.d, dtype=torch.float16, device="cuda")
    out = torch.empty_like(x)
    W = to_dev(synth.layer_weights(w, 0))
    kv = dv.kv_cache(K, K.clone())
    with pytest.raises(dv.DvError) as e:
        dv.sparse_attn(x, D, W, None, w.h_kv, kv, 4, out, ws, flags=dv.DV_KV_FILL)
    assert e.value.code in (dv.DV_ERR_NULL, dv.DV_ERR_ALIGN)


def test_multistep_missing_kv_batch4_union():
    # four sequences decoded together over one (union) set of units per step;
    # each sequence's cache gets its own recomputed rows from its own inputs
    setup_lib()
    w = synth.workload("opt-6.7b", d=1024, h=16, h_kv=16, dh=64, F=64)
    B, n0, T = 4, 30, 7
    rng = np.random.default_rng(4)
    W = synth.layer_weights(w, 0, seed=5, full_bias=True)
    n_max = n0 + T + 2
    K, V = synth.kv_cache(w, 0, n_max, B=B, seed=5)
    ys = [synth.hidden(w, B=B, seed=300 + t) for t in range(T)]
    sels = [sorted(rng.choice(w.h_kv, 6, replace=False).tolist()) for _ in range(T)]
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws = dv.workspace(D, B)
    Kd, Vd = K.cuda(), V.cuda()
    y_side = torch.zeros(B, n_max, w.d, dtype=torch.float16, device="cuda")
    miss = torch.zeros(B, n_max, (w.h_kv + 31) // 32, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(Kd, Vd, y_side=y_side, kv_missing=miss)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wd = to_dev(W)
    outs = []
    for t in range(T):
        out = torch.empty(B, w.d, dtype=torch.float16, device="cuda")
        sd = torch.tensor(sels[t], dtype=torch.int32, device="cuda")
        dv.sparse_attn(ys[t].cuda(), D, Wd, sd, len(sels[t]), kv, n0 + t, out, ws,
                       flags=dv.DV_NO_RESIDUAL | dv.DV_KV_FILL, dev_status=st)
        outs.append(out)
    torch.cuda.synchronize()
    assert st.item() == 0
    Wh = host(W)
    for b in range(B):
        ref, Kf, _ = oracle.attn_steps([np16(y[b]) for y in ys], Wh, np16(K[b]), np16(V[b]), n0,
                                       sels)
        for t in range(T):
            assert rel_err(npf(outs[t][b]), ref[t].delta) < TOL, (b, t)
        Kg = Kd[b].cpu().numpy()
        for u in range(w.h_kv):
            last = max([t for t in range(T) if u in sels[t]], default=-1)
            if last >= 0:
                rows = list(range(n0 + last + 1))
                assert rel_err(Kg[u, rows].astype(float), Kf[u, rows].astype(float)) < TOL, (b, u)


def test_multistep_missing_kv_with_retained_buffer():
    # composition ("Where Activation Sparsity and KV-Cache Sparsity Cross",
    # §3.2: neither branch discards state): attention reads the retained KV
    # buffer (kept positions of a selection, then every decoded token), the
    # units are head-sparse per step, and a unit's missing rows are recomputed
    # into the full cache and into their retained slots before it is read.
    # Reference: for each step and selected unit, the oracle's attention over
    # the kept positions plus the decoded tokens, every token's k, v from its
    # own input (oracle.token_kv), the new token's from this step's input.
    setup_lib()
    w = synth.workload("compose", d=512, h=16, h_kv=4, F=64, obs_window=16)
    n0, T, keep = 120, 8, 0.25
    rng = np.random.default_rng(7)
    W = synth.layer_weights(w, 0, seed=9, full_bias=True)
    n_max = n0 + T + 4
    K, V = synth.kv_cache(w, 0, n_max, B=1, seed=9)
    q_obs = synth.obs_queries(w, 0, seed=9)
    ys = [synth.hidden(w, B=1, seed=700 + t) for t in range(T)]
    sels = [sorted(rng.choice(w.h_kv, 2, replace=False).tolist()) for _ in range(T)]
    b = oracle.kv_budget(n0, keep)
    b_max = b + T + 8
    D = dv.dims(w.d, w.h, w.h_kv, w.dh, w.F, w.r, n_max)
    ws_sel = dv.workspace(D, 1, dv.DV_KV_RESELECT)
    ws = dv.workspace(D, 1)
    Kd, Vd = K.cuda(), V.cuda()
    Kr = torch.zeros(w.h_kv, b_max, w.dh, dtype=torch.float16, device="cuda")
    Vr = torch.zeros_like(Kr)
    kp = torch.zeros(w.h_kv, b_max, dtype=torch.int32, device="cuda")
    kc = torch.zeros(w.h_kv, dtype=torch.int32, device="cuda")
    y_side = torch.zeros(1, n_max, w.d, dtype=torch.float16, device="cuda")
    miss = torch.zeros(1, n_max, 1, dtype=torch.int32, device="cuda")
    kv = dv.kv_cache(Kd, Vd, y_side=y_side, kv_missing=miss, Kr=Kr, Vr=Vr, kept_pos=kp,
                     kept_count=kc, b_max=b_max)
    H = torch.zeros(w.h, w.dh, device="cuda")
    dv.kv_select_attn(torch.zeros(w.h, w.dh, device="cuda"), D, kv, n0, H, ws_sel,
                      q_obs=q_obs.cuda(), obs_window=w.obs_window, kv_keep=keep,
                      flags=dv.DV_KV_RESELECT)
    torch.cuda.synchronize()
    counts0 = kc.cpu().numpy().copy()
    kept0 = [kp[u, : counts0[u]].cpu().numpy().copy() for u in range(w.h_kv)]
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    Wd = to_dev(W)
    outs = []
    flags = dv.DV_NO_RESIDUAL | dv.DV_KV_FILL | dv.DV_KV_RETAINED | dv.DV_KV_ADVANCE
    for t in range(T):
        out = torch.empty(1, w.d, dtype=torch.float16, device="cuda")
        sd = torch.tensor(sels[t], dtype=torch.int32, device="cuda")
        dv.sparse_attn(ys[t].cuda(), D, Wd, sd, len(sels[t]), kv, n0 + t, out, ws, flags=flags,
                       dev_status=st)
        outs.append(out)
    torch.cuda.synchronize()
    assert st.item() == 0
    assert np.array_equal(kc.cpu().numpy(), counts0 + T)

    Wh = host(W)
    Kc, Vc = np16(K[0]).copy(), np16(V[0]).copy()
    bo = Wh.get("bo")
    bo = np.zeros(w.d) if bo is None else bo.astype(np.float64)
    for t in range(T):
        n = n0 + t
        y = np16(ys[t][0])
        want = bo.copy()
        for u in sels[t]:
            pos = np.concatenate([kept0[u], np.arange(n0, n)]).astype(np.int64)
            Ks = np.zeros((w.h_kv, len(pos) + 1, w.dh), np.float16)
            Vs = np.zeros_like(Ks)
            Ks[u, : len(pos)], Vs[u, : len(pos)] = Kc[u, pos], Vc[u, pos]
            a = oracle.attn_gather(y, Wh, Ks, Vs, len(pos), [u])
            want += a.delta - bo
        assert rel_err(npf(outs[t][0]), want) < TOL, t
        Kc[:, n], Vc[:, n] = oracle.token_kv(y, Wh, w.h_kv, w.dh)
    # the retained slots of the decoded tokens hold their own k (for the
    # positions up to each unit's last selection: later ones are still holes)
    Krg = Kr.cpu().numpy()
    for u in range(w.h_kv):
        last = max([t for t in range(T) if u in sels[t]], default=-1)
        if last >= 0:
            slots = counts0[u] + np.arange(last + 1)
            assert rel_err(Krg[u, slots].astype(float), Kc[u, n0:n0 + last + 1].astype(float)) < TOL, u
