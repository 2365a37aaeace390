"""CPU oracle for the Deja Vu contextual-sparsity decode step (test infrastructure).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package. The product path (``contextual_sparsity_gb300``) never does.

The arithmetic lives in ``dv_oracle.c`` (plain single-threaded C, fp64): this
module only loads it with ctypes and marshals numpy arrays. The byte account
(closed forms, pure Python) is in :mod:`oracle.byte_account`. Each function
below names the passage of the pages it follows:

* "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time"
  (arXiv 2310.17157): §2.3 Eq. 1-2, §4.1-4.3, App. C.1, C.3, D.
* "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding"
  (arXiv 2609.33889): §3, §4.1, App. A, App. C.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dv_oracle.c")
_LIB = os.path.join(_HERE, "libdv_oracle.so")

# -ffp-contract=off: no fused multiply-add contraction, so the oracle gives the
# same bits on x86-64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile dv_oracle.c into libdv_oracle.so next to it (gcc, no GPU)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


class _AttnDims(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int), ("h", ctypes.c_int), ("hkv", ctypes.c_int),
                ("dh", ctypes.c_int), ("n", ctypes.c_int), ("n_max", ctypes.c_int),
                ("eps", ctypes.c_double), ("scale", ctypes.c_double)]


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.or_h2d.restype = ctypes.c_double
        _lib.or_h2d.argtypes = [ctypes.c_uint16]
        _lib.or_d2h.restype = ctypes.c_uint16
        _lib.or_d2h.argtypes = [ctypes.c_double]
        _lib.or_topk.restype = ctypes.c_int
        _lib.or_union.restype = ctypes.c_int
        _lib.or_kv_choose.restype = ctypes.c_int
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _h(a):
    """fp16 array (or None) -> contiguous uint16 view."""
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    assert a.dtype == np.float16, a.dtype
    return a.view(np.uint16)


def _f64(shape):
    return np.zeros(shape, dtype=np.float64)


# --------------------------------------------------------------------------
# fp16 conversion
# --------------------------------------------------------------------------
def h2d(bits: np.ndarray) -> np.ndarray:
    """Exact binary16 -> double decode of an array of uint16 bit patterns."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = _f64(bits.shape)
    lib().or_h2d_array(_p(bits), _p(out), ctypes.c_int64(bits.size))
    return out


def d2h(x: np.ndarray) -> np.ndarray:
    """double -> binary16 (round to nearest even); returns uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint16)
    lib().or_d2h_array(_p(x), _p(out), ctypes.c_int64(x.size))
    return out


def round_fp16(x: np.ndarray) -> np.ndarray:
    """double -> nearest fp16, returned as a float16 array."""
    return d2h(x).view(np.float16)


# --------------------------------------------------------------------------
# a1 LayerNorm, a2 predictor, a3 top-k / union
# --------------------------------------------------------------------------
def layernorm(x, g=None, b=None, eps=1e-5):
    x = _h(x)
    z = _f64(x.shape[-1])
    lib().or_layernorm(_p(x), ctypes.c_int(x.shape[-1]), _p(_h(g)), _p(_h(b)),
                       ctypes.c_double(eps), _p(z))
    return z


def predict(y, P1, P2, relu=False):
    """Scores s = act(y P1^T) P2^T in fp64 (Deja Vu §4.1 "Design", §4.2)."""
    y, P1, P2 = _h(y), _h(P1), _h(P2)
    r, d = P1.shape
    N = P2.shape[0]
    assert P2.shape[1] == r and y.shape[-1] == d
    s = _f64(N)
    lib().or_predict(_p(y), ctypes.c_int(d), _p(P1), ctypes.c_int(r), _p(P2), ctypes.c_int(N),
                     ctypes.c_int(1 if relu else 0), _p(s))
    return s


def topk(scores, k):
    """k largest scores, ties to the lower index, returned ascending (int32)."""
    s = np.ascontiguousarray(scores, dtype=np.float64)
    idx = np.zeros(k, dtype=np.int32)
    rc = lib().or_topk(_p(s), ctypes.c_int(s.size), ctypes.c_int(k), _p(idx))
    if rc != 0:
        raise ValueError("or_topk: bad arguments or NaN score")
    return idx


def union(idx, N):
    """Union of the rows of idx [B][k] over [0, N), ascending (Deja Vu App. C.1)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    B, k = idx.shape
    out = np.zeros(N, dtype=np.int32)
    c = lib().or_union(_p(idx), ctypes.c_int(B), ctypes.c_int(k), ctypes.c_int(N), _p(out))
    return out[:c].copy()


def k_from_keep(keep: float, N: int) -> int:
    """Budget of Deja Vu §2.3: |S| <= (1 - sparsity) N, so k = max(1, floor(keep N))."""
    return max(1, int(math.floor(keep * N + 1e-9)))


# --------------------------------------------------------------------------
# a4 MLP block (Deja Vu §2.3 Eq. 1)
# --------------------------------------------------------------------------
def mlp_gather(x, fc1, b1, fc2T, b2, idx, ln_g=None, ln_b=None, eps=1e-5, return_act=False):
    x, fc1, fc2T = _h(x), _h(fc1), _h(fc2T)
    F, d = fc1.shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    delta, act = _f64(d), _f64(max(1, idx.size))
    lib().or_mlp_gather(_p(x), ctypes.c_int(d), _p(_h(ln_g)), _p(_h(ln_b)), ctypes.c_double(eps),
                        _p(fc1), _p(_h(b1)), _p(fc2T), _p(_h(b2)), _p(idx),
                        ctypes.c_int(idx.size), _p(delta), _p(act))
    return (delta, act[: idx.size]) if return_act else delta


def mlp_masked(x, fc1, b1, fc2T, b2, mask=None, ln_g=None, ln_b=None, eps=1e-5, return_act=False):
    x, fc1, fc2T = _h(x), _h(fc1), _h(fc2T)
    F, d = fc1.shape
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    delta, act = _f64(d), _f64(F)
    lib().or_mlp_masked(_p(x), ctypes.c_int(d), ctypes.c_int(F), _p(_h(ln_g)), _p(_h(ln_b)),
                        ctypes.c_double(eps), _p(fc1), _p(_h(b1)), _p(fc2T), _p(_h(b2)), _p(m),
                        _p(delta), _p(act))
    return (delta, act) if return_act else delta


# --------------------------------------------------------------------------
# a5-a7 MHA block (Deja Vu §2.3 Eq. 2) and a9 attention over retained KV
# --------------------------------------------------------------------------
class AttnOut:
    def __init__(self, delta, H, knew, vnew):
        self.delta, self.H, self.knew, self.vnew = delta, H, knew, vnew


def _attn_common(x, W, Kc, n, scale, eps):
    x = _h(x)
    d = x.shape[-1]
    Wq = _h(W["Wq"])
    dh = Kc.shape[-1]
    h = Wq.shape[0] // dh
    hkv = Kc.shape[0]
    n_max = Kc.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(dh)
    D = _AttnDims(d, h, hkv, dh, n, n_max, eps, scale)
    return x, D, h, hkv, dh


def _attn_args(W):
    return [_p(_h(W.get("ln1_g"))), _p(_h(W.get("ln1_b"))), _p(_h(W["Wq"])), _p(_h(W.get("bq"))),
            _p(_h(W["Wk"])), _p(_h(W.get("bk"))), _p(_h(W["Wv"])), _p(_h(W.get("bv"))),
            _p(_h(W["WoT"])), _p(_h(W.get("bo")))]


def attn_gather(x, W, Kc, Vc, n, sel, scale=None, eps=1e-5):
    """Sparse MHA over the selected units (KV heads; one head each under MHA)."""
    Kc16, Vc16 = _h(Kc), _h(Vc)
    x, D, h, hkv, dh = _attn_common(x, W, Kc16, n, scale, eps)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    knew = np.zeros((hkv, dh), np.uint16)
    vnew = np.zeros((hkv, dh), np.uint16)
    H, delta = _f64((h, dh)), _f64(D.d)
    lib().or_attn_gather(ctypes.byref(D), _p(x), *_attn_args(W), _p(Kc16), _p(Vc16), _p(sel),
                         ctypes.c_int(sel.size), _p(knew), _p(vnew), _p(H), _p(delta))
    return AttnOut(delta, H, knew.view(np.float16), vnew.view(np.float16))


def attn_masked(x, W, Kc, Vc, n, mask=None, scale=None, eps=1e-5):
    Kc16, Vc16 = _h(Kc), _h(Vc)
    x, D, h, hkv, dh = _attn_common(x, W, Kc16, n, scale, eps)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    knew = np.zeros((hkv, dh), np.uint16)
    vnew = np.zeros((hkv, dh), np.uint16)
    H, delta = _f64((h, dh)), _f64(D.d)
    lib().or_attn_masked(ctypes.byref(D), _p(x), *_attn_args(W), _p(Kc16), _p(Vc16), _p(m),
                         _p(knew), _p(vnew), _p(H), _p(delta))
    return AttnOut(delta, H, knew.view(np.float16), vnew.view(np.float16))


def attn_kvsel(x, W, Kc, Vc, n, kept, counts, scale=None, eps=1e-5):
    """Attention of every head over its KV head's retained positions plus the new token."""
    Kc16, Vc16 = _h(Kc), _h(Vc)
    x, D, h, hkv, dh = _attn_common(x, W, Kc16, n, scale, eps)
    kept = np.ascontiguousarray(kept, dtype=np.int32)
    counts = np.ascontiguousarray(counts, dtype=np.int32)
    knew = np.zeros((hkv, dh), np.uint16)
    vnew = np.zeros((hkv, dh), np.uint16)
    H, delta = _f64((h, dh)), _f64(D.d)
    lib().or_attn_kvsel(ctypes.byref(D), _p(x), *_attn_args(W), _p(Kc16), _p(Vc16), _p(kept),
                        ctypes.c_int(kept.shape[1]), _p(counts), _p(knew), _p(vnew), _p(H),
                        _p(delta))
    return AttnOut(delta, H, knew.view(np.float16), vnew.view(np.float16))


def attend(q, K, V, knew, vnew, scale, pos=None):
    """One query over cached rows K/V [*][dh] (positions pos, or all) plus a new key/value."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K16, V16 = _h(K), _h(V)
    dh = q.size
    cnt = K16.shape[0] if pos is None else len(pos)
    p = None if pos is None else np.ascontiguousarray(pos, dtype=np.int32)
    kn = np.ascontiguousarray(knew, dtype=np.float64)
    vn = np.ascontiguousarray(vnew, dtype=np.float64)
    out = _f64(dh)
    lib().or_attend(_p(q), ctypes.c_int(dh), _p(K16), _p(V16), _p(p), ctypes.c_int(cnt), _p(kn),
                    _p(vn), ctypes.c_double(scale), _p(out))
    return out


# --------------------------------------------------------------------------
# a8 attention-scored KV selection (ByteCross §4.1, App. A)
# --------------------------------------------------------------------------
def kv_pool(q_obs, K, n, scale=None):
    """Pooled causal attention of the observation window: [hkv][n]."""
    q16, K16 = _h(q_obs), _h(K)
    h, W, dh = q16.shape
    hkv, n_max, _ = K16.shape
    if scale is None:
        scale = 1.0 / math.sqrt(dh)
    out = _f64((hkv, n))
    lib().or_kv_pool(_p(q16), _p(K16), ctypes.c_int(h), ctypes.c_int(hkv), ctypes.c_int(dh),
                     ctypes.c_int(n), ctypes.c_int(n_max), ctypes.c_int(W), ctypes.c_double(scale),
                     _p(out))
    return out


def kv_smooth(pooled, width=7):
    pooled = np.ascontiguousarray(pooled, dtype=np.float64)
    out = np.zeros_like(pooled)
    rows = pooled.reshape(-1, pooled.shape[-1])
    o = out.reshape(-1, pooled.shape[-1])
    for r in range(rows.shape[0]):
        src = np.ascontiguousarray(rows[r])
        dst = np.zeros_like(src)
        lib().or_kv_smooth(_p(src), ctypes.c_int(src.size), ctypes.c_int(width), _p(dst))
        o[r] = dst
    return out


def kv_choose(smoothed, n_sinks, W, b):
    """Kept positions of one KV head, ascending."""
    sm = np.ascontiguousarray(smoothed, dtype=np.float64)
    n = sm.size
    kept = np.zeros(n, dtype=np.int32)
    c = lib().or_kv_choose(_p(sm), ctypes.c_int(n), ctypes.c_int(n_sinks), ctypes.c_int(W),
                           ctypes.c_int(b), _p(kept))
    return kept[:c].copy()


def kv_budget(n: int, keep: float) -> int:
    """Per-KV-head budget b = floor(n keep), sinks and window included."""
    return int(math.floor(n * keep + 1e-9))


def kv_select(q_obs, K, n, keep, n_sinks=4, width=7, scale=None):
    """All three steps for every KV head: (kept [hkv][*] list, smoothed [hkv][n])."""
    W = q_obs.shape[1]
    sm = kv_smooth(kv_pool(q_obs, K, n, scale), width)
    b = kv_budget(n, keep)
    return [kv_choose(sm[u], n_sinks, W, b) for u in range(sm.shape[0])], sm


# --------------------------------------------------------------------------
# One decode layer (Deja Vu App. C.3: y~ = y + MHA(y), y^ = y~ + MLP(y~))
# --------------------------------------------------------------------------
def layer(x, W, Kc, Vc, n, head_sel, neuron_idx, scale=None, eps=1e-5):
    """Sparse decode layer. The block outputs are rounded to fp16 where the
    library hands them on: h = fp16(x + MHA), y' = fp16(h + MLP(h))."""
    a = attn_gather(x, W, Kc, Vc, n, head_sel, scale=scale, eps=eps)
    xd = h2d(_h(x))
    hmid = round_fp16(xd + a.delta)
    m = mlp_gather(hmid, W["fc1"], W.get("b1"), W["fc2T"], W.get("b2"), neuron_idx,
                   ln_g=W.get("ln2_g"), ln_b=W.get("ln2_b"), eps=eps)
    y = round_fp16(h2d(_h(hmid)) + m)
    return y, hmid, a, m


def token_kv(x, W, hkv, dh, eps=1e-5):
    """k, v of every unit for one token (fp16 [hkv][dh] each): z = LN1(x)
    projected by W^K, W^V plus biases, rounded as the cache stores them. These
    are the rows "Deja Vu" §4.2 recomputes from a stored token embedding."""
    K0 = np.zeros((hkv, 1, dh), np.float16)
    a = attn_masked(x, W, K0, K0.copy(), 0, None, eps=eps)
    return a.knew, a.vnew


def attn_steps(ys, W, Kc, Vc, n0, sels, scale=None, eps=1e-5):
    """T decode steps of the head-sparse attention block ("Deja Vu" §2.3 Eq. 2,
    §4.2). Step t reads input ys[t] with n0 + t cached tokens and attends, for
    the units in sels[t], over positions 0..n0+t. A step computes k, v only for
    the units it selects; the units it skips keep a copy of the token's input,
    and their k, v are computed from that copy before a later step reads them.
    So every step sees, at every past position, the k, v of that position's own
    token: this function computes them directly. Returns the per-step outputs
    (AttnOut) and the completed caches K, V [hkv][n_max][dh] (fp16)."""
    K = np.array(Kc, dtype=np.float16, copy=True)
    V = np.array(Vc, dtype=np.float16, copy=True)
    hkv, dh = K.shape[0], K.shape[2]
    outs = []
    for t, (y, sel) in enumerate(zip(ys, sels)):
        n = n0 + t
        outs.append(attn_gather(y, W, K, V, n, sel, scale=scale, eps=eps))
        K[:, n], V[:, n] = token_kv(y, W, hkv, dh, eps=eps)
    return outs, K, V
