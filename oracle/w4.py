"""4-bit weights with 16-bit activations (W4A16) for the sparse MLP
(test infrastructure; numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

"Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time", §5.2 and
Table 7, combine contextual sparsity with 4-bit weight quantization and 16-bit
activations; the page names no quantization format. The format here is this
project's own choice, written out as its definition:

* groups of G = 128 consecutive columns of a weight row;
* scale s = fp16(max_i |w_i| / 7) per group (the division in fp32, IEEE
  round-to-nearest, then rounded to fp16 to nearest even);
* code q_i = clamp(rint(w_i / s), -8, 7), the division in fp32 and rint
  rounding half to even; a group of zeros gets s = 0 and q = 0;
* dequantized weight w'_i = q_i s (exact in fp64).

Packed row (the library's layout): d/2 bytes of codes, byte i holding columns
2i (low nibble) and 2i + 1 (high nibble) as q + 8 in 0..15, then the d/G
scales as fp16, then zero bytes up to a multiple of 16 (every row then starts
on a 16-byte boundary).

The MLP is "Deja Vu" Eq. 1 over the selected neurons S with the dequantized
weights: a_j = max(0, W1'_j . LN2(x) + b1_j), out = sum_j a_j W2'_j + b2,
computed in fp64.
"""
from __future__ import annotations

import numpy as np

from . import layernorm

GROUP = 128


def quantize(W16):
    """fp16 rows [rows][d] -> (codes int8 [rows][d], scales fp16 [rows][d/G])."""
    W16 = np.ascontiguousarray(W16, dtype=np.float16)
    rows, d = W16.shape
    assert d % GROUP == 0
    W = W16.astype(np.float32).reshape(rows, d // GROUP, GROUP)
    amax = np.abs(W).max(axis=2)
    s16 = (amax / np.float32(7.0)).astype(np.float16)
    s32 = s16.astype(np.float32)
    q = np.zeros_like(W)
    nz = s32 > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = W / np.where(nz, s32, np.float32(1.0))[..., None]
    q = np.where(nz[..., None], np.rint(r), np.float32(0.0))
    q = np.clip(q, -8, 7).astype(np.int8).reshape(rows, d)
    return q, s16


def dequantize(q, s16):
    """w' = q s in fp64, [rows][d]."""
    rows, d = q.shape
    return (q.reshape(rows, d // GROUP, GROUP).astype(np.float64)
            * s16.astype(np.float64)[..., None]).reshape(rows, d)


def row_bytes(d):
    return (d // 2 + d // 64 + 15) // 16 * 16


def pack(q, s16):
    """Packed rows (uint8 [rows][row_bytes(d)]) in the library's layout."""
    rows, d = q.shape
    u = (q.astype(np.int16) + 8).astype(np.uint8)
    codes = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    scales = np.ascontiguousarray(s16, dtype=np.float16).view(np.uint8).reshape(rows, -1)
    pad = np.zeros((rows, row_bytes(d) - d // 2 - d // 64), np.uint8)
    return np.concatenate([codes, scales, pad], axis=1)


def unpack(rows_u8, d):
    """Inverse of pack: (codes int8 [rows][d], scales fp16 [rows][d/G])."""
    rows_u8 = np.ascontiguousarray(rows_u8, dtype=np.uint8)
    rows = rows_u8.shape[0]
    codes = rows_u8[:, : d // 2]
    q = np.empty((rows, d), np.int8)
    q[:, 0::2] = (codes & 0xF).astype(np.int8) - 8
    q[:, 1::2] = (codes >> 4).astype(np.int8) - 8
    s16 = np.ascontiguousarray(rows_u8[:, d // 2: d // 2 + d // 64]).view(np.float16)
    s16 = s16.reshape(rows, d // GROUP)
    return q, s16


def mlp(x, fc1_q, fc1_s, b1, fc2T_q, fc2T_s, b2, idx, ln_g=None, ln_b=None, eps=1e-5):
    """Sparse MLP block output (residual excluded) with dequantized weights."""
    z = layernorm(x, ln_g, ln_b, eps)
    idx = np.asarray(idx, dtype=np.int64)
    W1 = dequantize(fc1_q[idx], fc1_s[idx])
    W2 = dequantize(fc2T_q[idx], fc2T_s[idx])
    pre = W1 @ z
    if b1 is not None:
        pre = pre + np.asarray(b1, dtype=np.float16).astype(np.float64)[idx]
    a = np.maximum(pre, 0.0)
    out = a @ W2
    if b2 is not None:
        out = out + np.asarray(b2, dtype=np.float16).astype(np.float64)
    return out


def attn(x, W, Kc, Vc, n, sel, scale=None, eps=1e-5):
    """Sparse MHA block output (residual excluded) of "Deja Vu" Eq. 2 with
    dequantized projection weights. W holds the packed-row codes and scales
    as (q, s) pairs under "Wq", "Wk", "Wv", "WoT", and fp16 biases / LN1
    parameters under their usual names. Kc, Vc [hkv][n_max][dh] fp16 hold
    positions 0..n-1; the new token's k, v are rounded to fp16 as the cache
    stores them and attended as position n. Returns (delta [d], knew, vnew
    [hkv][dh] fp16 for the selected units, zeros elsewhere)."""
    z = layernorm(x, W.get("ln1_g"), W.get("ln1_b"), eps)
    hkv, _, dh = Kc.shape
    Wq = dequantize(*W["Wq"])
    h = Wq.shape[0] // dh
    G = h // hkv
    scale = 1.0 / np.sqrt(dh) if scale is None else scale

    def proj(name, rows, bias):
        out = dequantize(*W[name])[rows] @ z
        if W.get(bias) is not None:
            out = out + np.asarray(W[bias], np.float16).astype(np.float64)[rows]
        return out

    WoT = dequantize(*W["WoT"])
    d = WoT.shape[1]
    delta = np.zeros(d)
    if W.get("bo") is not None:
        delta += np.asarray(W["bo"], np.float16).astype(np.float64)
    knew = np.zeros((hkv, dh), np.float16)
    vnew = np.zeros((hkv, dh), np.float16)
    for u in sel:
        r = np.arange(u * dh, (u + 1) * dh)
        knew[u] = proj("Wk", r, "bk").astype(np.float16)
        vnew[u] = proj("Wv", r, "bv").astype(np.float16)
        Ku = np.concatenate([np.asarray(Kc[u, :n], np.float16), knew[u][None]]).astype(np.float64)
        Vu = np.concatenate([np.asarray(Vc[u, :n], np.float16), vnew[u][None]]).astype(np.float64)
        for g in range(G):
            j = u * G + g
            q = proj("Wq", np.arange(j * dh, (j + 1) * dh), "bq") * scale
            s = Ku @ q
            p = np.exp(s - s.max())
            H = (p / p.sum()) @ Vu
            delta += H @ WoT[j * dh:(j + 1) * dh]
    return delta, knew, vnew


def layer(x, W, Kc, Vc, n, head_sel, neuron_idx, scale=None, eps=1e-5):
    """A decode layer with 4-bit projection and MLP weights: h = fp16(x + MHA),
    y' = fp16(h + MLP(h)) (the fp16 points of the library)."""
    a, _, _ = attn(x, W, Kc, Vc, n, head_sel, scale=scale, eps=eps)
    xd = np.asarray(x, np.float16).astype(np.float64)
    hmid = (xd + a).astype(np.float16)
    m = mlp(hmid, *W["fc1"], W.get("b1"), *W["fc2T"], W.get("b2"), neuron_idx,
            W.get("ln2_g"), W.get("ln2_b"), eps)
    return (hmid.astype(np.float64) + m).astype(np.float16), hmid
