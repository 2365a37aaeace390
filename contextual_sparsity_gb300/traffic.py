"""Algorithmic bytes of the decode step: what each kernel must move.

Used by the benchmark for achieved GB/s. Counts follow the sparsified blocks
of "Deja Vu" §2.3 (Eq. 1: one fc1 row and one fc2^T row per selected neuron;
Eq. 2: the query, key, value and output slices of each selected head plus its
KV-cache rows) and the byte account of "Where Activation Sparsity and KV-Cache
Sparsity Cross in LLM Decoding" §3.1-3.2 (projection bytes x keep + KV bytes x
KV keep). fp16 everywhere (2 bytes per element).
"""
from __future__ import annotations

import math

E = 2


def k_of(keep: float, N: int) -> int:
    return N if keep >= 1.0 else max(1, int(math.floor(keep * N + 1e-9)))


def qkv_bytes(d, G, dh, units):
    """Weights of the QKV gather-GEMV: (G + 2) dh rows of d per unit."""
    return units * (G + 2) * dh * d * E


def wo_bytes(d, G, dh, units):
    return units * G * dh * d * E


def mlp_bytes(d, neurons):
    return 2 * neurons * d * E


def kv_bytes(dh, units, keys):
    """K and V rows of the attended keys (the new token's write included)."""
    return units * 2 * dh * keys * E


def p1_bytes(d, r):
    """The predictor's first layer P1 [r][d]."""
    return r * d * E


def pred_bytes(d, r, rows):
    return 0 if rows == 0 else r * (d + rows) * E


def layer_bytes(w, keep_N=None, keep_H=None, keys=None, union=None):
    """(selected bytes, predictor bytes) of one decode layer of workload w.

    At batch B > 1 every row is computed over the union of the B sets
    ("Deja Vu" App. C.1): `union` = (|U_N|, |U_H|) replaces k_N, k_H for the
    weight rows, and each sequence reads its own cache rows of the union's
    units."""
    keep_N = w.keep_N if keep_N is None else keep_N
    keep_H = w.keep_H if keep_H is None else keep_H
    G = w.h // w.h_kv
    kN = k_of(keep_N, w.F)
    kH = k_of(keep_H, w.h_kv)
    if union is not None:
        kN, kH = union
    keys = (w.n + 1) if keys is None else keys
    sel = (qkv_bytes(w.d, G, w.dh, kH) + wo_bytes(w.d, G, w.dh, kH) + mlp_bytes(w.d, kN)
           + w.B * kv_bytes(w.dh, kH, keys))
    rows = (w.F if keep_N < 1 else 0) + (w.h_kv if keep_H < 1 else 0)
    return sel, pred_bytes(w.d, w.r, rows)


def w4_row_bytes(d):
    """Bytes of one packed 4-bit row: d/2 of codes, d/64 of fp16 group scales,
    padded to a multiple of 16."""
    return (d // 2 + d // 64 + 15) // 16 * 16


def layer_bytes_w4(w, keep_N=None, keep_H=None, keys=None):
    """Selected bytes of one decode layer with 4-bit projection and MLP rows
    (the KV cache stays fp16): (2G + 2) d_h packed rows per selected unit, two
    per selected neuron, plus the K, V rows of the attended keys."""
    keep_N = w.keep_N if keep_N is None else keep_N
    keep_H = w.keep_H if keep_H is None else keep_H
    G = w.h // w.h_kv
    kN, kH = k_of(keep_N, w.F), k_of(keep_H, w.h_kv)
    keys = (w.n + 1) if keys is None else keys
    return ((kH * (2 * G + 2) * w.dh + 2 * kN) * w4_row_bytes(w.d)
            + w.B * kv_bytes(w.dh, kH, keys))
