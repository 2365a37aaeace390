"""Decode-step byte account (test infrastructure; pure Python closed forms).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources:
* "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time", §2.2
  Table 2: per-layer attention and MLP FLOPs and I/O of OPT-175B (d = 12288);
  an OPT layer holds 4 d^2 attention and 8 d^2 MLP parameters (FFN 4d).
* "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM Decoding",
  §3.1 (a step reads the projection weights once plus a KV term that grows with
  context; other reads: LM head, one embedding row, norm weights), §3.2
  (projection keep r_P saves context-independent bytes, KV keep r_KV saves
  bytes that grow with n), §3.3 (the crossover n* is the context where both
  savings are equal; ideal speedup bounds = dense bytes / remaining bytes),
  App. C (crossover values).
"""
from __future__ import annotations

ELT = 2  # fp16 bytes


# --------------------------------------------------------------------------
# Deja Vu per-layer account (OPT, one token)
# --------------------------------------------------------------------------
def opt_attention_params(d: int) -> int:
    """W^Q, W^K, W^V, W^O: four d x d matrices."""
    return 4 * d * d


def opt_mlp_params(d: int) -> int:
    """W^1, W^2 in R^{d x 4d} (Deja Vu §2.3)."""
    return 2 * d * 4 * d


def table2_io_gib(d: int = 12288):
    """Per-layer I/O in GiB of the attention and MLP blocks (fp16)."""
    return (opt_attention_params(d) * ELT / 2**30, opt_mlp_params(d) * ELT / 2**30)


def table2_gflops(d: int = 12288):
    """Per-layer GFLOPs of one token: 2 FLOPs per weight."""
    return (2 * opt_attention_params(d) / 1e9, 2 * opt_mlp_params(d) / 1e9)


# --------------------------------------------------------------------------
# Selected bytes of one sparse decode layer
# --------------------------------------------------------------------------
def selected_bytes(d, h, h_kv, dh, F, n, k_N, k_H):
    """Bytes a sparse decode layer must move (batch 1).

    k_N selected neurons: one fc1 row and one fc2^T row of d fp16 each.
    k_H selected units (KV heads and their h/h_kv query heads): the query and
    output slices (h/h_kv * dh rows each), the key and value slices (dh rows
    each), and the K and V rows of the n cached tokens plus the new token.
    """
    G = h // h_kv
    mlp = 2 * k_N * d * ELT
    attn_w = k_H * (2 * G * dh + 2 * dh) * d * ELT
    kv = k_H * 2 * dh * (n + 1) * ELT
    return mlp + attn_w + kv


def predictor_bytes(d, r, rows):
    """P1 [r][d] plus the P2 rows that are scored: 2 r (d + rows); 0 if none."""
    return 0 if rows == 0 else ELT * r * (d + rows)


def dense_bytes(d, h, h_kv, dh, F, n):
    return selected_bytes(d, h, h_kv, dh, F, n, F, h_kv)


# --------------------------------------------------------------------------
# ByteCross crossover and bounds
# --------------------------------------------------------------------------
def crossover(w_proj_bytes: float, kv_bytes_per_token: float, r_P: float, r_KV: float) -> float:
    """n* where the projection saving (1-r_P) W equals the KV saving (1-r_KV) b n."""
    return (1.0 - r_P) * w_proj_bytes / ((1.0 - r_KV) * kv_bytes_per_token)


def llama_like_layer_bytes(d, h, h_kv, dh, ffn, gated=True):
    """Projection bytes of one Llama-style layer: q, o (d x h dh), k, v (d x h_kv dh),
    and three (gated) or two feed-forward matrices d x ffn."""
    attn = d * h * dh * 2 + d * h_kv * dh * 2
    ff = (3 if gated else 2) * d * ffn
    return ELT * attn, ELT * ff


def kv_bytes_per_token(h_kv, dh, layers=1):
    return layers * 2 * h_kv * dh * ELT


def step_bytes(L, w_layer, kv_tok_layer, n, lm_head=0, emb_row=0, norms=0):
    """Total bytes of one decode step (ByteCross §3.1)."""
    return L * w_layer + L * kv_tok_layer * n + lm_head + emb_row + norms


def bound(total, saved):
    return total / (total - saved)
