"""Byte account pinned to the values printed on the pages (tests/golden)."""
import json
import os

import pytest

from oracle import byte_account as ba

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def test_dejavu_table2():
    g = _load("dejavu_table2.json")
    att_gib, mlp_gib = ba.table2_io_gib(g["d"])
    att_gf, mlp_gf = ba.table2_gflops(g["d"])
    # I/O is printed cut to two decimals (1.125 -> 1.12, 2.25 -> 2.25)
    assert int(att_gib * 100) / 100 == g["attention"]["io_gb"]
    assert int(mlp_gib * 100) / 100 == g["mlp"]["io_gb"]
    assert att_gib == 1.125 and mlp_gib == 2.25
    assert abs(att_gf - g["attention"]["gflops"]) < 0.01
    assert abs(mlp_gf - g["mlp"]["gflops"]) < 0.01


def _model_bytes(m):
    attn, ff = ba.llama_like_layer_bytes(m["d"], m["h"], m["h_kv"], m["dh"], m["ffn"])
    return attn, ff, ba.kv_bytes_per_token(m["h_kv"], m["dh"])


def test_bytecross_layer_bytes():
    g = _load("bytecross_crossovers.json")
    m = g["models"][g["layer_bytes"]["model"]]
    attn, ff, kv = _model_bytes(m)
    assert round((attn + ff) / 1e6) == g["layer_bytes"]["proj_mb"]
    assert kv == g["layer_bytes"]["kv_bytes_per_token"]


@pytest.mark.parametrize("i", range(8))
def test_bytecross_crossovers(i):
    g = _load("bytecross_crossovers.json")
    c = g["crossovers"][i]
    attn, ff, kv = _model_bytes(g["models"][c["model"]])
    w = attn + ff if c["scope"] == "all" else ff
    assert round(ba.crossover(w, kv, c["r_P"], c["r_KV"])) == c["n_star"]


def test_bytecross_window_bound_at_128k():
    g = _load("bytecross_crossovers.json")
    wb = g["window_bound"]
    m = g["models"][wb["model"]]
    attn, ff, kv = _model_bytes(m)
    L = m["layers"]
    lm_head = m["vocab"] * m["d"] * ba.ELT
    emb = m["d"] * ba.ELT
    norms = (2 * L + 1) * m["d"] * ba.ELT
    total = ba.step_bytes(L, attn + ff, kv, wb["n"], lm_head, emb, norms)
    saved = (1 - wb["r_KV"]) * L * kv * wb["n"]
    assert round(ba.bound(total, saved), 2) == wb["bound"]


def test_opt_selected_bytes_matches_closed_form():
    # For MHA OPT (F = 4d, h dh = d) the selected bytes are
    # 2 (8 d^2 k_N/F + 4 d^2 k_H/h) + 4 d (n+1) k_H/h.
    for d, h, F, n, kN, kH in [(12288, 96, 49152, 1024, 4915, 48), (4096, 32, 16384, 512, 1638, 16),
                               (9216, 72, 36864, 2048, 3686, 36)]:
        got = ba.selected_bytes(d, h, h, d // h, F, n, kN, kH)
        ref = 2 * (8 * d * d * kN / F + 4 * d * d * kH / h) + 4 * d * (n + 1) * kH / h
        assert abs(got - ref) < 1e-6
    # dense = Table 2's 8 d^2 + 16 d^2 plus the cache of n + 1 tokens
    assert ba.dense_bytes(12288, 96, 96, 128, 49152, 1024) == 24 * 12288**2 + 4 * 12288 * 1025


def test_composition_crossover_is_32768():
    # d 4096, 32/8 heads x 128, two-matrix ReLU FFN 14336: n* with neuron keep
    # 1/2 (MLP weights only) and KV keep 1/8
    attn, ff = ba.llama_like_layer_bytes(4096, 32, 8, 128, 14336, gated=False)
    assert ba.crossover(ff, ba.kv_bytes_per_token(8, 128), 0.5, 0.125) == 32768
