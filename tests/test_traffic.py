"""The benchmark's byte counts agree with the oracle's byte account."""
import pytest

from contextual_sparsity_gb300 import synth, traffic
from oracle import byte_account as ba


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
@pytest.mark.parametrize("kn,kh", [(None, None), (0.25, 1.0), (1.0, 0.25), (0.5, 0.5)])
def test_layer_bytes_match_oracle(name, kn, kh):
    w = synth.workload(name)
    sel, pred = traffic.layer_bytes(w, kn, kh)
    kn = w.keep_N if kn is None else kn
    kh = w.keep_H if kh is None else kh
    k_N = w.F if kn >= 1 else max(1, int(kn * w.F + 1e-9))
    k_H = w.h_kv if kh >= 1 else max(1, int(kh * w.h_kv + 1e-9))
    assert sel == ba.selected_bytes(w.d, w.h, w.h_kv, w.dh, w.F, w.n, k_N, k_H)
    rows = (w.F if kn < 1 else 0) + (w.h_kv if kh < 1 else 0)
    assert pred == ba.predictor_bytes(w.d, w.r, rows)


def test_opt175b_headline_bytes():
    # 175B, 10 % neurons, 50 % heads, n = 1024: 870.8 MB selected, 123.1 MB predictor
    sel, pred = traffic.layer_bytes(synth.workload("opt-175b"))
    assert round(sel / 1e6, 1) == 870.8
    assert round(pred / 1e6, 1) == 123.1


def test_w4_layer_bytes():
    # opt-175b: 48 units x 4 x 128 packed rows + 2 x 4915 packed rows (6336 bytes each,
    # the oracle's packed-row size) + the fp16 K, V rows of 1025 keys
    from oracle import w4 as ow4
    w = synth.workload("opt-175b")
    assert traffic.w4_row_bytes(w.d) == ow4.row_bytes(w.d) == 6336
    want = (48 * 4 * 128 + 2 * 4915) * 6336 + 48 * 2 * 128 * 1025 * 2
    assert traffic.layer_bytes_w4(w) == want == 243186816
    assert traffic.layer_bytes_w4(w, keep_N=0.25) == (48 * 4 * 128 + 2 * 12288) * 6336 + 48 * 2 * 128 * 1025 * 2
