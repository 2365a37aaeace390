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
