"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory) and runs the pin suite against that copy: the suite
has to fail. The real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "unbiased_variance": ("var /= d;", "var /= (d - 1);"),
    "no_mean_subtraction": ("z[i] = (H(x, i) - mean) * inv", "z[i] = H(x, i) * inv"),
    "dropped_b1": ("double a = HOPT(b1, j, 0.0);", "double a = 0.0;"),
    "no_relu": ("if (a < 0.0) a = 0.0;", ""),
    "fc2_wrong_index": ("fc2T + (size_t)j * d;", "fc2T + (size_t)t * d;"),
    "dropped_new_token": ("for (int c = 0; c < dh; ++c) Hout[c] += sc[cnt] * vnew[c];", ""),
    "dropped_scale": ("sc[t] = s * scale;", "sc[t] = s;"),
    "gqa_interleaved": ("int j = u * G + g;", "int j = g * D->hkv + u;"),
    "wo_transposed": ("WoT + ((size_t)j * D->dh + c) * D->d", "WoT + ((size_t)c * D->h + j) * D->d"),
    "pool_unnormalised": ("pooled[(size_t)u * n + p] += sc[p] / Z;", "pooled[(size_t)u * n + p] += sc[p];"),
    "pool_not_causal": ("int pt = n - W + t;", "int pt = n - 1;"),
    "relu_always": ("u[j] = (relu && acc < 0.0) ? 0.0 : acc;", "u[j] = (acc < 0.0) ? 0.0 : acc;"),
    "ties_to_higher": ("return (x->i < y->i) ? -1 : (x->i > y->i);",
                       "return (x->i > y->i) ? -1 : (x->i < y->i);"),
    "window_off_by_one": ("if (p < n_sinks || p >= n - W) {", "if (p < n_sinks || p > n - W) {"),
    "round_half_away": ("double r = nearbyint(a / q);", "double r = round(a / q);"),
    "v_new_unrounded": ("vd[c] = or_h2d(vnew16[(size_t)u * dh + c]);", ""),
    "kvsel_table_stride_is_count": ("kept + (size_t)u * kept_ld, cnt[u]", "kept + (size_t)u * cnt[u], cnt[u]"),
    "kvsel_count_of_first_head": ("kept + (size_t)u * kept_ld, cnt[u], u,", "kept + (size_t)u * kept_ld, cnt[0], u,"),
    "predictor_transposed_p2": ("const uint16_t* row = P2 + (size_t)n * r;\n    for (int j = 0; j < r; ++j) acc += H(row, j) * u[j];",
                                "for (int j = 0; j < r; ++j) acc += H(P2, (size_t)j * N + n) * u[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "dv_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "oracle" / "dv_oracle.c").write_text(src.replace(old, new))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


GATE_MUTANTS = {
    "gate_no_new_token": ("kv = B * uH * 2 * dh * (tokens + 1) * ELT", "kv = B * uH * 2 * dh * tokens * ELT"),
    "gate_kv_shared_by_batch": ("kv = B * uH * 2 * dh", "kv = uH * 2 * dh"),
    "gate_no_predictor": ("return weights + kv + pred", "return weights + kv"),
    "gate_union_additive": ("return N * (1.0 - (1.0 - k / N) ** B)", "return min(N, k * B)"),
    "gate_keep_unfloored": ("kN, kH = keep_count(keep_N, F), keep_count(keep_H, h_kv)",
                            "kN, kH = keep_N * F, keep_H * h_kv"),
    "gate_budget_ignored": ("tokens = min(float(n), kv_budget) if kv_budget > 0 else keep_KV * n",
                            "tokens = keep_KV * n"),
    "gate_dense_linear": ("return math.exp(lys[i] + t * (lys[i + 1] - lys[i]))",
                          "return ys[i] + t * (ys[i + 1] - ys[i])"),
    "gate_select_every_step": ("t += linear(n, ctx, select_us) / steps", "t += linear(n, ctx, select_us)"),
    "gate_cost_unscaled": ("measured_us[DENSE][i] * bytes_at(m, c) / bytes_at(DENSE, c)",
                           "measured_us[DENSE][i]"),
    "gate_ties_to_higher": ("key=lambda m: (ts[m], m)", "key=lambda m: (ts[m], -m)"),
}


@pytest.mark.parametrize("name", sorted(GATE_MUTANTS))
def test_gate_pins_catch_mutant(name, tmp_path):
    old, new = GATE_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "gate.py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "oracle" / "gate.py").write_text(src.replace(old, new))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_gate_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_gate_pins.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


PY_MUTANTS = {
    "steps_position_off_by_one": ("K[:, n], V[:, n] = token_kv(y, W, hkv, dh, eps=eps)",
                                  "K[:, n - 1], V[:, n - 1] = token_kv(y, W, hkv, dh, eps=eps)"),
    "steps_skipped_units_left_stale": ("K[:, n], V[:, n] = token_kv(y, W, hkv, dh, eps=eps)",
                                       "K[sel, n], V[sel, n] = outs[-1].knew[sel], outs[-1].vnew[sel]"),
    "token_kv_no_layernorm": ("a = attn_masked(x, W, K0, K0.copy(), 0, None, eps=eps)",
                              "a = attn_masked(x, W, K0, K0.copy(), 0, None, eps=1e30)"),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_multistep_pins_catch_mutant(name, tmp_path):
    old, new = PY_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "oracle" / "__init__.py").write_text(src.replace(old, new))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "-k", "token_kv or attn_steps"],
                       cwd=tmp_path, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


W4_MUTANTS = {
    "w4_scale_over_8": ("amax / np.float32(7.0)", "amax / np.float32(8.0)"),
    "w4_round_half_up": ("np.rint(r)", "np.floor(r + np.float32(0.5))"),
    "w4_scale_unrounded": ("s32 = s16.astype(np.float32)", "s32 = amax / np.float32(7.0)"),
    "w4_nibbles_swapped": ("(u[:, 0::2] | (u[:, 1::2] << 4))", "(u[:, 1::2] | (u[:, 0::2] << 4))"),
    "w4_dequant_no_scale": ("* s16.astype(np.float64)[..., None]).reshape(rows, d)",
                            "* 1.0).reshape(rows, d)"),
    "w4_mlp_no_relu": ("a = np.maximum(pre, 0.0)", "a = pre"),
    "w4_mlp_no_b1": ("pre = pre + np.asarray(b1", "pre = pre + 0 * np.asarray(b1"),
    "w4_attn_no_scale": ('np.arange(j * dh, (j + 1) * dh), "bq") * scale',
                         'np.arange(j * dh, (j + 1) * dh), "bq")'),
    "w4_attn_gqa_interleaved": ("j = u * G + g", "j = g * hkv + u"),
    "w4_attn_cache_slot_for_new_token": (
        "Ku = np.concatenate([np.asarray(Kc[u, :n], np.float16), knew[u][None]])",
        "Ku = np.asarray(Kc[u, :n + 1], np.float16)"),
}


@pytest.mark.parametrize("name", sorted(W4_MUTANTS))
def test_w4_pins_catch_mutant(name, tmp_path):
    old, new = W4_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "w4.py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "oracle" / "w4.py").write_text(src.replace(old, new))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_w4_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_w4_pins.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


LAYER_MUTANTS = {
    "layer_mlp_reads_x": ("m = mlp_gather(hmid, W[\"fc1\"]", "m = mlp_gather(x, W[\"fc1\"]"),
    "layer_output_adds_unrounded_h": ("y = round_fp16(h2d(_h(hmid)) + m)",
                                      "y = round_fp16(xd + a.delta + m)"),
    "layer_output_unrounded": ("y = round_fp16(h2d(_h(hmid)) + m)", "y = h2d(_h(hmid)) + m"),
    "layer_attention_residual_dropped": ("hmid = round_fp16(xd + a.delta)",
                                         "hmid = round_fp16(a.delta)"),
}


@pytest.mark.parametrize("name", sorted(LAYER_MUTANTS))
def test_layer_pins_catch_mutant(name, tmp_path):
    old, new = LAYER_MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    (tmp_path / "oracle" / "__init__.py").write_text(src.replace(old, new))
    os.makedirs(tmp_path / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tmp_path / "tests" / "golden")
    env = dict(os.environ, PYTHONPATH=str(tmp_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py", "-k", "test_layer_"],
                       cwd=tmp_path, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
