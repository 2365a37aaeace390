"""Helpers of the GPU parity tests: building the library, moving seeded inputs
between torch and numpy, and the error measures the tests use."""
import numpy as np
import torch

from contextual_sparsity_gb300 import build, dv

# Tolerance on block outputs: max_i |gpu_i - ref_i| / max_i |ref_i| (fp16
# weights, fp32 accumulation against the fp64 oracle).
TOL = 2e-3


def setup_lib():
    build.build()
    return dv.lib()


def np16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy()


def npf(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def rel_err(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def to_dev(W: dict, device="cuda") -> dict:
    return {k: v.to(device) for k, v in W.items()}


def host(W: dict) -> dict:
    return {k: np16(v) for k, v in W.items()}


def check_sets(gpu_idx, ref_scores, k, rtol=1e-6):
    """Index-set parity: same size, and every index in the symmetric difference
    has a reference score within rtol (relative) of the k-th reference score."""
    gpu = set(int(i) for i in np.asarray(gpu_idx).ravel())
    order = np.argsort(-ref_scores, kind="stable")
    ref = set(int(i) for i in order[:k])
    assert len(gpu) == k
    sk = ref_scores[order[k - 1]]
    for i in gpu ^ ref:
        assert abs(ref_scores[i] - sk) <= rtol * abs(sk), (i, ref_scores[i], sk)
    return len(gpu ^ ref)


def check_kv_kept(gpu_kept, ref_kept, ref_scores, gpu_scores, forced):
    """KV-selection parity for one KV head: the GPU keeps as many positions as
    the oracle, every forced position (sinks and window) is kept, and a
    position kept by one side only must score, on the oracle's smoothed
    scores, within 2 eps of the oracle's cut score (the lowest score it keeps
    beyond the forced set), eps the largest GPU-vs-oracle difference of the
    smoothed scores of this head: a swap is only accepted between positions
    that the GPU's own rounding could have ordered either way."""
    gpu, ref = set(int(p) for p in gpu_kept), set(int(p) for p in ref_kept)
    assert len(gpu) == len(ref)
    assert set(forced) <= gpu and set(forced) <= ref
    diff = gpu ^ ref
    if not diff:
        return 0
    eps = float(np.max(np.abs(np.asarray(gpu_scores, float) - np.asarray(ref_scores, float))))
    cut = min(ref_scores[p] for p in ref - set(forced))
    for p in diff:
        assert abs(ref_scores[p] - cut) <= 2 * eps + 1e-6 * abs(cut), (p, ref_scores[p], cut, eps)
    return len(diff)
