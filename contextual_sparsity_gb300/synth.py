"""Seeded synthetic inputs for the decode-step hot path.

This module holds shapes, distributions and seeds only -- none of the method's
arithmetic -- so that both the CUDA path and the CPU oracle can be fed the same
tensors. There are no trained weights or datasets: every tensor is drawn from
the distribution its workload names (OPT-shaped layers with fp16 weights
N(0, 0.02), fc1 bias N(-0.5, 0.1) so that ReLU is sparse, predictor weights
N(0, 0.05), hidden state and KV cache N(0, 1)).

Each tensor has its own generator, seeded from (seed, workload, layer, name)
through CRC32, so a tensor does not depend on which others were drawn.
"""
from __future__ import annotations

import dataclasses
import zlib

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    d: int
    h: int
    h_kv: int
    dh: int
    F: int
    r: int
    n: int
    layers: int
    keep_N: float
    keep_H: float
    B: int = 1
    keep_KV: float = 1.0
    obs_window: int = 64
    n_sinks: int = 4
    smooth: int = 7

    @property
    def head_units(self) -> int:
        """Selectable attention units: KV heads (= heads when h_kv == h)."""
        return self.h_kv


WORKLOADS = {
    # Tiny OPT-style block: d 256, 4 heads x 64, FFN 1024, rank 32, 64 cached tokens.
    "tiny": Workload("tiny", 256, 4, 4, 64, 1024, 32, 64, 1, 0.25, 0.5),
    # OPT-6.7B shape, 32 layers, KV context 512.
    "opt-6.7b": Workload("opt-6.7b", 4096, 32, 32, 128, 16384, 1000, 512, 32, 0.10, 0.5),
    # OPT-66B shape, 16 layers, KV context 2048, batch 1 or 4.
    "opt-66b": Workload("opt-66b", 9216, 72, 72, 128, 36864, 1000, 2048, 16, 0.10, 0.5),
    # OPT-175B layer shape, 24 layers (~87 GB fp16), KV context 1024.
    "opt-175b": Workload("opt-175b", 12288, 96, 96, 128, 49152, 1000, 1024, 24, 0.10, 0.5),
    # Composition: d 4096, 32 query / 8 KV heads x 128, ReLU FFN 14336, 32 layers,
    # neuron keep 50 %, all heads, attention-scored KV keep 1/8.
    "compose": Workload("compose", 4096, 32, 8, 128, 14336, 1000, 32768, 32, 0.5, 1.0,
                        keep_KV=0.125),
}


def workload(name: str, **over) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **over)


def _seed(seed: int, wl: str, layer: int, name: str) -> int:
    return zlib.crc32(f"{seed}/{wl}/{layer}/{name}".encode()) & 0x7FFFFFFF


def normal(shape, mean, std, *, seed, wl, layer, name, device="cpu", dtype=torch.float16,
           chunk=1 << 26):
    """Seeded N(mean, std) tensor, drawn in fp32 and rounded to `dtype`."""
    g = torch.Generator(device=device)
    g.manual_seed(_seed(seed, wl, layer, name))
    out = torch.empty(shape, dtype=dtype, device=device)
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        t = torch.randn(e - s, generator=g, device=device, dtype=torch.float32)
        flat[s:e] = t.mul_(std).add_(mean).to(dtype)
    return out


def layer_weights(w: Workload, layer: int, *, seed=0, device="cpu", full_bias=False):
    """Weights of one decode layer in the library's layouts.

    Wq [h dh][d], Wk / Wv [h_kv dh][d], WoT [h dh][d] (W^O transposed),
    fc1 [F][d], fc2T [F][d] (W^2 transposed), P1 [r][d], P2 [F + h_kv][r].
    Biases other than b1 and LayerNorm parameters are absent (zero / unit)
    unless full_bias, which draws all of them to exercise every bias path.
    """
    kw = dict(seed=seed, wl=w.name, layer=layer, device=device)
    W = {
        "Wq": normal((w.h * w.dh, w.d), 0.0, 0.02, name="Wq", **kw),
        "Wk": normal((w.h_kv * w.dh, w.d), 0.0, 0.02, name="Wk", **kw),
        "Wv": normal((w.h_kv * w.dh, w.d), 0.0, 0.02, name="Wv", **kw),
        "WoT": normal((w.h * w.dh, w.d), 0.0, 0.02, name="WoT", **kw),
        "fc1": normal((w.F, w.d), 0.0, 0.02, name="fc1", **kw),
        "b1": normal((w.F,), -0.5, 0.1, name="b1", **kw),
        "fc2T": normal((w.F, w.d), 0.0, 0.02, name="fc2T", **kw),
        "P1": normal((w.r, w.d), 0.0, 0.05, name="P1", **kw),
        "P2": normal((w.F + w.head_units, w.r), 0.0, 0.05, name="P2", **kw),
    }
    if full_bias:
        W["bq"] = normal((w.h * w.dh,), 0.0, 0.1, name="bq", **kw)
        W["bk"] = normal((w.h_kv * w.dh,), 0.0, 0.1, name="bk", **kw)
        W["bv"] = normal((w.h_kv * w.dh,), 0.0, 0.1, name="bv", **kw)
        W["bo"] = normal((w.d,), 0.0, 0.1, name="bo", **kw)
        W["b2"] = normal((w.d,), 0.0, 0.1, name="b2", **kw)
        W["ln1_g"] = normal((w.d,), 1.0, 0.1, name="ln1_g", **kw)
        W["ln1_b"] = normal((w.d,), 0.0, 0.1, name="ln1_b", **kw)
        W["ln2_g"] = normal((w.d,), 1.0, 0.1, name="ln2_g", **kw)
        W["ln2_b"] = normal((w.d,), 0.0, 0.1, name="ln2_b", **kw)
    return W


def hidden(w: Workload, *, seed=0, device="cpu", B=None, name="x", layer=0):
    """Layer input y [B][d] ~ N(0, 1)."""
    return normal((B or w.B, w.d), 0.0, 1.0, seed=seed, wl=w.name, layer=layer, name=name,
                  device=device)


def kv_cache(w: Workload, layer: int, n_max: int, *, seed=0, device="cpu", B=None):
    """K and V caches [B][h_kv][n_max][dh] ~ N(0, 1) (every slot filled)."""
    shape = (B or w.B, w.h_kv, n_max, w.dh)
    kw = dict(seed=seed, wl=w.name, layer=layer, device=device)
    return normal(shape, 0.0, 1.0, name="K", **kw), normal(shape, 0.0, 1.0, name="V", **kw)


def obs_queries(w: Workload, layer: int, *, seed=0, device="cpu"):
    """Projected queries of the last obs_window prompt tokens [h][W][dh] ~ N(0, 1)."""
    return normal((w.h, w.obs_window, w.dh), 0.0, 1.0, seed=seed, wl=w.name, layer=layer,
                  name="q_obs", device=device)
