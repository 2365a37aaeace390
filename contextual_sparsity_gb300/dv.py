"""Python binding of libdv.so: the same entry points, argument marshalling only.

Every function takes torch CUDA tensors, passes their device pointers and the
current CUDA stream to the C ABI (``include/dv.h``) and raises ``DvError`` on a
negative status. All arithmetic happens in the library's CUDA kernels; there is
no fallback: if ``libdv.so`` is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdv.so")

DV_OK = 0
DV_ERR_NULL, DV_ERR_ALIGN, DV_ERR_DIMS, DV_ERR_KEEP = -1, -2, -3, -4
DV_ERR_K, DV_ERR_WORKSPACE, DV_ERR_LAUNCH, DV_ERR_UNSUPPORTED = -5, -6, -7, -8
DV_DEV_BAD_INDEX, DV_DEV_TIMEOUT, DV_DEV_NONFINITE = 1, 2, 4

DV_PRED_RELU = 1 << 0
DV_SKIP_INACTIVE = 1 << 1
DV_LOOKAHEAD = 1 << 2
DV_SYNC_PREDICT = 1 << 3
DV_KV_RESELECT = 1 << 4
DV_KV_DENSE = 1 << 5
DV_KV_RETAINED = 1 << 6
DV_KV_ADVANCE = 1 << 7
DV_JOIN = 1 << 8
DV_NO_RESIDUAL = 1 << 9
DV_KV_FILL = 1 << 10
DV_W4 = 1 << 11

_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


class DvError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class Dims(ctypes.Structure):
    _fields_ = [("d", _i), ("h", _i), ("h_kv", _i), ("d_h", _i), ("F", _i), ("r", _i),
                ("n_max", _i), ("ln_eps", _f)]


class Keep(ctypes.Structure):
    _fields_ = [("neuron", _f), ("head", _f), ("kv", _f)]


_W_FIELDS = ["ln1_g", "ln1_b", "Wq", "bq", "Wk", "bk", "Wv", "bv", "WoT", "bo", "ln2_g", "ln2_b",
             "fc1", "b1", "fc2T", "b2", "P1", "P2"]


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, _p) for n in _W_FIELDS]


class KvCache(ctypes.Structure):
    _fields_ = [("K", _p), ("V", _p), ("y_side", _p), ("kv_missing", _p), ("Kr", _p), ("Vr", _p),
                ("kept_pos", _p), ("kept_count", _p), ("b_max", _i)]


class Sets(ctypes.Structure):
    _fields_ = [("idx_N", _p), ("idx_H", _p), ("uN", _p), ("uH", _p), ("ucnt", _p),
                ("scores", _p)]


MODE_DENSE, MODE_ACT, MODE_KV, MODE_COMPOSED = 0, 1, 2, 3
MODES = ("dense", "act", "kv", "composed")
PLAN_MAX_CTX = 16
_d = ctypes.c_double


class Request(ctypes.Structure):
    _fields_ = [("B", _i), ("steps", _i), ("union_N", _i), ("union_H", _i), ("kv_budget", _i),
                ("modes", ctypes.c_uint)]


class CostModel(ctypes.Structure):
    _fields_ = [("n_ctx", _i), ("ctx", _d * PLAN_MAX_CTX), ("dense_us", _d * PLAN_MAX_CTX),
                ("cost_us", (_d * PLAN_MAX_CTX) * 4), ("select_us", _d * PLAN_MAX_CTX)]


class Plan(ctypes.Structure):
    _fields_ = [("bytes", _d * 4), ("us", _d * 4), ("choice", _i)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libdv.so not built ({LIB_PATH}); run contextual_sparsity_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        L.dv_version.restype = _i
        L.dv_status_string.restype = ctypes.c_char_p
        L.dv_status_string.argtypes = [_i]
        L.dv_workspace_size.restype = _sz
        L.dv_workspace_size.argtypes = [ctypes.POINTER(Dims), _i, _i]
        L.dv_set_tuning.argtypes = [_i, _i, _i, _i, _i, _i, _i]
        L.dv_predict.argtypes = [_p, _i, _i, _p, _i, _p, _i, _i, _p, _p, _sz, _p]
        L.dv_select_topk.argtypes = [_p, _i, _i, _i, _i, _p, _p, _p, _p, _p, _sz, _p]
        L.dv_sparse_mlp.argtypes = [_p, _i, ctypes.POINTER(Dims), ctypes.POINTER(LayerWeights),
                                    _p, _i, _p, _i, _p, _p, _p, _sz, _p]
        L.dv_sparse_attn.argtypes = [_p, _i, ctypes.POINTER(Dims), ctypes.POINTER(LayerWeights),
                                     _p, _i, _p, ctypes.POINTER(KvCache), _i, _f, _i, _p, _p, _p,
                                     _sz, _p]
        L.dv_kv_select_attn.argtypes = [_p, ctypes.POINTER(Dims), ctypes.POINTER(KvCache), _i, _p,
                                        _i, _i, _i, _f, _f, _i, _p, _p, _p, _p, _sz, _p]
        L.dv_decode_layer.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Keep), _i,
                                      ctypes.POINTER(LayerWeights), _p, _p,
                                      ctypes.POINTER(KvCache), _i, _f, ctypes.POINTER(Sets),
                                      ctypes.POINTER(Sets), _p, _p, _i, _p, _p, _sz, _p, _p, _p,
                                      _p]
        L.dv_decode_step.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Keep), _i, _i,
                                     ctypes.POINTER(LayerWeights), ctypes.POINTER(KvCache), _i, _f,
                                     ctypes.POINTER(Sets), _p, _p, _p, _i, _p, _p, _sz, _p, _p, _p,
                                     _p]
        L.dv_union_mlp_ws_size.restype = _sz
        L.dv_union_mlp_ws_size.argtypes = [_i, _i, _i]
        L.dv_union_mlp.argtypes = [_p, _i, ctypes.POINTER(Dims), ctypes.POINTER(LayerWeights), _p,
                                   _i, _p, _i, _p, _p, _p, _sz, _p]
        L.dv_w4_row_bytes.restype = _sz
        L.dv_w4_row_bytes.argtypes = [_i]
        L.dv_quantize_w4.argtypes = [_p, _i, _i, _p, _p]
        L.dv_sparse_mlp_w4.argtypes = [_p, _i, ctypes.POINTER(Dims), ctypes.POINTER(LayerWeights),
                                       _p, _p, _p, _i, _p, _i, _p, _p, _p, _sz, _p]
        _R, _C = ctypes.POINTER(Request), ctypes.POINTER(CostModel)
        _D, _K = ctypes.POINTER(Dims), ctypes.POINTER(Keep)
        L.dv_plan_bytes.argtypes = [_D, _K, _R, _d, ctypes.POINTER(_d)]
        L.dv_cost_calibrate.argtypes = [_D, _K, _R, _i, ctypes.POINTER(_d), ctypes.POINTER(_d),
                                        ctypes.POINTER(_d), _C]
        L.dv_plan_decode.argtypes = [_D, _K, _R, _C, _d, ctypes.POINTER(Plan)]
        L.dv_plan_crossing.argtypes = [_D, _K, _R, _C, _i, _i, _d, _d, ctypes.POINTER(_d)]
        _lib = L
    return _lib


EXPORTED = ["dv_version", "dv_status_string", "dv_workspace_size", "dv_set_tuning", "dv_profile",
            "dv_launch_count", "dv_predict",
            "dv_select_topk", "dv_sparse_mlp", "dv_sparse_attn", "dv_kv_select_attn",
            "dv_decode_layer", "dv_decode_step", "dv_sparse_mlp_noalloc", "dv_plan_bytes",
            "dv_cost_calibrate", "dv_plan_decode", "dv_plan_crossing", "dv_w4_row_bytes",
            "dv_quantize_w4", "dv_sparse_mlp_w4", "dv_union_mlp_ws_size", "dv_union_mlp",
            "dv_count_active"]


def status_string(code: int) -> str:
    return lib().dv_status_string(code).decode()


def _check(rc, where):
    if rc != DV_OK:
        raise DvError(rc, where)


def ptr(t):
    """Device pointer of a tensor (or None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def event(timing=False) -> "torch.cuda.Event":
    """A CUDA event whose handle exists now (torch creates handles lazily, on
    the first record), usable as ev_fork / ev_join or for profiling."""
    e = torch.cuda.Event(enable_timing=timing)
    e.record()
    return e


def _ev(e):
    if e is None:
        return None
    h = e.cuda_event
    if not h:
        raise ValueError("CUDA event has no handle yet; create it with dv.event()")
    return h


def dims(d, h, h_kv, d_h, F, r, n_max, ln_eps=1e-5) -> Dims:
    return Dims(d, h, h_kv, d_h, F, r, n_max, ln_eps)


def layer_weights(W: dict) -> LayerWeights:
    return LayerWeights(*[ptr(W.get(n)) for n in _W_FIELDS])


def workspace_size(D: Dims, B: int = 1, flags: int = 0) -> int:
    return lib().dv_workspace_size(ctypes.byref(D), B, flags)


def workspace(D: Dims, B=1, flags=0, device="cuda"):
    n = workspace_size(D, B, flags)
    if n == 0:
        raise DvError(DV_ERR_DIMS, "dv_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def set_tuning(main_ctas=0, side_ctas=0, main_ring_kb=160, side_ring_kb=32, attn_ctas=0, pdl=1,
               stage_kb=48):
    _check(lib().dv_set_tuning(main_ctas, side_ctas, main_ring_kb, side_ring_kb, attn_ctas, pdl,
                               stage_kb), "dv_set_tuning")


# ---------------------------------------------------------------------------
# Entry points
# ---------------------------------------------------------------------------
def predict(y, P1, P2, scores, ws, relu=False, stream=None):
    B, d = y.shape
    r = P1.shape[0]
    N = P2.shape[0]
    _check(lib().dv_predict(ptr(y), B, d, ptr(P1), r, ptr(P2), N, DV_PRED_RELU if relu else 0,
                            ptr(scores), ptr(ws), ws.numel(), _stream(stream)), "dv_predict")


def select_topk(scores, N, k, idx, union_idx=None, union_count=None, dev_status=None, ld=None,
                stream=None):
    B = scores.shape[0] if scores.dim() == 2 else 1
    ld = ld if ld is not None else scores.shape[-1]
    _check(lib().dv_select_topk(ptr(scores), B, ld, N, k, ptr(idx), ptr(union_idx),
                                ptr(union_count), ptr(dev_status), None, 0, _stream(stream)),
           "dv_select_topk")


def sparse_mlp(x, D: Dims, W: dict, idx, k, out, ws, dev_count=None, flags=0, dev_status=None,
               stream=None):
    lw = layer_weights(W)
    B = x.shape[0]
    _check(lib().dv_sparse_mlp(ptr(x), B, ctypes.byref(D), ctypes.byref(lw), ptr(idx), k,
                               ptr(dev_count), flags, ptr(out), ptr(dev_status), ptr(ws),
                               ws.numel(), _stream(stream)), "dv_sparse_mlp")


def union_mlp(x, D: Dims, W: dict, union_idx, k, out, dev_count=None, flags=0, dev_status=None,
              ws=None, stream=None):
    """Batched (B = 8..64) MLP over one union of neurons on the tensor cores."""
    import torch
    B = x.shape[0]
    need = lib().dv_union_mlp_ws_size(B, D.d, k)
    if ws is None:
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=x.device)
    lw = layer_weights(W)
    _check(lib().dv_union_mlp(ptr(x), B, ctypes.byref(D), ctypes.byref(lw), ptr(union_idx), k,
                              ptr(dev_count), flags, ptr(out), ptr(dev_status), ptr(ws), ws.numel(),
                              _stream(stream)), "dv_union_mlp")
    return ws


def w4_row_bytes(d: int) -> int:
    return lib().dv_w4_row_bytes(d)


def quantize_w4(W, out=None, stream=None):
    """Packed 4-bit rows [rows][w4_row_bytes(d)] (uint8) of fp16 rows W [rows][d]."""
    import torch
    rows, d = W.shape
    if out is None:
        out = torch.empty(rows, w4_row_bytes(d), dtype=torch.uint8, device=W.device)
    _check(lib().dv_quantize_w4(ptr(W), rows, d, ptr(out), _stream(stream)), "dv_quantize_w4")
    return out


def sparse_mlp_w4(x, D: Dims, W: dict, fc1_w4, fc2T_w4, idx, k, out, ws, dev_count=None, flags=0,
                  dev_status=None, stream=None):
    lw = layer_weights(W)
    _check(lib().dv_sparse_mlp_w4(ptr(x), x.shape[0], ctypes.byref(D), ctypes.byref(lw),
                                  ptr(fc1_w4), ptr(fc2T_w4), ptr(idx), k, ptr(dev_count), flags,
                                  ptr(out), ptr(dev_status), ptr(ws), ws.numel(), _stream(stream)),
           "dv_sparse_mlp_w4")


def kv_cache(K, V, y_side=None, kv_missing=None, Kr=None, Vr=None, kept_pos=None, kept_count=None,
             b_max=0) -> KvCache:
    return KvCache(ptr(K), ptr(V), ptr(y_side), ptr(kv_missing), ptr(Kr), ptr(Vr), ptr(kept_pos),
                   ptr(kept_count), b_max)


def sparse_attn(x, D: Dims, W: dict, head_idx, k_heads, kv: KvCache, n, out, ws, scale=None,
                dev_count=None, flags=0, dev_status=None, stream=None):
    lw = layer_weights(W)
    B = x.shape[0]
    if scale is None:
        scale = D.d_h ** -0.5
    _check(lib().dv_sparse_attn(ptr(x), B, ctypes.byref(D), ctypes.byref(lw), ptr(head_idx),
                                k_heads, ptr(dev_count), ctypes.byref(kv), n, scale, flags,
                                ptr(out), ptr(dev_status), ptr(ws), ws.numel(), _stream(stream)),
           "dv_sparse_attn")


def kv_select_attn(q, D: Dims, kv: KvCache, n, H, ws, q_obs=None, obs_window=64, n_sinks=4,
                   smooth=7, kv_keep=0.125, scale=None, flags=0, sel_scores=None, dev_status=None,
                   stream=None):
    if scale is None:
        scale = D.d_h ** -0.5
    _check(lib().dv_kv_select_attn(ptr(q), ctypes.byref(D), ctypes.byref(kv), n, ptr(q_obs),
                                   obs_window, n_sinks, smooth, kv_keep, scale, flags, ptr(H),
                                   ptr(sel_scores), ptr(dev_status), ptr(ws), ws.numel(),
                                   _stream(stream)), "dv_kv_select_attn")


def sets(B, F, h_units, kN, kH, device="cuda") -> tuple:
    """Device buffers of one layer's index sets and the ctypes struct pointing at them."""
    t = {
        "idx_N": torch.zeros(B, kN, dtype=torch.int32, device=device),
        "idx_H": torch.zeros(B, kH, dtype=torch.int32, device=device),
        "uN": torch.zeros(F, dtype=torch.int32, device=device),
        "uH": torch.zeros(max(h_units, 4), dtype=torch.int32, device=device),
        "ucnt": torch.zeros(4, dtype=torch.int32, device=device),
        "scores": torch.zeros(B, F + h_units, dtype=torch.float32, device=device),
    }
    s = Sets(ptr(t["idx_N"]), ptr(t["idx_H"]), ptr(t["uN"]), ptr(t["uH"]), ptr(t["ucnt"]),
             ptr(t["scores"]))
    return s, t


def decode_layer(D: Dims, keep: Keep, W: dict, P_next, kv: KvCache, n, cur: Sets, nxt: Sets,
                 y_in, y_out, ws, flags, ev_fork=None, ev_join=None, side=None, scale=None,
                 dev_status=None, stream=None):
    lw = layer_weights(W)
    if scale is None:
        scale = D.d_h ** -0.5
    P1n, P2n = (P_next if P_next is not None else (None, None))
    _check(lib().dv_decode_layer(ctypes.byref(D), ctypes.byref(keep), y_in.shape[0],
                                 ctypes.byref(lw), ptr(P1n), ptr(P2n), ctypes.byref(kv), n, scale,
                                 ctypes.byref(cur), ctypes.byref(nxt) if nxt is not None else None,
                                 ptr(y_in), ptr(y_out), flags, ptr(dev_status), ptr(ws),
                                 ws.numel(), _stream(stream),
                                 side.cuda_stream if side is not None else None,
                                 _ev(ev_fork), _ev(ev_join)),
           "dv_decode_layer")


def decode_step(D: Dims, keep: Keep, Ws: list, kvs: list, n, sets2: list, y_in, y_tmp, y_out, ws,
                flags, side, ev_fork, ev_join, scale=None, dev_status=None, stream=None):
    L = len(Ws)
    warr = (LayerWeights * L)(*[layer_weights(W) for W in Ws])
    karr = (KvCache * L)(*kvs)
    sarr = (Sets * 2)(*sets2)
    if scale is None:
        scale = D.d_h ** -0.5
    _check(lib().dv_decode_step(ctypes.byref(D), ctypes.byref(keep), y_in.shape[0], L, warr, karr,
                                n, scale, sarr, ptr(y_in), ptr(y_tmp), ptr(y_out), flags,
                                ptr(dev_status), ptr(ws), ws.numel(), _stream(stream),
                                side.cuda_stream, _ev(ev_fork), _ev(ev_join)),
           "dv_decode_step")


# ---------------------------------------------------------------------------
# Launch accounting (aux)
# ---------------------------------------------------------------------------
TAGS = {0: "qkv", 1: "splitk", 2: "wo", 3: "reduce", 4: "mlp", 5: "pred1", 6: "pred2", 7: "topk",
        8: "union", 9: "combine", 10: "kvsel", 11: "kvappend", 12: "kvadvance", 13: "kvfill"}


class Profiler:
    """Brackets every library kernel launch with CUDA events on its stream
    (``dv_profile``). Usable inside stream capture: the records become graph
    nodes and hold the timestamps of the latest replay."""

    def __init__(self, cap=4096):
        self.cap = cap
        self.events = [event(timing=True) for _ in range(2 * cap)]
        self._ev = (ctypes.c_void_p * (2 * cap))(*[e.cuda_event for e in self.events])
        self._tags = (ctypes.c_int * cap)()
        self.n = 0

    def start(self):
        lib().dv_profile.argtypes = [_p, _p, _i]
        lib().dv_profile(ctypes.cast(self._ev, _p), ctypes.cast(self._tags, _p), self.cap)

    def stop(self):
        self.n = lib().dv_profile(None, None, 0)
        return self.n

    def durations_ms(self):
        """[(tag name, ms)] of the recorded launches (call after synchronising)."""
        return [(TAGS.get(self._tags[i], str(self._tags[i])),
                 self.events[2 * i].elapsed_time(self.events[2 * i + 1])) for i in range(self.n)]


def count_active(counter=None):
    """MLP launches with DV_SKIP_INACTIVE add their streamed fc2T rows to the
    device int `counter` from now on (None stops; dv_count_active)."""
    lib().dv_count_active.argtypes = [_p]
    lib().dv_count_active(ptr(counter))


def launch_count() -> int:
    lib().dv_launch_count.restype = ctypes.c_longlong
    return lib().dv_launch_count()


class Step:
    """Prepared arguments of dv_decode_step for a fixed stack (the ctypes arrays
    are built once, so a step costs one C call)."""

    def __init__(self, D: Dims, keep: Keep, Ws: list, kvs: list, sets2: list, ws, flags,
                 side, ev_fork, ev_join, scale=None, dev_status=None):
        self.D, self.keep, self.flags = D, keep, flags
        self.L = len(Ws)
        self.warr = (LayerWeights * self.L)(*[layer_weights(W) for W in Ws])
        self.karr = (KvCache * self.L)(*kvs)
        self.sarr = (Sets * 2)(*sets2)
        self.ws = ws
        self.side, self.ev_fork, self.ev_join = side, ev_fork, ev_join
        self.scale = D.d_h ** -0.5 if scale is None else scale
        self.dev_status = dev_status

    def __call__(self, y_in, y_tmp, y_out, n, stream=None):
        _check(lib().dv_decode_step(ctypes.byref(self.D), ctypes.byref(self.keep), y_in.shape[0],
                                    self.L, self.warr, self.karr, n, self.scale, self.sarr,
                                    ptr(y_in), ptr(y_tmp), ptr(y_out), self.flags,
                                    ptr(self.dev_status), ptr(self.ws), self.ws.numel(),
                                    _stream(stream), self.side.cuda_stream,
                                    _ev(self.ev_fork), _ev(self.ev_join)),
               "dv_decode_step")


# ---------------------------------------------------------------------------
# latency gate (host-only calls: no device needed)
# ---------------------------------------------------------------------------
def request(B=1, steps=1, union_N=0, union_H=0, kv_budget=0, modes=0) -> Request:
    return Request(B, steps, union_N, union_H, kv_budget, modes)


def plan_bytes(D: Dims, keep: Keep, req: Request, n: float) -> list:
    out = (_d * 4)()
    _check(lib().dv_plan_bytes(ctypes.byref(D), ctypes.byref(keep), ctypes.byref(req), n, out),
           "dv_plan_bytes")
    return list(out)


def cost_calibrate(D: Dims, keep: Keep, req: Request, ctx, measured_us, select_us=None) -> CostModel:
    """measured_us[m][i]: mode m's layer time (µs) at ctx[i]; row 0 = dense."""
    nc = len(ctx)
    c = (_d * nc)(*ctx)
    m = (_d * (4 * nc))(*[float(v) for row in measured_us for v in row])
    s = (_d * nc)(*select_us) if select_us is not None else None
    cm = CostModel()
    _check(lib().dv_cost_calibrate(ctypes.byref(D), ctypes.byref(keep), ctypes.byref(req), nc, c,
                                   m, s, ctypes.byref(cm)), "dv_cost_calibrate")
    return cm


def cost_model(ctx, dense_us, cost_us, select_us=None) -> CostModel:
    cm = CostModel()
    cm.n_ctx = len(ctx)
    for i, c in enumerate(ctx):
        cm.ctx[i], cm.dense_us[i] = c, dense_us[i]
        cm.select_us[i] = 0.0 if select_us is None else select_us[i]
        for m in range(4):
            cm.cost_us[m][i] = cost_us[m][i]
    return cm


def plan_decode(D: Dims, keep: Keep, req: Request, cm: CostModel, n: float) -> dict:
    """Predicted per-layer µs of the four modes at context n and the chosen
    mode (the fastest admitted one)."""
    p = Plan()
    _check(lib().dv_plan_decode(ctypes.byref(D), ctypes.byref(keep), ctypes.byref(req),
                                ctypes.byref(cm), n, ctypes.byref(p)), "dv_plan_decode")
    return {"choice": p.choice, "us": list(p.us), "bytes": list(p.bytes)}


def plan_crossing(D: Dims, keep: Keep, req: Request, cm: CostModel, a: int, b: int, lo: float,
                  hi: float):
    """First context in [lo, hi] where modes a and b are predicted equal, or None."""
    x = _d()
    _check(lib().dv_plan_crossing(ctypes.byref(D), ctypes.byref(keep), ctypes.byref(req),
                                  ctypes.byref(cm), a, b, lo, hi, ctypes.byref(x)),
           "dv_plan_crossing")
    return None if x.value < 0 else x.value
