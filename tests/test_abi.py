"""The C ABI: libdv.so builds, exports every symbol include/dv.h declares, and
host-side validation rejects bad arguments with a status code before anything
is enqueued. No compute calls: every case here fails validation first (no
pointer given here is ever dereferenced)."""
import ctypes
import os
import re
import subprocess

import pytest

from contextual_sparsity_gb300 import build, dv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return dv.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "dv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w \t*]*?\b(dv_\w+)\s*\(", src, flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "dv_sparse_mlp" in names and "dv_decode_layer" in names and len(names) >= 11
    out = subprocess.run(["nm", "-D", "--defined-only", dv.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(dv_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert sorted(dv.EXPORTED) == names


def test_status_strings(L):
    assert dv.status_string(0) == "ok"
    for c in range(-8, 0):
        s = dv.status_string(c)
        assert s and s != "unknown status"
    assert dv.status_string(-99) == "unknown status"
    assert L.dv_version() >= 100


def _dims(**kw):
    base = dict(d=256, h=4, h_kv=4, d_h=64, F=1024, r=32, n_max=80, ln_eps=1e-5)
    base.update(kw)
    return dv.Dims(**base)


def test_workspace_size_rejects_bad_dims(L):
    assert dv.workspace_size(_dims()) > 0
    for bad in (dict(d=250), dict(d=0), dict(h=6, h_kv=4), dict(d_h=96), dict(F=0), dict(r=30),
                dict(n_max=0)):
        assert dv.workspace_size(_dims(**bad)) == 0, bad
    assert L.dv_workspace_size(ctypes.byref(_dims()), 5, 0) == 0
    assert L.dv_workspace_size(None, 1, 0) == 0


FAKE = 0x100000   # aligned, never dereferenced: every call below fails validation first
MISALIGNED = 0x100002


def _w(**kw):
    w = {n: FAKE for n in ("Wq", "Wk", "Wv", "WoT", "fc1", "fc2T", "P1", "P2")}
    w.update(kw)
    return dv.LayerWeights(*[w.get(n) for n in dv._W_FIELDS])


def _mlp(L, x=FAKE, B=1, D=None, w=None, idx=None, k=1, out=FAKE + 4096, ws=FAKE * 2, ws_bytes=0):
    D = D or _dims()
    w = w or _w()
    return L.dv_sparse_mlp(x, B, ctypes.byref(D), ctypes.byref(w), idx, k, None, 0, out, None, ws,
                           ws_bytes, None)


def test_sparse_mlp_validation(L):
    assert _mlp(L, x=None) == dv.DV_ERR_NULL
    assert _mlp(L, x=MISALIGNED) == dv.DV_ERR_ALIGN
    assert _mlp(L, D=_dims(d=100)) == dv.DV_ERR_DIMS
    assert _mlp(L, w=_w(fc1=None)) == dv.DV_ERR_NULL
    assert _mlp(L, w=_w(fc2T=MISALIGNED)) == dv.DV_ERR_ALIGN
    assert _mlp(L, B=5) == dv.DV_ERR_DIMS
    assert _mlp(L, idx=FAKE, k=0) == dv.DV_ERR_K
    assert _mlp(L, idx=FAKE, k=1025) == dv.DV_ERR_K
    assert _mlp(L, out=FAKE) == dv.DV_ERR_DIMS           # out aliases x
    assert _mlp(L, ws=FAKE + 16) == dv.DV_ERR_ALIGN       # workspace wants 256-byte alignment
    assert _mlp(L, idx=FAKE, k=8, ws_bytes=16) == dv.DV_ERR_WORKSPACE


def test_predict_and_topk_validation(L):
    f = L.dv_predict
    assert f(None, 1, 256, FAKE, 32, FAKE, 10, 0, FAKE, FAKE, 1 << 20, None) == dv.DV_ERR_NULL
    assert f(FAKE, 0, 256, FAKE, 32, FAKE, 10, 0, FAKE, FAKE, 1 << 20, None) == dv.DV_ERR_DIMS
    assert f(FAKE, 1, 256, FAKE, 30, FAKE, 10, 0, FAKE, FAKE, 1 << 20, None) == dv.DV_ERR_DIMS
    assert f(FAKE, 1, 256, FAKE, 32, FAKE, 10, 0, FAKE, FAKE, 8, None) == dv.DV_ERR_WORKSPACE
    t = L.dv_select_topk
    assert t(FAKE, 1, 10, 10, 0, FAKE, None, None, None, None, 0, None) == dv.DV_ERR_K
    assert t(FAKE, 1, 10, 10, 11, FAKE, None, None, None, None, 0, None) == dv.DV_ERR_K
    assert t(FAKE, 1, 5, 10, 3, FAKE, None, None, None, None, 0, None) == dv.DV_ERR_DIMS
    assert t(FAKE, 9, 10, 10, 3, FAKE, None, None, None, None, 0, None) == dv.DV_ERR_DIMS
    assert t(FAKE, 1, 10, 10, 3, FAKE, FAKE, None, None, None, 0, None) == dv.DV_ERR_NULL


def test_attention_and_layer_validation(L):
    D = _dims()
    w = _w()
    kv = dv.KvCache(FAKE, FAKE, None, None, None, None, None, None, 0)
    a = L.dv_sparse_attn
    args = lambda n=10, k=2, flags=0, kvp=kv: (FAKE, 1, ctypes.byref(D), ctypes.byref(w), FAKE, k,
                                                None, ctypes.byref(kvp), n, 0.125, flags,
                                                FAKE + 4096, None, FAKE * 2, 16, None)
    assert a(*args(n=80)) == dv.DV_ERR_DIMS          # n must be < n_max
    assert a(*args(n=-1)) == dv.DV_ERR_DIMS
    assert a(*args(k=5)) == dv.DV_ERR_K
    assert a(*args(flags=dv.DV_KV_RETAINED)) == dv.DV_ERR_NULL   # no retained buffers
    assert a(*args(flags=dv.DV_KV_FILL)) == dv.DV_ERR_NULL       # no kept inputs / marks
    kv_f = dv.KvCache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64)
    assert a(*args(flags=dv.DV_KV_FILL | dv.DV_KV_RESELECT, kvp=kv_f)) == dv.DV_ERR_UNSUPPORTED
    assert a(*args(flags=dv.DV_KV_FILL | dv.DV_KV_RETAINED, kvp=kv_f)) == dv.DV_ERR_WORKSPACE
    assert a(*args(flags=dv.DV_KV_FILL, kvp=kv_f)) == dv.DV_ERR_WORKSPACE
    assert a(*args(flags=dv.DV_W4 | dv.DV_KV_FILL, kvp=kv_f)) == dv.DV_ERR_WORKSPACE
    assert a(*args(flags=dv.DV_W4)) == dv.DV_ERR_WORKSPACE           # d 256: a multiple of 128
    D264 = _dims(d=264)
    assert a(FAKE, 1, ctypes.byref(D264), ctypes.byref(w), FAKE, 2, None, ctypes.byref(kv), 10,
             0.125, dv.DV_W4, FAKE + 4096, None, FAKE * 2, 16, None) == dv.DV_ERR_DIMS
    assert a(*args()) == dv.DV_ERR_WORKSPACE
    keep = dv.Keep(0.0, 0.5, 1.0)
    lay = L.dv_decode_layer
    s = dv.Sets(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE)
    call = lambda kp, B=1: lay(ctypes.byref(D), ctypes.byref(kp), B, ctypes.byref(w), None, None,
                                 ctypes.byref(kv), 10, 0.125, ctypes.byref(s), None, FAKE,
                                 FAKE + 4096, 0, None, FAKE * 2, 16, None, None, None, None)
    assert call(keep) == dv.DV_ERR_KEEP
    assert call(dv.Keep(1.5, 0.5, 1.0)) == dv.DV_ERR_KEEP
    assert call(dv.Keep(0.25, 0.5, 1.0), B=0) == dv.DV_ERR_DIMS
    assert call(dv.Keep(0.25, 0.5, 1.0)) == dv.DV_ERR_WORKSPACE


def test_kv_select_validation(L):
    D = _dims(h=8, h_kv=2, n_max=300)
    kv = dv.KvCache(FAKE, FAKE, None, None, FAKE, FAKE, FAKE, FAKE, 64)
    f = L.dv_kv_select_attn
    big = 1 << 40
    call = lambda n=200, W=64, sinks=4, sm=7, keep=0.125, flags=dv.DV_KV_RESELECT: f(
        FAKE, ctypes.byref(D), ctypes.byref(kv), n, FAKE, W, sinks, sm, keep, 0.1, flags, FAKE,
        None, None, FAKE * 2, big, None)
    assert call(W=0) == dv.DV_ERR_DIMS
    assert call(W=201) == dv.DV_ERR_DIMS
    assert call(sm=6) == dv.DV_ERR_DIMS
    assert call(keep=0.0) == dv.DV_ERR_KEEP
    assert call(keep=1.5) == dv.DV_ERR_KEEP
    assert call(n=300) == dv.DV_ERR_DIMS


def test_w4_validation(L):
    assert dv.w4_row_bytes(12288) == 6336 and dv.w4_row_bytes(256) == 144
    assert dv.w4_row_bytes(4096) == 2112 and dv.w4_row_bytes(100) == 0 and dv.w4_row_bytes(0) == 0
    q = L.dv_quantize_w4
    assert q(None, 4, 256, FAKE, None) == dv.DV_ERR_NULL
    assert q(MISALIGNED, 4, 256, FAKE, None) == dv.DV_ERR_ALIGN
    assert q(FAKE, 4, 200, FAKE, None) == dv.DV_ERR_DIMS
    assert q(FAKE, 0, 256, FAKE, None) == dv.DV_ERR_DIMS
    D = _dims()
    w = _w()
    m = L.dv_sparse_mlp_w4
    args = lambda fc1=FAKE, k=4, B=1, dd=D, ws_bytes=16: (
        FAKE, B, ctypes.byref(dd), ctypes.byref(w), fc1, FAKE + 8192, FAKE, k, None, 0,
        FAKE + 4096, None, FAKE * 2, ws_bytes, None)
    assert m(*args(fc1=None)) == dv.DV_ERR_NULL
    assert m(*args(fc1=MISALIGNED)) == dv.DV_ERR_ALIGN
    assert m(*args(k=0)) == dv.DV_ERR_K
    assert m(*args(B=5)) == dv.DV_ERR_DIMS
    assert m(*args(dd=_dims(d=264))) == dv.DV_ERR_DIMS      # not a multiple of 128
    assert m(*args()) == dv.DV_ERR_WORKSPACE


def test_union_mlp_validation(L):
    assert L.dv_union_mlp_ws_size(8, 512, 100) > 0 and L.dv_union_mlp_ws_size(24, 512, 100) == 0
    assert L.dv_union_mlp_ws_size(4, 512, 100) == 0 and L.dv_union_mlp_ws_size(128, 512, 100) == 0
    D = _dims()
    w = _w()
    u = L.dv_union_mlp
    args = lambda B=8, idx=FAKE, k=4, ws_bytes=16: (FAKE, B, ctypes.byref(D), ctypes.byref(w), idx,
                                                    k, None, 0, FAKE + 4096, None, FAKE * 2,
                                                    ws_bytes, None)
    assert u(*args(idx=None)) == dv.DV_ERR_NULL
    assert u(*args(k=0)) == dv.DV_ERR_K
    assert u(*args(B=12)) == dv.DV_ERR_UNSUPPORTED
    assert u(*args()) == dv.DV_ERR_WORKSPACE


_NOALLOC_CHECKS = r'''
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from contextual_sparsity_gb300 import dv
L = dv.lib()
f = L.dv_sparse_mlp_noalloc
f.restype = ctypes.c_int
f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(dv.Dims),
              ctypes.POINTER(dv.LayerWeights), ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
              ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
FAKE = 0x100000
D = dv.Dims(d=256, h=4, h_kv=4, d_h=64, F=1024, r=32, n_max=80, ln_eps=1e-5)
w = dv.LayerWeights(*[FAKE if n in ("fc1", "fc2T") else None for n in dv._W_FIELDS])
call = lambda D=D, w=w, B=1, idx=FAKE, k=4, flags=0, x=FAKE, out=FAKE + 4096: f(
    x, B, ctypes.byref(D), ctypes.byref(w), idx, k, None, flags, out, None, None)
res = {
    "w4": call(flags=dv.DV_W4),
    "w4_all": call(flags=dv.DV_W4 | dv.DV_SKIP_INACTIVE, idx=None),
    "eps": call(D=dv.Dims(d=256, h=4, h_kv=4, d_h=64, F=1024, r=32, n_max=80, ln_eps=-1.0)),
    "heads": call(D=dv.Dims(d=256, h=6, h_kv=4, d_h=64, F=1024, r=32, n_max=80, ln_eps=1e-5)),
    "ln2_misaligned": call(w=dv.LayerWeights(*[FAKE if n in ("fc1", "fc2T") else
                                             (FAKE + 2 if n == "ln2_g" else None)
                                             for n in dv._W_FIELDS])),
    "null_out": call(out=None),
    "alias": call(out=FAKE),
    "k": call(k=0),
    "B": call(B=5),
    # 4 rows of 16384 fp32 partial sums need 256 KiB per CTA, and 262144 rows
    # need at least 1024 CTAs of 256 rows: beyond the 8 MiB array
    "too_big": call(D=dv.Dims(d=16384, h=128, h_kv=128, d_h=128, F=262144, r=8, n_max=8,
                              ln_eps=1e-5), B=4, idx=None, k=0),
}
print(repr(res))
'''


def test_noalloc_validation_without_a_gpu():
    """dv_sparse_mlp_noalloc rejects what it cannot serve before it launches
    anything: packed 4-bit rows, the dimension and weight checks of
    dv_sparse_mlp, and problems beyond its built-in array. Run in a child
    process that sees no CUDA device, so a call that got past its checks would
    fail on the host (a launch error), never reach a GPU."""
    import ast
    import sys

    build.build()
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", _NOALLOC_CHECKS, ROOT], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    res = ast.literal_eval(r.stdout.strip().splitlines()[-1])
    assert res["w4"] == dv.DV_ERR_UNSUPPORTED
    assert res["w4_all"] == dv.DV_ERR_UNSUPPORTED
    assert res["eps"] == dv.DV_ERR_DIMS
    assert res["heads"] == dv.DV_ERR_DIMS
    assert res["ln2_misaligned"] == dv.DV_ERR_ALIGN
    assert res["null_out"] == dv.DV_ERR_NULL
    assert res["alias"] == dv.DV_ERR_DIMS
    assert res["k"] == dv.DV_ERR_K
    assert res["B"] == dv.DV_ERR_DIMS
    assert res["too_big"] == dv.DV_ERR_WORKSPACE
