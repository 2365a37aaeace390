// dv_abi.cu -- the extern "C" entry points of libdv.so (see include/dv.h).
//
// Host side only: argument validation (a bad argument returns a negative
// status before anything is enqueued), the workspace layout, and the order of
// kernel launches on the caller's streams. The decode driver follows "Deja
// Vu" §4.3: layer l's sets come from the look-ahead of layer l-1 (computed
// from y_{l-1} on a side stream while layer l-1 runs), layer 0 predicts
// synchronously, and a layer is y' = h + MLP(h), h = y + MHA(y) (App. C.3).
#include <cmath>
#include <cstdio>

#include "dv_internal.h"
#include "k_union_tc.h"

namespace dv {

struct Tuning {
  int main_ctas = 0;        // 0: one per SM
  int side_ctas = 0;        // predictor CTAs on the side stream; 0: two per SM
  int main_ring = 160 * 1024;
  int side_ring = 32 * 1024;
  int attn_ctas = 0;        // split-K CTA target; 0: two per SM
};
static Tuning g_tune;
int* g_count_active = nullptr;

int sm_count() {
  static int cached = 0;
  if (!cached) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    cached = n;
  }
  return cached;
}

static cudaEvent_t* g_prof_ev = nullptr;
static int* g_prof_tags = nullptr;
static int g_prof_cap = 0, g_prof_n = 0;
static long long g_launches = 0;

void note_launch(int tag, int phase, cudaStream_t s) {
  if (phase == 0) ++g_launches;
  if (!g_prof_ev || g_prof_n >= g_prof_cap) return;
  // External records become event nodes under stream capture (a plain record
  // would only express a dependency), so graph replays leave timestamps.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_prof_ev[2 * g_prof_n + phase], s, cudaEventRecordExternal);
  else
    cudaEventRecord(g_prof_ev[2 * g_prof_n + phase], s);
  if (phase == 0) {
    g_prof_tags[g_prof_n] = tag;
  } else {
    ++g_prof_n;
  }
}

static int side_ctas() { return g_tune.side_ctas > 0 ? g_tune.side_ctas : 2 * sm_count(); }
int main_ctas() { return g_tune.main_ctas > 0 ? g_tune.main_ctas : sm_count(); }
int main_ring_bytes() { return g_tune.main_ring; }

static bool g_pdl = true;

cudaError_t launch_k(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     void** args, bool pdl, int cluster_x) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pdl && g_pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (cluster_x > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelExC(&cfg, fn, args);
}
static int attn_ctas() { return g_tune.attn_ctas > 0 ? g_tune.attn_ctas : 2 * sm_count(); }

static int k_from_keep(float keep, int N) {
  const double k = std::floor((double)keep * (double)N + 1e-9);
  return std::max(1, (int)std::min<double>(k, N));
}

static bool aligned(const void* p, size_t a = 16) { return ((uintptr_t)p % a) == 0; }

#define REQ(c, e)          \
  do {                     \
    if (!(c)) return (e);  \
  } while (0)
#define REQ_PTR(p) \
  do {             \
    if (!(p)) return DV_ERR_NULL; \
    if (!aligned(p)) return DV_ERR_ALIGN; \
  } while (0)
#define OPT_PTR(p) \
  do {             \
    if ((p) && !aligned(p)) return DV_ERR_ALIGN; \
  } while (0)

int check_dims(const dv_dims* D) {
  REQ(D, DV_ERR_NULL);
  REQ(D->d >= 8 && D->d <= 16384 && D->d % 8 == 0, DV_ERR_DIMS);
  REQ(D->h >= 1 && D->h_kv >= 1 && D->h % D->h_kv == 0, DV_ERR_DIMS);
  const int G = D->h / D->h_kv;
  REQ(G == 1 || G == 2 || G == 4 || G == 8, DV_ERR_UNSUPPORTED);
  REQ(D->d_h == 64 || D->d_h == 128, DV_ERR_UNSUPPORTED);
  REQ(D->F >= 1, DV_ERR_DIMS);
  REQ(D->r >= 0 && D->r <= 4096 && D->r % 8 == 0, DV_ERR_DIMS);
  REQ(D->n_max >= 1, DV_ERR_DIMS);
  REQ(D->ln_eps >= 0.f, DV_ERR_DIMS);
  return DV_OK;
}

// ---- workspace layout ------------------------------------------------------
struct WsLayout {
  size_t part, qbuf, sk, hcomb, cnt, hmid, u_main, u_side, kvsel, total;
  size_t kvsel_floats;
  int S_max;
};

static size_t al(size_t x) { return (x + 255) / 256 * 256; }

static WsLayout ws_layout(const dv_dims* D, int B, int flags) {
  WsLayout L{};
  const int G = D->h / D->h_kv;
  const int target = main_ctas();
  const size_t part = std::max(stream_part_bytes(D->d, B, D->F, target),
                               stream_part_bytes(D->d, B, (long long)D->h * D->d_h, target));
  L.S_max = kSplitsMax;
  size_t off = 0;
  L.part = off;
  off += al(part);
  L.qbuf = off;
  off += al((size_t)B * D->h * D->d_h * 4);
  L.sk = off;
  off += al((size_t)B * D->h_kv * G * L.S_max * (D->d_h + 2) * 4);
  L.hcomb = off;
  off += al((size_t)B * D->h * D->d_h * 4);
  L.cnt = off;  // split-K counters [B][h_kv]
  off += al((size_t)B * D->h_kv * 4);
  L.hmid = off;
  off += al((size_t)B * D->d * 2);
  L.u_main = off;
  off += al((size_t)B * std::max(D->r, 8) * 4);
  L.u_side = off;
  off += al((size_t)B * std::max(D->r, 8) * 4);
  L.kvsel = off;
  if (flags & DV_KV_RESELECT) {
    const int W = std::min(D->n_max, 512 / G);
    L.kvsel_floats = kv_select_ws_floats(D->h, D->h_kv, W, D->n_max);
    off += al(L.kvsel_floats * 4);
  }
  L.total = off;
  return L;
}

template <class T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ---- the attention block and the MLP block (shared by the entry points) ----
// QKV gather-GEMV (+ KV append; optionally the look-ahead predictor's first
// layer on the same input, written to u_out).
static int attn_qkv(const uint16_t* x, int B, const dv_dims* D, const dv_layer_weights* w,
                    const int32_t* sel, int k, const int32_t* dev_count, dv_kv_cache* kv, int n,
                    float scale, int flags, const uint16_t* P1n, float* u_out, int* st, void* ws,
                    const WsLayout& L, cudaStream_t s, bool pdl, bool fill_done = false) {
  const int G = D->h / D->h_kv;
  const bool ret = (flags & DV_KV_RETAINED) != 0;
  const bool fill = (flags & DV_KV_FILL) != 0;
  if (fill && !fill_done) {
    // [DV] 4.2: the selected units' missing k, v first, from the kept inputs
    // (the QKV launch below then clears their marks).
    int rc = launch_kv_fill(kv->y_side, kv->kv_missing, B, D->d, D->h_kv, D->d_h, w->ln1_g,
                            w->ln1_b, D->ln_eps, w->Wk, w->bk, w->Wv, w->bv, sel, k, dev_count,
                            kv->K, kv->V, n, D->n_max, st, s, pdl, ret ? kv->Kr : nullptr,
                            ret ? kv->Vr : nullptr, kv->kept_count, kv->b_max,
                            (flags & DV_W4) != 0);
    if (rc != DV_OK) return rc;
    pdl = true;  // the fill waited for the index list before letting QKV start
  }
  return launch_qkv(x, B, D->d, G, D->d_h, D->h_kv, w->ln1_g, w->ln1_b, D->ln_eps, w->Wq, w->bq,
                    w->Wk, w->bk, w->Wv, w->bv, sel, k, dev_count, scale, at<float>(ws, L.qbuf),
                    kv->K, kv->V, n, D->n_max, ret ? kv->Kr : nullptr, ret ? kv->Vr : nullptr,
                    kv->kept_count, kv->b_max, kv->y_side, kv->kv_missing, fill ? 1 : 0,
                    at<int>(ws, L.cnt),
                    B * D->h_kv, P1n, D->r, (flags & DV_PRED_RELU) ? 1 : 0, u_out, st,
                    main_ctas(), g_tune.main_ring, s, pdl, (flags & DV_W4) != 0);
}

// Split-K attention with the combine fused, then the Wo^T gather-axpy and the
// residual.
static int attn_rest(const uint16_t* x, int B, const dv_dims* D, const dv_layer_weights* w,
                     const int32_t* sel, int k, const int32_t* dev_count, dv_kv_cache* kv, int n,
                     int flags, uint16_t* out, int* st, void* ws, const WsLayout& L,
                     cudaStream_t s) {
  const int G = D->h / D->h_kv;
  const bool ret = (flags & DV_KV_RETAINED) != 0;
  const int max_keys = ret ? kv->b_max : n + 1;
  SplitPlan plan = split_plan(max_keys, k, B, attn_ctas());
  if (plan.S > L.S_max) return DV_ERR_WORKSPACE;
  int rc = launch_splitk(at<float>(ws, L.qbuf), B, D->d_h, G, D->h_kv, sel, k, dev_count, kv->K,
                         kv->V, n, D->n_max, kv->Kr, kv->Vr, kv->kept_count, kv->b_max,
                         ret ? 1 : 0, plan, at<float>(ws, L.sk), at<float>(ws, L.hcomb),
                         at<int>(ws, L.cnt), st, s, true);
  if (rc != DV_OK) return rc;
  rc = launch_wo((flags & DV_NO_RESIDUAL) ? nullptr : x, B, D->d, G, D->d_h, D->h_kv, w->WoT,
                 w->bo, sel, k, dev_count, at<float>(ws, L.hcomb), out, st, at<float>(ws, L.part),
                 main_ctas(), g_tune.main_ring, s, (flags & DV_W4) != 0);
  if (rc != DV_OK) return rc;
  if (ret && (flags & DV_KV_ADVANCE)) rc = launch_kv_advance(kv->kept_count, D->h_kv, kv->b_max, s);
  return rc;
}

static int run_attn(const uint16_t* x, int B, const dv_dims* D, const dv_layer_weights* w,
                    const int32_t* sel, int k, const int32_t* dev_count, dv_kv_cache* kv, int n,
                    float scale, int flags, uint16_t* out, int* st, void* ws, const WsLayout& L,
                    cudaStream_t s) {
  int rc = attn_qkv(x, B, D, w, sel, k, dev_count, kv, n, scale, flags, nullptr, nullptr, st, ws, L,
                    s, false);
  if (rc != DV_OK) return rc;
  return attn_rest(x, B, D, w, sel, k, dev_count, kv, n, flags, out, st, ws, L, s);
}

static int run_mlp(const uint16_t* x, int B, const dv_dims* D, const dv_layer_weights* w,
                   const int32_t* sel, int k, const int32_t* dev_count, int flags, uint16_t* out,
                   int* st, void* ws, const WsLayout& L, cudaStream_t s, bool pdl) {
  if (flags & DV_W4)
    return launch_mlp_w4(x, B, D->d, D->F, w->ln2_g, w->ln2_b, D->ln_eps,
                         reinterpret_cast<const uint8_t*>(w->fc1), w->b1,
                         reinterpret_cast<const uint8_t*>(w->fc2T), w->b2, sel, k, dev_count,
                         flags & (DV_SKIP_INACTIVE | DV_NO_RESIDUAL), out, st,
                         at<float>(ws, L.part), main_ctas(), g_tune.main_ring, s, pdl);
  return launch_mlp(x, B, D->d, D->F, w->ln2_g, w->ln2_b, D->ln_eps, w->fc1, w->b1, w->fc2T, w->b2,
                    sel, k, dev_count, flags & (DV_SKIP_INACTIVE | DV_NO_RESIDUAL), out, st,
                    at<float>(ws, L.part),
                    main_ctas(), g_tune.main_ring, s, pdl);
}

// Second predictor layer on u, then per-row top-k and (B > 1) unions.
static int sets_from_u(const dv_dims* D, int B, const float* u, const uint16_t* P2, int kN,
                       bool neuron_dense, int kH, bool head_dense, dv_sets* sets, int* st,
                       int ctas, cudaStream_t s) {
  const int ld = D->F + D->h_kv;
  const int row0 = neuron_dense ? D->F : 0;
  const int row1 = head_dense ? D->F : ld;
  if (row1 <= row0) return DV_OK;
  int rc = launch_pred2(u, B, D->r, P2 + (size_t)row0 * D->r, row1 - row0, sets->scores + row0, ld,
                        ctas, s);
  if (rc != DV_OK) return rc;
  // The head set first: the next layer's first kernel needs it, the neuron
  // set only its last.
  if (!head_dense)
    rc = launch_topk(sets->scores + D->F, B, ld, D->h_kv, nullptr, kH, sets->idx_H, kH, st, s);
  if (rc == DV_OK && !neuron_dense)
    rc = launch_topk(sets->scores, B, ld, D->F, nullptr, kN, sets->idx_N, kN, st, s);
  if (rc != DV_OK) return rc;
  if (B > 1 && !neuron_dense) rc = launch_union(sets->idx_N, B, kN, D->F, sets->uN, sets->ucnt, s);
  if (rc == DV_OK && B > 1 && !head_dense)
    rc = launch_union(sets->idx_H, B, kH, D->h_kv, sets->uH, sets->ucnt + 1, s);
  if (rc != DV_OK) return rc;
  return DV_OK;
}

// Predict the sets of one layer from y (both predictor layers, top-k, unions).
static int run_sets(const dv_dims* D, int B, const uint16_t* y, const uint16_t* P1,
                    const uint16_t* P2, int kN, bool neuron_dense, int kH, bool head_dense,
                    int flags, dv_sets* sets, int* st, float* u, int ctas, int ring,
                    cudaStream_t s) {
  if (neuron_dense && head_dense) return DV_OK;
  int rc = launch_pred1(y, B, D->d, P1, D->r, (flags & DV_PRED_RELU) ? 1 : 0, u, ctas, ring, s);
  if (rc != DV_OK) return rc;
  return sets_from_u(D, B, u, P2, kN, neuron_dense, kH, head_dense, sets, st, ctas, s);
}

static int check_weights_attn(const dv_layer_weights* w) {
  REQ(w, DV_ERR_NULL);
  REQ_PTR(w->Wq); REQ_PTR(w->Wk); REQ_PTR(w->Wv); REQ_PTR(w->WoT);
  OPT_PTR(w->ln1_g); OPT_PTR(w->ln1_b);
  return DV_OK;
}

int check_weights_mlp(const dv_layer_weights* w) {
  REQ(w, DV_ERR_NULL);
  REQ_PTR(w->fc1); REQ_PTR(w->fc2T);
  OPT_PTR(w->ln2_g); OPT_PTR(w->ln2_b);
  return DV_OK;
}

static int check_w4(const dv_dims* D, int flags) {
  if (!(flags & DV_W4)) return DV_OK;
  REQ(D->d % 128 == 0, DV_ERR_DIMS);
  return DV_OK;
}

static int check_kv(const dv_dims* D, const dv_kv_cache* kv, int B, int n, int flags) {
  REQ(kv, DV_ERR_NULL);
  REQ_PTR(kv->K); REQ_PTR(kv->V);
  OPT_PTR(kv->y_side);
  REQ(n >= 0 && n < D->n_max, DV_ERR_DIMS);
  if (flags & DV_KV_FILL) {
    REQ_PTR(kv->y_side);
    REQ(kv->kv_missing, DV_ERR_NULL);
    REQ(!(flags & DV_KV_RESELECT), DV_ERR_UNSUPPORTED);
  }
  if (flags & (DV_KV_RETAINED | DV_KV_RESELECT)) {
    REQ(B == 1, DV_ERR_UNSUPPORTED);
    REQ_PTR(kv->Kr); REQ_PTR(kv->Vr);
    REQ(kv->kept_pos && kv->kept_count, DV_ERR_NULL);
    REQ(kv->b_max >= 1, DV_ERR_DIMS);
  }
  return DV_OK;
}

static int launch_status() {
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv

using namespace dv;

extern "C" {

int dv_version(void) { return 100; }

const char* dv_status_string(int status) {
  switch (status) {
    case DV_OK: return "ok";
    case DV_ERR_NULL: return "a required pointer is NULL";
    case DV_ERR_ALIGN: return "a pointer is not 16-byte aligned (workspace: 256)";
    case DV_ERR_DIMS: return "a dimension is out of range or inconsistent";
    case DV_ERR_KEEP: return "a keep ratio is outside (0, 1]";
    case DV_ERR_K: return "k is outside [1, N]";
    case DV_ERR_WORKSPACE: return "workspace smaller than dv_workspace_size()";
    case DV_ERR_LAUNCH: return "a CUDA launch or stream call failed";
    case DV_ERR_UNSUPPORTED: return "shape outside what the kernels implement";
    default: return "unknown status";
  }
}

size_t dv_workspace_size(const dv_dims* dims, int B, int flags) {
  if (check_dims(dims) != DV_OK || B < 1 || B > 4) return 0;
  return ws_layout(dims, B, flags).total;
}

int dv_profile(cudaEvent_t* events, int* tags, int cap) {
  const int n = g_prof_n;
  if (!events || !tags || cap <= 0) {
    g_prof_ev = nullptr;
    g_prof_tags = nullptr;
    g_prof_cap = 0;
    g_prof_n = 0;
    return n;
  }
  g_prof_ev = events;
  g_prof_tags = tags;
  g_prof_cap = cap;
  g_prof_n = 0;
  return DV_OK;
}

long long dv_launch_count(void) { return g_launches; }

int dv_count_active(int* dev_counter) {
  g_count_active = dev_counter;
  return DV_OK;
}

// Tuning knobs for launch shapes (aux; defaults need no call).
int dv_set_tuning(int main_ctas, int side_ctas, int main_ring_kb, int side_ring_kb,
                  int attn_ctas, int pdl, int stage_kb) {
  if (main_ctas < 0 || side_ctas < 0 || main_ring_kb < 16 || main_ring_kb > 200 ||
      side_ring_kb < 8 || side_ring_kb > 200 || attn_ctas < 0 || stage_kb < 4 ||
      stage_kb > 100)
    return DV_ERR_DIMS;
  g_stage_target = stage_kb * 1024;
  g_tune.main_ctas = main_ctas;
  g_tune.side_ctas = side_ctas;
  g_tune.main_ring = main_ring_kb * 1024;
  g_tune.side_ring = side_ring_kb * 1024;
  g_tune.attn_ctas = attn_ctas;
  g_pdl = pdl != 0;
  return DV_OK;
}

int dv_predict(const uint16_t* y, int B, int d, const uint16_t* P1, int r, const uint16_t* P2,
               int N, int flags, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream) {
  REQ_PTR(y); REQ_PTR(P1); REQ_PTR(P2); REQ(scores, DV_ERR_NULL); REQ(ws, DV_ERR_NULL);
  REQ(aligned(ws, 256), DV_ERR_ALIGN);
  REQ(B >= 1 && B <= 4, DV_ERR_DIMS);
  REQ(d >= 8 && d <= 16384 && d % 8 == 0, DV_ERR_DIMS);
  REQ(r >= 8 && r <= 4096 && r % 8 == 0, DV_ERR_DIMS);
  REQ(N >= 1, DV_ERR_DIMS);
  REQ(ws_bytes >= (size_t)B * r * 4, DV_ERR_WORKSPACE);
  return launch_predict(y, B, d, P1, r, P2, N, (flags & DV_PRED_RELU) ? 1 : 0, scores, N,
                        static_cast<float*>(ws), main_ctas(), g_tune.main_ring, stream);
}

int dv_select_topk(const float* scores, int B, int ld, int N, int k, int32_t* idx,
                   int32_t* union_idx, int32_t* union_count, int* dev_status, void* ws,
                   size_t ws_bytes, cudaStream_t stream) {
  (void)ws;
  (void)ws_bytes;
  REQ(scores && idx, DV_ERR_NULL);
  REQ(B >= 1 && B <= 8, DV_ERR_DIMS);
  REQ(N >= 1 && N <= (1 << 24) && ld >= N, DV_ERR_DIMS);
  REQ(k >= 1 && k <= N, DV_ERR_K);
  REQ(!union_idx || union_count, DV_ERR_NULL);
  int rc = launch_topk(scores, B, ld, N, nullptr, k, idx, k, dev_status, stream);
  if (rc == DV_OK && union_idx) rc = launch_union(idx, B, k, N, union_idx, union_count, stream);
  return rc;
}

int dv_sparse_mlp(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                  const int32_t* idx, int k, const int32_t* dev_count, int flags, uint16_t* out,
                  int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  REQ_PTR(x); REQ_PTR(out); REQ(ws, DV_ERR_NULL); REQ(aligned(ws, 256), DV_ERR_ALIGN);
  if ((rc = check_weights_mlp(w)) != DV_OK) return rc;
  if ((rc = check_w4(dims, flags)) != DV_OK) return rc;
  REQ(B >= 1 && B <= 4, DV_ERR_DIMS);
  if (!idx) k = dims->F;
  REQ(k >= 1 && k <= dims->F, DV_ERR_K);
  REQ(x != out, DV_ERR_DIMS);
  const WsLayout L = ws_layout(dims, B, 0);
  REQ(ws_bytes >= L.total, DV_ERR_WORKSPACE);
  return run_mlp(x, B, dims, w, idx, k, dev_count, flags, out, dev_status, ws, L, stream, false);
}

size_t dv_union_mlp_ws_size(int B, int d, int k) {
  if (B < 8 || B > 64 || (B & 7) || B == 24 || B == 40 || B == 48 || B == 56 || d < 64 ||
      d % 64 || k < 1)
    return 0;
  return union_tc_ws_bytes(B, d, k);
}

int dv_union_mlp(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                 const int32_t* union_idx, int k, const int32_t* dev_count, int flags,
                 uint16_t* out, int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  REQ_PTR(x); REQ_PTR(out); REQ(x != out, DV_ERR_DIMS);
  if ((rc = check_weights_mlp(w)) != DV_OK) return rc;
  REQ(union_idx, DV_ERR_NULL);
  REQ(dims->d % 64 == 0, DV_ERR_DIMS);
  REQ(k >= 1 && k <= dims->F, DV_ERR_K);
  const size_t need = dv_union_mlp_ws_size(B, dims->d, k);
  REQ(need > 0, DV_ERR_UNSUPPORTED);
  REQ(ws, DV_ERR_NULL); REQ(aligned(ws, 256), DV_ERR_ALIGN);
  REQ(ws_bytes >= need, DV_ERR_WORKSPACE);
  return launch_union_mlp_tc(x, B, dims->d, dims->F, w->ln2_g, w->ln2_b, dims->ln_eps, w->fc1,
                             w->b1, w->fc2T, w->b2, union_idx, k, dev_count,
                             !(flags & DV_NO_RESIDUAL), out, dev_status, ws, stream);
}

size_t dv_w4_row_bytes(int d) { return (d >= 128 && d % 128 == 0) ? w4_row_bytes_host(d) : 0; }

int dv_quantize_w4(const uint16_t* W, int rows, int d, uint8_t* out, cudaStream_t stream) {
  REQ_PTR(W); REQ_PTR(out);
  REQ(rows >= 1 && rows <= 65535 && d >= 128 && d % 128 == 0 && d <= 16384, DV_ERR_DIMS);
  return launch_quant_w4(W, rows, d, out, stream);
}

int dv_sparse_mlp_w4(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                     const uint8_t* fc1_w4, const uint8_t* fc2T_w4, const int32_t* idx, int k,
                     const int32_t* dev_count, int flags, uint16_t* out, int* dev_status,
                     void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  REQ(dims->d % 128 == 0, DV_ERR_DIMS);
  REQ_PTR(x); REQ_PTR(out); REQ(ws, DV_ERR_NULL); REQ(aligned(ws, 256), DV_ERR_ALIGN);
  REQ(w, DV_ERR_NULL);
  REQ_PTR(fc1_w4); REQ_PTR(fc2T_w4);
  OPT_PTR(w->b1); OPT_PTR(w->b2); OPT_PTR(w->ln2_g); OPT_PTR(w->ln2_b);
  REQ(B >= 1 && B <= 4, DV_ERR_DIMS);
  if (!idx) k = dims->F;
  REQ(k >= 1 && k <= dims->F, DV_ERR_K);
  REQ(x != out, DV_ERR_DIMS);
  const WsLayout L = ws_layout(dims, B, 0);
  REQ(ws_bytes >= L.total, DV_ERR_WORKSPACE);
  return launch_mlp_w4(x, B, dims->d, dims->F, w->ln2_g, w->ln2_b, dims->ln_eps, fc1_w4, w->b1,
                       fc2T_w4, w->b2, idx, k, dev_count,
                       flags & (DV_SKIP_INACTIVE | DV_NO_RESIDUAL), out, dev_status,
                       at<float>(ws, L.part), main_ctas(), g_tune.main_ring, stream, false);
}

int dv_sparse_attn(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                   const int32_t* head_idx, int k_heads, const int32_t* dev_count,
                   dv_kv_cache* kv, int n, float softmax_scale, int flags, uint16_t* out,
                   int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  REQ_PTR(x); REQ_PTR(out); REQ(ws, DV_ERR_NULL); REQ(aligned(ws, 256), DV_ERR_ALIGN);
  if ((rc = check_weights_attn(w)) != DV_OK) return rc;
  if ((rc = check_w4(dims, flags)) != DV_OK) return rc;
  REQ(B >= 1 && B <= 4, DV_ERR_DIMS);
  if ((rc = check_kv(dims, kv, B, n, flags)) != DV_OK) return rc;
  if (!head_idx) k_heads = dims->h_kv;
  REQ(k_heads >= 1 && k_heads <= dims->h_kv, DV_ERR_K);
  REQ(x != out, DV_ERR_DIMS);
  REQ(std::isfinite(softmax_scale), DV_ERR_DIMS);
  const WsLayout L = ws_layout(dims, B, 0);
  REQ(ws_bytes >= L.total, DV_ERR_WORKSPACE);
  return run_attn(x, B, dims, w, head_idx, k_heads, dev_count, kv, n, softmax_scale, flags, out,
                  dev_status, ws, L, stream);
}

int dv_kv_select_attn(const float* q, const dv_dims* dims, dv_kv_cache* kv, int n,
                      const uint16_t* q_obs, int obs_window, int n_sinks, int smooth,
                      float kv_keep, float softmax_scale, int flags, float* H, float* sel_scores,
                      int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  REQ(q && H, DV_ERR_NULL);
  REQ(ws, DV_ERR_NULL);
  REQ(aligned(ws, 256), DV_ERR_ALIGN);
  const bool dense = (flags & DV_KV_DENSE) != 0;
  if ((rc = check_kv(dims, kv, 1, n, dense ? 0 : DV_KV_RETAINED)) != DV_OK) return rc;
  const int G = dims->h / dims->h_kv;
  const bool resel = (flags & DV_KV_RESELECT) != 0;
  const WsLayout L = ws_layout(dims, 1, resel ? DV_KV_RESELECT : 0);
  REQ(ws_bytes >= L.total, DV_ERR_WORKSPACE);
  if (resel && !dense) {
    REQ_PTR(q_obs);
    REQ(obs_window >= 1 && obs_window <= n && G * obs_window <= 512 && (G * obs_window) % 4 == 0,
        DV_ERR_DIMS);
    REQ(n_sinks >= 0 && smooth >= 1 && smooth % 2 == 1, DV_ERR_DIMS);
    REQ(kv_keep > 0.f && kv_keep <= 1.f, DV_ERR_KEEP);
    const int b = (int)std::floor((double)kv_keep * n + 1e-9);
    if (kv_select_ws_floats(dims->h, dims->h_kv, obs_window, n) > L.kvsel_floats)
      return DV_ERR_WORKSPACE;
    rc = launch_kv_select(q_obs, dims->h, dims->h_kv, dims->d_h, obs_window, kv->K, kv->V, n,
                          dims->n_max, softmax_scale, n_sinks, smooth, b, kv->Kr, kv->Vr,
                          kv->kept_pos, kv->kept_count, kv->b_max, sel_scores,
                          at<float>(ws, L.kvsel), L.kvsel_floats, dev_status, stream);
    if (rc != DV_OK) return rc;
  }
  if (!dense) {
    rc = launch_kv_append(kv->K, kv->V, dims->h_kv, dims->d_h, n, dims->n_max, kv->Kr, kv->Vr,
                          kv->kept_count, kv->b_max, stream);
    if (rc != DV_OK) return rc;
  }
  const int max_keys = dense ? n + 1 : kv->b_max;
  SplitPlan plan = split_plan(max_keys, dims->h_kv, 1, attn_ctas());
  if (plan.S > L.S_max) return DV_ERR_WORKSPACE;
  if (cudaMemsetAsync(at<int>(ws, L.cnt), 0, sizeof(int) * dims->h_kv, stream) != cudaSuccess)
    return DV_ERR_LAUNCH;
  rc = launch_splitk(q, 1, dims->d_h, G, dims->h_kv, nullptr, dims->h_kv, nullptr, kv->K, kv->V, n,
                     dims->n_max, kv->Kr, kv->Vr, kv->kept_count, kv->b_max, dense ? 0 : 1, plan,
                     at<float>(ws, L.sk), H, at<int>(ws, L.cnt), dev_status, stream, false);
  if (rc != DV_OK) return rc;
  if (!dense && (flags & DV_KV_ADVANCE))
    rc = launch_kv_advance(kv->kept_count, dims->h_kv, kv->b_max, stream);
  return rc;
}

// One decode layer. With w_next / kv_next (the stacked driver), the missing
// K/V of the next layer are recomputed on the side stream as soon as its
// look-ahead sets exist (*side_filled is set), so that work leaves the main
// stream's path; fill_done says this layer's own recompute already ran there.
static int decode_layer(const dv_dims* dims, const dv_keep* keep, int B, const dv_layer_weights* w,
                        const uint16_t* P1_next, const uint16_t* P2_next, dv_kv_cache* kv, int n,
                        float softmax_scale, dv_sets* cur, dv_sets* next, const uint16_t* y_in,
                        uint16_t* y_out, int flags, int* dev_status, void* ws, size_t ws_bytes,
                        cudaStream_t main, cudaStream_t side, cudaEvent_t ev_fork,
                        cudaEvent_t ev_join, const dv_layer_weights* w_next,
                        dv_kv_cache* kv_next, bool fill_done, bool* side_filled) {
  if (side_filled) *side_filled = false;
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  REQ(keep, DV_ERR_NULL);
  REQ(keep->neuron > 0.f && keep->neuron <= 1.f && keep->head > 0.f && keep->head <= 1.f,
      DV_ERR_KEEP);
  REQ(B >= 1 && B <= 4, DV_ERR_DIMS);
  REQ_PTR(y_in); REQ_PTR(y_out); REQ(y_in != y_out, DV_ERR_DIMS);
  REQ(ws, DV_ERR_NULL); REQ(aligned(ws, 256), DV_ERR_ALIGN);
  if ((rc = check_weights_attn(w)) != DV_OK) return rc;
  if ((rc = check_weights_mlp(w)) != DV_OK) return rc;
  if ((rc = check_w4(dims, flags)) != DV_OK) return rc;
  if ((rc = check_kv(dims, kv, B, n, flags)) != DV_OK) return rc;
  const WsLayout L = ws_layout(dims, B, 0);
  REQ(ws_bytes >= L.total, DV_ERR_WORKSPACE);
  REQ(std::isfinite(softmax_scale), DV_ERR_DIMS);

  const bool nd = keep->neuron >= 1.f, hd = keep->head >= 1.f;
  const int kN = nd ? dims->F : k_from_keep(keep->neuron, dims->F);
  const int kH = hd ? dims->h_kv : k_from_keep(keep->head, dims->h_kv);
  const bool need_pred = !(nd && hd);
  if (need_pred) {
    REQ(dims->r >= 8, DV_ERR_DIMS);
    REQ(cur && cur->scores && cur->idx_N && cur->idx_H, DV_ERR_NULL);
    if (B > 1) REQ(cur->uN && cur->uH && cur->ucnt, DV_ERR_NULL);
  }
  const bool look = (flags & DV_LOOKAHEAD) && P1_next && P2_next && need_pred;
  if (look) {
    REQ(next && next->scores && next->idx_N && next->idx_H, DV_ERR_NULL);
    if (B > 1) REQ(next->uN && next->uH && next->ucnt, DV_ERR_NULL);
    REQ(side && ev_fork && ev_join, DV_ERR_NULL);
    REQ_PTR(P1_next);
    REQ_PTR(P2_next);
  }

  // (the previous layer recorded the join only if it predicted ahead)
  if ((flags & DV_JOIN) && ev_join && need_pred)
    if (cudaStreamWaitEvent(main, ev_join, 0) != cudaSuccess) return DV_ERR_LAUNCH;
  if ((flags & DV_SYNC_PREDICT) && need_pred) {
    REQ_PTR(w->P1); REQ_PTR(w->P2);
    rc = run_sets(dims, B, y_in, w->P1, w->P2, kN, nd, kH, hd, flags, cur, dev_status,
                  at<float>(ws, L.u_main), main_ctas(), g_tune.main_ring, main);
    if (rc != DV_OK) return rc;
  }
  // Attention block: h = y + MHA_{S_A}(y). The QKV kernel also streams the
  // next layer's first predictor layer on y ([DV] 4.3: S^{l+1} <- SP(y_l));
  // the rest of the prediction runs on the side stream alongside this layer.
  const int32_t* selH = hd ? nullptr : (B == 1 ? cur->idx_H : cur->uH);
  const int32_t* cntH = (hd || B == 1) ? nullptr : cur->ucnt + 1;
  const int kHe = (hd || B == 1) ? kH : std::min(dims->h_kv, B * kH);
  uint16_t* hmid = at<uint16_t>(ws, L.hmid);
  // PDL for the QKV kernel only when its index list was not produced by the
  // kernel right before it (a synchronous prediction on this stream).
  const bool pdl_qkv = !((flags & DV_SYNC_PREDICT) && need_pred) && (flags & DV_JOIN);
  // At batch 1 the next layer's P1 rows ride in this QKV launch; at B > 1
  // (the fused form would spill registers) and with 4-bit Q/K/V rows (P1
  // stays fp16) they run on the side stream.
  const bool fuse_p1 = look && B == 1 && !(flags & DV_W4);
  const bool fill_next = look && w_next && kv_next && (flags & DV_KV_FILL);
  if (fill_next) {
    if ((rc = check_kv(dims, kv_next, B, n, flags)) != DV_OK) return rc;
    if ((rc = check_weights_attn(w_next)) != DV_OK) return rc;
  }
  rc = attn_qkv(y_in, B, dims, w, selH, kHe, cntH, kv, n, softmax_scale, flags,
                fuse_p1 ? P1_next : nullptr, at<float>(ws, L.u_side), dev_status, ws, L, main,
                pdl_qkv, fill_done);
  if (rc != DV_OK) return rc;
  if (look) {
    if (cudaEventRecord(ev_fork, main) != cudaSuccess) return DV_ERR_LAUNCH;
    if (cudaStreamWaitEvent(side, ev_fork, 0) != cudaSuccess) return DV_ERR_LAUNCH;
    if (!fuse_p1) {
      rc = launch_pred1_gemv(y_in, B, dims->d, P1_next, dims->r, (flags & DV_PRED_RELU) ? 1 : 0,
                             at<float>(ws, L.u_side), side_ctas(), side);
      if (rc != DV_OK) return rc;
    }
    rc = sets_from_u(dims, B, at<float>(ws, L.u_side), P2_next, kN, nd, kH, hd, next, dev_status,
                     side_ctas(), side);
    if (rc != DV_OK) return rc;
    if (fill_next) {
      // [DV] 4.2 + 4.3: the next layer's missing k, v, from its kept inputs,
      // for the units its look-ahead just selected (small CTAs that fit
      // beside this layer's streaming CTAs).
      const int32_t* selHn = hd ? nullptr : (B == 1 ? next->idx_H : next->uH);
      const int32_t* cntHn = (hd || B == 1) ? nullptr : next->ucnt + 1;
      const bool retn = (flags & DV_KV_RETAINED) != 0;
      rc = launch_kv_fill(kv_next->y_side, kv_next->kv_missing, B, dims->d, dims->h_kv,
                          dims->d_h, w_next->ln1_g, w_next->ln1_b, dims->ln_eps, w_next->Wk,
                          w_next->bk, w_next->Wv, w_next->bv, selHn, kHe, cntHn, kv_next->K,
                          kv_next->V, n, dims->n_max, dev_status, side, false,
                          retn ? kv_next->Kr : nullptr, retn ? kv_next->Vr : nullptr,
                          kv_next->kept_count, kv_next->b_max, (flags & DV_W4) != 0);
      if (rc != DV_OK) return rc;
      if (side_filled) *side_filled = true;
    }
    if (cudaEventRecord(ev_join, side) != cudaSuccess) return DV_ERR_LAUNCH;
  }
  const int32_t* selN = nd ? nullptr : (B == 1 ? cur->idx_N : cur->uN);
  const int32_t* cntN = (nd || B == 1) ? nullptr : cur->ucnt;
  const int kNe = (nd || B == 1) ? kN : std::min(dims->F, B * kN);
  rc = attn_rest(y_in, B, dims, w, selH, kHe, cntH, kv, n, flags, hmid, dev_status, ws, L, main);
  if (rc != DV_OK) return rc;
  // MLP block: y' = h + MLP_{S_M}(h).
  rc = run_mlp(hmid, B, dims, w, selN, kNe, cntN, flags, y_out, dev_status, ws, L, main, true);
  if (rc != DV_OK) return rc;
  return launch_status();
}

int dv_decode_layer(const dv_dims* dims, const dv_keep* keep, int B, const dv_layer_weights* w,
                    const uint16_t* P1_next, const uint16_t* P2_next, dv_kv_cache* kv, int n,
                    float softmax_scale, dv_sets* cur, dv_sets* next, const uint16_t* y_in,
                    uint16_t* y_out, int flags, int* dev_status, void* ws, size_t ws_bytes,
                    cudaStream_t main, cudaStream_t side, cudaEvent_t ev_fork,
                    cudaEvent_t ev_join) {
  return decode_layer(dims, keep, B, w, P1_next, P2_next, kv, n, softmax_scale, cur, next, y_in,
                      y_out, flags, dev_status, ws, ws_bytes, main, side, ev_fork, ev_join,
                      nullptr, nullptr, false, nullptr);
}

int dv_decode_step(const dv_dims* dims, const dv_keep* keep, int B, int L,
                   const dv_layer_weights* w, dv_kv_cache* kv, int n, float softmax_scale,
                   dv_sets* sets, const uint16_t* y_in, uint16_t* y_tmp, uint16_t* y_out, int flags,
                   int* dev_status, void* ws, size_t ws_bytes, cudaStream_t main, cudaStream_t side,
                   cudaEvent_t ev_fork, cudaEvent_t ev_join) {
  REQ(dims && keep && w && kv && sets, DV_ERR_NULL);
  REQ(L >= 1, DV_ERR_DIMS);
  REQ_PTR(y_in); REQ_PTR(y_out);
  if (L > 1) REQ_PTR(y_tmp);
  const bool look = (flags & DV_LOOKAHEAD) != 0;
  const uint16_t* cur_in = y_in;
  bool filled = false;  // this layer's missing K/V were recomputed on the side stream
  for (int l = 0; l < L; ++l) {
    uint16_t* dst = (l == L - 1) ? y_out : y_tmp + (size_t)(l & 1) * B * dims->d;
    int f = flags & ~(DV_SYNC_PREDICT | DV_JOIN | DV_LOOKAHEAD);
    if (l == 0 || !look) f |= DV_SYNC_PREDICT;
    if (look && l > 0) f |= DV_JOIN;
    const bool has_next = look && (l + 1 < L);
    if (has_next) f |= DV_LOOKAHEAD;
    bool filled_next = false;
    int rc = decode_layer(dims, keep, B, &w[l], has_next ? w[l + 1].P1 : nullptr,
                          has_next ? w[l + 1].P2 : nullptr, &kv[l], n, softmax_scale,
                          &sets[l & 1], &sets[(l + 1) & 1], cur_in, dst, f, dev_status, ws,
                          ws_bytes, main, side, ev_fork, ev_join, has_next ? &w[l + 1] : nullptr,
                          has_next ? &kv[l + 1] : nullptr, filled, &filled_next);
    if (rc != DV_OK) return rc;
    filled = filled_next;
    cur_in = dst;
  }
  return DV_OK;
}

}  // extern "C"
