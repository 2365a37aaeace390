// dv_internal.h -- launchers shared between the libdv translation units.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "dv_common.cuh"

namespace dv {

// k_stream.cu ---------------------------------------------------------------
int launch_mlp(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g, const uint16_t* ln_b,
               float eps, const uint16_t* fc1, const uint16_t* b1, const uint16_t* fc2T,
               const uint16_t* b2, const int32_t* idx, int k, const int32_t* dev_count, int flags,
               uint16_t* out, int* st, float* part, int target_ctas, int ring_budget,
               cudaStream_t stream, bool pdl);

int launch_qkv(const uint16_t* x, int B, int d, int G, int dh, int h_kv, const uint16_t* ln_g,
               const uint16_t* ln_b, float eps, const uint16_t* Wq, const uint16_t* bq,
               const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv, const uint16_t* bv,
               const int32_t* idx, int k, const int32_t* dev_count, float scale, float* qbuf,
               uint16_t* K, uint16_t* V, int n, int n_max, uint16_t* Kr, uint16_t* Vr,
               const int32_t* kept_count, int b_max, uint16_t* y_side, uint32_t* kv_missing,
               int fill_clear, int* zero_cnt, int n_zero, const uint16_t* P1, int n_pred,
               int relu, float* u_out, int* st, int target_ctas, int ring_budget,
               cudaStream_t stream, bool pdl, bool w4 = false);

int launch_mlp_w4(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g,
                  const uint16_t* ln_b, float eps, const uint8_t* fc1q, const uint16_t* b1,
                  const uint8_t* fc2Tq, const uint16_t* b2, const int32_t* idx, int k,
                  const int32_t* dev_count, int flags, uint16_t* out, int* st, float* part,
                  int target_ctas, int ring_budget, cudaStream_t stream, bool pdl);

// k_w4.cu ---------------------------------------------------------------------
size_t w4_row_bytes_host(int d);
int launch_quant_w4(const uint16_t* W, int rows, int d, uint8_t* out, cudaStream_t stream);

// k_fill.cu -------------------------------------------------------------------
// Missing K/V of the selected units recomputed from the kept inputs.
int launch_kv_fill(const uint16_t* y_side, const uint32_t* missing, int B, int d, int h_kv,
                   int dh, const uint16_t* ln_g, const uint16_t* ln_b, float eps,
                   const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv,
                   const uint16_t* bv, const int32_t* idx, int k, const int32_t* dev_count,
                   uint16_t* K, uint16_t* V, int n, int n_max, int* st, cudaStream_t stream,
                   bool pdl, uint16_t* Kr = nullptr, uint16_t* Vr = nullptr,
                   const int32_t* kept_count = nullptr, int b_max = 0, bool w4 = false);

int launch_wo(const uint16_t* x, int B, int d, int G, int dh, int h_kv, const uint16_t* WoT,
              const uint16_t* bo, const int32_t* idx, int k, const int32_t* dev_count,
              const float* H, uint16_t* out, int* st, float* part, int target_ctas,
              int ring_budget, cudaStream_t stream, bool w4 = false);

int launch_predict(const uint16_t* y, int B, int d, const uint16_t* P1, int r,
                   const uint16_t* P2, int N, int relu, float* scores, int ld, float* u,
                   int target_ctas, int ring_budget, cudaStream_t stream);

int launch_pred1(const uint16_t* y, int B, int d, const uint16_t* P1, int r, int relu, float* u,
                 int target_ctas, int ring_budget, cudaStream_t stream);

int launch_pred1_gemv(const uint16_t* y, int B, int d, const uint16_t* P1, int r, int relu,
                      float* u, int target_ctas, cudaStream_t stream);
int launch_pred2(const float* u, int B, int r, const uint16_t* P2, int N, float* scores, int ld,
                 int target_ctas, cudaStream_t stream);

size_t stream_part_bytes(int d, int B, long long max_rows, int target_ctas);

// out[b] = fp16(x[b] + bias + sum_g part[g][b]) in a fixed order of g (x, bias
// nullable); programmatic dependent launch on the previous kernel.
int reduce_launch(const float* part, int G, int B, int d, const uint16_t* x, const uint16_t* bias,
                  uint16_t* out, cudaStream_t stream);

// k_attn.cu ------------------------------------------------------------------
struct SplitPlan {
  int C;  // keys per split
  int S;  // splits
};
constexpr int kSplitsMax = 64;  // splits per unit, any plan
SplitPlan split_plan(int max_keys, int units, int B, int target_ctas);

int launch_splitk(const float* q, int B, int dh, int G, int h_kv, const int32_t* idx, int k,
                  const int32_t* dev_count, const uint16_t* K, const uint16_t* V, int n, int n_max,
                  const uint16_t* Kr, const uint16_t* Vr, const int32_t* kept_count, int b_max,
                  int retained, SplitPlan plan, float* part, float* H, int* cnt, int* st,
                  cudaStream_t stream, bool pdl);

int launch_kv_select(const uint16_t* q_obs, int h, int h_kv, int dh, int W, const uint16_t* K,
                     const uint16_t* V, int n, int n_max, float scale, int n_sinks, int smooth,
                     int b, uint16_t* Kr, uint16_t* Vr, int32_t* kept_pos, int32_t* kept_count,
                     int b_max, float* sel_scores, float* ws_f, size_t ws_floats, int* st,
                     cudaStream_t stream);

size_t kv_select_ws_floats(int h, int h_kv, int W, int n);

// k_kvscore_tc.cu: the scoring pass of the KV selection on the tensor cores
// (pooled [h_kv][n]); DV_ERR_UNSUPPORTED for shapes it does not take.
int launch_kv_scores_tc(const uint16_t* q_obs, const uint16_t* K, int h, int h_kv, int dh, int W,
                        int n, int n_max, float scale2, float* stats, size_t stats_floats,
                        float* pooled, int* st, cudaStream_t stream);

int launch_kv_append(const uint16_t* K, const uint16_t* V, int h_kv, int dh, int n, int n_max,
                     uint16_t* Kr, uint16_t* Vr, const int32_t* kept_count, int b_max,
                     cudaStream_t stream);

int launch_kv_advance(int32_t* kept_count, int h_kv, int b_max, cudaStream_t stream);

// k_select.cu ----------------------------------------------------------------
int launch_topk(const float* scores, int B, int ld, int N, const int* k_per_row, int k,
                int32_t* idx, int ld_idx, int* st, cudaStream_t stream);

int launch_union(const int32_t* idx, int B, int k, int N, int32_t* out, int32_t* count,
                 cudaStream_t stream);

extern int g_stage_target;  // bytes per weight-stream ring stage
extern int* g_count_active; // dv_count_active: device counter of streamed fc2^T rows

// Device properties (cached).
int sm_count();

// dv_abi.cu: launch-shape tuning in force (dv_set_tuning) and the host-side
// argument checks the entry points share.
int main_ctas();        // CTAs of a weight-streaming launch
int main_ring_bytes();  // its shared-memory ring budget
int check_dims(const dv_dims* D);
int check_weights_mlp(const dv_layer_weights* w);

// Launch with (pdl) or without a programmatic dependency on the previous
// kernel of the stream.
cudaError_t launch_k(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     void** args, bool pdl, int cluster_x = 0);

// Launch accounting: call with phase 0 just before a kernel launch and phase 1
// just after it (see dv_profile / dv_launch_count).
void note_launch(int tag, int phase, cudaStream_t s);

}  // namespace dv
