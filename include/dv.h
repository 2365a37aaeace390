/*
 * dv.h -- C ABI of libdv.so: the batch-1 decode-step hot path of Deja Vu
 * contextual sparsity on one NVIDIA GB300 (sm_103a), composed with
 * attention-scored KV-token selection.
 *
 * Pages this interface follows:
 *   [DV] "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time"
 *        (arXiv 2310.17157): §2.3 Eq. 1 (sparsified MLP), Eq. 2 (sparsified
 *        MHA) and the keep budget; §4.1 "Design" and §4.2 "Approach"
 *        (predictors); §4.3 (look-ahead); §4.4 and App. D (fused gather +
 *        multiply, W2 and W^O stored transposed); App. C.1 (batch union);
 *        App. C.3 (residual form of a layer).
 *   [BX] "Where Activation Sparsity and KV-Cache Sparsity Cross in LLM
 *        Decoding" (arXiv 2609.33889): §3.2 (branches keep all state),
 *        §4.1 and App. A (attention-scored KV selection, split-K attention);
 *        §3.1-3.3, §5.4, App. D (byte account, latency gate, dispatch).
 *
 * Conventions (every entry point):
 *  - fp16 data are IEEE binary16 bit patterns (uint16_t). Accumulation is fp32.
 *  - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned,
 *    unless stated otherwise. The library allocates no device memory: scratch
 *    comes from the caller's workspace `ws` of at least dv_workspace_size()
 *    bytes (256-byte aligned).
 *  - Every call only enqueues work on the given stream(s) and returns; it
 *    never synchronises the host, so a sequence of calls can be captured in
 *    a CUDA graph.
 *  - Host-side argument errors return a negative dv_status and launch
 *    nothing. Data-dependent device errors (an index out of range, a bounded
 *    wait that gave up, a non-finite score) set bits in the caller's
 *    `dev_status` word (device int, nullable), which the caller reads after
 *    synchronising; the offending element is skipped, never dereferenced.
 *  - Matrices are row-major. Layouts: Wq [h*d_h][d] (row j*d_h+c = dim c of
 *    query head j), Wk / Wv [h_kv*d_h][d], WoT [h*d_h][d] (W^O transposed:
 *    row j*d_h+c = the output weights of dim c of head j), fc1 [F][d]
 *    (neuron j's input weights), fc2T [F][d] (W2 transposed: neuron j's output
 *    weights), P1 [r][d], P2 [F + h_kv][r] (rows 0..F-1 score neurons, rows
 *    F.. score attention units). KV cache K, V [B][h_kv][n_max][d_h].
 *  - An attention "unit" is one KV head with the h/h_kv query heads that read
 *    it; under MHA (h_kv == h) a unit is one head.
 */
#ifndef DV_H
#define DV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (returned) ---------------------------------------- */
#define DV_OK 0
#define DV_ERR_NULL (-1)        /* a required pointer is NULL */
#define DV_ERR_ALIGN (-2)       /* a pointer is not 16-byte aligned (ws: 256) */
#define DV_ERR_DIMS (-3)        /* a dimension is out of range or inconsistent */
#define DV_ERR_KEEP (-4)        /* a keep ratio is outside (0, 1] */
#define DV_ERR_K (-5)           /* k < 1 or k > N */
#define DV_ERR_WORKSPACE (-6)   /* ws_bytes < dv_workspace_size(...) */
#define DV_ERR_LAUNCH (-7)      /* a CUDA launch or stream call failed */
#define DV_ERR_UNSUPPORTED (-8) /* shape outside what the kernels implement */

/* ---- device status bits (written to *dev_status with atomicOr) --------- */
#define DV_DEV_BAD_INDEX 1      /* an index list held a value out of range */
#define DV_DEV_TIMEOUT 2        /* a bounded wait inside a kernel gave up */
#define DV_DEV_NONFINITE 4      /* a non-finite score reached top-k */

/* ---- flags ------------------------------------------------------------- */
#define DV_PRED_RELU (1u << 0)     /* ReLU between the two predictor layers */
#define DV_SKIP_INACTIVE (1u << 1) /* MLP: skip fc2T rows with a_j <= 0 (exact) */
#define DV_LOOKAHEAD (1u << 2)     /* driver: predict layer l+1 on the side stream */
#define DV_SYNC_PREDICT (1u << 3)  /* driver: predict this layer's sets from y first */
#define DV_KV_RESELECT (1u << 4)   /* KV: run the scoring pass, rebuild the retained set */
#define DV_KV_DENSE (1u << 5)      /* attention reads the full cache */
#define DV_KV_RETAINED (1u << 6)   /* attention reads the retained KV buffer */
#define DV_KV_ADVANCE (1u << 7)    /* retained counts grow by one after the step */
#define DV_JOIN (1u << 8)          /* driver: main waits for the previous side work */
#define DV_NO_RESIDUAL (1u << 9)   /* MLP / attention block: out = block output, without
                                      the residual x (the parallel form of [DV] App. C.3,
                                      y + MHA(y) + MLP(y), sums block outputs) */
#define DV_KV_FILL (1u << 10)      /* attention: first recompute the missing k, v of the
                                      selected units from y_side ([DV] §4.2) */
#define DV_W4 (1u << 11)           /* the layer's Wq, Wk, Wv, WoT, fc1, fc2T point to packed
                                      4-bit rows (dv_quantize_w4; [DV] §5.2, Table 7
                                      W4A16); P1, P2 stay fp16; d % 128 == 0; with
                                      DV_KV_FILL the recompute reads the 4-bit W^K, W^V */

/* ---- shapes ------------------------------------------------------------ */
typedef struct {
  int d;        /* model dim; multiple of 8, 8 <= d <= 16384 */
  int h;        /* query heads */
  int h_kv;     /* KV heads; h % h_kv == 0 (h_kv == h: MHA) */
  int d_h;      /* head dim: 64 or 128; h * d_h need not equal d */
  int F;        /* FFN width (neurons), >= 1 */
  int r;        /* predictor rank; multiple of 8, <= 4096 */
  int n_max;    /* KV cache capacity per KV head, tokens */
  float ln_eps; /* LayerNorm epsilon (1e-5 for OPT) */
} dv_dims;

/* Keep ratios ([DV] §2.3: |S| <= (1 - sparsity) N, so k = max(1, floor(keep N))).
 * keep == 1 skips prediction and selection for that segment (all selected). */
typedef struct {
  float neuron; /* MLP neurons */
  float head;   /* attention units */
  float kv;     /* KV tokens ([BX] App. A budget b = floor(n kv) per KV head) */
} dv_keep;

/* One layer's weights. Bias and LayerNorm pointers are nullable (0 bias,
 * gain 1, shift 0). P1 / P2 are this layer's predictor. */
typedef struct {
  const uint16_t *ln1_g, *ln1_b; /* [d] */
  const uint16_t *Wq, *bq;       /* [h*d_h][d], [h*d_h] */
  const uint16_t *Wk, *bk;       /* [h_kv*d_h][d], [h_kv*d_h] */
  const uint16_t *Wv, *bv;       /* [h_kv*d_h][d], [h_kv*d_h] */
  const uint16_t *WoT, *bo;      /* [h*d_h][d], [d] */
  const uint16_t *ln2_g, *ln2_b; /* [d] */
  const uint16_t *fc1, *b1;      /* [F][d], [F] */
  const uint16_t *fc2T, *b2;     /* [F][d], [d] */
  const uint16_t *P1, *P2;       /* [r][d], [F + h_kv][r] */
} dv_layer_weights;

/* One layer's KV state ([BX] §3.2: the full cache stays allocated and keeps
 * receiving entries; the retained buffer is read instead of it). */
typedef struct {
  uint16_t *K, *V;      /* [B][h_kv][n_max][d_h]; slot n receives the new token */
  uint16_t *y_side;     /* [B][n_max][d] nullable: copy of y per token ([DV] §4.2) */
  uint32_t *kv_missing; /* [B][n_max][(h_kv+31)/32] nullable: bit u set = unit u's
                           k, v were not computed for that token ([DV] §4.2) */
  uint16_t *Kr, *Vr;    /* [h_kv][b_max][d_h] nullable: retained KV (batch 1) */
  int32_t *kept_pos;    /* [h_kv][b_max]: cache position of each retained row */
  int32_t *kept_count;  /* [h_kv] device: retained rows before the new token */
  int b_max;            /* retained capacity per KV head */
} dv_kv_cache;

/* Index sets of one layer. Per-row sets are ascending. */
typedef struct {
  int32_t *idx_N; /* [B][k_N] neuron sets */
  int32_t *idx_H; /* [B][k_H] attention-unit sets */
  int32_t *uN;    /* [F] union of the B neuron sets (B > 1), ascending */
  int32_t *uH;    /* [h_kv] union of the B unit sets (B > 1), ascending */
  int32_t *ucnt;  /* [2] device: |uN|, |uH| */
  float *scores;  /* [B][F + h_kv] predictor scores */
} dv_sets;

/* ---- aux ----------------------------------------------------------------- */

/* Library version (major * 10000 + minor * 100 + patch). */
int dv_version(void);

/* Human-readable text of a dv_status code; never NULL. */
const char* dv_status_string(int status);

/* Workspace bytes any entry point below needs for these shapes at batch B,
 * with n_max from dims (split-K partials and KV scoring buffers scale with
 * it). One workspace of this size serves every entry point and the driver. */
size_t dv_workspace_size(const dv_dims* dims, int B, int flags);

/* Launch-shape tuning (aux, process-wide; the defaults need no call): CTAs of
 * the weight-streaming kernels (0: one per SM), CTAs of the side-stream
 * predictor (0: two per SM), shared-memory ring budgets in KB (main 16..200, side
 * 8..200), split-K CTA target (0: two per SM), whether consecutive kernels
 * of one call use programmatic dependent launch (pdl != 0, the default: the
 * next kernel's weight stream starts while the previous kernel drains), and the
 * target size in KB of one weight-stream ring stage (4..100; rows are grouped
 * up to it). DV_OK or DV_ERR_DIMS. */
int dv_set_tuning(int main_ctas, int side_ctas, int main_ring_kb, int side_ring_kb,
                  int attn_ctas, int pdl, int stage_kb);

/* Kernel-launch accounting (aux). dv_profile(events, tags, cap): from now on
 * every kernel launch of the library is bracketed by two cudaEventRecord calls
 * on its stream, using events[2i] (before) and events[2i+1] (after) of the
 * caller's timing-enabled events, and tags[i] receives the kernel kind
 * (DV_TAG_*), until cap pairs are used; works inside stream capture (the
 * records become graph nodes). dv_profile(NULL, NULL, 0) stops and returns the
 * number of pairs recorded. dv_launch_count() is the number of kernels this
 * process has launched through the library (captured launches count once). */
#define DV_TAG_QKV 0
#define DV_TAG_SPLITK 1
#define DV_TAG_WO 2
#define DV_TAG_REDUCE 3
#define DV_TAG_MLP 4
#define DV_TAG_PRED1 5
#define DV_TAG_PRED2 6
#define DV_TAG_TOPK 7
#define DV_TAG_UNION 8
#define DV_TAG_COMBINE 9
#define DV_TAG_KVSEL 10
#define DV_TAG_KVAPPEND 11
#define DV_TAG_KVADVANCE 12
#define DV_TAG_KVFILL 13
int dv_profile(cudaEvent_t* events, int* tags, int cap);
long long dv_launch_count(void);

/* Bytes actually read with DV_SKIP_INACTIVE (aux, process-wide): from now on
 * every MLP launch with DV_SKIP_INACTIVE adds to *dev_counter (a device int,
 * atomically; works inside stream capture, where the pointer is baked into
 * the launch) the number of fc2T rows it streamed, i.e. the selected neurons
 * whose activation is above zero. dv_count_active(NULL) stops. Always DV_OK. */
int dv_count_active(int* dev_counter);

/* ---- a2: predictor ([DV] §4.1 "Design", §4.2 "Approach") ------------------
 * scores[b][i] = sum_j act(sum_c y[b][c] P1[j][c]) * P2[i][j] for i < N,
 * act = identity, or ReLU with DV_PRED_RELU. y [B][d] fp16 is the layer input
 * y_l ([DV] §4.3); P2 points at the first row to score (e.g. P2 + F*r for the
 * head rows only). scores [B][N] fp32. B <= 4. ws holds the rank-r vector. */
int dv_predict(const uint16_t* y, int B, int d, const uint16_t* P1, int r, const uint16_t* P2,
               int N, int flags, float* scores, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a3: top-k selection ([DV] §2.3 budget, §4.1; App. C.1 union) ---------
 * For each row b < B: the k largest of scores[b*ld + 0 .. b*ld + N-1]; equal
 * scores go to the lower index, -0 equals +0; idx[b][0..k-1] ascending.
 * If union_idx != NULL: the ascending union of the B sets is written to
 * union_idx[0..c-1] and c to *union_count (device int). A NaN score sets
 * DV_DEV_NONFINITE. B <= 8, N <= 1 << 24. No workspace is needed. */
int dv_select_topk(const float* scores, int B, int ld, int N, int k, int32_t* idx,
                   int32_t* union_idx, int32_t* union_count, int* dev_status, void* ws,
                   size_t ws_bytes, cudaStream_t stream);

/* ---- a4: gather-fused sparse MLP ([DV] §2.3 Eq. 1, §4.4, App. D) ----------
 * out[b] = x[b] + sum_{j in S} relu(LN2(x[b]) . fc1[j] + b1[j]) fc2T[j] + b2,
 * S = idx[0..k-1] (shared by the B rows: for B > 1 pass the union), or, if
 * dev_count != NULL, idx[0..*dev_count-1] with *dev_count <= k read on the
 * device; idx == NULL means all F neurons (dense). Indices must be distinct
 * and in [0, F); one out of range is skipped and sets DV_DEV_BAD_INDEX.
 * x, out [B][d] fp16 (may not alias). B <= 4.
 * flags: DV_SKIP_INACTIVE, DV_NO_RESIDUAL (out = MLP(x) only). */
int dv_sparse_mlp(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                  const int32_t* idx, int k, const int32_t* dev_count, int flags, uint16_t* out,
                  int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream);

/* dv_sparse_mlp without a workspace, for callers that cannot allocate device
 * memory (a plugin inside a serving engine that owns all device memory, code
 * that must not allocate after start-up, a latency path that cannot take
 * cudaMalloc's synchronisation). The pages have no counterpart: this is a
 * deployment convenience. Same arguments, checks and result as dv_sparse_mlp
 * with fp16 rows, minus ws / ws_bytes (launch tuning from dv_set_tuning
 * applies the same way): the per-CTA partial sums live in a fixed 8 MiB array
 * inside the library, held on every device that loads it until the process
 * exits. The call allocates nothing. Its first call on a device looks the
 * array's device address up; make that first call before any stream capture.
 * Calls that overlap on the GPU share the array and race. Returns
 * DV_ERR_UNSUPPORTED for DV_W4 (packed 4-bit rows are not served here) and
 * DV_ERR_WORKSPACE when B * d fp32 partial sums per CTA cannot fit the array
 * at a launch that keeps at most 256 selected rows per CTA. */
int dv_sparse_mlp_noalloc(const uint16_t* x, int B, const dv_dims* dims,
                          const dv_layer_weights* w, const int32_t* idx, int k,
                          const int32_t* dev_count, int flags, uint16_t* out, int* dev_status,
                          cudaStream_t stream);

/* ---- batched union MLP on the tensor cores ([DV] §5.2, App. C.1) ------------
 * For a batch of B = 8, 16, 32 or 64 sequences sharing one union U of their
 * neuron sets (union_idx[0..k-1], or *dev_count of them, distinct, in [0, F)):
 * out[b] = x[b] + sum_{j in U} relu(LN2(x[b]) . fc1[j] + b1[j]) fc2T[j] + b2,
 * as two dense contractions on the fifth-generation tensor cores (tcgen05,
 * accumulators in TMEM; the union rows gathered into shared memory by TMA;
 * fp16 operands: LN2(x) and the activations rounded to fp16; fp32
 * accumulation, partial sums added in a fixed order). x, out [B][d] fp16,
 * d % 64 == 0, d >= 64. An entry of the union outside [0, F) sets
 * DV_DEV_BAD_INDEX and adds nothing. ws: dv_union_mlp_ws_size(B, d, k) bytes
 * (0 = unsupported shape); it holds LN2(x), the activations and partial sums.
 * flags: DV_NO_RESIDUAL. Errors as dv_sparse_mlp, DV_ERR_UNSUPPORTED for
 * another B. */
size_t dv_union_mlp_ws_size(int B, int d, int k);
int dv_union_mlp(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                 const int32_t* union_idx, int k, const int32_t* dev_count, int flags,
                 uint16_t* out, int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- W4A16: 4-bit weight rows for the sparse MLP ([DV] §5.2, Table 7) ------
 * The pages name no format; this library's: groups of DV_W4_GROUP = 128
 * columns of a row, scale s = fp16(max |w| / 7) (fp32 division), code
 * q = clamp(rint(w / s), -8, 7) (fp32 division, ties to even; a zero group
 * has s = 0, q = 0), weight q s. Packed row: d/2 bytes of codes (column 2i in
 * the low nibble of byte i, stored as q + 8), the d/128 fp16 scales, then zero
 * bytes up to dv_w4_row_bytes(d) (a multiple of 16). */
#define DV_W4_GROUP 128

/* Bytes of one packed row (0 unless d is a positive multiple of 128). Host. */
size_t dv_w4_row_bytes(int d);

/* Quantize rows W [rows][d] fp16 (finite values) into out [rows][dv_w4_row_bytes(d)]
 * (device, 16-byte aligned). 128 <= d <= 16384, d % 128 == 0, rows <= 65535.
 * Enqueued on stream. DV_OK, DV_ERR_NULL, DV_ERR_ALIGN, DV_ERR_DIMS. */
int dv_quantize_w4(const uint16_t* W, int rows, int d, uint8_t* out, cudaStream_t stream);

/* dv_sparse_mlp with packed 4-bit rows: fc1_w4 [F][row] and fc2T_w4 [F][row]
 * (row = dv_w4_row_bytes(d)) replace w->fc1 and w->fc2T (ignored); the
 * activations stay fp16 and LN2, b1, b2 come from w:
 * out[b] = x[b] + sum_{j in S} relu(LN2(x[b]) . (q s)1_j + b1[j]) (q s)2_j + b2,
 * accumulated in fp32. d % 128 == 0. Other arguments, flags and errors as
 * dv_sparse_mlp; the workspace is dv_workspace_size(dims, B, 0). */
int dv_sparse_mlp_w4(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                     const uint8_t* fc1_w4, const uint8_t* fc2T_w4, const int32_t* idx, int k,
                     const int32_t* dev_count, int flags, uint16_t* out, int* dev_status,
                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a5-a7: head-sparse attention block ([DV] §2.3 Eq. 2, §4.2, §4.4) ------
 * For each selected unit u in head_idx[0..k_heads-1] (or *dev_count of them;
 * head_idx == NULL: all h_kv units): project z = LN1(x[b]) to q (every query
 * head of u, scaled by softmax_scale), k and v of u (+ biases); write k, v as
 * fp16 to K/V[b][u][n]; attend over cache positions 0..n (n cached tokens
 * plus the new one) with split-K flash-decoding and a separate combine; then
 * out[b] = x[b] + sum_{query heads j of selected units} H_j WoT_j + bo.
 * Unselected units get no k, v at slot n: their kv_missing bit is set and
 * y_side[b][n] = x[b] (when those pointers are given).
 * With DV_KV_FILL (y_side and kv_missing required; not with DV_KV_RESELECT):
 * before the step reads the cache, every selected unit u
 * gets, for each position t < n whose kv_missing bit of u is set, k and v
 * recomputed from the kept input: z = LN1(y_side[b][t]), K[b][u][t] =
 * fp16(z W^K_u^T + bk_u), V likewise ([DV] §4.2: load the stored embeddings
 * and compute the missing keys and values); the bits are then cleared. A
 * unit's set bits must form a suffix t0..n-1 of the positions, which holds
 * when every step since the cache was complete ran with DV_KV_FILL (a step
 * that selects a unit fills all of its holes). With DV_KV_RETAINED as well, a
 * recomputed position t at or after the selection's context also goes to its
 * retained slot kept_count[u] - (n - t) (every step since the selection ran
 * with DV_KV_ADVANCE, so the decoded tokens follow the kept rows in order).
 * With DV_KV_RETAINED (batch 1): the new k, v also go to Kr/Vr[u][kept_count[u]]
 * and attention reads Kr/Vr[u][0..kept_count[u]] instead of the cache; with
 * DV_KV_ADVANCE the kept counts then grow by one.
 * 0 <= n < n_max. x, out [B][d]. B <= 4. DV_NO_RESIDUAL: out = MHA(x) only. */
int dv_sparse_attn(const uint16_t* x, int B, const dv_dims* dims, const dv_layer_weights* w,
                   const int32_t* head_idx, int k_heads, const int32_t* dev_count,
                   dv_kv_cache* kv, int n, float softmax_scale, int flags, uint16_t* out,
                   int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a8-a9: attention-scored KV selection + split-K attention --------------
 * ([BX] §4.1, App. A.) Batch 1. q [h][d_h] fp32: the new token's queries,
 * already projected and scaled; the new token's k, v are already in K/V[u][n].
 * With DV_KV_RESELECT: the observation window is the last W = obs_window
 * cached positions n-W..n-1 with queries q_obs [h][W][d_h] fp16; every
 * window query t attends causally to positions <= n-W+t (scores scaled by
 * softmax_scale); the softmax probabilities are summed over the window and
 * over the query heads of each KV head, smoothed by a centred width-`smooth`
 * mean (zero padded, divided by smooth); the positions 0..n_sinks-1 and the
 * window are forced, and the remaining budget b - forced (b = floor(n kv_keep))
 * is filled by the highest smoothed scores (ties to the lower position).
 * The kept positions, ascending, go to kept_pos[u][*], their count to
 * kept_count[u], and their K, V rows to Kr/Vr[u][*] (b <= b_max - 1).
 * Every call then appends K/V[u][n] at Kr/Vr[u][kept_count[u]] and computes
 * H[j] = attention of q[j] over Kr/Vr[u][0..kept_count[u]] (or, with
 * DV_KV_DENSE, over K/V[u][0..n]) by split-K and combine. H [h][d_h] fp32.
 * sel_scores [h_kv][n] fp32 (nullable) receives the smoothed scores. */
int dv_kv_select_attn(const float* q, const dv_dims* dims, dv_kv_cache* kv, int n,
                      const uint16_t* q_obs, int obs_window, int n_sinks, int smooth,
                      float kv_keep, float softmax_scale, int flags, float* H, float* sel_scores,
                      int* dev_status, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ---- a1 + a10: one decode layer with look-ahead ([DV] §4.3, App. C.3) --------
 * y_out = h + MLP_{S_M}(h), h = y_in + MHA_{S_A}(y_in), with S_A, S_M taken
 * from cur (per-row sets; for B > 1 their unions, [DV] App. C.1).
 * DV_SYNC_PREDICT: first compute cur from y_in with this layer's P1/P2 on
 *   `main` (used for layer 0 and for sync mode).
 * DV_LOOKAHEAD: record ev_fork on `main` once y_in is ready, and on `side`
 *   compute next (the sets of layer l+1) from y_in with P1_next / P2_next,
 *   then record ev_join ([DV] §4.3: S^{l+1} <- SP(y_l), in parallel with
 *   layer l). DV_JOIN: `main` first waits on ev_join (pass it for every layer
 *   after one that looked ahead).
 * keep->head == 1 uses all units; keep->neuron == 1 all neurons.
 * DV_KV_RETAINED / DV_KV_ADVANCE as in dv_sparse_attn. y_in, y_out [B][d]. */
int dv_decode_layer(const dv_dims* dims, const dv_keep* keep, int B, const dv_layer_weights* w,
                    const uint16_t* P1_next, const uint16_t* P2_next, dv_kv_cache* kv, int n,
                    float softmax_scale, dv_sets* cur, dv_sets* next, const uint16_t* y_in,
                    uint16_t* y_out, int flags, int* dev_status, void* ws, size_t ws_bytes,
                    cudaStream_t main, cudaStream_t side, cudaEvent_t ev_fork,
                    cudaEvent_t ev_join);

/* One decode step over L stacked layers: layer 0 predicts synchronously, each
 * layer l looks ahead for l+1 on `side` (when flags has DV_LOOKAHEAD), layer l
 * reads the sets written by layer l-1's look-ahead. sets[0], sets[1] are used
 * alternately. y_tmp [2][B][d] holds the intermediate layer outputs.
 * y_out = layer L-1's output. Same stream / event rules as above. */
int dv_decode_step(const dv_dims* dims, const dv_keep* keep, int B, int L,
                   const dv_layer_weights* w /* [L], host array */,
                   dv_kv_cache* kv /* [L], host array */, int n, float softmax_scale,
                   dv_sets* sets /* [2], host array */, const uint16_t* y_in, uint16_t* y_tmp,
                   uint16_t* y_out, int flags, int* dev_status, void* ws, size_t ws_bytes,
                   cudaStream_t main, cudaStream_t side, cudaEvent_t ev_fork,
                   cudaEvent_t ev_join);

/* ---- latency gate: choose the decode mode per request --------------------
 * ([BX] §3.1-3.3, §5.4, App. D, App. I; [DV] §2.3 Eq. 1-2, §4.1, App. C.1.)
 * Host-only: these take host pointers, make no CUDA call and can run on a
 * machine without a GPU. A step of one layer over B sequences with n cached
 * tokens each reads, in fp16 bytes:
 *   weights  U_H (2 G d_h + 2 d_h) d 2 + U_N 2 d 2      (G = h / h_kv)
 *   KV       B U_H 2 d_h (t + 1) 2                       (the new token's row included)
 *   predictor r (d + rows) 2, rows = F [keep->neuron < 1] + h_kv [keep->head < 1]
 * where the modes take
 *   DENSE     U_N = F, U_H = h_kv, t = n, no predictor;
 *   ACT       U_N, U_H = the selected counts k = max(1, floor(keep N)) (B = 1)
 *             or the union of the B sets (B > 1), t = n, the predictor;
 *   KV        U_N = F, U_H = h_kv, t = keep->kv n (or min(n, kv_budget));
 *   COMPOSED  ACT's rows and predictor with KV's t.
 * n and t are real numbers here (t is not floored), so times and crossings are
 * continuous in n. Per-layer time of one step in mode m at context n ([BX]
 * App. D): T_m(n) = D(n) bytes_m(n) / bytes_DENSE(n) + c_m(n)
 *                   [+ s(n) / steps for KV and COMPOSED: the scoring pass, run
 *                    once per request, spread over its decode steps]
 * with D the dense time interpolated piecewise-linearly in (log n, log D)
 * through the sweep contexts (the end segments extended beyond them), and the
 * kernel costs c_m and scoring times s interpolated piecewise-linearly in n
 * (held at the end values beyond them). */
#define DV_MODE_DENSE 0    /* every weight row, the full cache */
#define DV_MODE_ACT 1      /* projection branch: selected neurons / units, full cache */
#define DV_MODE_KV 2       /* every weight row, the retained KV */
#define DV_MODE_COMPOSED 3 /* selected rows and the retained KV */
#define DV_PLAN_MAX_CTX 16

typedef struct {
  int B;          /* sequences decoded together, >= 1 */
  int steps;      /* decode steps the request runs, >= 1 */
  int union_N;    /* B > 1: |union of the B neuron sets|, 0..F; 0 = independent
                     uniform draws: F (1 - (1 - k_N / F)^B) */
  int union_H;    /* B > 1: the same for attention units, 0..h_kv */
  int kv_budget;  /* > 0: a fixed budget, t = min(n, kv_budget) ([BX] §3.3:
                     r_KV = b / n); 0: t = keep->kv n */
  unsigned modes; /* admitted modes (quality admissibility, [BX] §6): bit m
                     admits mode m; 0 admits all four */
} dv_request;

typedef struct {
  int n_ctx;                          /* sweep contexts, 2..DV_PLAN_MAX_CTX */
  double ctx[DV_PLAN_MAX_CTX];        /* strictly ascending, > 0 */
  double dense_us[DV_PLAN_MAX_CTX];   /* DENSE layer time at ctx[i], > 0 */
  double cost_us[4][DV_PLAN_MAX_CTX]; /* c_m at ctx[i], µs (c_DENSE = 0) */
  double select_us[DV_PLAN_MAX_CTX];  /* one layer's scoring pass at ctx[i], >= 0 */
} dv_cost_model;

typedef struct {
  double bytes[4]; /* bytes_m(n) of one layer's step */
  double us[4];    /* T_m(n), µs per layer per step */
  int choice;      /* the admitted mode with the lowest T_m (ties: the lower
                      mode number); KV and COMPOSED are admitted only for
                      B == 1, the batch the retained buffers serve */
} dv_plan;

/* bytes[m] = bytes_m(n) of one layer's step for the four modes (n >= 0).
 * DV_OK, DV_ERR_NULL, DV_ERR_DIMS (d, h, h_kv, d_h, F >= 1, h % h_kv == 0,
 * r >= 0; B, steps >= 1; unions in range; kv_budget >= 0; n finite),
 * DV_ERR_KEEP (a keep ratio outside (0, 1]). */
int dv_plan_bytes(const dv_dims* dims, const dv_keep* keep, const dv_request* req, double n,
                  double bytes[4]);

/* Fit the kernel costs of a sweep ([BX] App. D): measured_us [4][n_ctx] holds
 * each mode's measured layer time at ctx[i] (row DV_MODE_DENSE = the dense
 * times); out->cost_us[m][i] = measured_us[m][i] - measured_us[0][i]
 * bytes_m(ctx[i]) / bytes_DENSE(ctx[i]); select_us [n_ctx] (nullable: 0) is
 * copied. All host arrays. Errors as dv_plan_bytes, plus DV_ERR_DIMS for
 * n_ctx outside 2..DV_PLAN_MAX_CTX, contexts not ascending or <= 0, a dense
 * time <= 0, a negative scoring time or a non-finite value. */
int dv_cost_calibrate(const dv_dims* dims, const dv_keep* keep, const dv_request* req, int n_ctx,
                      const double* ctx, const double* measured_us, const double* select_us,
                      dv_cost_model* out);

/* Predict T_m(n) for the four modes at context n > 0 and choose the fastest
 * admitted one. DV_ERR_UNSUPPORTED if no admitted mode can run (KV-only
 * admission at B > 1); other errors as dv_cost_calibrate. */
int dv_plan_decode(const dv_dims* dims, const dv_keep* keep, const dv_request* req,
                   const dv_cost_model* cm, double n, dv_plan* out);

/* The first context in [n_lo, n_hi] (0 < n_lo < n_hi) where modes a and b take
 * equal predicted time, T_a(n) = T_b(n) ([BX] App. D: solve for equal branch
 * latency), to a relative 1e-12; *n_star = -1 if T_a - T_b keeps its sign over
 * the range. A root is bracketed on 8192 log-spaced points, then bisected, so
 * two crossings closer than that spacing can be missed. Errors as
 * dv_plan_decode, DV_ERR_DIMS for a mode outside 0..3 or a == b. */
int dv_plan_crossing(const dv_dims* dims, const dv_keep* keep, const dv_request* req,
                     const dv_cost_model* cm, int mode_a, int mode_b, double n_lo, double n_hi,
                     double* n_star);

#ifdef __cplusplus
}
#endif

#endif /* DV_H */
