// k_stream.cu -- weight-streaming kernels of the decode step (sm_103a).
//
// One engine serves every weight-bound step: a CTA owns a contiguous slice of
// the selected rows of a matrix whose rows are contiguous in memory (fc1 and
// fc2^T rows are neurons, Wq/Wk/Wv and Wo^T rows are head dims, P1 rows are
// predictor units; "Deja Vu", §4.4 / App. D: W2 and W^O stored transposed so
// that a selected neuron or head is one contiguous read). One elected thread
// of a producer warp streams those rows into a ring of shared-memory stages
// with 1-D TMA bulk copies (cp.async.bulk + mbarrier complete_tx, L2
// evict-first); the consumer warps spread every row across the whole CTA, so
// each thread keeps its columns of the activation vector in registers:
//   dot phase   value[row] = z . W[row]           (fc1, QKV, P1)
//   axpy phase  acc       += coef[row] * W[row]   (fc2^T, Wo^T)
// The fused MLP runs both phases in one CTA: the producer keeps streaming fc2^T
// rows while the consumers reduce the fc1 dots, so the pipeline never drains
// between the two ("Deja Vu", §4.4 kernel fusion). Cross-CTA sums go through
// fp32 partials in the workspace and a fixed-order reduce kernel, so results
// are deterministic.
#include "dv_internal.h"

namespace dv {

// ---------------------------------------------------------------------------
// Shared-memory layout of a streaming CTA
// ---------------------------------------------------------------------------
struct StreamGeom {
  int T;             // consumer threads (multiple of 32)
  int R;             // rows per stage
  int NS;            // stages
  uint32_t row_bytes;
  uint32_t stage_bytes;
  int CH;            // max rows per CTA
  int B;
  // byte offsets
  uint32_t off_bar, off_red, off_coef, off_ln, off_list, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Rows per ring stage a consumer holds in registers: at most 8 vectors of 16 B.
__host__ __device__ constexpr int rows_max(int V) { return V >= 8 ? 1 : 8 / V; }

// `dot`: the launch has a dot phase (its per-warp row sums need `red`; a
// Wo launch has none, and the smaller footprint lets one split-K CTA share
// the SM with it).
__host__ __device__ inline void stream_layout(StreamGeom& g, bool dot = true) {
  const int nwc = g.T / 32;
  uint32_t off = g.NS * g.stage_bytes;
  off = align_up(off, 16);
  g.off_bar = off;
  off += (2 * g.NS + 2) * 8;
  off = align_up(off, 16);
  g.off_red = off;
  if (dot) off += g.CH * g.B * nwc * 4;
  g.off_coef = off;
  off += g.B * g.CH * 4;
  g.off_ln = off;
  off += g.B * nwc * 2 * 4 + g.B * 2 * 4;
  g.off_list = off;
  off += (g.CH + 4) * 4;
  g.total = align_up(off, 128);
}

// ---------------------------------------------------------------------------
// Kernel parameters
// ---------------------------------------------------------------------------
enum StreamKind { KIND_MLP = 0, KIND_QKV = 1, KIND_P1 = 2, KIND_WO = 3, KIND_MLP4 = 4,
                  KIND_QKV4 = 5, KIND_WO4 = 6 };
// KIND_MLP4: the MLP with 4-bit weight rows ("Deja Vu" §5.2, Table 7: W4A16).
// A packed row holds d/2 bytes of codes (column 2i in the low nibble of byte
// i, code + 8), then the d/128 fp16 group scales, padded to 16 bytes.
__host__ __device__ constexpr bool is_mlp(int k) { return k == KIND_MLP || k == KIND_MLP4; }
__host__ __device__ constexpr bool is_qkv(int k) { return k == KIND_QKV || k == KIND_QKV4; }
__host__ __device__ constexpr bool is_wo(int k) { return k == KIND_WO || k == KIND_WO4; }
// Kinds whose rows are 4-bit packed rows (the Q/K/V and Wo kinds carry no
// fused predictor rows: the predictor stays fp16).
__host__ __device__ constexpr bool is_w4(int k) {
  return k == KIND_MLP4 || k == KIND_QKV4 || k == KIND_WO4;
}
constexpr int kW4StageRows = 8;  // rows per ring stage for 4-bit rows
constexpr int kW4Ilp = 4;        // 4-bit rows a consumer works on at once
constexpr int kW4Threads = 768;  // consumer threads at B = 1 (24 warps + the producer)
__host__ __device__ inline uint32_t w4_row_bytes(int d) { return (uint32_t)((d / 2 + d / 64 + 15) / 16 * 16); }

// The 8 codes of one 32-bit word (q = nibble - 8) as exact fp16 pairs:
// h[k] = {q_k, q_{k+4}}. Nibbles k and k + 4 sit 16 bits apart, so one mask
// puts a pair into the two halves of a half2: w & 0x000F000F | 0x6400.. reads
// as 1024 + n (minus 1032 gives q), w & 0x00F000F0 | 0x6400.. as 1024 + 16 n
// (times 1/16 minus 72 gives q, exact in one fused multiply-add); the same on
// w >> 8 gives codes 2, 6 and 3, 7.
DV_DEV void w4_decode_h2(uint32_t w, __half2* h) {
  const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 s16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
  const __half2 off16 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
  const uint32_t w8 = w >> 8;
  const uint32_t b0 = (w & 0x000F000Fu) | 0x64006400u;
  const uint32_t b1 = (w & 0x00F000F0u) | 0x64006400u;
  const uint32_t b2 = (w8 & 0x000F000Fu) | 0x64006400u;
  const uint32_t b3 = (w8 & 0x00F000F0u) | 0x64006400u;
  h[0] = __hsub2(*reinterpret_cast<const __half2*>(&b0), off);
  h[1] = __hfma2(*reinterpret_cast<const __half2*>(&b1), s16, off16);
  h[2] = __hsub2(*reinterpret_cast<const __half2*>(&b2), off);
  h[3] = __hfma2(*reinterpret_cast<const __half2*>(&b3), s16, off16);
}

// The same decode fused with its use, as explicit f16x2 instructions (the
// bits of the pairs are carried in 32-bit registers): five integer
// instructions and four f16x2 instructions decode a word.
// w4_axpy8: h[k] += {q_k, q_{k+4}} * cf.
DV_DEV void w4_axpy8(uint32_t w, uint32_t cf, uint32_t* h) {
  asm("{\n\t.reg .b32 t0, t1, t2, t3, w8, c0, c1, c2;\n\t"
      "mov.b32 c0, 0x64086408;\n\t"
      "mov.b32 c1, 0x2C002C00;\n\t"
      "mov.b32 c2, 0xD480D480;\n\t"
      "lop3.b32 t0, %4, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t1, %4, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "shr.u32 w8, %4, 8;\n\t"
      "lop3.b32 t2, w8, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t3, w8, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "sub.rn.f16x2 t0, t0, c0;\n\t"
      "fma.rn.f16x2 t1, t1, c1, c2;\n\t"
      "sub.rn.f16x2 t2, t2, c0;\n\t"
      "fma.rn.f16x2 t3, t3, c1, c2;\n\t"
      "fma.rn.f16x2 %0, t0, %5, %0;\n\t"
      "fma.rn.f16x2 %1, t1, %5, %1;\n\t"
      "fma.rn.f16x2 %2, t2, %5, %2;\n\t"
      "fma.rn.f16x2 %3, t3, %5, %3;\n\t}"
      : "+r"(h[0]), "+r"(h[1]), "+r"(h[2]), "+r"(h[3])
      : "r"(w), "r"(cf));
}

// w4_dot8: the fp16 pair sum {sum_k q_k z_k, sum_k q_{k+4} z_{k+4}} of a word
// against z[k] = {z_k, z_{k+4}} (a product, then three fused multiply-adds).
DV_DEV uint32_t w4_dot8(uint32_t w, const uint32_t* z) {
  uint32_t r;
  asm("{\n\t.reg .b32 t0, t1, t2, t3, w8, c0, c1, c2;\n\t"
      "mov.b32 c0, 0x64086408;\n\t"
      "mov.b32 c1, 0x2C002C00;\n\t"
      "mov.b32 c2, 0xD480D480;\n\t"
      "lop3.b32 t0, %1, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t1, %1, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "shr.u32 w8, %1, 8;\n\t"
      "lop3.b32 t2, w8, 0x000F000F, 0x64006400, 0xEA;\n\t"
      "lop3.b32 t3, w8, 0x00F000F0, 0x64006400, 0xEA;\n\t"
      "sub.rn.f16x2 t0, t0, c0;\n\t"
      "fma.rn.f16x2 t1, t1, c1, c2;\n\t"
      "sub.rn.f16x2 t2, t2, c0;\n\t"
      "fma.rn.f16x2 t3, t3, c1, c2;\n\t"
      "mul.rn.f16x2 %0, t0, %2;\n\t"
      "fma.rn.f16x2 %0, t1, %3, %0;\n\t"
      "fma.rn.f16x2 %0, t2, %4, %0;\n\t"
      "fma.rn.f16x2 %0, t3, %5, %0;\n\t}"
      : "=r"(r)
      : "r"(w), "r"(z[0]), "r"(z[1]), "r"(z[2]), "r"(z[3]));
  return r;
}

// Both halves of an f16x2 register as floats.
DV_DEV float2 h2bits_to_f2(uint32_t x) {
  float lo, hi;
  asm("{\n\t.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(x));
  return make_float2(lo, hi);
}

// Batch-1 launches of 4-bit rows give each consumer thread V consecutive
// 8-column vectors (tid V .. tid V + V - 1), so its words of a row are one
// vector load and usually share one group scale; other launches stride the
// vectors by the thread count (tid + m T).
template <int KIND, int B, int V>
DV_DEV int vec_of(int tid, int m, int T) {
  if constexpr (is_w4(KIND) && B == 1) return tid * V + m;
  else return tid + m * T;
}

// This thread's V code words of a staged 4-bit row (vectors v0 .. v0 + V - 1,
// all inside the row), from their address.
template <int V>
DV_DEV void w4_words_at(const uint8_t* src, uint32_t* w) {
  if constexpr (V == 2) {
    const uint2 t = *reinterpret_cast<const uint2*>(src);
    w[0] = t.x; w[1] = t.y;
  } else if constexpr (V % 4 == 0) {
#pragma unroll
    for (int i = 0; i < V; i += 4) {
      const uint4 t = *reinterpret_cast<const uint4*>(src + i * 4);
      w[i] = t.x; w[i + 1] = t.y; w[i + 2] = t.z; w[i + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) w[i] = *reinterpret_cast<const uint32_t*>(src + i * 4);
  }
}

template <int V>
DV_DEV void w4_words(const uint8_t* row, int v0, uint32_t* w) {
  w4_words_at<V>(row + (size_t)v0 * 4, w);
}

// Sums of four values over the warp's lanes, four rows at once: after a
// pairwise exchange at distances 16 and 8 each lane keeps one row, then
// three shuffles finish it. Returns the full sum of row 2 (lane / 16 % 2) +
// (lane / 8 % 2), the same in every lane of that group of 8.
DV_DEV float warp_sum4(const float* a, int lane) {
  const bool h16 = lane & 16, h8 = lane & 8;
  float x0 = h16 ? a[2] : a[0], x1 = h16 ? a[3] : a[1];
  const float s0 = h16 ? a[0] : a[2], s1 = h16 ? a[1] : a[3];
  x0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  x1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  float y = h8 ? x1 : x0;
  y += __shfl_xor_sync(0xffffffffu, h8 ? x0 : x1, 8);
  y += __shfl_xor_sync(0xffffffffu, y, 4);
  y += __shfl_xor_sync(0xffffffffu, y, 2);
  y += __shfl_xor_sync(0xffffffffu, y, 1);
  return y;
}

struct StreamParams {
  StreamGeom g;
  int d, B;
  const uint16_t* x;   // [B][d] input of the block (LN applied for MLP / QKV)
  const uint16_t* ln_g;
  const uint16_t* ln_b;
  float eps;
  // rows
  const uint16_t* W0;  // fc1 / Wq / P1 / WoT
  const uint16_t* W1;  // fc2T / Wk
  const uint16_t* W2;  // Wv
  const uint16_t* bias0;  // b1 / bq
  const uint16_t* bias1;  // bk
  const uint16_t* bias2;  // bv
  const int32_t* idx;     // selected rows (neurons or units); NULL = identity
  int k;                  // number of selected entries (upper bound)
  const int32_t* dev_count;
  int n_rows_total;       // rows of the addressed matrix (bounds check)
  int flags;
  // QKV
  int G, dh, h_kv, n, n_max;
  float scale;
  float* qbuf;            // [B][k][G][dh]
  uint16_t *K, *V;        // [B][h_kv][n_max][dh]
  uint16_t *Kr, *Vr;      // retained [h_kv][b_max][dh]
  const int32_t* kept_count;
  int b_max;
  uint16_t* y_side;
  uint32_t* kv_missing;
  int fill_clear;         // QKV: the selected units' missing K/V were just recomputed
  // predictor first layer: P1 rows streamed after the QKV rows (look-ahead,
  // on the raw layer input) or alone (KIND_P1)
  const uint16_t* P1;
  int n_pred;             // P1 rows appended to a QKV launch
  float* u_out;           // [B][r]
  int relu;
  // WO: combined head outputs [B][k][G][dh]
  const float* Hc;
  // QKV: split-K counters to clear for the attention launch that follows
  int* zero_cnt;
  int n_zero;
  // partial outputs
  float* part;            // [gridDim][B][d]
  int* st;
  // MLP with DV_SKIP_INACTIVE: each CTA adds the fc2^T rows it streams here
  // (dv_count_active; NULL: not counted)
  int* active_cnt;
};

// Number of selected entries this launch processes.
DV_DEV int eff_count(const StreamParams& p) {
  int k = p.k;
  if (p.dev_count) {
    int c = *p.dev_count;
    k = c < k ? (c < 0 ? 0 : c) : k;
  }
  return k;
}

// Rows streamed per selected entry (1 for neurons / predictor rows; (G+2) dh
// for a QKV unit; G dh for a Wo unit).
DV_DEV int rows_per_entry(const StreamParams& p, int kind) {
  if (is_qkv(kind)) return (p.G + 2) * p.dh;
  if (is_wo(kind)) return p.G * p.dh;
  return 1;
}

// Global address of virtual row v of the launch's row list (phase: 0 dot
// phase, 1 axpy phase). Out-of-range indices are replaced by row 0 and
// reported; the consumers see coef 0 / discard the value.
DV_DEV const uint16_t* row_addr(const StreamParams& p, int kind, int phase, int v, int qkv_rows,
                                bool& bad) {
  const size_t d = (size_t)p.d;
  if (kind == KIND_QKV && v >= qkv_rows) {  // appended predictor rows
    bad = false;
    return p.P1 + (size_t)(v - qkv_rows) * d;
  }
  if (is_mlp(kind) || kind == KIND_P1) {
    int j = p.idx ? p.idx[v] : v;
    bad = (j < 0 || j >= p.n_rows_total);
    if (bad) j = 0;
    const uint16_t* base = (is_mlp(kind) && phase == 1) ? p.W1 : p.W0;
    if (kind == KIND_MLP4)
      return reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(base) +
                                               (size_t)j * w4_row_bytes(p.d));
    return base + (size_t)j * d;
  }
  const int per = rows_per_entry(p, kind);
  const int e = v / per, r = v % per;
  int u = p.idx ? p.idx[e] : e;
  bad = (u < 0 || u >= p.h_kv);
  if (bad) u = 0;
  // the matrix and row this virtual row reads
  const uint16_t* base;
  size_t row;
  if (is_wo(kind)) {  // r = g * dh + c ; query head u*G + g
    base = p.W0;
    row = (size_t)u * p.G * p.dh + r;
  } else {
    const int qrows = p.G * p.dh;
    if (r < qrows) {
      base = p.W0;
      row = (size_t)u * qrows + r;
    } else if (r < qrows + p.dh) {
      base = p.W1;
      row = (size_t)u * p.dh + (r - qrows);
    } else {
      base = p.W2;
      row = (size_t)u * p.dh + (r - qrows - p.dh);
    }
  }
  if (is_w4(kind))
    return reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(base) +
                                             row * w4_row_bytes(p.d));
  return base + row * d;
}

// Vector v (8 columns, 16 bytes of fp16) of a staged row (fp16 kinds; the
// 4-bit kinds read their words in place).
DV_DEV uint4 stage_vec(const uint8_t* row, int v) {
  return *reinterpret_cast<const uint4*>(row + v * 16);
}
// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int KIND, int B, int V>
DV_DEV void consume(const StreamParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                    uint64_t* act_ready, float* red, float* coef, float* lnred, int* list,
                    volatile int* abort_flag, volatile int* list_count, const int kk,
                    const int per, const int qkv_rows, const int r0, const int nrows,
                    const bool has_dot, const bool has_axpy, const bool skip);

template <int KIND, int B, int V>
__global__ void __launch_bounds__((is_w4(KIND) && B == 1) ? kW4Threads + 32 : (B == 1 ? 544 : 416), 1)
    k_stream(const StreamParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const StreamGeom& g = p.g;
  const int T = g.T, nwc = T / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem + g.off_bar);
  uint64_t* empty = full + g.NS;
  uint64_t* act_ready = empty + g.NS;
  float* red = reinterpret_cast<float*>(smem + g.off_red);
  float* coef = reinterpret_cast<float*>(smem + g.off_coef);
  float* lnred = reinterpret_cast<float*>(smem + g.off_ln);
  int* list = reinterpret_cast<int*>(smem + g.off_list);
  volatile int* abort_flag = list + g.CH;
  volatile int* list_count = list + g.CH + 1;

  // This CTA's slice of the selected entries.
  const int kk = eff_count(p);
  const int per = rows_per_entry(p, KIND);
  const int qkv_rows = is_qkv(KIND) ? kk * per : 0;
  const long long tot_rows = (long long)kk * per + (KIND == KIND_QKV ? p.n_pred : 0);
  const int r0 = (int)(tot_rows * blockIdx.x / gridDim.x);
  const int r1 = (int)(tot_rows * (blockIdx.x + 1) / gridDim.x);
  const int nrows = r1 - r0;
  const bool has_dot = !is_wo(KIND);
  const bool has_axpy = (is_mlp(KIND) || is_wo(KIND));
  const bool skip = is_mlp(KIND) && (p.flags & DV_SKIP_INACTIVE);

  if (tid == 0) {
    for (int s = 0; s < g.NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], nwc);
    }
    mbar_init(act_ready, 1);
    *abort_flag = 0;
    *list_count = nrows;
    fence_mbar_init();
  }
  __syncthreads();

  // ======================= producer warp =======================
  if (warp == nwc && is_w4(KIND)) {
    // 4-bit rows are short, so one thread fetching each row's index before
    // its copy would set the pace: the warp's lanes issue a stage's rows
    // together (lane c: row c), after lane 0 has claimed the slot.
    const uint64_t pol = policy_evict_first();
    int it = 0;
    bool bad_any = false, stop = false;
    for (int phase = 0; phase < 2 && !stop; ++phase) {
      if (phase == 0 && !has_dot) continue;
      if (phase == 1 && !has_axpy) continue;
      int n_this = nrows;
      if (phase == 1 && skip) {
        const bool got = mbar_wait(act_ready, 0);  // every lane reads the list below
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) {
            *abort_flag = 1;
            flag(p.st, DV_DEV_TIMEOUT);
          }
          break;
        }
        n_this = *list_count;
      }
      for (int q0 = 0; q0 < n_this; q0 += g.R, ++it) {
        const int cnt = min(g.R, n_this - q0);
        const int s = it % g.NS;
        const uint32_t ph = (it / g.NS) & 1;
        int go = 1;
        if (lane == 0) {
          if (*abort_flag) {
            go = 0;
          } else if (it >= g.NS && !mbar_wait(&empty[s], ph ^ 1)) {
            *abort_flag = 1;
            flag(p.st, DV_DEV_TIMEOUT);
            go = 0;
          }
          if (go) mbar_arrive_expect_tx(&full[s], cnt * g.row_bytes);
        }
        if (!__shfl_sync(0xffffffffu, go, 0)) {
          stop = true;
          break;
        }
        if (lane < cnt) {
          const int local = (phase == 1 && skip) ? list[q0 + lane] : (q0 + lane);
          bool bad;
          const uint16_t* src = row_addr(p, KIND, phase, r0 + local, qkv_rows, bad);
          bad_any |= bad;
          bulk_g2s(smem + (size_t)s * g.stage_bytes + (size_t)lane * g.row_bytes, src,
                   g.row_bytes, &full[s], pol);
        }
        __syncwarp();
      }
    }
    if (__any_sync(0xffffffffu, bad_any) && lane == 0) flag(p.st, DV_DEV_BAD_INDEX);
    if (lane == 0)  // drain: every issued copy must land before the CTA exits
      for (int j = (it > g.NS ? it - g.NS : 0); j < it; ++j)
        if (!mbar_wait(&full[j % g.NS], (j / g.NS) & 1)) flag(p.st, DV_DEV_TIMEOUT);
    __syncwarp();
  } else if (warp == nwc) {
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int it = 0;
      int bad_any = 0;
      for (int phase = 0; phase < 2; ++phase) {
        if (phase == 0 && !has_dot) continue;
        if (phase == 1 && !has_axpy) continue;
        int n_this = nrows;
        if (phase == 1 && skip) {
          if (!mbar_wait(act_ready, 0)) {
            *abort_flag = 1;
            flag(p.st, DV_DEV_TIMEOUT);
          }
          n_this = *list_count;
        }
        for (int q0 = 0; q0 < n_this && !*abort_flag; q0 += g.R, ++it) {
          const int cnt = min(g.R, n_this - q0);
          const int s = it % g.NS;
          const uint32_t ph = (it / g.NS) & 1;
          if (it >= g.NS && !mbar_wait(&empty[s], ph ^ 1)) {
            *abort_flag = 1;
            flag(p.st, DV_DEV_TIMEOUT);
            break;
          }
          mbar_arrive_expect_tx(&full[s], cnt * g.row_bytes);
          for (int c = 0; c < cnt; ++c) {
            const int local = (phase == 1 && skip) ? list[q0 + c] : (q0 + c);
            bool bad;
            const uint16_t* src = row_addr(p, KIND, phase, r0 + local, qkv_rows, bad);
            bad_any |= bad;
            bulk_g2s(smem + (size_t)s * g.stage_bytes + (size_t)c * g.row_bytes, src, g.row_bytes,
                     &full[s], pol);
          }
        }
      }
      if (bad_any) flag(p.st, DV_DEV_BAD_INDEX);
      // Drain: every issued copy must land before the CTA exits.
      for (int j = (it > g.NS ? it - g.NS : 0); j < it; ++j)
        if (!mbar_wait(&full[j % g.NS], (j / g.NS) & 1)) flag(p.st, DV_DEV_TIMEOUT);
    }
    __syncwarp();
  } else {
    consume<KIND, B, V>(p, smem, full, empty, act_ready, red, coef, lnred, list, abort_flag,
                        list_count, kk, per, qkv_rows, r0, nrows, has_dot, has_axpy, skip);
  }
  // Both roles meet here once, with converged warps.
  __syncthreads();
}

// ======================= consumer warps =======================
template <int KIND, int B, int V>
DV_DEV void consume(const StreamParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                    uint64_t* act_ready, float* red, float* coef, float* lnred, int* list,
                    volatile int* abort_flag, volatile int* list_count, const int kk,
                    const int per, const int qkv_rows, const int r0, const int nrows,
                    const bool has_dot, const bool has_axpy, const bool skip) {
  const StreamGeom& g = p.g;
  const int T = g.T, nwc = T / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = p.d >> 3;
  constexpr int RM = rows_max(V);  // rows per stage held in registers
  // The weight stream may already be running; activations and every global
  // write wait until the previous kernel of the stream has completed.
  pdl_wait();
  if (tid == 0) pdl_launch_dependents();
  // Activation columns of this thread: vectors v_m = tid + m T (8 columns each).
  float z[B][V][8];
  __half2 zh[is_w4(KIND) ? B : 1][is_w4(KIND) ? V : 1][4];
  // The raw fp16 input, for predictor rows fused into a QKV launch (they read
  // y, not LN(y)); batch-1 launches only (at B = 4 the extra registers would
  // spill: the predictor's first layer then runs as its own launch).
  constexpr bool kRaw = (KIND == KIND_QKV && B == 1);
  uint4 xraw[kRaw ? B : 1][kRaw ? V : 1];
  int it = 0;
  if (has_dot) {
    // --- load x, optional LayerNorm ("Deja Vu" App. C.3: blocks read LN(y)).
    float s1[B];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      s1[b] = 0.f;
#pragma unroll
      for (int m = 0; m < V; ++m) {
        const int v = vec_of<KIND, B, V>(tid, m, T);
#pragma unroll
        for (int e = 0; e < 8; ++e) z[b][m][e] = 0.f;
        if (kRaw) xraw[kRaw ? b : 0][kRaw ? m : 0] = make_uint4(0, 0, 0, 0);
        if (v < nvec && b < p.B) {
          uint4 xv = *reinterpret_cast<const uint4*>(p.x + (size_t)b * p.d + v * 8);
          if (kRaw) xraw[kRaw ? b : 0][kRaw ? m : 0] = xv;
          h8_to_f8(xv, z[b][m]);
#pragma unroll
          for (int e = 0; e < 8; ++e) s1[b] += z[b][m][e];
        }
      }
    }
    if (KIND != KIND_P1) {
      float* mean_inv = lnred + B * nwc * 2;
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float t = warp_sum(s1[b]);
        if (lane == 0) lnred[b * nwc + warp] = t;
      }
      consumer_sync(T);
      if (tid < B) {
        float t = 0.f;
        for (int w = 0; w < nwc; ++w) t += lnred[tid * nwc + w];
        mean_inv[tid * 2] = t / p.d;
      }
      consumer_sync(T);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float mu = mean_inv[b * 2];
        float s2 = 0.f;
#pragma unroll
        for (int m = 0; m < V; ++m) {
          const int v = vec_of<KIND, B, V>(tid, m, T);
          if (v < nvec) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float c = z[b][m][e] - mu;
              s2 = fmaf(c, c, s2);
            }
          }
        }
        s2 = warp_sum(s2);
        if (lane == 0) lnred[B * nwc + b * nwc + warp] = s2;
      }
      consumer_sync(T);
      if (tid < B) {
        float t = 0.f;
        for (int w = 0; w < nwc; ++w) t += lnred[B * nwc + tid * nwc + w];
        mean_inv[tid * 2 + 1] = 1.0f / sqrtf(t / p.d + p.eps);
      }
      consumer_sync(T);
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const float mu = mean_inv[b * 2], inv = mean_inv[b * 2 + 1];
#pragma unroll
        for (int m = 0; m < V; ++m) {
          const int v = vec_of<KIND, B, V>(tid, m, T);
          if (v < nvec) {
            float gg[8], bb[8];
            if (p.ln_g) {
              h8_to_f8(*reinterpret_cast<const uint4*>(p.ln_g + v * 8), gg);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) gg[e] = 1.f;
            }
            if (p.ln_b) {
              h8_to_f8(*reinterpret_cast<const uint4*>(p.ln_b + v * 8), bb);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) bb[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) z[b][m][e] = (z[b][m][e] - mu) * inv * gg[e] + bb[e];
          }
        }
      }
    }

    if constexpr (is_w4(KIND)) {
      // fp16 pairs of the activations in the codes' order: {z_k, z_{k+4}}
#pragma unroll
      for (int b = 0; b < B; ++b)
#pragma unroll
        for (int m = 0; m < V; ++m)
#pragma unroll
          for (int k = 0; k < 4; ++k) zh[b][m][k] = __floats2half2_rn(z[b][m][k], z[b][m][k + 4]);
    }
    // --- dot phase: red[row][b][warp] = warp's share of z . W[row]. A warp
    // copies its columns of the stage's rows into registers, releases the
    // slot, then computes (the slot is held only for the shared-memory reads).
    for (int q0 = 0; q0 < nrows; q0 += g.R, ++it) {
      const int cnt = min(g.R, nrows - q0);
      const int s = it % g.NS;
      const uint32_t ph = (it / g.NS) & 1;
      bool ok = !*abort_flag;
      if (ok && !mbar_wait(&full[s], ph)) {
        *abort_flag = 1;
        flag(p.st, DV_DEV_TIMEOUT);
        ok = false;
      }
      ok = __all_sync(0xffffffffu, ok);  // warp-uniform: the row sums below shuffle
      if constexpr (is_w4(KIND) && B == 1) {
        // 4-bit rows, batch 1: four rows at a time, each thread over its V
        // consecutive words (one vector load, one group scale when V divides
        // 16); products of the exact codes and the fp16 activations summed
        // in fp16 pairs over each word, then scaled and accumulated in fp32.
        if (ok) {
          const uint8_t* st0 = smem + (size_t)s * g.stage_bytes;
          const int v0 = tid * V;
          const bool act = v0 < nvec;
          if (16 % V == 0 && cnt == kW4StageRows && T * V == nvec) {
            // a full stage and every thread on whole words: no per-row tests
            const uint8_t* wp = st0 + (size_t)v0 * 4;
            const uint16_t* sp = reinterpret_cast<const uint16_t*>(st0 + p.d / 2) + (v0 >> 4);
            const int rb = (int)g.row_bytes;
#pragma unroll
            for (int c0 = 0; c0 < kW4StageRows; c0 += 4) {
              float a[4];
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                uint32_t wd[V];
                w4_words_at<V>(wp + (c0 + r) * rb, wd);
                const float sc = h2f(sp[(c0 + r) * (rb >> 1)]);
                float t = 0.f;
#pragma unroll
                for (int m = 0; m < V; ++m) {
                  const float2 hf =
                      h2bits_to_f2(w4_dot8(wd[m], reinterpret_cast<const uint32_t*>(zh[0][m])));
                  t += hf.x + hf.y;
                }
                a[r] = t * sc;
              }
              const float sum = warp_sum4(a, lane);
              const int rr = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
              if ((lane & 7) == 0) red[(q0 + c0 + rr) * nwc + warp] = sum;
            }
          } else
          for (int c0 = 0; c0 < cnt; c0 += 4) {
            float a[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              a[r] = 0.f;
              if (c0 + r < cnt && act) {
                const uint8_t* row = st0 + (size_t)(c0 + r) * g.row_bytes;
                const uint16_t* scl = reinterpret_cast<const uint16_t*>(row + p.d / 2);
                uint32_t wd[V];
                w4_words<V>(row, v0, wd);
                float t = 0.f;
#pragma unroll
                for (int m = 0; m < V; ++m) {
                  if (16 % V != 0 && v0 + m >= nvec) break;
                  const float2 hf =
                      h2bits_to_f2(w4_dot8(wd[m], reinterpret_cast<const uint32_t*>(zh[0][m])));
                  if constexpr (16 % V == 0) {
                    t += hf.x + hf.y;
                  } else {
                    t = fmaf(h2f(scl[(v0 + m) >> 4]), hf.x + hf.y, t);
                  }
                }
                a[r] = (16 % V == 0) ? t * h2f(scl[v0 >> 4]) : t;
              }
            }
            const float sum = warp_sum4(a, lane);
            const int rr = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            if ((lane & 7) == 0 && c0 + rr < cnt) red[(q0 + c0 + rr) * nwc + warp] = sum;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      } else if constexpr (is_w4(KIND)) {
        // 4-bit rows: decode straight from the stage, release it afterwards
        if (ok) {
          const uint8_t* st0 = smem + (size_t)s * g.stage_bytes;
          // kW4Ilp rows at a time: independent chains, and their row sums
          // shuffle together. The 16-bit activations ("A16") times the exact
          // codes are summed in fp16 pairs over each 8 columns, then scaled
          // and accumulated in fp32.
          for (int c0 = 0; c0 < cnt; c0 += kW4Ilp) {
            float acc[kW4Ilp][B];
#pragma unroll
            for (int r = 0; r < kW4Ilp; ++r)
#pragma unroll
              for (int b = 0; b < B; ++b) acc[r][b] = 0.f;
#pragma unroll
            for (int m = 0; m < V; ++m) {
              const int v = vec_of<KIND, B, V>(tid, m, T);
              if (v >= nvec) continue;
#pragma unroll
              for (int r = 0; r < kW4Ilp; ++r) {
                if (c0 + r >= cnt) break;
                const uint8_t* row = st0 + (size_t)(c0 + r) * g.row_bytes;
                __half2 q2[4];
                w4_decode_h2(*reinterpret_cast<const uint32_t*>(row + v * 4), q2);
                const float sc =
                    h2f(*reinterpret_cast<const uint16_t*>(row + p.d / 2 + (v >> 4) * 2));
#pragma unroll
                for (int b = 0; b < B; ++b) {
                  __half2 t = __hmul2(q2[0], zh[b][m][0]);
#pragma unroll
                  for (int k = 1; k < 4; ++k) t = __hfma2(q2[k], zh[b][m][k], t);
                  const float2 tf = __half22float2(t);
                  acc[r][b] = fmaf(sc, tf.x + tf.y, acc[r][b]);
                }
              }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
              for (int r = 0; r < kW4Ilp; ++r)
#pragma unroll
                for (int b = 0; b < B; ++b)
                  acc[r][b] += __shfl_xor_sync(0xffffffffu, acc[r][b], off);
            if (lane == 0)
#pragma unroll
              for (int r = 0; r < kW4Ilp; ++r)
                if (c0 + r < cnt)
#pragma unroll
                  for (int b = 0; b < B; ++b) red[((q0 + c0 + r) * B + b) * nwc + warp] = acc[r][b];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      uint4 wv[RM][V];
      if (ok) {
        const uint8_t* st0 = smem + (size_t)s * g.stage_bytes;
#pragma unroll
        for (int c = 0; c < RM; ++c)
#pragma unroll
          for (int m = 0; m < V; ++m) {
            const int v = vec_of<KIND, B, V>(tid, m, T);
            wv[c][m] = (c < cnt && v < nvec) ? stage_vec(st0 + (size_t)c * g.row_bytes, v)
                                             : make_uint4(0, 0, 0, 0);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (ok) {
#pragma unroll
        for (int c = 0; c < RM; ++c) {
          if (c >= cnt) break;
          const bool raw = (KIND == KIND_QKV) && (r0 + q0 + c >= qkv_rows);
          float acc[B];
#pragma unroll
          for (int b = 0; b < B; ++b) acc[b] = 0.f;
#pragma unroll
          for (int m = 0; m < V; ++m) {
            float w[8];
            h8_to_f8(wv[c][m], w);
            if (kRaw && raw) {
#pragma unroll
              for (int b = 0; b < B; ++b) {
                float xf[8];
                h8_to_f8(xraw[kRaw ? b : 0][kRaw ? m : 0], xf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[b] = fmaf(xf[e], w[e], acc[b]);
              }
            } else {
#pragma unroll
              for (int b = 0; b < B; ++b)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[b] = fmaf(z[b][m][e], w[e], acc[b]);
            }
          }
#pragma unroll
          for (int b = 0; b < B; ++b) {
            const float t = warp_sum(acc[b]);
            if (lane == 0) red[((q0 + c) * B + b) * nwc + warp] = t;
          }
        }
      }
    }
    consumer_sync(T);

    // --- finalize the dot values (fixed-order sum over the warps)
    for (int i = tid; i < nrows; i += T) {
      const int v = r0 + i;
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float val = 0.f;
        for (int w = 0; w < nwc; ++w) val += red[(i * B + b) * nwc + w];
        if (is_mlp(KIND)) {
          int j = p.idx ? p.idx[v] : v;
          const bool badj = (j < 0 || j >= p.n_rows_total);
          float a = val + ((p.bias0 && !badj) ? h2f(p.bias0[j]) : 0.f);
          a = a > 0.f ? a : 0.f;
          coef[b * g.CH + i] = (badj || b >= p.B) ? 0.f : a;
        } else if (KIND == KIND_P1) {
          if (b < p.B) {
            float u = val;
            if (p.relu && u < 0.f) u = 0.f;
            p.u_out[(size_t)b * p.n_rows_total + v] = u;
          }
        } else if (is_qkv(KIND) && v >= qkv_rows) {
          if (b < p.B) {
            float u = val;
            if (p.relu && u < 0.f) u = 0.f;
            p.u_out[(size_t)b * p.n_pred + (v - qkv_rows)] = u;
          }
        } else if (is_qkv(KIND)) {
          const int e = v / per, r = v % per;
          const int u = p.idx ? p.idx[e] : e;
          if (u < 0 || u >= p.h_kv || b >= p.B) continue;
          const int qrows = p.G * p.dh;
          if (r < qrows) {
            const float bq = p.bias0 ? h2f(p.bias0[u * qrows + r]) : 0.f;
            p.qbuf[((size_t)b * p.k + e) * qrows + r] = (val + bq) * p.scale;
          } else {
            const bool isk = r < qrows + p.dh;
            const int c = isk ? r - qrows : r - qrows - p.dh;
            const uint16_t* bb = isk ? p.bias1 : p.bias2;
            const float bv = bb ? h2f(bb[u * p.dh + c]) : 0.f;
            const uint16_t hv = f2h(val + bv);
            uint16_t* cache = isk ? p.K : p.V;
            cache[(((size_t)b * p.h_kv + u) * p.n_max + p.n) * p.dh + c] = hv;
            if (p.Kr) {
              const int slot = p.kept_count[u];
              uint16_t* rc = isk ? p.Kr : p.Vr;
              if (slot >= 0 && slot < p.b_max) rc[((size_t)u * p.b_max + slot) * p.dh + c] = hv;
            }
          }
        }
      }
    }
    if (is_qkv(KIND) && blockIdx.x == 0)
      for (int i = tid; i < p.n_zero; i += T) p.zero_cnt[i] = 0;
    if (is_qkv(KIND) && blockIdx.x == 0) {
      // Missing-KV bookkeeping ("Deja Vu" §4.2): keep a copy of y for the
      // units that did not get their k, v at this token.
      const int words = (p.h_kv + 31) / 32;
      for (int b = 0; b < p.B; ++b) {
        if (p.y_side)
          for (int v = tid; v < nvec; v += T)
            *reinterpret_cast<uint4*>(p.y_side + ((size_t)b * p.n_max + p.n) * p.d + v * 8) =
                *reinterpret_cast<const uint4*>(p.x + (size_t)b * p.d + v * 8);
        if (p.kv_missing)
          for (int w = tid; w < words; w += T) {
            uint32_t bits = 0;
            for (int u = w * 32; u < min(p.h_kv, w * 32 + 32); ++u) bits |= 1u << (u - w * 32);
            if (p.idx) {
              for (int e = 0; e < kk; ++e) {
                const int u = p.idx[e];
                if (u >= w * 32 && u < w * 32 + 32) bits &= ~(1u << (u - w * 32));
              }
            } else {
              bits = 0;
            }
            p.kv_missing[((size_t)b * p.n_max + p.n) * words + w] = bits;
          }
      }
    }
    if (is_qkv(KIND) && blockIdx.x == 0 && p.fill_clear && p.kv_missing) {
      // The recompute that ran right before this launch filled every marked
      // position of the selected units ("Deja Vu" §4.2): clear those marks.
      // A unit's marks are a suffix of the positions; scan back from n - 1.
      const int words = (p.h_kv + 31) / 32;
      for (int be = warp; be < p.B * kk; be += nwc) {
        const int b = be / kk, e = be % kk;
        const int u = p.idx ? p.idx[e] : e;
        if (u < 0 || u >= p.h_kv) continue;
        uint32_t* marks = p.kv_missing + (size_t)b * p.n_max * words + (u >> 5);
        const uint32_t bit = 1u << (u & 31);
        for (int top = p.n - 1; top >= 0; top -= 32) {
          const int t = top - lane;
          const bool miss = t >= 0 && (marks[(size_t)t * words] & bit);
          if (miss) atomicAnd(&marks[(size_t)t * words], ~bit);
          if (__ballot_sync(0xffffffffu, !miss)) break;
        }
      }
    }
    if (skip) {
      consumer_sync(T);
      if (tid == 0) {
        int c = 0;
        for (int i = 0; i < nrows; ++i) {
          float any = 0.f;
#pragma unroll
          for (int b = 0; b < B; ++b) any = fmaxf(any, coef[b * g.CH + i]);
          if (any > 0.f) list[c++] = i;
        }
        *list_count = c;
        mbar_arrive(act_ready);
        if (p.active_cnt) atomicAdd(p.active_cnt, c);
      }
    }
    consumer_sync(T);
  }

  if (has_axpy) {
    if (is_wo(KIND)) {
      // Coefficients: the combined attention output of each row's (head, dim).
      for (int i = tid; i < nrows * B; i += T) {
        const int li = i % nrows, b = i / nrows;
        const int v = r0 + li;
        const int e = v / per, r = v % per;  // r = g dh + c
        float H = 0.f;
        if (b < p.B) {
          const int u = p.idx ? p.idx[e] : e;
          if (u >= 0 && u < p.h_kv) H = p.Hc[((size_t)b * p.k + e) * per + r];
        }
        coef[b * g.CH + li] = H;
      }
      consumer_sync(T);
    }
    const int n_ax = skip ? *list_count : nrows;
    float acc[B][V][8];
#pragma unroll
    for (int b = 0; b < B; ++b)
#pragma unroll
      for (int m = 0; m < V; ++m)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[b][m][e] = 0.f;
    for (int q0 = 0; q0 < n_ax; q0 += g.R, ++it) {
      const int cnt = min(g.R, n_ax - q0);
      const int s = it % g.NS;
      const uint32_t ph = (it / g.NS) & 1;
      bool ok = !*abort_flag;
      if (ok && !mbar_wait(&full[s], ph)) {
        *abort_flag = 1;
        flag(p.st, DV_DEV_TIMEOUT);
        ok = false;
      }
      ok = __all_sync(0xffffffffu, ok);
      if constexpr (is_w4(KIND) && B == 1) {
        // 4-bit rows, batch 1: the thread's V consecutive words of each row
        // (one vector load, one group scale when V divides 16), coefficient
        // a_j s rounded to fp16, the stage's rows summed in fp16 pairs, then
        // added to the fp32 accumulators once per stage.
        if (ok) {
          const uint8_t* st0 = smem + (size_t)s * g.stage_bytes;
          const int v0 = tid * V;
          if (v0 < nvec) {
            uint32_t h[V][4];
#pragma unroll
            for (int m = 0; m < V; ++m)
#pragma unroll
              for (int k = 0; k < 4; ++k) h[m][k] = 0u;  // +0.0 in both halves
            if (16 % V == 0 && cnt == kW4StageRows && T * V == nvec) {
              // a full stage and every thread on whole words: no per-row tests
              const uint8_t* wp = st0 + (size_t)v0 * 4;
              const uint16_t* sp = reinterpret_cast<const uint16_t*>(st0 + p.d / 2) + (v0 >> 4);
              const int rb = (int)g.row_bytes;
#pragma unroll
              for (int c = 0; c < kW4StageRows; ++c) {
                const float a = coef[skip ? list[q0 + c] : (q0 + c)];
                uint32_t wd[V];
                w4_words_at<V>(wp + c * rb, wd);
                const __half2 cf = __float2half2_rn(a * h2f(sp[c * (rb >> 1)]));
#pragma unroll
                for (int m = 0; m < V; ++m)
                  w4_axpy8(wd[m], *reinterpret_cast<const uint32_t*>(&cf), h[m]);
              }
            } else
            for (int c = 0; c < cnt; ++c) {
              const uint8_t* row = st0 + (size_t)c * g.row_bytes;
              const uint16_t* scl = reinterpret_cast<const uint16_t*>(row + p.d / 2);
              const float a = coef[skip ? list[q0 + c] : (q0 + c)];
              uint32_t wd[V];
              w4_words<V>(row, v0, wd);
              __half2 cf = __float2half2_rn(a * h2f(scl[v0 >> 4]));
#pragma unroll
              for (int m = 0; m < V; ++m) {
                if (16 % V != 0 && v0 + m >= nvec) break;
                if (16 % V != 0 && m > 0) cf = __float2half2_rn(a * h2f(scl[(v0 + m) >> 4]));
                w4_axpy8(wd[m], *reinterpret_cast<const uint32_t*>(&cf), h[m]);
              }
            }
#pragma unroll
            for (int m = 0; m < V; ++m)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = h2bits_to_f2(h[m][k]);
                acc[0][m][k] += f.x;
                acc[0][m][k + 4] += f.y;
              }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      } else if constexpr (is_w4(KIND)) {
        if (ok) {
          const uint8_t* st0 = smem + (size_t)s * g.stage_bytes;
          // The stage's rows (at most kW4StageRows) are summed in fp16 pairs,
          // each row's coefficient a_j s rounded to fp16, then added to the
          // fp32 accumulators once per stage.
#pragma unroll
          for (int m = 0; m < V; ++m) {
            const int v = vec_of<KIND, B, V>(tid, m, T);
            if (v >= nvec) continue;
            __half2 h[B][4];
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
              for (int k = 0; k < 4; ++k) h[b][k] = __float2half2_rn(0.f);
            for (int c = 0; c < cnt; ++c) {
              const uint8_t* row = st0 + (size_t)c * g.row_bytes;
              const int li = skip ? list[q0 + c] : (q0 + c);
              __half2 q2[4];
              w4_decode_h2(*reinterpret_cast<const uint32_t*>(row + v * 4), q2);
              const float sc = h2f(*reinterpret_cast<const uint16_t*>(row + p.d / 2 + (v >> 4) * 2));
#pragma unroll
              for (int b = 0; b < B; ++b) {
                const __half2 cf = __float2half2_rn(coef[b * g.CH + li] * sc);
#pragma unroll
                for (int k = 0; k < 4; ++k) h[b][k] = __hfma2(q2[k], cf, h[b][k]);
              }
            }
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(h[b][k]);
                acc[b][m][k] += f.x;
                acc[b][m][k + 4] += f.y;
              }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      uint4 wv[RM][V];
      if (ok) {
        const uint8_t* st0 = smem + (size_t)s * g.stage_bytes;
#pragma unroll
        for (int c = 0; c < RM; ++c)
#pragma unroll
          for (int m = 0; m < V; ++m) {
            const int v = vec_of<KIND, B, V>(tid, m, T);
            wv[c][m] = (c < cnt && v < nvec) ? stage_vec(st0 + (size_t)c * g.row_bytes, v)
                                             : make_uint4(0, 0, 0, 0);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (ok) {
#pragma unroll
        for (int c = 0; c < RM; ++c) {
          if (c >= cnt) break;
          const int li = skip ? list[q0 + c] : (q0 + c);
          float a[B];
#pragma unroll
          for (int b = 0; b < B; ++b) a[b] = coef[b * g.CH + li];
#pragma unroll
          for (int m = 0; m < V; ++m) {
            float w[8];
            h8_to_f8(wv[c][m], w);
#pragma unroll
            for (int b = 0; b < B; ++b)
#pragma unroll
              for (int e = 0; e < 8; ++e) acc[b][m][e] = fmaf(a[b], w[e], acc[b][m][e]);
          }
        }
      }
    }
    // Partial output of this CTA.
#pragma unroll
    for (int b = 0; b < B; ++b) {
      if (b >= p.B) break;
      float* dst = p.part + ((size_t)blockIdx.x * p.B + b) * p.d;
#pragma unroll
      for (int m = 0; m < V; ++m) {
        const int v = vec_of<KIND, B, V>(tid, m, T);
        if (v < nvec) {
          float4* o = reinterpret_cast<float4*>(dst + v * 8);
          o[0] = make_float4(acc[b][m][0], acc[b][m][1], acc[b][m][2], acc[b][m][3]);
          o[1] = make_float4(acc[b][m][4], acc[b][m][5], acc[b][m][6], acc[b][m][7]);
        }
      }
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// Fixed-order reduce of the CTA partials: out = x + bias + sum_g part[g].
// A CTA covers 64 columns: 16 slices of 16 lanes, each lane a float4 of
// columns; slice j sums partials j, j+16, ... with all its loads in flight,
// then slice 0 adds the 16 slices in order.
// ---------------------------------------------------------------------------
constexpr int kRedSlices = 16;

__global__ void __launch_bounds__(256) k_reduce(const float* __restrict__ part, int G, int B, int d,
                                                const uint16_t* __restrict__ x,
                                                const uint16_t* __restrict__ bias,
                                                uint16_t* __restrict__ out) {
  __shared__ float4 sl[kRedSlices][16];
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int cg = threadIdx.x & 15, slice = threadIdx.x >> 4;
  const int c4 = blockIdx.x * 16 + cg;  // group of 4 columns
  const int b = blockIdx.y;
  const bool on = c4 * 4 < d;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (on) {
    const size_t stride = (size_t)B * d;
    const float* src = part + (size_t)b * d + c4 * 4;
    for (int g0 = slice; g0 < G; g0 += kRedSlices * 12) {
      float4 t[12];
#pragma unroll
      for (int j = 0; j < 12; ++j) {
        const int gi = g0 + kRedSlices * j;
        t[j] = gi < G ? __ldcg(reinterpret_cast<const float4*>(src + gi * stride))
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int j = 0; j < 12; ++j) { s.x += t[j].x; s.y += t[j].y; s.z += t[j].z; s.w += t[j].w; }
    }
  }
  sl[slice][cg] = s;
  __syncthreads();
  if (slice != 0 || !on) return;
  float r[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < kRedSlices; ++k) {
    r[0] += sl[k][cg].x; r[1] += sl[k][cg].y; r[2] += sl[k][cg].z; r[3] += sl[k][cg].w;
  }
  const uint16_t* xr = x ? x + (size_t)b * d + c4 * 4 : nullptr;
  uint16_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float bb = bias ? h2f(bias[c4 * 4 + e]) : 0.f;
    o[e] = f2h((xr ? h2f(xr[e]) : 0.f) + (r[e] + bb));
  }
  uint2 pk;
  pk.x = (uint32_t)o[0] | ((uint32_t)o[1] << 16);
  pk.y = (uint32_t)o[2] | ((uint32_t)o[3] << 16);
  *reinterpret_cast<uint2*>(out + (size_t)b * d + c4 * 4) = pk;
}

// ---------------------------------------------------------------------------
// Predictor GEMVs ("Deja Vu" §4.1 "Design": a small two-layer fully connected
// network; low-rank chain y -> P1 -> r -> P2 -> scores). Dense, contiguous
// rows, so plain 16-byte loads: one warp per row (two rows per step for short
// rows), each lane keeping U independent loads in flight. These kernels are
// small (256 threads, no dynamic shared memory) so that, launched on the side
// stream, their CTAs fit next to a weight-streaming CTA on every SM.
// out[b][row] = act(sum_c in[b][c] W[row][c]); `in` is fp16 (first layer) or
// fp32 (second layer); Kahan-compensated per-lane sums of 8-term chunks.
// ---------------------------------------------------------------------------
template <typename TIn>
DV_DEV void load_in8(const TIn* p, float* f);
template <>
DV_DEV void load_in8<uint16_t>(const uint16_t* p, float* f) {
  h8_to_f8(*reinterpret_cast<const uint4*>(p), f);
}
template <>
DV_DEV void load_in8<float>(const float* p, float* f) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

template <typename TIn, int B, int RPW>
__global__ void __launch_bounds__(256, 4) k_gemv(const TIn* __restrict__ in, int nB, int len,
                                              const uint16_t* __restrict__ W, int N,
                                              float* __restrict__ out, int ld, int relu) {
  constexpr int U = 4;  // loads in flight per lane and row (64 registers: fits next to a
                        // weight-streaming CTA on the same SM)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int nv = len >> 3;
  for (int row0 = (blockIdx.x * nw + warp) * RPW; row0 < N; row0 += gridDim.x * nw * RPW) {
    float acc[RPW][B], cmp[RPW][B];
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
      for (int b = 0; b < B; ++b) acc[q][b] = cmp[q][b] = 0.f;
    for (int v0 = lane; v0 < nv; v0 += 32 * U) {
      uint4 w[RPW][U];
#pragma unroll
      for (int q = 0; q < RPW; ++q)
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int v = v0 + 32 * j;
          const int row = row0 + q;
          w[q][j] = (v < nv && row < N) ? ld_nc_v4(W + (size_t)row * len + v * 8)
                                        : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
      for (int j = 0; j < U; ++j) {
        const int v = v0 + 32 * j;
        if (v >= nv) break;
#pragma unroll
        for (int b = 0; b < B; ++b) {
          if (b >= nB) break;
          float xin[8];
          load_in8<TIn>(in + (size_t)b * len + v * 8, xin);
#pragma unroll
          for (int q = 0; q < RPW; ++q) {
            float wf[8];
            h8_to_f8(w[q][j], wf);
            float t = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) t = fmaf(xin[e], wf[e], t);
            kahan_add(acc[q][b], cmp[q][b], t);
          }
        }
      }
    }
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
      for (int b = 0; b < B; ++b) {
        float t = warp_sum(acc[q][b] - cmp[q][b]);
        if (relu && t < 0.f) t = 0.f;
        if (lane == 0 && b < nB && row0 + q < N) out[(size_t)b * ld + row0 + q] = t;
      }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static int pick_V(int nvec, int tmax) { return (nvec + tmax - 1) / tmax; }

int g_stage_target = 48 * 1024;  // bytes per ring stage (rows are grouped up to this)

static bool make_geom(StreamGeom& g, int d, int B, int ring_budget, int CH, bool w4 = false,
                      bool dot = true) {
  const int nvec = d / 8;
  // 4-bit rows cost more instructions per byte: up to 24 consumer warps at B = 1
  const int tmax = (w4 && B == 1) ? kW4Threads : (B == 1) ? 512 : 384;
  const int V = pick_V(nvec, tmax);
  g.T = ((nvec + V - 1) / V + 31) / 32 * 32;
  g.B = B;
  g.row_bytes = w4 ? w4_row_bytes(d) : (uint32_t)d * 2;
  // 4-bit rows are read from the stage in place (no register copy), so a
  // stage can hold more of them
  g.R = w4 ? std::min(kW4StageRows, std::max(1, ring_budget / (2 * (int)g.row_bytes)))
            : std::min(rows_max(V == 7 ? 8 : V), std::max(1, (int)(g_stage_target / g.row_bytes)));
  g.stage_bytes = g.R * g.row_bytes;
  g.NS = std::min(16, ring_budget / (int)g.stage_bytes);
  if (g.NS < 2) g.NS = 2;
  g.CH = CH;
  stream_layout(g, dot);
  return g.total <= 227 * 1024;
}

template <int KIND, int B>
static void* stream_kernel_for_V(int V) {
  switch (V) {
    case 1: return (void*)k_stream<KIND, B, 1>;
    case 2: return (void*)k_stream<KIND, B, 2>;
    case 3: return (void*)k_stream<KIND, B, 3>;
    case 4: return (void*)k_stream<KIND, B, 4>;
    case 5: return B == 1 ? (void*)k_stream<KIND, 1, 5> : nullptr;
    case 6: return B == 1 ? (void*)k_stream<KIND, 1, 6> : nullptr;
    case 8: return B == 1 ? (void*)k_stream<KIND, 1, 8> : nullptr;
    default: return nullptr;
  }
}

template <int KIND>
static void* stream_kernel(int B, int V) {
  if (V == 7) V = 8;
  return B == 1 ? stream_kernel_for_V<KIND, 1>(V) : stream_kernel_for_V<KIND, 4>(V);
}

int stream_ctas_max(int CH_rows, long long rows, int target) {
  long long need = (rows + CH_rows - 1) / CH_rows;
  long long gsz = std::max<long long>(need, std::min<long long>(target, rows));
  return (int)std::max<long long>(1, gsz);
}

static int launch_stream(int kind, StreamParams& p, long long rows, int target_ctas,
                         int ring_budget, cudaStream_t stream, int* grid_out, bool pdl) {
  const int Bt = p.B == 1 ? 1 : 4;
  // At most 256 rows per CTA, or more when the CTA target (one per SM) would
  // otherwise need a second wave of CTAs (a dense or nearly dense MLP) and the
  // larger per-row arrays still fit in shared memory.
  int CH = 256;
  if (target_ctas > 0) {
    const long long per = (rows + target_ctas - 1) / target_ctas;
    StreamGeom wide;
    if (per > CH && per <= 1024 &&
        make_geom(wide, p.d, Bt, ring_budget, (int)per, is_w4(kind), !is_wo(kind)))
      CH = (int)per;
  }
  if (!make_geom(p.g, p.d, Bt, ring_budget, CH, is_w4(kind), !is_wo(kind))) return DV_ERR_UNSUPPORTED;
  const int V = pick_V(p.d / 8, (is_w4(kind) && Bt == 1) ? kW4Threads : (Bt == 1 ? 512 : 384));
  void* fn = nullptr;
  switch (kind) {
    case KIND_MLP: fn = stream_kernel<KIND_MLP>(Bt, V); break;
    case KIND_MLP4: fn = stream_kernel<KIND_MLP4>(Bt, V); break;
    case KIND_QKV: fn = stream_kernel<KIND_QKV>(Bt, V); break;
    case KIND_WO: fn = stream_kernel<KIND_WO>(Bt, V); break;
    case KIND_QKV4: fn = stream_kernel<KIND_QKV4>(Bt, V); break;
    case KIND_WO4: fn = stream_kernel<KIND_WO4>(Bt, V); break;
    case KIND_P1: fn = stream_kernel<KIND_P1>(Bt, V); break;
  }
  if (!fn) return DV_ERR_UNSUPPORTED;
  int grid = stream_ctas_max(CH, rows, target_ctas);
  if (rows == 0) grid = 1;
  if (grid_out) *grid_out = grid;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, p.g.total) !=
      cudaSuccess)
    return DV_ERR_LAUNCH;
  void* args[] = {&p};
  static const int tags[7] = {DV_TAG_MLP, DV_TAG_QKV, DV_TAG_PRED1, DV_TAG_WO, DV_TAG_MLP,
                              DV_TAG_QKV, DV_TAG_WO};
  note_launch(tags[kind], 0, stream);
  const cudaError_t e = launch_k(fn, dim3(grid), dim3(p.g.T + 32), p.g.total, stream, args, pdl);
  note_launch(tags[kind], 1, stream);
  return e == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

int reduce_launch(const float* part, int G, int B, int d, const uint16_t* x, const uint16_t* bias,
                  uint16_t* out, cudaStream_t stream) {
  dim3 grid((d + 63) / 64, B);
  void* args[] = {&part, &G, &B, &d, &x, &bias, &out};
  note_launch(DV_TAG_REDUCE, 0, stream);
  const cudaError_t e = launch_k((const void*)k_reduce, grid, dim3(256), 0, stream, args, true);
  note_launch(DV_TAG_REDUCE, 1, stream);
  return e == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

// ---- public launchers (declared in dv_internal.h) -------------------------

int launch_mlp(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g, const uint16_t* ln_b,
               float eps, const uint16_t* fc1, const uint16_t* b1, const uint16_t* fc2T,
               const uint16_t* b2, const int32_t* idx, int k, const int32_t* dev_count, int flags,
               uint16_t* out, int* st, float* part, int target_ctas, int ring_budget,
               cudaStream_t stream, bool pdl) {
  const uint16_t* resid = (flags & DV_NO_RESIDUAL) ? nullptr : x;
  StreamParams p{};
  p.d = d; p.B = B; p.x = x; p.ln_g = ln_g; p.ln_b = ln_b; p.eps = eps;
  p.W0 = fc1; p.W1 = fc2T; p.bias0 = b1; p.idx = idx; p.k = k; p.dev_count = dev_count;
  p.n_rows_total = F; p.flags = flags; p.part = part; p.st = st;
  p.active_cnt = (flags & DV_SKIP_INACTIVE) ? g_count_active : nullptr;
  int grid = 0;
  int rc = launch_stream(KIND_MLP, p, k, target_ctas, ring_budget, stream, &grid, pdl);
  if (rc != DV_OK) return rc;
  return reduce_launch(part, grid, B, d, resid, b2, out, stream);
}

int launch_mlp_w4(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g,
                  const uint16_t* ln_b, float eps, const uint8_t* fc1q, const uint16_t* b1,
                  const uint8_t* fc2Tq, const uint16_t* b2, const int32_t* idx, int k,
                  const int32_t* dev_count, int flags, uint16_t* out, int* st, float* part,
                  int target_ctas, int ring_budget, cudaStream_t stream, bool pdl) {
  const uint16_t* resid = (flags & DV_NO_RESIDUAL) ? nullptr : x;
  StreamParams p{};
  p.d = d; p.B = B; p.x = x; p.ln_g = ln_g; p.ln_b = ln_b; p.eps = eps;
  p.W0 = reinterpret_cast<const uint16_t*>(fc1q); p.W1 = reinterpret_cast<const uint16_t*>(fc2Tq);
  p.bias0 = b1; p.idx = idx; p.k = k; p.dev_count = dev_count;
  p.n_rows_total = F; p.flags = flags; p.part = part; p.st = st;
  int grid = 0;
  int rc = launch_stream(KIND_MLP4, p, k, target_ctas, ring_budget, stream, &grid, pdl);
  if (rc != DV_OK) return rc;
  return reduce_launch(part, grid, B, d, resid, b2, out, stream);
}

int launch_qkv(const uint16_t* x, int B, int d, int G, int dh, int h_kv, const uint16_t* ln_g,
               const uint16_t* ln_b, float eps, const uint16_t* Wq, const uint16_t* bq,
               const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv, const uint16_t* bv,
               const int32_t* idx, int k, const int32_t* dev_count, float scale, float* qbuf,
               uint16_t* K, uint16_t* V, int n, int n_max, uint16_t* Kr, uint16_t* Vr,
               const int32_t* kept_count, int b_max, uint16_t* y_side, uint32_t* kv_missing,
               int fill_clear, int* zero_cnt, int n_zero, const uint16_t* P1, int n_pred,
               int relu, float* u_out, int* st, int target_ctas, int ring_budget,
               cudaStream_t stream, bool pdl, bool w4) {
  StreamParams p{};
  p.fill_clear = fill_clear;
  if (w4) P1 = nullptr;  // 4-bit Q/K/V rows: the predictor's fp16 rows run on their own
  p.zero_cnt = zero_cnt; p.n_zero = n_zero;
  p.P1 = P1; p.n_pred = P1 ? n_pred : 0; p.relu = relu; p.u_out = u_out;
  p.d = d; p.B = B; p.x = x; p.ln_g = ln_g; p.ln_b = ln_b; p.eps = eps;
  p.W0 = Wq; p.W1 = Wk; p.W2 = Wv; p.bias0 = bq; p.bias1 = bk; p.bias2 = bv;
  p.idx = idx; p.k = k; p.dev_count = dev_count; p.G = G; p.dh = dh; p.h_kv = h_kv;
  p.scale = scale; p.qbuf = qbuf; p.K = K; p.V = V; p.n = n; p.n_max = n_max;
  p.Kr = Kr; p.Vr = Vr; p.kept_count = kept_count; p.b_max = b_max;
  p.y_side = y_side; p.kv_missing = kv_missing; p.st = st;
  return launch_stream(w4 ? KIND_QKV4 : KIND_QKV, p, (long long)k * (G + 2) * dh + p.n_pred,
                       target_ctas, ring_budget, stream, nullptr, pdl);
}

int launch_wo(const uint16_t* x, int B, int d, int G, int dh, int h_kv, const uint16_t* WoT,
              const uint16_t* bo, const int32_t* idx, int k, const int32_t* dev_count,
              const float* H, uint16_t* out, int* st, float* part, int target_ctas,
              int ring_budget, cudaStream_t stream, bool w4) {
  // x: residual added by the reduce (NULL: none)
  StreamParams p{};
  p.d = d; p.B = B; p.x = x; p.W0 = WoT; p.idx = idx; p.k = k; p.dev_count = dev_count;
  p.G = G; p.dh = dh; p.h_kv = h_kv; p.Hc = H; p.part = part; p.st = st;
  int grid = 0;
  int rc = launch_stream(w4 ? KIND_WO4 : KIND_WO, p, (long long)k * G * dh, target_ctas,
                         ring_budget, stream,
                         &grid, true);
  if (rc != DV_OK) return rc;
  return reduce_launch(part, grid, B, d, x, bo, out, stream);
}

// First predictor layer on the side stream (batch > 1, where it is not fused
// into the QKV launch): u[b][j] = act(sum_c y[b][c] P1[j][c]), small CTAs that
// share SMs with the main-stream kernels.
int launch_pred1_gemv(const uint16_t* y, int B, int d, const uint16_t* P1, int r, int relu,
                      float* u, int target_ctas, cudaStream_t stream) {
  const int threads = 256, nw = threads / 32;
  const int g1 = std::max(1, std::min(target_ctas, (r + 2 * nw - 1) / (2 * nw)));
  note_launch(DV_TAG_PRED1, 0, stream);
  if (B == 1)
    k_gemv<uint16_t, 1, 2><<<g1, threads, 0, stream>>>(y, B, d, P1, r, u, r, relu);
  else
    k_gemv<uint16_t, 4, 2><<<g1, threads, 0, stream>>>(y, B, d, P1, r, u, r, relu);
  note_launch(DV_TAG_PRED1, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

// Second predictor layer: scores[b][row] = sum_j u[b][j] P2[row][j].
int launch_pred2(const float* u, int B, int r, const uint16_t* P2, int N, float* scores, int ld,
                 int target_ctas, cudaStream_t stream) {
  const int threads = 256, nw = threads / 32;
  const int g2 = std::max(1, std::min(target_ctas, (N + 2 * nw - 1) / (2 * nw)));
  note_launch(DV_TAG_PRED2, 0, stream);
  if (B == 1)
    k_gemv<float, 1, 2><<<g2, threads, 0, stream>>>(u, B, r, P2, N, scores, ld, 0);
  else
    k_gemv<float, 4, 2><<<g2, threads, 0, stream>>>(u, B, r, P2, N, scores, ld, 0);
  note_launch(DV_TAG_PRED2, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

// Both predictor layers: P1 streamed by the weight-streaming engine (dense
// rows, raw input, no LayerNorm), then the second layer.
int launch_pred1(const uint16_t* y, int B, int d, const uint16_t* P1, int r, int relu, float* u,
                 int target_ctas, int ring_budget, cudaStream_t stream) {
  StreamParams p{};
  p.d = d; p.B = B; p.x = y; p.W0 = P1; p.idx = nullptr; p.k = r; p.n_rows_total = r;
  p.u_out = u; p.relu = relu; p.n_pred = r;
  return launch_stream(KIND_P1, p, r, target_ctas, ring_budget, stream, nullptr, false);
}

int launch_predict(const uint16_t* y, int B, int d, const uint16_t* P1, int r,
                   const uint16_t* P2, int N, int relu, float* scores, int ld, float* u,
                   int target_ctas, int ring_budget, cudaStream_t stream) {
  int rc = launch_pred1(y, B, d, P1, r, relu, u, target_ctas, ring_budget, stream);
  if (rc != DV_OK) return rc;
  return launch_pred2(u, B, r, P2, N, scores, ld, target_ctas, stream);
}

size_t stream_part_bytes(int d, int B, long long max_rows, int target_ctas) {
  const int CH = 256;
  const int grid = stream_ctas_max(CH, max_rows, target_ctas);
  return (size_t)grid * B * d * sizeof(float);
}

}  // namespace dv
