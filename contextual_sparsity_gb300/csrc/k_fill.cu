// k_fill.cu -- recompute of missing K/V rows before a decode step (sm_103a).
//
// "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time", §4.2:
// a step computes k, v only for the attention units it selects; for the other
// units the token's input y is kept aside and its k, v are marked missing.
// When a later step selects such a unit, the missing rows are computed from
// the kept inputs before that step's attention reads them:
//   k_t = LN1(y_t) W^K_u^T + b^K_u,  v_t = LN1(y_t) W^V_u^T + b^V_u  (fp16),
// for every position t of the unit still marked missing. LN1(y_t) is held in
// shared memory as fp16 (two tokens per pass), so the recomputed rows can
// differ from the QKV launch's fp32 form in the last bit.
//
// A unit's missing positions are always a suffix [n - depth, n) of the cache:
// positions are marked when the unit is skipped, and a step that selects the
// unit fills all of its marks (the marks themselves are cleared by that step's
// QKV launch, which runs after this kernel). So each CTA finds `depth` by
// scanning the marks backwards from n - 1, 32 positions per warp step.
#include "dv_internal.h"

namespace dv {

constexpr int kFillRows = 24;   // K/V rows of one unit per CTA (12 warps x 2 rows)
constexpr int kFillRowsW = 2;   // rows per warp
constexpr int kFillUnroll = 4;  // 16-byte loads per row in flight per lane
constexpr int kFillTok = 2;     // missing tokens per pass (their LN1(y) in shared memory, fp16)
constexpr int kFillGroups = 8;  // CTAs that split a unit's passes between them
constexpr int kFillThreads = 384;

struct FillParams {
  const uint16_t* y_side;    // [B][n_max][d]
  const uint32_t* missing;   // [B][n_max][words]
  const uint16_t *ln_g, *ln_b;
  float eps;
  const uint16_t *Wk, *bk, *Wv, *bv;
  const int32_t* idx;        // selected units (NULL: all)
  const int32_t* dev_count;
  int k, h_kv, dh, d, n, n_max;
  uint16_t *K, *V;           // [B][h_kv][n_max][dh]
  // The retained buffer (batch 1, nullable): the tokens decoded since the
  // selection sit after the kept rows, position t at slot
  // kept_count[u] - (n - t), and get the recomputed rows too.
  uint16_t *Kr, *Vr;         // [h_kv][b_max][dh]
  const int32_t* kept_count;
  int b_max;
  int* st;
};

// 12 warps and 2 d bytes of shared memory per token slot (48 KB at d = 12288):
// on the side stream a CTA runs beside the Wo / MLP streaming CTAs where their
// registers leave room (measured faster than 8 warps of <= 64 registers).
// 4-bit rows (DV_W4): a packed row holds d/2 bytes of codes (column 2i in the
// low nibble of byte i, stored as q + 8), then the d/128 fp16 group scales,
// padded to 16 bytes; a weight is q s, exact in fp32.
__host__ __device__ inline size_t fill_w4_row_bytes(int d) { return (size_t)((d / 2 + d / 64 + 15) / 16 * 16); }

// Eight codes of a 32-bit word as exact floats q in column order.
DV_DEV void fill_w4_decode(uint32_t w, float* f) {
#pragma unroll
  for (int k = 0; k < 8; ++k) f[k] = (float)((int)((w >> (4 * k)) & 15u) - 8);
}

template <bool W4>
__global__ void __launch_bounds__(kFillThreads, 2) k_kv_fill(const FillParams p) {
  extern __shared__ __align__(16) uint16_t zs[];  // [kFillTok][d]: LN1 of the pass's tokens
  __shared__ float red[kFillThreads / 32][kFillTok];
  __shared__ float stat[kFillTok][2];
  __shared__ int depth_s;
  // The marks, the kept inputs and the index list come from earlier kernels.
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();

  const int rb = blockIdx.x, e = blockIdx.y;
  const int b = blockIdx.z / kFillGroups, grp = blockIdx.z % kFillGroups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int kk = p.k;
  if (p.dev_count) kk = min(kk, *p.dev_count);
  if (e >= kk) return;
  const int u = p.idx ? p.idx[e] : e;
  if (u < 0 || u >= p.h_kv) {
    if (threadIdx.x == 0) flag(p.st, DV_DEV_BAD_INDEX);
    return;
  }
  const int words = (p.h_kv + 31) >> 5;
  const uint32_t* marks = p.missing + (size_t)b * p.n_max * words + (u >> 5);
  const uint32_t bit = 1u << (u & 31);
  if (warp == 0) {
    int depth = 0;
    for (int top = p.n - 1; top >= 0; top -= 32) {
      const int t = top - lane;
      const bool miss = t >= 0 && (marks[(size_t)t * words] & bit);
      const unsigned present = __ballot_sync(0xffffffffu, !miss);
      if (present) {
        depth += __ffs(present) - 1;
        break;
      }
      depth += 32;
    }
    if (lane == 0) depth_s = depth;
  }
  __syncthreads();
  const int depth = depth_s;
  if (depth == 0) return;

  const int d = p.d, nvec = d >> 3;
  // This warp's rows of the unit's [W^K; W^V] (2 dh rows).
  const uint8_t* wrow[kFillRowsW];
  int rrow[kFillRowsW];
  const size_t rbytes = W4 ? fill_w4_row_bytes(d) : (size_t)d * 2;
#pragma unroll
  for (int r = 0; r < kFillRowsW; ++r) {
    int row = rb * kFillRows + warp * kFillRowsW + r;
    rrow[r] = row;
    if (row >= 2 * p.dh) row = 0;  // (no such row: computed, never stored)
    const bool isk = row < p.dh;
    const int c = isk ? row : row - p.dh;
    wrow[r] = reinterpret_cast<const uint8_t*>(isk ? p.Wk : p.Wv) + ((size_t)u * p.dh + c) * rbytes;
  }

  // Passes of kFillTok tokens; the kFillGroups CTAs of a row block take
  // every kFillGroups-th pass.
  for (int t0 = p.n - depth + grp * kFillTok; t0 < p.n; t0 += kFillGroups * kFillTok) {
    const int nt = min(kFillTok, p.n - t0);
    // --- LN1 of the kept inputs (two passes over the stored fp16 rows)
    float s1[kFillTok];
#pragma unroll
    for (int j = 0; j < kFillTok; ++j) {
      s1[j] = 0.f;
      if (j < nt) {
        const uint16_t* y = p.y_side + ((size_t)b * p.n_max + t0 + j) * d;
        for (int v = threadIdx.x; v < nvec; v += kFillThreads) {
          const uint4 yv = *reinterpret_cast<const uint4*>(y + v * 8);
          *reinterpret_cast<uint4*>(zs + (size_t)j * d + v * 8) = yv;
          float f[8];
          h8_to_f8(yv, f);
#pragma unroll
          for (int i = 0; i < 8; ++i) s1[j] += f[i];
        }
      }
      s1[j] = warp_sum(s1[j]);
      if (lane == 0) red[warp][j] = s1[j];
    }
    __syncthreads();
    if (threadIdx.x < kFillTok) {
      float t = 0.f;
      for (int w = 0; w < kFillThreads / 32; ++w) t += red[w][threadIdx.x];
      stat[threadIdx.x][0] = t / d;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kFillTok; ++j) {
      float s2 = 0.f;
      if (j < nt) {
        const float mu = stat[j][0];
        for (int v = threadIdx.x; v < nvec; v += kFillThreads) {
          float f[8];
          h8_to_f8(*reinterpret_cast<const uint4*>(zs + (size_t)j * d + v * 8), f);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float c = f[i] - mu;
            s2 = fmaf(c, c, s2);
          }
        }
      }
      s2 = warp_sum(s2);
      if (lane == 0) red[warp][j] = s2;
    }
    __syncthreads();
    if (threadIdx.x < kFillTok) {
      float t = 0.f;
      for (int w = 0; w < kFillThreads / 32; ++w) t += red[w][threadIdx.x];
      stat[threadIdx.x][1] = 1.0f / sqrtf(t / d + p.eps);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nt * d; i += kFillThreads) {
      const int j = i / d, c = i - j * d;
      const float g = p.ln_g ? h2f(p.ln_g[c]) : 1.f;
      const float bb = p.ln_b ? h2f(p.ln_b[c]) : 0.f;
      zs[i] = f2h((h2f(zs[i]) - stat[j][0]) * stat[j][1] * g + bb);
    }
    __syncthreads();

    // --- kFillRowsW rows x nt tokens per warp: lanes stride over d, 16 bytes
    // per row per step, kFillUnroll steps of loads in flight
    float acc[kFillRowsW][kFillTok];
#pragma unroll
    for (int r = 0; r < kFillRowsW; ++r)
#pragma unroll
      for (int j = 0; j < kFillTok; ++j) acc[r][j] = 0.f;
    if constexpr (W4) {
      // The fp16 loop's shape over 8-column vectors: one 32-bit word of codes
      // per vector (byte offset 4 v), its group's scale (group v / 16).
      for (int v0 = lane; v0 < nvec; v0 += 32 * kFillUnroll) {
        uint32_t wc[kFillUnroll][kFillRowsW];
        float sc[kFillUnroll][kFillRowsW];
#pragma unroll
        for (int q = 0; q < kFillUnroll; ++q) {
          const int v = v0 + q * 32;
#pragma unroll
          for (int r = 0; r < kFillRowsW; ++r) {
            const bool on = v < nvec;
            wc[q][r] = on ? __ldg(reinterpret_cast<const unsigned int*>(wrow[r]) + v) : 0u;
            sc[q][r] = on ? __half2float(__ldg(reinterpret_cast<const __half*>(wrow[r] + d / 2) + (v >> 4)))
                          : 0.f;
          }
        }
#pragma unroll
        for (int q = 0; q < kFillUnroll; ++q) {
          const int v = v0 + q * 32;
          if (v >= nvec) break;
          float wf[kFillRowsW][8];
#pragma unroll
          for (int r = 0; r < kFillRowsW; ++r) {
            fill_w4_decode(wc[q][r], wf[r]);
#pragma unroll
            for (int i = 0; i < 8; ++i) wf[r][i] *= sc[q][r];
          }
#pragma unroll
          for (int j = 0; j < kFillTok; ++j) {
            if (j >= nt) break;
            float z[8];
            h8_to_f8(*reinterpret_cast<const uint4*>(zs + (size_t)j * d + v * 8), z);
#pragma unroll
            for (int r = 0; r < kFillRowsW; ++r)
#pragma unroll
              for (int i = 0; i < 8; ++i) acc[r][j] = fmaf(z[i], wf[r][i], acc[r][j]);
          }
        }
      }
    } else
    for (int v0 = lane; v0 < nvec; v0 += 32 * kFillUnroll) {
      uint4 w[kFillUnroll][kFillRowsW];
#pragma unroll
      for (int q = 0; q < kFillUnroll; ++q) {
        const int v = v0 + q * 32;
#pragma unroll
        for (int r = 0; r < kFillRowsW; ++r)
          w[q][r] = v < nvec ? ld_nc_v4(wrow[r] + (size_t)v * 16) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kFillUnroll; ++q) {
        const int v = v0 + q * 32;
        if (v >= nvec) break;
        float wf[kFillRowsW][8];
#pragma unroll
        for (int r = 0; r < kFillRowsW; ++r) h8_to_f8(w[q][r], wf[r]);
#pragma unroll
        for (int j = 0; j < kFillTok; ++j) {
          if (j >= nt) break;
          float z[8];
          h8_to_f8(*reinterpret_cast<const uint4*>(zs + (size_t)j * d + v * 8), z);
#pragma unroll
          for (int r = 0; r < kFillRowsW; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[r][j] = fmaf(z[i], wf[r][i], acc[r][j]);
        }
      }
    }
    // Lanes leave the loops above after different trip counts; the warp
    // reconverges here before the shuffles sum the partials.
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kFillRowsW; ++r)
#pragma unroll
      for (int j = 0; j < kFillTok; ++j) acc[r][j] = warp_sum(acc[r][j]);
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kFillRowsW; ++r) {
        if (rrow[r] >= 2 * p.dh) continue;
        const bool isk = rrow[r] < p.dh;
        const int c = isk ? rrow[r] : rrow[r] - p.dh;
        const uint16_t* bias = isk ? p.bk : p.bv;
        const float bv = bias ? h2f(bias[u * p.dh + c]) : 0.f;
        uint16_t* cache = isk ? p.K : p.V;
        uint16_t* kept = isk ? p.Kr : p.Vr;
        const int kc = kept ? p.kept_count[u] : 0;
        for (int j = 0; j < nt; ++j) {
          const uint16_t val = f2h(acc[r][j] + bv);
          cache[(((size_t)b * p.h_kv + u) * p.n_max + t0 + j) * p.dh + c] = val;
          if (kept) {
            const int slot = kc - (p.n - (t0 + j));
            if (slot >= 0 && slot < p.b_max) kept[((size_t)u * p.b_max + slot) * p.dh + c] = val;
          }
        }
      }
    }
    __syncthreads();  // the next pass overwrites zs
  }
}

int launch_kv_fill(const uint16_t* y_side, const uint32_t* missing, int B, int d, int h_kv,
                   int dh, const uint16_t* ln_g, const uint16_t* ln_b, float eps,
                   const uint16_t* Wk, const uint16_t* bk, const uint16_t* Wv,
                   const uint16_t* bv, const int32_t* idx, int k, const int32_t* dev_count,
                   uint16_t* K, uint16_t* V, int n, int n_max, int* st, cudaStream_t stream,
                   bool pdl, uint16_t* Kr, uint16_t* Vr, const int32_t* kept_count, int b_max,
                   bool w4) {
  FillParams p{};
  p.Kr = Kr; p.Vr = Vr; p.kept_count = kept_count; p.b_max = b_max;
  p.y_side = y_side; p.missing = missing; p.ln_g = ln_g; p.ln_b = ln_b; p.eps = eps;
  p.Wk = Wk; p.bk = bk; p.Wv = Wv; p.bv = bv; p.idx = idx; p.dev_count = dev_count;
  p.k = k; p.h_kv = h_kv; p.dh = dh; p.d = d; p.n = n; p.n_max = n_max; p.K = K; p.V = V;
  p.st = st;
  const size_t smem = (size_t)kFillTok * d * sizeof(uint16_t);
  const void* fn = w4 ? (const void*)k_kv_fill<true> : (const void*)k_kv_fill<false>;
  if (w4 && d % 128 != 0) return DV_ERR_DIMS;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
      cudaSuccess)
    return DV_ERR_LAUNCH;
  dim3 grid((2 * dh + kFillRows - 1) / kFillRows, k, B * kFillGroups);
  void* args[] = {&p};
  note_launch(DV_TAG_KVFILL, 0, stream);
  const cudaError_t e =
      launch_k(fn, grid, dim3(kFillThreads), smem, stream, args, pdl);
  note_launch(DV_TAG_KVFILL, 1, stream);
  return e == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
