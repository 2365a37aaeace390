// k_select.cu -- set formation on the device (sm_103a).
//
// Top-k ("Deja Vu", §2.3: |S| <= (1 - sparsity) N; §4.1: the predictor's set at
// a test-time sparsity level): one CTA per row runs an MSB-first radix select
// over order-preserving 32-bit keys (4 passes of 8 bits, shared-memory
// histogram), finds the k-th largest key T and how many keys equal to T are
// needed, then compacts in index order with two block scans, so the set comes
// out ascending and equal scores go to the lower index -- bit-exact and
// deterministic. The union of a batch's sets ("Deja Vu", App. C.1) is a
// shared-memory bitmap compacted the same way.
#include <cooperative_groups.h>

#include "dv_internal.h"

namespace cg = cooperative_groups;

namespace dv {

constexpr int kTopkThreads = 256;  // small: fits next to a weight-streaming CTA

// Order-preserving key: larger float -> larger key; -0 and +0 map together.
DV_DEV uint32_t fkey(float f) {
  if (f == 0.f) return 0x80000000u;
  const uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the total to *total. Uses `tmp` (32 ints) in shared memory.
DV_DEV int block_exscan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    tmp[lane] = w;  // inclusive prefix of warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
  *total = tmp[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kTopkThreads) k_topk(const float* __restrict__ scores, int ld,
                                                       int N, const int* __restrict__ k_per_row,
                                                       int k_default, int32_t* __restrict__ idx,
                                                       int ld_idx, int* st) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t whist[256 * (kTopkThreads / 32)];
  __shared__ int tmp[32];
  __shared__ uint32_t sh_prefix, sh_krem;
  const int row = blockIdx.x;
  const float* s = scores + (size_t)row * ld;
  int32_t* out = idx + (size_t)row * ld_idx;
  int k = k_per_row ? k_per_row[row] : k_default;
  k = max(0, min(k, N));
  const int tid = threadIdx.x;
  if (k == 0) return;

  // NaN check (sets the status bit; NaN keys sort below everything finite).
  bool nan_seen = false;
  for (int i = tid; i < N; i += blockDim.x) nan_seen |= isnan(s[i]);
  if (__syncthreads_or(nan_seen) && tid == 0) flag(st, DV_DEV_NONFINITE);

  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  const int warp = tid >> 5, nwarp = blockDim.x >> 5;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256 * nwarp; i += blockDim.x) whist[i] = 0;
    __syncthreads();
    uint32_t* my = whist + warp * 256;  // per-warp histogram: no cross-warp contention
    for (int i = tid; i < N; i += blockDim.x) {
      const float f = s[i];
      const uint32_t key = isnan(f) ? 0u : fkey(f);
      if ((key & mask) == prefix) atomicAdd(&my[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    for (int i = tid; i < 256; i += blockDim.x) {
      uint32_t t = 0;
      for (int w = 0; w < nwarp; ++w) t += whist[w * 256 + i];
      hist[i] = t;
    }
    __syncthreads();
    if (tid < 32) {
      // lane L owns digits [255 - 8L - 7, 255 - 8L], scanned from the top.
      uint32_t c[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * tid - j];
        loc += c[j];
      }
      uint32_t incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      const uint32_t excl = incl - loc;  // keys with a higher digit than my range
      if (excl < krem && krem <= incl) {
        uint32_t above = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= krem) {
            const uint32_t digit = 255 - 8 * tid - j;
            sh_prefix = prefix | (digit << shift);
            sh_krem = krem - above;
            break;
          }
          above += c[j];
        }
      }
    }
    __syncthreads();
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // the k-th largest key; krem of the keys == T are taken

  // Ordered compaction: thread t owns [c0, c1).
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int c0 = min(N, tid * per), c1 = min(N, c0 + per);
  int gt = 0, eq = 0;
  for (int i = c0; i < c1; ++i) {
    const float f = s[i];
    const uint32_t key = isnan(f) ? 0u : fkey(f);
    gt += key > T;
    eq += key == T;
  }
  int tot;
  const int eq_before = block_exscan(eq, tmp, &tot);
  int take_eq = min(eq, max(0, (int)krem - eq_before));
  const int pos0 = block_exscan(gt + take_eq, tmp, &tot);
  int pos = pos0;
  for (int i = c0; i < c1; ++i) {
    const float f = s[i];
    const uint32_t key = isnan(f) ? 0u : fkey(f);
    if (key > T) {
      out[pos++] = i;
    } else if (key == T && take_eq > 0) {
      out[pos++] = i;
      --take_eq;
    }
  }
}

// ---------------------------------------------------------------------------
// Cluster top-k: one cluster of 8 CTAs per row. CTA r of the cluster owns
// positions [r C, (r+1) C) (C = ceil(N / 8)); its thread t keeps the KPT
// consecutive keys starting at r C + t KPT in registers. Each radix pass builds
// per-warp histograms, sums them into a CTA histogram, and every CTA reads the
// 8 CTA histograms through distributed shared memory in rank order (so every
// CTA takes the same, deterministic decision). The compaction offsets come
// from the CTAs' totals exchanged the same way. No global atomics, no spin.
// ---------------------------------------------------------------------------
constexpr int kClusterTopk = 8;

template <int KPT>
__global__ void __cluster_dims__(kClusterTopk, 1, 1) __launch_bounds__(256, 4)
    k_topk_cluster(const float* __restrict__ scores, int ld, int N, int k,
                   int32_t* __restrict__ idx, int ld_idx, int* st) {
  cg::cluster_group cluster = cg::this_cluster();
  __shared__ uint32_t whist[8][256];
  __shared__ uint32_t ctah[256];
  __shared__ int tmp[32];
  __shared__ uint32_t sh_prefix, sh_krem;
  __shared__ int tot[2];  // this CTA's count of keys > T, == T
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.x / kClusterTopk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const float* s = scores + (size_t)row * ld;
  int32_t* out = idx + (size_t)row * ld_idx;
  const int C = (N + kClusterTopk - 1) / kClusterTopk;
  const int c0 = min(N, rank * C), c1 = min(N, c0 + C);
  const int p0 = c0 + tid * KPT;
  k = max(1, min(k, N));

  uint32_t key[KPT];
  bool nan_seen = false;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int i = p0 + j;
    key[j] = 0u;
    if (i < c1) {
      const float f = s[i];
      nan_seen |= isnan(f);
      key[j] = isnan(f) ? 0u : fkey(f);
    }
  }
  if (__syncthreads_or(nan_seen) && tid == 0) flag(st, DV_DEV_NONFINITE);

  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 8 * 256; i += blockDim.x) (&whist[0][0])[i] = 0;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (p0 + j < c1 && (key[j] & mask) == prefix)
        atomicAdd(&whist[warp][(key[j] >> shift) & 255u], 1u);
    __syncthreads();
    {
      uint32_t t = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) t += whist[w][tid];
      ctah[tid] = t;
    }
    cluster.sync();
    {
      // Cluster histogram: thread t gathers bin t from the 8 CTAs (rank order).
      uint32_t t = 0;
#pragma unroll
      for (int r = 0; r < kClusterTopk; ++r) t += cluster.map_shared_rank(ctah, r)[tid];
      whist[0][tid] = t;
    }
    __syncthreads();
    if (warp == 0) {
      // lane L owns digits [255 - 8L - 7, 255 - 8L], scanned from the top.
      uint32_t c[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = whist[0][255 - 8 * lane - j];
        loc += c[j];
      }
      uint32_t incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - loc;
      if (excl < krem && krem <= incl) {
        uint32_t above = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (above + c[j] >= krem) {
            sh_prefix = prefix | ((uint32_t)(255 - 8 * lane - j) << shift);
            sh_krem = krem - above;
            break;
          }
          above += c[j];
        }
      }
    }
    cluster.sync();  // every CTA is done reading the others' histograms
    prefix = sh_prefix;
    krem = sh_krem;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;

  // Ordered compaction.
  int gt = 0, eq = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j)
    if (p0 + j < c1) {
      gt += key[j] > T;
      eq += key[j] == T;
    }
  int cta_eq, cta_gt;
  const int eq_before_local = block_exscan(eq, tmp, &cta_eq);
  const int gt_dummy = block_exscan(gt, tmp, &cta_gt);
  (void)gt_dummy;
  if (tid == 0) {
    tot[0] = cta_gt;
    tot[1] = cta_eq;
  }
  cluster.sync();
  int eq_before_cta = 0, out_before_cta = 0;
  for (int r = 0; r < rank; ++r) {
    const int* o = cluster.map_shared_rank(tot, r);
    const int g_r = o[0], e_r = o[1];
    const int take_r = min(e_r, max(0, (int)krem - eq_before_cta));
    out_before_cta += g_r + take_r;
    eq_before_cta += e_r;
  }
  int take_eq = min(eq, max(0, (int)krem - (eq_before_cta + eq_before_local)));
  int total_unused;
  int pos = out_before_cta + block_exscan(gt + take_eq, tmp, &total_unused);
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    if (p0 + j >= c1) break;
    if (key[j] > T) {
      out[pos++] = p0 + j;
    } else if (key[j] == T && take_eq > 0) {
      out[pos++] = p0 + j;
      --take_eq;
    }
  }
  cluster.sync();  // keep this CTA's shared memory alive until all peers read it
}

// ---------------------------------------------------------------------------
// Short rows (N <= kSmallN, e.g. the head scores): one CTA of 256 threads per
// row (small enough to share an SM with a weight-streaming CTA) loads the
// row's keys into shared memory once, runs the 4-pass radix select there and
// compacts in index order with warp ballots over per-warp segments.
// ---------------------------------------------------------------------------
constexpr int kSmallN = 4096;

DV_DEV uint32_t key_of(float f) { return isnan(f) ? 0u : fkey(f); }

// Scanning hist[0, nb) from the top bin down, find the bin where the running
// count reaches krem: sh[0] = that bin, sh[1] = krem minus the keys above it.
DV_DEV void select_bin(const uint32_t* hist, int nb, uint32_t krem, uint32_t* sh, int* tmp) {
  const int per = nb / (int)blockDim.x;
  const int top = nb - 1 - per * (int)threadIdx.x;
  uint32_t loc = 0;
  for (int j = 0; j < per; ++j) loc += hist[top - j];
  int total;
  const uint32_t excl = (uint32_t)block_exscan((int)loc, tmp, &total);
  if (excl < krem && krem <= excl + loc) {
    uint32_t above = excl;
    for (int j = 0; j < per; ++j) {
      const uint32_t c = hist[top - j];
      if (above + c >= krem) {
        sh[0] = (uint32_t)(top - j);
        sh[1] = krem - above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTopkThreads, 4) k_topk_small(const float* __restrict__ scores,
                                                                 int ld, int N, int k,
                                                                 int32_t* __restrict__ idx,
                                                                 int ld_idx, int* st) {
  constexpr int NW = kTopkThreads / 32;
  __shared__ uint32_t keys[kSmallN];
  __shared__ uint32_t hist[256];
  __shared__ int tmp[32];
  __shared__ uint32_t sh[2];
  __shared__ int wgt[NW], weq[NW];
  const float* s = scores + (size_t)blockIdx.x * ld;
  int32_t* out = idx + (size_t)blockIdx.x * ld_idx;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  k = max(1, min(k, N));

  bool nan_seen = false;
  for (int i = tid; i < N; i += kTopkThreads) {
    const float f = s[i];
    nan_seen |= isnan(f);
    keys[i] = key_of(f);
  }
  if (__syncthreads_or(nan_seen) && tid == 0) flag(st, DV_DEV_NONFINITE);

  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += kTopkThreads) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += kTopkThreads)
      if ((keys[i] & mask) == prefix) atomicAdd(&hist[(keys[i] >> shift) & 255u], 1u);
    __syncthreads();
    select_bin(hist, 256, krem, sh, tmp);
    prefix |= sh[0] << shift;
    krem = sh[1];
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;  // the k-th largest key; krem of the keys equal to T are taken

  // Ordered compaction over warp segments (multiples of 32 positions).
  const int seg = (N + kTopkThreads - 1) / kTopkThreads * 32;
  const int w0 = min(N, warp * seg), w1 = min(N, w0 + seg);
  int gt = 0, eq = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool v = i < w1;
    const uint32_t key = v ? keys[i] : 0u;
    gt += __popc(__ballot_sync(0xffffffffu, v && key > T));
    eq += __popc(__ballot_sync(0xffffffffu, v && key == T));
  }
  if (lane == 0) {
    wgt[warp] = gt;
    weq[warp] = eq;
  }
  __syncthreads();
  int pos = 0, eqb = 0;
  for (int w = 0; w < warp; ++w) {
    pos += wgt[w] + min(weq[w], max(0, (int)krem - eqb));
    eqb += weq[w];
  }
  const unsigned lt = (1u << lane) - 1u;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const bool v = i < w1;
    const uint32_t key = v ? keys[i] : 0u;
    const unsigned me = __ballot_sync(0xffffffffu, v && key == T);
    const bool take = v && (key > T || (key == T && eqb + __popc(me & lt) < (int)krem));
    const unsigned mt = __ballot_sync(0xffffffffu, take);
    if (take) out[pos + __popc(mt & lt)] = i;
    pos += __popc(mt);
    eqb += __popc(me);
  }
}

template <int KPT>
static int launch_topk_cluster(const float* scores, int B, int ld, int N, int k, int32_t* idx,
                               int ld_idx, int* st, cudaStream_t stream) {
  k_topk_cluster<KPT><<<B * kClusterTopk, 256, 0, stream>>>(scores, ld, N, k, idx, ld_idx, st);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

int launch_topk(const float* scores, int B, int ld, int N, const int* k_per_row, int k,
                int32_t* idx, int ld_idx, int* st, cudaStream_t stream) {
  const int per = (N + kClusterTopk * 256 - 1) / (kClusterTopk * 256);  // keys per thread
  int rc = DV_ERR_UNSUPPORTED;
  note_launch(DV_TAG_TOPK, 0, stream);
  if (!k_per_row && N <= kSmallN) {
    k_topk_small<<<B, kTopkThreads, 0, stream>>>(scores, ld, N, k, idx, ld_idx, st);
    rc = cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
  } else if (!k_per_row && per <= 64) {
    if (per <= 1) rc = launch_topk_cluster<1>(scores, B, ld, N, k, idx, ld_idx, st, stream);
    else if (per <= 4) rc = launch_topk_cluster<4>(scores, B, ld, N, k, idx, ld_idx, st, stream);
    else if (per <= 8) rc = launch_topk_cluster<8>(scores, B, ld, N, k, idx, ld_idx, st, stream);
    else if (per <= 16) rc = launch_topk_cluster<16>(scores, B, ld, N, k, idx, ld_idx, st, stream);
    else if (per <= 24) rc = launch_topk_cluster<24>(scores, B, ld, N, k, idx, ld_idx, st, stream);
    else if (per <= 32) rc = launch_topk_cluster<32>(scores, B, ld, N, k, idx, ld_idx, st, stream);
    else rc = launch_topk_cluster<64>(scores, B, ld, N, k, idx, ld_idx, st, stream);
  } else {
    k_topk<<<B, kTopkThreads, 0, stream>>>(scores, ld, N, k_per_row, k, idx, ld_idx, st);
    rc = cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
  }
  note_launch(DV_TAG_TOPK, 1, stream);
  return rc;
}

// Union of B ascending sets of width k over [0, N): bitmap, then ordered
// compaction over 32-bit words.
__global__ void __launch_bounds__(256) k_union(const int32_t* __restrict__ idx, int B, int k,
                                                int N, int32_t* __restrict__ out,
                                                int32_t* __restrict__ count) {
  extern __shared__ uint32_t bits[];
  __shared__ int tmp[32];
  const int words = (N + 31) / 32;
  for (int w = threadIdx.x; w < words; w += blockDim.x) bits[w] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < B * k; i += blockDim.x) {
    const int j = idx[i];
    if (j >= 0 && j < N) atomicOr(&bits[j >> 5], 1u << (j & 31));
  }
  __syncthreads();
  const int per = (words + blockDim.x - 1) / blockDim.x;
  const int w0 = min(words, (int)threadIdx.x * per), w1 = min(words, w0 + per);
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bits[w]);
  int tot;
  int pos = block_exscan(c, tmp, &tot);
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bits[w];
    while (m) {
      const int b = __ffs(m) - 1;
      out[pos++] = w * 32 + b;
      m &= m - 1;
    }
  }
  if (threadIdx.x == 0) *count = tot;
}

int launch_union(const int32_t* idx, int B, int k, int N, int32_t* out, int32_t* count,
                 cudaStream_t stream) {
  const size_t smem = (size_t)((N + 31) / 32) * 4;
  if (smem > 200 * 1024) return DV_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(k_union, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  note_launch(DV_TAG_UNION, 0, stream);
  k_union<<<1, 256, smem, stream>>>(idx, B, k, N, out, count);
  note_launch(DV_TAG_UNION, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
