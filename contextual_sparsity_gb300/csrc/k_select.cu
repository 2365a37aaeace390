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
#include "dv_internal.h"

namespace dv {

constexpr int kTopkThreads = 1024;

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
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < N; i += blockDim.x) {
      const float f = s[i];
      const uint32_t key = isnan(f) ? 0u : fkey(f);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
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

int launch_topk(const float* scores, int B, int ld, int N, const int* k_per_row, int k,
                int32_t* idx, int ld_idx, int* st, cudaStream_t stream) {
  note_launch(DV_TAG_TOPK, 0, stream);
  k_topk<<<B, kTopkThreads, 0, stream>>>(scores, ld, N, k_per_row, k, idx, ld_idx, st);
  note_launch(DV_TAG_TOPK, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

// Union of B ascending sets of width k over [0, N): bitmap, then ordered
// compaction over 32-bit words.
__global__ void __launch_bounds__(1024) k_union(const int32_t* __restrict__ idx, int B, int k,
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
  k_union<<<1, 1024, smem, stream>>>(idx, B, k, N, out, count);
  note_launch(DV_TAG_UNION, 1, stream);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
