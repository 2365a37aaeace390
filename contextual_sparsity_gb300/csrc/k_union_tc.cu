// k_union_tc.cu -- the sparse MLP of a batch of 8..64 sequences over the union
// of their neuron sets, on the tensor cores (sm_103a, mma.sync m16n8k16).
//
// "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time", §5.2
// and App. C.1: a batch computes every row over the union U of its sequences'
// sets, which turns the per-sequence gathers into one dense contraction:
//   H = relu(Z W1_U^T + b1_U)   (B x |U|),  Z = LN2(x) in fp16
//   out = x + H W2_U + b2       (B x d)
// fp16 operands (the 16-bit activations), fp32 accumulation. Three launches:
// LN2 of the B inputs; the fc1 contraction in tiles of 16 union rows x B, K
// split over the CTA's warps; the fc2^T contraction in tiles of 16 output
// columns x B over the union rows, K split over the warps.
#include "dv_internal.h"
#include "k_union_tc.h"

namespace dv {

constexpr int kTcWarps = 4;

// D (16 x 8, fp32) += A (16 x 16, fp16, row-major) * B (16 x 8, fp16, column-major).
// Fragments (g = lane / 4, c = lane % 4): a[0] = A[g][2c..2c+1],
// a[1] = A[g+8][2c..], a[2] = A[g][2c+8..], a[3] = A[g+8][2c+8..];
// b[0] = B[2c..2c+1][g], b[1] = B[2c+8..2c+9][g]; d[0..1] = D[g][2c..2c+1],
// d[2..3] = D[g+8][2c..2c+1].
DV_DEV void mma16816(float* d, const uint32_t* a, const uint32_t* b) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

DV_DEV uint32_t ld32(const uint16_t* p) { return *reinterpret_cast<const uint32_t*>(p); }
DV_DEV uint32_t pack2(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

// Z[b] = fp16(LN2(x[b])): one CTA per sequence, two passes in fp32.
__global__ void __launch_bounds__(256) k_union_ln(const uint16_t* __restrict__ x, int d,
                                                  const uint16_t* __restrict__ g,
                                                  const uint16_t* __restrict__ bb, float eps,
                                                  uint16_t* __restrict__ Z) {
  __shared__ float red[8];
  __shared__ float stat[2];
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t* xr = x + (size_t)b * d;
  float s = 0.f;
  for (int i = threadIdx.x; i < d; i += 256) s += h2f(xr[i]);
  s = warp_sum(s);
  if (lane == 0) red[warp] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += red[w];
    stat[0] = t / d;
  }
  __syncthreads();
  const float mu = stat[0];
  float q = 0.f;
  for (int i = threadIdx.x; i < d; i += 256) {
    const float c = h2f(xr[i]) - mu;
    q = fmaf(c, c, q);
  }
  q = warp_sum(q);
  __syncthreads();
  if (lane == 0) red[warp] = q;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += red[w];
    stat[1] = 1.0f / sqrtf(t / d + eps);
  }
  __syncthreads();
  const float inv = stat[1];
  for (int i = threadIdx.x; i < d; i += 256) {
    const float gg = g ? h2f(g[i]) : 1.f, be = bb ? h2f(bb[i]) : 0.f;
    Z[(size_t)b * d + i] = f2h((h2f(xr[i]) - mu) * inv * gg + be);
  }
}

// H[b][j] = fp16(relu(Z[b] . fc1[U[j]] + b1[U[j]])) for a tile of 16 union rows.
template <int NT>
__global__ void __launch_bounds__(kTcWarps * 32) k_union_fc1(
    const uint16_t* __restrict__ Z, int B, int d, const uint16_t* __restrict__ fc1,
    const uint16_t* __restrict__ b1, int F, const int32_t* __restrict__ U, int k,
    const int32_t* __restrict__ dev_count, uint16_t* __restrict__ H, int ldh, int* st) {
  __shared__ float red[kTcWarps][16][NT * 8];
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  int kk = k;
  if (dev_count) kk = min(kk, *dev_count);
  const int j0 = blockIdx.x * 16;
  if (j0 >= kk) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  // the two union rows this thread reads (rows beyond the union: row 0, zero weight)
  // (an entry inside the union that is negative or >= F is reported and skipped)
  int ra = j0 + g < kk ? U[j0 + g] : -1, rb = j0 + g + 8 < kk ? U[j0 + g + 8] : -1;
  const bool bad_a = j0 + g < kk && (ra < 0 || ra >= F);
  const bool bad_b = j0 + g + 8 < kk && (rb < 0 || rb >= F);
  if (bad_a || bad_b) {
    flag(st, DV_DEV_BAD_INDEX);
    if (bad_a) ra = -1;
    if (bad_b) rb = -1;
  }
  const uint16_t* wa = fc1 + (size_t)(ra < 0 ? 0 : ra) * d;
  const uint16_t* wb = fc1 + (size_t)(rb < 0 ? 0 : rb) * d;
  const uint32_t ma = ra < 0 ? 0u : 0xffffffffu, mb = rb < 0 ? 0u : 0xffffffffu;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
  const int ksteps = d / 16;
  for (int s = warp; s < ksteps; s += kTcWarps) {
    const int k0 = s * 16 + 2 * c;
    uint32_t a[4] = {ld32(wa + k0) & ma, ld32(wb + k0) & mb, ld32(wa + k0 + 8) & ma,
                     ld32(wb + k0 + 8) & mb};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint16_t* zr = Z + (size_t)(t * 8 + g) * d;
      const uint32_t bf[2] = {ld32(zr + k0), ld32(zr + k0 + 8)};
      mma16816(acc[t], a, bf);
    }
  }
  // the warps' K slices, summed in warp order
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    red[warp][g][t * 8 + 2 * c] = acc[t][0];
    red[warp][g][t * 8 + 2 * c + 1] = acc[t][1];
    red[warp][g + 8][t * 8 + 2 * c] = acc[t][2];
    red[warp][g + 8][t * 8 + 2 * c + 1] = acc[t][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * B; i += blockDim.x) {
    const int r = i / B, b = i % B, j = j0 + r;
    if (j >= kk) continue;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kTcWarps; ++w) v += red[w][r][b];
    const int u = U[j];
    const bool ok = u >= 0 && u < F;
    v += (b1 && ok) ? h2f(b1[u]) : 0.f;
    H[(size_t)b * ldh + j] = f2h(ok && v > 0.f ? v : 0.f);
  }
}

// out[b][col] = x[b][col] + b2[col] + sum_j H[b][j] fc2T[U[j]][col], a tile of
// 16 output columns.
template <int NT>
__global__ void __launch_bounds__(kTcWarps * 32) k_union_fc2(
    const uint16_t* __restrict__ H, int ldh, int B, int d, const uint16_t* __restrict__ fc2T,
    int F, const uint16_t* __restrict__ b2, const int32_t* __restrict__ U, int k,
    const int32_t* __restrict__ dev_count, const uint16_t* __restrict__ x,
    uint16_t* __restrict__ out, int* st) {
  __shared__ float red[kTcWarps][16][NT * 8];
  pdl_wait();
  if (threadIdx.x == 0) pdl_launch_dependents();
  int kk = k;
  if (dev_count) kk = min(kk, *dev_count);
  const int c0 = blockIdx.x * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.f;
  const int ksteps = (kk + 15) / 16;
  bool bad = false;
  for (int s = warp; s < ksteps; s += kTcWarps) {
    const int j = s * 16 + 2 * c;  // this thread's union rows: j, j+1, j+8, j+9
    uint16_t v[8];
    int jj[4] = {j, j + 1, j + 8, j + 9};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      int u = jj[q] < kk ? U[jj[q]] : -1;
      if (jj[q] < kk && (u < 0 || u >= F)) {  // reported and skipped
        bad = true;
        u = -1;
      }
      const uint16_t* row = fc2T + (size_t)(u < 0 ? 0 : u) * d + c0;
      v[2 * q] = u < 0 ? 0 : row[g];           // A[g][row jj[q]]
      v[2 * q + 1] = u < 0 ? 0 : row[g + 8];   // A[g+8][row jj[q]]
    }
    const uint32_t a[4] = {pack2(v[0], v[2]), pack2(v[1], v[3]), pack2(v[4], v[6]),
                           pack2(v[5], v[7])};
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint16_t* hr = H + (size_t)(t * 8 + g) * ldh;
      // H beyond the union's count is never written: those rows carry zero A
      const uint32_t bf[2] = {j + 1 < kk ? ld32(hr + j) : (j < kk ? (uint32_t)hr[j] : 0u),
                              j + 9 < kk ? ld32(hr + j + 8) : (j + 8 < kk ? (uint32_t)hr[j + 8] : 0u)};
      mma16816(acc[t], a, bf);
    }
  }
  if (bad) flag(st, DV_DEV_BAD_INDEX);
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    red[warp][g][t * 8 + 2 * c] = acc[t][0];
    red[warp][g][t * 8 + 2 * c + 1] = acc[t][1];
    red[warp][g + 8][t * 8 + 2 * c] = acc[t][2];
    red[warp][g + 8][t * 8 + 2 * c + 1] = acc[t][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * B; i += blockDim.x) {
    const int r = i / B, b = i % B, col = c0 + r;
    if (col >= d) continue;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kTcWarps; ++w) v += red[w][r][b];
    v += b2 ? h2f(b2[col]) : 0.f;
    v += x ? h2f(x[(size_t)b * d + col]) : 0.f;
    out[(size_t)b * d + col] = f2h(v);
  }
}

template <int NT>
static int union_launch(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g,
                        const uint16_t* ln_b, float eps, const uint16_t* fc1, const uint16_t* b1,
                        const uint16_t* fc2T, const uint16_t* b2, const int32_t* U, int k,
                        const int32_t* dev_count, bool resid, uint16_t* out, int* st,
                        uint16_t* Z, uint16_t* H, int ldh, cudaStream_t s) {
  note_launch(DV_TAG_MLP, 0, s);
  k_union_ln<<<B, 256, 0, s>>>(x, d, ln_g, ln_b, eps, Z);
  note_launch(DV_TAG_MLP, 1, s);
  if (cudaGetLastError() != cudaSuccess) return DV_ERR_LAUNCH;
  {
    void* args[] = {&Z, &B, &d, &fc1, &b1, &F, &U, &k, &dev_count, &H, &ldh, &st};
    note_launch(DV_TAG_MLP, 0, s);
    const cudaError_t e = launch_k((const void*)k_union_fc1<NT>, dim3((k + 15) / 16),
                                   dim3(kTcWarps * 32), 0, s, args, true);
    note_launch(DV_TAG_MLP, 1, s);
    if (e != cudaSuccess) return DV_ERR_LAUNCH;
  }
  const uint16_t* xr = resid ? x : nullptr;
  void* args[] = {&H, &ldh, &B, &d, &fc2T, &F, &b2, &U, &k, &dev_count, &xr, &out, &st};
  note_launch(DV_TAG_MLP, 0, s);
  const cudaError_t e = launch_k((const void*)k_union_fc2<NT>, dim3((d + 15) / 16),
                                 dim3(kTcWarps * 32), 0, s, args, true);
  note_launch(DV_TAG_MLP, 1, s);
  return e == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

int union_tc_ldh(int k);

size_t union_tc_ws_bytes(int B, int d, int k) {
  const size_t z = ((size_t)B * d * 2 + 255) / 256 * 256;
  return z + (size_t)B * union_tc_ldh(k) * 2;
}

int union_tc_ldh(int k) { return (k + 15) / 16 * 16; }

int launch_union_mlp_tc(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g,
                        const uint16_t* ln_b, float eps, const uint16_t* fc1, const uint16_t* b1,
                        const uint16_t* fc2T, const uint16_t* b2, const int32_t* U, int k,
                        const int32_t* dev_count, bool resid, uint16_t* out, int* st, void* ws,
                        cudaStream_t s) {
  uint16_t* Z = static_cast<uint16_t*>(ws);
  uint16_t* H = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(ws) +
                                            ((size_t)B * d * 2 + 255) / 256 * 256);
  const int ldh = union_tc_ldh(k);
  switch (B / 8) {
    case 1: return union_launch<1>(x, B, d, F, ln_g, ln_b, eps, fc1, b1, fc2T, b2, U, k, dev_count, resid, out, st, Z, H, ldh, s);
    case 2: return union_launch<2>(x, B, d, F, ln_g, ln_b, eps, fc1, b1, fc2T, b2, U, k, dev_count, resid, out, st, Z, H, ldh, s);
    case 4: return union_launch<4>(x, B, d, F, ln_g, ln_b, eps, fc1, b1, fc2T, b2, U, k, dev_count, resid, out, st, Z, H, ldh, s);
    case 8: return union_launch<8>(x, B, d, F, ln_g, ln_b, eps, fc1, b1, fc2T, b2, U, k, dev_count, resid, out, st, Z, H, ldh, s);
    default: return DV_ERR_UNSUPPORTED;
  }
}

}  // namespace dv
