// k_w4.cu -- 4-bit weight rows for the sparse MLP (W4A16, sm_103a).
//
// "Deja Vu: Contextual Sparsity for Efficient LLMs at Inference Time", §5.2
// and Table 7, combine contextual sparsity with 4-bit weights and 16-bit
// activations; the page gives no format, so this library defines one:
// groups of 128 columns, scale s = fp16(max |w| / 7) (the division in fp32),
// code q = clamp(rint(w / s), -8, 7) (fp32 division, ties to even; a zero
// group has s = 0 and q = 0), dequantized weight q s. A packed row holds d/2
// bytes of codes (column 2i in the low nibble of byte i, stored as q + 8),
// then the d/128 fp16 scales, then zero bytes up to a multiple of 16 (so that
// every row starts on a 16-byte boundary for the bulk copies).
#include "dv_internal.h"

namespace dv {

size_t w4_row_bytes_host(int d) { return ((size_t)d / 2 + (size_t)d / 64 + 15) / 16 * 16; }

// One warp per 128-column group: each lane quantizes 4 adjacent columns.
__global__ void __launch_bounds__(256) k_quant_w4(const uint16_t* __restrict__ W, int rows, int d,
                                                  size_t row_bytes, uint8_t* __restrict__ out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * 8 + warp, row = blockIdx.y;
  const int ng = d / 128;
  if (g >= ng || row >= rows) return;
  const uint2 raw = *reinterpret_cast<const uint2*>(W + (size_t)row * d + g * 128 + lane * 4);
  const uint16_t h[4] = {(uint16_t)(raw.x & 0xFFFF), (uint16_t)(raw.x >> 16),
                         (uint16_t)(raw.y & 0xFFFF), (uint16_t)(raw.y >> 16)};
  float w[4], amax = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    w[e] = h2f(h[e]);
    amax = fmaxf(amax, fabsf(w[e]));
  }
  amax = warp_max(amax);
  const uint16_t s16 = f2h(amax / 7.0f);
  const float sf = h2f(s16);
  uint32_t nib[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    int q = 0;
    if (sf > 0.f) q = (int)fminf(fmaxf(rintf(w[e] / sf), -8.f), 7.f);
    nib[e] = (uint32_t)(q + 8);
  }
  uint8_t* orow = out + (size_t)row * row_bytes;
  *reinterpret_cast<uint16_t*>(orow + (g * 128 + lane * 4) / 2) =
      (uint16_t)(nib[0] | (nib[1] << 4) | (nib[2] << 8) | (nib[3] << 12));
  if (lane == 0) *reinterpret_cast<uint16_t*>(orow + d / 2 + g * 2) = s16;
  if (g == 0)  // zero padding after the scales
    for (size_t i = (size_t)d / 2 + d / 64 + lane; i < row_bytes; i += 32) orow[i] = 0;
}

int launch_quant_w4(const uint16_t* W, int rows, int d, uint8_t* out, cudaStream_t stream) {
  dim3 grid((d / 128 + 7) / 8, rows);
  k_quant_w4<<<grid, 256, 0, stream>>>(W, rows, d, w4_row_bytes_host(d), out);
  return cudaGetLastError() == cudaSuccess ? DV_OK : DV_ERR_LAUNCH;
}

}  // namespace dv
