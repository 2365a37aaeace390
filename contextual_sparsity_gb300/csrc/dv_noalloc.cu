// dv_noalloc.cu -- dv_sparse_mlp_noalloc: the sparse MLP block for callers
// that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers: a plugin
// running inside a serving engine that owns every byte of device memory, code
// that must not allocate once it has started, or a latency path that cannot
// afford cudaMalloc's implicit synchronisation. dv_sparse_mlp needs a caller
// workspace for its per-CTA partial sums; this entry point keeps those partial
// sums in a fixed array that lives in the library image instead, so the call
// allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
//
// The array holds kNoAllocScratchBytes (8 MiB) on every device that loads the
// library, until the process exits. All calls share it: two calls that
// overlap on the GPU (different streams, or different host threads, without
// ordering between them) race on it. Nothing in it has to start at zero: each
// launch writes every partial it later reads.
#include <mutex>

#include "dv_internal.h"

namespace dv {

constexpr size_t kNoAllocScratchBytes = 8u << 20;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

// Device address of the array, looked up once per device (the host-side name
// is only a stand-in: a kernel given it would read the wrong memory).
static float* noalloc_scratch_ptr(int* status) {
  static std::mutex mu;
  static float* ptr[kNoAllocMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    *status = DV_ERR_LAUNCH;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      *status = DV_ERR_LAUNCH;
      return nullptr;
    }
    ptr[dev] = static_cast<float*>(p);
  }
  *status = DV_OK;
  return ptr[dev];
}

}  // namespace dv

using namespace dv;

extern "C" int dv_sparse_mlp_noalloc(const uint16_t* x, int B, const dv_dims* dims,
                                     const dv_layer_weights* w, const int32_t* idx, int k,
                                     const int32_t* dev_count, int flags, uint16_t* out,
                                     int* dev_status, cudaStream_t stream) {
  auto al16 = [](const void* p) { return ((uintptr_t)p % 16) == 0; };
  if (!dims || !w || !x || !out || !w->fc1 || !w->fc2T) return DV_ERR_NULL;
  if (!al16(x) || !al16(out) || !al16(w->fc1) || !al16(w->fc2T) || !al16(w->ln2_g) ||
      !al16(w->ln2_b))
    return DV_ERR_ALIGN;
  if (dims->d < 8 || dims->d > 16384 || dims->d % 8 != 0 || dims->F < 1 || B < 1 || B > 4 ||
      x == out)
    return DV_ERR_DIMS;
  if (!idx) k = dims->F;
  if (k < 1 || k > dims->F) return DV_ERR_K;

  // One CTA per SM, as dv_sparse_mlp, when the partial sums fit; fewer CTAs
  // (each streaming more rows, at most 256) when they would not; otherwise the
  // problem is too large for the built-in array.
  const size_t per_cta = (size_t)B * dims->d * sizeof(float);
  const long long max_ctas = (long long)(kNoAllocScratchBytes / per_cta);
  const long long need = ((long long)k + 255) / 256;
  if (max_ctas < need || max_ctas < 1) return DV_ERR_WORKSPACE;
  const int target = (int)std::min<long long>(sm_count(), max_ctas);

  int rc = DV_OK;
  float* scratch = noalloc_scratch_ptr(&rc);
  if (rc != DV_OK) return rc;
  return launch_mlp(x, B, dims->d, dims->F, w->ln2_g, w->ln2_b, dims->ln_eps, w->fc1, w->b1,
                    w->fc2T, w->b2, idx, k, dev_count, flags & (DV_SKIP_INACTIVE | DV_NO_RESIDUAL),
                    out, dev_status, scratch, target, 160 * 1024, stream, false);
}
