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
  // The same host-side checks as dv_sparse_mlp (dimensions including ln_eps,
  // weight pointers and their alignment), then what is particular to this
  // entry point: fp16 rows only, and the size limit of the built-in array.
  int rc = check_dims(dims);
  if (rc != DV_OK) return rc;
  if (!x || !out) return DV_ERR_NULL;
  auto al16 = [](const void* p) { return ((uintptr_t)p % 16) == 0; };
  if (!al16(x) || !al16(out)) return DV_ERR_ALIGN;
  if ((rc = check_weights_mlp(w)) != DV_OK) return rc;
  // Packed 4-bit rows (DV_W4) are not served here: their rows have another
  // size, and reading them as fp16 rows would run past the caller's buffers.
  if (flags & DV_W4) return DV_ERR_UNSUPPORTED;
  if (B < 1 || B > 4 || x == out) return DV_ERR_DIMS;
  if (!idx) k = dims->F;
  if (k < 1 || k > dims->F) return DV_ERR_K;

  // As many CTAs as dv_sparse_mlp launches (one per SM, or the dv_set_tuning
  // count) when their partial sums fit the array; fewer CTAs, each streaming
  // more rows (at most 256), when they would not; otherwise the problem is
  // too large for the built-in array.
  const size_t per_cta = (size_t)B * dims->d * sizeof(float);
  const long long max_ctas = (long long)(kNoAllocScratchBytes / per_cta);
  const long long need = ((long long)k + 255) / 256;
  if (max_ctas < need || max_ctas < 1) return DV_ERR_WORKSPACE;
  const int target = (int)std::min<long long>(main_ctas(), max_ctas);

  float* scratch = noalloc_scratch_ptr(&rc);
  if (rc != DV_OK) return rc;
  return launch_mlp(x, B, dims->d, dims->F, w->ln2_g, w->ln2_b, dims->ln_eps, w->fc1, w->b1,
                    w->fc2T, w->b2, idx, k, dev_count, flags & (DV_SKIP_INACTIVE | DV_NO_RESIDUAL),
                    out, dev_status, scratch, target, main_ring_bytes(), stream, false);
}
