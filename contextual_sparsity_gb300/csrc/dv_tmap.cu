// dv_tmap.cu -- host side of the tiled TMA loads: tensor maps encoded through
// the driver's cuTensorMapEncodeTiled, looked up once through the runtime's
// entry-point query (no link-time dependency on libcuda).
#include <mutex>

#include "dv_tc.cuh"

namespace dv {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiled encode_fn() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

bool make_tmap_f16_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t pitch_elems, uint32_t box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn || !base || ((uintptr_t)base & 15) || (pitch_elems * 2) % 16 || cols < 64 ||
      box_rows < 1 || box_rows > 256)
    return false;
  const cuuint64_t dim[2] = {cols, rows};
  const cuuint64_t stride[1] = {pitch_elems * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dim, stride, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace dv
