// k_union_tc.h -- launcher of the batch-union MLP on the tensor cores
// (k_union_tc.cu), used by the C ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace dv {

// Workspace of one call: LN2(x) of the B inputs and the activations H.
size_t union_tc_ws_bytes(int B, int d, int k);

int launch_union_mlp_tc(const uint16_t* x, int B, int d, int F, const uint16_t* ln_g,
                        const uint16_t* ln_b, float eps, const uint16_t* fc1, const uint16_t* b1,
                        const uint16_t* fc2T, const uint16_t* b2, const int32_t* U, int k,
                        const int32_t* dev_count, bool resid, uint16_t* out, int* st, void* ws,
                        cudaStream_t s);

}  // namespace dv
