#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace kvs {

size_t surrogate_smem_bytes(int Dh, int Hkv);

cudaError_t launch_surrogate(const bf16_t* h, int L, int T, int Dh, int Hkv, const bf16_t* W,
                             const float* b, float* z, float tau, int w, uint8_t* mask,
                             int* keep, cudaStream_t s);

}  // namespace kvs
