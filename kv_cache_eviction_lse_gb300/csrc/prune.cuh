#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvs {

// mode 0: threshold (tau, w); mode 1: top-k (k, w).  rows = L * H_kv rows of T scores.
cudaError_t launch_prune(const float* score, int rows, int T, int mode, float tau, int k, int w,
                         uint8_t* mask, int* keep, cudaStream_t s);

}  // namespace kvs
