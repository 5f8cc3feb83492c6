// Launcher of the KVzap-MLP surrogate (two-layer MLP per layer, D_h -> D_mid -> H_kv).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvs {

struct MlpArgs {
  const bf16_t* h = nullptr;   // [L][T][Dh]
  const bf16_t* W1 = nullptr;  // [L][Dm][Dh]
  const float* b1 = nullptr;   // [L][Dm]
  const bf16_t* W2 = nullptr;  // [L][H][Dm]
  const float* b2 = nullptr;   // [L][H]
  float* z = nullptr;          // [L][H][T], zeroed by the launcher, then accumulated
  int L = 0, T = 0, Dh = 0, Dm = 0, H = 0;
};

// Number of column parts D_mid is split into (each part is one CTA's accumulator of at
// most 256 columns, a multiple of 32), or 0 when D_mid cannot be split that way.
int mlp_parts(int Dm);

// True when the kernels support this (Dh, Dm, H).
bool mlp_supported(int Dh, int Dm, int H);

cudaError_t launch_mlp_surrogate(const MlpArgs& a, cudaStream_t s);

// Reads (and with `clear` resets) the device error word of the MLP kernel.
cudaError_t mlp_device_error(int* code, bool clear, cudaStream_t s);

}  // namespace kvs
