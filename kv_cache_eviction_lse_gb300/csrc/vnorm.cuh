#pragma once
#include <cuda_runtime.h>
#include <stddef.h>

#include "common.cuh"

namespace kvs {

size_t vnorm_workspace_bytes(int L, int Hq, int d);

// vn [L][Hq][T] = ||W_O^{(hq)} v_i||; ws: vnorm_workspace_bytes() bytes (Gram matrices).
cudaError_t launch_vnorm(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                         const bf16_t* w_o, float* vn, void* ws, cudaStream_t s);

// Same result without a caller workspace: one layer at a time through a built-in
// device scratch array of vnorm_noalloc_scratch_bytes() (needs Hq*d*d*4 <= that).
size_t vnorm_noalloc_scratch_bytes();
cudaError_t launch_vnorm_noalloc(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                                 const bf16_t* w_o, float* vn, cudaStream_t s);

}  // namespace kvs
