// Launchers of the two attention-scoring passes (pass 1: LSE; pass 2: transposed
// KVzip max / KVpop future mass) and the hidden-norm prologue.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvs {

struct AttnArgs {
  const bf16_t* q = nullptr;       // [L][Hq][n_q][d]
  const bf16_t* k_ctx = nullptr;   // [L][Hkv][T][d]
  const bf16_t* k_tail = nullptr;  // [L][Hkv][n_tail][d]
  const float* lse = nullptr;      // [L][Hq][n_q]
  const float* vnorm = nullptr;    // [L][Hq][T] or null
  const float* hlog = nullptr;     // [L][n_q] ln||h_j|| or null
  const bf16_t* gpair = nullptr;   // [L][Hq][2d][d] Gram pairs (hi rows, lo rows); vnorm only
  float* out = nullptr;
  int L = 0, Hq = 0, Hkv = 0, d = 0, n_q = 0, T = 0, n_tail = 0;
  int w = 0, accumulate = 0;
  int causal = 1;                  // 0: every query sees every key (internal callers)
  uint16_t* rows = nullptr;        // softmax rows: [L][Hq][n_q][rows_ld] fp16
  int rows_ld = 0;                 // padded row length (multiple of 64, >= T)
  // KVzip max (pass 2): per-query constants -(lse_j + ln||h_j||) / sqrt(d), split into
  // three bf16 parts [L][Hq][n_q_pad][16] (n_q_pad = n_q rounded up to 256; padding rows
  // hold -1e30), and a [128][16] tile of (1, 1, 1, 0, ...) rows: one extra K = 16 MMA
  // step adds the constant to every accumulator column
  const bf16_t* ccol = nullptr;
  const bf16_t* ones = nullptr;
};

// Score-max / future-mass workspace: the constants, then the ones tile above.
size_t score_max_ws_bytes(int L, int Hq, int n_q);
// Writes the constants -lse_j sqrt(d) and the ones tile into the workspace.
cudaError_t launch_score_constants(const float* lse, int L, int Hq, int n_q,
                                   int d, bf16_t* ccol, bf16_t* ones, cudaStream_t s);

cudaError_t launch_lse(const AttnArgs& a, cudaStream_t s);
// Softmax rows a_ji = exp(x_ji - lse_j) over the T context keys (lse given), written as
// fp16 into rows (zero past T up to rows_ld); no tail keys.
cudaError_t launch_softmax_rows(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_score_max(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_future_sum(const AttnArgs& a, cudaStream_t s);

// vn[l][hq][i] = sqrt(v_i^T (G_hi + G_lo) v_i) on tcgen05: k_ctx = v [L][Hkv][T][d],
// gpair = Gram pairs, out = vn [L][Hq][T]; needs Hq / Hkv <= 16.
cudaError_t launch_vnorm_quad(const AttnArgs& a, cudaStream_t s);

struct FwdArgs {
  const bf16_t* q = nullptr;       // [L][Hq][n_q][d]
  const bf16_t* k_ctx = nullptr;   // [L][Hkv][T][d]
  const bf16_t* v_ctx = nullptr;   // [L][Hkv][T][d]
  const bf16_t* k_tail = nullptr;  // [L][Hkv][n_tail][d]
  const bf16_t* v_tail = nullptr;  // [L][Hkv][n_tail][d]
  bf16_t* o = nullptr;             // [L][Hq][n_q][d], bf16 (fp16 when o_f16)
  int o_f16 = 0;                   // write O as fp16 (the value refit's target)
  float* lse = nullptr;            // [L][Hq][n_q]
  int L = 0, Hq = 0, Hkv = 0, d = 0, n_q = 0, T = 0, n_tail = 0;
  int causal = 1;                  // 0: every query sees every key (internal callers)
};

// Attention forward (bottom-right causal over [context | tail]) with its LSE.
cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t s);
cudaError_t fwd_device_error(int* code, bool clear, cudaStream_t s);

// Reads (and with `clear` resets) the device error word of the scoring kernels.
cudaError_t attn_device_error(int* code, bool clear, cudaStream_t s);

// The same constants with the hidden-state factor ln ||h[l][j]||_2 (over D_h bf16
// channels) reduced from h in the same pass.
cudaError_t launch_hidden_constants(const bf16_t* h, int Dh, const float* lse, int L, int Hq,
                                    int n_q, int d, bf16_t* ccol, bf16_t* ones, cudaStream_t s);

}  // namespace kvs
