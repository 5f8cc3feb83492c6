#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvs {

// mode 0: threshold (tau, w); mode 1: top-k (k, w).  rows = L * H_kv rows of T scores.
cudaError_t launch_prune(const float* score, int rows, int T, int mode, float tau, int k, int w,
                         uint8_t* mask, int* keep, cudaStream_t s);

// Per-layer quantile threshold: tau[l] = rank floor(q (N - 1)) of the N = Hkv (T - w)
// non-window scores of layer l (NaN lowest), then the threshold rule with tau[l].
cudaError_t launch_prune_quantile(const float* score, int L, int Hkv, int T, float q, int w,
                                  float* tau, uint8_t* mask, int* keep, cudaStream_t s);

constexpr int kMaxTopkBudgets = 8;
struct TopkBudgets {
  int k[kMaxTopkBudgets];
};

// Top-k masks of n_budgets budgets over the same rows in one launch: mask
// [n_budgets][rows][T], keep [n_budgets][rows].
cudaError_t launch_topk(const float* score, int rows, int T, int n_budgets, const TopkBudgets& kb,
                        int w, uint8_t* mask, int* keep, cudaStream_t s);

}  // namespace kvs
