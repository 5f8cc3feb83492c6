// Launchers of the value refit's linear algebra: the batched X^T Y products on the
// tensor cores and the per-problem Cholesky solve of the ridge normal equations.
// The refit's products run on fp16 operands (softmax weights in [0, 1] and the attention
// output, 2^-12 relative each) with fp32 accumulation (launch_refit_products); the
// value-norm Gram of o_proj runs on bf16 with its result split into bf16 hi/lo pairs.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvs {

// The value norms' Gram pairs: the diagonal d x d blocks of X^T X for X = o_proj.weight,
// the Gram matrix of each d-column slice (one head), written as bf16 pairs
// pair[batch][M / d][2][d][d] (hi rows, then lo = bf16(G - hi)).
struct GramArgs {
  const bf16_t* x = nullptr;  // [batch][rows][ldx]
  bf16_t* pair = nullptr;
  int batch = 0, rows = 0, M = 0, ldx = 0, pair_d = 0;
};

cudaError_t launch_gram(const GramArgs& a, cudaStream_t s);

// The value refit's normal equations in one launch, fp16 operands, fp32 results:
//   g[b] = A_S[b]^T A_S[b] (upper block triangle, k_ld x k_ld)   r[b] = A_S[b]^T O[b] (k_ld x d)
struct RefitProdArgs {
  const uint16_t* a_s = nullptr;  // [batch][rows][k_ld] fp16 softmax rows, zero past k
  const uint16_t* o = nullptr;    // [batch][rows][d] fp16 attention outputs
  float* g = nullptr;             // [batch][k_ld][k_ld]
  float* r = nullptr;             // [batch][k_ld][d]
  int batch = 0, rows = 0, k_ld = 0, d = 0;
};
cudaError_t launch_refit_products(const RefitProdArgs& a, cudaStream_t s);
cudaError_t gram_device_error(int* code, bool clear, cudaStream_t s);

struct CholArgs {
  float* g = nullptr;      // [batch][M][ldg]: Gram (upper block triangle), overwritten by U
  float* r = nullptr;      // [batch][M][d]: right-hand sides, used as scratch by the solves
  float* x = nullptr;      // [batch][k][d]: output, the first k rows of the solution
  int batch = 0, M = 0, ldg = 0, k = 0, d = 0;
  float lam_rel = 0.f;     // ridge weight relative to the mean of the first k diagonal entries
};

// Solves (G + lam I) X = R per problem, lam = lam_rel * trace(G[:k, :k]) / k, by a blocked
// upper Cholesky factorisation in fp32 (one launch per step over all problems; R rides
// along as extra columns) and one backward-solve launch.  M <= kCholMaxM.
constexpr int kCholMaxM = 8192;
cudaError_t launch_chol_solve(const CholArgs& a, cudaStream_t s);
cudaError_t chol_device_error(int* code, bool clear, cudaStream_t s);

}  // namespace kvs
