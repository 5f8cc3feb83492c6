// Ridge solve of the value refit's normal equations, one CTA per (layer, KV head):
//   (G + lam I) X = R,   lam = lam_rel * mean(diag G[:k, :k])
// by an upper Cholesky factorisation G + lam I = U^T U in fp32 (blocked, right-looking,
// panels of 16 rows in shared memory) and two blocked triangular solves U^T Y = R,
// U X = Y with one thread per right-hand-side column.  G arrives as its upper block
// triangle (the Gram kernel writes only those tiles); the lower triangle is never read.
// Rows/columns k .. M-1 (padding of the kept-key dimension) are decoupled: their
// diagonal gets 1 and their right-hand side is 0, so their solution is 0.
#include <math.h>

#include "gram.cuh"

namespace kvs {

__device__ int g_chol_error = 0;

namespace {

constexpr int NB = 16;
constexpr int kThreads = 1024;
constexpr int kErrNotSpd = 6;  // a pivot of the factorisation was not positive

// Upper-triangle index of micro-tile t among the n x n tiles with tj >= ti (row-major).
__device__ __forceinline__ void upper_tile(long t, int n, int& ti, int& tj) {
  const double b = 2.0 * n + 1.0;
  int i = (int)((b - sqrt(b * b - 8.0 * (double)t)) * 0.5);
  auto start = [&](int r) { return (long)r * n - (long)r * (r - 1) / 2; };
  while (i > 0 && start(i) > t) --i;
  while (i + 1 < n && start(i + 1) <= t) ++i;
  ti = i;
  tj = i + (int)(t - start(i));
}

__global__ void __launch_bounds__(kThreads) chol_solve_kernel(const CholArgs a) {
  extern __shared__ float sm[];
  const int M = a.M, ld = a.ldg, d = a.d;
  float* ub = sm;                      // [NB][NB + 1] diagonal block of U
  float* panel = ub + NB * (NB + 1);   // [NB][M] row panel of U (trailing columns)
  float* yb = panel + NB * M;          // [NB][d] solved rows of the current block
  __shared__ float red[kThreads / 32];
  __shared__ float lam_s;
  const int tid = threadIdx.x, lane = tid & 31;
  float* G = a.g + (size_t)blockIdx.x * M * ld;
  float* R = a.r + (size_t)blockIdx.x * M * d;

  // ---- ridge weight from the trace, then the shifted diagonal
  float t = 0.f;
  for (int i = tid; i < a.k; i += kThreads) t += G[(size_t)i * ld + i];
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if (lane == 0) red[tid >> 5] = t;
  __syncthreads();
  if (tid == 0) {
    float s = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) s += red[w];
    lam_s = a.lam_rel * s / (float)max(a.k, 1);
  }
  __syncthreads();
  const float lam = lam_s;
  for (int i = tid; i < M; i += kThreads) {
    float* gi = G + (size_t)i * ld + i;
    if (i < a.k) {
      *gi += lam;
    } else {  // padding: decouple it
      *gi = 1.f;
    }
  }
  for (size_t idx = tid; idx < (size_t)(M - a.k) * d; idx += kThreads)
    R[(size_t)a.k * d + idx] = 0.f;

  // ---- factorisation G = U^T U (upper), in place
  for (int p = 0; p < M; p += NB) {
    const int nb = min(NB, M - p);
    const int nrest = M - p - nb;
    __syncthreads();
    for (int idx = tid; idx < nb * nb; idx += kThreads) {
      const int r = idx / nb, c = idx % nb;
      ub[r * (NB + 1) + c] = (c >= r) ? G[(size_t)(p + r) * ld + p + c] : 0.f;
    }
    __syncthreads();
    if (tid < 32) {
      for (int r = 0; r < nb; ++r) {
        if (lane == r) {
          const float v = ub[r * (NB + 1) + r];
          if (!(v > 0.f)) atomicCAS(&g_chol_error, 0, kErrNotSpd);
          ub[r * (NB + 1) + r] = sqrtf(fmaxf(v, 1e-30f));
        }
        __syncwarp();
        const float piv = ub[r * (NB + 1) + r];
        if (lane > r && lane < nb) ub[r * (NB + 1) + lane] /= piv;
        __syncwarp();
        for (int s = r + 1; s < nb; ++s)
          if (lane >= s && lane < nb) ub[s * (NB + 1) + lane] -= ub[r * (NB + 1) + s] * ub[r * (NB + 1) + lane];
        __syncwarp();
      }
    }
    __syncthreads();
    for (int idx = tid; idx < nb * nb; idx += kThreads) {
      const int r = idx / nb, c = idx % nb;
      if (c >= r) G[(size_t)(p + r) * ld + p + c] = ub[r * (NB + 1) + c];
    }
    // row panel: U[p..p+nb][j] = U_pp^-T G[p..p+nb][j] for the trailing columns j
    for (int jj = tid; jj < nrest; jj += kThreads) {
      const int j = p + nb + jj;
      float x[NB];
#pragma unroll
      for (int r = 0; r < NB; ++r) x[r] = r < nb ? G[(size_t)(p + r) * ld + j] : 0.f;
#pragma unroll
      for (int r = 0; r < NB; ++r) {
        if (r < nb) {
          float v = x[r];
#pragma unroll
          for (int s = 0; s < r; ++s) v -= ub[s * (NB + 1) + r] * x[s];
          x[r] = v / ub[r * (NB + 1) + r];
        }
      }
#pragma unroll
      for (int r = 0; r < NB; ++r)
        if (r < nb) {
          G[(size_t)(p + r) * ld + j] = x[r];
          panel[r * M + jj] = x[r];
        }
    }
    __syncthreads();
    // trailing update of the upper triangle: G[i][j] -= sum_r U[p+r][i] U[p+r][j]
    const int n4 = (nrest + 3) / 4;
    const long ntiles = (long)n4 * (n4 + 1) / 2;
    for (long tt = tid; tt < ntiles; tt += kThreads) {
      int ti, tj;
      upper_tile(tt, n4, ti, tj);
      const int i0 = 4 * ti, j0 = 4 * tj;
      float acc[4][4] = {};
      for (int r = 0; r < nb; ++r) {
        float xi[4], xj[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          xi[u] = i0 + u < nrest ? panel[r * M + i0 + u] : 0.f;
          xj[u] = j0 + u < nrest ? panel[r * M + j0 + u] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(xi[u], xj[v], acc[u][v]);
      }
      const bool full = i0 + 4 <= nrest && j0 + 4 <= nrest && tj > ti && ((p + nb + j0) & 3) == 0 &&
                        (ld & 3) == 0;
      if (full) {  // an off-diagonal micro-tile: four 16-byte read-modify-writes
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float4* gp = reinterpret_cast<float4*>(G + (size_t)(p + nb + i0 + u) * ld + p + nb + j0);
          float4 g4 = *gp;
          g4.x -= acc[u][0]; g4.y -= acc[u][1]; g4.z -= acc[u][2]; g4.w -= acc[u][3];
          *gp = g4;
        }
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v)
            if (i0 + u < nrest && j0 + v < nrest && j0 + v >= i0 + u)
              G[(size_t)(p + nb + i0 + u) * ld + p + nb + j0 + v] -= acc[u][v];
      }
    }
  }
  __syncthreads();

  // ---- U^T Y = R (forward, by blocks of NB rows), in place in R
  for (int p = 0; p < M; p += NB) {
    const int nb = min(NB, M - p);
    const int nrest = M - p - nb;
    for (int idx = tid; idx < nb * nb; idx += kThreads) {
      const int r = idx / nb, c = idx % nb;
      ub[r * (NB + 1) + c] = (c >= r) ? G[(size_t)(p + r) * ld + p + c] : 0.f;
    }
    for (int idx = tid; idx < nb * nrest; idx += kThreads) {
      const int r = idx / nrest, q = idx % nrest;
      panel[r * M + q] = G[(size_t)(p + r) * ld + p + nb + q];
    }
    __syncthreads();
    for (int c = tid; c < d; c += kThreads) {
      float y[NB];
#pragma unroll
      for (int r = 0; r < NB; ++r) {
        if (r < nb) {
          float v = R[(size_t)(p + r) * d + c];
#pragma unroll
          for (int s = 0; s < r; ++s) v -= ub[s * (NB + 1) + r] * y[s];
          y[r] = v / ub[r * (NB + 1) + r];
          R[(size_t)(p + r) * d + c] = y[r];
          yb[r * d + c] = y[r];
        }
      }
    }
    __syncthreads();
    for (size_t idx = tid; idx < (size_t)nrest * d; idx += kThreads) {
      const int q = (int)(idx / d), c = (int)(idx % d);
      float v = 0.f;
      for (int r = 0; r < nb; ++r) v = fmaf(panel[r * M + q], yb[r * d + c], v);
      R[(size_t)(p + nb + q) * d + c] -= v;
    }
    __syncthreads();
  }

  // ---- U X = Y (backward, by blocks of NB rows from the bottom), in place in R
  const int nblk = (M + NB - 1) / NB;
  for (int bk = nblk - 1; bk >= 0; --bk) {
    const int p = bk * NB, nb = min(NB, M - p);
    for (int idx = tid; idx < nb * nb; idx += kThreads) {
      const int r = idx / nb, c = idx % nb;
      ub[r * (NB + 1) + c] = (c >= r) ? G[(size_t)(p + r) * ld + p + c] : 0.f;
    }
    // column panel U[q][p..p+nb] for the rows q < p, stored [r][q]
    for (int idx = tid; idx < nb * p; idx += kThreads) {
      const int q = idx / nb, r = idx % nb;
      panel[r * M + q] = G[(size_t)q * ld + p + r];
    }
    __syncthreads();
    for (int c = tid; c < d; c += kThreads) {
      float x[NB];
#pragma unroll
      for (int r = NB - 1; r >= 0; --r) {
        if (r < nb) {
          float v = R[(size_t)(p + r) * d + c];
#pragma unroll
          for (int s = r + 1; s < NB; ++s)
            if (s < nb) v -= ub[r * (NB + 1) + s] * x[s];
          x[r] = v / ub[r * (NB + 1) + r];
          R[(size_t)(p + r) * d + c] = x[r];
          yb[r * d + c] = x[r];
        }
      }
    }
    __syncthreads();
    for (size_t idx = tid; idx < (size_t)p * d; idx += kThreads) {
      const int q = (int)(idx / d), c = (int)(idx % d);
      float v = 0.f;
      for (int r = 0; r < nb; ++r) v = fmaf(panel[r * M + q], yb[r * d + c], v);
      R[(size_t)q * d + c] -= v;
    }
    __syncthreads();
  }

  // ---- the first k rows are the refitted values
  float* X = a.x + (size_t)blockIdx.x * a.k * d;
  for (size_t idx = tid; idx < (size_t)a.k * d; idx += kThreads) X[idx] = R[idx];
}

}  // namespace

cudaError_t launch_chol_solve(const CholArgs& a, cudaStream_t s) {
  if (a.batch <= 0 || a.M <= 0) return cudaSuccess;
  if (a.M > kCholMaxM || a.k > a.M || a.d > 256) return cudaErrorInvalidValue;
  const size_t smem = sizeof(float) * ((size_t)NB * (NB + 1) + (size_t)NB * a.M + (size_t)NB * a.d);
  cudaError_t e = cudaFuncSetAttribute(chol_solve_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  count_launches(1);
  chol_solve_kernel<<<a.batch, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t chol_device_error(int* code, bool clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_chol_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && *code) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_chol_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace kvs
