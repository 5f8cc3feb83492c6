// Ridge solve of the value refit's normal equations, batched over (layer, KV head):
//   (G + lam I) X = R,   lam = lam_rel * mean(diag G[:k, :k])
// by a blocked right-looking upper Cholesky factorisation G + lam I = U^T U in fp32
// and two blocked triangular solves U^T Y = R, U X = Y.  Every step is one launch over
// all problems, so the trailing updates (the bulk of the work) spread over the whole
// GPU instead of one CTA per problem:
//   per 64-row panel p:  factor the diagonal block (one CTA per problem), solve the row
//                        panel U_pp^T X = G[p][p+64:] (CTAs over 64-column blocks), update
//                        the trailing upper triangle G -= X^T X (CTAs over 64 x 64 tiles)
//   per 64-row block of the solves: the diagonal block's triangular solve, then the
//                        update of every remaining block row (64 x 64 x 64 products)
// G arrives as its upper block triangle (the Gram kernel writes only those tiles); the
// lower triangle is never read.  Rows/columns k .. M-1 (padding of the kept-key
// dimension) are decoupled: their diagonal becomes 1 and their right-hand side 0.
#include <math.h>

#include "gram.cuh"

namespace kvs {

__device__ int g_chol_error = 0;

namespace {

constexpr int NB = 64;         // panel / block size (M is a multiple of 64)
constexpr int kErrNotSpd = 6;  // a pivot of the factorisation was not positive

__device__ __forceinline__ float* prob(float* base, size_t stride) {
  return base + (size_t)blockIdx.y * stride;
}

// lam from the trace of the first k diagonal entries; shift the diagonal; decouple padding
__global__ void __launch_bounds__(256) shift_kernel(const CholArgs a) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  __shared__ float red[8];
  float t = 0.f;
  for (int i = threadIdx.x; i < a.k; i += 256) t += G[(size_t)i * a.ldg + i];
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < 8; ++w) s += red[w];
  const float lam = a.lam_rel * s / (float)max(a.k, 1);
  __syncthreads();
  for (int i = threadIdx.x; i < a.M; i += 256) {
    float* gi = G + (size_t)i * a.ldg + i;
    *gi = i < a.k ? *gi + lam : 1.f;
  }
  for (size_t idx = threadIdx.x; idx < (size_t)(a.M - a.k) * a.d; idx += 256)
    R[(size_t)a.k * a.d + idx] = 0.f;
}

// Cholesky of the diagonal block at p (upper, in place), one CTA per problem
__global__ void __launch_bounds__(256) potrf_kernel(const CholArgs a, int p) {
  float* G = prob(a.g, (size_t)a.M * a.ldg) + (size_t)p * a.ldg + p;
  __shared__ float u[NB][NB + 1];
  for (int idx = threadIdx.x; idx < NB * NB; idx += 256) {
    const int r = idx / NB, c = idx % NB;
    u[r][c] = c >= r ? G[(size_t)r * a.ldg + c] : 0.f;
  }
  __syncthreads();
  for (int r = 0; r < NB; ++r) {
    if (threadIdx.x == 0) {
      const float v = u[r][r];
      if (!(v > 0.f)) atomicCAS(&g_chol_error, 0, kErrNotSpd);
      u[r][r] = sqrtf(fmaxf(v, 1e-30f));
    }
    __syncthreads();
    const float piv = u[r][r];
    if (threadIdx.x > r && threadIdx.x < NB) u[r][threadIdx.x] /= piv;
    __syncthreads();
    // rank-1 update of rows s > r, columns c >= s
    for (int idx = threadIdx.x; idx < NB * NB; idx += 256) {
      const int s = idx / NB, c = idx % NB;
      if (s > r && c >= s) u[s][c] -= u[r][s] * u[r][c];
    }
    __syncthreads();
  }
  for (int idx = threadIdx.x; idx < NB * NB; idx += 256) {
    const int r = idx / NB, c = idx % NB;
    if (c >= r) G[(size_t)r * a.ldg + c] = u[r][c];
  }
}

// Row panel: G[p..p+64][j] = U_pp^-T G[p..p+64][j] for the 64 columns j of block
// blockIdx.x after the diagonal block; one thread per column
__global__ void __launch_bounds__(64) trsm_row_kernel(const CholArgs a, int p) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  const int j = p + NB + blockIdx.x * NB + threadIdx.x;
  __shared__ float u[NB][NB + 1];
  for (int idx = threadIdx.x; idx < NB * NB; idx += 64) {
    const int r = idx / NB, c = idx % NB;
    u[r][c] = c >= r ? G[(size_t)(p + r) * a.ldg + p + c] : 0.f;
  }
  __syncthreads();
  if (j >= a.M) return;
  float x[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) x[r] = G[(size_t)(p + r) * a.ldg + j];
#pragma unroll
  for (int r = 0; r < NB; ++r) {
    float v = x[r];
#pragma unroll
    for (int s = 0; s < r; ++s) v = fmaf(-u[s][r], x[s], v);
    x[r] = v / u[r][r];
  }
#pragma unroll
  for (int r = 0; r < NB; ++r) G[(size_t)(p + r) * a.ldg + j] = x[r];
}

// Trailing update of the upper triangle after panel p: tile (ti, tj), ti <= tj, of the
// trailing 64-blocks: G[i][j] -= sum_r U[p+r][i] U[p+r][j]; 256 threads, 4 x 4 each
__global__ void __launch_bounds__(256) syrk_kernel(const CholArgs a, int p) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  const int q0 = p + NB, nt = (a.M - q0) / NB;
  int t = blockIdx.x, ti = 0;
  while (t >= nt - ti) {
    t -= nt - ti;
    ++ti;
  }
  const int tj = ti + t;
  const int i0 = q0 + ti * NB, j0 = q0 + tj * NB;
  __shared__ __align__(16) float xi[NB][NB + 4];  // [r][column]
  __shared__ __align__(16) float xj[NB][NB + 4];
  for (int idx = threadIdx.x; idx < NB * NB / 4; idx += 256) {
    const int r = idx / (NB / 4), c = (idx % (NB / 4)) * 4;
    *reinterpret_cast<float4*>(&xi[r][c]) =
        *reinterpret_cast<const float4*>(G + (size_t)(p + r) * a.ldg + i0 + c);
    *reinterpret_cast<float4*>(&xj[r][c]) =
        *reinterpret_cast<const float4*>(G + (size_t)(p + r) * a.ldg + j0 + c);
  }
  __syncthreads();
  const int tr = (threadIdx.x / 16) * 4, tc = (threadIdx.x % 16) * 4;
  float acc[4][4] = {};
#pragma unroll 8
  for (int r = 0; r < NB; ++r) {
    const float4 a4 = *reinterpret_cast<const float4*>(&xi[r][tr]);
    const float4 b4 = *reinterpret_cast<const float4*>(&xj[r][tc]);
    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float4* gp = reinterpret_cast<float4*>(G + (size_t)(i0 + tr + u) * a.ldg + j0 + tc);
    float4 g4 = *gp;
    g4.x -= acc[u][0]; g4.y -= acc[u][1]; g4.z -= acc[u][2]; g4.w -= acc[u][3];
    *gp = g4;  // entries below the diagonal of a diagonal tile are never read
  }
}

// Triangular solve of block row p of the right-hand sides, one thread per column:
// forward (U_pp^T y = r) or backward (U_pp x = y)
__global__ void __launch_bounds__(128) solve_diag_kernel(const CholArgs a, int p, int backward) {
  const float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  __shared__ float u[NB][NB + 1];
  for (int idx = threadIdx.x; idx < NB * NB; idx += 128) {
    const int r = idx / NB, c = idx % NB;
    u[r][c] = c >= r ? G[(size_t)(p + r) * a.ldg + p + c] : 0.f;
  }
  __syncthreads();
  const int c = blockIdx.x * 128 + threadIdx.x;
  if (c >= a.d) return;
  float x[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) x[r] = R[(size_t)(p + r) * a.d + c];
  if (!backward) {
#pragma unroll
    for (int r = 0; r < NB; ++r) {
      float v = x[r];
#pragma unroll
      for (int s = 0; s < r; ++s) v = fmaf(-u[s][r], x[s], v);
      x[r] = v / u[r][r];
    }
  } else {
#pragma unroll
    for (int r = NB - 1; r >= 0; --r) {
      float v = x[r];
#pragma unroll
      for (int s = r + 1; s < NB; ++s) v = fmaf(-u[r][s], x[s], v);
      x[r] = v / u[r][r];
    }
  }
#pragma unroll
  for (int r = 0; r < NB; ++r) R[(size_t)(p + r) * a.d + c] = x[r];
}

// Update of the block rows after (forward) or before (backward) block p:
//   forward:  R[q] -= U[p][q]^T Y[p]  for q > p      backward: R[q] -= U[q][p] X[p]  for q < p
// CTA (q block, 64 right-hand-side columns); 256 threads, 4 x 4 each
__global__ void __launch_bounds__(256) solve_update_kernel(const CholArgs a, int p, int backward) {
  const float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  const int q0 = backward ? blockIdx.x * NB : p + NB + blockIdx.x * NB;
  const int c0 = blockIdx.z * NB;
  __shared__ __align__(16) float us[NB][NB + 4];  // [r][q]: coefficient of row r of block p in row q
  __shared__ __align__(16) float ys[NB][NB + 4];  // [r][c]: solved rows of block p
  for (int idx = threadIdx.x; idx < NB * NB; idx += 256) {
    const int r = idx / NB, q = idx % NB;
    us[r][q] = backward ? G[(size_t)(q0 + q) * a.ldg + p + r] : G[(size_t)(p + r) * a.ldg + q0 + q];
    ys[r][q] = R[(size_t)(p + r) * a.d + c0 + q];
  }
  __syncthreads();
  const int tq = (threadIdx.x / 16) * 4, tc = (threadIdx.x % 16) * 4;
  float acc[4][4] = {};
#pragma unroll 8
  for (int r = 0; r < NB; ++r) {
    const float4 a4 = *reinterpret_cast<const float4*>(&us[r][tq]);
    const float4 b4 = *reinterpret_cast<const float4*>(&ys[r][tc]);
    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    float4* rp = reinterpret_cast<float4*>(R + (size_t)(q0 + tq + u) * a.d + c0 + tc);
    float4 r4 = *rp;
    r4.x -= acc[u][0]; r4.y -= acc[u][1]; r4.z -= acc[u][2]; r4.w -= acc[u][3];
    *rp = r4;
  }
}

__global__ void __launch_bounds__(256) copy_out_kernel(const CholArgs a) {
  const float* R = prob(a.r, (size_t)a.M * a.d);
  float* X = prob(a.x, (size_t)a.k * a.d);
  for (size_t idx = (size_t)blockIdx.x * 256 + threadIdx.x; idx < (size_t)a.k * a.d;
       idx += (size_t)gridDim.x * 256)
    X[idx] = R[idx];
}

}  // namespace

cudaError_t launch_chol_solve(const CholArgs& a, cudaStream_t s) {
  if (a.batch <= 0 || a.M <= 0) return cudaSuccess;
  if (a.M > kCholMaxM || a.M % NB || a.k > a.M || a.d % NB || a.d > 1024 || a.ldg % 4 ||
      a.ldg < a.M)
    return cudaErrorInvalidValue;
  const int nb = a.M / NB, B = a.batch, dcb = a.d / NB;
  int launches = 0;
  shift_kernel<<<dim3(1, B), 256, 0, s>>>(a);
  ++launches;
  for (int b = 0; b < nb; ++b) {  // G + lam I = U^T U
    const int p = b * NB, rest = nb - b - 1;
    potrf_kernel<<<dim3(1, B), 256, 0, s>>>(a, p);
    ++launches;
    if (rest > 0) {
      trsm_row_kernel<<<dim3(rest, B), 64, 0, s>>>(a, p);
      syrk_kernel<<<dim3(rest * (rest + 1) / 2, B), 256, 0, s>>>(a, p);
      launches += 2;
    }
  }
  for (int b = 0; b < nb; ++b) {  // U^T Y = R
    const int p = b * NB, rest = nb - b - 1;
    solve_diag_kernel<<<dim3((a.d + 127) / 128, B), 128, 0, s>>>(a, p, 0);
    ++launches;
    if (rest > 0) {
      solve_update_kernel<<<dim3(rest, B, dcb), 256, 0, s>>>(a, p, 0);
      ++launches;
    }
  }
  for (int b = nb - 1; b >= 0; --b) {  // U X = Y
    const int p = b * NB;
    solve_diag_kernel<<<dim3((a.d + 127) / 128, B), 128, 0, s>>>(a, p, 1);
    ++launches;
    if (b > 0) {
      solve_update_kernel<<<dim3(b, B, dcb), 256, 0, s>>>(a, p, 1);
      ++launches;
    }
  }
  copy_out_kernel<<<dim3(64, B), 256, 0, s>>>(a);
  ++launches;
  count_launches(launches);
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
