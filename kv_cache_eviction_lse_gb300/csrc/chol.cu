// Ridge solve of the value refit's normal equations, batched over (layer, KV head):
//   (G + lam I) X = R,   lam = lam_rel * mean(diag G[:k, :k])
// by a blocked right-looking upper Cholesky factorisation G + lam I = U^T U in fp32
// and two blocked triangular solves U^T Y = R, U X = Y.  Every factorisation step is one
// launch over all problems, so the trailing updates (the bulk of the work) spread over
// the whole GPU instead of one CTA per problem:
//   per 64-row panel p:  factor the diagonal block (one CTA per problem), solve the row
//                        panel U_pp^T X = G[p][p+64:] (CTAs over 64-column blocks), update
//                        the trailing upper triangle G -= X^T X (CTAs over 64 x 64 tiles)
// The solves then run as one launch: the 64-column blocks of right-hand sides are
// independent, so one CTA per (problem, column block) takes both sweeps, each a diagonal
// block's triangular solve followed by the update of every remaining block row.
// G arrives as its upper block triangle (the Gram kernel writes only those tiles); the
// lower triangle is never read.  Rows/columns k .. M-1 (padding of the kept-key
// dimension) are decoupled: their diagonal becomes 1 and their right-hand side 0.
#include <math.h>

#include "gram.cuh"

namespace kvs {

__device__ int g_chol_error = 0;

namespace {

constexpr int NB = 64;         // panel / block size (M is a multiple of 64)
constexpr int kLd = NB + 4;    // row stride of staged 64 x 64 blocks: 16-byte aligned rows
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

// The diagonal-block kernels run once per panel with one small CTA per problem, so they
// are latency chains and their code is fetched once per launch: fully unrolled 64 x 64
// loops (thousands of instructions) are bound by that fetch.  Each keeps a column in
// registers under a rolled pivot loop instead: the column is shifted by one register per
// step (x[i] holds row r + i), fused with the update x[i-1] = x[i] - w[i] x[0], so the
// pivot is always x[0] and the step's line of U is staged pre-shifted (w[i] = U[r][r+i])
// for aligned 16-byte reads.

// Cholesky of the diagonal block at p (upper, in place), one CTA of 64 threads per
// problem: thread c keeps column c of the block in registers; per pivot r the owner of
// column r takes the square root, every later column scales its row-r entry, stores it
// and publishes it, and each column applies the rank-1 update to its own entries.
__global__ void __launch_bounds__(NB) potrf_kernel(const CholArgs a, int p) {
  float* G = prob(a.g, (size_t)a.M * a.ldg) + (size_t)p * a.ldg + p;
  const int c = threadIdx.x;
  __shared__ __align__(16) float prow[NB];  // prow[i] = U[r][r + i] (i >= 1), 0 past the block
  __shared__ float pinv;
  float x[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i) x[i] = i <= c ? G[(size_t)i * a.ldg + c] : 0.f;
  prow[c] = 0.f;
#pragma unroll 1
  for (int r = 0; r < NB; ++r) {
    if (c == r) {
      const float v = x[0];
      if (!(v > 0.f)) atomicCAS(&g_chol_error, 0, kErrNotSpd);
      const float piv = sqrtf(fmaxf(v, 1e-30f));
      G[(size_t)r * a.ldg + r] = piv;
      pinv = 1.f / piv;
    }
    __syncthreads();
    float xr = 0.f;
    if (c > r) {
      xr = x[0] * pinv;
      G[(size_t)r * a.ldg + c] = xr;
      prow[c - r] = xr;
    }
    __syncthreads();
    // columns c > r: rows r+1 .. c; past c the registers hold nothing that is stored
#pragma unroll
    for (int i4 = 0; i4 < NB; i4 += 4) {
      const float4 w = *reinterpret_cast<const float4*>(&prow[i4]);
      const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (i4 + e >= 1) x[i4 + e - 1] = fmaf(-wv[e], xr, x[i4 + e]);
    }
    x[NB - 1] = 0.f;
    __syncthreads();  // prow is rewritten by the next pivot
    if (c > r) prow[c - r] = 0.f;
  }
}

// Triangular solve of 64 rows in registers against the staged diagonal block (rows of w
// pre-shifted as above, dinv = 1 / diag), one column per thread; row r of the solution
// is written to out[r * ld] as soon as it is final.  Forward: U^T y = x with x[i] = row i
// initially; backward: U y = x with x[i] = row 63 - i initially.
template <bool BACKWARD>
__device__ __forceinline__ void tri_solve_col(float (&x)[NB], const float (*w)[NB],
                                              const float* dinv, float* out, size_t ld) {
#pragma unroll 1
  for (int k = 0; k < NB; ++k) {
    const int r = BACKWARD ? NB - 1 - k : k;
    const float xr = x[0] * dinv[r];
    out[(size_t)r * ld] = xr;
#pragma unroll
    for (int i4 = 0; i4 < NB; i4 += 4) {
      const float4 q = *reinterpret_cast<const float4*>(&w[r][i4]);
      const float qv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (i4 + e >= 1) x[i4 + e - 1] = fmaf(-qv[e], xr, x[i4 + e]);
    }
    x[NB - 1] = 0.f;
  }
}

// Stages the diagonal block at p pre-shifted for a forward solve (w[r][i] = U[r][r+i]) or
// a backward one (w[r][i] = U[r-i][r]), zero past the block, and 1 / diag (nt threads).
__device__ __forceinline__ void load_diag_block(const float* G, int ldg, int p, int nt,
                                                bool backward, float (*w)[NB], float* dinv) {
  for (int idx = threadIdx.x; idx < NB * NB; idx += nt) w[idx / NB][idx % NB] = 0.f;
  __syncthreads();
  for (int idx = threadIdx.x; idx < NB * NB; idx += nt) {
    const int r = idx / NB, c = idx % NB;  // U[r][c], c >= r
    if (c >= r) {
      const float v = G[(size_t)(p + r) * ldg + p + c];
      if (backward)
        w[c][c - r] = v;
      else
        w[r][c - r] = v;
    }
  }
  __syncthreads();
  if (threadIdx.x < NB) dinv[threadIdx.x] = 1.f / w[threadIdx.x][0];
  __syncthreads();
}

// Row panel: G[p..p+64][j] = U_pp^-T G[p..p+64][j] for the 64 columns j of block
// blockIdx.x after the diagonal block; one thread per column
__global__ void __launch_bounds__(NB) trsm_row_kernel(const CholArgs a, int p) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  const int j = p + NB + blockIdx.x * NB + threadIdx.x;
  __shared__ __align__(16) float w[NB][NB];
  __shared__ float dinv[NB];
  load_diag_block(G, a.ldg, p, NB, false, w, dinv);
  if (j >= a.M) return;
  float x[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) x[r] = G[(size_t)(p + r) * a.ldg + j];
  tri_solve_col<false>(x, w, dinv, G + (size_t)p * a.ldg + j, a.ldg);
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

// Both triangular solves (U^T Y = R, then U X = Y) of one problem and one 64-column block
// of right-hand sides; the column blocks are independent, so each CTA runs the whole
// chain with no other launch.  Per 64-row block p (forward ascending, backward
// descending): the diagonal solve in registers (threads 0..63, one column each) into the
// stage ys, then every remaining block row q is updated, forward R[q] -= U[p][q]^T Y[p],
// backward R[q] -= U[q][p] X[p] (64 x 64 x 64, a 4 x 4 tile per thread).  Y goes back to
// R; X rows below k go to the output.
__global__ void __launch_bounds__(256) solve_kernel(const CholArgs a) {
  const float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  float* X = prob(a.x, (size_t)a.k * a.d);
  const int c0 = blockIdx.x * NB, tid = threadIdx.x, nb = a.M / NB;
  __shared__ __align__(16) float w[NB][NB];   // diagonal block, pre-shifted
  __shared__ float dinv[NB];
  __shared__ __align__(16) float ys[NB][kLd];  // solved rows of block p
  __shared__ __align__(16) float us[NB][kLd];  // coefficients of block p in block row q
  const int tq = (tid / 16) * 4, tc = (tid % 16) * 4;
  for (int pass = 0; pass < 2; ++pass) {
    const bool back = pass == 1;
    for (int bi = 0; bi < nb; ++bi) {
      const int p = (back ? nb - 1 - bi : bi) * NB;
      __syncthreads();  // the previous block's reads of w, ys and us are done
      load_diag_block(G, a.ldg, p, 256, back, w, dinv);
      if (tid < NB) {
        float x[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i)
          x[i] = R[(size_t)(p + (back ? NB - 1 - i : i)) * a.d + c0 + tid];
        if (back)
          tri_solve_col<true>(x, w, dinv, &ys[0][tid], kLd);
        else
          tri_solve_col<false>(x, w, dinv, &ys[0][tid], kLd);
      }
      __syncthreads();
      for (int idx = tid; idx < NB * NB; idx += 256) {
        const int r = idx / NB, c = idx % NB;
        if (!back)
          R[(size_t)(p + r) * a.d + c0 + c] = ys[r][c];
        else if (p + r < a.k)
          X[(size_t)(p + r) * a.d + c0 + c] = ys[r][c];
      }
      const int q_begin = back ? 0 : p + NB, q_end = back ? p : a.M;
      for (int q = q_begin; q < q_end; q += NB) {
        for (int idx = tid; idx < NB * NB; idx += 256) {
          const int i = idx / NB, j = idx % NB;  // consecutive threads read consecutive addresses
          if (back)
            us[j][i] = G[(size_t)(q + i) * a.ldg + p + j];  // U[q+i][p+j]
          else
            us[i][j] = G[(size_t)(p + i) * a.ldg + q + j];  // U[p+i][q+j]
        }
        __syncthreads();
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
          float4* rp = reinterpret_cast<float4*>(R + (size_t)(q + tq + u) * a.d + c0 + tc);
          float4 r4 = *rp;
          r4.x -= acc[u][0]; r4.y -= acc[u][1]; r4.z -= acc[u][2]; r4.w -= acc[u][3];
          *rp = r4;
        }
        __syncthreads();  // us is reloaded for the next block row
      }
    }
  }
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
    potrf_kernel<<<dim3(1, B), NB, 0, s>>>(a, p);
    ++launches;
    if (rest > 0) {
      trsm_row_kernel<<<dim3(rest, B), NB, 0, s>>>(a, p);
      syrk_kernel<<<dim3(rest * (rest + 1) / 2, B), 256, 0, s>>>(a, p);
      launches += 2;
    }
  }
  solve_kernel<<<dim3(dcb, B), 256, 0, s>>>(a);  // U^T Y = R, U X = Y, X = rows < k
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
