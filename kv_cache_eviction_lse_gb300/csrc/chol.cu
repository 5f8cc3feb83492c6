// Ridge solve of the value refit's normal equations, batched over (layer, KV head):
//   (G + lam I) X = R,   lam = lam_rel * mean(diag G[:k, :k])
// by a blocked right-looking upper Cholesky factorisation G + lam I = U^T U in fp32
// and two blocked triangular solves U^T Y = R, U X = Y.  Every factorisation step is one
// launch over all problems, so the trailing updates (the bulk of the work) spread over
// the whole GPU instead of one CTA per problem:
//   per 64-row panel p:  factor the diagonal block (one CTA per problem), solve the row
//                        panel U_pp^T X = [G[p][p+64:] | R[p]] (CTAs over 64-column
//                        blocks), update the trailing upper triangle G -= X^T X and the
//                        trailing rows of R (CTAs over 64 x 64 tiles)
// R rides along as extra columns of the factorised matrix, so the forward solve U^T Y = R
// is done when the factorisation is.  The backward solve U X = Y then runs as one launch:
// the column blocks of right-hand sides are independent, so one CTA per (problem, column
// block) takes the whole sweep, each diagonal block's triangular solve followed by the
// update of every block row above it.
// G arrives as its upper block triangle (the Gram kernel writes only those tiles); the
// lower triangle is never read.  Rows/columns k .. M-1 (padding of the kept-key
// dimension) are decoupled: their diagonal becomes 1 and their right-hand side 0.
#include <math.h>

#include <algorithm>

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
// for aligned 16-byte reads.  After 16 steps the top 16 registers hold only finished
// rows, so the 64 steps run as four rolled loops over 64, 48, 32 and 16 registers.
static_assert(NB == 64, "the diagonal-block chains run in four phases of 16 steps");

// x[i-1] = x[i] - wrow[i] xr for i = 1 .. W-1, x[W-1] = 0 (wrow 16-byte aligned)
template <int W>
__device__ __forceinline__ void shift_axpy(float (&x)[NB], const float* wrow, float xr) {
#pragma unroll
  for (int i4 = 0; i4 < W; i4 += 4) {
    const float4 q = *reinterpret_cast<const float4*>(&wrow[i4]);
    const float qv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (i4 + e >= 1) x[i4 + e - 1] = fmaf(-qv[e], xr, x[i4 + e]);
  }
  x[W - 1] = 0.f;
}

// Pivots r0 .. r0+15 of the diagonal block (see potrf_kernel); W registers are live.
template <int W>
__device__ __forceinline__ void potrf_steps(float (&x)[NB], int r0, int c, float* G, int ldg,
                                            float* prow, float* pinv) {
#pragma unroll 1
  for (int r = r0; r < r0 + 16; ++r) {
    if (c == r) {
      const float v = x[0];
      if (!(v > 0.f)) atomicCAS(&g_chol_error, 0, kErrNotSpd);
      const float piv = sqrtf(fmaxf(v, 1e-30f));
      G[(size_t)r * ldg + r] = piv;
      *pinv = 1.f / piv;
    }
    __syncthreads();
    float xr = 0.f;
    if (c > r) {
      xr = x[0] * *pinv;
      G[(size_t)r * ldg + c] = xr;
      prow[c - r] = xr;
    }
    __syncthreads();
    // columns c > r: rows r+1 .. c; past c the registers hold nothing that is stored
    shift_axpy<W>(x, prow, xr);
    __syncthreads();  // prow is rewritten by the next pivot
    if (c > r) prow[c - r] = 0.f;
  }
}

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
  potrf_steps<64>(x, 0, c, G, a.ldg, prow, &pinv);
  potrf_steps<48>(x, 16, c, G, a.ldg, prow, &pinv);
  potrf_steps<32>(x, 32, c, G, a.ldg, prow, &pinv);
  potrf_steps<16>(x, 48, c, G, a.ldg, prow, &pinv);
}

// Triangular solve of 64 rows in registers against the staged diagonal block (rows of w
// pre-shifted as above, dinv = 1 / diag), one column per thread; row r of the solution
// is written to out[r * ld] as soon as it is final.  Forward: U^T y = x with x[i] = row i
// initially; backward: U y = x with x[i] = row 63 - i initially.
template <bool BACKWARD, int W>
__device__ __forceinline__ void tri_steps(float (&x)[NB], const float (*w)[kLd],
                                          const float* dinv, float* out, size_t ld, int k0) {
#pragma unroll 1
  for (int k = k0; k < k0 + 16; ++k) {
    const int r = BACKWARD ? NB - 1 - k : k;
    const float xr = x[0] * dinv[r];
    out[(size_t)r * ld] = xr;
    shift_axpy<W>(x, w[r], xr);
  }
}

template <bool BACKWARD>
__device__ __forceinline__ void tri_solve_col(float (&x)[NB], const float (*w)[kLd],
                                              const float* dinv, float* out, size_t ld) {
  tri_steps<BACKWARD, 64>(x, w, dinv, out, ld, 0);
  tri_steps<BACKWARD, 48>(x, w, dinv, out, ld, 16);
  tri_steps<BACKWARD, 32>(x, w, dinv, out, ld, 32);
  tri_steps<BACKWARD, 16>(x, w, dinv, out, ld, 48);
}

// Stages the diagonal block at p pre-shifted for a forward solve (w[r][i] = U[r][r+i]) or
// a backward one (w[r][i] = U[r-i][r]), zero past the block, and 1 / diag, with NT
// threads in one pass: each thread issues all its (coalesced) loads before it stores, and
// the lower-triangle positions it visits map one to one onto the zero slots (forward:
// (r, c < r) -> w[r][63 - c]; backward: (r > c, c) -> w[c][r]).
template <int NT, bool BACKWARD>
__device__ __forceinline__ void load_diag_block(const float* G, int ldg, int p,
                                                float (*w)[kLd], float* dinv) {
  constexpr int PER = NB * NB / NT;
  float v[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = (int)threadIdx.x + e * NT, r = idx / NB, c = idx % NB;
    v[e] = c >= r ? G[(size_t)(p + r) * ldg + p + c] : 0.f;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = (int)threadIdx.x + e * NT, r = idx / NB, c = idx % NB;
    if (BACKWARD) {
      if (c >= r)
        w[c][c - r] = v[e];
      else
        w[c][r] = 0.f;
    } else {
      if (c >= r)
        w[r][c - r] = v[e];
      else
        w[r][NB - 1 - c] = 0.f;
    }
  }
  __syncthreads();
  if (threadIdx.x < NB) dinv[threadIdx.x] = 1.f / w[threadIdx.x][0];
  __syncthreads();
}

// Row panel: X = U_pp^-T B for the 64 columns of block blockIdx.x of [G[p][p+64:] | R[p]]
// (the first `rest` blocks are G's, the next d / 64 are R's); one thread per column
__global__ void __launch_bounds__(NB) trsm_row_kernel(const CholArgs a, int p, int rest) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  const bool in_r = (int)blockIdx.x >= rest;
  float* col = in_r ? R + (size_t)p * a.d + (blockIdx.x - rest) * NB + threadIdx.x
                    : G + (size_t)p * a.ldg + p + NB + blockIdx.x * NB + threadIdx.x;
  const size_t ld = in_r ? (size_t)a.d : (size_t)a.ldg;
  __shared__ __align__(16) float w[NB][kLd];
  __shared__ float dinv[NB];
  load_diag_block<NB, false>(G, a.ldg, p, w, dinv);
  float x[NB];
#pragma unroll
  for (int r = 0; r < NB; ++r) x[r] = col[(size_t)r * ld];
  tri_solve_col<false>(x, w, dinv, col, ld);
}

// Trailing update after panel p, 256 threads, 4 x 4 each.  Blocks below nt (nt + 1) / 2:
// tile (ti, tj), ti <= tj, of the trailing 64-blocks, G[i][j] -= sum_r U[p+r][i] U[p+r][j];
// the rest: tile (ti, column block cb) of R's trailing rows, R[i][c] -= sum_r U[p+r][i] Y[p+r][c]
__global__ void __launch_bounds__(256) syrk_kernel(const CholArgs a, int p) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  const int q0 = p + NB, nt = (a.M - q0) / NB;
  int t = blockIdx.x, ti = 0;
  const bool in_r = t >= nt * (nt + 1) / 2;
  const float* src_j;  // rows p .. p+63 of the right factor, and its row stride
  size_t ldj;
  float* dst;          // the updated tile and its row stride
  size_t ldd;
  if (in_r) {
    t -= nt * (nt + 1) / 2;
    const int ncb = a.d / NB;
    ti = t / ncb;
    const int c0 = (t % ncb) * NB;
    src_j = R + (size_t)p * a.d + c0;
    ldj = a.d;
    dst = R + (size_t)(q0 + ti * NB) * a.d + c0;
    ldd = a.d;
  } else {
    while (t >= nt - ti) {
      t -= nt - ti;
      ++ti;
    }
    const int j0 = q0 + (ti + t) * NB;
    src_j = G + (size_t)p * a.ldg + j0;
    ldj = a.ldg;
    dst = G + (size_t)(q0 + ti * NB) * a.ldg + j0;
    ldd = a.ldg;
  }
  const int i0 = q0 + ti * NB;
  __shared__ __align__(16) float xi[NB][NB + 4];  // [r][column]
  __shared__ __align__(16) float xj[NB][NB + 4];
  for (int idx = threadIdx.x; idx < NB * NB / 4; idx += 256) {
    const int r = idx / (NB / 4), c = (idx % (NB / 4)) * 4;
    *reinterpret_cast<float4*>(&xi[r][c]) =
        *reinterpret_cast<const float4*>(G + (size_t)(p + r) * a.ldg + i0 + c);
    *reinterpret_cast<float4*>(&xj[r][c]) =
        *reinterpret_cast<const float4*>(src_j + (size_t)r * ldj + c);
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
    float4* gp = reinterpret_cast<float4*>(dst + (size_t)(tr + u) * ldd + tc);
    float4 g4 = *gp;
    g4.x -= acc[u][0]; g4.y -= acc[u][1]; g4.z -= acc[u][2]; g4.w -= acc[u][3];
    *gp = g4;  // entries below the diagonal of a diagonal tile are never read
  }
}

// Backward solve U X = Y of one problem and one block of CB right-hand-side columns (Y
// is in R: the forward solve rode along with the factorisation); the column blocks are
// independent, so each CTA runs the whole chain with no other launch (narrow blocks give
// more CTAs, whose latency chains overlap).  Per 64-row block p, descending: the diagonal
// solve in registers (threads 0..CB-1, one column each) into the stage ys, then every
// block row q above it is updated, R[q] -= U[q][p] X[p] (64 x 64 x CB; a thread owns
// CB/16 rows x 4 columns).  The next block row's U block is loaded into registers while
// the current one is multiplied, and a thread's R tile is read before the products so
// that its loads overlap them.  X rows below k go to the output.
template <int CB>
__global__ void __launch_bounds__(256, CB == 64 ? 1 : 2) solve_kernel(const CholArgs a) {
  constexpr int CG = CB / 4;      // groups of 4 columns
  constexpr int RPT = CB / 16;    // rows per thread in the updates
  constexpr int LDY = CB + 4;     // ys row stride (16-byte aligned rows)
  constexpr int UPT = NB * NB / 256;  // U block elements per thread
  static_assert(RPT >= 1 && (256 / CG) * RPT == NB, "column block of 16, 32 or 64");
  const float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  float* X = prob(a.x, (size_t)a.k * a.d);
  const int c0 = blockIdx.x * CB, tid = threadIdx.x, nb = a.M / NB;
  __shared__ __align__(16) float w[NB][kLd];  // diagonal block, pre-shifted
  __shared__ float dinv[NB];
  __shared__ __align__(16) float ys[NB][LDY];  // solved rows of block p
  __shared__ __align__(16) float us[NB][kLd];  // us[r][i] = U[q+i][p+r]
  const int tq = (tid / CG) * RPT, tc = (tid % CG) * 4;
  for (int p = (nb - 1) * NB; p >= 0; p -= NB) {
    // the previous block's reads of w, ys and us are done and its updates of R visible
    __syncthreads();
    float x[NB];
    if (tid < CB) {  // the block's right-hand sides, in flight while w is staged
#pragma unroll
      for (int i = 0; i < NB; ++i) x[i] = R[(size_t)(p + NB - 1 - i) * a.d + c0 + tid];
    }
    load_diag_block<256, true>(G, a.ldg, p, w, dinv);
    if (tid < CB) tri_solve_col<true>(x, w, dinv, &ys[0][tid], LDY);
    __syncthreads();
    for (int idx = tid; idx < NB * CB; idx += 256) {
      const int r = idx / CB, c = idx % CB;
      if (p + r < a.k) X[(size_t)(p + r) * a.d + c0 + c] = ys[r][c];
    }
    // U[q+i][p+j] of block row q (consecutive threads read consecutive addresses)
    float ureg[UPT];
    auto load_u = [&](int q) {
#pragma unroll
      for (int e = 0; e < UPT; ++e) {
        const int idx = tid + 256 * e, i = idx / NB, j = idx % NB;
        ureg[e] = G[(size_t)(q + i) * a.ldg + p + j];
      }
    };
    if (p > 0) load_u(0);
    for (int q = 0; q < p; q += NB) {
#pragma unroll
      for (int e = 0; e < UPT; ++e) {
        const int idx = tid + 256 * e, i = idx / NB, j = idx % NB;
        us[j][i] = ureg[e];
      }
      float4 r4[RPT];
#pragma unroll
      for (int u = 0; u < RPT; ++u)
        r4[u] = *reinterpret_cast<const float4*>(R + (size_t)(q + tq + u) * a.d + c0 + tc);
      __syncthreads();
      if (q + NB < p) load_u(q + NB);  // in flight during the products
      float acc[RPT][4] = {};
#pragma unroll 8
      for (int r = 0; r < NB; ++r) {
        const float4 b4 = *reinterpret_cast<const float4*>(&ys[r][tc]);
        const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
        float av[RPT];
#pragma unroll
        for (int u = 0; u < RPT; ++u) av[u] = us[r][tq + u];
#pragma unroll
        for (int u = 0; u < RPT; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
      }
#pragma unroll
      for (int u = 0; u < RPT; ++u) {
        r4[u].x -= acc[u][0];
        r4[u].y -= acc[u][1];
        r4[u].z -= acc[u][2];
        r4[u].w -= acc[u][3];
        *reinterpret_cast<float4*>(R + (size_t)(q + tq + u) * a.d + c0 + tc) = r4[u];
      }
      __syncthreads();  // us is rewritten for the next block row
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
  for (int b = 0; b < nb; ++b) {  // G + lam I = U^T U, and Y = U^-T R alongside
    const int p = b * NB, rest = nb - b - 1;
    potrf_kernel<<<dim3(1, B), NB, 0, s>>>(a, p);
    trsm_row_kernel<<<dim3(rest + dcb, B), NB, 0, s>>>(a, p, rest);
    launches += 2;
    if (rest > 0) {
      syrk_kernel<<<dim3(rest * (rest + 1) / 2 + rest * dcb, B), 256, 0, s>>>(a, p);
      ++launches;
    }
  }
  // U X = Y, X = rows < k: the narrowest right-hand-side blocks (16 or 32
  // columns) whose CTAs are all resident at once (two per SM), else blocks of 64 columns
  static int nsm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!nsm[dev]) cudaDeviceGetAttribute(&nsm[dev], cudaDevAttrMultiProcessorCount, dev);
  const size_t resident = 2 * (size_t)std::max(1, nsm[dev]);
  if ((size_t)dcb * 4 * B <= resident)
    solve_kernel<16><<<dim3(dcb * 4, B), 256, 0, s>>>(a);
  else if ((size_t)dcb * 2 * B <= resident)
    solve_kernel<32><<<dim3(dcb * 2, B), 256, 0, s>>>(a);
  else
    solve_kernel<64><<<dim3(dcb, B), 256, 0, s>>>(a);
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
