// Ridge solve of the value refit's normal equations, batched over (layer, KV head):
//   (G + lam I) X = R,   lam = lam_rel * mean(diag G[:k, :k])
// by a blocked right-looking upper Cholesky factorisation G + lam I = U^T U in fp32
// and two blocked triangular solves U^T Y = R, U X = Y.  Every factorisation step is one
// launch over all problems, so the trailing updates (the bulk of the work) spread over
// the whole GPU instead of one CTA per problem:
//   per 64-row panel p:  factor the diagonal block and invert it, W = U_pp^-T (one CTA
//                        per problem; the identity rides along the elimination), form
//                        the row panel X = W [G[p][p+64:] | R[p]] (CTAs over 64-column
//                        blocks), update the trailing upper triangle G -= X^T X and the
//                        trailing rows of R (CTAs over 64 x 64 tiles)
// R rides along as extra columns of the factorised matrix, so the forward solve U^T Y = R
// is done when the factorisation is.  The backward solve U X = Y then runs as one launch:
// the column blocks of right-hand sides are independent, so one CTA per (problem, column
// block) takes the whole sweep, each diagonal block's product X[p] = W^T Y[p] followed by
// the update of every block row above it.  Only the diagonal blocks' factorisations are
// serial chains (64 pivots each); the triangular solves are products with the inverted
// diagonal blocks.
// G arrives as its upper block triangle (the Gram kernel writes only those tiles); its
// lower triangle is never read, and the factorisation keeps each W in the strictly lower
// part of its diagonal block.  Rows/columns k .. M-1 (padding of the kept-key dimension)
// are decoupled: their diagonal becomes 1 and their right-hand side 0.
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
// One barrier per pivot: the owners of the block's columns c >= r publish their raw
// row-r entries into raw[r & 1] (two buffers, so a pivot's writes never meet the
// previous pivot's reads), and every thread derives the pivot's inverse square root
// from raw[r & 1][0] itself.  With d = A'[r][r], U[r][c] = A'[r][c] / sqrt(d), and the
// rank-1 update of column c is x[i] -= A'[r][r+i] * (A'[r][c] / d).
template <int W>
__device__ __forceinline__ void potrf_steps(float (&x)[NB], int r0, int c, bool carried,
                                            float* D, int ldg, float (*raw)[NB]) {
#pragma unroll 1
  for (int r = r0; r < r0 + 16; ++r) {
    float* row = raw[r & 1];
    if (!carried && c >= r) row[c - r] = x[0];
    __syncthreads();
    const float dv = fmaxf(row[0], 1e-30f);
    const float pinv = rsqrtf(dv);  // 1 / U[r][r]
    const float xr = x[0] * pinv;  // U[r][c] (block columns) or W[r][c] (carried identity)
    float t = 0.f;
    if (!carried) {
      if (c == r) {
        if (!(row[0] > 0.f)) atomicCAS(&g_chol_error, 0, kErrNotSpd);
        D[(size_t)r * ldg + r] = dv * pinv;
      } else if (c > r) {
        D[(size_t)r * ldg + c] = xr;
        t = xr * pinv;
      }
    } else {
      if (r > c) D[(size_t)r * ldg + c] = xr;  // W strictly below the diagonal
      t = xr * pinv;
    }
    // columns c > r: rows r+1 .. c; past c (and past the block) the registers hold
    // nothing that is stored
    shift_axpy<W>(x, row, t);
  }
}

// Cholesky of the diagonal block at p (upper, in place) and W = U_pp^-T, one CTA of 128
// threads per problem.  Threads 0..63 keep column c of the block in registers; threads
// 64..127 keep column c of the identity, which rides along as right-hand sides, so the
// forward elimination that factors the block turns it into U_pp^-T.  Per pivot r the
// block's columns store U[r][c] and the identity's store W[r][c] (r > c) into the
// block's lower triangle, which nothing else reads; W's diagonal is 1 / U[r][r].
__global__ void __launch_bounds__(2 * NB) potrf_kernel(const CholArgs a, int p) {
  float* D = prob(a.g, (size_t)a.M * a.ldg) + (size_t)p * a.ldg + p;
  const bool carried = threadIdx.x >= NB;
  const int c = threadIdx.x & (NB - 1);
  __shared__ __align__(16) float raw[2][NB];
  float x[NB];
#pragma unroll
  for (int i = 0; i < NB; ++i)
    x[i] = carried ? (i == c ? 1.f : 0.f) : (i <= c ? D[(size_t)i * a.ldg + c] : 0.f);
  raw[0][c] = 0.f;
  raw[1][c] = 0.f;
  __syncthreads();
  potrf_steps<64>(x, 0, c, carried, D, a.ldg, raw);
  potrf_steps<48>(x, 16, c, carried, D, a.ldg, raw);
  potrf_steps<32>(x, 32, c, carried, D, a.ldg, raw);
  potrf_steps<16>(x, 48, c, carried, D, a.ldg, raw);
}

// W = U_pp^-T of the diagonal block at p, staged in shared memory by NT threads: with
// TRANSPOSE, w[j][i] = W[i][j] (the columns of W as rows), else w[j][i] = W[j][i].  W's
// strictly lower part is read from the block's lower triangle, its diagonal is
// 1 / U[i][i], and its upper part is 0.  Each thread issues all its loads (coalesced
// along rows of W) before it stores, so their latencies overlap.
template <int NT, bool TRANSPOSE>
__device__ __forceinline__ void load_winv(const float* G, int ldg, int p, float (*w)[kLd]) {
  constexpr int PER = NB * NB / NT;
  const float* D = G + (size_t)p * ldg + p;
  float v[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = (int)threadIdx.x + e * NT, i = idx / NB, j = idx % NB;  // W[i][j]
    v[e] = i >= j ? D[(size_t)i * ldg + j] : 0.f;
  }
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int idx = (int)threadIdx.x + e * NT, i = idx / NB, j = idx % NB;
    const float wv = i == j ? 1.f / v[e] : v[e];
    if (TRANSPOSE)
      w[j][i] = wv;
    else
      w[i][j] = wv;
  }
}

// Row panel: X = W B for the 64 columns of block blockIdx.x of [G[p][p+64:] | R[p]] (the
// first `rest` blocks are G's, the next d / 64 are R's), W = U_pp^-T from the diagonal
// block; 256 threads, 4 x 4 results each, written over B.
__global__ void __launch_bounds__(256) panel_kernel(const CholArgs a, int p, int rest) {
  float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  const bool in_r = (int)blockIdx.x >= rest;
  float* blk = in_r ? R + (size_t)p * a.d + (blockIdx.x - rest) * NB
                    : G + (size_t)p * a.ldg + p + NB + blockIdx.x * NB;
  const size_t ld = in_r ? (size_t)a.d : (size_t)a.ldg;
  __shared__ __align__(16) float wt[NB][kLd];  // wt[j][i] = W[i][j]
  __shared__ __align__(16) float bs[NB][kLd];  // bs[j][c] = B[j][c]
  load_winv<256, true>(G, a.ldg, p, wt);
  for (int idx = threadIdx.x; idx < NB * NB / 4; idx += 256) {
    const int r = idx / (NB / 4), c = (idx % (NB / 4)) * 4;
    *reinterpret_cast<float4*>(&bs[r][c]) =
        *reinterpret_cast<const float4*>(blk + (size_t)r * ld + c);
  }
  __syncthreads();
  const int tr = (threadIdx.x / 16) * 4, tc = (threadIdx.x % 16) * 4;
  float acc[4][4] = {};
#pragma unroll 8
  for (int j = 0; j < NB; ++j) {  // X[i][c] = sum_j W[i][j] B[j][c]
    const float4 a4 = *reinterpret_cast<const float4*>(&wt[j][tr]);
    const float4 b4 = *reinterpret_cast<const float4*>(&bs[j][tc]);
    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, bv[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<float4*>(blk + (size_t)(tr + u) * ld + tc) =
        make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
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
// independent, so each CTA runs the whole sweep with no other launch.  Per 64-row block
// p, descending: X[p] = U_pp^-1 Y[p] = W^T Y[p] with the factorisation's W = U_pp^-T
// (64 x 64 x CB), then every block row q above it is updated, R[q] -= U[q][p] X[p]
// (64 x 64 x CB); a thread owns CB/16 rows x 4 columns of both products.  The next block
// row's U block is loaded into registers while the current one is multiplied, and a
// thread's R tile is read before the products so that its loads overlap them.  X rows
// below k go to the output.
template <int CB>
__global__ void __launch_bounds__(256, CB == 64 ? 1 : 2) solve_kernel(const CholArgs a) {
  constexpr int CG = CB / 4;      // groups of 4 columns
  constexpr int RPT = CB / 16;    // rows per thread in the products
  constexpr int LDY = CB + 4;     // row stride of yin / ys (16-byte aligned rows)
  constexpr int UPT = NB * NB / 256;  // U block elements per thread
  static_assert(RPT >= 1 && (256 / CG) * RPT == NB, "column block of 16, 32 or 64");
  const float* G = prob(a.g, (size_t)a.M * a.ldg);
  float* R = prob(a.r, (size_t)a.M * a.d);
  float* X = prob(a.x, (size_t)a.k * a.d);
  const int c0 = blockIdx.x * CB, tid = threadIdx.x, nb = a.M / NB;
  __shared__ __align__(16) float yin[NB][LDY];  // right-hand sides of block p
  __shared__ __align__(16) float ys[NB][LDY];   // solved rows of block p
  __shared__ __align__(16) float us[NB][kLd];   // W of block p, then us[r][i] = U[q+i][p+r]
  const int tq = (tid / CG) * RPT, tc = (tid % CG) * 4;
  for (int p = (nb - 1) * NB; p >= 0; p -= NB) {
    // the previous block's reads of ys and us are done and its updates of R visible
    __syncthreads();
    load_winv<256, false>(G, a.ldg, p, us);  // us[j][i] = W[j][i]
    for (int idx = tid; idx < NB * CG; idx += 256) {
      const int r = idx / CG, c = (idx % CG) * 4;
      *reinterpret_cast<float4*>(&yin[r][c]) =
          *reinterpret_cast<const float4*>(R + (size_t)(p + r) * a.d + c0 + c);
    }
    __syncthreads();
    {  // X[p][i][c] = sum_j W[j][i] Y[p][j][c]
      float acc[RPT][4] = {};
#pragma unroll 8
      for (int j = 0; j < NB; ++j) {
        const float4 b4 = *reinterpret_cast<const float4*>(&yin[j][tc]);
        const float bv[4] = {b4.x, b4.y, b4.z, b4.w};
        float av[RPT];
#pragma unroll
        for (int u = 0; u < RPT; ++u) av[u] = us[j][tq + u];
#pragma unroll
        for (int u = 0; u < RPT; ++u)
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
      }
#pragma unroll
      for (int u = 0; u < RPT; ++u) {
        const float4 x4 = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
        *reinterpret_cast<float4*>(&ys[tq + u][tc]) = x4;
        if (p + tq + u < a.k)
          *reinterpret_cast<float4*>(X + (size_t)(p + tq + u) * a.d + c0 + tc) = x4;
      }
    }
    __syncthreads();  // ys is complete and us free for the U blocks
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
    potrf_kernel<<<dim3(1, B), 2 * NB, 0, s>>>(a, p);
    panel_kernel<<<dim3(rest + dcb, B), 256, 0, s>>>(a, p, rest);
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
