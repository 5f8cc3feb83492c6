// Products X^T Y on the tensor cores (tcgen05 + TMEM + TMA), fp32 accumulation:
//   gram_tc_kernel         the value norms' Gram pairs: the diagonal d x d blocks of
//                          o_proj^T o_proj (bf16 operands), written as bf16 hi/lo pairs
//   refit_products_kernel  the value refit's normal equations A_S^T A_S and A_S^T O
//                          (fp16 operands), below
//
// Both operands are read MN-major straight from their row-major [rows][cols] storage:
// a TMA box of 64 rows x 64 columns is one 128-byte-swizzled MN-major atom column, so
// a 128-column tile is two boxes (leading byte offset 8 KB) and each MMA takes 16 rows.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "gram.cuh"
#include "tc.cuh"

namespace kvs {

__device__ int g_gram_error = 0;

namespace {

constexpr int BT = 128;                 // output tile edge
constexpr int BK = 64;                  // rows per k-block
constexpr uint32_t kBox = 64 * 128;     // 64 rows x 64 bf16 = 8 KB
constexpr uint32_t kOp = 2 * kBox;      // one 128-column operand tile of a k-block
// The value-norm Gram streams one operand (16 KB per k-block) straight from HBM; a
// 4-stage ring lets three CTAs share an SM, so all (layer, head) tiles of a call run at
// once and the heads of a layer walk the rows of o_proj.weight together.
constexpr int kStages = 4;
constexpr uint32_t kRingDiag = kStages * kOp;
constexpr int kMaxStages = 12;          // barrier slots (the refit products use 3)
constexpr int kThreads = 64 + 128;
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t OFF_BAR = 0;  // barriers and the TMEM address first, the ring after
constexpr uint32_t NBAR = 2 * kMaxStages + 1;  // full[S], empty[S], done
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
constexpr uint32_t OFF_RING = 1024;
static_assert(OFF_MISC + 16 <= OFF_RING, "barrier block");
constexpr uint32_t kDiagSmem = OFF_RING + kRingDiag + 1024;
constexpr int kErrWaitTimeout = 1;
constexpr int kErrSmemAlign = 3;

// One CTA per 128 x 128 diagonal tile of X^T X (X = o_proj.weight [D_h][H_q d], tile tm
// covers the 128 / d heads whose slices it holds): warp 0 streams 64-row k-blocks through
// the ring, warp 1 issues the MMAs (X^T against itself) into one TMEM accumulator, warps
// 2-5 write each head's d x d block as bf16 hi and lo parts.
__global__ void __launch_bounds__(kThreads, 1)
    gram_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const GramArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + OFF_RING + kRingDiag > kDiagSmem) {
    if (threadIdx.x == 0) atomicCAS(&g_gram_error, 0, kErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t bar0 = sb + OFF_BAR;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  const uint32_t bar_done = bar0 + 8u * (2 * kMaxStages);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + OFF_MISC);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tm = blockIdx.x, b = blockIdx.y;
  const int nkb = (a.rows + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(bar_full(s), 1);
      tc::mbar_init(bar_empty(s), 1);
    }
    tc::mbar_init(bar_done, 1);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sb + OFF_MISC, kTmemCols);
    tc::tmem_relinquish();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    if (lane == 0) {
      int kb = 0;
      bool ok = true;
      for (; kb < nkb; ++kb) {
        const int s = kb % kStages;
        if (!tc::mbar_wait(bar_empty(s), ((kb / kStages) & 1) ^ 1u)) {
          ok = false;
          break;
        }
        const uint32_t st = sb + OFF_RING + s * kOp;
        tc::mbar_expect_tx(bar_full(s), kOp);
        for (int c = 0; c < 2; ++c)  // two 64-column boxes
          tc::tma_load_3d(st + c * kBox, &tm_x, bar_full(s), tm * BT + 64 * c, kb * BK, b);
      }
      if (!ok) {
        atomicCAS(&g_gram_error, 0, kErrWaitTimeout);
        for (int j = max(0, kb - kStages); j < kb; ++j)
          tc::mbar_wait(bar_full(j % kStages), (j / kStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_bmn(BT, BT) | (1u << 15);  // A and B MN-major
      int kb = 0;
      bool ok = true;
      for (; kb < nkb; ++kb) {
        const int s = kb % kStages;
        if (!tc::mbar_wait(bar_full(s), (kb / kStages) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t st = sb + OFF_RING + s * kOp;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint64_t xd = tc::sdesc_sw128_mn(st + 2048u * k, kBox);  // 16 rows of 128 B
          tc::mma_bf16(tmem, xd, xd, idesc, (kb | k) != 0 ? 1u : 0u);
        }
        tc::commit(bar_empty(s));
      }
      if (!ok) atomicCAS(&g_gram_error, 0, kErrWaitTimeout);
      tc::commit(bar_done);  // lands once every MMA above has completed
      tc::mbar_wait(bar_done, 0);
    }
    __syncwarp();
  } else {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) ..; row ml of the tile per thread
    // belongs to slice (head) r = ml / d; write that slice's row of its d x d Gram block
    // as bf16 hi and lo parts
    const int eq = warp & 3;
    const bool ok = tc::mbar_wait(bar_done, 0);
    if (!ok) atomicCAS(&g_gram_error, 0, kErrWaitTimeout);
    tc::fence_after_sync();
    const int dd = a.pair_d, ml = eq * 32 + lane, r = ml / dd, i = ml % dd;
    const int head = (tm * BT) / dd + r, nheads = a.M / dd;
    bf16_t* gh = a.pair + (((size_t)b * nheads + head) * 2 * dd + i) * dd;
#pragma unroll
    for (int cb = 0; cb < BT / 32; ++cb) {
      uint32_t v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(eq * 32) << 16) + 32u * cb, v);
      tc::tmem_ld_wait();
      const int c0 = 32 * cb - r * dd;  // column within the slice
      if (ok && head < nheads && c0 >= 0 && c0 < dd) {
#pragma unroll
        for (int c = 0; c < 32; c += 8) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float x0 = __uint_as_float(v[c + 2 * e]), x1 = __uint_as_float(v[c + 2 * e + 1]);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
            hi[e] = *reinterpret_cast<uint32_t*>(&h2);
            __nv_bfloat162 l2 = __floats2bfloat162_rn(x0 - __low2float(h2), x1 - __high2float(h2));
            lo[e] = *reinterpret_cast<uint32_t*>(&l2);
          }
          *reinterpret_cast<uint4*>(gh + c0 + c) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          *reinterpret_cast<uint4*>(gh + (size_t)dd * dd + c0 + c) =
              make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ refit products
//
// The value refit's normal equations in one launch, on single-part fp16 operands:
//   G = A_S^T A_S  (upper block triangle of 256 x 256 blocks)   and   R = A_S^T O
// One CTA per 256 x WN output block (WN = 256 for G, 128 for R, so R's blocks carry no
// empty columns), its two 128-row halves in two TMEM accumulators of WN columns.  Per
// 64-row k-block the CTA loads 64 x 256 of A_S and 64 x WN of A_S or O and issues 2 x 4
// MMAs of 128 x WN x 16: a byte of operand feeds twice the flops of a 128 x 128 tile
// (these products stream their operands from L2, and that is what bounds them), and the
// G and R blocks share one wave of CTAs.
constexpr int WM = 256;                    // output rows per CTA (two MMA halves)
constexpr int kWideThreads = 64 + 256;     // producer, MMA issuer, 8 epilogue warps
constexpr int kWideStages = 3;             // 64 KB per stage (X and Y tiles)
constexpr uint32_t kWideStage = 8 * kBox;  // X: 4 boxes, Y: up to 4 boxes
constexpr uint32_t kWideSmem = OFF_RING + kWideStages * kWideStage + 1024;
constexpr uint32_t kWideCols = 512;        // TMEM: two accumulators of up to 256 columns
static_assert(kWideSmem <= 232448, "shared-memory plan exceeds the per-block limit");

__global__ void __launch_bounds__(kWideThreads, 1)
    refit_products_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_o,
                          const RefitProdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + OFF_RING + kWideStages * kWideStage > kWideSmem) {
    if (threadIdx.x == 0) atomicCAS(&g_gram_error, 0, kErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t bar0 = sb + OFF_BAR;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
  const uint32_t bar_done = bar0 + 8u * (2 * kMaxStages);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  constexpr uint32_t kY = 4 * kBox;  // Y tile offset within a stage

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // blocks [0, n_up): G's upper block triangle; the next nt blocks: R's row blocks
  const int nt = (a.k_ld + WM - 1) / WM, n_up = nt * (nt + 1) / 2;
  const bool rhs = (int)blockIdx.x >= n_up;
  int tm, tn = 0;
  if (rhs) {
    tm = (int)blockIdx.x - n_up;
  } else {
    int t = blockIdx.x, row = 0;
    while (t >= nt - row) {
      t -= nt - row;
      ++row;
    }
    tm = row;
    tn = row + t;
  }
  const int wn = rhs ? 128 : 256;
  const int b = blockIdx.y;
  const int nkb = (a.rows + BK - 1) / BK;
  // Only the block's rows and columns inside k_ld (d for R) are computed: a second
  // 128-row half made only of padding is skipped, N follows the valid columns (rounded
  // up to the MMA's multiple of 16), and the second half of a diagonal block of G, whose
  // first 128 columns lie below the diagonal (never read), covers only the rest.
  const int m_valid = min(WM, a.k_ld - tm * WM);
  const int n_valid = min(wn, (rhs ? a.d : a.k_ld) - tn * wn);
  const int n_mma = (n_valid + 15) & ~15;
  const bool half1 = m_valid > 128;
  const bool diag = !rhs && tm == tn;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWideStages; ++s) {
      tc::mbar_init(bar_full(s), 1);
      tc::mbar_init(bar_empty(s), 1);
    }
    tc::mbar_init(bar_done, 1);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sb + OFF_MISC, kWideCols);
    tc::tmem_relinquish();
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    if (lane == 0) {
      // boxes loaded; a diagonal block of G multiplies A_S's column block by itself, so
      // its Y operand is the X tile
      const int nxb = (m_valid + 63) / 64, nyb = diag ? 0 : (n_valid + 63) / 64;
      const uint32_t bytes = (uint32_t)(nxb + nyb) * kBox;
      const CUtensorMap* ym = rhs ? &tm_o : &tm_a;
      int kb = 0;
      bool ok = true;
      for (; kb < nkb; ++kb) {
        const int s = kb % kWideStages;
        if (!tc::mbar_wait(bar_empty(s), ((kb / kWideStages) & 1) ^ 1u)) {
          ok = false;
          break;
        }
        const uint32_t st = sb + OFF_RING + s * kWideStage;
        tc::mbar_expect_tx(bar_full(s), bytes);
        for (int c = 0; c < nxb; ++c)  // X: A_S columns tm*256 .., 64-column boxes
          tc::tma_load_3d(st + c * kBox, &tm_a, bar_full(s), tm * WM + 64 * c, kb * BK, b);
        for (int c = 0; c < nyb; ++c)
          tc::tma_load_3d(st + kY + c * kBox, ym, bar_full(s), tn * wn + 64 * c, kb * BK, b);
      }
      if (!ok) {
        atomicCAS(&g_gram_error, 0, kErrWaitTimeout);
        for (int j = max(0, kb - kWideStages); j < kb; ++j)
          tc::mbar_wait(bar_full(j % kWideStages), (j / kWideStages) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // A and B MN-major, fp16 (format fields 0); N = n_mma, or the columns from 128 on
      // for the second half of a diagonal block.  The boxes a trimmed MMA reads past the
      // loaded ones hold stale data that reaches only discarded rows and columns.
      auto idesc_n = [](int n) {
        return (tc::idesc_bf16_bmn(128, n) | (1u << 15)) & ~((1u << 7) | (1u << 10));
      };
      const uint32_t idesc0 = idesc_n(n_mma);
      const int n1 = diag ? n_mma - 128 : n_mma;  // > 0 whenever half1
      const uint32_t idesc1 = idesc_n(n1 > 0 ? n1 : 16);
      const uint32_t c1 = diag ? 128u : 0u;       // first column of the second half
      const uint32_t y_off = diag ? 0u : kY;       // the Y tile within a stage
      int kb = 0;
      bool ok = true;
      for (; kb < nkb; ++kb) {
        const int s = kb % kWideStages;
        if (!tc::mbar_wait(bar_full(s), (kb / kWideStages) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t st = sb + OFF_RING + s * kWideStage;
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {
          const uint32_t o = 2048u * k;  // 16 rows of 128 bytes
          const uint32_t acc = (kb | k) != 0 ? 1u : 0u;
          tc::mma_bf16(tmem, tc::sdesc_sw128_mn(st + o, kBox),
                       tc::sdesc_sw128_mn(st + y_off + o, kBox), idesc0, acc);
          if (half1)
            tc::mma_bf16(tmem + (uint32_t)wn + c1, tc::sdesc_sw128_mn(st + 2 * kBox + o, kBox),
                         tc::sdesc_sw128_mn(st + y_off + (c1 / 64) * kBox + o, kBox), idesc1,
                         acc);
        }
        tc::commit(bar_empty(s));
      }
      if (!ok) atomicCAS(&g_gram_error, 0, kErrWaitTimeout);
      tc::commit(bar_done);
      tc::mbar_wait(bar_done, 0);
    }
    __syncwarp();
  } else {
    // epilogue: warp w reads TMEM lanes 32 (w % 4) .. of accumulator hh = (w - 2) / 4
    const int eq = warp & 3, hh = (warp - 2) >> 2;
    const int m = tm * WM + hh * 128 + eq * 32 + lane;
    const bool ok = tc::mbar_wait(bar_done, 0);
    if (!ok) atomicCAS(&g_gram_error, 0, kErrWaitTimeout);
    tc::fence_after_sync();
    const int N = rhs ? a.d : a.k_ld, ldc = rhs ? a.d : a.k_ld;
    float* crow = (rhs ? a.r : a.g) + ((size_t)b * a.k_ld + m) * ldc + tn * wn;
    const int nmax = min(wn, N - tn * wn);
    const uint32_t t0 = tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(hh * wn);
    // the columns this half computed: none for a skipped half, from 128 on for the
    // second half of a diagonal block
    const int cb0 = hh == 1 ? (half1 ? (diag ? 4 : 0) : wn / 32) : 0;
#pragma unroll 1
    for (int cb = cb0; cb < (nmax + 31) / 32; ++cb) {
      uint32_t v[32];
      tc::tmem_ld32(t0 + 32u * cb, v);
      tc::tmem_ld_wait();
      if (ok && m < a.k_ld) {
        if (32 * cb + 32 <= nmax) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(crow + 32 * cb + c) =
                make_float4(__uint_as_float(v[c]), __uint_as_float(v[c + 1]),
                            __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
        } else {
          for (int c = 0; c < 32 && 32 * cb + c < nmax; ++c) crow[32 * cb + c] = __uint_as_float(v[c]);
        }
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kWideCols);
  }
}

}  // namespace

cudaError_t launch_gram(const GramArgs& a, cudaStream_t s) {
  if (a.M <= 0 || a.batch <= 0) return cudaSuccess;
  if (!a.x || !a.pair || a.pair_d <= 0 || BT % a.pair_d || a.M % a.pair_d || a.pair_d % 8 ||
      a.ldx % 8)
    return cudaErrorInvalidValue;
  CUtensorMap x;
  cudaError_t e = tma_map_bf16_3d(&x, a.x, a.ldx, a.rows, a.batch, BK);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gram_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kDiagSmem);
  if (e != cudaSuccess) return e;
  count_launches(1);
  gram_tc_kernel<<<dim3((a.M + BT - 1) / BT, a.batch), kThreads, kDiagSmem, s>>>(x, a);
  return cudaGetLastError();
}

cudaError_t launch_refit_products(const RefitProdArgs& a, cudaStream_t s) {
  if (a.batch <= 0 || a.k_ld <= 0 || a.rows <= 0) return cudaSuccess;
  if (a.k_ld % 64 || a.d % 8 || a.d > 128) return cudaErrorInvalidValue;
  CUtensorMap ma, mo;
  cudaError_t e = tma_map_bf16_3d(&ma, a.a_s, a.k_ld, a.rows, a.batch, BK);
  if (e == cudaSuccess) e = tma_map_bf16_3d(&mo, a.o, a.d, a.rows, a.batch, BK);
  if (e != cudaSuccess) return e;
  const int nt = (a.k_ld + WM - 1) / WM;
  e = cudaFuncSetAttribute(refit_products_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kWideSmem);
  if (e != cudaSuccess) return e;
  count_launches(1);
  refit_products_kernel<<<dim3(nt * (nt + 1) / 2 + nt, a.batch), kWideThreads, kWideSmem, s>>>(
      ma, mo, a);
  return cudaGetLastError();
}

cudaError_t gram_device_error(int* code, bool clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_gram_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && *code) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_gram_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace kvs
