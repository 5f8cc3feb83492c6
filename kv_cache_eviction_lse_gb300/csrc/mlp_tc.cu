// KVzap-MLP surrogate on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Per layer a two-layer MLP maps each hidden state h_t (D_h) to one predicted log-score
// per KV head: z_t = W2 GELU(W1 h_t + b1) + b2, hidden width D_mid = D_h / 8
// [KVzap review, 3.3 KVzap and the training setup table; the activation is a reading:
// exact (erf) GELU].  The first layer is the GEMM [T x D_h] x [D_h x D_mid]
// (D_h^2 / 4 flop per token); everything after it is fused into the GEMM's epilogue.
//
// Work item = (layer, 128-token tile, column part).  D_mid is split into P parts of
// N <= 256 columns so that two 256-column fp32 accumulators fit in TMEM and the
// epilogue of one item overlaps the MMAs of the next.  The CTAs of a persistent grid
// (one per SM, grid a multiple of P) take items round-robin, so the P CTAs that share
// a token tile run side by side and its h rows are read from HBM once (the other
// reads hit L2).
//   warp 0      TMA producer: per 64-wide k-block one A box (128 tokens x 64) and one
//               B box (N rows of W1 x 64) into a STAGES-deep ring (128-byte swizzle)
//   warp 1      owns TMEM (512 columns = two accumulators), issues the K-loop of
//               128 x N x 16 MMAs (bf16 x bf16 -> fp32) of an item into one of them
//   warps 2-9   epilogue, two groups of four warps (one per TMEM lane quarter), each
//               group half of the item's N columns: u = acc + b1, g = GELU(u),
//               partial z_h += g W2[h][c]; the two groups' partials meet in shared
//               memory and one fp32 atomic add per (token, head) adds the part's sum
//               (plus b2 for part 0) into z, which the launcher zeroes first.  With P
//               = 2 the result does not depend on the order of the two adds.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

#include "mlp.cuh"
#include "tc.cuh"

namespace kvs {

__device__ int g_mlp_error = 0;

namespace {

constexpr int BM = 128;  // tokens per item = TMEM lanes
constexpr int BK = 64;   // k-block: one 128-byte swizzle span of bf16
constexpr int kMaxN = 256;
constexpr int kGroupThreads = 128;
constexpr int kEpiThreads = 2 * kGroupThreads;
constexpr int kThreads = 64 + kEpiThreads;
constexpr uint32_t kBoxA = BM * 128;      // 16 KB
constexpr uint32_t kBoxBMax = kMaxN * 128;  // 32 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kMaxSmem = 232448;
constexpr int kStages = 4;
constexpr int kErrWaitTimeout = 1;
constexpr int kErrSmemAlign = 3;

template <int H>
struct MCfg {
  static constexpr uint32_t OFF_B = kStages * kBoxA;
  static constexpr uint32_t OFF_W = OFF_B + kStages * kBoxBMax;  // W2 slice [N][H] fp32
  static constexpr uint32_t OFF_B1 = OFF_W + kMaxN * H * 4;      // b1 slice [N] fp32
  static constexpr uint32_t OFF_Z = OFF_B1 + kMaxN * 4;          // group-1 partials [H][BM]
  static constexpr uint32_t OFF_BAR = OFF_Z + H * BM * 4;
  static constexpr uint32_t NBAR = 2 * kStages + 4;  // full[S], empty[S], tfull[2], tempty[2]
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM = (USED + 1024 <= kMaxSmem) ? USED + 1024 : kMaxSmem;
  static_assert(USED <= kMaxSmem, "shared-memory plan exceeds the per-block limit");
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, int code) {
  *abort_flag = 1u;
  atomicCAS(&g_mlp_error, 0, code);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// GELU(u) = u Phi(u) = u (1 + erf(u / sqrt 2)) / 2.
__device__ __forceinline__ float gelu(float u) {
  return 0.5f * u * (1.0f + erff(u * 0.70710678118654752f));
}

// 16 accumulator columns starting at column c0 of this group's part: z_h += GELU(acc +
// b1[c]) * W2[h][c].
template <int H>
__device__ __forceinline__ void mlp_cols(const uint32_t* v, const float* b1s, const float* ws,
                                         int c0, float* z) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int c = c0 + j;
    const float g = gelu(__uint_as_float(v[j]) + b1s[c]);
    const float* wc = ws + c * H;
#pragma unroll
    for (int hh = 0; hh < H; ++hh) z[hh] = fmaf(g, wc[hh], z[hh]);
  }
}

struct Item {
  int l, tile, part;
};

__device__ __forceinline__ Item item_of(int i, int P, int ntile) {
  Item it;
  it.part = i % P;
  const int lt = i / P;
  it.l = lt / ntile;
  it.tile = lt % ntile;
  return it;
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
    mlp_tc_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w1,
                  const MlpArgs a, int P, int N) {
  using C = MCfg<H>;
  constexpr int S = kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + C::USED > C::SMEM) {  // uniform; never overflow the allocation
    if (threadIdx.x == 0) atomicCAS(&g_mlp_error, 0, kErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sA = sb, sB = sb + C::OFF_B;
  float* wsm = reinterpret_cast<float*>(smem + C::OFF_W);
  float* b1sm = reinterpret_cast<float*>(smem + C::OFF_B1);
  float* zx = reinterpret_cast<float*>(smem + C::OFF_Z);
  const uint32_t bar0 = sb + C::OFF_BAR;
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto bar_tfull = [&](int x) { return bar0 + 8u * (2 * S + x); };
  auto bar_tempty = [&](int x) { return bar0 + 8u * (2 * S + 2 + x); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = a.Dh / BK;
  const int ntile = (a.T + BM - 1) / BM;
  const int nitems = a.L * ntile * P;
  const uint32_t b_bytes = (uint32_t)N * 128u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(bar_full(s), 1);
      tc::mbar_init(bar_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(bar_tfull(x), 1);
      tc::mbar_init(bar_tempty(x), kEpiThreads);
    }
    misc[1] = 0u;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sb + C::OFF_MISC, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_h);
    tc::tma_prefetch_desc(&tm_w1);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < nitems && ok; i += gridDim.x) {
        const Item it = item_of(i, P, ntile);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = g % S;
          const uint32_t ph = (uint32_t)(g / S) & 1u;
          if (!tc::mbar_wait(bar_empty(s), ph ^ 1u) || *abort_flag) {
            ok = false;
            break;
          }
          tc::mbar_expect_tx(bar_full(s), kBoxA + b_bytes);
          tc::tma_load_3d(sA + s * kBoxA, &tm_h, bar_full(s), kb * BK, it.tile * BM, it.l);
          tc::tma_load_3d(sB + s * kBoxBMax, &tm_w1, bar_full(s), kb * BK, it.part * N, it.l);
        }
      }
      if (!ok) {
        fail(abort_flag, kErrWaitTimeout);
        // let the copies already in flight land before the CTA exits
        for (int j = max(0, g - S); j < g; ++j) tc::mbar_wait(bar_full(j % S), (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(BM, N);
      int g = 0, n = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < nitems && ok; i += gridDim.x, ++n) {
        const int acc = n & 1;
        const uint32_t aph = (uint32_t)(n >> 1) & 1u;
        if (!tc::mbar_wait(bar_tempty(acc), aph ^ 1u) || *abort_flag) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d_t = tmem + (uint32_t)(acc * kMaxN);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          const int s = g % S;
          const uint32_t ph = (uint32_t)(g / S) & 1u;
          if (!tc::mbar_wait(bar_full(s), ph) || *abort_flag) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a_s = sA + s * kBoxA, b_s = sB + s * kBoxBMax;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            tc::mma_bf16(d_t, tc::sdesc_sw128(a_s + 32u * k), tc::sdesc_sw128(b_s + 32u * k),
                         idesc, (kb | k) != 0 ? 1u : 0u);
          tc::commit(bar_empty(s));
        }
        if (!ok) break;
        tc::commit(bar_tfull(acc));
      }
      if (!ok) fail(abort_flag, kErrWaitTimeout);
      if (g > 0) tc::mbar_wait(bar_empty((g - 1) % S), ((g - 1) / S) & 1);
    }
    __syncwarp();
  } else {
    // ============================================================ epilogue
    const int grp = (warp - 2) >> 2;  // half of the item's N columns
    const int eq = warp & 3;          // TMEM lane quarter this warp may access
    const int row = eq * 32 + lane;   // token within the tile
    const int et = threadIdx.x - 64;  // 0..255
    const int ncol = N / 2;           // columns of this group, a multiple of 16
    const int c_begin = grp * ncol;
    bool failed = false;
    int n = 0;
    for (int i = blockIdx.x; i < nitems; i += gridDim.x, ++n) {
      const Item it = item_of(i, P, ntile);
      // this item's slices of b1 and W2 (fp32) into shared memory; the barrier in front
      // also orders the previous item's reads of wsm, b1sm and zx before these writes
      named_sync(1, kEpiThreads);
      const int col0 = it.part * N;
      for (int idx = et; idx < N * H; idx += kEpiThreads) {
        const int c = idx / H, hh = idx - c * H;
        const uint16_t wb = a.W2[((size_t)it.l * H + hh) * a.Dm + col0 + c];
        wsm[idx] = __uint_as_float((uint32_t)wb << 16);
      }
      for (int c = et; c < N; c += kEpiThreads) b1sm[c] = a.b1[(size_t)it.l * a.Dm + col0 + c];
      named_sync(1, kEpiThreads);

      const int acc = n & 1;
      const uint32_t aph = (uint32_t)(n >> 1) & 1u;
      const bool ok = tc::mbar_wait(bar_tfull(acc), aph) && !*abort_flag;
      if (tc::bar_or(2, kEpiThreads, !ok)) {
        failed = true;
        break;
      }
      tc::fence_after_sync();
      float z[H];
#pragma unroll
      for (int hh = 0; hh < H; ++hh) z[hh] = 0.f;
      const uint32_t t_base =
          tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(acc * kMaxN + c_begin);
      const int nch = ncol / 16;
      uint32_t v0[16], v1[16];
      tc::tmem_ld16(t_base, v0);
      tc::tmem_ld_wait();
      tc::reg_fence16(v0);
      for (int cb = 0; cb < nch; cb += 2) {
        if (cb + 1 < nch) tc::tmem_ld16(t_base + 16u * (cb + 1), v1);
        mlp_cols<H>(v0, b1sm, wsm, c_begin + 16 * cb, z);
        tc::tmem_ld_wait();
        tc::reg_fence16(v1);
        if (cb + 1 < nch) {
          if (cb + 2 < nch) tc::tmem_ld16(t_base + 16u * (cb + 2), v0);
          mlp_cols<H>(v1, b1sm, wsm, c_begin + 16 * (cb + 1), z);
          tc::tmem_ld_wait();
          tc::reg_fence16(v0);
        }
      }
      // every column of this accumulator has been read
      tc::fence_before_sync();
      tc::mbar_arrive(bar_tempty(acc));

      if (grp == 1) {
#pragma unroll
        for (int hh = 0; hh < H; ++hh) zx[hh * BM + row] = z[hh];
      }
      named_sync(3, kEpiThreads);
      if (grp == 0) {
        const int t = it.tile * BM + row;
        if (t < a.T) {
#pragma unroll
          for (int hh = 0; hh < H; ++hh) {
            float zz = z[hh] + zx[hh * BM + row];
            if (it.part == 0) zz += a.b2[it.l * H + hh];
            atomicAdd(a.z + ((size_t)it.l * H + hh) * a.T + t, zz);
          }
        }
      }
    }
    if (failed) atomicCAS(&g_mlp_error, 0, (int)kErrWaitTimeout);
  }

  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

int sm_count() {
  static int n[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev];
}

template <int H>
cudaError_t launch_h(const MlpArgs& a, cudaStream_t s) {
  using C = MCfg<H>;
  const int P = mlp_parts(a.Dm);
  const int N = a.Dm / P;
  CUtensorMap th, tw;
  cudaError_t e = tma_map_bf16_3d(&th, a.h, a.Dh, a.T, a.L, BM);
  if (e == cudaSuccess) e = tma_map_bf16_3d(&tw, a.W1, a.Dh, a.Dm, a.L, N);
  if (e != cudaSuccess) return e;
  const int nitems = a.L * ((a.T + BM - 1) / BM) * P;
  const int nsm = sm_count();
  if (nsm <= 0) return cudaErrorInvalidDevice;
  const int grid = std::min(nitems, std::max(P, nsm / P * P));
  auto kern = mlp_tc_kernel<H>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  count_launches(1);
  kern<<<grid, kThreads, C::SMEM, s>>>(th, tw, a, P, N);
  return cudaGetLastError();
}

}  // namespace

int mlp_parts(int Dm) {
  if (Dm <= 0 || Dm % 32) return 0;
  for (int P = (Dm + kMaxN - 1) / kMaxN; P <= Dm / 32; ++P)
    if (Dm % P == 0 && (Dm / P) % 32 == 0) return P;
  return 0;
}

bool mlp_supported(int Dh, int Dm, int H) {
  return Dh > 0 && Dh % BK == 0 && mlp_parts(Dm) > 0 &&
         (H == 1 || H == 2 || H == 4 || H == 8 || H == 16);
}

cudaError_t launch_mlp_surrogate(const MlpArgs& a, cudaStream_t s) {
  if (!mlp_supported(a.Dh, a.Dm, a.H)) return cudaErrorInvalidValue;
  if (a.T == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(a.z, 0, (size_t)a.L * a.H * a.T * sizeof(float), s);
  if (e != cudaSuccess) return e;
  switch (a.H) {
    case 1: return launch_h<1>(a, s);
    case 2: return launch_h<2>(a, s);
    case 4: return launch_h<4>(a, s);
    case 8: return launch_h<8>(a, s);
    default: return launch_h<16>(a, s);
  }
}

cudaError_t mlp_device_error(int* code, bool clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_mlp_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && *code) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_mlp_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace kvs
