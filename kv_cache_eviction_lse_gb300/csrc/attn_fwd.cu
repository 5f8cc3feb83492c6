// Attention forward that returns its LSE normaliser, on the 5th-generation tensor cores.
//
// For every query head h and query j (bottom-right causal over the concatenated
// [context | tail] keys of the head's KV head):
//   o^h_j = sum_i a_ji v_i,   a_ji = exp(q_j.k_i / sqrt d - LSE_j)
// [KVzap review 3.2, Eq. 2: the head output that W_O maps into the residual stream]
// together with LSE_j, the normaliser the transposed scoring pass reuses [KVpop review,
// 1. Key Terms], so that pruning pays only for pass 2 when the attention runs anyway.
//
// A persistent grid (one CTA per SM) works through units of 128 queries of one head;
// keys in tiles of 128 (online softmax):
//   warp 0      TMA: K and V tiles through two 2-stage rings
//   warp 1      owns TMEM (two S buffers: 2 x 128 columns; P: 64; Q: d/2; O: d) and
//               issues S(j) = Q K(j)^T with Q read from TMEM as the A operand, then
//               O += P(j-1) V(j-1) with P read from TMEM as the A operand and V as an
//               MN-major operand straight from its TMA box: shared memory feeds only
//               the B operand of either product (half of what a shared-memory A would
//               add to the QK^T product, whose N = 128 tile would otherwise need the
//               whole shared-memory bandwidth)
//   warps 2-9   first copy the CTA's query rows into TMEM (two threads per row, 16-byte
//               loads, tcgen05.st), then the softmax, two threads per query row (one per
//               64-key half): read S with tcgen05.ld and release its buffer at once, agree
//               on the row max through shared memory, p = 2^(x - m) with one ex2 each,
//               store P as bf16 pairs into the P columns (tcgen05.st) once the previous
//               P V product has read them, and rescale O in TMEM when the running max
//               grows by more than 2^8 (otherwise the stale max is kept: p <= 256 stays
//               exact enough in bf16 and the final normalisation uses the same max)
// S(j + 1) only waits for the softmax to have read S(j - 1), so the tensor pipe runs
// S(j + 1) while the softmax of tile j works; P V(j) waits for P(j).  TMEM, barriers and
// rings carry over between units: the next unit's K/V tiles load during this unit's last
// ones, and its query rows are read into registers before this unit's O is finished.
// The epilogue divides O by the row sum, writes it as bf16 and writes the LSE.
#include <algorithm>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "attn.cuh"
#include "tc.cuh"

namespace kvs {

__device__ int g_fwd_error = 0;

namespace {

constexpr int BM = 128;  // queries per CTA = TMEM lanes
constexpr int BN = 128;  // keys per tile
constexpr int NQ = 2;          // softmax threads per query row, each on BN / NQ keys
constexpr int KC = BN / NQ;    // keys per softmax thread and tile
constexpr int kSoftThreads = NQ * 128;
constexpr int kThreads = 64 + kSoftThreads;
constexpr uint32_t kBox = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr uint32_t kTmemCols = 512;
constexpr int NSB = 2;  // S buffers in TMEM
constexpr uint32_t kMaxSmem = 232448;
constexpr int kErrWaitTimeout = 1;
constexpr int kErrSmemAlign = 3;
constexpr float kRescale = 8.f;  // log2 growth of the row max that forces a rescale of O

template <int D>
struct FCfg {
  static constexpr int KH = D / 64;
  static constexpr uint32_t TILE = KH * kBox;  // one K or V tile
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + 2 * TILE;
  // separate K and V rings: K(j) is released as soon as S(j) = Q K(j)^T is done, so the
  // load of K(j+2) overlaps the softmax and P V of tile j; V(j) is held until P V(j)
  static constexpr uint32_t OFF_XM = OFF_V + 2 * TILE;     // row max exchange [2][NQ][BM]
  static constexpr uint32_t OFF_XL = OFF_XM + 2 * NQ * BM * 4;  // row sum exchange [NQ][BM]
  static constexpr uint32_t OFF_BAR = OFF_XL + NQ * BM * 4;
  // q, k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], s_empty[2], p[2], o[2], done
  static constexpr uint32_t NBAR = 18;
  // TMEM columns: S buffers, then P (bf16 pairs of one tile), Q (bf16 pairs), O
  static constexpr uint32_t COL_P = NSB * BN;
  static constexpr uint32_t COL_Q = COL_P + BN / 2;
  static constexpr uint32_t COL_O = COL_Q + D / 2;
  static_assert(COL_O + D <= kTmemCols, "TMEM plan");
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM = (USED + 1024 <= kMaxSmem) ? USED + 1024 : kMaxSmem;
  static_assert(USED <= kMaxSmem, "shared-memory plan exceeds the per-block limit");
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, int code) {
  *abort_flag = 1u;
  atomicCAS(&g_fwd_error, 0, code);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// One unit of the persistent grid: 128 queries of one (layer, query head).  A CTA's
// units visit one residue class of query tiles modulo dg = gcd(grid, tiles per head);
// a causal unit's cost grows with its query tile, so odd groups of dg tiles are taken in
// reverse order, giving every residue class the same mean cost.
struct FwdUnit {
  int l, hq, hk, row0, n_ctx, ntiles;
};

__device__ __forceinline__ FwdUnit fwd_unit(const FwdArgs& a, int u, int nqt, int dg, int G,
                                            int off) {
  FwdUnit f;
  const int r = u % nqt, k = r / dg, sr = r - k * dg;
  f.row0 = (k * dg + ((k & 1) ? dg - 1 - sr : sr)) * BM;
  f.hq = (u / nqt) % a.Hq;
  f.l = u / (nqt * a.Hq);
  f.hk = f.hq / G;
  // key tiles the unit sees: context tiles, then tail tiles
  const int kv_end = off + min(f.row0 + BM, a.n_q);  // keys [0, kv_end) are visible to some query
  f.n_ctx = (min(a.T, kv_end) + BN - 1) / BN;
  f.ntiles = f.n_ctx + (min(a.n_tail, max(0, kv_end - a.T)) + BN - 1) / BN;
  return f;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kt,
                    const __grid_constant__ CUtensorMap tm_vt, const FwdArgs a) {
  using C = FCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + C::USED > C::SMEM) {
    if (threadIdx.x == 0) atomicCAS(&g_fwd_error, 0, kErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sK = sb + C::OFF_K, sV = sb + C::OFF_V;
  float* xm = reinterpret_cast<float*>(smem + C::OFF_XM);
  float* xl = reinterpret_cast<float*>(smem + C::OFF_XL);
  const uint32_t bar0 = sb + C::OFF_BAR;
  const uint32_t bar_q = bar0;  // the query rows are in TMEM (softmax threads arrive)
  auto bar_kfull = [&](int s) { return bar0 + 8u * (1 + s); };
  auto bar_kempty = [&](int s) { return bar0 + 8u * (3 + s); };
  auto bar_vfull = [&](int s) { return bar0 + 8u * (5 + s); };
  auto bar_vempty = [&](int s) { return bar0 + 8u * (7 + s); };
  auto bar_sfull = [&](int s) { return bar0 + 8u * (9 + s); };    // S buffer s = j & 1
  auto bar_sempty = [&](int s) { return bar0 + 8u * (11 + s); };  // the softmax read it
  // P(i) is ready on p[i & 1] and O += P(i) V(i) completes on o[i & 1]: the softmax waits
  // for P V(i - 1) before it writes P(i), so neither barrier can run two phases ahead of
  // a waiter and every parity wait is unambiguous
  auto bar_p = [&](int i) { return bar0 + 8u * (13 + (i & 1)); };
  auto bar_o = [&](int i) { return bar0 + 8u * (15 + (i & 1)); };
  const uint32_t bar_done = bar0 + 8u * 17;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int n_k = a.T + a.n_tail;
  const int off = a.causal ? n_k - a.n_q : n_k;  // non-causal: every key is visible
  // Persistent grid: this CTA takes units blockIdx.x, blockIdx.x + gridDim.x, ... of all
  // (layer, query head, 128-query tile), query tile fastest.  TMEM, the barriers and the
  // K/V rings carry over from unit to unit (their phases follow global tile counters).
  const int nqt = (a.n_q + BM - 1) / BM;
  const int total = nqt * a.Hq * a.L;
  const int nunits = (int)blockIdx.x < total ? (total - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  int dg = (int)gridDim.x;  // gcd(grid, nqt)
  for (int x = nqt; x > 0;) {
    const int t = dg % x;
    dg = x;
    x = t;
  }
  auto unit = [&](int n) {
    return fwd_unit(a, (int)blockIdx.x + n * (int)gridDim.x, nqt, dg, G, off);
  };

  if (threadIdx.x == 0) {
    tc::mbar_init(bar_q, kSoftThreads);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(bar_kfull(s), 1);
      tc::mbar_init(bar_kempty(s), 1);
      tc::mbar_init(bar_vfull(s), 1);
      tc::mbar_init(bar_vempty(s), 1);
      tc::mbar_init(bar_o(s), 1);
      tc::mbar_init(bar_p(s), kSoftThreads);
      tc::mbar_init(bar_sfull(s), 1);
      tc::mbar_init(bar_sempty(s), kSoftThreads);
    }
    tc::mbar_init(bar_done, 1);
    misc[1] = 0u;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sb + C::OFF_MISC, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_k);
    tc::tma_prefetch_desc(&tm_v);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];
  const uint32_t t_p = tmem + C::COL_P;  // P of the current tile: BN / 2 columns
  const uint32_t t_q = tmem + C::COL_Q;  // the query rows: D / 2 columns
  const uint32_t t_o = tmem + C::COL_O;  // O accumulator: D columns

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      // per unit, loads in the order the MMAs use them: K(0), K(1), V(0), K(2), V(1), ...;
      // the next unit's first tiles load while this unit's last ones are consumed
      int gk = 0, gv = 0;  // K and V tiles issued (all units)
      bool ok = true;
      for (int n = 0; n < nunits && ok; ++n) {
        const FwdUnit U = unit(n);
        const int head = U.l * a.Hkv + U.hk;
        auto load = [&](bool is_v, int j, int g) -> bool {  // tile j of the unit, g-th overall
          const int s = g & 1;
          const uint32_t empty = is_v ? bar_vempty(s) : bar_kempty(s);
          if (!tc::mbar_wait(empty, ((g >> 1) & 1) ^ 1u) || *abort_flag) return false;
          const bool ctx = j < U.n_ctx;
          const CUtensorMap* m = is_v ? (ctx ? &tm_v : &tm_vt) : (ctx ? &tm_k : &tm_kt);
          const int row = ctx ? j * BN : (j - U.n_ctx) * BN;
          const uint32_t full = is_v ? bar_vfull(s) : bar_kfull(s);
          const uint32_t dst = (is_v ? sV : sK) + s * C::TILE;
          tc::mbar_expect_tx(full, C::TILE);
#pragma unroll
          for (int kh = 0; kh < C::KH; ++kh) tc::tma_load_3d(dst + kh * kBox, m, full, kh * 64, row, head);
          return true;
        };
        for (int t = 0; ok && t <= U.ntiles; ++t) {
          if (t < U.ntiles) {
            ok = load(false, t, gk);
            if (ok) ++gk;
          }
          if (ok && t >= 1) {
            ok = load(true, t - 1, gv);
            if (ok) ++gv;
          }
        }
      }
      if (!ok) {
        fail(abort_flag, kErrWaitTimeout);
        // let the copies already in flight land before the CTA exits
        for (int i = max(0, gk - 2); i < gk; ++i) tc::mbar_wait(bar_kfull(i & 1), (i >> 1) & 1);
        for (int i = max(0, gv - 2); i < gv; ++i) tc::mbar_wait(bar_vfull(i & 1), (i >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16(BM, BN);
      constexpr uint32_t idesc_o = tc::idesc_bf16_bmn(BM, D);
      int gs = 0, gp = 0;  // S and P V products issued (all units)
      int issued = 0;      // MMA groups issued (for the final drain)
      bool ok = true;
      for (int n = 0; n < nunits && ok; ++n) {
        const int ntiles = unit(n).ntiles;
        // the unit's query rows are in TMEM, and the softmax threads have read the
        // previous unit's O (they arrive after both), so P V(0) may overwrite it
        if (!tc::mbar_wait(bar_q, (uint32_t)n & 1u) || *abort_flag) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        for (int j = 0; ok && j <= ntiles; ++j) {
          if (j < ntiles) {  // S = Q K^T into S buffer gs & 1 (Q from TMEM)
            const int s = gs & 1;
            const uint32_t ph = (uint32_t)(gs >> 1) & 1u;
            if (!tc::mbar_wait(bar_kfull(s), ph) || !tc::mbar_wait(bar_sempty(s), ph ^ 1u) ||
                *abort_flag) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t d_s = tmem + (uint32_t)(s * BN);
            const uint32_t k_s = sK + s * C::TILE;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
              const uint32_t o = (uint32_t)(k >> 2) * kBox + (uint32_t)(k & 3) * 32u;
              tc::mma_bf16_ts(d_s, t_q + 8u * k, tc::sdesc_sw128(k_s + o), idesc_s, k > 0 ? 1u : 0u);
            }
            tc::commit(bar_sfull(s));
            tc::commit(bar_kempty(s));
            ++gs;
            ++issued;
          }
          if (j >= 1) {  // O += P V of the unit's tile j - 1
            const int s = gp & 1;
            if (!tc::mbar_wait(bar_p(gp), (uint32_t)(gp >> 1) & 1u) ||
                !tc::mbar_wait(bar_vfull(s), (uint32_t)(gp >> 1) & 1u) || *abort_flag) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t v_s = sV + s * C::TILE;
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
              tc::mma_bf16_ts(t_o, t_p + 8u * k, tc::sdesc_sw128_mn(v_s + 2048u * k, kBox), idesc_o,
                              (j > 1 || k > 0) ? 1u : 0u);
            tc::commit(bar_vempty(s));
            tc::commit(bar_o(gp));
            ++gp;
            ++issued;
          }
        }
      }
      if (!ok) fail(abort_flag, kErrWaitTimeout);
      // drain: every MMA issued so far has completed once this commit lands
      if (issued > 0) {
        tc::commit(bar_done);
        tc::mbar_wait(bar_done, 0);
      }
    }
    __syncwarp();
  } else {
    // ============================================================ softmax + epilogue
    constexpr int OC = D / NQ;          // O columns of this thread in the rescale / epilogue
    constexpr int QW = D / (2 * NQ);    // 32-bit words (bf16 pairs) of the query row per thread
    const int h = (warp - 2) >> 2;      // key part of each tile (and D / NQ of O)
    const int eq = warp & 3;            // TMEM lane quarter
    const int row = eq * 32 + lane;     // query row within the tile
    const uint32_t lane_off = (uint32_t)(eq * 32) << 16;
    const float sc2 = rsqrtf((float)D) * kLog2e;
    // this thread's part of a unit's query row (zeros past the last query)
    uint32_t qv[QW];
    auto load_q = [&](const FwdUnit& U) {
      const int qr = U.row0 + row;
      if (qr < a.n_q) {
        const uint4* src = reinterpret_cast<const uint4*>(
            a.q + ((size_t)(U.l * a.Hq + U.hq) * a.n_q + qr) * D + h * (D / NQ));
#pragma unroll
        for (int c = 0; c < QW / 4; ++c) {
          const uint4 x = __ldg(src + c);
          qv[4 * c] = x.x;
          qv[4 * c + 1] = x.y;
          qv[4 * c + 2] = x.z;
          qv[4 * c + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < QW; ++c) qv[c] = 0u;
      }
    };
    if (nunits > 0) load_q(unit(0));
    int gs = 0;  // tiles processed (all units): S buffer, exchange buffer, P and O barriers
    bool failed = false, wait_failed = false;
    for (int n = 0; n < nunits && !failed; ++n) {
      const FwdUnit U = unit(n);
      const int qr = U.row0 + row;  // query index
      // the unit's query rows into TMEM: the previous unit's S products are complete (its
      // last P V was waited for below) and its O is in registers
      if constexpr (QW == 32)
        tc::tmem_st32(t_q + lane_off + (uint32_t)(h * QW), qv);
      else if constexpr (QW == 16)
        tc::tmem_st16(t_q + lane_off + (uint32_t)(h * QW), qv);
      else
        tc::tmem_st8(t_q + lane_off + (uint32_t)(h * QW), qv);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      tc::mbar_arrive(bar_q);
      float m_used = -1e30f, lsum = 0.f;
      for (int j = 0; j < U.ntiles; ++j, ++gs) {
        const int s = gs & 1;  // max-exchange buffer and S buffer
        bool ok = tc::mbar_wait(bar_sfull(s), (uint32_t)(gs >> 1) & 1u) && !*abort_flag;
        if (tc::bar_or(2, kSoftThreads, !ok || wait_failed)) {
          failed = true;
          break;
        }
        tc::fence_after_sync();
        uint32_t v[KC];
#pragma unroll
        for (int c = 0; c < KC; c += 32)
          tc::tmem_ld32(tmem + lane_off + (uint32_t)(s * BN + h * KC + c), v + c);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        tc::mbar_arrive(bar_sempty(s));  // the next S into this buffer may start now

        const bool ctx = j < U.n_ctx;
        const int kb = (ctx ? j * BN : a.T + (j - U.n_ctx) * BN) + h * KC;
        const int lim = ctx ? a.T : n_k;
        if (kb + KC > lim || kb + KC - 1 > off + qr) {
#pragma unroll
          for (int c = 0; c < KC; ++c)
            if (kb + c >= lim || kb + c > off + qr) v[c] = __float_as_uint(-CUDART_INF_F);
        }
        float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F, mx2 = -CUDART_INF_F, mx3 = -CUDART_INF_F;
#pragma unroll
        for (int c = 0; c < KC; c += 8) {
          mx0 = tc::max3(mx0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
          mx1 = tc::max3(mx1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
          mx2 = tc::max3(mx2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
          mx3 = tc::max3(mx3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
        }
        const float mine = tc::max3(mx0, mx1, fmaxf(mx2, mx3)) * sc2;
        float* xmj = xm + s * NQ * BM;
        xmj[h * BM + row] = mine;
        // the NQ threads of a row are the warps eq + 2 + 4g: one named barrier per lane
        // quarter (ids 3..6) pairs them without holding up the other quarters
        named_sync(3 + eq, 32 * NQ);
        float mt = mine;
#pragma unroll
        for (int g = 1; g < NQ; ++g) mt = fmaxf(mt, xmj[((h + g) % NQ) * BM + row]);
        const bool need = mt > m_used + kRescale;
        float factor = 1.f;
        if (need) {
          factor = fast_exp2(m_used - mt);
          m_used = mt;
          lsum *= factor;
        }
        // p = 2^(x sc2 - m) with packed fp32 pairs (FFMA2 / FADD2): half the FMA-pipe
        // instructions of scalar code, one MUFU ex2 per key
        uint32_t pk[KC / 2];
        const float2 k2 = make_float2(sc2, sc2), nm = make_float2(-m_used, -m_used);
        float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
        for (int c = 0; c < KC; c += 4) {
          const float2 y0 = __ffma2_rn(tc::f2(v[c], v[c + 1]), k2, nm);
          const float2 y1 = __ffma2_rn(tc::f2(v[c + 2], v[c + 3]), k2, nm);
          const float p0 = fast_exp2(y0.x), p1 = fast_exp2(y0.y);
          const float p2 = fast_exp2(y1.x), p3 = fast_exp2(y1.y);
          a0 = __fadd2_rn(a0, make_float2(p0, p1));
          a1 = __fadd2_rn(a1, make_float2(p2, p3));
          pk[c / 2] = pack_bf16(p0, p1);
          pk[c / 2 + 1] = pack_bf16(p2, p3);
        }
        a0 = __fadd2_rn(a0, a1);
        lsum += a0.x + a0.y;

        // P V of the previous tile has read its P (and finished O) before P is written;
        // O is rescaled only when this row's max grew past the threshold.  The unit's
        // first tile needs no wait: the previous unit's last P V was waited for below.
        const bool any_need = __any_sync(0xffffffffu, need);
        if (j > 0) {
          ok = tc::mbar_wait(bar_o(gs - 1), (uint32_t)((gs - 1) >> 1) & 1u) && !*abort_flag;
          ok = __all_sync(0xffffffffu, ok);  // the TMEM accesses below are warp-wide
          if (!ok) wait_failed = true;       // reported at the next vote
          tc::fence_after_sync();
          if (ok && any_need) {
            const uint32_t to = t_o + lane_off + (uint32_t)(h * OC);
            if constexpr (OC >= 32) {
#pragma unroll
              for (int cb = 0; cb < OC; cb += 32) {
                tc::tmem_ld32(to + cb, v);
                tc::tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * factor);
                tc::tmem_st32(to + cb, v);
              }
            } else {
              tc::tmem_ld16(to, v);
              tc::tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 16; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * factor);
              tc::tmem_st16(to, v);
            }
            tc::tmem_st_wait();
          }
        }
        if (wait_failed) continue;  // the P columns may still be in use: leave them alone
        // P of this thread's keys h*KC .. h*KC+KC-1 as bf16 pairs into P columns h*KC/2 ..
        if constexpr (KC == 64)
          tc::tmem_st32(t_p + lane_off + (uint32_t)(h * (KC / 2)), pk);
        else
          tc::tmem_st16(t_p + lane_off + (uint32_t)(h * (KC / 2)), pk);
        tc::tmem_st_wait();
        tc::fence_before_sync();
        tc::mbar_arrive(bar_p(gs));
      }
      if (failed) break;
      // the next unit's query rows load while this unit's O is finished and written
      if (n + 1 < nunits) load_q(unit(n + 1));
      // the last two P V products of the unit (on o[0] and o[1]) complete O
      bool ok = U.ntiles < 2 || tc::mbar_wait(bar_o(gs - 2), (uint32_t)((gs - 2) >> 1) & 1u);
      ok = ok && tc::mbar_wait(bar_o(gs - 1), (uint32_t)((gs - 1) >> 1) & 1u) && !*abort_flag;
      failed = tc::bar_or(2, kSoftThreads, !ok || wait_failed);
      if (failed) break;
      tc::fence_after_sync();
      xl[h * BM + row] = lsum;
      named_sync(1, kSoftThreads);
      float ltot = lsum;
#pragma unroll
      for (int g = 1; g < NQ; ++g) ltot += xl[((h + g) % NQ) * BM + row];
      const float inv = 1.f / ltot;
      uint32_t v[OC];
      uint32_t ob[OC / 2];
      if constexpr (OC >= 32) {
#pragma unroll
        for (int cb = 0; cb < OC; cb += 32) tc::tmem_ld32(t_o + lane_off + (uint32_t)(h * OC + cb), v + cb);
      } else {
        tc::tmem_ld16(t_o + lane_off + (uint32_t)(h * OC), v);
      }
      tc::tmem_ld_wait();
      if (a.o_f16) {
#pragma unroll
        for (int c = 0; c < OC; c += 2)
          ob[c / 2] = pack_f16(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv);
      } else {
#pragma unroll
        for (int c = 0; c < OC; c += 2)
          ob[c / 2] = pack_bf16(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv);
      }
      if (qr < a.n_q) {
        uint4* dst = reinterpret_cast<uint4*>(
            a.o + ((size_t)(U.l * a.Hq + U.hq) * a.n_q + qr) * D + h * OC);
#pragma unroll
        for (int c = 0; c < OC / 8; ++c)
          dst[c] = make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
        if (h == 0)
          a.lse[(size_t)(U.l * a.Hq + U.hq) * a.n_q + qr] = (m_used + fast_log2(ltot)) * kLn2;
      }
      // xl is rewritten at the next unit's end only after the rows' pair barriers of its
      // tiles, which every partner reaches after reading xl here
    }
    if (failed) atomicCAS(&g_fwd_error, 0, (int)kErrWaitTimeout);
  }

  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_fwd_d(const FwdArgs& a, cudaStream_t s) {
  using C = FCfg<D>;
  CUtensorMap tk, tv, tkt, tvt;
  cudaError_t e = a.T > 0 ? tma_map_bf16_3d(&tk, a.k_ctx, D, a.T, a.L * a.Hkv, BN)
                          : tma_map_bf16_3d(&tk, a.q, D, 1, 1, BN);
  if (e == cudaSuccess)
    e = a.T > 0 ? tma_map_bf16_3d(&tv, a.v_ctx, D, a.T, a.L * a.Hkv, BN)
                : tma_map_bf16_3d(&tv, a.q, D, 1, 1, BN);
  if (e == cudaSuccess)
    e = a.n_tail > 0 ? tma_map_bf16_3d(&tkt, a.k_tail, D, a.n_tail, a.L * a.Hkv, BN)
                     : tma_map_bf16_3d(&tkt, a.q, D, 1, 1, BN);
  if (e == cudaSuccess)
    e = a.n_tail > 0 ? tma_map_bf16_3d(&tvt, a.v_tail, D, a.n_tail, a.L * a.Hkv, BN)
                     : tma_map_bf16_3d(&tvt, a.q, D, 1, 1, BN);
  if (e != cudaSuccess) return e;
  static int nsm[64] = {0};
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!nsm[dev]) {
    e = cudaDeviceGetAttribute(&nsm[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
  }
  const long long units = (long long)((a.n_q + BM - 1) / BM) * a.Hq * a.L;
  dim3 grid((unsigned)std::min<long long>(units, std::max(1, nsm[dev])));  // one CTA per SM
  auto kern = attn_fwd_kernel<D>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  count_launches(1);
  kern<<<grid, kThreads, C::SMEM, s>>>(tk, tv, tkt, tvt, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const FwdArgs& a, cudaStream_t s) {
  if (a.n_q == 0) return cudaSuccess;
  return a.d == 128 ? launch_fwd_d<128>(a, s) : launch_fwd_d<64>(a, s);
}

cudaError_t fwd_device_error(int* code, bool clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_fwd_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && *code) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_fwd_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace kvs
