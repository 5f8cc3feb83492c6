// Attention-scoring passes on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Every pass runs one warp-specialised CTA per SM (a persistent grid).  A CTA takes
// 128-row units of operand A round-robin over (layer, head, row block) and, for each,
// streams 256-row tiles of operand B; each B tile is one chain of 128 x 256 x 16 MMAs
// (the wide N keeps the tensor core's shared-memory operand traffic at 96 bytes per
// clock).  Two A buffers alternate between consecutive units, the next unit's A tile
// loading as soon as its buffer's previous unit has finished its MMAs:
//   warp 0      TMA producer: A tiles into the two A buffers, B tiles through a ring of
//               two 64 KB tiles at d = 128 (four at d = 64), handed out per 64-column box
//               for the key-side maximum so that its loads lead the MMAs by 1.5 tiles
//   warp 1      allocates all 512 TMEM columns (two 256-column accumulators) and issues
//               tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32) into one of them;
//               with A = queries, a key tile reaching past the unit's causal limit is
//               multiplied only up to its last visible column (N rounded up to 16)
//   warps 2-17  epilogue, four groups of four warps (one warp per TMEM lane quarter per
//               group), 64 accumulator columns each: a thread reads its row's columns
//               with tcgen05.ld, releases the accumulator, and reduces them while the
//               MMA fills the other accumulator; the groups' partials of each row meet in
//               shared memory at the end of the unit (the quadratic form keeps two groups)
// Modes (x = q.k / sqrt(d), never written to memory):
//   kLse     A = queries,  B = key tiles (context, then tail): online max and
//            sum of 2^(x log2 e) per query -> ln sum exp(x)
//   kMax     A = context keys, B = query tiles of every head of the group: per key
//            max of x - lse_j - ln||h_j||, folded per head with ln ||W_O^{(h)} v_i||; the
//            per-query constant enters the accumulator through one extra K = 16 MMA
//            step (a ones tile against the constant split into three bf16 parts), so
//            the epilogue is a plain 3-input max
//   kFuture  A = keys, B = query tiles j >= i0 + w: per key sum over the group of
//            2^((x - lse_j) log2 e) for j >= i + w, with -lse_j sqrt(d) folded into the
//            accumulator by the same extra MMA step as kMax
//   kQuad    A = values, B = the head's Gram pair [G_hi | G_lo]: v^T G v per key and
//            query head of the group (the value norms)
//   kRows    A = queries, B = kept keys: the softmax rows 2^(x log2 e - lse_j log2 e) as
//            fp16, written through a per-warp stage (value refit)
// Sources: KVpop review, 1. Key Terms (LSE reuse, transposed-attention pass);
// KVzap review, 3.1 Eq. 1 and 3.2 Eq. 3.
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include "attn.cuh"
#include "tc.cuh"

namespace kvs {

__device__ int g_attn_error = 0;

namespace {

constexpr int BM = 128;     // rows of operand A per CTA = TMEM lanes
constexpr int BN = 256;     // rows per B tile = accumulator columns (N of each MMA)
constexpr int kGroupThreads = 128;  // one epilogue group: a warp per TMEM lane quarter
constexpr int kAllBar = 6;          // named barrier of all epilogue warps (groups use 1..4)
constexpr uint32_t kBoxBytesA = 128 * 128;  // 128 rows x 64 bf16 (one 128-byte swizzle span)
constexpr uint32_t kBoxBytesB = 256 * 128;  // 256 rows x 64 bf16
constexpr uint32_t kTmemCols = 2 * BN;       // two accumulators of 256 columns
constexpr int kErrWaitTimeout = 1;   // a bounded mbarrier wait ran out
constexpr int kErrSmemAlign = 3;     // dynamic shared memory window not 1024-byte aligned
constexpr uint32_t kMaxSmem = 232448;  // per-block opt-in limit (227 KB)

enum Mode { kLse = 0, kMax = 1, kFuture = 2, kQuad = 3, kRows = 4 };
// modes whose operand A is a tile of queries (B: key tiles)
template <int MODE>
__host__ __device__ constexpr bool a_is_queries() { return MODE == kLse || MODE == kRows; }
// Two A buffers per CTA, alternating between consecutive units, so the next unit's A tile
// loads and its MMAs start while the epilogue drains the current one.
constexpr int kABufs = 2;
constexpr int kMaxGroup = 16;  // query heads per KV head handled by kQuad

template <int D, int MODE>
struct Cfg {
  // epilogue groups, each owning COLS accumulator columns of every row: four groups of
  // 64 columns (four warps per SM sub-partition to hide the reductions' latency); the
  // quadratic form needs its rows' halves and keeps two
  static constexpr int NG = MODE == kQuad ? 2 : 4;
  static constexpr int COLS = BN / NG;
  // The maximum and the future mass split the tiles between two pairs of groups: pair p
  // takes the tiles of accumulator p (every other tile), each group of the pair 128 of
  // the 256 columns in two chunks of 64, so the pairs run half a tile apart and one
  // pair's TMEM loads overlap the other's arithmetic.  (The LSE pass measured slower
  // that way: its rescaled online sum pays per chunk, and its accumulator is released
  // later; it keeps every group on every tile.)
  static constexpr bool PAIRED = MODE == kMax || MODE == kFuture;
  static constexpr int EPI = NG * kGroupThreads;
  static constexpr int TEMPTY = PAIRED ? EPI / 2 : EPI;  // arrivals that release an accumulator
  static constexpr int THREADS = 64 + EPI;
  static constexpr int KH = D / 64;
  static constexpr int STAGES = D == 128 ? 2 : 4;  // B tiles in the ring
  // Ring slots per B tile.  The key-side passes (the maximum and the future mass) hand the
  // ring out by box (64 columns of d): a tile's first box is refilled while the MMAs read
  // its second, so the loads lead the MMAs by 1.5 tiles at d = 128 instead of one (the
  // future mass ran 4 % faster on c4 that way).  The other modes keep whole-tile slots:
  // their epilogues bound them and the extra barrier traffic of box slots costs them more
  // than the deeper lead gains (the LSE pass measured 2.5 % slower with box slots).
  static constexpr int PARTS = (MODE == kMax || MODE == kFuture) ? KH : 1;
  static constexpr int NS = STAGES * PARTS;
  static constexpr uint32_t SLOT_BYTES = KH / PARTS * kBoxBytesB;
  static constexpr uint32_t A_BYTES = KH * kBoxBytesA;  // one of kABufs A buffers
  static constexpr uint32_t B_BYTES = KH * kBoxBytesB;
  static constexpr uint32_t OFF_B = kABufs * A_BYTES;
  // kMax: the K = 16 operands of the constant-adding MMA step: a ones tile for A and,
  // per stage, the B tile's per-query constants (32-byte rows, 32-byte swizzle)
  static constexpr bool AUG = MODE == kMax || MODE == kFuture;
  static constexpr uint32_t AUG_A_BYTES = BM * 32, AUG_B_BYTES = BN * 32;
  static constexpr uint32_t OFF_AUG_A = OFF_B + STAGES * B_BYTES;
  static constexpr uint32_t OFF_AUG_B = OFF_AUG_A + (AUG ? AUG_A_BYTES : 0);
  static constexpr uint32_t OFF_X = OFF_AUG_B + (AUG ? STAGES * AUG_B_BYTES : 0);  // [2][NG-1][BM][2]
  // the softmax rows need no exchange of partials; their warps stage 32 rows x 64 bytes
  // each instead, so the rows leave in whole 64-byte segments
  static constexpr uint32_t ROWS_STAGE = 32 * 64;
  static constexpr uint32_t OFF_P =
      OFF_X + (MODE == kRows ? (EPI / 32) * ROWS_STAGE : 2 * (NG - 1) * BM * 2 * 4);  // kQuad [2][16][BM]
  static constexpr uint32_t OFF_BAR = OFF_P + (MODE == kQuad ? 2 * kMaxGroup * BM * 4 : 0);
  // a_full[kABufs], full[NS], empty[NS], tfull[2], tempty[2], a_empty[kABufs]
  static constexpr uint32_t NBAR = 2 * kABufs + 2 * NS + 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM = (USED + 1024 <= kMaxSmem) ? USED + 1024 : kMaxSmem;
  static constexpr uint32_t IDESC = tc::idesc_bf16(BM, BN);
  static_assert(USED <= kMaxSmem, "shared-memory plan exceeds the per-block limit");
};

__device__ __forceinline__ void fail(volatile uint32_t* abort_flag, int code) {
  *abort_flag = 1u;
  atomicCAS(&g_attn_error, 0, code);
}

using tc::f2;
using tc::max3;

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// LSE reduction of 64 columns: running max m (log2 units) and sum s.
__device__ __forceinline__ void lse_cols(const uint32_t* v, float sc2, float& m, float& ssum) {
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F, mx2 = -CUDART_INF_F, mx3 = -CUDART_INF_F;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    mx0 = max3(mx0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
    mx1 = max3(mx1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
    mx2 = max3(mx2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
    mx3 = max3(mx3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
  }
  const float mn = fmaxf(m, max3(mx0, mx1, fmaxf(mx2, mx3)) * sc2);
  ssum *= fast_exp2(m - mn);
  m = mn;
  const float2 k2 = make_float2(sc2, sc2), nm = make_float2(-m, -m);
  float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    const float2 y0 = __ffma2_rn(f2(v[c], v[c + 1]), k2, nm);
    const float2 y1 = __ffma2_rn(f2(v[c + 2], v[c + 3]), k2, nm);
    const float2 y2 = __ffma2_rn(f2(v[c + 4], v[c + 5]), k2, nm);
    const float2 y3 = __ffma2_rn(f2(v[c + 6], v[c + 7]), k2, nm);
    a0 = __fadd2_rn(a0, make_float2(fast_exp2(y0.x), fast_exp2(y0.y)));
    a1 = __fadd2_rn(a1, make_float2(fast_exp2(y1.x), fast_exp2(y1.y)));
    a2 = __fadd2_rn(a2, make_float2(fast_exp2(y2.x), fast_exp2(y2.y)));
    a3 = __fadd2_rn(a3, make_float2(fast_exp2(y3.x), fast_exp2(y3.y)));
  }
  a0 = __fadd2_rn(__fadd2_rn(a0, a1), __fadd2_rn(a2, a3));
  ssum += a0.x + a0.y;
}

// Max of 64 raw accumulator columns (the KVzip max with the constants folded in).
__device__ __forceinline__ float max_raw_cols(const uint32_t* v, float r) {
  float r0 = r, r1 = -CUDART_INF_F, r2 = -CUDART_INF_F, r3 = -CUDART_INF_F;
#pragma unroll
  for (int c = 0; c < 64; c += 8) {
    r0 = max3(r0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
    r1 = max3(r1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
    r2 = max3(r2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
    r3 = max3(r3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
  }
  return fmaxf(max3(r0, r1, r2), r3);
}

// Future mass of 64 columns: sum_c 2^(acc_c * sc2) (the column's -lse_j sqrt(d) is in the
// accumulator); in a band chunk (BAND) the columns c < jlim are zeroed.  The band test is
// a template argument so that the chunks off the band (nearly all) carry no per-column
// compare and select.
template <bool BAND>
__device__ __forceinline__ float future_cols(const uint32_t* v, float sc2, int jlim) {
  const float2 k2 = make_float2(sc2, sc2);
  float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const float2 y0 = __fmul2_rn(f2(v[4 * q], v[4 * q + 1]), k2);
    const float2 y1 = __fmul2_rn(f2(v[4 * q + 2], v[4 * q + 3]), k2);
    float e0 = fast_exp2(y0.x), e1 = fast_exp2(y0.y);
    float e2 = fast_exp2(y1.x), e3 = fast_exp2(y1.y);
    if constexpr (BAND) {
      if (4 * q < jlim) e0 = 0.f;
      if (4 * q + 1 < jlim) e1 = 0.f;
      if (4 * q + 2 < jlim) e2 = 0.f;
      if (4 * q + 3 < jlim) e3 = 0.f;
    }
    a0 = __fadd2_rn(a0, make_float2(e0, e1));
    a1 = __fadd2_rn(a1, make_float2(e2, e3));
  }
  a0 = __fadd2_rn(a0, a1);
  return a0.x + a0.y;
}

__device__ __forceinline__ uint32_t pack2_f16(float lo, float hi) {
  __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Softmax weights of 32 columns (keys kb .. kb+31) of the warp's 32 query rows, written
// as fp16 (weights in [0, 1]: 11 significant bits, 2^-12 relative): p = 2^(x sc2 - l2),
// 0 for keys >= lim.  Each thread computes its own row; the rows then pass through the
// warp's 2 KB stage (32 rows x 64 bytes), so every store instruction writes eight whole
// 64-byte row segments (a thread writing 16 bytes into each of 32 rows would make 32
// transactions).  row_base = element offset of the warp's first row (row stride ld);
// rows at or past nvalid (from the warp's first row) and columns at or past ld are not
// written.
__device__ __forceinline__ void rows_cols(const uint32_t* v, int kb, int lim, float l2, float sc2,
                                          uint16_t* rows, size_t row_base, int ld, int nvalid,
                                          uint8_t* stage, int lane) {
  if (kb >= ld) return;  // warp-uniform: ld is a multiple of 64, kb of 32
  const uint32_t sbase = smem_u32(stage);
  float pv[32];
#pragma unroll
  for (int c = 0; c < 32; ++c)
    pv[c] = (kb + c < lim) ? fast_exp2(fmaf(__uint_as_float(v[c]), sc2, -l2)) : 0.f;
  // this row's 64 bytes into the stage, 16-byte chunk j at position j ^ (row & 3)
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) w4[e] = pack2_f16(pv[8 * j + 2 * e], pv[8 * j + 2 * e + 1]);
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(
                     sbase + (uint32_t)(lane * 64 + ((j ^ (lane & 3)) << 4))),
                 "r"(w4[0]), "r"(w4[1]), "r"(w4[2]), "r"(w4[3])
                 : "memory");
  }
  __syncwarp();
  uint16_t* out = rows + row_base + kb;
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // lanes 4i..4i+3 write row 8q + i, 16 bytes each
    const int r = 8 * q + (lane >> 2), j = lane & 3;
    uint4 u;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                 : "r"(sbase + (uint32_t)(r * 64 + ((j ^ (r & 3)) << 4)))
                 : "memory");
    if (r < nvalid) *reinterpret_cast<uint4*>(out + (size_t)r * ld + 8 * j) = u;
  }
  __syncwarp();
}

// B-tile space of the 128-row unit starting at row0.
struct Tiles {
  int row0, ntiles, n_ctx, per_head, qt_begin;
};

template <int MODE>
__device__ __forceinline__ Tiles tiles_of(const AttnArgs& a, int row0, int G, int off) {
  Tiles t;
  t.row0 = row0;
  t.n_ctx = 0;
  t.per_head = 1;
  t.qt_begin = 0;
  if (a_is_queries<MODE>()) {
    const int j_last = min(row0 + BM, a.n_q) - 1;
    const int kv_end = off + j_last + 1;  // keys [0, kv_end) are visible to some query
    t.n_ctx = (min(a.T, kv_end) + BN - 1) / BN;
    const int tail_need = min(a.n_tail, max(0, kv_end - a.T));
    t.ntiles = t.n_ctx + (tail_need + BN - 1) / BN;
  } else if (MODE == kQuad) {
    t.ntiles = G;  // one B tile (the head's Gram pair) per query head of the group
  } else {
    const int nqt = (a.n_q + BN - 1) / BN;
    if (MODE == kFuture) t.qt_begin = (row0 + a.w) / BN;
    t.per_head = max(0, nqt - t.qt_begin);
    t.ntiles = G * t.per_head;
  }
  return t;
}

template <int D, int MODE>
__global__ void __launch_bounds__(Cfg<D, MODE>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_b2, const __grid_constant__ CUtensorMap tm_auga,
                   const __grid_constant__ CUtensorMap tm_augb, const AttnArgs a) {
  using C = Cfg<D, MODE>;
  constexpr int S = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  if (pad + C::USED > C::SMEM) {  // uniform; never overflow the allocation
    if (threadIdx.x == 0) atomicCAS(&g_attn_error, 0, kErrSmemAlign);
    return;
  }
  uint8_t* smem = smem_raw + pad;
  const uint32_t sb = raw + pad;
  const uint32_t sA = sb, sB = sb + C::OFF_B;
  float* xchg_all = reinterpret_cast<float*>(smem + C::OFF_X);
  float* part = reinterpret_cast<float*>(smem + C::OFF_P);
  const uint32_t bar0 = sb + C::OFF_BAR;
  auto bar_afull = [&](int b) { return bar0 + 8u * b; };
  constexpr int NS = C::NS;  // box slots of the B ring
  auto bar_full = [&](int j) { return bar0 + 8u * (kABufs + j); };
  auto bar_empty = [&](int j) { return bar0 + 8u * (kABufs + NS + j); };
  auto bar_tfull = [&](int x) { return bar0 + 8u * (kABufs + 2 * NS + x); };
  auto bar_tempty = [&](int x) { return bar0 + 8u * (kABufs + 2 * NS + 2 + x); };
  auto bar_aempty = [&](int b) { return bar0 + 8u * (kABufs + 2 * NS + 4 + b); };
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile uint32_t* abort_flag = misc + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.Hq / a.Hkv;
  const int n_k = a.T + a.n_tail;
  const int off = a.causal ? n_k - a.n_q : n_k;  // non-causal: every key is visible
  const float scale = rsqrtf((float)D);
  const float sc2 = scale * kLog2e;
  constexpr bool kQ = a_is_queries<MODE>();
  const int a_rows = kQ ? a.n_q : a.T;
  const int nrb = (a_rows + BM - 1) / BM;  // 128-row units per (layer, head)
  const int NH = kQ ? a.Hq : a.Hkv;
  // The CTA's units (a persistent grid of one CTA per SM): units blockIdx.x,
  // blockIdx.x + gridDim.x, ... of all (layer, head, row block), row block fastest, the two
  // A buffers alternating, the setup paid once per SM.
  const int nunits = (nrb * NH * a.L - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
  // A CTA's units visit one residue class of row blocks modulo dg = gcd(grid, row blocks);
  // the cost of a causal unit grows (or falls) with its row block, so odd groups of dg
  // row blocks are taken in reverse order, giving every residue class the same mean cost.
  int dg = (int)gridDim.x;
  for (int x = nrb; x > 0;) {
    const int t = dg % x;
    dg = x;
    x = t;
  }
  auto unit_of = [&](int n, int& l, int& hy) -> int {  // returns the unit's first row
    const int u = (int)blockIdx.x + n * (int)gridDim.x;
    const int r = u % nrb, k = r / dg, sr = r - k * dg;
    const int rb = k * dg + ((k & 1) ? dg - 1 - sr : sr);
    hy = (u / nrb) % NH;
    l = u / (nrb * NH);
    return rb * BM;
  };


  if (threadIdx.x == 0) {
    for (int n = 0; n < kABufs; ++n) {
      tc::mbar_init(bar_afull(n), 1);
      // the quadratic form's epilogue reads its value rows from A, so its threads also
      // release the buffer
      tc::mbar_init(bar_aempty(n), MODE == kQuad ? 1 + C::EPI : 1);
    }
    for (int j = 0; j < NS; ++j) {
      tc::mbar_init(bar_full(j), 1);
      tc::mbar_init(bar_empty(j), 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(bar_tfull(x), 1);
      tc::mbar_init(bar_tempty(x), C::TEMPTY);
    }
    misc[1] = 0u;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(sb + C::OFF_MISC, kTmemCols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_a);
    tc::tma_prefetch_desc(&tm_b);
    if (kQ) tc::tma_prefetch_desc(&tm_b2);
  }
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    // ============================================================ TMA producer
    if (lane == 0) {
      int gt = 0, na = 0, nb = 0;  // B tiles, A tiles and B boxes issued
      // A tile of unit na into buffer na & 1, whose previous unit (na - 2) is done: the
      // MMA issuer commits a_empty of the buffer once that unit's products complete
      auto issue_a = [&]() {
        int l, hy;
        const int row0 = unit_of(na, l, hy);
        const int b = na & 1;
        tc::mbar_expect_tx(bar_afull(b), C::A_BYTES + (C::AUG && na == 0 ? C::AUG_A_BYTES : 0));
        if (C::AUG && na == 0) tc::tma_load_3d(sb + C::OFF_AUG_A, &tm_auga, bar_afull(0), 0, 0, 0);
#pragma unroll
        for (int kh = 0; kh < C::KH; ++kh)
          tc::tma_load_3d(sA + b * C::A_BYTES + kh * kBoxBytesA, &tm_a, bar_afull(b), kh * 64, row0,
                          l * (kQ ? a.Hq : a.Hkv) + hy);
        ++na;
      };
      bool ok = true;
      for (int n = 0; n < nunits && ok; ++n) {
        int l, hy;
        const int row0 = unit_of(n, l, hy);
        const int hk = kQ ? hy / G : hy;
        if (na == n) {  // not prefetched: wait for the buffer
          if (!tc::mbar_wait(bar_aempty(n & 1), ((n >> 1) & 1) ^ 1u) || *abort_flag) {
            ok = false;
            break;
          }
          issue_a();
        }
        const Tiles U = tiles_of<MODE>(a, row0, G, off);
        for (int it = 0; it < U.ntiles && ok; ++it, ++gt) {
          // prefetch the next unit's A tile as soon as its buffer is free
          if (na == n + 1 && na < nunits && tc::mbar_test(bar_aempty(na & 1), ((na >> 1) & 1) ^ 1u))
            issue_a();
          const CUtensorMap* map;
          int row, head;
          if (kQ) {
            head = l * a.Hkv + hk;
            if (it < U.n_ctx) {
              map = &tm_b;
              row = it * BN;
            } else {
              map = &tm_b2;
              row = (it - U.n_ctx) * BN;
            }
          } else {
            map = &tm_b;
            head = l * a.Hq + hk * G + it / U.per_head;
            row = (U.qt_begin + it % U.per_head) * BN;
          }
          constexpr int BPP = C::KH / C::PARTS;  // boxes per slot
#pragma unroll
          for (int pt = 0; pt < C::PARTS; ++pt, ++nb) {  // part pt of the tile into slot nb % NS
            const int j = nb % NS;
            if (!tc::mbar_wait(bar_empty(j), (uint32_t)((nb / NS) & 1) ^ 1u) || *abort_flag) {
              ok = false;
              break;
            }
            const bool last = pt == C::PARTS - 1;
            tc::mbar_expect_tx(bar_full(j), C::SLOT_BYTES + (C::AUG && last ? C::AUG_B_BYTES : 0));
#pragma unroll
            for (int q = 0; q < BPP; ++q)
              tc::tma_load_3d(sB + j * C::SLOT_BYTES + q * kBoxBytesB, map, bar_full(j),
                              (pt * BPP + q) * 64, row, head);
            if (C::AUG && last)  // the tile's per-query constants (rows padded to whole tiles)
              tc::tma_load_3d(sb + C::OFF_AUG_B + (gt % S) * C::AUG_B_BYTES, &tm_augb, bar_full(j),
                              0, row, head);
          }
        }
      }
      if (!ok) {
        fail(abort_flag, kErrWaitTimeout);
        // let the copies already in flight land before the CTA exits
        for (int n = max(0, na - 2); n < na; ++n) tc::mbar_wait(bar_afull(n & 1), (n >> 1) & 1);
        for (int u = max(0, nb - NS); u < nb; ++u) tc::mbar_wait(bar_full(u % NS), (u / NS) & 1);
      }
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      int gt = 0, nb = 0;  // B tiles and boxes consumed
      bool ok = true;
      for (int n = 0; n < nunits && ok; ++n) {
        int l, hy;
        const Tiles U = tiles_of<MODE>(a, unit_of(n, l, hy), G, off);
        const int b = n & 1;
        if (!tc::mbar_wait(bar_afull(b), (n >> 1) & 1)) {
          ok = false;
          break;
        }
        const uint32_t a_n = sA + b * C::A_BYTES;
        for (int it = 0; it < U.ntiles && ok; ++it, ++gt) {
          const int acc = gt & 1;
          const uint32_t aph = (uint32_t)(gt >> 1) & 1u;
          if (!tc::mbar_wait(bar_tempty(acc), aph ^ 1u) || *abort_flag) {
            ok = false;
            break;
          }
          const uint32_t d_t = tmem + (uint32_t)(acc * BN);
          uint32_t idesc = C::IDESC;
          if constexpr (MODE == kLse || MODE == kRows) {
            // a tile past the causal limit of the unit's last query (or past the end of its
            // key range) is multiplied only up to its last visible column, rounded up to
            // 16; the epilogue masks, skips or zeroes every column past it
            const bool ctx = it < U.n_ctx;
            const int kb0 = ctx ? it * BN : a.T + (it - U.n_ctx) * BN;
            const int vis = min(ctx ? a.T : n_k, off + min(U.row0 + BM, a.n_q)) - kb0;
            if (vis < BN) idesc = tc::idesc_bf16(BM, max(16, (vis + 15) & ~15));
          }
          constexpr int BPP = C::KH / C::PARTS;  // boxes per slot
#pragma unroll
          for (int pt = 0; pt < C::PARTS; ++pt, ++nb) {  // part pt of the tile, in slot nb % NS
            const int j = nb % NS;
            if (!tc::mbar_wait(bar_full(j), (uint32_t)(nb / NS) & 1u) || *abort_flag) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
            const uint32_t b_j = sB + j * C::SLOT_BYTES;
#pragma unroll
            for (int k = 0; k < 4 * BPP; ++k) {  // 16 columns of d per MMA
              const int kh = pt * BPP + (k >> 2);  // box of the tile
              const uint32_t kk = (uint32_t)(k & 3) * 32u;
              tc::mma_bf16(d_t, tc::sdesc_sw128(a_n + kh * kBoxBytesA + kk),
                           tc::sdesc_sw128(b_j + (k >> 2) * kBoxBytesB + kk), idesc,
                           (pt | k) ? 1u : 0u);
            }
            if (C::AUG && pt == C::PARTS - 1)  // + (1,1,1,0..) . (c_hi, c_mid, c_lo, 0..)
              tc::mma_bf16(d_t, tc::sdesc_sw32(sb + C::OFF_AUG_A),
                           tc::sdesc_sw32(sb + C::OFF_AUG_B + (gt % S) * C::AUG_B_BYTES),
                           C::IDESC, 1u);
            tc::commit(bar_empty(j));  // the slot is free once these MMAs complete
          }
          if (ok) tc::commit(bar_tfull(acc));
        }
        // the producer reuses this A buffer for unit n + 2 once the unit's MMAs complete
        // (no commit after the last use, so nothing arrives once the CTA may have exited)
        if (n + 2 < nunits) tc::commit(bar_aempty(b));
      }
      if (!ok) fail(abort_flag, kErrWaitTimeout);
      if (nb > 0) tc::mbar_wait(bar_empty((nb - 1) % NS), (uint32_t)((nb - 1) / NS) & 1u);
    }
    __syncwarp();
  } else {
    // ============================================================ epilogue
    constexpr int NG = C::NG, COLS = C::COLS, EPI = C::EPI;
    const int h = (warp - 2) >> 2;               // epilogue group: columns [h COLS, (h+1) COLS)
    const int eq = warp & 3;                     // TMEM lane quarter this warp may access
    const int row = eq * 32 + lane;              // accumulator row
    const uint32_t t_lane = tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(h * COLS);
    const int bar_id = 1 + h;
    int gt = 0;
    bool failed = false;

    for (int n = 0; n < nunits; ++n) {
      int l, hy;
      const Tiles U = tiles_of<MODE>(a, unit_of(n, l, hy), G, off);
      const int hq_a = kQ ? hy : 0;
      const int hk = kQ ? hy / G : hy;
      const int ra = U.row0 + row;  // this thread's query (kLse, kRows) or key
      float l2row = 0.f;              // kRows: this query's LSE in log2 units
      // kRows: the warp's first row (of 32) in the output and how many of its rows exist
      const int warp_row0 = U.row0 + eq * 32;
      const size_t rows_base = ((size_t)(l * a.Hq + hq_a) * a.n_q + warp_row0) * a.rows_ld;
      if (MODE == kRows && ra < a.n_q) l2row = a.lse[(size_t)(l * a.Hq + hq_a) * a.n_q + ra] * kLog2e;

      // ||W_O v|| of this key for the head of tile it (1 without value norms); the
      // logarithm is taken only when the head's maximum is folded, tiles later, so the
      // load's latency never delays the release of an accumulator
      auto vn_of = [&](int it) -> float {
        if (!a.vnorm || ra >= a.T) return 1.f;
        return a.vnorm[(size_t)(l * a.Hq + hk * G + it / U.per_head) * a.T + ra];
      };

      float m = -1e30f, ssum = 0.f;                  // kLse
      float r = -CUDART_INF_F, tot = -CUDART_INF_F;  // kMax
      float vn = 1.f;                                // kMax: vnorm of the current head
      int cur_head = -1;                             // kMax: head of r (-1: none yet)
      float f = 0.f;                                 // kFuture

      // kQuad: this thread's D/2 elements of its value row, from the swizzled A tile
      uint32_t vrow[MODE == kQuad ? D / 4 : 1];
      bool bad = false;  // a wait of this group ran out: skip to the end-of-unit vote
      if (MODE == kQuad)
        bad = tc::bar_or(bar_id, kGroupThreads, !tc::mbar_wait(bar_afull(n & 1), (n >> 1) & 1));
      if (MODE == kQuad && !bad) {
        const uint32_t a_n = sA + (n & 1) * C::A_BYTES;
#pragma unroll
        for (int jj = 0; jj < D / 16; ++jj) {  // 16-byte chunks of 8 elements
          const int c = h * (D / 2) + 8 * jj;
          const uint32_t addr = a_n + (uint32_t)(c / 64) * kBoxBytesA + (uint32_t)row * 128u +
                                ((uint32_t)(((c % 64) / 8) ^ (row & 7)) << 4);
          uint4 u;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                       : "r"(addr));
          vrow[4 * jj] = u.x;
          vrow[4 * jj + 1] = u.y;
          vrow[4 * jj + 2] = u.z;
          vrow[4 * jj + 3] = u.w;
        }
        // the rows are in registers: the buffer may take unit n + 2 once the MMAs are done
        if (n + 2 < nunits) tc::mbar_arrive(bar_aempty(n & 1));
      }

      for (int it = 0; it < U.ntiles && !bad; ++it, ++gt) {
        const int acc = gt & 1;
        const uint32_t aph = (uint32_t)(gt >> 1) & 1u;
        if (C::PAIRED && acc != (h >> 1)) continue;  // the other pair's tile
        // a wait that runs out raises the CTA's abort flag, so every other thread leaves
        // at its next wait and all meet at the end-of-unit vote
        if (!tc::mbar_wait(bar_tfull(acc), aph) || *abort_flag) {
          *abort_flag = 1u;
          bad = true;
          break;
        }
        tc::fence_after_sync();
        if constexpr (MODE == kQuad) {
          uint32_t v[128];
          // columns [h D/2, (h+1) D/2) of V G_hi and of V G_lo (which starts at column D)
          const uint32_t tq =
              tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(acc * BN + h * (D / 2));
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            tc::tmem_ld32(tq + 32 * c, v + 32 * c);
            tc::tmem_ld32(tq + D + 32 * c, v + 64 + 32 * c);
          }
          tc::tmem_ld_wait();
          tc::fence_before_sync();
          tc::mbar_arrive(bar_tempty(acc));
          float p0 = 0.f, p1 = 0.f;
#pragma unroll
          for (int c = 0; c < D / 2; c += 2) {
            const uint32_t pr = vrow[c / 2];
            p0 = fmaf(__uint_as_float(v[c]) + __uint_as_float(v[64 + c]), bf16_lo(pr), p0);
            p1 = fmaf(__uint_as_float(v[c + 1]) + __uint_as_float(v[64 + c + 1]), bf16_hi(pr), p1);
          }
          part[(h * kMaxGroup + it) * BM + row] = p0 + p1;
          continue;
        } else {
          // this group's COLS columns; the accumulator is released as soon as they are in
          // registers, so the MMA of tile it+2 can start while they reduce
          const uint32_t ta = t_lane + (uint32_t)(acc * BN);
          if constexpr (MODE == kRows) {
            // softmax weights of this tile's columns, 32 at a time (their registers are the
            // kernel's tightest), written through the warp's stage; then the accumulator
            // is released
#pragma unroll 1
            for (int c = 0; c < COLS; c += 32) {
              uint32_t v32[32];
              tc::tmem_ld32(ta + c, v32);
              tc::tmem_ld_wait();
              rows_cols(v32, it * BN + h * COLS + c, a.T, l2row, sc2, a.rows,
                        rows_base, a.rows_ld, a.n_q - warp_row0,
                        smem + C::OFF_X + (warp - 2) * C::ROWS_STAGE, lane);
            }
            tc::fence_before_sync();
            tc::mbar_arrive(bar_tempty(acc));
          } else {
            if (MODE == kMax) {  // a new query head: fold the previous head's maximum
              const int hd = it / U.per_head;
              if (hd != cur_head) {
                if (cur_head >= 0) tot = fmaxf(tot, r * scale + logf(vn));
                r = -CUDART_INF_F;
                vn = vn_of(it);
                cur_head = hd;
              }
            }
            // paired modes: this group's 128 columns in two chunks of 64; otherwise its 64
            // columns in one chunk.  The accumulator is released once the last chunk is in
            // registers.
            constexpr int NCH = C::PAIRED ? 2 : 1;
            const int cbase = C::PAIRED ? (h & 1) * 128 : h * COLS;
            const uint32_t ta2 =
                tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)(acc * BN) + (uint32_t)cbase;
#pragma unroll 1
            for (int ch = 0; ch < NCH; ++ch) {
              uint32_t w[64];
              tc::tmem_ld32(ta2 + 64 * ch, w);
              tc::tmem_ld32(ta2 + 64 * ch + 32, w + 32);
              tc::tmem_ld_wait();
              if (ch == NCH - 1) {
                tc::fence_before_sync();
                tc::mbar_arrive(bar_tempty(acc));
              }
              const int c0 = cbase + 64 * ch;  // first column of the chunk in the tile
              if (MODE == kLse) {
                const bool ctx = it < U.n_ctx;
                const int kb = (ctx ? it * BN : a.T + (it - U.n_ctx) * BN) + c0;
                const int lim = ctx ? a.T : n_k;
                if (kb >= lim || kb > off + ra) continue;  // no visible key in these 64
                if (kb + 64 > lim || kb + 63 > off + ra) {
#pragma unroll
                  for (int c = 0; c < 64; ++c)
                    if (kb + c >= lim || kb + c > off + ra) w[c] = __float_as_uint(-CUDART_INF_F);
                }
                lse_cols(w, sc2, m, ssum);
              } else if (MODE == kMax) {
                r = max_raw_cols(w, r);  // q.k / scale-units minus the column's constant
              } else {
                const int j0 = (U.qt_begin + it % U.per_head) * BN + c0;
                const bool band = j0 < U.row0 + BM - 1 + a.w;
                if (band) {
                  if (ra + a.w - j0 >= 64) continue;  // all 64 queries in the window
                  f += future_cols<true>(w, sc2, ra + a.w - j0);
                } else {
                  f += future_cols<false>(w, sc2, 0);
                }
              }
            }
          }
        }
      }
      // results of this unit: combine the groups' partial results of each row (kQuad:
      // the per-head partial dot products).  All groups vote on failure here, so they
      // leave the unit loop together and never wait at a barrier another has abandoned.
      if (MODE == kMax && cur_head >= 0) tot = fmaxf(tot, r * scale + logf(vn));
      float* xchg = xchg_all + (n & 1) * (NG - 1) * BM * 2;
      if (MODE != kQuad && MODE != kRows && h > 0 && !bad) {
        float* xg = xchg + (h - 1) * BM * 2;
        if (MODE == kLse) {
          xg[row * 2] = m;
          xg[row * 2 + 1] = ssum;
        } else {
          xg[row * 2] = (MODE == kMax) ? tot : f;
        }
      }
      if (tc::bar_or(kAllBar, EPI, bad)) {
        failed = true;
        break;
      }
      if (MODE == kRows) continue;  // rows were written tile by tile
      if (MODE == kQuad) {
        if (h == 0 && ra < a.T) {
          for (int it = 0; it < U.ntiles; ++it) {
            const float q2 = part[it * BM + row] + part[(kMaxGroup + it) * BM + row];
            a.out[(size_t)(l * a.Hq + hk * G + it) * a.T + ra] = sqrtf(fmaxf(q2, 0.f));
          }
        }
        if (n + 1 < nunits) named_sync(kAllBar, EPI);  // part[] is rewritten by the next unit
        continue;
      }
      if (h == 0) {
        if (MODE == kLse) {
          float mn = m;
#pragma unroll
          for (int g2 = 0; g2 < NG - 1; ++g2) mn = fmaxf(mn, xchg[g2 * BM * 2 + row * 2]);
          float st = ssum * fast_exp2(m - mn);
#pragma unroll
          for (int g2 = 0; g2 < NG - 1; ++g2)
            st += xchg[g2 * BM * 2 + row * 2 + 1] * fast_exp2(xchg[g2 * BM * 2 + row * 2] - mn);
          if (ra < a.n_q)
            a.out[(size_t)(l * a.Hq + hq_a) * a.n_q + ra] = (mn + fast_log2(st)) * kLn2;
        } else if (MODE == kMax) {
          float t2 = tot;
#pragma unroll
          for (int g2 = 0; g2 < NG - 1; ++g2) t2 = fmaxf(t2, xchg[g2 * BM * 2 + row * 2]);
          if (ra < a.T) {
            float* o = a.out + (size_t)(l * a.Hkv + hk) * a.T + ra;
            *o = a.accumulate ? fmaxf(*o, t2) : t2;
          }
        } else {
          float ft = f;
#pragma unroll
          for (int g2 = 0; g2 < NG - 1; ++g2) ft += xchg[g2 * BM * 2 + row * 2];
          if (ra < a.T) a.out[(size_t)(l * a.Hkv + hk) * a.T + ra] = ft;
        }
      }
    }
    if (failed) atomicCAS(&g_attn_error, 0, (int)kErrWaitTimeout);
  }

  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D map over [heads][rows][16] bf16 with box_rows x 16 boxes, 32-byte swizzle.
cudaError_t make_map_k16(CUtensorMap* m, const void* base, int rows, int heads, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {16, (cuuint64_t)rows, (cuuint64_t)heads};
  cuuint64_t strides[2] = {32, (cuuint64_t)rows * 32};
  cuuint32_t box[3] = {16, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over [heads][rows][d] bf16 with 128-row x 64-element boxes, 128-byte swizzle;
// rows past the end read as zeros.
cudaError_t make_map(CUtensorMap* m, const void* base, int d, int rows, int heads, int box_rows) {
  auto enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)heads};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int MODE>
cudaError_t launch_d(const AttnArgs& a, cudaStream_t s) {
  using C = Cfg<D, MODE>;
  CUtensorMap ta, tb, tb2;
  cudaError_t e;
  if (a_is_queries<MODE>()) {
    e = make_map(&ta, a.q, D, a.n_q, a.L * a.Hq, BM);
    if (e == cudaSuccess)
      e = a.T > 0 ? make_map(&tb, a.k_ctx, D, a.T, a.L * a.Hkv, BN)
                  : make_map(&tb, a.q, D, 1, 1, BN);
    if (e == cudaSuccess)
      e = a.n_tail > 0 ? make_map(&tb2, a.k_tail, D, a.n_tail, a.L * a.Hkv, BN)
                       : make_map(&tb2, a.q, D, 1, 1, BN);
  } else if (MODE == kQuad) {
    e = make_map(&ta, a.k_ctx, D, a.T, a.L * a.Hkv, BM);
    if (e == cudaSuccess) e = make_map(&tb, a.gpair, D, 2 * D, a.L * a.Hq, BN);
    tb2 = tb;
  } else {
    e = make_map(&ta, a.k_ctx, D, a.T, a.L * a.Hkv, BM);
    // with no scoring queries no B tile is loaded (every key gets the empty reduction)
    if (e == cudaSuccess)
      e = a.n_q > 0 ? make_map(&tb, a.q, D, a.n_q, a.L * a.Hq, BN)
                    : make_map(&tb, a.k_ctx, D, 1, 1, BN);
    tb2 = tb;
  }
  if (e != cudaSuccess) return e;
  CUtensorMap tauga = ta, taugb = ta;  // the constant-adding operands (kMax only)
  if (C::AUG) {
    if (!a.ccol || !a.ones) return cudaErrorInvalidValue;
    const int nq_pad = (a.n_q + BN - 1) / BN * BN;
    e = make_map_k16(&taugb, a.ccol, nq_pad, a.L * a.Hq, BN);
    if (e == cudaSuccess) e = make_map_k16(&tauga, a.ones, BM, 1, BM);
    if (e != cudaSuccess) return e;
  }
  const int rows = a_is_queries<MODE>() ? a.n_q : a.T;
  const int nrb = (rows + BM - 1) / BM, nh = a_is_queries<MODE>() ? a.Hq : a.Hkv;
  // one CTA per SM (fewer when there are fewer units), each looping over its units
  static int nsm[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!nsm[dev]) cudaDeviceGetAttribute(&nsm[dev], cudaDevAttrMultiProcessorCount, dev);
  const long units = (long)nrb * nh * a.L;
  const dim3 grid((unsigned)std::min(units, (long)std::max(1, nsm[dev])), 1, 1);
  auto kern = attn_tc_kernel<D, MODE>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  count_launches(1);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(ta, tb, tb2, tauga, taugb, a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_mode(const AttnArgs& a, cudaStream_t s) {
  const int rows = a_is_queries<MODE>() ? a.n_q : a.T;
  if (rows == 0) return cudaSuccess;
  return a.d == 128 ? launch_d<128, MODE>(a, s) : launch_d<64, MODE>(a, s);
}

// The per-query constants of the maximum with the hidden-state factor, from h directly:
// one warp per (layer, query row j) reduces ln ||h_j|| and writes the constants of all
// H_q query heads for that row, so ||h_j|| never makes a round trip through memory.
__global__ void __launch_bounds__(256) hidden_constants_kernel(
    const bf16_t* __restrict__ h, int Dh, const float* __restrict__ lse, int L, int Hq, int n_q,
    int nq_pad, float inv_scale, bf16_t* ccol, bf16_t* ones) {
  if (blockIdx.x == 0 && threadIdx.x < BM) {
    const uint32_t one = 0x3F80u;  // bf16 1.0
    uint4* o = reinterpret_cast<uint4*>(ones + threadIdx.x * 16);
    o[0] = make_uint4(one | (one << 16), one, 0u, 0u);
    o[1] = make_uint4(0u, 0u, 0u, 0u);
  }
  const int wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wg >= L * nq_pad) return;
  const int l = wg / nq_pad, j = wg % nq_pad;
  float hl = 0.f;
  if (j < n_q) {
    const bf16_t* p = h + ((size_t)l * n_q + j) * Dh;
    float s = 0.f;
    for (int c = lane * 8; c < Dh; c += 256) {
      const uint4 u = ld_nc_v4(p + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float lo = bf16_lo(w[k]), hi = bf16_hi(w[k]);
        s = fmaf(lo, lo, s);
        s = fmaf(hi, hi, s);
      }
    }
    hl = 0.5f * logf(warp_sum(s));
  }
  for (int hq = lane; hq < Hq; hq += 32) {
    const size_t lh = (size_t)l * Hq + hq;
    const float v = j < n_q ? -(lse[lh * n_q + j] + hl) * inv_scale : -1e30f;
    const __nv_bfloat16 bh = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(bh);
    const __nv_bfloat16 bm = __float2bfloat16_rn(r1);
    const __nv_bfloat16 bl = __float2bfloat16_rn(r1 - __bfloat162float(bm));
    const uint32_t w0 = (uint32_t)__bfloat16_as_ushort(bh) | ((uint32_t)__bfloat16_as_ushort(bm) << 16);
    const uint32_t w1 = (uint32_t)__bfloat16_as_ushort(bl);
    uint4* o = reinterpret_cast<uint4*>(ccol + (lh * nq_pad + j) * 16);
    o[0] = make_uint4(w0, w1, 0u, 0u);
    o[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

cudaError_t tma_map_bf16_3d(CUtensorMap* m, const void* base, int inner, int rows, int outer,
                            int box_rows) {
  return make_map(m, base, inner, rows, outer, box_rows);
}

cudaError_t tma_map_bf16_k16(CUtensorMap* m, const void* base, int rows, int outer, int box_rows) {
  return make_map_k16(m, base, rows, outer, box_rows);
}

namespace {

// Row (l, hq, j) of the KVzip max constants: -(lse_j + ln||h_j||) / scale as a sum of
// three bf16 (hi, mid, lo: ~24 bits), then zeros; rows past n_q hold -1e30 (they are
// padding queries and must never win the max).  Block 0 also writes the ones tile.
__global__ void __launch_bounds__(256) score_constants_kernel(const float* __restrict__ lse,
                                                              int L, int Hq, int n_q, int nq_pad,
                                                              float inv_scale, bf16_t* ccol,
                                                              bf16_t* ones) {
  const size_t row = (size_t)blockIdx.x * 256 + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x < BM) {
    const uint32_t one = 0x3F80u;  // bf16 1.0
    uint4* o = reinterpret_cast<uint4*>(ones + threadIdx.x * 16);
    o[0] = make_uint4(one | (one << 16), one, 0u, 0u);
    o[1] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (row >= (size_t)L * Hq * nq_pad) return;
  const int j = (int)(row % nq_pad);
  const size_t lh = row / nq_pad;  // l * Hq + hq
  float v = -1e30f;
  if (j < n_q) v = -lse[lh * n_q + j] * inv_scale;
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(hi);
  const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
  const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
  const uint32_t w0 = (uint32_t)__bfloat16_as_ushort(hi) | ((uint32_t)__bfloat16_as_ushort(mid) << 16);
  const uint32_t w1 = (uint32_t)__bfloat16_as_ushort(lo);
  uint4* o = reinterpret_cast<uint4*>(ccol + row * 16);
  o[0] = make_uint4(w0, w1, 0u, 0u);
  o[1] = make_uint4(0u, 0u, 0u, 0u);
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t score_max_ws_bytes(int L, int Hq, int n_q) {
  const size_t nq_pad = (size_t)(n_q + BN - 1) / BN * BN;
  return align256((size_t)L * Hq * nq_pad * 32) + (size_t)BM * 32;
}

cudaError_t launch_score_constants(const float* lse, int L, int Hq, int n_q,
                                   int d, bf16_t* ccol, bf16_t* ones, cudaStream_t s) {
  const int nq_pad = (n_q + BN - 1) / BN * BN;
  const size_t rows = (size_t)L * Hq * nq_pad;
  count_launches(1);
  score_constants_kernel<<<(unsigned)((rows + 255) / 256), 256, 0, s>>>(
      lse, L, Hq, n_q, nq_pad, sqrtf((float)d), ccol, ones);
  return cudaGetLastError();
}

cudaError_t launch_hidden_constants(const bf16_t* h, int Dh, const float* lse, int L, int Hq,
                                    int n_q, int d, bf16_t* ccol, bf16_t* ones, cudaStream_t s) {
  const int nq_pad = (n_q + BN - 1) / BN * BN;
  const size_t warps = (size_t)L * nq_pad;
  count_launches(1);
  hidden_constants_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, s>>>(h, Dh, lse, L, Hq, n_q, nq_pad,
                                                                      sqrtf((float)d), ccol, ones);
  return cudaGetLastError();
}

cudaError_t launch_lse(const AttnArgs& a, cudaStream_t s) { return launch_mode<kLse>(a, s); }
cudaError_t launch_softmax_rows(const AttnArgs& a, cudaStream_t s) {
  return launch_mode<kRows>(a, s);
}
cudaError_t launch_score_max(const AttnArgs& a, cudaStream_t s) { return launch_mode<kMax>(a, s); }
cudaError_t launch_future_sum(const AttnArgs& a, cudaStream_t s) {
  return launch_mode<kFuture>(a, s);
}
cudaError_t launch_vnorm_quad(const AttnArgs& a, cudaStream_t s) {
  if (a.Hq / a.Hkv > kMaxGroup) return cudaErrorInvalidValue;
  return launch_mode<kQuad>(a, s);
}

cudaError_t attn_device_error(int* code, bool clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_attn_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && *code) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_attn_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace kvs
