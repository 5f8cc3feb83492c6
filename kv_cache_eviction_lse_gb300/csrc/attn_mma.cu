// Attention-scoring passes on the warp-level tensor-core path (mma.sync m16n8k16).
//
// Pass 1 (LSE) and pass 2 (transposed scoring) share one tile engine: a block holds
// 64 rows of operand A in registers (4 warps x 16 rows) and streams 64-row tiles of
// operand B through double-buffered shared memory (cp.async), computing S = A B^T
// with fp32 accumulation; each mode reduces S in registers without ever writing it:
//   kLse     A = queries, B = keys:   online max / sum of 2^(x log2 e) per query
//   kMax     A = keys,    B = queries: running max of x - lse_j - ln||h_j|| per key,
//                                     folded per query head with ln ||W_O v_i||
//   kFuture  A = keys,    B = queries: sum of 2^((x - lse_j) log2 e) over j >= i + w
// x = q.k / sqrt(d).  Sources: KVpop review, 1. Key Terms (LSE reuse, transposed pass);
// KVzap review, 3.1 Eq. 1 and 3.2 Eq. 3.
#include <math_constants.h>

#include "attn.cuh"

namespace kvs {
namespace {

constexpr int BM = 64;
constexpr int BN = 64;
constexpr int NTHR = 128;

enum Mode { kLse = 0, kMax = 1, kFuture = 2 };

template <int D>
struct alignas(16) AttnSmem {
  bf16_t b[2][BN][D + 8];  // +8 elements: rows 16 B apart in bank space (ldmatrix conflict-free)
  float cv[2][BN];         // per-column constant of the B tile (mode dependent)
};

template <int D, int MODE>
__global__ void __launch_bounds__(NTHR) attn_mma_kernel(const AttnArgs a) {
  __shared__ AttnSmem<D> sm;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const int l = blockIdx.z;
  const int G = a.Hq / a.Hkv;
  const int n_k = a.T + a.n_tail;
  const int off = n_k - a.n_q;
  const float scale = rsqrtf((float)D);
  const float sc2 = scale * kLog2e;
  const int row0 = blockIdx.x * BM;
  const int hq_a = (MODE == kLse) ? (int)blockIdx.y : 0;
  const int hk = (MODE == kLse) ? hq_a / G : (int)blockIdx.y;

  // ---------------------------------------------------------------- operand A -> registers
  {
    const bf16_t* base;
    int nrows;
    if (MODE == kLse) {
      base = a.q + (size_t)(l * a.Hq + hq_a) * a.n_q * D;
      nrows = a.n_q;
    } else {
      base = a.k_ctx + (size_t)(l * a.Hkv + hk) * a.T * D;
      nrows = a.T;
    }
    for (int idx = tid; idx < BM * (D / 8); idx += NTHR) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      const int row = row0 + r;
      const bool ok = row < nrows;
      cp_async16(smem_u32(&sm.b[0][r][c * 8]), ok ? base + (size_t)row * D + c * 8 : base,
                 ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
  }
  uint32_t af[D / 16][4];
#pragma unroll
  for (int kc = 0; kc < D / 16; ++kc)
    ldmatrix_x4(smem_u32(&sm.b[0][warp * 16 + (lane & 15)][kc * 16 + (lane >> 4) * 8]),
                af[kc][0], af[kc][1], af[kc][2], af[kc][3]);
  __syncthreads();

  // ---------------------------------------------------------------- tile space of B
  const int nqt = (a.n_q + BN - 1) / BN;
  int ntiles = 0, per_head = 0, qt_begin = 0;
  if (MODE == kLse) {
    const int j_last = min(row0 + BM, a.n_q) - 1;
    ntiles = (off + j_last + 1 + BN - 1) / BN;
  } else if (MODE == kMax) {
    per_head = nqt;
    ntiles = G * per_head;
  } else {
    qt_begin = (row0 + a.w) / BN;
    per_head = max(0, nqt - qt_begin);
    ntiles = G * per_head;
  }

  auto issue = [&](int it, int buf) {
    if (MODE == kLse) {
      const int i0 = it * BN;
      const bf16_t* kc = a.k_ctx + (size_t)(l * a.Hkv + hk) * a.T * D;
      const bf16_t* kt = a.k_tail + (size_t)(l * a.Hkv + hk) * a.n_tail * D;
      for (int idx = tid; idx < BN * (D / 8); idx += NTHR) {
        const int r = idx / (D / 8), c = idx % (D / 8);
        const int i = i0 + r;
        const bf16_t* src = a.q;  // never read when nb == 0
        int nb = 0;
        if (i < a.T) {
          src = kc + (size_t)i * D + c * 8;
          nb = 16;
        } else if (i < n_k) {
          src = kt + (size_t)(i - a.T) * D + c * 8;
          nb = 16;
        }
        cp_async16(smem_u32(&sm.b[buf][r][c * 8]), src, nb);
      }
    } else {
      const int hq = hk * G + it / per_head;
      const int j0 = (qt_begin + it % per_head) * BN;
      const bf16_t* qb = a.q + (size_t)(l * a.Hq + hq) * a.n_q * D;
      for (int idx = tid; idx < BN * (D / 8); idx += NTHR) {
        const int r = idx / (D / 8), c = idx % (D / 8);
        const int j = j0 + r;
        const bool ok = j < a.n_q;
        cp_async16(smem_u32(&sm.b[buf][r][c * 8]), ok ? qb + (size_t)j * D + c * 8 : qb,
                   ok ? 16 : 0);
      }
      if (tid < BN) {
        const int j = j0 + tid;
        float c = -CUDART_INF_F;
        if (j < a.n_q) {
          const float lj = a.lse[(size_t)(l * a.Hq + hq) * a.n_q + j];
          if (MODE == kMax)
            c = -(lj + (a.hlog ? a.hlog[(size_t)l * a.n_q + j] : 0.f));
          else
            c = -lj * kLog2e;
        }
        sm.cv[buf][tid] = c;
      }
    }
  };

  // per-thread state for rows g and g+8 of this warp's 16 A rows
  const int ra0 = row0 + warp * 16 + g, ra1 = ra0 + 8;
  float m0 = -1e30f, m1 = -1e30f, s0 = 0.f, s1 = 0.f;                  // kLse
  float r0 = -CUDART_INF_F, r1 = -CUDART_INF_F;                       // kMax: per head
  float tot0 = -CUDART_INF_F, tot1 = -CUDART_INF_F;                   // kMax: over heads
  float f0 = 0.f, f1 = 0.f;                                           // kFuture
  const int lim0 = off + ra0, lim1 = off + ra1;                       // kLse: last visible key

  if (ntiles > 0) {
    issue(0, 0);
    cp_async_commit();
  }
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < ntiles) {
      issue(it + 1, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    float acc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
      for (int k2 = 0; k2 < D / 32; ++k2) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(&sm.b[buf][nt * 8 + (lane & 7)][k2 * 32 + (lane >> 3) * 8]), b0,
                    b1, b2, b3);
        mma_bf16_16816(acc[nt], af[2 * k2], b0, b1);
        mma_bf16_16816(acc[nt], af[2 * k2 + 1], b2, b3);
      }
    }

    if (MODE == kLse) {
      const int i0 = it * BN;
      const bool need_mask = (i0 + BN - 1 > off + row0 + warp * 16);
      float tm0 = -CUDART_INF_F, tm1 = -CUDART_INF_F;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = acc[nt][e] * sc2;
          if (need_mask) {
            const int i = i0 + nt * 8 + 2 * t4 + (e & 1);
            if (i > (e < 2 ? lim0 : lim1)) x = -CUDART_INF_F;
          }
          acc[nt][e] = x;
          if (e < 2) tm0 = fmaxf(tm0, x); else tm1 = fmaxf(tm1, x);
        }
      }
      const float mn0 = fmaxf(m0, tm0), mn1 = fmaxf(m1, tm1);
      s0 *= fast_exp2(m0 - mn0);
      s1 *= fast_exp2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s0 += fast_exp2(acc[nt][0] - m0) + fast_exp2(acc[nt][1] - m0);
        s1 += fast_exp2(acc[nt][2] - m1) + fast_exp2(acc[nt][3] - m1);
      }
    } else if (MODE == kMax) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const float c0 = sm.cv[buf][nt * 8 + 2 * t4], c1 = sm.cv[buf][nt * 8 + 2 * t4 + 1];
        r0 = fmaxf(r0, fmaxf(fmaf(acc[nt][0], scale, c0), fmaf(acc[nt][1], scale, c1)));
        r1 = fmaxf(r1, fmaxf(fmaf(acc[nt][2], scale, c0), fmaf(acc[nt][3], scale, c1)));
      }
      if ((it + 1) % per_head == 0) {  // last query tile of this query head
        const int hq = hk * G + it / per_head;
        float lv0 = 0.f, lv1 = 0.f;
        if (a.vnorm) {
          const float* vn = a.vnorm + (size_t)(l * a.Hq + hq) * a.T;
          lv0 = ra0 < a.T ? logf(vn[ra0]) : 0.f;
          lv1 = ra1 < a.T ? logf(vn[ra1]) : 0.f;
        }
        tot0 = fmaxf(tot0, r0 + lv0);
        tot1 = fmaxf(tot1, r1 + lv1);
        r0 = r1 = -CUDART_INF_F;
      }
    } else {
      const int j0 = (qt_begin + it % per_head) * BN;
      const bool need_band = j0 < row0 + warp * 16 + 15 + a.w;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = nt * 8 + 2 * t4 + (e & 1);
          float ev = fast_exp2(fmaf(acc[nt][e], sc2, sm.cv[buf][col]));
          if (need_band && j0 + col < (e < 2 ? ra0 : ra1) + a.w) ev = 0.f;
          if (e < 2) f0 += ev; else f1 += ev;
        }
      }
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- quad reduce + store
  if (MODE == kLse) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      const float mo0 = __shfl_xor_sync(0xffffffffu, m0, o), so0 = __shfl_xor_sync(0xffffffffu, s0, o);
      const float mo1 = __shfl_xor_sync(0xffffffffu, m1, o), so1 = __shfl_xor_sync(0xffffffffu, s1, o);
      const float mn0 = fmaxf(m0, mo0), mn1 = fmaxf(m1, mo1);
      s0 = s0 * fast_exp2(m0 - mn0) + so0 * fast_exp2(mo0 - mn0);
      s1 = s1 * fast_exp2(m1 - mn1) + so1 * fast_exp2(mo1 - mn1);
      m0 = mn0;
      m1 = mn1;
    }
    if (t4 == 0) {
      float* out = a.out + (size_t)(l * a.Hq + hq_a) * a.n_q;
      if (ra0 < a.n_q) out[ra0] = (m0 + fast_log2(s0)) * kLn2;
      if (ra1 < a.n_q) out[ra1] = (m1 + fast_log2(s1)) * kLn2;
    }
  } else if (MODE == kMax) {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      tot0 = fmaxf(tot0, __shfl_xor_sync(0xffffffffu, tot0, o));
      tot1 = fmaxf(tot1, __shfl_xor_sync(0xffffffffu, tot1, o));
    }
    if (t4 == 0) {
      float* out = a.out + (size_t)(l * a.Hkv + hk) * a.T;
      if (ra0 < a.T) out[ra0] = a.accumulate ? fmaxf(out[ra0], tot0) : tot0;
      if (ra1 < a.T) out[ra1] = a.accumulate ? fmaxf(out[ra1], tot1) : tot1;
    }
  } else {
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
      f0 += __shfl_xor_sync(0xffffffffu, f0, o);
      f1 += __shfl_xor_sync(0xffffffffu, f1, o);
    }
    if (t4 == 0) {
      float* out = a.out + (size_t)(l * a.Hkv + hk) * a.T;
      if (ra0 < a.T) out[ra0] = f0;
      if (ra1 < a.T) out[ra1] = f1;
    }
  }
}

template <int MODE>
cudaError_t launch_mode(const AttnArgs& a, cudaStream_t s) {
  const int rows = (MODE == kLse) ? a.n_q : a.T;
  if (rows == 0) return cudaSuccess;
  dim3 grid((rows + BM - 1) / BM, MODE == kLse ? a.Hq : a.Hkv, a.L);
  count_launches(1);
  if (a.d == 128)
    attn_mma_kernel<128, MODE><<<grid, NTHR, 0, s>>>(a);
  else
    attn_mma_kernel<64, MODE><<<grid, NTHR, 0, s>>>(a);
  return cudaGetLastError();
}

__global__ void hidden_log_norm_kernel(const bf16_t* __restrict__ h, int rows, int Dh,
                                       float* __restrict__ out) {
  const int wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wg >= rows) return;
  const bf16_t* p = h + (size_t)wg * Dh;
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
  s = warp_sum(s);
  if (lane == 0) out[wg] = 0.5f * logf(s);
}

}  // namespace

cudaError_t launch_lse(const AttnArgs& a, cudaStream_t s) { return launch_mode<kLse>(a, s); }
cudaError_t launch_score_max(const AttnArgs& a, cudaStream_t s) { return launch_mode<kMax>(a, s); }
cudaError_t launch_future_sum(const AttnArgs& a, cudaStream_t s) {
  return launch_mode<kFuture>(a, s);
}

cudaError_t launch_hidden_log_norm(const bf16_t* h, int L, int n, int Dh, float* hlog,
                                   cudaStream_t s) {
  const int rows = L * n;
  if (rows == 0) return cudaSuccess;
  count_launches(1);
  hidden_log_norm_kernel<<<(rows + 7) / 8, 256, 0, s>>>(h, rows, Dh, hlog);
  return cudaGetLastError();
}

}  // namespace kvs
