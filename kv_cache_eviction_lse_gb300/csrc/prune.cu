// Keep masks per (layer, KV head) row of scores.
//   threshold: keep t <=> score >= tau || t >= T - w     (KVzap review, thresholding;
//              Algorithm 1 sets the window scores to +inf and keeps scores >= threshold)
//   top-k:     keep the window plus the k best of the other T - w tokens
//              (KVpop review, 3. Method: per-head top-k within a fixed budget)
//   quantile:  threshold with tau_l = the lower nearest-rank quantile q of the layer's
//              non-window scores over all its KV heads (KVzip review, Methods: a
//              ratio-based threshold; the threshold rule as above)
// Top-k ranks by (score descending, position ascending) with NaN below everything;
// the k-th key is found by an exact 4-pass radix select on order-preserving 32-bit
// keys (shared-memory histograms), then ties at the k-th key go to the lowest
// positions via a block-wide ordered scan.  Deterministic, no sorting.  One launch
// selects any number (up to kMaxTopkBudgets) of budgets over the same scores.  The
// quantile's select runs the same radix passes over a whole layer, spread over many
// blocks per layer for long rows (one launch per digit).
#include <algorithm>

#include "common.cuh"
#include "prune.cuh"

namespace kvs {
namespace {

constexpr int kPruneThreads = 1024;
constexpr int kStageMaxT = 16384;  // rows staged in shared memory (64 KB of order keys)

// Order-preserving 32-bit key of a score: -0 and +0 get the same key (they compare equal,
// so a tie between them goes to the earlier position like any other tie).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = f == 0.f ? 0u : __float_as_uint(f);
  if (f != f) return 0u;  // NaN below -inf (whose key is 0x007fffff)
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Block-wide sum of an int (any block size that is a multiple of 32, <= 1024).
__device__ int block_sum(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum_int(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int r = lane < nw ? red[lane] : 0;
  if (warp == 0) r = warp_sum_int(r);
  if (threadIdx.x == 0) red[32] = r;
  __syncthreads();
  return red[32];
}

// Exclusive scan of a 0/1 flag over the block; returns the prefix, *total = sum.
__device__ int block_excl_scan_flag(bool f, int* red, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, f);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();
  if (lane == 0) red[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nw ? red[lane] : 0;
    int incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane < nw) red[lane] = incl - x;
    if (lane == 31) red[32] = incl;
  }
  __syncthreads();
  *total = red[32];
  return red[warp] + in_warp;
}

constexpr int kThrThreads = 256;
constexpr int kThrPer = 16;  // tokens per thread

// Grid (chunks of 4096 tokens, rows).  keep[row] must be zero on entry (the launcher
// clears it); each block adds its count with one atomic.
// With tau_l != NULL the threshold of row r is tau_l[r / rows_per_tau] (per layer).
__global__ void __launch_bounds__(kThrThreads) threshold_kernel(const float* __restrict__ score,
                                                                int T, float tau_c, int w,
                                                                const float* __restrict__ tau_l,
                                                                int rows_per_tau,
                                                                uint8_t* __restrict__ mask,
                                                                int* __restrict__ keep) {
  __shared__ int red[33];
  const size_t row = blockIdx.y;
  const float tau = tau_l ? tau_l[row / rows_per_tau] : tau_c;
  const float* s = score + row * T;
  uint8_t* m = mask + row * T;
  const int t0 = (blockIdx.x * kThrThreads + threadIdx.x) * kThrPer;
  int cnt = 0;
  if ((T & 15) == 0) {
    if (t0 < T) {
      uint32_t mb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(s + t0 + 4 * q);
        const float x[4] = {v.x, v.y, v.z, v.w};
        uint32_t word = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = t0 + 4 * q + e;
          const uint32_t k = (x[e] >= tau) || (t >= T - w);
          word |= k << (8 * e);
          cnt += (int)k;
        }
        mb[q] = word;
      }
      *reinterpret_cast<uint4*>(m + t0) = make_uint4(mb[0], mb[1], mb[2], mb[3]);
    }
  } else {
    for (int t = t0; t < min(t0 + kThrPer, T); ++t) {
      const int k = (s[t] >= tau) || (t >= T - w);
      m[t] = (uint8_t)k;
      cnt += k;
    }
  }
  cnt = block_sum(cnt, red);
  if (threadIdx.x == 0 && cnt) atomicAdd(keep + row, cnt);
}

// Float value of an order key (the inverse of order_key; key 0 is NaN).
__device__ __forceinline__ float key_value(uint32_t k) {
  if (k == 0u) return __uint_as_float(0x7fc00000u);
  return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k);
}

// One block per layer: tau[l] = the rank-r smallest (0-based, r = floor(q (N - 1))) of
// the layer's N = H_kv (T - w) non-window scores, NaN lowest, by an exact 4-pass radix
// select from the bottom (shared-memory histograms over order keys).  N = 0: +inf.
__global__ void __launch_bounds__(kPruneThreads) quantile_kernel(const float* __restrict__ score,
                                                                 int Hkv, int T, int w, float q,
                                                                 float* __restrict__ tau) {
  __shared__ unsigned hist[256];
  __shared__ uint32_t s_prefix;
  __shared__ long long s_rem;
  const int l = blockIdx.x;
  const int n = T - min(max(w, 0), T);
  const long long N = (long long)Hkv * n;
  if (N <= 0) {
    if (threadIdx.x == 0) tau[l] = __uint_as_float(0x7f800000u);
    return;
  }
  const float* s = score + (size_t)l * Hkv * T;
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_rem = (long long)floor((double)q * (double)(N - 1));
  }
  uint32_t hi_mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int h = 0; h < Hkv; ++h)
      for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const uint32_t u = order_key(s[(size_t)h * T + t]);
        if ((u & hi_mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l owns digits 8l .. 8l+7; find the digit at which the count of keys from the
      // bottom passes the remaining rank
      const int lane = threadIdx.x;
      long long c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[8 * lane + i];
        tot += c[i];
      }
      long long incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const long long r = s_rem;
      const unsigned hit = __ballot_sync(0xffffffffu, incl > r);
      const int src = __ffs(hit) - 1;  // first lane whose range passes rank r
      if (lane == src) {
        long long cum = incl - tot;
        int i = 0;
        for (; i < 7; ++i) {
          if (cum + c[i] > r) break;
          cum += c[i];
        }
        s_rem = r - cum;
        s_prefix = prefix | ((uint32_t)(8 * lane + i) << shift);
      }
    }
    hi_mask |= 255u << shift;
    __syncthreads();
  }
  if (threadIdx.x == 0) tau[l] = key_value(s_prefix);
}

// The same selection spread over many blocks per layer, one launch per 8-bit digit:
// block (h, b) of layer l histograms its part of row h (keys that match the digits
// already chosen) and stores the histogram; the block that finishes last (an atomic
// ticket, so nobody waits) adds the layer's histograms, picks the digit and the rank
// left inside it, and after the last digit writes tau[l].  The layer's mask rows, which
// the threshold pass rewrites afterwards, hold this state (16-byte aligned at the start
// of the layer's H_kv T mask bytes): the chosen prefix and remaining rank, then one
// 256-bin histogram per block.  keep[l H_kv] (zeroed before the first digit) counts the
// tickets and is zeroed again after the last.
constexpr int kQThreads = 256;
constexpr long long kQuantileMultiMin = 65536;  // fewer values: one block per layer
constexpr int kQuantilePerBlock = 4096;         // values per block (at least)
constexpr int kQuantileMaxSplit = 8;            // blocks per row (at most)

struct QuantileState {
  uint32_t prefix;
  uint32_t pad;
  long long rem;
};

__device__ __forceinline__ QuantileState* quantile_state(uint8_t* mask, int l, size_t slice) {
  uintptr_t p = reinterpret_cast<uintptr_t>(mask + (size_t)l * slice);
  p = (p + 15u) & ~(uintptr_t)15u;
  return reinterpret_cast<QuantileState*>(p);
}

__global__ void __launch_bounds__(kQThreads) quantile_digit_kernel(
    const float* __restrict__ score, int Hkv, int T, int w, float q, int split, int pass,
    float* __restrict__ tau, uint8_t* __restrict__ mask, int* __restrict__ keep) {
  __shared__ unsigned hist[256];
  __shared__ int s_last;
  const int l = blockIdx.y, blk = blockIdx.x, nblk = Hkv * split;
  const int h = blk / split, b = blk % split;
  const int n = T - min(max(w, 0), T);
  QuantileState* st = quantile_state(mask, l, (size_t)Hkv * T);
  unsigned* partial = reinterpret_cast<unsigned*>(st + 1);
  const int shift = 24 - 8 * pass;
  const uint32_t hi_mask = pass == 0 ? 0u : 0xffffffffu << (32 - 8 * pass);
  const uint32_t prefix = pass == 0 ? 0u : st->prefix;  // chosen by the previous launch
  const int tid = threadIdx.x;
  hist[tid] = 0u;
  __syncthreads();
  const int chunk = (n + split - 1) / split;
  const int t0 = b * chunk, t1 = min(n, t0 + chunk);
  const float* s = score + ((size_t)l * Hkv + h) * T;
  constexpr int kBatch = 8;  // loads in flight per thread before the histogram updates
  for (int tb = t0 + tid; tb < t1; tb += kBatch * kQThreads) {
    float x[kBatch];
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const int t = tb + e * kQThreads;
      x[e] = t < t1 ? __ldg(s + t) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < kBatch; ++e) {
      const uint32_t u = order_key(x[e]);
      if (tb + e * kQThreads < t1 && (u & hi_mask) == prefix)
        atomicAdd(&hist[(u >> shift) & 255u], 1u);
    }
  }
  __syncthreads();
  partial[(size_t)blk * 256 + tid] = hist[tid];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&keep[(size_t)l * Hkv], 1) == (pass + 1) * nblk - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  unsigned acc[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};  // eight loads in flight
  int i = 0;
  for (; i + 8 <= nblk; i += 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __ldcg(&partial[(size_t)(i + e) * 256 + tid]);
  }
  for (; i < nblk; ++i) acc[0] += __ldcg(&partial[(size_t)i * 256 + tid]);
  hist[tid] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
  __syncthreads();
  if (tid < 32) {
    // lane l owns digits 8l .. 8l+7; find the digit at which the count of keys from the
    // bottom passes the remaining rank
    const int lane = tid;
    long long c[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = hist[8 * lane + i];
      sum += c[i];
    }
    long long incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const long long N = (long long)Hkv * n;
    const long long r = pass == 0 ? (long long)floor((double)q * (double)(N - 1)) : st->rem;
    const unsigned hit = __ballot_sync(0xffffffffu, incl > r);
    const int src = __ffs(hit) - 1;  // first lane whose range passes rank r
    if (lane == src) {
      long long cum = incl - sum;
      int i = 0;
      for (; i < 7; ++i) {
        if (cum + c[i] > r) break;
        cum += c[i];
      }
      const uint32_t pre = prefix | ((uint32_t)(8 * lane + i) << shift);
      if (pass == 3) {
        tau[l] = key_value(pre);
        keep[(size_t)l * Hkv] = 0;
      } else {
        st->prefix = pre;
        st->rem = r - cum;
      }
    }
  }
}

// One block per (row, budget): grid (rows, n_budgets).  Rows of up to kStageMaxT scores
// are staged once in shared memory as order keys (the radix passes then read shared
// memory); longer rows are read from global memory in every pass.  The last radix pass
// also counts the candidates equal to the k-th key: when all of them are kept (no tie
// crosses the budget, the usual case) the mask is a plain u >= kth compare, written four
// tokens per store; otherwise the ties go to the lowest positions by an ordered scan.
// keep = min(k, T - w) + min(w, T) exactly: top-k keeps that many by construction.
__global__ void __launch_bounds__(kPruneThreads) topk_kernel(const float* __restrict__ score,
                                                             int rows, int T, TopkBudgets kb,
                                                             int w, uint8_t* __restrict__ mask,
                                                             int* __restrict__ keep) {
  extern __shared__ uint32_t keys_s[];
  __shared__ unsigned hist[256];
  __shared__ int red[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem, s_eq;
  const int b = blockIdx.y;
  const size_t row = blockIdx.x;
  const float* s = score + row * T;
  uint8_t* m = mask + ((size_t)b * rows + row) * T;
  const int wn = min(max(w, 0), T);
  const int n = T - wn;                    // candidate tokens (outside the window)
  const int kk = min(max(kb.k[b], 0), n);  // how many of them to keep
  const bool staged = T <= kStageMaxT;
  const bool vec = (T & 3) == 0;
  if (staged && kk > 0 && kk < n) {
    if (vec) {
      for (int t4 = threadIdx.x; 4 * t4 < n; t4 += blockDim.x) {
        const float4 x = *reinterpret_cast<const float4*>(s + 4 * t4);
        *reinterpret_cast<uint4*>(keys_s + 4 * t4) =
            make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
      }
    } else {
      for (int t = threadIdx.x; t < n; t += blockDim.x) keys_s[t] = order_key(s[t]);
    }
    __syncthreads();
  }
  auto key_at = [&](int t) -> uint32_t { return staged ? keys_s[t] : order_key(s[t]); };

  uint32_t kth = 0;  // key of the kk-th best candidate
  int rem = 0;       // how many candidates equal to kth to keep
  int eq_all = 0;    // how many candidates equal kth
  if (kk > 0 && kk < n) {
    if (threadIdx.x == 0) {
      s_prefix = 0u;
      s_rem = kk;
    }
    uint32_t hi_mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0u;
      __syncthreads();
      const uint32_t prefix = s_prefix;
      for (int t = threadIdx.x; t < n; t += blockDim.x) {
        const uint32_t u = key_at(t);
        if ((u & hi_mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l owns digits 255-8l .. 248-8l; find the digit at which the count of
        // keys from the top reaches the remaining rank
        const int lane = threadIdx.x;
        int c[8], tot = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          c[i] = (int)hist[255 - 8 * lane - i];
          tot += c[i];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const int r = s_rem;
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= r);
        const int src = __ffs(hit) - 1;  // first lane whose range reaches rank r
        if (lane == src) {
          int cum = incl - tot, i = 0;
          for (; i < 7; ++i) {
            if (cum + c[i] >= r) break;
            cum += c[i];
          }
          s_rem = r - cum;
          s_eq = c[i];  // after the last pass: the candidates whose key equals kth
          s_prefix = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
        }
      }
      hi_mask |= 255u << shift;
      __syncthreads();
    }
    kth = s_prefix;
    rem = s_rem;
    eq_all = s_eq;
  }
  if (threadIdx.x == 0) keep[(size_t)b * rows + row] = kk + wn;

  if (kk == 0 || kk == n || rem == eq_all) {
    // every candidate at or above the k-th key is kept (kk == n: all, kk == 0: none)
    const uint32_t lo = kk == 0 ? 0xffffffffu : kk == n ? 0u : kth;
    auto kept = [&](int t) -> uint32_t {
      if (t >= n) return 1u;
      if (kk == 0) return 0u;
      if (kk == n) return 1u;
      return key_at(t) >= lo ? 1u : 0u;
    };
    if (vec) {
      for (int t4 = threadIdx.x; 4 * t4 < T; t4 += blockDim.x) {
        const int t = 4 * t4;
        const uint32_t word = kept(t) | (kept(t + 1) << 8) | (kept(t + 2) << 16) | (kept(t + 3) << 24);
        *reinterpret_cast<uint32_t*>(m + t) = word;
      }
    } else {
      for (int t = threadIdx.x; t < T; t += blockDim.x) m[t] = (uint8_t)kept(t);
    }
    return;
  }

  // ties at the k-th key cross the budget: they go to the lowest positions
  int carry = 0;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    bool gt = false, eq = false;
    if (t < n) {
      const uint32_t u = key_at(t);
      gt = u > kth;
      eq = u == kth;
    }
    int tot;
    const int rank = block_excl_scan_flag(eq, red, &tot) + carry;
    carry += tot;
    if (t < T) m[t] = (uint8_t)((t >= n) || gt || (eq && rank < rem));
  }
}

}  // namespace

cudaError_t launch_prune(const float* score, int rows, int T, int mode, float tau, int k, int w,
                         uint8_t* mask, int* keep, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (mode == 0) {
    cudaError_t e = cudaMemsetAsync(keep, 0, sizeof(int) * (size_t)rows, s);
    if (e != cudaSuccess) return e;
    if (T == 0) return cudaSuccess;
    const int per_block = kThrThreads * kThrPer;
    count_launches(1);
    threshold_kernel<<<dim3((T + per_block - 1) / per_block, rows), kThrThreads, 0, s>>>(
        score, T, tau, w, nullptr, 1, mask, keep);
    return cudaGetLastError();
  }
  TopkBudgets kb;
  kb.k[0] = k;
  return launch_topk(score, rows, T, 1, kb, w, mask, keep, s);
}

cudaError_t launch_topk(const float* score, int rows, int T, int n_budgets, const TopkBudgets& kb,
                        int w, uint8_t* mask, int* keep, cudaStream_t s) {
  if (rows == 0 || n_budgets == 0) return cudaSuccess;
  if (n_budgets < 0 || n_budgets > kMaxTopkBudgets) return cudaErrorInvalidValue;
  const size_t smem = T <= kStageMaxT ? (size_t)T * sizeof(uint32_t) : 0;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)(kStageMaxT * sizeof(uint32_t)));
  if (e != cudaSuccess) return e;
  count_launches(1);
  topk_kernel<<<dim3(rows, n_budgets), kPruneThreads, smem, s>>>(score, rows, T, kb, w, mask, keep);
  return cudaGetLastError();
}

cudaError_t launch_prune_quantile(const float* score, int L, int Hkv, int T, float q, int w,
                                  float* tau, uint8_t* mask, int* keep, cudaStream_t s) {
  if (L == 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(keep, 0, sizeof(int) * (size_t)L * Hkv, s);
  if (e != cudaSuccess) return e;
  const int n = T - std::min(std::max(w, 0), T);
  const long long N = (long long)Hkv * n;
  if (N >= kQuantileMultiMin && n >= kQuantilePerBlock) {  // state fits in a quarter of the mask
    const int split = std::max(1, std::min(kQuantileMaxSplit, n / kQuantilePerBlock));
    count_launches(4);
    for (int pass = 0; pass < 4; ++pass)
      quantile_digit_kernel<<<dim3(Hkv * split, L), kQThreads, 0, s>>>(score, Hkv, T, w, q,
                                                                       split, pass, tau, mask, keep);
  } else {
    count_launches(1);
    quantile_kernel<<<L, kPruneThreads, 0, s>>>(score, Hkv, T, w, q, tau);
  }
  if (T == 0) return cudaGetLastError();
  const int per_block = kThrThreads * kThrPer;
  count_launches(1);
  threshold_kernel<<<dim3((T + per_block - 1) / per_block, L * Hkv), kThrThreads, 0, s>>>(
      score, T, 0.f, w, tau, Hkv, mask, keep);
  return cudaGetLastError();
}

}  // namespace kvs
