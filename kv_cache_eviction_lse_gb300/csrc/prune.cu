// Keep masks per (layer, KV head) row of scores.
//   threshold: keep t <=> score >= tau || t >= T - w     (KVzap review, thresholding;
//              Algorithm 1 sets the window scores to +inf and keeps scores >= threshold)
//   top-k:     keep the window plus the k best of the other T - w tokens
//              (KVpop review, 3. Method: per-head top-k within a fixed budget)
// Top-k ranks by (score descending, position ascending) with NaN below everything;
// the k-th key is found by an exact 4-pass radix select on order-preserving 32-bit
// keys (shared-memory histograms), then ties at the k-th key go to the lowest
// positions via a block-wide ordered scan.  Deterministic, no sorting.
#include "common.cuh"
#include "prune.cuh"

namespace kvs {
namespace {

constexpr int kPruneThreads = 1024;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f);
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
__global__ void __launch_bounds__(kThrThreads) threshold_kernel(const float* __restrict__ score,
                                                                int T, float tau, int w,
                                                                uint8_t* __restrict__ mask,
                                                                int* __restrict__ keep) {
  __shared__ int red[33];
  const size_t row = blockIdx.y;
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

__global__ void __launch_bounds__(kPruneThreads) topk_kernel(const float* __restrict__ score,
                                                             int T, int k, int w,
                                                             uint8_t* __restrict__ mask,
                                                             int* __restrict__ keep) {
  __shared__ unsigned hist[256];
  __shared__ int red[33];
  __shared__ uint32_t s_prefix;
  __shared__ int s_rem;
  const size_t row = blockIdx.x;
  const float* s = score + row * T;
  uint8_t* m = mask + row * T;
  const int wn = min(max(w, 0), T);
  const int n = T - wn;              // candidate tokens (outside the window)
  const int kk = min(max(k, 0), n);  // how many of them to keep

  uint32_t kth = 0;  // key of the kk-th best candidate
  int rem = 0;       // how many candidates equal to kth to keep
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
        const uint32_t u = order_key(s[t]);
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
          s_prefix = prefix | ((uint32_t)(255 - 8 * lane - i) << shift);
        }
      }
      hi_mask |= 255u << shift;
      __syncthreads();
    }
    kth = s_prefix;
    rem = s_rem;
  }

  int cnt = 0, carry = 0;
  for (int base = 0; base < T; base += blockDim.x) {
    const int t = base + threadIdx.x;
    bool gt = false, eq = false;
    if (t < n && kk > 0) {
      if (kk == n) {
        gt = true;
      } else {
        const uint32_t u = order_key(s[t]);
        gt = u > kth;
        eq = u == kth;
      }
    }
    int tot;
    const int rank = block_excl_scan_flag(eq, red, &tot) + carry;
    carry += tot;
    if (t < T) {
      const int kp = (t >= n) || gt || (eq && rank < rem);
      m[t] = (uint8_t)kp;
      cnt += kp;
    }
  }
  cnt = block_sum(cnt, red);
  if (threadIdx.x == 0) keep[row] = cnt;
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
        score, T, tau, w, mask, keep);
  } else {
    count_launches(1);
    topk_kernel<<<rows, kPruneThreads, 0, s>>>(score, T, k, w, mask, keep);
  }
  return cudaGetLastError();
}

}  // namespace kvs
