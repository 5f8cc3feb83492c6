// KVzap-Linear surrogate score (KVzap review, 3.3; Algorithm 1 step 1), optionally
// fused with the threshold rule and sliding window (KVzap review, thresholding):
//   z[l][hk][t] = sum_c h[l][t][c] W[l][c][hk] + b[l][hk]
//   mask = z >= tau || t >= T - w;  keep[l][hk] = count
//
// The op streams h (D_h bf16 per token, 8 KiB at D_h = 4096) once and is bound by
// HBM bandwidth.  At 8 flop per byte an fp32 CUDA-core dot product would need ~75%
// of the FMA issue rate just to keep up with HBM, so the per-token contraction
// against the D_h x H_kv weight runs on warp MMAs (m16n8k16, N = 8 heads).  Each lane
// loads 16-byte pieces of two token rows with non-allocating loads and feeds them to
// the MMA directly as A fragments: the reduction runs over channels,
// so any channel permutation works as long as the B fragments (W, staged once per
// block in shared memory) use the same one.  No shared-memory staging of h.
#include <cooperative_groups.h>

#include "common.cuh"
#include "surrogate.cuh"

namespace kvs {
namespace {

constexpr int kWarps = 8;

struct SurArgs {
  const bf16_t* h;
  const bf16_t* W;
  const float* b;
  float* z;
  uint8_t* mask;
  int* keep;
  int T, Dh, Hkv, w, tiles_per_warp;
  float tau;
  int ksplit;  // 1: each warp owns whole token tiles; kWarps: the warps of a block split
               // the channels of one tile (few tokens, e.g. one per sequence in decode)
};

// Channel permutation: in superblock sb (128 channels), lane (g, t) (lane = 4*g + t) loads
// channels sb*128 + 32*p + 8*t + e (e = 0..7) of token rows g and g+8 for p = 0..3, so the
// four lanes of a row read 64 contiguous bytes per load instruction (two full sectors).
// MMA 2p takes e = 0..3 and MMA 2p+1 takes e = 4..7 as k-slots {2t, 2t+1, 2t+8, 2t+9}.
// Shared layout of W: [superblock][n-tile][p][lane] x 16 bytes, holding
// W[sb*128 + 32*p + 8*t + e][nt*8 + g] for e = 0..7: the same permutation.
template <int NT>
__global__ void __launch_bounds__(kWarps * 32) surrogate_kernel(const SurArgs a) {
  extern __shared__ uint4 wsm[];
  const int l = blockIdx.y;
  const int nsb = a.Dh / 128;
  const bf16_t* Wl = a.W + (size_t)l * a.Dh * a.Hkv;
  if (NT == 1 && a.Hkv == 8) {
    // 8 heads: a channel's weights are one 16-byte row.  Each thread reads the 8 rows of
    // one group of 8 channels (128 contiguous bytes) and writes its 8 x 8 transpose:
    // one 16-byte entry (8 channels of one head) per head
    for (int grp = threadIdx.x; grp < nsb * 16; grp += blockDim.x) {
      const int sb = grp >> 4, p = (grp >> 2) & 3, t = grp & 3;
      const uint4* src = reinterpret_cast<const uint4*>(Wl + (size_t)(sb * 128 + 32 * p + 8 * t) * 8);
      uint32_t r[8][4];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint4 u = __ldg(src + e);
        r[e][0] = u.x; r[e][1] = u.y; r[e][2] = u.z; r[e][3] = u.w;
      }
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        const int sh = (gg & 1) * 16;
        uint32_t wv[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
          wv[e2] = ((r[2 * e2][gg >> 1] >> sh) & 0xffffu) | (((r[2 * e2 + 1][gg >> 1] >> sh) & 0xffffu) << 16);
        wsm[(sb * 4 + p) * 32 + 4 * gg + t] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
  } else
  for (int idx = threadIdx.x; idx < nsb * NT * 128; idx += blockDim.x) {
    const int ln = idx & 31, p = (idx >> 5) & 3, nt = (idx >> 7) % NT, sb = (idx >> 7) / NT;
    const int head = nt * 8 + (ln >> 2);
    const int ch0 = sb * 128 + 32 * p + 8 * (ln & 3);
    uint32_t wv[4];
#pragma unroll
    for (int e2 = 0; e2 < 4; ++e2) {
      uint32_t lo = 0, hi = 0;
      if (head < a.Hkv) {
        lo = Wl[(size_t)(ch0 + 2 * e2) * a.Hkv + head];
        hi = Wl[(size_t)(ch0 + 2 * e2 + 1) * a.Hkv + head];
      }
      wv[e2] = lo | (hi << 16);
    }
    wsm[idx] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int ntile = (a.T + 15) / 16;
  const float* bl = a.b + (size_t)l * a.Hkv;
  int cnt[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) cnt[nt][0] = cnt[nt][1] = 0;

  // partial sums of the channel superblocks [sb0, sb1) of token tile t0
  auto contract = [&](int t0, int sb0, int sb1, float (*acc)[4]) {
    const int ra = min(t0 + g, a.T - 1), rb = min(t0 + g + 8, a.T - 1);
    const bf16_t* pa = a.h + ((size_t)l * a.T + ra) * a.Dh + 8 * t4;
    const bf16_t* pb = a.h + ((size_t)l * a.T + rb) * a.Dh + 8 * t4;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll 2
    for (int sb = sb0; sb < sb1; ++sb) {
      uint4 xa[4], xb[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        xa[p] = ld_nc_v4(pa + sb * 128 + 32 * p);
        xb[p] = ld_nc_v4(pb + sb * 128 + 32 * p);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const uint4 wv = wsm[((sb * NT + nt) * 4 + p) * 32 + lane];
          const uint32_t A0[4] = {xa[p].x, xb[p].x, xa[p].y, xb[p].y};
          mma_bf16_16816(acc[nt], A0, wv.x, wv.y);
          const uint32_t A1[4] = {xa[p].z, xb[p].z, xa[p].w, xb[p].w};
          mma_bf16_16816(acc[nt], A1, wv.z, wv.w);
        }
      }
    }
  };
  // bias, score store and the fused threshold of one finished tile
  auto finish = [&](int t0, float (*acc)[4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int head = nt * 8 + 2 * t4 + (e & 1);
        const int tok = t0 + g + (e >> 1) * 8;
        if (head < a.Hkv && tok < a.T) {
          const float zz = acc[nt][e] + bl[head];
          const size_t o = ((size_t)l * a.Hkv + head) * a.T + tok;
          a.z[o] = zz;
          if (a.mask) {
            const int kp = (zz >= a.tau) || (tok >= a.T - a.w);
            a.mask[o] = (uint8_t)kp;
            cnt[nt][e & 1] += kp;
          }
        }
      }
    }
  };

  if (a.ksplit > 1) {
    // one tile per block; warp w contracts the w-th slice of the channel superblocks and
    // warp 0 adds the slices up (fixed order: deterministic)
    float* red = reinterpret_cast<float*>(wsm + (size_t)nsb * NT * 128);
    const int t0 = blockIdx.x * 16;
    float acc[NT][4];
    contract(t0, warp * nsb / kWarps, (warp + 1) * nsb / kWarps, acc);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) red[((warp * NT + nt) * 4 + e) * 32 + lane] = acc[nt][e];
    __syncthreads();
    if (warp == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float sum = 0.f;
          for (int w8 = 0; w8 < kWarps; ++w8) sum += red[((w8 * NT + nt) * 4 + e) * 32 + lane];
          acc[nt][e] = sum;
        }
      finish(t0, acc);
    }
  } else {
    int tile = (blockIdx.x * kWarps + warp) * a.tiles_per_warp;
    for (int k = 0; k < a.tiles_per_warp && tile < ntile; ++k, ++tile) {
      float acc[NT][4];
      contract(tile * 16, 0, nsb, acc);
      finish(tile * 16, acc);
    }
  }
  if (a.mask) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        int c = cnt[nt][e2];
        c += __shfl_xor_sync(0xffffffffu, c, 4);
        c += __shfl_xor_sync(0xffffffffu, c, 8);
        c += __shfl_xor_sync(0xffffffffu, c, 16);
        const int head = nt * 8 + 2 * t4 + e2;
        if (g == 0 && head < a.Hkv && c) atomicAdd(a.keep + (size_t)l * a.Hkv + head, c);
      }
    }
  }
}

// W fragments of superblock sb for up to 8 heads (the B-operand layout of
// surrogate_kernel: entry (p, lane) = W[sb*128 + 32p + 8t + e][g] for e = 0..7, lane =
// 4g + t), written by one warp into dst[4 * 32].
__device__ __forceinline__ void stage_w_superblock(const bf16_t* Wl, int Hkv, int sb, uint4* dst,
                                                   int lane) {
  if (Hkv == 8) {
    // a channel's weights are one 16-byte row: lanes 0..15 each read the 8 rows of one
    // group of 8 channels and write their 8 x 8 transpose
    if (lane < 16) {
      const int p = lane >> 2, t = lane & 3;
      const uint4* src = reinterpret_cast<const uint4*>(Wl + (size_t)(sb * 128 + 32 * p + 8 * t) * 8);
      uint32_t r[8][4];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint4 u = __ldg(src + e);
        r[e][0] = u.x; r[e][1] = u.y; r[e][2] = u.z; r[e][3] = u.w;
      }
#pragma unroll
      for (int gg = 0; gg < 8; ++gg) {
        const int sh = (gg & 1) * 16;
        uint32_t wv[4];
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
          wv[e2] = ((r[2 * e2][gg >> 1] >> sh) & 0xffffu) | (((r[2 * e2 + 1][gg >> 1] >> sh) & 0xffffu) << 16);
        dst[p * 32 + 4 * gg + t] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
    }
  } else {
    for (int idx = lane; idx < 4 * 32; idx += 32) {
      const int ln = idx & 31, p = idx >> 5, head = ln >> 2;
      const int ch0 = sb * 128 + 32 * p + 8 * (ln & 3);
      uint32_t wv[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        uint32_t lo = 0, hi = 0;
        if (head < Hkv) {
          lo = Wl[(size_t)(ch0 + 2 * e2) * Hkv + head];
          hi = Wl[(size_t)(ch0 + 2 * e2 + 1) * Hkv + head];
        }
        wv[e2] = lo | (hi << 16);
      }
      dst[idx] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  }
  __syncwarp();
}

// Few tokens (decode: one per sequence), up to 8 heads: a cluster of kSplit blocks per
// (layer, 16-token tile) splits the channels.  Block rank r takes superblocks
// [r nsb / kSplit, (r+1) nsb / kSplit), its warps one superblock at a time (each stages
// only that superblock's W, 2 KB); the warps' partial sums meet in shared memory and the
// blocks' partials in the rank-0 block's shared memory (distributed shared memory),
// which adds them in rank order (deterministic) and applies bias, threshold and window.
constexpr int kSplit = 4;
__global__ void __cluster_dims__(kSplit, 1, 1) __launch_bounds__(kWarps * 32)
    surrogate_split_kernel(const SurArgs a) {
  namespace cg = cooperative_groups;
  __shared__ uint4 wst[kWarps][4 * 32];          // per warp: one superblock's W fragments
  __shared__ float red[kWarps][4][32];            // per warp partial sums
  __shared__ float cred[kSplit][4][32];           // rank 0: the blocks' partial sums
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int l = blockIdx.y, t0 = (blockIdx.x / kSplit) * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int nsb = a.Dh / 128;
  const bf16_t* Wl = a.W + (size_t)l * a.Dh * a.Hkv;
  const int ra = min(t0 + g, a.T - 1), rb = min(t0 + g + 8, a.T - 1);
  const bf16_t* pa = a.h + ((size_t)l * a.T + ra) * a.Dh + 8 * t4;
  const bf16_t* pb = a.h + ((size_t)l * a.T + rb) * a.Dh + 8 * t4;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int sb = rank * nsb / kSplit + warp; sb < (rank + 1) * nsb / kSplit; sb += kWarps) {
    uint4 xa[4], xb[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {  // issue the token loads before staging W
      xa[p] = ld_nc_v4(pa + sb * 128 + 32 * p);
      xb[p] = ld_nc_v4(pb + sb * 128 + 32 * p);
    }
    stage_w_superblock(Wl, a.Hkv, sb, wst[warp], lane);
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint4 wv = wst[warp][p * 32 + lane];
      const uint32_t A0[4] = {xa[p].x, xb[p].x, xa[p].y, xb[p].y};
      mma_bf16_16816(acc, A0, wv.x, wv.y);
      const uint32_t A1[4] = {xa[p].z, xb[p].z, xa[p].w, xb[p].w};
      mma_bf16_16816(acc, A1, wv.z, wv.w);
    }
    __syncwarp();  // wst[warp] is restaged for the next superblock
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) red[warp][e][lane] = acc[e];
  __syncthreads();
  if (warp == 0) {
    float* dst = cluster.map_shared_rank(&cred[0][0][0], 0);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float sum = 0.f;
      for (int w8 = 0; w8 < kWarps; ++w8) sum += red[w8][e][lane];
      dst[(rank * 4 + e) * 32 + lane] = sum;
    }
  }
  cluster.sync();  // every block reaches it once: the partials are in rank 0
  if (rank != 0 || warp != 0) return;
  const float* bl = a.b + (size_t)l * a.Hkv;
  int cnt[2] = {0, 0};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float zz = 0.f;
    for (int r = 0; r < kSplit; ++r) zz += cred[r][e][lane];
    const int head = 2 * t4 + (e & 1), tok = t0 + g + (e >> 1) * 8;
    if (head < a.Hkv && tok < a.T) {
      zz += bl[head];
      const size_t o = ((size_t)l * a.Hkv + head) * a.T + tok;
      a.z[o] = zz;
      if (a.mask) {
        const int kp = (zz >= a.tau) || (tok >= a.T - a.w);
        a.mask[o] = (uint8_t)kp;
        cnt[e & 1] += kp;
      }
    }
  }
  if (a.mask) {
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      int c = cnt[e2];
      c += __shfl_xor_sync(0xffffffffu, c, 4);
      c += __shfl_xor_sync(0xffffffffu, c, 8);
      c += __shfl_xor_sync(0xffffffffu, c, 16);
      const int head = 2 * t4 + e2;
      if (g == 0 && head < a.Hkv && c) atomicAdd(a.keep + (size_t)l * a.Hkv + head, c);
    }
  }
}

}  // namespace

size_t surrogate_smem_bytes(int Dh, int Hkv) { return (size_t)Dh * ((Hkv + 7) / 8) * 16; }

cudaError_t launch_surrogate(const bf16_t* h, int L, int T, int Dh, int Hkv, const bf16_t* W,
                             const float* b, float* z, float tau, int w, uint8_t* mask,
                             int* keep, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (mask) {
    cudaError_t e = cudaMemsetAsync(keep, 0, sizeof(int) * (size_t)L * Hkv, s);
    if (e != cudaSuccess) return e;
  }
  SurArgs a{h, W, b, z, mask, keep, T, Dh, Hkv, w, 8, tau, 1};
  const int ntile = (T + 15) / 16;
  // few token tiles (decode: one token per sequence): split each tile's channels over
  // the blocks of a cluster (up to 8 heads) or the warps of a block, instead of leaving
  // most of the GPU idle
  if ((long)L * ntile < 304) {
    if (Hkv <= 8 && Dh % (128 * kSplit) == 0) {
      count_launches(1);
      surrogate_split_kernel<<<dim3(ntile * kSplit, L), kWarps * 32, 0, s>>>(a);
      return cudaGetLastError();
    }
    a.ksplit = kWarps;
  }
  // fewer tiles per warp when the grid would not fill the GPU twice over
  while (a.tiles_per_warp > 1 &&
         (long)L * ((ntile + kWarps * a.tiles_per_warp - 1) / (kWarps * a.tiles_per_warp)) < 304)
    a.tiles_per_warp >>= 1;
  dim3 grid(a.ksplit > 1 ? ntile : (ntile + kWarps * a.tiles_per_warp - 1) /
                                        (kWarps * a.tiles_per_warp), L);
  size_t smem = surrogate_smem_bytes(Dh, Hkv);
  if (a.ksplit > 1) smem += (size_t)kWarps * ((Hkv + 7) / 8) * 4 * 32 * sizeof(float);
  count_launches(1);
  if (Hkv <= 8) {
    cudaFuncSetAttribute(surrogate_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    surrogate_kernel<1><<<grid, kWarps * 32, smem, s>>>(a);
  } else {
    cudaFuncSetAttribute(surrogate_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    surrogate_kernel<2><<<grid, kWarps * 32, smem, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kvs
