// Value factor of KVzip+ (KVzap review, 3.2 Eq. 2/Eq. 3): ||W_O^{(h)} v_i||_2.
//
// Computed through the Gram matrix of each head's output-projection slice:
//   G_h = W_h^T W_h   (d x d; W_h = o_proj.weight[:, h*d:(h+1)*d], D_h x d)
//   ||W_h v||^2 = v^T G_h v
// which costs 2 D_h d^2 + 4 T d^2 flops per head instead of 2 T d D_h for the direct
// product (5x fewer at D_h = 1536, T = 2048; 14x fewer at D_h = 4096, T = 32768).
// Both contractions run on warp MMAs (bf16 in, fp32 accumulate):
//   gram  G = W_h^T W_h, operands read transposed with ldmatrix.trans; G is stored as a
//         bf16 pair G = G_hi + G_lo (G_lo = bf16(G - G_hi)), exact to ~2^-17 |G|
//   quad  u = V (G_hi + G_lo) for a tile of tokens, then v_i . u_i in the epilogue
#include <mutex>

#include "common.cuh"
#include "vnorm.cuh"

namespace kvs {
namespace {

constexpr int kKc = 32;  // rows of W_h per pipeline stage

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint16_t f2bf(float x) {  // round to nearest even
  const uint32_t u = __float_as_uint(x);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

// One block per (head, layer): 8 warps as 4 (M) x 2 (N), each a 32 x 64 tile of the
// 128 x 128 Gram matrix (D = 128), or 16 x 32 for D = 64.  K = D_h streams through a
// double-buffered cp.async ring of kKc-row slices of W_h.
template <int D>
__global__ void __launch_bounds__(256) gram_mma_kernel(const bf16_t* __restrict__ w_o, int Dh,
                                                       int Hq, bf16_t* __restrict__ G) {
  constexpr int MT = D / 64;      // m16 tiles per warp (2 for D=128)
  constexpr int NT = D / 16;      // n8 tiles per warp (8 for D=128)
  constexpr int LD = D + 8;
  __shared__ __align__(16) bf16_t ws[2][kKc][LD];
  const int hq = blockIdx.x, l = blockIdx.y, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int wm = warp >> 1, wn = warp & 1;
  const int m0 = wm * (D / 4), n0 = wn * (D / 2);
  const bf16_t* base = w_o + (size_t)l * Dh * Hq * D + (size_t)hq * D;

  auto issue = [&](int r0, int buf) {
    for (int idx = tid; idx < kKc * D / 8; idx += 256) {
      const int r = idx / (D / 8), c = (idx % (D / 8)) * 8;
      const bool ok = r0 + r < Dh;
      cp_async16(smem_u32(&ws[buf][r][c]), ok ? base + (size_t)(r0 + r) * Hq * D + c : base,
                 ok ? 16 : 0);
    }
  };

  float acc[MT][NT][4];
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[i][j][0] = acc[i][j][1] = acc[i][j][2] = acc[i][j][3] = 0.f;

  const int nchunks = (Dh + kKc - 1) / kKc;
  issue(0, 0);
  cp_async_commit();
  for (int ch = 0; ch < nchunks; ++ch) {
    const int buf = ch & 1;
    if (ch + 1 < nchunks) {
      issue((ch + 1) * kKc, buf ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int kc = 0; kc < kKc; kc += 16) {
      // A = W^T: rows of the stored tile are k; .trans gives A[m][k] fragments
      uint32_t af[MT][4];
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const int mat = lane >> 3, rr = lane & 7;
        const int k = kc + (mat >> 1) * 8 + rr;
        const int m = m0 + i * 16 + (mat & 1) * 8;
        ldmatrix_x4_trans(smem_u32(&ws[buf][k][m]), af[i][0], af[i][1], af[i][2], af[i][3]);
      }
#pragma unroll
      for (int j = 0; j < NT; j += 2) {
        // B = W: matrices (k0, n), (k0+8, n), (k0, n+8), (k0+8, n+8)
        const int mat = lane >> 3, rr = lane & 7;
        const int k = kc + (mat & 1) * 8 + rr;
        const int n = n0 + j * 8 + (mat >> 1) * 8;
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(smem_u32(&ws[buf][k][n]), b0, b1, b2, b3);
#pragma unroll
        for (int i = 0; i < MT; ++i) {
          mma_bf16_16816(acc[i][j], af[i], b0, b1);
          mma_bf16_16816(acc[i][j + 1], af[i], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  bf16_t* Gh = G + ((size_t)l * Hq + hq) * 2 * D * D;  // [hi: D x D][lo: D x D]
#pragma unroll
  for (int i = 0; i < MT; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = m0 + i * 16 + g + (e >> 1) * 8;
        const int col = n0 + j * 8 + 2 * t4 + (e & 1);
        const float x = acc[i][j][e];
        const uint16_t hi = f2bf(x);
        const uint16_t lo = f2bf(x - __uint_as_float((uint32_t)hi << 16));
        Gh[row * D + col] = hi;
        Gh[D * D + row * D + col] = lo;
      }
}

// vn = sqrt(v^T (G_hi + G_lo) v) for 128-token tiles (32 per warp, two m16 tiles that
// share every G fragment); G_hi, G_lo (bf16, symmetric, so their rows serve directly as
// the k-contiguous B operand) stay in shared memory while the block walks kTokTiles
// consecutive token tiles of one (layer, query head).
constexpr int kTokTiles = 4;
constexpr int kQuadTok = 128;

template <int D>
__global__ void __launch_bounds__(128) quad_mma_kernel(const bf16_t* __restrict__ v,
                                                       const bf16_t* __restrict__ G, int T,
                                                       int Hq, int Hkv, float* __restrict__ vn) {
  constexpr int LD = D + 8;
  extern __shared__ __align__(16) uint8_t qsm[];
  bf16_t(*gs)[LD] = reinterpret_cast<bf16_t(*)[LD]>(qsm);                   // [2D][LD]
  bf16_t(*vs)[LD] = reinterpret_cast<bf16_t(*)[LD]>(qsm + 2 * D * LD * 2);  // [128][LD]
  const int hq = blockIdx.y, l = blockIdx.z, tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t4 = lane & 3;
  const int hk = hq / (Hq / Hkv);
  const bf16_t* Gh = G + ((size_t)l * Hq + hq) * 2 * D * D;
  for (int idx = tid; idx < 2 * D * D / 8; idx += 128) {
    const int r = idx / (D / 8), c = (idx % (D / 8)) * 8;
    cp_async16(smem_u32(&gs[r][c]), Gh + (size_t)r * D + c, 16);
  }
  cp_async_commit();
  const bf16_t* vb = v + (size_t)(l * Hkv + hk) * T * D;
  for (int tt = 0; tt < kTokTiles; ++tt) {
    const int i0 = (blockIdx.x * kTokTiles + tt) * kQuadTok;
    if (i0 >= T) break;
    for (int idx = tid; idx < kQuadTok * D / 8; idx += 128) {
      const int r = idx / (D / 8), c = (idx % (D / 8)) * 8;
      const bool ok = i0 + r < T;
      cp_async16(smem_u32(&vs[r][c]), ok ? vb + (size_t)(i0 + r) * D + c : vb, ok ? 16 : 0);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    uint32_t af[2][D / 16][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int kc = 0; kc < D / 16; ++kc)
        ldmatrix_x4(smem_u32(&vs[warp * 32 + mt * 16 + (lane & 15)][kc * 16 + (lane >> 4) * 8]),
                    af[mt][kc][0], af[mt][kc][1], af[mt][kc][2], af[mt][kc][3]);
    float p[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll 1
    for (int nt = 0; nt < D / 8; ++nt) {
      float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int k2 = 0; k2 < D / 32; ++k2) {
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(smem_u32(&gs[half * D + nt * 8 + (lane & 7)][k2 * 32 + (lane >> 3) * 8]), b0,
                      b1, b2, b3);
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            mma_bf16_16816(acc[mt], af[mt][2 * k2], b0, b1);
            mma_bf16_16816(acc[mt], af[mt][2 * k2 + 1], b2, b3);
          }
        }
      }
      const int col = nt * 8 + 2 * t4;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint32_t va = *reinterpret_cast<const uint32_t*>(&vs[warp * 32 + mt * 16 + g][col]);
        const uint32_t vc = *reinterpret_cast<const uint32_t*>(&vs[warp * 32 + mt * 16 + g + 8][col]);
        p[mt][0] = fmaf(acc[mt][0], bf16_lo(va), fmaf(acc[mt][1], bf16_hi(va), p[mt][0]));
        p[mt][1] = fmaf(acc[mt][2], bf16_lo(vc), fmaf(acc[mt][3], bf16_hi(vc), p[mt][1]));
      }
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x = p[mt][hh];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        const int i = i0 + warp * 32 + mt * 16 + g + hh * 8;
        if (t4 == 0 && i < T) vn[((size_t)l * Hq + hq) * T + i] = sqrtf(fmaxf(x, 0.f));
      }
    __syncthreads();
  }
}

}  // namespace

size_t vnorm_workspace_bytes(int L, int Hq, int d) {
  return (size_t)L * Hq * 2 * d * d * sizeof(bf16_t);
}

cudaError_t launch_vnorm(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                         const bf16_t* w_o, float* vn, void* ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  bf16_t* G = static_cast<bf16_t*>(ws);
  dim3 gg(Hq, L);
  dim3 gq((T + kQuadTok * kTokTiles - 1) / (kQuadTok * kTokTiles), Hq, L);
  count_launches(2);
  if (d == 128) {
    constexpr size_t smem = (2 * 128 + kQuadTok) * (128 + 8) * 2;
    gram_mma_kernel<128><<<gg, 256, 0, s>>>(w_o, Dh, Hq, G);
    cudaFuncSetAttribute(quad_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    quad_mma_kernel<128><<<gq, 128, smem, s>>>(v, G, T, Hq, Hkv, vn);
  } else {
    constexpr size_t smem = (2 * 64 + kQuadTok) * (64 + 8) * 2;
    gram_mma_kernel<64><<<gg, 256, 0, s>>>(w_o, Dh, Hq, G);
    cudaFuncSetAttribute(quad_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    quad_mma_kernel<64><<<gq, 128, smem, s>>>(v, G, T, Hq, Hkv, vn);
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------------ allocation-free variant
//
// Some callers of this library cannot allocate device memory for the Gram scratch:
// code that runs as a plugin inside a host framework which owns every device
// allocation (its caching allocator and memory accounting must see all of them), and
// latency-critical serving loops that forbid allocation, with its implicit
// synchronisation, after warm-up.  For them the value norm can use a scratch buffer
// built into the library: a file-scope device array of kNoAllocScratchBytes, which
// every GPU that loads the library holds until the process exits.  The layers are
// processed one after another on the caller's stream, each reusing the array, so the
// limit is one layer's Gram matrices: H_q * d * d * 4 bytes <= kNoAllocScratchBytes
// (H_q <= 128 at d = 128).  The array keeps the last call's contents; the Gram kernel
// overwrites every byte a call reads, so nothing needs clearing, but calls that overlap
// on the GPU (different streams, or different host threads) race on it.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_vnorm_scratch[kNoAllocScratchBytes];
constexpr int kMaxDevices = 64;
}  // namespace

size_t vnorm_noalloc_scratch_bytes() { return kNoAllocScratchBytes; }

// Device address of the built-in scratch on the current device, looked up once per
// device (the first call on a device does the lookup, so it must not be made while a
// stream is being captured).
static cudaError_t vnorm_noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_vnorm_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
  }
  *out = addr[dev];
  return cudaSuccess;
}

cudaError_t launch_vnorm_noalloc(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                                 const bf16_t* w_o, float* vn, cudaStream_t s) {
  void* scratch = nullptr;
  cudaError_t e = vnorm_noalloc_scratch(&scratch);
  if (e != cudaSuccess) return e;
  for (int l = 0; l < L && e == cudaSuccess; ++l)
    e = launch_vnorm(v + (size_t)l * Hkv * T * d, 1, Hq, Hkv, d, T, Dh,
                     w_o + (size_t)l * Dh * Hq * d, vn + (size_t)l * Hq * T, scratch, s);
  return e;
}

}  // namespace kvs
