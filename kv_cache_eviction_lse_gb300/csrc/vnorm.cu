// Value factor of KVzip+ (KVzap review, 3.2 Eq. 2/Eq. 3): ||W_O^{(h)} v_i||_2.
//
// Computed through the Gram matrix of each head's output-projection slice:
//   G_h = W_h^T W_h   (d x d; W_h = o_proj.weight[:, h*d:(h+1)*d], D_h x d)
//   ||W_h v||^2 = v^T G_h v
// which costs 2 D_h d^2 + 4 T d^2 flops per head instead of 2 T d D_h for the direct
// product (5x fewer at D_h = 1536, T = 2048; 14x fewer at D_h = 4096, T = 32768).
// Both contractions run on tensor cores (bf16 in, fp32 accumulate):
//   gram  G = W_h^T W_h on warp MMAs, operands read transposed with ldmatrix.trans; G is
//         stored as a bf16 pair G = G_hi + G_lo (G_lo = bf16(G - G_hi)), ~2^-17 |G| exact
//   quad  [V G_hi | V G_lo] for 128-token tiles on tcgen05 (the scoring kernel's kQuad
//         mode: one M=128 N=256 MMA chain per query head), then v_i . u_i per token
#include <mutex>

#include "attn.cuh"
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

}  // namespace

size_t vnorm_workspace_bytes(int L, int Hq, int d) {
  return (size_t)L * Hq * 2 * d * d * sizeof(bf16_t);
}

cudaError_t launch_vnorm(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                         const bf16_t* w_o, float* vn, void* ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  bf16_t* G = static_cast<bf16_t*>(ws);
  dim3 gg(Hq, L);
  count_launches(1);
  if (d == 128)
    gram_mma_kernel<128><<<gg, 256, 0, s>>>(w_o, Dh, Hq, G);
  else
    gram_mma_kernel<64><<<gg, 256, 0, s>>>(w_o, Dh, Hq, G);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  AttnArgs a;  // quadratic form on the tensor cores (tcgen05), see attn_tc.cu
  a.k_ctx = v;
  a.gpair = G;
  a.out = vn;
  a.L = L; a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.T = T;
  return launch_vnorm_quad(a, s);
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
