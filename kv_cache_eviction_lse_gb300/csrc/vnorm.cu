// Value factor of KVzip+ (KVzap review, 3.2 Eq. 2/Eq. 3): ||W_O^{(h)} v_i||_2.
//
// Computed through the Gram matrix of each head's output-projection slice:
//   G_h = W_h^T W_h  (d x d, fp32; W_h = o_proj.weight[:, h*d:(h+1)*d], D_h x d)
//   ||W_h v||^2 = v^T G_h v
// which costs 2 D_h d^2 + 2 T d^2 flops per head instead of 2 T d D_h for the direct
// product (7x fewer at D_h=1536, T=2048; 28x fewer at D_h=4096, T=32768).
#include "common.cuh"
#include "vnorm.cuh"

namespace kvs {
namespace {

constexpr int kGramRows = 32;

// G[l][hq] = W_h^T W_h.  One block per (head, layer); 256 threads each own a
// (D/16 x D/16) block of G and stream the D_h rows of W_h through shared memory.
template <int D>
__global__ void __launch_bounds__(256) gram_kernel(const bf16_t* __restrict__ w_o, int Dh,
                                                   int Hq, float* __restrict__ G) {
  constexpr int TB = D / 16;
  __shared__ __align__(16) float ws[kGramRows][D];
  const int hq = blockIdx.x, l = blockIdx.y, tid = threadIdx.x;
  const int ta = tid / 16, tb = tid % 16;
  const bf16_t* base = w_o + (size_t)l * Dh * Hq * D + (size_t)hq * D;
  float acc[TB][TB];
#pragma unroll
  for (int i = 0; i < TB; ++i)
#pragma unroll
    for (int j = 0; j < TB; ++j) acc[i][j] = 0.f;

  for (int r0 = 0; r0 < Dh; r0 += kGramRows) {
    for (int idx = tid; idx < kGramRows * D / 8; idx += 256) {
      const int r = idx / (D / 8), c = (idx % (D / 8)) * 8;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (r0 + r < Dh) u = ld_nc_v4(base + (size_t)(r0 + r) * Hq * D + c);
      float4* dst = reinterpret_cast<float4*>(&ws[r][c]);
      dst[0] = make_float4(bf16_lo(u.x), bf16_hi(u.x), bf16_lo(u.y), bf16_hi(u.y));
      dst[1] = make_float4(bf16_lo(u.z), bf16_hi(u.z), bf16_lo(u.w), bf16_hi(u.w));
    }
    __syncthreads();
#pragma unroll 4
    for (int r = 0; r < kGramRows; ++r) {
      float va[TB], vb[TB];
#pragma unroll
      for (int i = 0; i < TB; ++i) {
        va[i] = ws[r][ta * TB + i];
        vb[i] = ws[r][tb * TB + i];
      }
#pragma unroll
      for (int i = 0; i < TB; ++i)
#pragma unroll
        for (int j = 0; j < TB; ++j) acc[i][j] = fmaf(va[i], vb[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* Gh = G + ((size_t)l * Hq + hq) * D * D;
#pragma unroll
  for (int i = 0; i < TB; ++i)
#pragma unroll
    for (int j = 0; j < TB; ++j) Gh[(ta * TB + i) * D + tb * TB + j] = acc[i][j];
}

// vn[l][hq][i] = sqrt(v_i^T G_hq v_i); one token per thread, v_i in registers, G in
// shared memory (read as broadcasts).
template <int D>
__global__ void __launch_bounds__(128) quad_kernel(const bf16_t* __restrict__ v,
                                                   const float* __restrict__ G, int T, int Hq,
                                                   int Hkv, float* __restrict__ vn) {
  extern __shared__ float4 gs4[];
  const int hq = blockIdx.y, l = blockIdx.z;
  const int hk = hq / (Hq / Hkv);
  const float4* Gh = reinterpret_cast<const float4*>(G + ((size_t)l * Hq + hq) * D * D);
  for (int idx = threadIdx.x; idx < D * D / 4; idx += blockDim.x) gs4[idx] = Gh[idx];
  __syncthreads();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T) return;
  const bf16_t* vp = v + ((size_t)(l * Hkv + hk) * T + i) * D;
  float x[D];
#pragma unroll
  for (int c = 0; c < D; c += 8) {
    const uint4 u = ld_nc_v4(vp + c);
    x[c + 0] = bf16_lo(u.x); x[c + 1] = bf16_hi(u.x);
    x[c + 2] = bf16_lo(u.y); x[c + 3] = bf16_hi(u.y);
    x[c + 4] = bf16_lo(u.z); x[c + 5] = bf16_hi(u.z);
    x[c + 6] = bf16_lo(u.w); x[c + 7] = bf16_hi(u.w);
  }
  float acc = 0.f;
#pragma unroll 1
  for (int a2 = 0; a2 < D; ++a2) {
    const float4* Ga = gs4 + a2 * (D / 4);
    float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
    for (int b4 = 0; b4 < D / 4; ++b4) {
      const float4 gg = Ga[b4];
      u0 = fmaf(gg.x, x[4 * b4 + 0], u0);
      u1 = fmaf(gg.y, x[4 * b4 + 1], u1);
      u2 = fmaf(gg.z, x[4 * b4 + 2], u2);
      u3 = fmaf(gg.w, x[4 * b4 + 3], u3);
    }
    const float xa = __uint_as_float(static_cast<uint32_t>(vp[a2]) << 16);
    acc = fmaf(xa, (u0 + u1) + (u2 + u3), acc);
  }
  vn[((size_t)l * Hq + hq) * T + i] = sqrtf(fmaxf(acc, 0.f));
}

}  // namespace

size_t vnorm_workspace_bytes(int L, int Hq, int d) { return (size_t)L * Hq * d * d * sizeof(float); }

cudaError_t launch_vnorm(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                         const bf16_t* w_o, float* vn, float* G, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dim3 gg(Hq, L);
  dim3 gq((T + 127) / 128, Hq, L);
  const size_t smem = (size_t)d * d * sizeof(float);
  count_launches(2);
  if (d == 128) {
    gram_kernel<128><<<gg, 256, 0, s>>>(w_o, Dh, Hq, G);
    cudaFuncSetAttribute(quad_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    quad_kernel<128><<<gq, 128, smem, s>>>(v, G, T, Hq, Hkv, vn);
  } else {
    gram_kernel<64><<<gg, 256, 0, s>>>(w_o, Dh, Hq, G);
    quad_kernel<64><<<gq, 128, smem, s>>>(v, G, T, Hq, Hkv, vn);
  }
  return cudaGetLastError();
}

}  // namespace kvs
