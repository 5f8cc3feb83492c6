// Value factor of KVzip+ (KVzap review, 3.2 Eq. 2/Eq. 3): ||W_O^{(h)} v_i||_2.
//
// Computed through the Gram matrix of each head's output-projection slice:
//   G_h = W_h^T W_h   (d x d; W_h = o_proj.weight[:, h*d:(h+1)*d], D_h x d)
//   ||W_h v||^2 = v^T G_h v
// which costs 2 D_h d^2 + 4 T d^2 flops per head instead of 2 T d D_h for the direct
// product (5x fewer at D_h = 1536, T = 2048; 14x fewer at D_h = 4096, T = 32768).
// Both contractions run on the tcgen05 tensor cores (bf16 in, fp32 accumulate):
//   gram  G = W_h^T W_h, the diagonal d x d blocks of W_O^T W_O (gram_tc.cu, both operands
//         MN-major straight from o_proj.weight); G is stored as a bf16 pair
//         G = G_hi + G_lo (G_lo = bf16(G - G_hi)), ~2^-17 |G| exact
//   quad  [V G_hi | V G_lo] for 128-token tiles on tcgen05 (the scoring kernel's kQuad
//         mode: one M=128 N=256 MMA chain per query head), then v_i . u_i per token
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "attn.cuh"
#include "common.cuh"
#include "gram.cuh"
#include "vnorm.cuh"

namespace kvs {

size_t vnorm_workspace_bytes(int L, int Hq, int d) {
  return (size_t)L * Hq * 2 * d * d * sizeof(bf16_t);
}

cudaError_t launch_vnorm(const bf16_t* v, int L, int Hq, int Hkv, int d, int T, int Dh,
                         const bf16_t* w_o, float* vn, void* ws, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  bf16_t* G = static_cast<bf16_t*>(ws);
  // G_h = W_h^T W_h for every head: the diagonal d x d blocks of W_O^T W_O on tcgen05,
  // written as bf16 hi/lo pairs
  GramArgs g;
  g.x = w_o; g.pair = G; g.pair_d = d;
  g.batch = L; g.rows = Dh; g.M = Hq * d; g.ldx = Hq * d;
  cudaError_t e = launch_gram(g, s);
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

// The driver's current-context calls, fetched through the runtime (the library links no
// driver library directly).
struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

static const CtxFns& ctx_fns() {
  static CtxFns f = [] {
    CtxFns r;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      r.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      r.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return r;
  }();
  return f;
}

// Unique id of the calling thread's current CUDA context (0 when there is none yet).
// Context ids are never reused within a process, unlike context handles.
static cudaError_t current_ctx_id(unsigned long long* id) {
  const CtxFns& f = ctx_fns();
  if (!f.get_current || !f.get_id) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS) return cudaErrorUnknown;
  *id = 0;
  if (ctx && f.get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorUnknown;
  return cudaSuccess;
}

// Device address of the built-in scratch in the current context.  It is looked up on
// the first call in each context and cached with that context's id; a call in a new
// context (another device, or the same device after cudaDeviceReset re-created its
// context) looks it up again.  A lookup must not happen while a stream is being captured.
static cudaError_t vnorm_noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  e = current_ctx_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || id == 0 || ctx_of[dev] != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_vnorm_scratch);  // makes the device's context current
    if (e != cudaSuccess) return e;
    e = current_ctx_id(&id);
    if (e != cudaSuccess) return e;
    addr[dev] = p;
    ctx_of[dev] = id;
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
