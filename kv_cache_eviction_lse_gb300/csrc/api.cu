// C ABI of the kvs library: argument validation, then launches on the caller's stream.
// Declarations and argument documentation: include/kvs.h.
#include <stdarg.h>
#include <stdio.h>

#include <atomic>
#include <string>

#include "../../include/kvs.h"
#include "attn.cuh"
#include "compact.cuh"
#include "decode.cuh"
#include "gram.cuh"
#include "mlp.cuh"
#include "prune.cuh"
#include "surrogate.cuh"
#include "vnorm.cuh"

namespace kvs {
static std::atomic<uint64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace kvs

namespace {

thread_local std::string g_last_error;

kvs_status fail(kvs_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

kvs_status ok() {
  g_last_error.clear();
  return KVS_OK;
}

kvs_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(KVS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define REQUIRE(cond, st, ...) \
  do {                         \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

#define REQUIRE_PTR(p)                                                       \
  do {                                                                       \
    if (!(p)) return fail(KVS_ERR_ARG, "%s: " #p " is NULL", __func__);      \
    if (!aligned16(p)) return fail(KVS_ERR_ALIGN, "%s: " #p " is not 16-byte aligned", __func__); \
  } while (0)

#define REQUIRE_OPT_PTR(p)                                                   \
  do {                                                                       \
    if ((p) && !aligned16(p))                                                \
      return fail(KVS_ERR_ALIGN, "%s: " #p " is not 16-byte aligned", __func__); \
  } while (0)

kvs_status check_dims(const kvs_dims* dm, const char* fn, bool need_heads = true) {
  if (!dm) return fail(KVS_ERR_ARG, "%s: dims is NULL", fn);
  if (dm->L < 1) return fail(KVS_ERR_SHAPE, "%s: L = %d must be >= 1", fn, dm->L);
  if (dm->H_kv < 1) return fail(KVS_ERR_SHAPE, "%s: H_kv = %d must be >= 1", fn, dm->H_kv);
  if (need_heads) {
    if (dm->H_q < 1 || dm->H_q % dm->H_kv)
      return fail(KVS_ERR_SHAPE, "%s: H_q = %d must be a positive multiple of H_kv = %d", fn,
                  dm->H_q, dm->H_kv);
    if (dm->d != 64 && dm->d != 128)
      return fail(KVS_ERR_UNSUPPORTED, "%s: head dim d = %d (supported: 64, 128)", fn, dm->d);
  }
  if (dm->L > 65535 || dm->H_q > 65535 || dm->H_kv > 65535)
    return fail(KVS_ERR_UNSUPPORTED, "%s: L/H_q/H_kv above 65535", fn);
  return KVS_OK;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

const char* kvs_version(void) { return "kvs 0.1.0 (sm_103a)"; }

const char* kvs_last_error(void) { return g_last_error.c_str(); }

uint64_t kvs_launch_count(void) { return kvs::g_launches.load(std::memory_order_relaxed); }

kvs_status kvs_device_error(int32_t* code_out, int32_t clear, void* stream) {
  REQUIRE(code_out, KVS_ERR_ARG, "kvs_device_error: code_out is NULL");
  int codes[6] = {0, 0, 0, 0, 0, 0};
  cudaError_t e = kvs::attn_device_error(&codes[0], clear != 0, as_stream(stream));
  if (e == cudaSuccess) e = kvs::mlp_device_error(&codes[1], clear != 0, as_stream(stream));
  if (e == cudaSuccess) e = kvs::fwd_device_error(&codes[2], clear != 0, as_stream(stream));
  if (e == cudaSuccess) e = kvs::decode_device_error(&codes[3], clear != 0, as_stream(stream));
  if (e == cudaSuccess) e = kvs::gram_device_error(&codes[4], clear != 0, as_stream(stream));
  if (e == cudaSuccess) e = kvs::chol_device_error(&codes[5], clear != 0, as_stream(stream));
  if (e != cudaSuccess) return cuda_status(e, "kvs_device_error");
  *code_out = 0;
  for (int c : codes)
    if (c && !*code_out) *code_out = c;
  return ok();
}

kvs_status kvs_lse(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q, const kvs_bf16* k_ctx,
                   int32_t T, const kvs_bf16* k_tail, int32_t n_tail, float* lse, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(n_q >= 0 && T >= 0 && n_tail >= 0, KVS_ERR_ARG, "kvs_lse: negative size");
  REQUIRE(n_q <= T + n_tail, KVS_ERR_SHAPE, "kvs_lse: n_q = %d exceeds keys T + n_tail = %d", n_q,
          T + n_tail);
  if (n_q == 0) return ok();
  REQUIRE_PTR(q);
  REQUIRE_PTR(lse);
  if (T > 0) REQUIRE_PTR(k_ctx);
  if (n_tail > 0) REQUIRE_PTR(k_tail);
  kvs::AttnArgs a;
  a.q = q; a.k_ctx = k_ctx; a.k_tail = k_tail; a.out = lse;
  a.L = dims->L; a.Hq = dims->H_q; a.Hkv = dims->H_kv; a.d = dims->d;
  a.n_q = n_q; a.T = T; a.n_tail = n_tail;
  return cuda_status(kvs::launch_lse(a, as_stream(stream)), "kvs_lse");
}

size_t kvs_score_max_workspace_size(const kvs_dims* dims, int32_t n_q, int32_t with_h) {
  if (!dims || n_q <= 0 || dims->L <= 0 || dims->H_q <= 0) return 0;
  (void)with_h;  // ln ||h_j|| is folded into the constants in the same pass: same size
  return kvs::score_max_ws_bytes(dims->L, dims->H_q, n_q);
}

kvs_status kvs_attn_fwd(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                        const kvs_bf16* k_ctx, const kvs_bf16* v_ctx, int32_t T,
                        const kvs_bf16* k_tail, const kvs_bf16* v_tail, int32_t n_tail,
                        kvs_bf16* o, float* lse, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(n_q >= 0 && T >= 0 && n_tail >= 0, KVS_ERR_ARG, "kvs_attn_fwd: negative size");
  REQUIRE(n_q <= T + n_tail, KVS_ERR_SHAPE, "kvs_attn_fwd: n_q = %d exceeds keys T + n_tail = %d",
          n_q, T + n_tail);
  if (n_q == 0) return ok();
  REQUIRE_PTR(q);
  REQUIRE_PTR(o);
  REQUIRE_PTR(lse);
  if (T > 0) {
    REQUIRE_PTR(k_ctx);
    REQUIRE_PTR(v_ctx);
  }
  if (n_tail > 0) {
    REQUIRE_PTR(k_tail);
    REQUIRE_PTR(v_tail);
  }
  kvs::FwdArgs a;
  a.q = q; a.k_ctx = k_ctx; a.v_ctx = v_ctx; a.k_tail = k_tail; a.v_tail = v_tail;
  a.o = o; a.lse = lse;
  a.L = dims->L; a.Hq = dims->H_q; a.Hkv = dims->H_kv; a.d = dims->d;
  a.n_q = n_q; a.T = T; a.n_tail = n_tail;
  return cuda_status(kvs::launch_attn_fwd(a, as_stream(stream)), "kvs_attn_fwd");
}

kvs_status kvs_score_max(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                         const kvs_bf16* k_ctx, int32_t T, const float* lse, const float* vnorm,
                         const kvs_bf16* h, int32_t accumulate, float* log_score, void* ws,
                         size_t ws_bytes, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(n_q >= 0 && T >= 0, KVS_ERR_ARG, "kvs_score_max: negative size");
  if (T == 0) return ok();
  REQUIRE_PTR(k_ctx);
  REQUIRE_PTR(log_score);
  REQUIRE_OPT_PTR(vnorm);
  REQUIRE_OPT_PTR(h);
  if (n_q > 0) {
    REQUIRE_PTR(q);
    REQUIRE_PTR(lse);
  }
  if (h) {
    REQUIRE(dims->D_h > 0 && dims->D_h % 8 == 0, KVS_ERR_SHAPE,
            "kvs_score_max: D_h = %d must be a positive multiple of 8 when h is given", dims->D_h);
  }
  const size_t need = kvs_score_max_workspace_size(dims, n_q, h != nullptr);
  if (n_q > 0) {
    REQUIRE_PTR(ws);
    REQUIRE(ws_bytes >= need, KVS_ERR_CAPACITY,
            "kvs_score_max: workspace of %zu bytes, %zu needed", ws_bytes, need);
  }
  cudaStream_t s = as_stream(stream);
  kvs::AttnArgs a;
  a.q = q; a.k_ctx = k_ctx; a.lse = lse; a.vnorm = vnorm; a.out = log_score;
  a.L = dims->L; a.Hq = dims->H_q; a.Hkv = dims->H_kv; a.d = dims->d;
  a.n_q = n_q; a.T = T; a.accumulate = accumulate != 0;
  if (n_q > 0) {
    uint8_t* w = static_cast<uint8_t*>(ws);
    auto* ccol = reinterpret_cast<kvs::bf16_t*>(w);
    auto* ones = reinterpret_cast<kvs::bf16_t*>(w + need - 128 * 32);
    // the per-query constants lse_j (+ ln ||h_j||) of the folded MMA step
    cudaError_t e = h ? kvs::launch_hidden_constants(h, dims->D_h, lse, dims->L, dims->H_q, n_q,
                                                     dims->d, ccol, ones, s)
                      : kvs::launch_score_constants(lse, dims->L, dims->H_q, n_q, dims->d, ccol,
                                                    ones, s);
    if (e != cudaSuccess) return cuda_status(e, "kvs_score_max (constants)");
    a.ccol = ccol;
    a.ones = ones;
  }
  return cuda_status(kvs::launch_score_max(a, s), "kvs_score_max");
}

size_t kvs_score_future_sum_workspace_size(const kvs_dims* dims, int32_t T) {
  if (!dims || T <= 0 || dims->L <= 0 || dims->H_q <= 0) return 0;
  return kvs::score_max_ws_bytes(dims->L, dims->H_q, T);
}

kvs_status kvs_score_future_sum(const kvs_dims* dims, const kvs_bf16* q, const kvs_bf16* k,
                                int32_t T, const float* lse, int32_t w, float* score, void* ws,
                                size_t ws_bytes, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(T >= 0 && w >= 0, KVS_ERR_ARG, "kvs_score_future_sum: negative T or w");
  if (T == 0) return ok();
  REQUIRE_PTR(q);
  REQUIRE_PTR(k);
  REQUIRE_PTR(lse);
  REQUIRE_PTR(score);
  REQUIRE_PTR(ws);
  const size_t need = kvs_score_future_sum_workspace_size(dims, T);
  REQUIRE(ws_bytes >= need, KVS_ERR_CAPACITY,
          "kvs_score_future_sum: workspace of %zu bytes, %zu needed", ws_bytes, need);
  cudaStream_t s = as_stream(stream);
  auto* ccol = static_cast<kvs::bf16_t*>(ws);
  auto* ones = reinterpret_cast<kvs::bf16_t*>(static_cast<uint8_t*>(ws) + need - 128 * 32);
  cudaError_t e = kvs::launch_score_constants(lse, dims->L, dims->H_q, T, dims->d, ccol, ones, s);
  if (e != cudaSuccess) return cuda_status(e, "kvs_score_future_sum (constants)");
  kvs::AttnArgs a;
  a.q = q; a.k_ctx = k; a.lse = lse; a.out = score;
  a.L = dims->L; a.Hq = dims->H_q; a.Hkv = dims->H_kv; a.d = dims->d;
  a.n_q = T; a.T = T; a.w = w;
  a.ccol = ccol; a.ones = ones;
  return cuda_status(kvs::launch_future_sum(a, s), "kvs_score_future_sum");
}

size_t kvs_vnorm_workspace_size(const kvs_dims* dims) {
  if (!dims || dims->L <= 0 || dims->H_q <= 0 || dims->d <= 0) return 0;
  return kvs::vnorm_workspace_bytes(dims->L, dims->H_q, dims->d);
}

kvs_status kvs_vnorm(const kvs_dims* dims, const kvs_bf16* v, int32_t T, const kvs_bf16* w_o,
                     float* vnorm, void* ws, size_t ws_bytes, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(T >= 0, KVS_ERR_ARG, "kvs_vnorm: negative T");
  REQUIRE(dims->H_q / dims->H_kv <= 16, KVS_ERR_UNSUPPORTED,
          "kvs_vnorm: %d query heads per KV head (at most 16)", dims->H_q / dims->H_kv);
  REQUIRE(dims->D_h > 0 && dims->D_h % 8 == 0, KVS_ERR_SHAPE,
          "kvs_vnorm: D_h = %d must be a positive multiple of 8", dims->D_h);
  if (T == 0) return ok();
  REQUIRE_PTR(v);
  REQUIRE_PTR(w_o);
  REQUIRE_PTR(vnorm);
  REQUIRE_PTR(ws);
  const size_t need = kvs_vnorm_workspace_size(dims);
  REQUIRE(ws_bytes >= need, KVS_ERR_CAPACITY, "kvs_vnorm: workspace of %zu bytes, %zu needed",
          ws_bytes, need);
  return cuda_status(kvs::launch_vnorm(v, dims->L, dims->H_q, dims->H_kv, dims->d, T, dims->D_h,
                                       w_o, vnorm, ws, as_stream(stream)),
                     "kvs_vnorm");
}

kvs_status kvs_vnorm_noalloc(const kvs_dims* dims, const kvs_bf16* v, int32_t T,
                             const kvs_bf16* w_o, float* vnorm, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(T >= 0, KVS_ERR_ARG, "kvs_vnorm_noalloc: negative T");
  REQUIRE(dims->D_h > 0 && dims->D_h % 8 == 0, KVS_ERR_SHAPE,
          "kvs_vnorm_noalloc: D_h = %d must be a positive multiple of 8", dims->D_h);
  const size_t per_layer = kvs::vnorm_workspace_bytes(1, dims->H_q, dims->d);
  REQUIRE(per_layer <= kvs::vnorm_noalloc_scratch_bytes(), KVS_ERR_CAPACITY,
          "kvs_vnorm_noalloc: one layer needs %zu bytes of scratch (H_q * d * d * 4) but the "
          "built-in scratch holds %zu; use kvs_vnorm with a caller workspace",
          per_layer, kvs::vnorm_noalloc_scratch_bytes());
  REQUIRE(dims->H_q / dims->H_kv <= 16, KVS_ERR_UNSUPPORTED,
          "kvs_vnorm_noalloc: %d query heads per KV head (at most 16)", dims->H_q / dims->H_kv);
  if (T == 0) return ok();
  REQUIRE_PTR(v);
  REQUIRE_PTR(w_o);
  REQUIRE_PTR(vnorm);
  return cuda_status(kvs::launch_vnorm_noalloc(v, dims->L, dims->H_q, dims->H_kv, dims->d, T,
                                               dims->D_h, w_o, vnorm, as_stream(stream)),
                     "kvs_vnorm_noalloc");
}

kvs_status kvs_surrogate(const kvs_dims* dims, const kvs_bf16* h, int32_t T, const kvs_bf16* W,
                         const float* b, float* score, float tau, int32_t w, uint8_t* mask,
                         int32_t* keep, void* stream) {
  kvs_status st = check_dims(dims, __func__, false);
  if (st) return st;
  REQUIRE(T >= 0 && w >= 0, KVS_ERR_ARG, "kvs_surrogate: negative T or w");
  REQUIRE(dims->H_kv <= 16, KVS_ERR_UNSUPPORTED, "kvs_surrogate: H_kv = %d (at most 16)",
          dims->H_kv);
  REQUIRE(dims->D_h > 0 && dims->D_h % 128 == 0, KVS_ERR_UNSUPPORTED,
          "kvs_surrogate: D_h = %d must be a positive multiple of 128", dims->D_h);
  REQUIRE(kvs::surrogate_smem_bytes(dims->D_h, dims->H_kv) <= 200 * 1024, KVS_ERR_UNSUPPORTED,
          "kvs_surrogate: D_h * ceil(H_kv/8) = %d above 12800",
          dims->D_h * ((dims->H_kv + 7) / 8));
  if (T == 0) return ok();
  REQUIRE_PTR(h);
  REQUIRE_PTR(W);
  REQUIRE_PTR(b);
  REQUIRE_PTR(score);
  if (mask) {
    REQUIRE_PTR(keep);
  }
  return cuda_status(kvs::launch_surrogate(h, dims->L, T, dims->D_h, dims->H_kv, W, b, score, tau,
                                           w, mask, keep, as_stream(stream)),
                     "kvs_surrogate");
}

kvs_status kvs_surrogate_mlp(const kvs_dims* dims, const kvs_bf16* h, int32_t T, int32_t D_mid,
                             const kvs_bf16* W1, const float* b1, const kvs_bf16* W2,
                             const float* b2, float* score, float tau, int32_t w, uint8_t* mask,
                             int32_t* keep, void* stream) {
  kvs_status st = check_dims(dims, __func__, false);
  if (st) return st;
  REQUIRE(T >= 0 && w >= 0, KVS_ERR_ARG, "kvs_surrogate_mlp: negative T or w");
  const int H = dims->H_kv;
  REQUIRE(H == 1 || H == 2 || H == 4 || H == 8 || H == 16, KVS_ERR_UNSUPPORTED,
          "kvs_surrogate_mlp: H_kv = %d (supported: 1, 2, 4, 8, 16)", H);
  REQUIRE(dims->D_h > 0 && dims->D_h % 64 == 0, KVS_ERR_UNSUPPORTED,
          "kvs_surrogate_mlp: D_h = %d must be a positive multiple of 64", dims->D_h);
  REQUIRE(kvs::mlp_parts(D_mid) > 0, KVS_ERR_UNSUPPORTED,
          "kvs_surrogate_mlp: D_mid = %d must be a positive multiple of 32", D_mid);
  REQUIRE((int64_t)dims->L * H * T <= ((int64_t)1 << 40) && (int64_t)dims->L * T < INT32_MAX,
          KVS_ERR_UNSUPPORTED, "kvs_surrogate_mlp: L * T too large");
  if (T == 0) return ok();
  REQUIRE_PTR(h);
  REQUIRE_PTR(W1);
  REQUIRE_PTR(b1);
  REQUIRE_PTR(W2);
  REQUIRE_PTR(b2);
  REQUIRE_PTR(score);
  if (mask) {
    REQUIRE_PTR(keep);
  }
  kvs::MlpArgs a;
  a.h = h;
  a.W1 = W1;
  a.b1 = b1;
  a.W2 = W2;
  a.b2 = b2;
  a.z = score;
  a.L = dims->L;
  a.T = T;
  a.Dh = dims->D_h;
  a.Dm = D_mid;
  a.H = H;
  cudaError_t e = kvs::launch_mlp_surrogate(a, as_stream(stream));
  if (e == cudaSuccess && mask)
    e = kvs::launch_prune(score, dims->L * H, T, KVS_THRESHOLD, tau, 0, w, mask, keep,
                          as_stream(stream));
  return cuda_status(e, "kvs_surrogate_mlp");
}

kvs_status kvs_decode_step(const kvs_dims* dims, int32_t B, int32_t w, int32_t* pos,
                           const float* new_score, const kvs_bf16* new_k, const kvs_bf16* new_v,
                           float* ring_score, kvs_bf16* ring_k, kvs_bf16* ring_v, float tau,
                           int32_t page_size, kvs_bf16* k_pages, kvs_bf16* v_pages,
                           int32_t capacity_pages, int32_t* next_page, int32_t* block_table,
                           int32_t max_pages, int32_t* seq_lens, int32_t advance_pos,
                           void* stream) {
  kvs_status st = check_dims(dims, __func__, false);
  if (st) return st;
  REQUIRE(dims->d == 64 || dims->d == 128, KVS_ERR_UNSUPPORTED,
          "kvs_decode_step: head dim d = %d (supported: 64, 128)", dims->d);
  REQUIRE(B >= 0 && w >= 0 && capacity_pages >= 0, KVS_ERR_ARG, "kvs_decode_step: negative size");
  REQUIRE(page_size >= 1 && page_size <= 4096, KVS_ERR_UNSUPPORTED,
          "kvs_decode_step: page_size = %d (1..4096)", page_size);
  REQUIRE(max_pages >= 1, KVS_ERR_SHAPE, "kvs_decode_step: max_pages = %d must be >= 1", max_pages);
  REQUIRE((int64_t)dims->L * dims->H_kv * B < INT32_MAX / 32, KVS_ERR_UNSUPPORTED,
          "kvs_decode_step: too many rows");
  if (B == 0) return ok();
  REQUIRE_PTR(pos);
  REQUIRE_PTR(new_score);
  REQUIRE_PTR(new_k);
  REQUIRE_PTR(new_v);
  if (w > 0) {
    REQUIRE_PTR(ring_score);
    REQUIRE_PTR(ring_k);
    REQUIRE_PTR(ring_v);
  }
  REQUIRE_PTR(next_page);
  REQUIRE_PTR(block_table);
  REQUIRE_PTR(seq_lens);
  if (capacity_pages > 0) {
    REQUIRE_PTR(k_pages);
    REQUIRE_PTR(v_pages);
  }
  kvs::DecodeArgs a;
  a.rows = dims->L * dims->H_kv * B;
  a.B = B; a.w = w; a.d = dims->d; a.page_size = page_size; a.max_pages = max_pages;
  a.capacity = capacity_pages; a.tau = tau;
  a.pos = pos; a.new_score = new_score; a.new_k = new_k; a.new_v = new_v;
  a.ring_score = ring_score; a.ring_k = ring_k; a.ring_v = ring_v;
  a.k_pages = k_pages; a.v_pages = v_pages; a.next_page = next_page;
  a.block_table = block_table; a.seq_lens = seq_lens;
  return cuda_status(kvs::launch_decode_step(a, advance_pos != 0, as_stream(stream)),
                     "kvs_decode_step");
}

namespace {
struct RefitPlan {
  int g, rows, k_ld;
  size_t off_o, off_lse, off_a, off_g, off_r, total;
};
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
RefitPlan refit_plan(const kvs_dims* dm, int n_q, int k) {
  RefitPlan p{};
  p.g = dm->H_q / dm->H_kv;
  p.rows = p.g * n_q;
  p.k_ld = (k + 63) / 64 * 64;
  const size_t nq_all = (size_t)dm->L * dm->H_q * n_q, batch = (size_t)dm->L * dm->H_kv;
  size_t o = 0;
  p.off_o = o;   o = align256(o + nq_all * dm->d * 2);
  p.off_lse = o; o = align256(o + nq_all * 4);
  p.off_a = o;   o = align256(o + nq_all * p.k_ld * 2);
  p.off_g = o;   o = align256(o + batch * p.k_ld * p.k_ld * 4);
  p.off_r = o;   o = align256(o + batch * p.k_ld * dm->d * 4);
  p.total = o;
  return p;
}
}  // namespace

size_t kvs_value_refit_workspace_size(const kvs_dims* dims, int32_t n_q, int32_t k) {
  if (!dims || dims->L <= 0 || dims->H_kv <= 0 || dims->H_q <= 0 || dims->H_q % dims->H_kv ||
      n_q < 0 || k < 0)
    return 0;
  return refit_plan(dims, n_q, k).total;
}

kvs_status kvs_value_refit(const kvs_dims* dims, const kvs_bf16* q, int32_t n_q,
                           const kvs_bf16* k_ctx, const kvs_bf16* v_ctx, int32_t T,
                           const kvs_bf16* k_kept, int32_t k, float lambda_rel, float* v_fit,
                           void* ws, size_t ws_bytes, void* stream) {
  kvs_status st = check_dims(dims, __func__);
  if (st) return st;
  REQUIRE(n_q >= 0 && T >= 0 && k >= 0, KVS_ERR_ARG, "kvs_value_refit: negative size");
  REQUIRE(k <= T, KVS_ERR_SHAPE, "kvs_value_refit: k = %d kept keys exceed T = %d", k, T);
  REQUIRE(lambda_rel >= 0.f, KVS_ERR_ARG, "kvs_value_refit: lambda_rel = %g < 0",
          (double)lambda_rel);
  REQUIRE((k + 63) / 64 * 64 <= kvs::kCholMaxM, KVS_ERR_UNSUPPORTED,
          "kvs_value_refit: k = %d above %d", k, kvs::kCholMaxM);
  if (n_q == 0 || k == 0) return ok();
  const RefitPlan pl = refit_plan(dims, n_q, k);
  REQUIRE((int64_t)pl.rows * pl.k_ld < INT32_MAX, KVS_ERR_UNSUPPORTED,
          "kvs_value_refit: n_q * g * k too large");
  REQUIRE_PTR(q);
  REQUIRE_PTR(k_ctx);
  REQUIRE_PTR(v_ctx);
  REQUIRE_PTR(k_kept);
  REQUIRE_PTR(v_fit);
  REQUIRE_PTR(ws);
  REQUIRE(ws_bytes >= pl.total, KVS_ERR_CAPACITY,
          "kvs_value_refit: workspace of %zu bytes, %zu needed", ws_bytes, pl.total);
  uint8_t* w = static_cast<uint8_t*>(ws);
  auto* o_ws = reinterpret_cast<kvs::bf16_t*>(w + pl.off_o);
  auto* lse_ws = reinterpret_cast<float*>(w + pl.off_lse);
  auto* a_s = reinterpret_cast<uint16_t*>(w + pl.off_a);  // fp16 softmax rows
  auto* gm = reinterpret_cast<float*>(w + pl.off_g);
  auto* rm = reinterpret_cast<float*>(w + pl.off_r);
  cudaStream_t s = as_stream(stream);
  const int L = dims->L, Hq = dims->H_q, Hkv = dims->H_kv, d = dims->d;
  // 1. target: attention output of every scoring query over the whole context
  kvs::FwdArgs f;
  f.q = q; f.k_ctx = k_ctx; f.v_ctx = v_ctx; f.o = o_ws; f.lse = lse_ws;
  f.L = L; f.Hq = Hq; f.Hkv = Hkv; f.d = d; f.n_q = n_q; f.T = T; f.causal = 0; f.o_f16 = 1;
  cudaError_t e = kvs::launch_attn_fwd(f, s);
  // 2. softmax rows over the kept keys: their LSE, then the rows as fp16
  kvs::AttnArgs r;
  r.q = q; r.k_ctx = k_kept; r.lse = lse_ws; r.out = lse_ws;
  r.L = L; r.Hq = Hq; r.Hkv = Hkv; r.d = d; r.n_q = n_q; r.T = k; r.causal = 0;
  r.rows = a_s; r.rows_ld = pl.k_ld;
  if (e == cudaSuccess) e = kvs::launch_lse(r, s);
  if (e == cudaSuccess) e = kvs::launch_softmax_rows(r, s);
  // 3. normal equations: Gram (upper block triangle) and right-hand side, one launch
  kvs::RefitProdArgs rp;
  rp.a_s = a_s; rp.o = reinterpret_cast<const uint16_t*>(o_ws); rp.g = gm; rp.r = rm;
  rp.batch = L * Hkv; rp.rows = pl.rows; rp.k_ld = pl.k_ld; rp.d = d;
  if (e == cudaSuccess) e = kvs::launch_refit_products(rp, s);
  // 4. ridge solve per (layer, KV head)
  kvs::CholArgs c;
  c.g = gm; c.r = rm; c.x = v_fit; c.batch = L * Hkv; c.M = pl.k_ld; c.ldg = pl.k_ld;
  c.k = k; c.d = d; c.lam_rel = lambda_rel;
  if (e == cudaSuccess) e = kvs::launch_chol_solve(c, s);
  return cuda_status(e, "kvs_value_refit");
}

kvs_status kvs_prune_mask(const kvs_dims* dims, const float* score, int32_t T, int32_t mode,
                          float tau, int32_t k, int32_t w, uint8_t* mask, int32_t* keep,
                          void* stream) {
  kvs_status st = check_dims(dims, __func__, false);
  if (st) return st;
  REQUIRE(T >= 0 && w >= 0 && k >= 0, KVS_ERR_ARG, "kvs_prune_mask: negative T, k or w");
  REQUIRE(mode == KVS_THRESHOLD || mode == KVS_TOPK, KVS_ERR_ARG, "kvs_prune_mask: mode = %d",
          mode);
  REQUIRE_PTR(keep);
  if (T > 0) {
    REQUIRE_PTR(score);
    REQUIRE_PTR(mask);
  }
  return cuda_status(kvs::launch_prune(score, dims->L * dims->H_kv, T, mode, tau, k, w, mask, keep,
                                       as_stream(stream)),
                     "kvs_prune_mask");
}

kvs_status kvs_prune_quantile(const kvs_dims* dims, const float* score, int32_t T, float q,
                              int32_t w, float* tau, uint8_t* mask, int32_t* keep, void* stream) {
  kvs_status st = check_dims(dims, __func__, false);
  if (st) return st;
  REQUIRE(T >= 0 && w >= 0, KVS_ERR_ARG, "kvs_prune_quantile: negative T or w");
  REQUIRE(q >= 0.f && q <= 1.f, KVS_ERR_ARG, "kvs_prune_quantile: q = %g outside [0, 1]", (double)q);
  REQUIRE_PTR(tau);
  REQUIRE_PTR(keep);
  if (T > 0) {
    REQUIRE_PTR(score);
    REQUIRE_PTR(mask);
  }
  return cuda_status(kvs::launch_prune_quantile(score, dims->L, dims->H_kv, T, q, w, tau, mask,
                                                keep, as_stream(stream)),
                     "kvs_prune_quantile");
}

size_t kvs_compact_workspace_size(const kvs_dims* dims, int32_t T) {
  return kvs_compact_multi_workspace_size(dims, T, 1);
}

size_t kvs_compact_multi_workspace_size(const kvs_dims* dims, int32_t T, int32_t n_masks) {
  if (!dims || dims->L <= 0 || dims->H_kv <= 0 || T < 0 || n_masks < 1) return 0;
  return kvs::compact_workspace_bytes(dims->L * dims->H_kv * n_masks, T);
}

static kvs_status compact_paged(const char* fn, const kvs_dims* dims, const kvs_bf16* k,
                                const kvs_bf16* v, int32_t T, int32_t n_masks, const uint8_t* mask,
                                int32_t page_size, kvs_bf16* k_pages, kvs_bf16* v_pages,
                                int32_t capacity_pages, int32_t* block_table, int32_t max_pages,
                                int32_t* seq_lens, int32_t* needed_pages, void* ws,
                                size_t ws_bytes, void* stream) {
  kvs_status st = check_dims(dims, fn, false);
  if (st) return st;
  REQUIRE(dims->d == 64 || dims->d == 128, KVS_ERR_UNSUPPORTED,
          "%s: head dim d = %d (supported: 64, 128)", fn, dims->d);
  REQUIRE(T >= 0 && capacity_pages >= 0, KVS_ERR_ARG, "%s: negative size", fn);
  REQUIRE(n_masks >= 1, KVS_ERR_ARG, "%s: n_masks = %d (at least 1)", fn, n_masks);
  REQUIRE((long long)dims->L * dims->H_kv * n_masks <= (1LL << 30), KVS_ERR_SHAPE,
          "%s: %d masks of %d rows", fn, n_masks, dims->L * dims->H_kv);
  REQUIRE(page_size >= 1 && page_size <= 4096, KVS_ERR_UNSUPPORTED,
          "%s: page_size = %d (1..4096)", fn, page_size);
  REQUIRE(max_pages >= (T + page_size - 1) / page_size, KVS_ERR_SHAPE,
          "%s: max_pages = %d below ceil(T / page_size) = %d", fn, max_pages,
          (T + page_size - 1) / page_size);
  if (!seq_lens) return fail(KVS_ERR_ARG, "%s: seq_lens is NULL", fn);
  if (!needed_pages) return fail(KVS_ERR_ARG, "%s: needed_pages is NULL", fn);
  if (!ws) return fail(KVS_ERR_ARG, "%s: ws is NULL", fn);
  if (!aligned16(seq_lens) || !aligned16(needed_pages) || !aligned16(ws))
    return fail(KVS_ERR_ALIGN, "%s: seq_lens, needed_pages or ws is not 16-byte aligned", fn);
  if (max_pages > 0) {
    if (!block_table) return fail(KVS_ERR_ARG, "%s: block_table is NULL", fn);
    if (!aligned16(block_table)) return fail(KVS_ERR_ALIGN, "%s: block_table is not 16-byte aligned", fn);
  }
  if (T > 0) {
    if (!k || !v || !mask) return fail(KVS_ERR_ARG, "%s: k, v or mask is NULL", fn);
    if (!aligned16(k) || !aligned16(v) || !aligned16(mask))
      return fail(KVS_ERR_ALIGN, "%s: k, v or mask is not 16-byte aligned", fn);
  }
  if (capacity_pages > 0) {
    if (!k_pages || !v_pages) return fail(KVS_ERR_ARG, "%s: k_pages or v_pages is NULL", fn);
    if (!aligned16(k_pages) || !aligned16(v_pages))
      return fail(KVS_ERR_ALIGN, "%s: k_pages or v_pages is not 16-byte aligned", fn);
  }
  const size_t need = kvs_compact_multi_workspace_size(dims, T, n_masks);
  REQUIRE(ws_bytes >= need, KVS_ERR_CAPACITY, "%s: workspace of %zu bytes, %zu needed", fn,
          ws_bytes, need);
  return cuda_status(kvs::launch_compact(k, v, dims->L * dims->H_kv, n_masks, T, dims->d, mask,
                                         page_size, k_pages, v_pages, capacity_pages, block_table,
                                         max_pages, seq_lens, needed_pages, ws, as_stream(stream)),
                     fn);
}

kvs_status kvs_compact_paged(const kvs_dims* dims, const kvs_bf16* k, const kvs_bf16* v, int32_t T,
                             const uint8_t* mask, int32_t page_size, kvs_bf16* k_pages,
                             kvs_bf16* v_pages, int32_t capacity_pages, int32_t* block_table,
                             int32_t max_pages, int32_t* seq_lens, int32_t* needed_pages,
                             void* ws, size_t ws_bytes, void* stream) {
  return compact_paged(__func__, dims, k, v, T, 1, mask, page_size, k_pages, v_pages,
                       capacity_pages, block_table, max_pages, seq_lens, needed_pages, ws,
                       ws_bytes, stream);
}

kvs_status kvs_compact_paged_multi(const kvs_dims* dims, const kvs_bf16* k, const kvs_bf16* v,
                                   int32_t T, int32_t n_masks, const uint8_t* masks,
                                   int32_t page_size, kvs_bf16* k_pages, kvs_bf16* v_pages,
                                   int32_t capacity_pages, int32_t* block_table, int32_t max_pages,
                                   int32_t* seq_lens, int32_t* needed_pages, void* ws,
                                   size_t ws_bytes, void* stream) {
  return compact_paged(__func__, dims, k, v, T, n_masks, masks, page_size, k_pages, v_pages,
                       capacity_pages, block_table, max_pages, seq_lens, needed_pages, ws,
                       ws_bytes, stream);
}

kvs_status kvs_prune_topk_multi(const kvs_dims* dims, const float* score, int32_t T,
                                int32_t n_budgets, const int32_t* k, int32_t w, uint8_t* masks,
                                int32_t* keeps, void* stream) {
  kvs_status st = check_dims(dims, __func__, false);
  if (st) return st;
  REQUIRE(T >= 0 && w >= 0, KVS_ERR_ARG, "kvs_prune_topk_multi: negative T or w");
  REQUIRE(n_budgets >= 1 && n_budgets <= kvs::kMaxTopkBudgets, KVS_ERR_UNSUPPORTED,
          "kvs_prune_topk_multi: n_budgets = %d (1..%d)", n_budgets, kvs::kMaxTopkBudgets);
  REQUIRE(k != nullptr, KVS_ERR_ARG, "kvs_prune_topk_multi: k is NULL");
  kvs::TopkBudgets kb = {};
  for (int b = 0; b < n_budgets; ++b) {
    REQUIRE(k[b] >= 0, KVS_ERR_ARG, "kvs_prune_topk_multi: k[%d] = %d is negative", b, k[b]);
    kb.k[b] = k[b];
  }
  REQUIRE_PTR(keeps);
  if (T > 0) {
    REQUIRE_PTR(score);
    REQUIRE_PTR(masks);
  }
  return cuda_status(kvs::launch_topk(score, dims->L * dims->H_kv, T, n_budgets, kb, w, masks,
                                      keeps, as_stream(stream)),
                     "kvs_prune_topk_multi");
}

}  // extern "C"
