// Decode-time pruning at the window boundary [KVzap review: the criterion is phase-
// agnostic and runs while decoding; KVpop review, 1. Key Terms: a token is decided when
// it leaves the protected window].
//
// One decode step for every (layer, KV head, sequence) row: the token that arrives now
// (position pos[b]) enters a ring of the last w tokens; the token it displaces
// (position pos[b] - w) is appended to the row's paged cache iff its score >= tau.  One
// warp per row moves the 2 x d bf16 of K and V in 16-byte lanes; a row that starts a
// new page takes the next page id of a shared pool with one atomic add and zero-fills
// the page, so its unused rows read as zeros.
#include "common.cuh"
#include "decode.cuh"

namespace kvs {

__device__ int g_decode_error = 0;

namespace {

constexpr int kErrPoolFull = 4;    // the page pool ran out: the token was not appended
constexpr int kErrTableFull = 5;   // the row's block table is full: not appended

template <int D>
__global__ void __launch_bounds__(256) decode_step_kernel(const DecodeArgs a) {
  constexpr int kChunks = D / 8;  // 16-byte chunks per row of K (or V)
  const int row = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.rows) return;
  const int b = row % a.B;
  const size_t rd = (size_t)row * D;
  // lane c < 2 * kChunks moves 16-byte chunk c of [K | V]
  const bool mover = lane < 2 * kChunks;
  const int ck = lane < kChunks ? lane : lane - kChunks;

  // independent loads first (one round trip): position, fill level, the arriving token
  const int p = a.pos[b];
  const int n = a.seq_lens[row];
  const float s_new = a.new_score[row];
  uint4 x_new = make_uint4(0, 0, 0, 0);
  if (mover)
    x_new = reinterpret_cast<const uint4*>((lane < kChunks ? a.new_k : a.new_v) + rd)[ck];
  const int pi = n / a.page_size, pr = n % a.page_size;
  // second round trip: the leaving token (ring slot of p) and the row's current page
  bool append;
  uint4 x_out = x_new;
  size_t slot_off = 0;
  if (a.w > 0) {
    slot_off = (size_t)row * a.w + p % a.w;
    const float s_old = a.ring_score[slot_off];
    if (mover)
      x_out = reinterpret_cast<const uint4*>((lane < kChunks ? a.ring_k : a.ring_v) +
                                             slot_off * D)[ck];
    append = p >= a.w && s_old >= a.tau;  // NaN compares false
  } else {
    append = s_new >= a.tau;
  }
  int pg = -1;
  if (append && pr != 0 && pi < a.max_pages) pg = a.block_table[(size_t)row * a.max_pages + pi];

  if (append) {
    if (pr == 0) {  // the row needs a new page
      if (pi >= a.max_pages) {
        if (lane == 0) atomicCAS(&g_decode_error, 0, kErrTableFull);
      } else {
        if (lane == 0) pg = atomicAdd(a.next_page, 1);
        pg = __shfl_sync(0xffffffffu, pg, 0);
        if (pg >= a.capacity) {
          if (lane == 0) atomicCAS(&g_decode_error, 0, kErrPoolFull);
          pg = -1;
        } else {
          if (lane == 0) a.block_table[(size_t)row * a.max_pages + pi] = pg;
          // zero rows 1 .. page_size-1 of the new page (row 0 is written below)
          const size_t base = (size_t)pg * a.page_size * D;
          const int n16 = (a.page_size - 1) * kChunks;
          for (int c = lane; c < n16; c += 32) {
            reinterpret_cast<uint4*>(a.k_pages + base + D)[c] = make_uint4(0, 0, 0, 0);
            reinterpret_cast<uint4*>(a.v_pages + base + D)[c] = make_uint4(0, 0, 0, 0);
          }
        }
      }
    }
    if (pg >= 0) {
      const size_t dst = ((size_t)pg * a.page_size + pr) * D;
      if (mover) reinterpret_cast<uint4*>((lane < kChunks ? a.k_pages : a.v_pages) + dst)[ck] = x_out;
      if (lane == 0) a.seq_lens[row] = n + 1;
    }
  }

  // the arriving token takes the freed ring slot
  if (a.w > 0) {
    if (mover)
      reinterpret_cast<uint4*>((lane < kChunks ? a.ring_k : a.ring_v) + slot_off * D)[ck] = x_new;
    if (lane == 0) a.ring_score[slot_off] = s_new;
  }
}

__global__ void advance_pos_kernel(int* pos, int B) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) pos[b] += 1;
}

}  // namespace

cudaError_t launch_decode_step(const DecodeArgs& a, bool advance, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  const int blocks = (int)(((size_t)a.rows * 32 + 255) / 256);
  count_launches(1);
  if (a.d == 128)
    decode_step_kernel<128><<<blocks, 256, 0, s>>>(a);
  else
    decode_step_kernel<64><<<blocks, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess && advance) {
    count_launches(1);
    advance_pos_kernel<<<(a.B + 255) / 256, 256, 0, s>>>(a.pos, a.B);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t decode_device_error(int* code, bool clear, cudaStream_t s) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(code, g_decode_error, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess && clear && *code) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(g_decode_error, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  }
  return e;
}

}  // namespace kvs
