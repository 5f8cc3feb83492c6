// Paged per-head variable-length compaction of the kept K/V rows (KVzap review,
// Algorithm 1: keys[indices], values[indices]; limitation 3: non-uniform head
// lengths need PagedAttention-like storage).
//
// Any number of masks over the same K/V rows go through one set of launches: mask row r
// takes its K/V from row r % (L H_kv), and the pages of all masks share one pool, in
// mask-major order.  Three launches, all bandwidth-bound:
//   1. seg_count   : kept tokens per (row, segment of 256, 1024 or 4096 tokens)  reads the mask
//   2. page_plan   : per-row exclusive scan of segment counts, page counts
//                    ceil(kept/page), exclusive scan of pages over rows (layer-major,
//                    then head), capacity check, seq_lens, needed_pages
//   3. scatter     : per (row, segment) ordered rank of each kept token (block scan),
//                    then a block-cooperative 16-byte copy of the kept K and V rows
//                    into (page, slot); the last segment zero-fills the tail of the
//                    row's last page; every block fills its share of block_table.
#include "common.cuh"
#include "compact.cuh"

namespace kvs {
namespace {

constexpr int kSegThreads = 256;  // P mask bytes per thread, segments of 256 * P tokens
constexpr int kTinySeg = 256;     // short rows (T <= kShortRow): P = 1, more blocks
constexpr int kMinSeg = 1024;     // medium rows: P = 4
constexpr int kMaxSeg = 4096;     // long rows (T >= kLongRow): P = 16, fewer, larger blocks
constexpr int kShortRow = 4096;
constexpr int kLongRow = 8192;

struct Plan {            // lives at the start of the workspace
  int ok;                // total pages <= capacity
  int total_pages;
  int pad[2];
};


// Mask bytes t0 .. t0+P-1 of a row as 0/1 flags (vector loads when T allows).
template <int P>
__device__ __forceinline__ void load_flags(const uint8_t* m, int T, int t0, uint8_t* f) {
  if constexpr (P == 1) {
    f[0] = t0 < T ? (m[t0] != 0) : 0;
    return;
  } else if ((T & (P - 1)) == 0 && t0 < T) {
    uint32_t wd[P / 4];
    if constexpr (P == 16) {
      const uint4 u = *reinterpret_cast<const uint4*>(m + t0);
      wd[0] = u.x;
      wd[1] = u.y;
      wd[2] = u.z;
      wd[3] = u.w;
    } else {
      static_assert(P == 4, "1, 4 or 16 mask bytes per thread");
      wd[0] = *reinterpret_cast<const uint32_t*>(m + t0);
    }
#pragma unroll
    for (int i = 0; i < P; ++i) f[i] = ((wd[i >> 2] >> (8 * (i & 3))) & 255u) != 0;
  } else {
#pragma unroll
    for (int i = 0; i < P; ++i) f[i] = (t0 + i < T) ? (m[t0 + i] != 0) : 0;
  }
}

// Kept count of each (row, segment).
template <int P>
__global__ void __launch_bounds__(kSegThreads) seg_count_kernel(const uint8_t* __restrict__ mask,
                                                                int T, int nseg,
                                                                int* __restrict__ seg) {
  __shared__ int red[kSegThreads / 32];
  const int s = blockIdx.x, row = blockIdx.y;
  const uint8_t* m = mask + (size_t)row * T;
  const int t0 = s * (kSegThreads * P) + threadIdx.x * P;
  uint8_t f[P];
  load_flags<P>(m, T, t0, f);
  int c = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) c += f[i];
  c = warp_sum_int(c);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
  __syncthreads();
  if (threadIdx.x == 0) {
    int tot = 0;
    for (int i = 0; i < kSegThreads / 32; ++i) tot += red[i];
    seg[(size_t)row * nseg + s] = tot;
  }
}

// One block: segment offsets per row, page offsets over rows, capacity check.
__global__ void __launch_bounds__(1024) page_plan_kernel(int rows, int nseg, int page_size,
                                                         int capacity, int* __restrict__ seg,
                                                         int* __restrict__ first_page,
                                                         Plan* __restrict__ plan,
                                                         int* __restrict__ seq_lens,
                                                         int* __restrict__ needed) {
  __shared__ int warp_tot[32];
  __shared__ int carry_s;
  if (threadIdx.x == 0) carry_s = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int base = 0; base < rows; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int pages = 0;
    if (r < rows) {
      int* sr = seg + (size_t)r * nseg;
      int acc = 0;
      for (int s = 0; s < nseg; ++s) {
        const int c = sr[s];
        sr[s] = acc;
        acc += c;
      }
      seq_lens[r] = acc;
      pages = (acc + page_size - 1) / page_size;
    }
    // block exclusive scan of pages
    int incl = pages;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int x = lane < nw ? warp_tot[lane] : 0;
      int wi = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wi, o);
        if (lane >= o) wi += y;
      }
      if (lane < nw) warp_tot[lane] = wi - x;
    }
    __syncthreads();
    const int excl = carry_s + warp_tot[warp] + incl - pages;
    if (r < rows) first_page[r] = excl;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry_s = excl + pages;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    plan->total_pages = carry_s;
    plan->ok = carry_s <= capacity;
    *needed = carry_s;
  }
}

template <int P>
__global__ void __launch_bounds__(kSegThreads) scatter_kernel(
    const bf16_t* __restrict__ k, const bf16_t* __restrict__ v, const uint8_t* __restrict__ mask,
    int T, int d, int nseg, int kv_rows, int page_size, const int* __restrict__ seg,
    const int* __restrict__ first_page, const Plan* __restrict__ plan,
    const int* __restrict__ seq_lens, bf16_t* __restrict__ k_pages, bf16_t* __restrict__ v_pages,
    int* __restrict__ block_table, int max_pages) {
  constexpr int kSeg = kSegThreads * P;
  __shared__ uint16_t list[kSeg];
  __shared__ int red[33];
  const int s = blockIdx.x, row = blockIdx.y;
  const bool ok = plan->ok != 0;
  const int first = first_page[row];
  const int kept = seq_lens[row];
  const int npages = (kept + page_size - 1) / page_size;

  // block_table entries [s*ppseg, (s+1)*ppseg), the last segment also covers the rest
  {
    const int ppseg = (kSeg + page_size - 1) / page_size;
    const int p0 = s * ppseg;
    const int p1 = (s == nseg - 1) ? max_pages : min(max_pages, p0 + ppseg);
    int* bt = block_table + (size_t)row * max_pages;
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x)
      bt[p] = (ok && p < npages) ? first + p : -1;
  }
  if (!ok) return;

  // ordered ranks of the kept tokens of this segment
  const uint8_t* m = mask + (size_t)row * T;
  const int t0 = s * kSeg + threadIdx.x * P;
  uint8_t f[P];
  load_flags<P>(m, T, t0, f);
  int c = 0;
#pragma unroll
  for (int i = 0; i < P; ++i) c += f[i];
  // block exclusive scan of c
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) red[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int x = lane < nw ? red[lane] : 0;
    int wi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < nw) red[lane] = wi - x;
    if (lane == nw - 1) red[32] = wi;
  }
  __syncthreads();
  int pos = red[warp] + incl - c;
  const int n_local = red[32];
#pragma unroll
  for (int i = 0; i < P; ++i)
    if (f[i]) list[pos++] = (uint16_t)(threadIdx.x * P + i);
  __syncthreads();

  // cooperative copy: (d/8) 16-byte chunks per kept row, for K and V
  const int base_rank = seg[(size_t)row * nseg + s];
  const int cpr = d / 8;
  const size_t src_row0 = (size_t)(row % kv_rows) * T + (size_t)s * kSeg;  // mask row -> K/V row
  const int total = n_local * cpr;
  constexpr int U = 4;
  for (int i0 = threadIdx.x; i0 < total; i0 += blockDim.x * U) {
    uint4 kv[U], vv[U];
    size_t dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = i0 + u * blockDim.x;
      if (idx < total) {
        const int e = idx / cpr, ch = idx % cpr;
        const size_t src = (src_row0 + list[e]) * d + ch * 8;
        const int rank = base_rank + e;
        dst[u] = ((size_t)(first + rank / page_size) * page_size + rank % page_size) * d + ch * 8;
        kv[u] = ld_nc_v4(k + src);
        vv[u] = ld_nc_v4(v + src);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = i0 + u * blockDim.x;
      if (idx < total) {
        *reinterpret_cast<uint4*>(k_pages + dst[u]) = kv[u];
        *reinterpret_cast<uint4*>(v_pages + dst[u]) = vv[u];
      }
    }
  }

  // zero the unused rows of the row's last page (one block per row does it)
  if (s == nseg - 1 && kept % page_size) {
    const int pad_rows = page_size - kept % page_size;
    const size_t base = ((size_t)(first + npages - 1) * page_size + kept % page_size) * d;
    for (int i = threadIdx.x; i < pad_rows * cpr; i += blockDim.x) {
      *reinterpret_cast<uint4*>(k_pages + base + (size_t)i * 8) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(v_pages + base + (size_t)i * 8) = make_uint4(0, 0, 0, 0);
    }
  }
}

}  // namespace

size_t compact_workspace_bytes(int rows, int T) {
  const int nseg = (T + kTinySeg - 1) / kTinySeg;  // the finest segmentation bounds all
  return sizeof(Plan) + sizeof(int) * ((size_t)rows * (nseg > 0 ? nseg : 1) + rows);
}

cudaError_t launch_compact(const bf16_t* k, const bf16_t* v, int kv_rows, int n_masks, int T, int d,
                           const uint8_t* mask, int page_size, bf16_t* k_pages, bf16_t* v_pages,
                           int capacity, int* block_table, int max_pages, int* seq_lens,
                           int* needed, void* ws, cudaStream_t s) {
  const int rows = kv_rows * n_masks;  // mask rows: mask-major, then the K/V rows
  if (rows == 0) return cudaSuccess;
  const bool long_rows = T >= kLongRow, short_rows = T <= kShortRow;
  const int seg_len = long_rows ? kMaxSeg : short_rows ? kTinySeg : kMinSeg;
  const int nseg = T > 0 ? (T + seg_len - 1) / seg_len : 1;
  Plan* plan = reinterpret_cast<Plan*>(ws);
  int* seg = reinterpret_cast<int*>(plan + 1);
  int* first = seg + (size_t)rows * nseg;
  count_launches(3);
  if (long_rows)
    seg_count_kernel<16><<<dim3(nseg, rows), kSegThreads, 0, s>>>(mask, T, nseg, seg);
  else if (short_rows)
    seg_count_kernel<1><<<dim3(nseg, rows), kSegThreads, 0, s>>>(mask, T, nseg, seg);
  else
    seg_count_kernel<4><<<dim3(nseg, rows), kSegThreads, 0, s>>>(mask, T, nseg, seg);
  page_plan_kernel<<<1, 1024, 0, s>>>(rows, nseg, page_size, capacity, seg, first, plan, seq_lens,
                                      needed);
  if (long_rows)
    scatter_kernel<16><<<dim3(nseg, rows), kSegThreads, 0, s>>>(
        k, v, mask, T, d, nseg, kv_rows, page_size, seg, first, plan, seq_lens, k_pages, v_pages,
        block_table, max_pages);
  else if (short_rows)
    scatter_kernel<1><<<dim3(nseg, rows), kSegThreads, 0, s>>>(
        k, v, mask, T, d, nseg, kv_rows, page_size, seg, first, plan, seq_lens, k_pages, v_pages,
        block_table, max_pages);
  else
    scatter_kernel<4><<<dim3(nseg, rows), kSegThreads, 0, s>>>(
        k, v, mask, T, d, nseg, kv_rows, page_size, seg, first, plan, seq_lens, k_pages, v_pages,
        block_table, max_pages);
  return cudaGetLastError();
}

}  // namespace kvs
