#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace kvs {

size_t compact_workspace_bytes(int rows, int T);

// n_masks masks [n_masks][kv_rows][T] over the same K/V rows [kv_rows][T][d]: block_table
// [n_masks][kv_rows][max_pages], seq_lens [n_masks][kv_rows]; workspace for
// n_masks * kv_rows rows.
cudaError_t launch_compact(const bf16_t* k, const bf16_t* v, int kv_rows, int n_masks, int T, int d,
                           const uint8_t* mask, int page_size, bf16_t* k_pages, bf16_t* v_pages,
                           int capacity, int* block_table, int max_pages, int* seq_lens,
                           int* needed, void* ws, cudaStream_t s);

}  // namespace kvs
