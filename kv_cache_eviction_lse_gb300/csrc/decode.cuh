// Launcher of the decode-time pruning step (window ring -> paged cache).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace kvs {

struct DecodeArgs {
  int rows = 0, B = 0, w = 0, d = 0, page_size = 0, max_pages = 0, capacity = 0;
  float tau = 0.f;
  int* pos = nullptr;               // [B]
  const float* new_score = nullptr; // [rows]
  const bf16_t* new_k = nullptr;    // [rows][d]
  const bf16_t* new_v = nullptr;    // [rows][d]
  float* ring_score = nullptr;      // [rows][w]
  bf16_t* ring_k = nullptr;         // [rows][w][d]
  bf16_t* ring_v = nullptr;         // [rows][w][d]
  bf16_t* k_pages = nullptr;        // [capacity][page_size][d]
  bf16_t* v_pages = nullptr;
  int* next_page = nullptr;         // [1]
  int* block_table = nullptr;       // [rows][max_pages]
  int* seq_lens = nullptr;          // [rows]
};

// One decode step over every row; with `advance`, pos[b] += 1 afterwards.
cudaError_t launch_decode_step(const DecodeArgs& a, bool advance, cudaStream_t s);
cudaError_t decode_device_error(int* code, bool clear, cudaStream_t s);

}  // namespace kvs
