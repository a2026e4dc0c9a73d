// dsa_common.cuh -- shared launch parameters and small device helpers of the
// sm_103a DSA indexer kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_indexer.h"

namespace dsa {

constexpr int kHeads = 64;      // H
constexpr int kDim = 128;       // D
constexpr int kPage = 64;       // positions per page
constexpr int kMaxDevices = 64; // per-device launch state is kept for this many devices

// Everything a kernel needs about one call (device pointers and sizes).
struct RowsParams {
  const uint16_t* q;           // bf16 bits [rows, 64, 128]
  const float* w;              // [rows, 64]
  const uint8_t* kcache;       // page p at kcache + p * page_stride
  const uint8_t* kscale;       // page p's scales at kscale + p*page_stride, or null
  long long page_stride;       // bytes
  int num_pages;
  int kv_dtype;                // DSA_KV_FP8_E4M3 / DSA_KV_BF16
  const int* block_table;      // row r at block_table + r * bt_stride
  long long bt_stride;
  const int* seqlens;          // [rows]
  int rows;
  int W;                       // pages per row (block-table width)
  float* out;                  // row r at out + r * out_stride
  long long out_stride;
  int* status;                 // nullable
  int fill;                    // decode: 1 = write the -inf past each row's last valid
                               // page; 0 = leave it (top-k reads only t < L)
  int sel_k;                   // decode, balanced mode: > 0 = fused top-k, each chunk's
                               // sel_k best positions into the slots at sel_ws
  float* sel_ws;               // the fused top-k's workspace (topk_slots.cuh)
};

// Prefill of several requests in one launch: request b's query rows are
// rows row0[b] .. row0[b+1]-1 of the call, grouped into query tiles
// tile0[b] .. tile0[b+1]-1 of four rows (the last one ragged), and read
// the keys through block-table row b.  n_req = 0: one request, every row
// reads table row 0.
constexpr int kMaxPrefillRequests = 128;
struct PrefillRequests {
  int n_req;
  int tile0[kMaxPrefillRequests + 1];
  int row0[kMaxPrefillRequests + 1];
};

__device__ __forceinline__ void raise_status(int* status, int code) {
  if (status != nullptr) atomicMax(status, code);
}

}  // namespace dsa
