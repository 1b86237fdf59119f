// Internal interface between the C ABI (rca_attn.cu) and the paged decode
// kernels (decode.cu). Not installed; callers use include/rca_attn.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rca {

// Positions of one request handled by one work item of the decode kernel. A
// request of length L yields ceil(L / kDecodeChunk) items per KV head group;
// requests with one item write their output directly, longer ones leave one
// partial (max, sum, unnormalised output) per item for the combine kernel.
#ifndef DEC_CHUNK
#define DEC_CHUNK 256
#endif
constexpr int kDecodeChunk = DEC_CHUNK;

// Largest request count the decode kernel accepts: each CTA keeps the prefix
// sums of the per-request item counts in shared memory (4 bytes a request).
constexpr int64_t kDecodeMaxBatch = 8192;

struct DecodeParams {
  const void* q;             // [B, Hq, Dh]
  const void* k_pool;        // [P, Hkv, page_size, Dh]
  const void* v_pool;        // [P, Hkv, page_size, Dh]
  const int32_t* page_table; // [B, max_pages]
  const int32_t* seq_lens;   // [B]
  void* out;                 // [B, Hq, Dh]
  float* lse;                // [B, Hq]
  float* part_ml;            // [B, Hq, max_chunks, 2]   (workspace)
  float* part_acc;           // [B, Hq, max_chunks, Dh]  (workspace)
  int* status;
  int64_t B, Hq, Hkv, Dh, page_size, max_pages, num_pages;
  bool bf16;
  int sms;
  unsigned long long timeout_ns;  // device-side wait limit
};

inline int64_t decode_max_chunks(int64_t page_size, int64_t max_pages) {
  return (page_size * max_pages + kDecodeChunk - 1) / kDecodeChunk;
}

// Enqueues the decode kernel and, when some request can span several items,
// the combine kernel (a programmatic dependent launch). Arguments are validated
// by the caller.
cudaError_t launch_paged_decode(const DecodeParams& p, cudaStream_t st);

}  // namespace rca
