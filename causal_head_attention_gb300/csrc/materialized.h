// Internal interface between the C ABI (rca_attn.cu) and the materialized
// attention path (materialized.cu). Not installed; callers use include/rca_attn.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

namespace rca {

struct MatParams {
  const void* q;      // [B,T,Hq,Dh]  storage dtype
  const void* k;      // [B,T,Hkv,Dh]
  const void* v;      // [B,T,Hkv,Dh]
  const void* dout;   // [B,T,Hq,Dh]  (backward)
  const float* dprobs;  // [B,Hq,T,T] upstream gradient of the probabilities, or null (backward)
  float* probs;       // [B,Hq,T,T]  written by the forward, read by the backward
  float* lse;         // [B,Hq,T]    (forward)
  void* out;          // [B,T,Hq,Dh] (forward)
  void* dq;           // [B,T,Hq,Dh] (backward)
  void* dk;           // [B,T,Hkv,Dh]
  void* dv;           // [B,T,Hkv,Dh]
  int64_t B, Hq, Hkv, T, Dh;
  bool bf16;
  void* workspace;
  size_t workspace_bytes;
  int* status;                    // the library's device status word (bounded waits)
  unsigned long long timeout_ns;  // device-side wait limit
};

// TMA descriptor of a [B, T, H, Dh] bf16 tensor, boxes of one 64-element
// (128-byte, swizzled) panel x one head x box_rows positions; positions past T
// and columns past Dh read as zero. Defined with the library's other
// descriptors (rca_attn.cu).
bool encode_rows_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t H, int64_t Dh,
                     unsigned box_rows, std::string& err);

// Bytes of scratch the materialized backward needs (the forward needs less).
size_t materialized_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, bool bf16);

// Enqueue the forward / backward on `st`. Arguments are validated by the
// caller. Returns false and fills `err` on a CUDA failure.
bool materialized_fwd(const MatParams& p, cudaStream_t st, std::string& err);
bool materialized_bwd(const MatParams& p, cudaStream_t st, std::string& err);

// The fused causal softmax and its VJP on N independent [T, T] score matrices
// (in place), as used by the two calls above.
bool causal_softmax_fwd(float* scores, float* lse, int64_t N, int64_t T, float scale, cudaStream_t st,
                        std::string& err);
// The VJP writes row i for columns j < min(T, tile * (i / tile + 1)) (tile >= T:
// whole rows).
bool causal_softmax_bwd(const float* probs, float* grad, const float* grad_extra, int64_t N, int64_t T, int64_t tile,
                        float scale, cudaStream_t st, std::string& err);

}  // namespace rca
