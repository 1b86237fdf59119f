// Variable-length batches: work lists that leave out the tiles made only of
// padding, and the zero fill of the rows those tiles would have written.
//
// A batch of B sequences is right-padded to T positions; sequence b has
// nq_b = ceil(L_b / 128) tiles of 128 positions that hold real tokens.
//  * forward items (b, h, qt) exist for qt < nq_b; an item of query tile qt
//    has qt + 1 key tiles, so the list is ordered by decreasing qt (the order
//    the dense schedule uses, longest items first);
//  * backward items (b, kvh, j) exist for key tiles j < nq_b and iterate over
//    the n_i = nq_b - j query tiles j .. nq_b - 1, so the list is ordered by
//    decreasing n_i.
// One CTA builds both lists: a counting sort of the sequences by nq_b gives,
// for every level, the sequences that reach it as a prefix of the sorted
// order, and prefix sums over the levels give where each level starts.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "bwd.cuh"
#include "tc.cuh"

namespace rca {

constexpr int kVarlenPlanThreads = 1024;

struct VarlenPlanArgs {
  const int* lens;
  int4* fwd_items;  // {b, h, qt, 0}
  int* fwd_count;
  int4* bwd_items;  // {b, kvh, j, n_i}
  int* bwd_count;
  int* status;
  int B, Hq, Hkv, T, n_qt;
};

// Shared memory sm: nq[B], order[B], cnt[n_qt + 1] (#sequences with
// nq_b > l for level l), fwd_off[n_qt + 1], bwd_off[n_qt + 1]. One block, any
// number of threads.
__device__ __forceinline__ void varlen_plan_block(const VarlenPlanArgs& a, int* sm) {
  int* nq = sm;
  int* order = nq + a.B;
  int* cnt = order + a.B;           // cnt[l] = #{b : nq_b > l}, l = 0 .. n_qt
  int* fwd_off = cnt + a.n_qt + 1;  // start of forward level l (qt = n_qt - 1 - l)
  int* bwd_off = fwd_off + a.n_qt + 1;  // start of backward level l (n_i = n_qt - l)
  const int tid = threadIdx.x;
  for (int l = tid; l <= a.n_qt; l += blockDim.x) cnt[l] = 0;
  __syncthreads();
  for (int b = tid; b < a.B; b += blockDim.x) {
    int L = __ldg(a.lens + b);
    if (L < 0 || L > a.T) {
      atomicExch(a.status, kStatusBadInput);
      L = L < 0 ? 0 : a.T;
    }
    nq[b] = (L + 127) / 128;
    atomicAdd(&cnt[nq[b]], 1);  // histogram of nq for now
  }
  __syncthreads();
  if (tid == 0) {
    // Counting sort by decreasing nq: first slot of each value's run.
    int pos = 0;
    for (int v = a.n_qt; v >= 0; --v) {
      const int c = cnt[v];
      cnt[v] = pos;
      pos += c;
    }
  }
  __syncthreads();
  for (int b = tid; b < a.B; b += blockDim.x) order[atomicAdd(&cnt[nq[b]], 1)] = b;
  __syncthreads();
  if (tid == 0) {
    // cnt[v] is now the end of value v's run = #{b : nq_b >= v}; shift to
    // #{b : nq_b > l} = #{b : nq_b >= l + 1}, then the level offsets.
    for (int l = 0; l < a.n_qt; ++l) cnt[l] = cnt[l + 1];
    cnt[a.n_qt] = 0;
    int f = 0, g = 0;
    for (int l = 0; l < a.n_qt; ++l) {
      fwd_off[l] = f;
      f += a.Hq * cnt[a.n_qt - 1 - l];  // query tile qt = n_qt - 1 - l: sequences with nq_b > qt
      bwd_off[l] = g;
      g += a.Hkv * cnt[a.n_qt - 1 - l];  // n_i = n_qt - l: sequences with nq_b >= n_i
    }
    fwd_off[a.n_qt] = f;
    bwd_off[a.n_qt] = g;
    *a.fwd_count = f;
    *a.bwd_count = g;
  }
  __syncthreads();
  // Entry e of a level: rank r = e / heads among the sorted sequences that
  // reach the level, head e % heads.
  auto level_of = [&](const int* off, int e) {
    int lo = 0, hi = a.n_qt;  // off[lo] <= e < off[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= e) lo = mid;
      else hi = mid;
    }
    return lo;
  };
  const int nf = fwd_off[a.n_qt];
  for (int e = tid; e < nf; e += blockDim.x) {
    const int l = level_of(fwd_off, e), r = (e - fwd_off[l]) / a.Hq, h = (e - fwd_off[l]) % a.Hq;
    a.fwd_items[e] = make_int4(order[r], h, a.n_qt - 1 - l, 0);
  }
  const int nb = bwd_off[a.n_qt];
  for (int e = tid; e < nb; e += blockDim.x) {
    const int l = level_of(bwd_off, e), r = (e - bwd_off[l]) / a.Hkv, kvh = (e - bwd_off[l]) % a.Hkv;
    const int b = order[r], ni = a.n_qt - l;
    a.bwd_items[e] = make_int4(b, kvh, nq[b] - ni, ni);
  }
}

__global__ void __launch_bounds__(kVarlenPlanThreads) varlen_plan_kernel(const VarlenPlanArgs a) {
  grid_dep_sync();
  extern __shared__ int sm[];
  varlen_plan_block(a, sm);
}

// Zero the rows of positions t >= L_b of a [B, T, H, Dh] tensor (storage
// dtype, ES bytes) and, if lse is given, set lse[b, h, t] = -inf there: block
// bx of the gx blocks given to sequence b. The padding is one contiguous range
// of 16-byte vectors, [L_b * vpr, T * vpr) of the sequence's slab, so no
// thread divides to find its row and none touches a real row.
template <int ES>
__device__ __forceinline__ void varlen_zero_block(void* __restrict__ x, float* __restrict__ lse,
                                                  const int* __restrict__ lens, int T, int H, int Dh, int b,
                                                  unsigned bx, unsigned gx) {
  int L = __ldg(lens + b);
  L = L < 0 ? 0 : (L > T ? T : L);
  const long long vpr = static_cast<long long>(H) * Dh * ES / 16;  // vectors per position
  uint4* slab = reinterpret_cast<uint4*>(x) + static_cast<long long>(b) * T * vpr;
  const long long stride = static_cast<long long>(gx) * blockDim.x;
  const long long first = static_cast<long long>(bx) * blockDim.x + threadIdx.x;
  for (long long i = L * vpr + first; i < T * vpr; i += stride) slab[i] = make_uint4(0, 0, 0, 0);
  if (lse) {
    const int np = T - L;  // padding positions of each head's LSE row
    for (long long k = first; k < static_cast<long long>(H) * np; k += stride) {
      const int h = static_cast<int>(k / np), t = L + static_cast<int>(k - static_cast<long long>(h) * np);
      lse[(static_cast<long long>(b) * H + h) * T + t] = -INFINITY;
    }
  }
}

// The same as a kernel: blockIdx.y is the sequence; blockIdx.z = 1 (when x2 is
// given) zeroes the padding of x2 instead, a second tensor of the same shape.
template <int ES>
__global__ void __launch_bounds__(256)
    varlen_zero_kernel(void* __restrict__ x, void* __restrict__ x2, float* __restrict__ lse,
                       const int* __restrict__ lens, int T, int H, int Dh) {
  grid_dep_sync();
  if (blockIdx.z == 1) {
    x = x2;
    lse = nullptr;
  }
  varlen_zero_block<ES>(x, lse, lens, T, H, Dh, blockIdx.y, blockIdx.x, gridDim.x);
}

// One launch ahead of a variable-length call's attention kernel, 256 threads a
// block: block 0 builds the work lists; the next nz = zgx * B * (x2 ? 2 : 1)
// blocks zero the padding rows of x (and x2; LSE -inf with x) as above, zgx
// blocks a sequence; the last pgx * B blocks (backward only) run the
// preprocess over the rows of real tiles, pgx blocks a sequence. The three
// parts touch disjoint memory and none reads what another writes, so they
// share one launch; the attention kernel after it waits for all of it
// (programmatic launch: its griddepcontrol.wait).
struct VarlenPrologue {
  VarlenPlanArgs plan;
  void* zx;
  void* zx2;
  float* zlse;
  int zH, Dh, zgx;
  PreArgs pre;
  int pgx;  // 0: no preprocess part
};

template <int ES, int PRE>  // PRE: 0 none, 1 bf16 storage, 2 fp32 storage
__global__ void __launch_bounds__(256) varlen_prologue_kernel(const VarlenPrologue p) {
  grid_dep_sync();
  extern __shared__ int sm[];
  unsigned blk = blockIdx.x;
  if (blk == 0) {
    varlen_plan_block(p.plan, sm);
    return;
  }
  blk -= 1;
  const unsigned B = static_cast<unsigned>(p.plan.B);
  const unsigned nz = static_cast<unsigned>(p.zgx) * B * (p.zx2 ? 2u : 1u);
  if (blk < nz) {
    const unsigned per = static_cast<unsigned>(p.zgx) * B;
    const bool second = blk >= per;
    const unsigned r = second ? blk - per : blk;
    varlen_zero_block<ES>(second ? p.zx2 : p.zx, second ? nullptr : p.zlse, p.plan.lens, p.plan.T, p.zH, p.Dh,
                          static_cast<int>(r / p.zgx), r % p.zgx, p.zgx);
    return;
  }
  if constexpr (PRE != 0) {
    blk -= nz;
    const unsigned pg = static_cast<unsigned>(p.pgx);
    preprocess_varlen_block<PRE == 2>(p.pre, static_cast<int>(blk / pg), blk % pg, pg);
  }
}

// dQ = scale * accumulator for a variable-length batch: blockIdx.y is the
// sequence b; rows t < L_b are converted, rows past it written as zeros
// without reading the accumulator (the backward leaves those rows stale).
// row4 = Hq * Dh / 4 float4 groups per position; U loads in flight per thread.
template <bool F32>
__global__ void __launch_bounds__(256)
    varlen_dq_convert_kernel(const float* __restrict__ acc, void* __restrict__ dq, const int* __restrict__ lens,
                             int T, long long row4, float scale) {
  grid_dep_sync();
  constexpr int U = 4;
  const int b = blockIdx.y;
  int L = __ldg(lens + b);
  L = L < 0 ? 0 : (L > T ? T : L);
  const long long base = static_cast<long long>(b) * T * row4, n = T * row4, real = L * row4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += U * stride) {
    float4 v[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const long long j = i + k * stride;
      v[k] = j < real ? reinterpret_cast<const float4*>(acc)[base + j] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const long long j = i + k * stride;
      if (j >= n) continue;
      if constexpr (F32) {
        reinterpret_cast<float4*>(dq)[base + j] =
            make_float4(v[k].x * scale, v[k].y * scale, v[k].z * scale, v[k].w * scale);
      } else {
        reinterpret_cast<uint2*>(dq)[base + j] = make_uint2(pack_bf16(v[k].x * scale, v[k].y * scale),
                                                           pack_bf16(v[k].z * scale, v[k].w * scale));
      }
    }
  }
}

}  // namespace rca
