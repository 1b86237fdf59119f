// Causal attention backward (vector-Jacobian product) for sm_103a.
//
// The riftco-transformer page "Execution Backends and the Python ABI", section
// "What the Metal slice does", specifies the memory-linear backward: scores and
// probabilities are recomputed from Q, K and the saved per-row statistics
// instead of reading a stored [T,T] probability tensor. With P = exp(S - LSE)
// the softmax VJP is
//   D = rowsum(dO * O),  dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),
//   dQ = scale dS K,     dK = scale dS^T Q.
// Grouped-query attention (algo-v1-codepoint "docs/ARCHITECTURE.md",
// "config.py"): dK and dV sum over the query heads that share a KV head.
//
// Three kernels:
//   attn_bwd_preprocess_kernel  -D and -LSE in base 2 (padded rows: 0 and -inf),
//                               zeroes the fp32 dQ accumulator. HBM-bound.
//   attn_bwd_main_kernel        work item = (batch, KV head, 128-key tile j); loops
//                               over every query head of the group and every query
//                               tile i >= j; dK, dV accumulate in TMEM; dQ partials
//                               are added into the fp32 accumulator. bf16 storage
//                               with a 64-column head: P^T stays in TMEM (dV reads
//                               it from there) and the CTAs are persistent, one per
//                               SM walking several items, with the next item's K/V
//                               and first S^T / dP^T fetched during the current
//                               item's last iteration; otherwise one CTA per item.
//   attn_bwd_dq_convert_kernel  dQ = scale * accumulator in the storage dtype.
//   split_hilo_kernel           fp32 storage only: bf16 hi/lo copies of Q, K, V, dO
//                               for the main kernel (see BwdCfg).
#pragma once

#include <type_traits>

#include "tc.cuh"

namespace rca {

// ----------------------------------------------------------------------------
// preprocess
// ----------------------------------------------------------------------------
struct PreArgs {
  const void* out;
  const float* lse;
  const void* dout;
  float* dq_acc;  // [B, T, Hq, Dh]
  float* lse2;    // [B, Hq, Tpad]  -LSE * log2(e); -inf on padded rows
  float* dvec;    // [B, Hq, Tpad]  -D; 0 on padded rows
  const int* lens;  // per-sequence lengths (right padding), or null
  int* status;
  int B, Hq, T, Dh, Tpad;
  int lg_lpr;     // log2 of the 16-byte segments per row (Dh * element size / 16)
  uint32_t hq_m;  // n / Hq = (umulhi(hq_m, n) + n) >> hq_l for n < 2^31
  int hq_l;
  int bpb;        // dense kernel: blocks per batch entry
};

// Segments (16 bytes of O and of dO) per thread in the dense kernel.
constexpr int kPreSegs = 1;

// Row r = t * Hq + h of one batch entry split into (t, h). For r < 2^31 the
// quotient is a multiply-high by a constant the host derives from Hq
// (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994); the sum below stays under 2^32 there.
__device__ __forceinline__ void pre_split_row(const PreArgs& a, uint32_t r, int& t, int& h) {
  const uint32_t q = (__umulhi(a.hq_m, r) + r) >> a.hq_l;
  t = static_cast<int>(q);
  h = static_cast<int>(r - q * static_cast<uint32_t>(a.Hq));
}
__device__ __forceinline__ void pre_split_row(const PreArgs& a, unsigned long long r, int& t, int& h) {
  t = static_cast<int>(r / static_cast<unsigned>(a.Hq));
  h = static_cast<int>(r - static_cast<unsigned long long>(t) * a.Hq);
}

// The share of rowsum(dO * O) held in one 16-byte segment of each.
template <bool F32>
__device__ __forceinline__ float pre_dot(const uint4 o, const uint4 g) {
  const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (F32) {
      acc = fmaf(__uint_as_float(ow[i]), __uint_as_float(gw[i]), acc);
    } else {
      const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[i]));
      const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[i]));
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
  }
  return acc;
}

// -D and base-2 -LSE of row (b, t, h); a padding row gets 0 and -inf, which
// keeps it out of the backward (its recomputed probabilities are exactly 0).
__device__ __forceinline__ void pre_write_row(const PreArgs& a, int b, int t, int h, bool real, float acc) {
  const size_t so = (static_cast<size_t>(b) * a.Hq + h) * a.Tpad + t;
  a.dvec[so] = real ? -acc : 0.f;
  a.lse2[so] = real ? -(a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.T + t] * 1.4426950408889634f) : -INFINITY;
}

// Dense preprocess. The rows of batch entry b, r = t * Hq + h for t < Tpad,
// are 2^lg_lpr consecutive 16-byte segments each, and segment s of the entry
// sits at 16-byte index s of its O and dO rows (contiguous [T, Hq, Dh]). Each
// block takes bpb-th of one entry: kPreSegs * 256 consecutive segments, one
// per thread per 256, all loads issued before any arithmetic. The lanes of a
// row are a power-of-two group of one warp, so its sum is a shuffle tree; the
// first lane of the row splits r into (t, h) and writes D and LSE2. Rows at
// or past T (or past the sequence's length) are padding: not read, their
// accumulator rows not zeroed (the conversion writes those dQ rows as zeros).
// WIDE: 64-bit segment indices (an entry with 2^31 or more segments).
template <bool F32, bool WIDE>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(const PreArgs a) {
  grid_dep_sync();
  using IT = typename std::conditional<WIDE, unsigned long long, uint32_t>::type;
  constexpr int ES = F32 ? 4 : 2;
  constexpr int Z4 = 16 / ES / 4;  // float4 groups of the accumulator per segment
  constexpr int U = kPreSegs;
  const int lg = a.lg_lpr;
  const IT pmask = (IT(1) << lg) - 1;
  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.bpb));
  const IT blk = blockIdx.x - static_cast<unsigned>(b) * static_cast<unsigned>(a.bpb);
  const IT nseg = (static_cast<IT>(a.Tpad) * static_cast<IT>(a.Hq)) << lg;
  IT real_rows = static_cast<IT>(a.T) * static_cast<IT>(a.Hq);
  if (a.lens) {
    int L = __ldg(a.lens + b);
    if (L < 0 || L > a.T) {
      if (threadIdx.x == 0) atomicExch(a.status, kStatusBadInput);
      L = L < 0 ? 0 : a.T;
    }
    real_rows = static_cast<IT>(L) * static_cast<IT>(a.Hq);
  }
  const size_t seg0 = static_cast<size_t>(b) * a.T * a.Hq << lg;  // the entry's first segment
  const uint4* ob = reinterpret_cast<const uint4*>(a.out) + seg0;
  const uint4* gb = reinterpret_cast<const uint4*>(a.dout) + seg0;
  float4* zb = reinterpret_cast<float4*>(a.dq_acc) + seg0 * Z4;
  const IT s0 = blk * static_cast<IT>(256 * U) + threadIdx.x;

  uint4 o[U], g[U];
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const IT s = s0 + static_cast<IT>(k * 256);
    if (s < nseg && (s >> lg) < real_rows) {
      o[k] = ob[s];
      g[k] = gb[s];
    } else {
      o[k] = make_uint4(0u, 0u, 0u, 0u);
      g[k] = o[k];
    }
  }
  float acc[U];
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const IT s = s0 + static_cast<IT>(k * 256);
    acc[k] = pre_dot<F32>(o[k], g[k]);
    if (s < nseg && (s >> lg) < real_rows) {
#pragma unroll
      for (int z = 0; z < Z4; ++z) zb[s * Z4 + z] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  const int lpr = 1 << lg;
#pragma unroll
  for (int k = 0; k < U; ++k)
    for (int x = lpr >> 1; x > 0; x >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], x, lpr);
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const IT s = s0 + static_cast<IT>(k * 256);
    if (s < nseg && (s & pmask) == 0) {
      const IT r = s >> lg;
      int t, h;
      pre_split_row(a, r, t, h);
      pre_write_row(a, b, t, h, r < real_rows, acc[k]);
    }
  }
}

// Variable-length batch, one block of the gx blocks (bx = 0 .. gx - 1) given to
// sequence b: only the rows the backward reads are visited, positions
// t < 128 * ceil(L_b / 128) (the query tiles that hold real rows). Real rows
// (t < L_b) get D and LSE2 and a zeroed accumulator row; the rest of their
// last tile gets D = 0, LSE2 = -inf. Rows past it are never read and not
// written. Segments as in the dense kernel, one per thread per pass; indices
// are 32-bit (the caller checks they fit). Run as part of the
// variable-length backward's prologue launch.
template <bool F32>
__device__ __forceinline__ void preprocess_varlen_block(const PreArgs& a, int b, unsigned bx, unsigned gx) {
  constexpr int ES = F32 ? 4 : 2;
  constexpr int Z4 = 16 / ES / 4;
  int L = __ldg(a.lens + b);
  if (L < 0 || L > a.T) {
    if (threadIdx.x == 0 && bx == 0) atomicExch(a.status, kStatusBadInput);
    L = L < 0 ? 0 : a.T;
  }
  const int lg = a.lg_lpr;
  const unsigned pmask = (1u << lg) - 1u;
  const unsigned rows = static_cast<unsigned>((L + 127) / 128 * 128) * a.Hq;  // (t, h) rows of real tiles
  const unsigned real_rows = static_cast<unsigned>(L) * a.Hq;
  const size_t seg0 = static_cast<size_t>(b) * a.T * a.Hq << lg;
  const uint4* ob = reinterpret_cast<const uint4*>(a.out) + seg0;
  const uint4* gb = reinterpret_cast<const uint4*>(a.dout) + seg0;
  float4* zb = reinterpret_cast<float4*>(a.dq_acc) + seg0 * Z4;
  const unsigned stride = gx * blockDim.x;
  const int lpr = 1 << lg;
  for (unsigned i0 = bx * blockDim.x; i0 < (rows << lg); i0 += stride) {  // uniform per block
    const unsigned s = i0 + threadIdx.x;
    const unsigned r = s >> lg;
    const bool in = r < rows;
    const bool real = r < real_rows;
    float acc = 0.f;
    if (real) {
      acc = pre_dot<F32>(ob[s], gb[s]);
#pragma unroll
      for (int z = 0; z < Z4; ++z) zb[static_cast<size_t>(s) * Z4 + z] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int x = lpr >> 1; x > 0; x >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, x, lpr);
    if (in && (s & pmask) == 0) {
      int t, h;
      pre_split_row(a, r, t, h);
      pre_write_row(a, b, t, h, real, acc);
    }
  }
}

// ----------------------------------------------------------------------------
// dQ convert
// ----------------------------------------------------------------------------
// Grid-stride over float4 groups, up to four loads in flight per thread per
// pass (the host launches one group per thread).
// STRIDED: the output rows (one position, all heads) are dq_row4 groups of 4
// elements apart instead of row4 (a row of a fused QKV gradient buffer).
template <bool F32, bool STRIDED>
__global__ void __launch_bounds__(256)
    attn_bwd_dq_convert_kernel(const float* __restrict__ acc, void* __restrict__ dq, long long n4,
                               float scale, long long row4, long long dq_row4) {
  grid_dep_sync();
  constexpr int U = 4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += U * stride) {
    float4 v[U];
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (i + k * stride < n4) v[k] = reinterpret_cast<const float4*>(acc)[i + k * stride];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      long long j = i + k * stride;
      if (j >= n4) continue;
      if constexpr (STRIDED) j = (j / row4) * dq_row4 + j % row4;
      if constexpr (F32) {
        reinterpret_cast<float4*>(dq)[j] =
            make_float4(v[k].x * scale, v[k].y * scale, v[k].z * scale, v[k].w * scale);
      } else {
        reinterpret_cast<uint2*>(dq)[j] = make_uint2(pack_bf16(v[k].x * scale, v[k].y * scale),
                                                     pack_bf16(v[k].z * scale, v[k].w * scale));
      }
    }
  }
}

// ----------------------------------------------------------------------------
// fp32 storage mode: bf16 hi/lo split of an operand (x = hi + lo)
// ----------------------------------------------------------------------------
// STRIDED: source rows are src_row4 groups of 4 apart (a fused QKV buffer);
// the copies are contiguous.
template <bool STRIDED>
__global__ void __launch_bounds__(256)
    split_hilo_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ hi,
                      __nv_bfloat16* __restrict__ lo, long long n4, long long row4, long long src_row4) {
  grid_dep_sync();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const long long si = STRIDED ? (i / row4) * src_row4 + i % row4 : i;
    const float4 v = reinterpret_cast<const float4*>(src)[si];
    uint32_t h0, l0, h1, l1;
    split_bf16x2(v.x, v.y, h0, l0);
    split_bf16x2(v.z, v.w, h1, l1);
    reinterpret_cast<uint2*>(hi)[i] = make_uint2(h0, h1);
    reinterpret_cast<uint2*>(lo)[i] = make_uint2(l0, l1);
  }
}

// ----------------------------------------------------------------------------
// main
// ----------------------------------------------------------------------------
// All tensor-core operands are bf16 tiles with DHB head columns (128-byte
// swizzle, 64-column panels). bf16 storage: one part per operand. fp32 storage
// (HL): two parts, hi and lo, and every product A.B is computed as
// Ahi.Bhi + Ahi.Blo + Alo.Bhi with fp32 accumulation. (Products over key or
// query positions need MN-major operands; kind::tf32 gave no result with
// MN-major operands on this GPU, so fp32 storage uses the bf16 split.)
template <bool HL, int DHB>
struct BwdCfg {
  static constexpr int NPART = HL ? 2 : 1;
  static constexpr int PANEL = 128 * 128;
  static constexpr int DPANELS = DHB / 64;
  static constexpr int TILE = DPANELS * PANEL;          // one part of a 128-row operand tile
  static constexpr int OPND = NPART * TILE;             // all parts of it
  static constexpr int PT_HALF = 2 * PANEL;             // 128 x 128 bf16
  static constexpr int P_BYTES = NPART * PT_HALF;
  // bf16 storage with a 64-column head: P^T stays in TMEM (dV = P^T dO reads
  // its A operand from there), which frees the shared-memory P^T buffer for a
  // second K/V buffer, and CTAs are persistent: the next work item's K/V tiles
  // and first S^T / dP^T are fetched and computed during the current item's
  // last iteration.
  static constexpr bool PTB = !HL && DHB == 64;
  static constexpr int KVB = PTB ? 2 : 1;               // K/V buffers
  static constexpr int P_SMEM = PTB ? 0 : P_BYTES;      // shared-memory P^T buffer
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int STAGE_BYTES = 2 * OPND + 1024;   // Q, dO, LSE2[128], D[128]
  // dQ is staged as fp32, 32 columns at a time, for bulk tensor reductions in
  // a 16 KB panel of its own (per-thread vector reductions of a whole dQ
  // partial per iteration saturate the load/store queue).
  static constexpr int DQS_BYTES = PANEL;
  static constexpr int AVAIL = SMEM_LIMIT - 1024 - BAR_BYTES - KVB * 2 * OPND - DQS_BYTES;
  static constexpr int NQS_SEP = (AVAIL - P_SMEM - P_BYTES) / STAGE_BYTES;
  static constexpr int NQS_SHR = (AVAIL - P_BYTES) / STAGE_BYTES;
  // P^T and dS^T share one buffer only when separate buffers leave < 2 stages.
  static constexpr bool SHARE = !PTB && NQS_SEP < 2 && NQS_SHR > NQS_SEP;
  static constexpr int NQS_RAW = SHARE ? NQS_SHR : NQS_SEP;
  static constexpr int NQS = NQS_RAW > 4 ? 4 : NQS_RAW;
  static_assert(NQS >= 1, "backward needs at least one Q/dO stage");
  static constexpr int OFF_K = 0;                       // K of buffer x at OFF_K + x * 2 * OPND
  static constexpr int OFF_V = OPND;                    // V of buffer x at OFF_V + x * 2 * OPND
  static constexpr int OFF_P = KVB * 2 * OPND;
  static constexpr int OFF_DS = SHARE ? OFF_P : OFF_P + P_SMEM;
  static constexpr int OFF_DQS = OFF_DS + P_BYTES;
  static constexpr int OFF_STAGE = OFF_DQS + DQS_BYTES;
  static constexpr int OFF_BAR = OFF_STAGE + NQS * STAGE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  // TMEM columns
  static constexpr int TM_S = 0, TM_DP = 128, TM_DV = 256, TM_DK = 256 + DHB;
  // dQ gets its own columns when they fit; otherwise it reuses the dP^T columns
  // once both compute warpgroups have read dP^T.
  static constexpr bool DQ_ALIAS = 256 + 3 * DHB > 512;
  static constexpr int TM_DQ = DQ_ALIAS ? TM_DP : 256 + 2 * DHB;
  static constexpr int TM_P = 256 + 3 * DHB;            // PTB: P^T, query pair (2c, 2c+1) in column c
  static_assert(!PTB || TM_P + 64 <= 512, "TMEM budget for P^T");
  // S^T / dP^T of the next iteration are computed while this iteration's dK and
  // dQ products are pending; that needs a second Q/dO stage, separate P^T and
  // dS^T buffers and dQ columns of its own.
  static constexpr bool PREFETCH = (NQS >= 2) && !DQ_ALIAS && !SHARE;
  static_assert(!PTB || PREFETCH, "persistent CTAs assume the prefetch schedule");
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_T = make_idesc(false, 128, 128, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_KV = make_idesc(false, 128, DHB, false, true);   // dV, dK
  static constexpr uint32_t IDESC_Q = make_idesc(false, 128, DHB, true, true);     // dQ
  // Warpgroups (4 warps each): 0 dQ drain, 1 and 2 compute, 3 = TMA producer
  // (warp 12), MMA issuer (warp 13) and two idle warps. Registers are split
  // per warpgroup from the 128 per thread the CTA is launched with.
  static constexpr int NTHREADS = 512;
  static constexpr int LAUNCH_REGS = 128;
  static constexpr int REG_DQ = 64, REG_CTL = 96, REG_CMP = 176;
  static_assert(128 * REG_DQ + 256 * REG_CMP + 128 * REG_CTL <= NTHREADS * LAUNCH_REGS, "register split");
  // barriers
  static constexpr int B_KVF = 0;            // [KVB] K/V tiles of a work item landed
  static constexpr int B_KVE = B_KVF + KVB;  // [KVB] K/V buffer free (last dQ of its item done)
  static constexpr int B_QF = B_KVE + KVB;
  static constexpr int B_QE = B_QF + NQS;
  static constexpr int B_SR = B_QE + NQS;   // S^T(it) in TMEM
  static constexpr int B_DPR = B_SR + 1;    // dP^T(it) in TMEM
  static constexpr int B_PR = B_DPR + 1;    // [2] P^T half g written
  static constexpr int B_SDPF = B_PR + 2;   // S^T, dP^T of it read by both warpgroups
  static constexpr int B_DVD = B_SDPF + 1;  // [2] dV half g done (P^T in TMEM / shared P, dS buffer)
  static constexpr int B_DSR = B_DVD + 2;   // [2] dS^T half g written
  static constexpr int B_DQF = B_DSR + 2;   // dQ(it) in TMEM (all MMAs of it done)
  static constexpr int B_ITF = B_DQF + 1;   // dQ(it) drained by both warpgroups
  static constexpr int B_KVFREE = B_ITF + 1;  // dK, dV of a work item read (drain warpgroup)
  static constexpr int B_KVD = B_KVFREE + 1;   // dK, dV of a work item final (its last dK done)
  static constexpr int B_FIN = B_KVD + 1;
  // Aliased dQ columns: the drain stages the four 32-column blocks of a dQ
  // partial in the P^T and dS^T buffers (idle while dQ is drained) and
  // releases the columns as soon as they are read; this barrier (one arrival
  // per drain warp) says the bulk reductions have finished reading them.
  static constexpr int B_STGF = B_FIN + 1;
  static constexpr int NBAR = B_STGF + 1;
  static_assert(!DQ_ALIAS || (!SHARE && P_SMEM == 2 * PANEL * NPART && NPART == 1 && DHB == 128),
                "dQ staging in the P^T / dS^T buffers assumes separate 32 KB buffers");
  // parts multiplied for one product: (hi,hi) [, (hi,lo), (lo,hi)]
  static constexpr int NPROD = HL ? 3 : 1;
  __device__ static constexpr int pa(int t) { return t == 2 ? 1 : 0; }
  __device__ static constexpr int pb(int t) { return t == 1 ? 1 : 0; }
};

// bf16 tensor maps of every operand: [0] = bf16 storage or hi part, [1] = lo part;
// dq: the fp32 dQ accumulator [B,T,Hq,Dh], 128 rows x 32 columns per box.
struct BwdMaps {
  CUtensorMap q[2], k[2], v[2], dO[2], dq;
};

struct BwdArgs {
  void* dk;
  void* dv;
  long long dkv_row;   // elements between consecutive positions of dK, dV (Hkv * Dh if contiguous)
  const int4* items;       // variable-length batches: work list {b, kvh, j, n_i} (null: all items)
  const int* n_items_dev;  // its length (device)
  const float* lse2;   // [B, Hq, Tpad]
  const float* dvec;   // [B, Hq, Tpad]
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, Dh, group, n_t, Tpad;
  int n_items;  // B * Hkv * n_t work items (one key tile of one KV head each)
  float scale, scale_log2;
};

// Work item k (k = 0, 1, ...) of this CTA: items are ordered by decreasing
// work (key tile j = 0 of every KV head first: it meets every query tile) and
// dealt out in a snake over the grid (round k gives item k G + c for even k,
// k G + G - 1 - c for odd k). Item (b, kvh, j) runs n_it = group * (n_t - j)
// iterations: every query head of the group times query tiles j .. n_t - 1.
struct BwdItem {
  int b, kvh, j, n_i, n_it;
};
template <bool LIST>
__device__ __forceinline__ bool bwd_item(const BwdArgs& a, int k, BwdItem& it) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const long long idx = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if constexpr (LIST) {  // variable-length batch: the planned list (tiles of padding left out)
    if (idx >= __ldg(a.n_items_dev)) return false;
    const int4 e = __ldg(a.items + idx);
    it.b = e.x;
    it.kvh = e.y;
    it.j = e.z;
    it.n_i = e.w;
    it.n_it = a.group * it.n_i;
    return true;
  }
  if (idx >= a.n_items) return false;
  const int bk_count = a.B * a.Hkv;
  it.j = static_cast<int>(idx / bk_count);
  const int bk = static_cast<int>(idx % bk_count);
  it.b = bk / a.Hkv;
  it.kvh = bk % a.Hkv;
  it.n_i = a.n_t - it.j;
  it.n_it = a.group * it.n_i;
  return true;
}

// Thread row `rl` of one 64-column panel of a 128 x 128 bf16 (hi[/lo])
// operand tile, K-major with the 128-byte swizzle: 8 chunks of 8 values.
template <bool HL>
__device__ __forceinline__ void store_half_row_bf16(uint32_t panel, int rl, const float (&x)[64], int half_bytes) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t addr = panel + rl * 128 + ((c ^ (rl & 7)) << 4);
    if constexpr (HL) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) split_bf16x2(x[8 * c + 2 * i], x[8 * c + 2 * i + 1], hi[i], lo[i]);
      st_shared_v4(addr, hi[0], hi[1], hi[2], hi[3]);
      st_shared_v4(addr + half_bytes, lo[0], lo[1], lo[2], lo[3]);
    } else {
      st_shared_v4(addr, pack_bf16(x[8 * c], x[8 * c + 1]), pack_bf16(x[8 * c + 2], x[8 * c + 3]),
                   pack_bf16(x[8 * c + 4], x[8 * c + 5]), pack_bf16(x[8 * c + 6], x[8 * c + 7]));
    }
  }
}

template <bool HL, int DHB, bool LIST>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_main_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = BwdCfg<HL, DHB>;
  grid_dep_sync();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  auto stage = [&](int s) -> uint32_t { return sbase + C::OFF_STAGE + s * C::STAGE_BYTES; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A CTA past the end of a planned work list has no item at all.
  if constexpr (LIST) {
    if (static_cast<int>(blockIdx.x) >= __ldg(a.n_items_dev)) return;
  }

  if (threadIdx.x == 0) {
    for (int x = 0; x < C::KVB; ++x) {
      mbar_init(bar(C::B_KVF + x), 1);
      mbar_init(bar(C::B_KVE + x), 1);
    }
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(bar(C::B_QF + s), 1);
      mbar_init(bar(C::B_QE + s), 1);
    }
    mbar_init(bar(C::B_SR), 1);
    mbar_init(bar(C::B_DPR), 1);
    mbar_init(bar(C::B_SDPF), 256);
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar(C::B_PR + g), 128);
      mbar_init(bar(C::B_DVD + g), 1);
      mbar_init(bar(C::B_DSR + g), 128);
    }
    mbar_init(bar(C::B_DQF), 1);
    mbar_init(bar(C::B_ITF), 128);  // the dQ drain warpgroup
    mbar_init(bar(C::B_KVFREE), 128);  // the dQ drain warpgroup writes dK, dV
    mbar_init(bar(C::B_KVD), 1);
    mbar_init(bar(C::B_FIN), 1);
    mbar_init(bar(C::B_STGF), 4);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{a.status, abort_flag, a.timeout_ns};
  // Every role ends in end_role(): the TMEM owner (warp 13) waits until all
  // 512 threads have finished with TMEM and releases it; the others only
  // arrive. No code follows the role branches (each warpgroup runs with its
  // own register budget).
  auto end_role = [&]() {
    tc_fence_before();
    if (warp == 13) {
      named_bar(1, C::NTHREADS);
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    } else {
      named_bar_arrive(1, C::NTHREADS);
    }
  };

  // Every role walks the same sequence of work items; iterations are numbered
  // gi = 0, 1, ... across all of this CTA's items, and the Q/dO ring position
  // and every per-iteration barrier phase is a function of gi.
  if (warp >= 12) {
   reg_dealloc<C::REG_CTL>();
   if (warp == 12) {
    // ---------------- TMA producer (one elected thread) ----------------
    if (elect_one()) {
      for (int part = 0; part < C::NPART; ++part) {
        tma_prefetch_desc(&maps.q[part]);
        tma_prefetch_desc(&maps.k[part]);
        tma_prefetch_desc(&maps.v[part]);
        tma_prefetch_desc(&maps.dO[part]);
      }
      bool ok = true;
      int gi = 0, n = 0;
      BwdItem itm{};
      for (; ok && bwd_item<LIST>(a, n, itm); ++n) {
        // K_j, V_j of the item into K/V buffer n % KVB.
        const int x = n % C::KVB;
        if (n >= C::KVB && !mbar_wait(bar(C::B_KVE + x), ((n / C::KVB) - 1) & 1, w)) break;
        mbar_expect_tx(bar(C::B_KVF + x), 2 * C::OPND);
        for (int part = 0; part < C::NPART; ++part)
          for (int p = 0; p < C::DPANELS; ++p) {
            tma_load_4d(sbase + C::OFF_K + x * 2 * C::OPND + part * C::TILE + p * C::PANEL, &maps.k[part],
                        bar(C::B_KVF + x), p * 64, itm.kvh, itm.j * 128, itm.b);
            tma_load_4d(sbase + C::OFF_V + x * 2 * C::OPND + part * C::TILE + p * C::PANEL, &maps.v[part],
                        bar(C::B_KVF + x), p * 64, itm.kvh, itm.j * 128, itm.b);
          }
        for (int it = 0; it < itm.n_it; ++it, ++gi) {
          const int s = gi % C::NQS;
          if (gi >= C::NQS && !mbar_wait(bar(C::B_QE + s), ((gi / C::NQS) - 1) & 1, w)) {
            ok = false;
            break;
          }
          const int h = itm.kvh * a.group + it / itm.n_i;
          const int i = itm.j + it % itm.n_i;
          const uint32_t st = stage(s);
          mbar_expect_tx(bar(C::B_QF + s), 2 * C::OPND + 1024);
          for (int part = 0; part < C::NPART; ++part)
            for (int p = 0; p < C::DPANELS; ++p) {
              tma_load_4d(st + part * C::TILE + p * C::PANEL, &maps.q[part], bar(C::B_QF + s), p * 64, h, i * 128,
                          itm.b);
              tma_load_4d(st + C::OPND + part * C::TILE + p * C::PANEL, &maps.dO[part], bar(C::B_QF + s), p * 64,
                          h, i * 128, itm.b);
            }
          const size_t ro = (static_cast<size_t>(itm.b) * a.Hq + h) * a.Tpad + static_cast<size_t>(i) * 128;
          bulk_load(st + 2 * C::OPND, a.lse2 + ro, 512, bar(C::B_QF + s));
          bulk_load(st + 2 * C::OPND + 512, a.dvec + ro, 512, bar(C::B_QF + s));
        }
      }
      // Exit path: every load issued has landed before shared memory is
      // released. n K/V loads were issued, minus one if the loop left before
      // the load of item n - 1 (only when a wait gave up).
      const int nkv = n;
      for (int x = 0; x < C::KVB && x < nkv; ++x) {
        const int last = x + ((nkv - 1 - x) / C::KVB) * C::KVB;
        mbar_drain(bar(C::B_KVF + x), (last / C::KVB) & 1, a.timeout_ns);
      }
      for (int s = 0; s < C::NQS && s < gi; ++s) {
        const int last = s + ((gi - 1 - s) / C::NQS) * C::NQS;
        mbar_drain(bar(C::B_QF + s), (last / C::NQS) & 1, a.timeout_ns);
      }
    }
    __syncwarp();
   } else if (warp == 13) {
    // ---------------- tcgen05 MMA issuer (one elected thread) ----------------
    if (elect_one()) {
      // Shared-memory descriptors are built once and moved by constant
      // offsets (desc_add): the issuing thread shares its sub-partition with
      // compute warps, so every instruction it saves shortens the gaps
      // between products. K-major operands (16-byte leading offset) and
      // MN-major ones (a 64-column panel apart) of each buffer:
      const uint64_t k_km = make_sdesc(sbase + C::OFF_K, 16, 1024);        // K: A of S^T
      const uint64_t v_km = make_sdesc(sbase + C::OFF_V, 16, 1024);        // V: A of dP^T
      const uint64_t k_mn = make_sdesc(sbase + C::OFF_K, C::PANEL, 1024);  // K: B of dQ
      const uint64_t q_km = make_sdesc(stage(0), 16, 1024);                // Q: B of S^T
      const uint64_t q_mn = make_sdesc(stage(0), C::PANEL, 1024);          // Q: B of dK
      const uint64_t do_km = make_sdesc(stage(0) + C::OPND, 16, 1024);     // dO: B of dP^T
      const uint64_t do_mn = make_sdesc(stage(0) + C::OPND, C::PANEL, 1024);  // dO: B of dV
      const uint64_t ds_km = make_sdesc(sbase + C::OFF_DS, 16, 1024);      // dS^T: A of dK
      const uint64_t ds_mn = make_sdesc(sbase + C::OFF_DS, C::PANEL, 1024);  // dS: A of dQ
      const uint64_t p_km = make_sdesc(sbase + C::OFF_P, 16, 1024);        // P^T in shared memory: A of dV
      // S^T = K Q^T (M = keys, N = queries, K = head dim) into TMEM_S, for
      // iteration gi2 whose item uses K/V buffer x2.
      auto issue_s = [&](int gi2, int x2) {
        const uint64_t db = desc_add(q_km, (gi2 % C::NQS) * C::STAGE_BYTES);
        const uint64_t da = desc_add(k_km, x2 * 2 * C::OPND);
#pragma unroll
        for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
          for (int k = 0; k < DHB / 16; ++k) {
            const uint32_t off = (k / 4) * C::PANEL + (k % 4) * 32;
            mma_ss<false>(tmem + C::TM_S, desc_add(da, C::pa(t) * C::TILE + off),
                          desc_add(db, C::pb(t) * C::TILE + off), C::IDESC_T, (t > 0 || k > 0) ? 1u : 0u);
          }
        tc_commit(bar(C::B_SR));
      };
      // dP^T = V dO^T into TMEM_DP
      auto issue_dp = [&](int gi2, int x2) {
        const uint64_t db = desc_add(do_km, (gi2 % C::NQS) * C::STAGE_BYTES);
        const uint64_t da = desc_add(v_km, x2 * 2 * C::OPND);
#pragma unroll
        for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
          for (int k = 0; k < DHB / 16; ++k) {
            const uint32_t off = (k / 4) * C::PANEL + (k % 4) * 32;
            mma_ss<false>(tmem + C::TM_DP, desc_add(da, C::pa(t) * C::TILE + off),
                          desc_add(db, C::pb(t) * C::TILE + off), C::IDESC_T, (t > 0 || k > 0) ? 1u : 0u);
          }
        tc_commit(bar(C::B_DPR));
      };
      BwdItem itm{};
      int n = 0, gi = 0;
      bool ok = bwd_item<LIST>(a, 0, itm);
      if (ok) ok = mbar_wait(bar(C::B_KVF), 0, w) && mbar_wait(bar(C::B_QF), 0, w);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        issue_dp(0, 0);
      }
      while (ok) {
        const int x = n % C::KVB;
        const uint64_t kx_mn = desc_add(k_mn, x * 2 * C::OPND);  // this item's K as the B operand of dQ
        BwdItem nxt{};
        const bool has_next = bwd_item<LIST>(a, n + 1, nxt);
        for (int it = 0; ok && it < itm.n_it; ++it, ++gi) {
          const int s = gi % C::NQS;
          const uint64_t qs_mn = desc_add(q_mn, s * C::STAGE_BYTES), dos_mn = desc_add(do_mn, s * C::STAGE_BYTES);
          // The next iteration: in this item, or the first of the next item.
          const bool more_here = it + 1 < itm.n_it;
          const bool more = more_here || (C::KVB > 1 && has_next);
          if constexpr (C::PREFETCH) {
            // The next iteration's S^T and dP^T go first: they need only this
            // iteration's S^T / dP^T to have been read (and the next Q/dO
            // stage), so the compute warps find them ready when they finish
            // this iteration.
            if (more) {
              const int x2 = more_here ? x : (n + 1) % C::KVB;
              if (!mbar_wait(bar(C::B_QF + (gi + 1) % C::NQS), ((gi + 1) / C::NQS) & 1, w) ||
                  (!more_here && !mbar_wait(bar(C::B_KVF + x2), ((n + 1) / C::KVB) & 1, w)) ||
                  !mbar_wait(bar(C::B_SDPF), gi & 1, w)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(gi + 1, x2);
              issue_dp(gi + 1, x2);
            }
          }
          // The previous item's dK and dV must have been read before this
          // item's first products overwrite them (waited here, after the
          // prefetch above, so that S^T / dP^T never wait for it).
          if (it == 0 && n >= 1 && !mbar_wait(bar(C::B_KVFREE), (n - 1) & 1, w)) {
            ok = false;
            break;
          }
          // dV += P^T dO, one query half per warpgroup as soon as it is written
          // (M = keys, N = head dim, K = queries 64g .. 64g+63).
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!mbar_wait(bar(C::B_PR + g), gi & 1, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
              for (int k = 4 * g; k < 4 * g + 4; ++k) {
                const uint32_t acc = (it > 0 || g > 0 || t > 0 || k > 0) ? 1u : 0u;
                const uint64_t bd = desc_add(dos_mn, C::pb(t) * C::TILE + k * 16 * 128);
                if constexpr (C::PTB) {
                  mma_ts(tmem + C::TM_DV, tmem + C::TM_P + 8 * k, bd, C::IDESC_KV, acc);
                } else {
                  const uint32_t aoff = (k / 4) * C::PANEL + (k % 4) * 32;
                  mma_ss<false>(tmem + C::TM_DV, desc_add(p_km, C::pa(t) * C::PT_HALF + aoff), bd, C::IDESC_KV, acc);
                }
              }
            // P^T half g is free again once this product is done (it no longer
            // precedes the next S^T / dP^T in issue order).
            if constexpr (C::SHARE || C::PTB) tc_commit(bar(C::B_DVD + g));
          }
          if (!ok) break;
          // dK += dS^T Q, one query half at a time (M = keys, N = head dim).
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!mbar_wait(bar(C::B_DSR + g), gi & 1, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
              for (int k = 4 * g; k < 4 * g + 4; ++k) {
                const uint32_t aoff = (k / 4) * C::PANEL + (k % 4) * 32;
                mma_ss<false>(tmem + C::TM_DK, desc_add(ds_km, C::pa(t) * C::PT_HALF + aoff),
                              desc_add(qs_mn, C::pb(t) * C::TILE + k * 16 * 128), C::IDESC_KV,
                              (it > 0 || g > 0 || t > 0 || k > 0) ? 1u : 0u);
              }
          }
          if (!ok) break;
          // The Q/dO stage is no longer read (dQ reads dS^T and K): release it now.
          tc_commit(bar(C::B_QE + s));
          if (!more_here) tc_commit(bar(C::B_KVD));  // the item's dK and dV are final
          // dQ partial = dS K (M = queries, N = head dim, K = keys): the previous
          // partial must have been drained, and (aliased columns) dP^T fully read.
          if (gi > 0 && !mbar_wait(bar(C::B_ITF), (gi - 1) & 1, w)) {
            ok = false;
            break;
          }
          if constexpr (!C::PREFETCH) {
            if (!mbar_wait(bar(C::B_SDPF), gi & 1, w)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
#pragma unroll
          for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
            for (int k = 0; k < 128 / 16; ++k)
              mma_ss<false>(tmem + C::TM_DQ, desc_add(ds_mn, C::pa(t) * C::PT_HALF + k * 16 * 128),
                            desc_add(kx_mn, C::pb(t) * C::TILE + k * 16 * 128), C::IDESC_Q, (t > 0 || k > 0) ? 1u : 0u);
          tc_commit(bar(C::B_DQF));
          if (!more_here) tc_commit(bar(C::B_KVE + x));  // the item's last read of K and V
          if constexpr (!C::PREFETCH) {
            if (more_here) {
              // With aliased dQ columns, dP^T(gi+1) may only be written once
              // dQ(gi) has been drained.
              if (!mbar_wait(bar(C::B_QF + (gi + 1) % C::NQS), ((gi + 1) / C::NQS) & 1, w) ||
                  (C::DQ_ALIAS && !mbar_wait(bar(C::B_ITF), gi & 1, w))) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(gi + 1, x);
              issue_dp(gi + 1, x);
            }
          }
        }
        if (!ok || !has_next || C::KVB == 1) break;
        itm = nxt;
        ++n;
      }
      // Exit path: all issued MMAs finish before TMEM is released.
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
    __syncwarp();
   }
   end_role();  // warps 14 and 15 have no role
  } else if (warp < 4) {
    reg_dealloc<C::REG_DQ>();
    // ---------------- dQ drain warpgroup ----------------
    // It also writes each work item's dK and dV once the item's last product
    // is done, so the compute warpgroups go straight on to the next item.
    // Warp q reads TMEM lanes 32 q .. 32 q + 31 (query rows) of every dQ
    // partial, 32 head columns at a time, and adds them to the fp32
    // accumulator: each 32 x 32 block is staged in the warp's 4 KB,
    // 128-byte-swizzled slice of the staging panel and added with a bulk
    // tensor reduction issued by the warp's lane 0 (the slice is rewritten only
    // after that lane's previous reduction has read it).
    const int quarter = warp;
    const int rl = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = true;
    int gi = 0;
    BwdItem itm{};
    for (int n = 0; ok && bwd_item<LIST>(a, n, itm); ++n) {
      for (int it = 0; it < itm.n_it; ++it, ++gi) {
        if (it == itm.n_it - 1) {
          // ---- dK, dV of the item, written as soon as its last dK product is
          // done (before its last dQ is drained). Key row rl of the key tile,
          // 32 head columns at a time; dK carries the softmax scale.
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_KVD), n & 1, w));
          if (!ok) break;
          tc_fence_after();
          const int key = itm.j * 128 + rl;
          const bool valid = key < a.T;
          const size_t row_off = (static_cast<size_t>(itm.b) * a.T + key) * a.dkv_row + static_cast<size_t>(itm.kvh) * a.Dh;
#pragma unroll
          for (int which = 0; which < 2; ++which) {
#pragma unroll
            for (int c = 0; c < DHB / 32; ++c) {
              uint32_t r[32];
              tmem_ld32(tl + (which == 0 ? C::TM_DV : C::TM_DK) + 32 * c, r);
              if (which == 1 && c == DHB / 32 - 1) {
                tc_fence_before();
                mbar_arrive(bar(C::B_KVFREE));  // the next item's products may overwrite dK, dV
              }
              const float mul = which == 0 ? 1.f : a.scale;
              const int ncol = a.Dh - 32 * c;
              if (!valid || ncol <= 0) continue;
              void* base = which == 0 ? a.dv : a.dk;
              if constexpr (HL) {
                float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + row_off + 32 * c);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  if (4 * u < ncol)
                    dst[u] = make_float4(__uint_as_float(r[4 * u]) * mul, __uint_as_float(r[4 * u + 1]) * mul,
                                         __uint_as_float(r[4 * u + 2]) * mul, __uint_as_float(r[4 * u + 3]) * mul);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row_off + 32 * c);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                  if (8 * u < ncol)
                    dst[u] = make_uint4(
                        pack_bf16(__uint_as_float(r[8 * u]) * mul, __uint_as_float(r[8 * u + 1]) * mul),
                        pack_bf16(__uint_as_float(r[8 * u + 2]) * mul, __uint_as_float(r[8 * u + 3]) * mul),
                        pack_bf16(__uint_as_float(r[8 * u + 4]) * mul, __uint_as_float(r[8 * u + 5]) * mul),
                        pack_bf16(__uint_as_float(r[8 * u + 6]) * mul, __uint_as_float(r[8 * u + 7]) * mul));
              }
            }
          }
        }
        const int h = itm.kvh * a.group + it / itm.n_i;
        const int i = itm.j + it % itm.n_i;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DQF), gi & 1, w));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < DHB / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tl + C::TM_DQ + 32 * c, r);
          if (c == DHB / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(C::B_ITF));  // dQ(gi) read: its columns may be overwritten
          }
          // Aliased dQ columns: block c goes to its own slice of the P^T / dS^T
          // buffers (no wait between blocks); otherwise the one staging panel,
          // rewritten once the previous block's reduction has read it.
          const uint32_t panel = C::DQ_ALIAS ? sbase + C::OFF_P + c * 16384 : sbase + C::OFF_DQS;
          if (!C::DQ_ALIAS && lane == 0) bulk_wait_read0();
          __syncwarp();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_shared_v4(panel + rl * 128 + ((k ^ (rl & 7)) << 4), r[4 * k], r[4 * k + 1], r[4 * k + 2],
                         r[4 * k + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            // A block past the head width has nothing to add; columns and rows
            // past the tensor's edge (a head narrower than the 32-column box, a
            // partial last query tile) are clipped by the reduction itself.
            if (32 * c < a.Dh)
              tma_reduce_add_4d(&maps.dq, panel + quarter * 4096, 32 * c, h, i * 128 + quarter * 32, itm.b);
            bulk_commit();
          }
        }
        if constexpr (C::DQ_ALIAS) {
          // The next iteration's P^T and dS^T may overwrite the slices once
          // these reductions have read them.
          if (lane == 0) {
            bulk_wait_read0();
            mbar_arrive(bar(C::B_STGF));
          }
          __syncwarp();
        }
      }
    }
    if (lane == 0) bulk_wait0();  // every bulk reduction this warp issued has landed
    __syncwarp();
    end_role();
  } else {
    reg_alloc<C::REG_CMP>();
    // ---------------- compute warpgroups ----------------
    // Warpgroup g owns query columns 64g .. 64g+63 of every S^T / dP^T tile.
    const int g = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // key row of P^T / dS^T
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    bool ok = true;
    int gi = 0;
    BwdItem itm{};
    for (int n = 0; ok && bwd_item<LIST>(a, n, itm); ++n) {
      const int j = itm.j;
      for (int it = 0; it < itm.n_it; ++it, ++gi) {
        const int s = gi % C::NQS;
        const int i = j + it % itm.n_i;  // query tile
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SR), gi & 1, w) &&
                                         mbar_wait(bar(C::B_QF + s), (gi / C::NQS) & 1, w));
        if (!ok) break;
        const float* lse2s = reinterpret_cast<const float*>(smem + (stage(s) - sbase) + 2 * C::OPND) + 64 * g;
        const float* dvs = lse2s + 128;
        float p[64];
        uint32_t dpr[64];  // prefetch schedule: dP^T half, loaded together with S^T
        if constexpr (C::PREFETCH) {
          // S^T(gi) and dP^T(gi) are issued together: one TMEM round trip for both.
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DPR), gi & 1, w));
          if (!ok) break;
          tc_fence_after();
          uint32_t r[64];
          tmem_ld64x2(tl + C::TM_S + 64 * g, tl + C::TM_DP + 64 * g, r, dpr);
          tc_fence_before();
          mbar_arrive(bar(C::B_SDPF));
#pragma unroll
          for (int q = 0; q < 64; ++q) p[q] = __uint_as_float(r[q]);
        } else {
          tc_fence_after();
          uint32_t r[64];
          tmem_ld64(tl + C::TM_S + 64 * g, r);
#pragma unroll
          for (int q = 0; q < 64; ++q) p[q] = __uint_as_float(r[q]);
        }
        // P^T = 2^(S^T * scale * log2 e - LSE * log2 e) (the stage holds the
        // negated base-2 LSE), two columns per packed FMA; key rl is after query
        // 64g + c on the diagonal tile: dropped.
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(lse2s + c);
          float x0, x1, x2, x3;
          f2unpack(ffma2(f2pack(p[c], p[c + 1]), sl2x2, f2pack(l4.x, l4.y)), x0, x1);
          f2unpack(ffma2(f2pack(p[c + 2], p[c + 3]), sl2x2, f2pack(l4.z, l4.w)), x2, x3);
          p[c] = ex2(x0);
          p[c + 1] = ex2(x1);
          p[c + 2] = ex2(x2);
          p[c + 3] = ex2(x3);
        }
        if (i == j) {  // diagonal tile (uniform across the CTA)
          const int lim = rl - 64 * g;
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < lim) p[c] = 0.f;
        }
        if constexpr (C::PTB) {
          // P^T half g in TMEM was last read by dV(gi - 1).
          if (gi > 0) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DVD + g), (gi - 1) & 1, w));
            if (!ok) break;
            tc_fence_after();
          }
          // P^T row -> TMEM: queries (2c, 2c + 1) of this half in column 32 g + c.
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(p[32 * hh + 2 * c], p[32 * hh + 2 * c + 1]);
            tmem_st16(tl + C::TM_P + 32 * g + 16 * hh, pk);
          }
        } else {
          if constexpr (C::DQ_ALIAS) {
            // The P^T / dS^T buffers held dQ(gi - 1) blocks for its reductions.
            if (gi > 0) {
              ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_STGF), (gi - 1) & 1, w));
              if (!ok) break;
            }
          }
          store_half_row_bf16<HL>(sbase + C::OFF_P + g * C::PANEL, rl, p, C::PT_HALF);
          fence_async_smem();
        }
        tc_fence_before();
        mbar_arrive(bar(C::B_PR + g));
        // dS^T = P^T * (dP^T - D)
        if constexpr (!C::PREFETCH) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DPR), gi & 1, w));
          if (!ok) break;
          tc_fence_after();
          tmem_ld64(tl + C::TM_DP + 64 * g, dpr);
          tc_fence_before();
          mbar_arrive(bar(C::B_SDPF));
        }
        // (the stage holds -D), two columns per packed add and multiply
#pragma unroll
        for (int q = 0; q < 64; q += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dvs + q);
          float y0, y1, y2, y3;
          f2unpack(fmul2(f2pack(p[q], p[q + 1]),
                         fadd2(f2pack(__uint_as_float(dpr[q]), __uint_as_float(dpr[q + 1])), f2pack(d4.x, d4.y))),
                   y0, y1);
          f2unpack(fmul2(f2pack(p[q + 2], p[q + 3]),
                         fadd2(f2pack(__uint_as_float(dpr[q + 2]), __uint_as_float(dpr[q + 3])), f2pack(d4.z, d4.w))),
                   y2, y3);
          p[q] = y0;
          p[q + 1] = y1;
          p[q + 2] = y2;
          p[q + 3] = y3;
        }
        // The dS^T buffer is free once dK(gi-1) and dQ(gi-1) are done.
        if (gi > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DQF), (gi - 1) & 1, w));
          if (!ok) break;
        }
        if constexpr (C::SHARE) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DVD + g), gi & 1, w));
          if (!ok) break;
        }
        store_half_row_bf16<HL>(sbase + C::OFF_DS + g * C::PANEL, rl, p, C::PT_HALF);
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::B_DSR + g));
      }
      if (!ok) break;
    }
    end_role();
  }
}

}  // namespace rca
