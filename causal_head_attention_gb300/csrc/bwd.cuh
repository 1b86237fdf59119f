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
//   attn_bwd_preprocess_kernel  D, LSE in base 2 (padded rows: D = 0, LSE = +inf),
//                               zeroes the fp32 dQ accumulator. HBM-bound.
//   attn_bwd_main_kernel        one CTA per (batch, KV head, 128-key tile j); loops
//                               over every query head of the group and every query
//                               tile i >= j; dK, dV accumulate in TMEM; dQ partials
//                               are added into the fp32 accumulator.
//   attn_bwd_dq_convert_kernel  dQ = scale * accumulator in the storage dtype.
//   split_hilo_kernel           fp32 storage only: bf16 hi/lo copies of Q, K, V, dO
//                               for the main kernel (see BwdCfg).
#pragma once

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
  float* lse2;    // [B, Hq, Tpad]
  float* dvec;    // [B, Hq, Tpad]
  int B, Hq, T, Dh, Tpad;
};

// A group of LPR consecutive lanes handles one (b, t, h) row of Dh elements,
// each lane 16 bytes, so every load instruction is fully coalesced.
template <bool F32>
__global__ void __launch_bounds__(256) attn_bwd_preprocess_kernel(const PreArgs a) {
  constexpr int ES = F32 ? 4 : 2;
  constexpr int EPL = 16 / ES;  // elements per lane
  const int lpr = a.Dh / EPL;   // lanes per row: power of two in [2, 32]
  const long long gid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long rows = static_cast<long long>(a.B) * a.Tpad * a.Hq;
  const long long row = gid / lpr;
  const int part = static_cast<int>(gid % lpr);
  const bool in = row < rows;
  int b = 0, t = 0, h = 0;
  if (in) {
    h = static_cast<int>(row % a.Hq);
    const long long bt = row / a.Hq;
    t = static_cast<int>(bt % a.Tpad);
    b = static_cast<int>(bt / a.Tpad);
  }
  const bool live = in && t < a.T;
  float acc = 0.f;
  if (live) {
    const size_t off = ((static_cast<size_t>(b) * a.T + t) * a.Hq + h) * a.Dh + part * EPL;
    const uint4 o = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.out) + off * ES);
    const uint4 g = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.dout) + off * ES);
    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
    const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
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
    float4* z = reinterpret_cast<float4*>(a.dq_acc + off);
#pragma unroll
    for (int i = 0; i < EPL / 4; ++i) z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int o = lpr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o, lpr);
  if (in && part == 0) {
    const size_t so = (static_cast<size_t>(b) * a.Hq + h) * a.Tpad + t;
    a.dvec[so] = live ? acc : 0.f;
    a.lse2[so] = live ? a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.T + t] * 1.4426950408889634f
                      : INFINITY;
  }
}

// ----------------------------------------------------------------------------
// dQ convert
// ----------------------------------------------------------------------------
template <bool F32>
__global__ void __launch_bounds__(256)
    attn_bwd_dq_convert_kernel(const float* __restrict__ acc, void* __restrict__ dq, long long n4,
                               float scale) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = reinterpret_cast<const float4*>(acc)[i];
    if constexpr (F32) {
      reinterpret_cast<float4*>(dq)[i] = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
    } else {
      reinterpret_cast<uint2*>(dq)[i] = make_uint2(pack_bf16(v.x * scale, v.y * scale),
                                                   pack_bf16(v.z * scale, v.w * scale));
    }
  }
}

// ----------------------------------------------------------------------------
// fp32 storage mode: bf16 hi/lo split of an operand (x = hi + lo)
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    split_hilo_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ hi,
                      __nv_bfloat16* __restrict__ lo, long long n4) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    const float4 v = reinterpret_cast<const float4*>(src)[i];
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
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int STAGE_BYTES = 2 * OPND + 1024;   // Q, dO, LSE2[128], D[128]
  // bf16 storage with a 64-column head: dQ halves are staged as fp32 for bulk
  // tensor reductions in a buffer of their own (two 16 KB panels).
  static constexpr bool TMA_DQ = !HL && DHB == 64;
  static constexpr int DQS_BYTES = TMA_DQ ? 2 * PANEL : 0;
  static constexpr int AVAIL = SMEM_LIMIT - 1024 - BAR_BYTES - 2 * OPND - DQS_BYTES;
  static constexpr int NQS_SEP = (AVAIL - 2 * P_BYTES) / STAGE_BYTES;
  static constexpr int NQS_SHR = (AVAIL - P_BYTES) / STAGE_BYTES;
  // P^T and dS^T share one buffer only when separate buffers leave < 2 stages.
  static constexpr bool SHARE = NQS_SEP < 2 && NQS_SHR > NQS_SEP;
  static constexpr int NQS_RAW = SHARE ? NQS_SHR : NQS_SEP;
  static constexpr int NQS = NQS_RAW > 4 ? 4 : NQS_RAW;
  static_assert(NQS >= 1, "backward needs at least one Q/dO stage");
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OPND;
  static constexpr int OFF_P = 2 * OPND;
  static constexpr int OFF_DS = SHARE ? OFF_P : OFF_P + P_BYTES;
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
  // S^T / dP^T of the next iteration are computed while this iteration's dK and
  // dQ products are pending; that needs a second Q/dO stage, separate P^T and
  // dS^T buffers and dQ columns of its own.
  static constexpr bool PREFETCH = (NQS >= 2) && !DQ_ALIAS && !SHARE;
  static_assert(!TMA_DQ || PREFETCH, "bulk dQ reduction assumes the prefetch schedule");
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_T = make_idesc(false, 128, 128, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_KV = make_idesc(false, 128, DHB, false, true);   // dV, dK
  static constexpr uint32_t IDESC_Q = make_idesc(false, 128, DHB, true, true);     // dQ
  static constexpr int NTHREADS = 320;
  // barriers
  static constexpr int B_KV = 0;
  static constexpr int B_QF = 1;
  static constexpr int B_QE = B_QF + NQS;
  static constexpr int B_SR = B_QE + NQS;   // S^T(it) in TMEM
  static constexpr int B_DPR = B_SR + 1;    // dP^T(it) in TMEM
  static constexpr int B_PR = B_DPR + 1;    // [2] P^T half g written
  static constexpr int B_SDPF = B_PR + 2;   // S^T, dP^T of it read by both warpgroups
  static constexpr int B_DVD = B_SDPF + 1;  // [2] dV half g done (shared P/dS buffer only)
  static constexpr int B_DSR = B_DVD + 2;   // [2] dS^T half g written
  static constexpr int B_DQF = B_DSR + 2;   // dQ(it) in TMEM (all MMAs of it done)
  static constexpr int B_ITF = B_DQF + 1;   // dQ(it) drained by both warpgroups
  static constexpr int B_FIN = B_ITF + 1;
  static constexpr int NBAR = B_FIN + 1;
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
  float* dq_acc;       // [B, T, Hq, Dh]
  const float* lse2;   // [B, Hq, Tpad]
  const float* dvec;   // [B, Hq, Tpad]
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, Dh, group, n_t, Tpad;
  float scale, scale_log2;
};

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

template <bool HL, int DHB>
__global__ void __launch_bounds__(320, 1)
    attn_bwd_main_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = BwdCfg<HL, DHB>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  auto stage = [&](int s) -> uint32_t { return sbase + C::OFF_STAGE + s * C::STAGE_BYTES; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bk_count = a.B * a.Hkv;
  const int lin = blockIdx.x;
  const int j = lin / bk_count;  // key tile; small j = most work, scheduled first
  const int bk = lin % bk_count;
  const int b = bk / a.Hkv, kvh = bk % a.Hkv;
  const int n_i = a.n_t - j;           // query tiles j .. n_t-1
  const int n_it = a.group * n_i;      // times every query head of the group

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KV), 1);
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
    mbar_init(bar(C::B_ITF), 256);
    mbar_init(bar(C::B_FIN), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{a.status, abort_flag, a.timeout_ns};

  if (warp == 0) {
    // ---------------- TMA producer (whole warp; one elected lane issues) ----------------
    const bool leader = elect_one();
    if (leader) {
      for (int part = 0; part < C::NPART; ++part) {
        tma_prefetch_desc(&maps.q[part]);
        tma_prefetch_desc(&maps.k[part]);
        tma_prefetch_desc(&maps.v[part]);
        tma_prefetch_desc(&maps.dO[part]);
      }
      mbar_expect_tx(bar(C::B_KV), 2 * C::OPND);
      for (int part = 0; part < C::NPART; ++part)
        for (int p = 0; p < C::DPANELS; ++p) {
          tma_load_4d(sbase + C::OFF_K + part * C::TILE + p * C::PANEL, &maps.k[part], bar(C::B_KV), p * 64,
                      kvh, j * 128, b);
          tma_load_4d(sbase + C::OFF_V + part * C::TILE + p * C::PANEL, &maps.v[part], bar(C::B_KV), p * 64,
                      kvh, j * 128, b);
        }
    }
    int it = 0;
    for (; it < n_it; ++it) {
      const int s = it % C::NQS;
      if (it >= C::NQS && !mbar_wait_warp(bar(C::B_QE + s), ((it / C::NQS) - 1) & 1, w)) break;
      const int h = kvh * a.group + it / n_i;
      const int i = j + it % n_i;
      const uint32_t st = stage(s);
      if (leader) {
        mbar_expect_tx(bar(C::B_QF + s), 2 * C::OPND + 1024);
        for (int part = 0; part < C::NPART; ++part)
          for (int p = 0; p < C::DPANELS; ++p) {
            tma_load_4d(st + part * C::TILE + p * C::PANEL, &maps.q[part], bar(C::B_QF + s), p * 64, h,
                        i * 128, b);
            tma_load_4d(st + C::OPND + part * C::TILE + p * C::PANEL, &maps.dO[part], bar(C::B_QF + s),
                        p * 64, h, i * 128, b);
          }
        const size_t ro = (static_cast<size_t>(b) * a.Hq + h) * a.Tpad + static_cast<size_t>(i) * 128;
        bulk_load(st + 2 * C::OPND, a.lse2 + ro, 512, bar(C::B_QF + s));
        bulk_load(st + 2 * C::OPND + 512, a.dvec + ro, 512, bar(C::B_QF + s));
      }
    }
    if (leader) {
      mbar_drain(bar(C::B_KV), 0, a.timeout_ns);
      for (int s = 0; s < C::NQS && s < it; ++s) {
        const int last = s + ((it - 1 - s) / C::NQS) * C::NQS;
        mbar_drain(bar(C::B_QF + s), (last / C::NQS) & 1, a.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- tcgen05 MMA issuer (whole warp; one elected lane issues) ----------------
    const bool leader = elect_one();
    const uint32_t kb = sbase + C::OFF_K, vb = sbase + C::OFF_V;
    const uint32_t pb = sbase + C::OFF_P, dsb = sbase + C::OFF_DS;
    // S^T = K Q^T (M = keys, N = queries, K = head dim) into TMEM_S
    auto issue_s = [&](int it2) {
      const uint32_t qb = stage(it2 % C::NQS);
#pragma unroll
      for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
        for (int k = 0; k < DHB / 16; ++k) {
          const uint32_t off = (k / 4) * C::PANEL + (k % 4) * 32;
          const uint64_t ad = make_sdesc(kb + C::pa(t) * C::TILE + off, 16, 1024);
          const uint64_t bd = make_sdesc(qb + C::pb(t) * C::TILE + off, 16, 1024);
          if (leader) mma_ss<false>(tmem + C::TM_S, ad, bd, C::IDESC_T, (t > 0 || k > 0) ? 1u : 0u);
        }
      if (leader) tc_commit(bar(C::B_SR));
    };
    // dP^T = V dO^T into TMEM_DP
    auto issue_dp = [&](int it2) {
      const uint32_t dob = stage(it2 % C::NQS) + C::OPND;
#pragma unroll
      for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
        for (int k = 0; k < DHB / 16; ++k) {
          const uint32_t off = (k / 4) * C::PANEL + (k % 4) * 32;
          const uint64_t ad = make_sdesc(vb + C::pa(t) * C::TILE + off, 16, 1024);
          const uint64_t bd = make_sdesc(dob + C::pb(t) * C::TILE + off, 16, 1024);
          if (leader) mma_ss<false>(tmem + C::TM_DP, ad, bd, C::IDESC_T, (t > 0 || k > 0) ? 1u : 0u);
        }
      if (leader) tc_commit(bar(C::B_DPR));
    };
    bool ok = mbar_wait_warp(bar(C::B_KV), 0, w) && mbar_wait_warp(bar(C::B_QF), 0, w);
    if (ok) {
      tc_fence_after();
      issue_s(0);
      issue_dp(0);
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it % C::NQS;
      const uint32_t qb = stage(s), dob = stage(s) + C::OPND;
      // dV += P^T dO, one query half per warpgroup as soon as it is written
      // (M = keys, N = head dim, K = queries 64g .. 64g+63).
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (!mbar_wait_warp(bar(C::B_PR + g), it & 1, w)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
          for (int k = 4 * g; k < 4 * g + 4; ++k) {
            const uint32_t aoff = (k / 4) * C::PANEL + (k % 4) * 32;
            const uint64_t ad = make_sdesc(pb + C::pa(t) * C::PT_HALF + aoff, 16, 1024);
            const uint64_t bd = make_sdesc(dob + C::pb(t) * C::TILE + k * 16 * 128, C::PANEL, 1024);
            if (leader)
              mma_ss<false>(tmem + C::TM_DV, ad, bd, C::IDESC_KV, (it > 0 || g > 0 || t > 0 || k > 0) ? 1u : 0u);
          }
        if constexpr (C::SHARE) {
          if (leader) tc_commit(bar(C::B_DVD + g));
        }
      }
      if (!ok) break;
      const bool more = it + 1 < n_it;
      if constexpr (C::PREFETCH) {
        // Next iteration's S^T and dP^T while dK and dQ of this one are pending.
        if (more) {
          if (!mbar_wait_warp(bar(C::B_QF + (it + 1) % C::NQS), ((it + 1) / C::NQS) & 1, w) ||
              !mbar_wait_warp(bar(C::B_SDPF), it & 1, w)) { ok = false; break; }
          tc_fence_after();
          issue_s(it + 1);
          issue_dp(it + 1);
        }
      }
      // dK += dS^T Q, one query half at a time (M = keys, N = head dim).
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (!mbar_wait_warp(bar(C::B_DSR + g), it & 1, w)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
          for (int k = 4 * g; k < 4 * g + 4; ++k) {
            const uint32_t aoff = (k / 4) * C::PANEL + (k % 4) * 32;
            const uint64_t ad = make_sdesc(dsb + C::pa(t) * C::PT_HALF + aoff, 16, 1024);
            const uint64_t bd = make_sdesc(qb + C::pb(t) * C::TILE + k * 16 * 128, C::PANEL, 1024);
            if (leader)
              mma_ss<false>(tmem + C::TM_DK, ad, bd, C::IDESC_KV, (it > 0 || g > 0 || t > 0 || k > 0) ? 1u : 0u);
          }
      }
      if (!ok) break;
      // The Q/dO stage is no longer read (dQ reads dS^T and K): release it now.
      if (leader) tc_commit(bar(C::B_QE + s));
      // dQ partial = dS K (M = queries, N = head dim, K = keys): the previous
      // partial must have been drained, and (aliased columns) dP^T fully read.
      if (it > 0 && !mbar_wait_warp(bar(C::B_ITF), (it - 1) & 1, w)) { ok = false; break; }
      if constexpr (!C::PREFETCH) {
        if (!mbar_wait_warp(bar(C::B_SDPF), it & 1, w)) { ok = false; break; }
      }
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < C::NPROD; ++t)
#pragma unroll
        for (int k = 0; k < 128 / 16; ++k) {
          const uint64_t ad = make_sdesc(dsb + C::pa(t) * C::PT_HALF + k * 16 * 128, C::PANEL, 1024);
          const uint64_t bd = make_sdesc(kb + C::pb(t) * C::TILE + k * 16 * 128, C::PANEL, 1024);
          if (leader) mma_ss<false>(tmem + C::TM_DQ, ad, bd, C::IDESC_Q, (t > 0 || k > 0) ? 1u : 0u);
        }
      if (leader) tc_commit(bar(C::B_DQF));
      if constexpr (!C::PREFETCH) {
        if (more) {
          // With aliased dQ columns, dP^T(it+1) may only be written once dQ(it)
          // has been drained.
          if (!mbar_wait_warp(bar(C::B_QF + (it + 1) % C::NQS), ((it + 1) / C::NQS) & 1, w)) { ok = false; break; }
          if (C::DQ_ALIAS && !mbar_wait_warp(bar(C::B_ITF), it & 1, w)) { ok = false; break; }
          tc_fence_after();
          issue_s(it + 1);
          issue_dp(it + 1);
        }
      }
    }
    if (leader) {
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
  } else {
    // ---------------- compute warpgroups ----------------
    // Warpgroup g owns query columns 64g .. 64g+63 of every S^T / dP^T tile
    // and drains head columns [g W, g W + W) of dQ, dK and dV.
    const int g = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // key row for P^T/dS^T, query row for dQ
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    constexpr int W = DHB / 2;  // 32 or 64 head columns drained per warpgroup
    bool ok = true;
    const int t = threadIdx.x - 64 - 128 * g;  // 0..127 within the warpgroup
    // dQ(it2) partial -> fp32 accumulator, rows of query tile i2 of head h2.
    auto drain_dq = [&](int it2) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_DQF), it2 & 1, w))) return false;
      tc_fence_after();
      const int h2 = kvh * a.group + it2 / n_i;
      const int i2 = j + it2 % n_i;
      uint32_t r[W];
      if constexpr (W == 64) tmem_ld64(tl + C::TM_DQ + g * W, r);
      else tmem_ld32(tl + C::TM_DQ + g * W, r);
      tc_fence_before();
      mbar_arrive(bar(C::B_ITF));
      if constexpr (C::TMA_DQ) {
        // Stage the fp32 [128 x 32] half in 128-byte-swizzled rows of this
        // warpgroup's staging panel, then one thread adds the whole box to
        // global memory. The panel is rewritten only after the previous
        // reduction (one iteration earlier) has finished reading it.
        const uint32_t panel = sbase + C::OFF_DQS + g * C::PANEL;
        if (t == 0) bulk_wait_read0();
        named_bar(2 + g, 128);
#pragma unroll
        for (int c = 0; c < 8; ++c)
          st_shared_v4(panel + rl * 128 + ((c ^ (rl & 7)) << 4), r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
        fence_async_smem();
        named_bar(2 + g, 128);
        if (t == 0 && g * W < a.Dh) {  // a half past the head width has nothing to add
          tma_reduce_add_4d(&maps.dq, panel, g * W, h2, i2 * 128, b);
          bulk_commit();
        }
      } else {
        const int qrow = i2 * 128 + rl;
        float* dst = a.dq_acc + ((static_cast<size_t>(b) * a.T + qrow) * a.Hq + h2) * a.Dh + g * W;
        const int ncol = a.Dh - g * W;
        if (qrow < a.T && ncol > 0) {
#pragma unroll
          for (int u = 0; u < W / 4; ++u)
            if (4 * u < ncol)
              red_add_v4(dst + 4 * u, __uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                         __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3]));
        }
      }
      return true;
    };
    for (int it = 0; it < n_it; ++it) {
      const int s = it % C::NQS;
      const int i = j + it % n_i;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SR), it & 1, w) &&
                                       mbar_wait(bar(C::B_QF + s), (it / C::NQS) & 1, w));
      if (!ok) break;
      const float* lse2s = reinterpret_cast<const float*>(smem + (stage(s) - sbase) + 2 * C::OPND) + 64 * g;
      const float* dvs = lse2s + 128;
      float p[64];
      uint32_t dpr[64];  // prefetch schedule: dP^T half, loaded together with S^T
      if constexpr (C::PREFETCH) {
        // S^T(it) and dP^T(it) are issued together: one TMEM round trip for both.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DPR), it & 1, w));
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
      // P^T = 2^(S^T * scale * log2 e - LSE2); key rl is after query 64g + c on
      // the diagonal tile: dropped.
      const bool diag = (i == j);
      const int lim = rl - 64 * g;
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lse2s + c);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float e = ex2(fmaf(p[c + u], sl2, -lv[u]));
          p[c + u] = (diag && c + u < lim) ? 0.f : e;
        }
      }
      store_half_row_bf16<HL>(sbase + C::OFF_P + g * C::PANEL, rl, p, C::PT_HALF);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PR + g));
      // dS^T = P^T * (dP^T - D)
      if constexpr (!C::PREFETCH) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DPR), it & 1, w));
        if (!ok) break;
        tc_fence_after();
        tmem_ld64(tl + C::TM_DP + 64 * g, dpr);
        tc_fence_before();
        mbar_arrive(bar(C::B_SDPF));
      }
#pragma unroll
      for (int q = 0; q < 64; q += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(dvs + q);
        p[q + 0] *= __uint_as_float(dpr[q + 0]) - d4.x;
        p[q + 1] *= __uint_as_float(dpr[q + 1]) - d4.y;
        p[q + 2] *= __uint_as_float(dpr[q + 2]) - d4.z;
        p[q + 3] *= __uint_as_float(dpr[q + 3]) - d4.w;
      }
      if constexpr (C::PREFETCH) {
        // The dS^T buffer is free once dK(it-1) and dQ(it-1) are done.
        if (it > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DQF), (it - 1) & 1, w));
          if (!ok) break;
        }
      }
      if constexpr (C::SHARE) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DVD + g), it & 1, w));
        if (!ok) break;
      }
      store_half_row_bf16<HL>(sbase + C::OFF_DS + g * C::PANEL, rl, p, C::PT_HALF);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSR + g));
      // dQ of the previous iteration (prefetch schedule), or of this one (dP^T
      // of the next iteration may reuse dQ's columns), goes to the accumulator.
      if constexpr (C::PREFETCH) {
        if (it > 0) {
          ok = drain_dq(it - 1);
          if (!ok) break;
        }
      } else {
        ok = drain_dq(it);
        if (!ok) break;
      }
    }
    if (C::PREFETCH && ok) ok = drain_dq(n_it - 1);
    if constexpr (C::TMA_DQ) {
      if (t == 0) bulk_wait0();  // every bulk reduction of this CTA has landed
    }
    if (ok) {
      // The last dQ commit covered every MMA, including the final dK/dV updates.
      const int key = j * 128 + rl;
      const bool valid = key < a.T;
      const size_t row_off = ((static_cast<size_t>(b) * a.T + key) * a.Hkv + kvh) * a.Dh + g * W;
      const int ncol = a.Dh - g * W;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t col0 = (which == 0 ? C::TM_DV : C::TM_DK) + g * W;
        const float mul = which == 0 ? 1.f : a.scale;
        void* base = which == 0 ? a.dv : a.dk;
        uint32_t r[W];
        if constexpr (W == 64) tmem_ld64(tl + col0, r);
        else tmem_ld32(tl + col0, r);
        if (!valid || ncol <= 0) continue;
        if constexpr (HL) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + row_off);
#pragma unroll
          for (int u = 0; u < W / 4; ++u)
            if (4 * u < ncol)
              dst[u] = make_float4(__uint_as_float(r[4 * u]) * mul, __uint_as_float(r[4 * u + 1]) * mul,
                                   __uint_as_float(r[4 * u + 2]) * mul, __uint_as_float(r[4 * u + 3]) * mul);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + row_off);
#pragma unroll
          for (int u = 0; u < W / 8; ++u)
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

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace rca
