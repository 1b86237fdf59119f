// Tensor-core products of the materialized causal attention path (sm_103a).
//
// The materialized path of the riftco-transformer page "Execution Backends and
// the Python ABI" (section "What the Metal slice does") forms the [T, T] score
// matrix, normalises it with a causal softmax, keeps the probabilities P for
// the VJP, and multiplies. The five products it needs are computed here, over
// the kept (causal) triangle only:
//
//   mat_scores_kernel     C[i, j] = A[i] . B[j]   for 128 x 128 tiles j <= i
//                         (S = Q K^T in the forward, dP = dO V^T in the
//                         backward); the epilogue writes C (fp32 into the
//                         [E, T, T] rows), or per-row statistics of C, or
//                         the probabilities 2^(c C - LSE2) (see MODE)
//   mat_reduce_kernel<0>  R[i] = sum_{j <= i} X[i, j] Y[j]
//                         (O = P V, dQ = dS K): one item per 128 query rows
//   mat_reduce_kernel<1>  R[j] = sum_h sum_{i >= j} X_h[i, j] Y_h[i]
//                         (dK = dS^T Q, dV = P^T dO, summed over the g query
//                         heads of a KV head): one item per 128 key rows
//
// E = B * Hq row blocks; X is one of the fp32 [E, T, T] matrices (P or dS,
// exactly zero above the diagonal); A, B, Y are [B, T, H, Dh] tensors read by
// TMA in 128-byte swizzled panels of 64 bf16 elements (head widths below 64
// are zero-padded by the copy).
//
// Precision. The MMAs take bf16 operands with fp32 accumulation. fp32 data is
// split into bf16 parts x = x0 + x1 (+ x2) with x0 = bf16(x), x1 = bf16(x - x0),
// x2 = bf16(x - x0 - x1); the products of parts whose indices sum to less than
// the part count are summed (3 parts: 6 products, relative error ~2^-24 like
// fp32 itself; 2 parts: 3 products, ~2^-17). X (P or dS) is split into two
// parts by the converting warps as it is loaded; bf16 operands are exact.
//
// Scheduling: persistent CTAs (one per SM) take items c, c + G, ... (the
// reduce kernel's items differ in length and are dealt in alternating
// directions, see reduce_deal); roles are a TMA warp, a single-thread MMA
// issuer, a TMEM owner, epilogue warps (TMEM lanes 32 q .. 32 q + 31: four in
// the reduce kernel; in the scores kernel four per lane quarter with bf16
// operands, one 32-column block of the tile each, or two with fp32 operands,
// one 64-column half each) and, in the reduce kernel, sixteen
// converting warps that load X straight from global memory (the next chunk's
// loads in flight while the current one is stored) and store its bf16 parts
// in the swizzled layout the MMA reads. Two TMEM accumulators alternate between items so one item's
// epilogue overlaps the next item's products. Every wait is time-bounded.
#pragma once

#include "tc.cuh"

namespace rca {
namespace mat {

constexpr int kPanel64 = 128 * 128;  // 128 rows x 128 bytes

// Products (part of A, part of B) summed for NA x NB parts: indices a + b < max(NA, NB).
template <int NA, int NB>
struct Products {
  static constexpr int NMAX = NA > NB ? NA : NB;
  static constexpr int count() {
    int n = 0;
    for (int a = 0; a < NA; ++a)
      for (int b = 0; b < NB; ++b)
        if (a + b < NMAX) ++n;
    return n;
  }
};

// ---------------------------------------------------------------------------
// Scores: 128 x 128 fp32 tiles of A B^T over the causal triangle of tiles.
// ---------------------------------------------------------------------------
template <int NP, int DHP>
struct ScoresCfg {
  // Epilogue warps: four per TMEM lane quarter (one 32-column block of the
  // tile each) with bf16 operands, two (one 64-column half each) with the
  // three-part fp32 operands, whose stages leave less room for staging.
  static constexpr int NEPI = NP == 1 ? 16 : 8;
  static constexpr int NGRP = NEPI / 4;                // column groups of a tile
  static constexpr int GCOLS = 128 / NGRP;             // columns per epilogue warp
  static constexpr int NTHREADS = 128 + 32 * NEPI;     // warps 0-3 roles, then the epilogue
  static constexpr int DP = DHP / 64;                  // 64-column panels across the head width
  static constexpr int PART = DP * kPanel64;           // one bf16 part of a 128-row tile
  static constexpr int STAGE = 2 * NP * PART;          // A parts then B parts
  static constexpr int STAGING = NEPI * 32 * 128;      // per epilogue warp: 32 rows x 128 bytes
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int BAR_BYTES = 256;
  static constexpr int NS_FIT = (SMEM_LIMIT - 1024 - BAR_BYTES - STAGING) / STAGE;
  static constexpr int NS = NS_FIT > 3 ? 3 : NS_FIT;
  static_assert(NS >= 1, "scores stage does not fit");
  static constexpr int OFF_STG = NS * STAGE;
  static constexpr int OFF_BAR = OFF_STG + STAGING;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  static constexpr int B_FULL = 0, B_EMPTY = NS, B_ACCF = 2 * NS, B_ACCE = 2 * NS + 2, B_FIN = 2 * NS + 4;
  static constexpr int NBAR = B_FIN + 1;
  static_assert(8 * NBAR + 8 <= BAR_BYTES, "barrier area");
  static constexpr uint32_t IDESC = make_idesc(false, 128, 128, false, false);
};

struct ScoresArgs {
  float* out;         // [E, T, T]
  float2* part;       // row statistics mode: (max, sum) of row r, tile j, column group g at [e, r, j, g]
  const float* lse2;  // probabilities mode: base-2 LSE of each row, [E, T]
  float c;            // both modes: scale * log2(e)
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, group, n_t;
  long long n_tri;    // tiles per row block: n_t (n_t + 1) / 2
  long long n_items;  // E * n_tri
};

struct ScoresMaps {
  CUtensorMap a[3];  // parts of the row operand (Q or dO), query heads
  CUtensorMap b[3];  // parts of the column operand (K or V), KV heads
};

// Item idx -> (row block e, query tile i, key tile j <= i).
__device__ __forceinline__ void scores_item(const ScoresArgs& a, long long idx, int& e, int& i, int& j) {
  e = static_cast<int>(idx / a.n_tri);
  const long long r = idx - static_cast<long long>(e) * a.n_tri;
  int ii = static_cast<int>((sqrtf(8.0f * static_cast<float>(r) + 1.0f) - 1.0f) * 0.5f);
  while (static_cast<long long>(ii + 1) * (ii + 2) / 2 <= r) ++ii;
  while (static_cast<long long>(ii) * (ii + 1) / 2 > r) --ii;
  i = ii;
  j = static_cast<int>(r - static_cast<long long>(ii) * (ii + 1) / 2);
}

// MODE (what the epilogue does with a tile's scores S = A B^T):
//   kScoresRaw    write S (fp32) into the kept tiles; blocks of the diagonal
//                 tile that lie wholly above a warp's rows are not written;
//   kScoresStats  write, per row and tile, x = c S's (max m, sum of 2^(x - m))
//                 over the row's kept columns, nothing else;
//   kScoresProbs  write P = 2^(c S - LSE2) on and below the diagonal, 0 above it
//                 inside the diagonal tile (the whole tile is written).
enum { kScoresRaw = 0, kScoresStats = 1, kScoresProbs = 2 };

template <int NP, int DHP, bool VEC, int MODE>
__global__ void __launch_bounds__(ScoresCfg<NP, DHP>::NTHREADS, 1)
    mat_scores_kernel(const __grid_constant__ ScoresMaps maps, const ScoresArgs a) {
  using C = ScoresCfg<NP, DHP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int k) -> uint32_t { return sbase + C::OFF_BAR + 8u * k; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long G = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar(C::B_FULL + s), 1);
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(C::B_ACCF + k), 1);
      mbar_init(bar(C::B_ACCE + k), C::NEPI);  // the epilogue warps
    }
    mbar_init(bar(C::B_FIN), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{a.status, abort_flag, a.timeout_ns};
  const long long n_mine = a.n_items > blockIdx.x ? (a.n_items - 1 - blockIdx.x) / G + 1 : 0;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (elect_one()) {
      for (int p = 0; p < NP; ++p) {
        tma_prefetch_desc(&maps.a[p]);
        tma_prefetch_desc(&maps.b[p]);
      }
      long long n = 0;
      for (; n < n_mine; ++n) {
        int e, i, j;
        scores_item(a, blockIdx.x + n * G, e, i, j);
        const int b = e / a.Hq, h = e - b * a.Hq, kvh = h / a.group;
        const int s = static_cast<int>(n % C::NS);
        if (n >= C::NS && !mbar_wait(bar(C::B_EMPTY + s), static_cast<uint32_t>((n / C::NS - 1) & 1), w)) break;
        mbar_expect_tx(bar(C::B_FULL + s), C::STAGE);
        const uint32_t st = sbase + s * C::STAGE;
        for (int p = 0; p < NP; ++p)
          for (int d = 0; d < C::DP; ++d) {
            tma_load_4d(st + (p * C::DP + d) * kPanel64, &maps.a[p], bar(C::B_FULL + s), d * 64, h, i * 128, b);
            tma_load_4d(st + ((NP + p) * C::DP + d) * kPanel64, &maps.b[p], bar(C::B_FULL + s), d * 64, kvh,
                        j * 128, b);
          }
      }
      // Exit: the loads issued have landed before shared memory is released.
      for (int s = 0; s < C::NS && s < n; ++s) {
        const long long last = s + ((n - 1 - s) / C::NS) * C::NS;
        mbar_drain(bar(C::B_FULL + s), static_cast<uint32_t>((last / C::NS) & 1), a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one()) {
      for (long long n = 0; n < n_mine; ++n) {
        const int s = static_cast<int>(n % C::NS);
        const int acc = static_cast<int>(n & 1);
        if (!mbar_wait(bar(C::B_FULL + s), static_cast<uint32_t>((n / C::NS) & 1), w)) break;
        if (n >= 2 && !mbar_wait(bar(C::B_ACCE + acc), static_cast<uint32_t>(((n >> 1) - 1) & 1), w)) break;
        tc_fence_after();
        const uint32_t st = sbase + s * C::STAGE;
        const uint32_t d = tmem + acc * 128;
        uint32_t first = 1;
#pragma unroll
        for (int pa = 0; pa < NP; ++pa)
#pragma unroll
          for (int pb = 0; pb < NP; ++pb) {
            if (pa + pb >= NP) continue;
#pragma unroll
            for (int k = 0; k < DHP / 16; ++k) {
              const uint32_t off = (k >> 2) * kPanel64 + (k & 3) * 32;
              mma_ss<false>(d, make_sdesc(st + pa * C::PART + off, 16, 1024),
                            make_sdesc(st + (NP + pb) * C::PART + off, 16, 1024), C::IDESC, first ? 0u : 1u);
              first = 0;
            }
          }
        tc_commit(bar(C::B_EMPTY + s));
        tc_commit(bar(C::B_ACCF + acc));
      }
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------- epilogue: TMEM -> staging -> coalesced row stores ----------------
    // Warps 4 + 4 g + q read TMEM lanes 32 q .. 32 q + 31 (tile rows) and the
    // tile's column group g (GCOLS columns): several warps per sub-partition,
    // so one's latency hides behind the others' work.
    const int q = warp & 3;
    const int grp = (warp - 4) >> 2;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t stg = sbase + C::OFF_STG + (warp - 4) * (32 * 128);
    const int rsub = lane >> 3, cq = lane & 7;  // staging read: row within a group of 4, 16-byte chunk
    for (long long n = 0; n < n_mine; ++n) {
      int e, i, j;
      scores_item(a, blockIdx.x + n * G, e, i, j);
      const int acc = static_cast<int>(n & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_ACCF + acc), static_cast<uint32_t>((n >> 1) & 1), w))) break;
      tc_fence_after();
      float* orow = a.out + static_cast<size_t>(e) * a.T * a.T;
      const int my_row = i * 128 + 32 * q + lane;  // this thread's TMEM lane
      if constexpr (MODE == kScoresStats) {
        // The group's columns in one load, this warp's share of the
        // accumulator released at once; then their maximum (of S: c > 0) and
        // the sum of 2^(c S - m) over the kept columns k <= lim, in four
        // chains each. A group wholly above the diagonal gives (-inf, 0).
        uint32_t rr[C::GCOLS];
        if constexpr (C::GCOLS == 64)
          tmem_ld64(tl + acc * 128 + C::GCOLS * grp, rr);
        else
          tmem_ld32(tl + acc * 128 + C::GCOLS * grp, rr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_ACCE + acc));
        const int lim = i == j ? my_row - (j * 128 + C::GCOLS * grp) : C::GCOLS - 1;
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < C::GCOLS; ++k)
          if (k <= lim) mx[k & 3] = fmaxf(mx[k & 3], __uint_as_float(rr[k]));
        const float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * a.c;
        float sm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < C::GCOLS; ++k)
          if (k <= lim) sm[k & 3] += ex2(fmaf(__uint_as_float(rr[k]), a.c, -m));
        if (my_row < a.T)
          a.part[((static_cast<size_t>(e) * a.T + my_row) * a.n_t + j) * C::NGRP + grp] =
              make_float2(m, (sm[0] + sm[1]) + (sm[2] + sm[3]));
        continue;
      }
      float lse2_row = 0.f;  // kScoresProbs
      if constexpr (MODE == kScoresProbs)
        if (my_row < a.T) lse2_row = a.lse2[static_cast<size_t>(e) * a.T + my_row];
      constexpr int CPW = C::GCOLS / 32;  // 32-column blocks per epilogue warp
      for (int c = CPW * grp; c < CPW * grp + CPW; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + acc * 128 + 32 * c, r);
        if (c == CPW * grp + CPW - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_ACCE + acc));
        }
        // On a diagonal tile a block whose columns all lie above this warp's
        // rows is skipped (its probabilities, all 0, are still written).
        if (MODE == kScoresRaw && i == j && c > q) continue;
        if constexpr (MODE == kScoresProbs) {
          // Column j 128 + 32 c + k is kept for this row unless it lies above
          // the diagonal, which only happens in the diagonal tile.
          const int lim = i == j ? my_row - (j * 128 + 32 * c) : 31;  // kept: k <= lim
#pragma unroll
          for (int k = 0; k < 32; ++k)
            r[k] = __float_as_uint(k <= lim ? ex2(fmaf(__uint_as_float(r[k]), a.c, -lse2_row)) : 0.f);
        }
        // This thread's row (32 fp32 = 8 chunks of 16 bytes), chunk index swizzled by row.
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(stg + lane * 128 + ((u ^ (lane & 7)) << 4), r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
        __syncwarp();
        const int col = j * 128 + 32 * c + 4 * cq;
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          const int rr = 4 * g4 + rsub;  // row within this warp's 32
          const int row = i * 128 + 32 * q + rr;
          float4 v;
          asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                       : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                       : "r"(stg + rr * 128 + ((cq ^ (rr & 7)) << 4)));
          if (row < a.T) {
            float* dst = orow + static_cast<size_t>(row) * a.T + col;
            if constexpr (VEC) {
              if (col < a.T) *reinterpret_cast<float4*>(dst) = v;  // T % 4 == 0: all four or none
            } else {
              if (col < a.T) dst[0] = v.x;
              if (col + 1 < a.T) dst[1] = v.y;
              if (col + 2 < a.T) dst[2] = v.z;
              if (col + 3 < a.T) dst[3] = v.w;
            }
          }
        }
        __syncwarp();
      }
    }
  }
  // TMEM is released once every role is done with it.
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------------------
// Reductions over the causal triangle: R = X Y (rows) or R = X^T Y (columns).
// ---------------------------------------------------------------------------
template <bool TRANS, int NPY, int DHP>
struct ReduceCfg {
  static constexpr int NCONV = 16;                      // converting warps 8 .. 8 + NCONV - 1
  static constexpr int CONV_THREADS = 32 * NCONV;
  static constexpr int SEG = 2048 / CONV_THREADS;      // 16-byte segments of a chunk per converting thread
  static constexpr int NTHREADS = 256 + CONV_THREADS;
  static constexpr int DP = DHP / 64;
  static constexpr int XPART = 128 * 64 * 2;            // 128 (M) x 64 (K) bf16 = 16 KB
  static constexpr int YPANEL = 64 * 128;               // 64 rows (K) x 128 bytes
  static constexpr int YPART = DP * YPANEL;
  static constexpr int STAGE = 2 * XPART + NPY * YPART;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int BAR_BYTES = 256;
  static constexpr int NS_FIT = (SMEM_LIMIT - 1024 - BAR_BYTES) / STAGE;
  static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
  static_assert(NS >= 2, "reduce stages do not fit");
  static constexpr int OFF_BAR = NS * STAGE;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;
  static constexpr int B_FULL = 0, B_EMPTY = NS, B_ACCF = 2 * NS, B_ACCE = 2 * NS + 2, B_FIN = 2 * NS + 4;
  static constexpr int NBAR = B_FIN + 1;
  static_assert(8 * NBAR + 8 <= BAR_BYTES, "barrier area");
  // X parts: K-major (rows) or MN-major (columns); Y: MN-major (head width contiguous).
  static constexpr uint32_t IDESC = make_idesc(false, 128, DHP, TRANS, true);
  static constexpr int TMEM_COLS = 2 * DHP > 32 ? 2 * DHP : 32;
};

struct ReduceArgs {
  const float* x;     // [E, T, T] fp32, zero above the diagonal
  void* out;          // rows: [B, T, Hq, Dh]; columns: [B, T, Hkv, Dh] (storage dtype)
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, Dh, group, n_t;
  int n_items;        // rows: B * Hq * n_t; columns: B * Hkv * n_t
  int out_f32;        // output element type: fp32 (1) or bf16 (0)
};

struct ReduceMaps {
  CUtensorMap y[2];   // parts of Y (64-row boxes): rows: V or K (KV heads); columns: Q or dO (query heads)
};

// Item idx -> (b, head, tile): rows: (b, h, i), the longest (largest i) first;
// columns: (b, kvh, j), the longest (smallest j) first.
template <bool TRANS>
__device__ __forceinline__ void reduce_item(const ReduceArgs& a, int idx, int& b, int& hd, int& t) {
  const int per = TRANS ? a.B * a.Hkv : a.B * a.Hq;
  const int level = idx / per, bh = idx - level * per;
  const int H = TRANS ? a.Hkv : a.Hq;
  b = bh / H;
  hd = bh - b * H;
  t = TRANS ? level : a.n_t - 1 - level;
}

// 64-position chunks of one item's contraction: rows: keys 0 .. min(128 (i+1), T);
// columns: for each of the group's query heads, queries 128 j .. T.
template <bool TRANS>
__device__ __forceinline__ int reduce_chunks_per_head(const ReduceArgs& a, int t) {
  if constexpr (TRANS) return (a.T - 128 * t + 63) / 64;
  const int kend = 128 * (t + 1) < a.T ? 128 * (t + 1) : a.T;
  return (kend + 63) / 64;
}

// The n-th item of CTA c among G: items are dealt in rounds of G, even rounds
// in CTA order and odd rounds in reverse, so that a CTA given one of the
// longest items of a round gets one of the shortest of the next (the items
// are ordered longest first). reduce_count is how many items CTA c gets.
__device__ __forceinline__ int reduce_deal(int c, int n, int G) { return n * G + ((n & 1) ? G - 1 - c : c); }
__device__ __forceinline__ int reduce_count(int c, int n_items, int G) {
  const int full = n_items / G, rem = n_items - full * G;
  const int pos = (full & 1) ? G - 1 - c : c;
  return full + (pos < rem ? 1 : 0);
}

template <bool TRANS, int NPY, int DHP>
__global__ void __launch_bounds__(ReduceCfg<TRANS, NPY, DHP>::NTHREADS, 1)
    mat_reduce_kernel(const __grid_constant__ ReduceMaps maps, const ReduceArgs a) {
  using C = ReduceCfg<TRANS, NPY, DHP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int k) -> uint32_t { return sbase + C::OFF_BAR + 8u * k; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar(C::B_FULL + s), C::NCONV + 1);  // the converting warps + the TMA thread
      mbar_init(bar(C::B_EMPTY + s), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(C::B_ACCF + k), 1);
      mbar_init(bar(C::B_ACCE + k), 4);
    }
    mbar_init(bar(C::B_FIN), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{a.status, abort_flag, a.timeout_ns};
  const int n_mine = reduce_count(static_cast<int>(blockIdx.x), a.n_items, G);

  if (warp == 0) {
    // ---------------- TMA producer: Y chunks ----------------
    if (elect_one()) {
      tma_prefetch_desc(&maps.y[0]);
      if (NPY > 1) tma_prefetch_desc(&maps.y[1]);
      long long u = 0;  // chunk counter across items
      bool ok = true;
      for (int n = 0; ok && n < n_mine; ++n) {
        int b, hd, t;
        reduce_item<TRANS>(a, reduce_deal(blockIdx.x, n, G), b, hd, t);
        const int nch = reduce_chunks_per_head<TRANS>(a, t);
        const int nh = TRANS ? a.group : 1;
        for (int r = 0; ok && r < nh; ++r)
          for (int c = 0; c < nch; ++c, ++u) {
            const int s = static_cast<int>(u % C::NS);
            if (u >= C::NS && !mbar_wait(bar(C::B_EMPTY + s), static_cast<uint32_t>((u / C::NS - 1) & 1), w)) {
              ok = false;
              break;
            }
            mbar_expect_tx(bar(C::B_FULL + s), NPY * C::YPART);
            const uint32_t yb = sbase + s * C::STAGE + 2 * C::XPART;
            const int head = TRANS ? hd * a.group + r : hd / a.group;
            const int pos = TRANS ? 128 * t + 64 * c : 64 * c;
            for (int p = 0; p < NPY; ++p)
              for (int d = 0; d < C::DP; ++d)
                tma_load_4d(yb + (p * C::DP + d) * C::YPANEL, &maps.y[p], bar(C::B_FULL + s), d * 64, head, pos, b);
          }
      }
      for (int s = 0; s < C::NS && s < u; ++s) {
        const long long last = s + ((u - 1 - s) / C::NS) * C::NS;
        mbar_drain(bar(C::B_FULL + s), static_cast<uint32_t>((last / C::NS) & 1), a.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (elect_one()) {
      long long u = 0;
      bool ok = true;
      for (int n = 0; ok && n < n_mine; ++n) {
        int b, hd, t;
        reduce_item<TRANS>(a, reduce_deal(blockIdx.x, n, G), b, hd, t);
        const int nch = reduce_chunks_per_head<TRANS>(a, t) * (TRANS ? a.group : 1);
        const int acc = n & 1;
        const uint32_t d = tmem + acc * DHP;
        if (n >= 2 && !mbar_wait(bar(C::B_ACCE + acc), static_cast<uint32_t>(((n >> 1) - 1) & 1), w)) break;
        for (int c = 0; c < nch; ++c, ++u) {
          const int s = static_cast<int>(u % C::NS);
          if (!mbar_wait(bar(C::B_FULL + s), static_cast<uint32_t>((u / C::NS) & 1), w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xb = sbase + s * C::STAGE;
          const uint32_t yb = xb + 2 * C::XPART;
#pragma unroll
          for (int px = 0; px < 2; ++px)
#pragma unroll
            for (int py = 0; py < NPY; ++py) {
              if (px + py >= 2) continue;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                // X: rows = K-major (k step = 32 bytes within a row); columns =
                // MN-major (k step = 16 rows of 128 bytes, M panels 8 KB apart).
                const uint64_t ad = TRANS ? make_sdesc(xb + px * C::XPART + k * 16 * 128, 8192, 1024)
                                          : make_sdesc(xb + px * C::XPART + k * 32, 16, 1024);
                const uint64_t bd = make_sdesc(yb + py * C::YPART + k * 16 * 128, C::YPANEL, 1024);
                mma_ss<false>(d, ad, bd, C::IDESC, (c == 0 && px == 0 && py == 0 && k == 0) ? 0u : 1u);
              }
            }
          tc_commit(bar(C::B_EMPTY + s));
        }
        if (!ok) break;
        tc_commit(bar(C::B_ACCF + acc));
      }
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
    __syncwarp();
  } else if (warp >= 8) {
    // ---------------- converting warps: X (fp32, global) -> bf16 parts (shared) ----------------
    // Per 64-position chunk, 2048 16-byte segments: rows: 128 rows x 16 segments
    // of K; columns: 64 rows (K) x 32 segments of M. Thread ct takes segments
    // ct + CONV_THREADS v, v < SEG; the next chunk's loads are issued before
    // this chunk's stores.
    const int ct = threadIdx.x - 256;
    long long u = 0;
    bool ok = true;
    float4 cur[C::SEG], nxt[C::SEG];
    // Loads of chunk (item n, head r, chunk c) into regs.
    auto load = [&](float4 (&rg)[C::SEG], int b, int hd, int t, int r, int c) {
      const int e = TRANS ? b * a.Hq + hd * a.group + r : b * a.Hq + hd;
      const float* xe = a.x + static_cast<size_t>(e) * a.T * a.T;
#pragma unroll
      for (int v = 0; v < C::SEG; ++v) {
        const int sg = ct + C::CONV_THREADS * v;
        int row, col;
        if constexpr (TRANS) {
          row = 128 * t + 64 * c + (sg >> 5);  // query position i
          col = 128 * t + 4 * (sg & 31);       // key position j
        } else {
          row = 128 * t + (sg >> 4);
          col = 64 * c + 4 * (sg & 15);
        }
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (row < a.T && col < a.T) {
          const float* src = xe + static_cast<size_t>(row) * a.T + col;
          if ((a.T & 3) == 0) {
            asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                         : "l"(src));
          } else {
            x.x = src[0];
            if (col + 1 < a.T) x.y = src[1];
            if (col + 2 < a.T) x.z = src[2];
            if (col + 3 < a.T) x.w = src[3];
          }
        }
        rg[v] = x;
      }
    };
    // Walk of the chunk sequence (items, heads, chunks) shared by the two cursors.
    struct Cur {
      int n, r, c, b, hd, t, nch, nh;
      bool valid;
    };
    auto start = [&](Cur& q, int n) {
      q.n = n;
      q.r = 0;
      q.c = 0;
      q.valid = n < n_mine;
      if (q.valid) {
        reduce_item<TRANS>(a, reduce_deal(blockIdx.x, n, G), q.b, q.hd, q.t);
        q.nch = reduce_chunks_per_head<TRANS>(a, q.t);
        q.nh = TRANS ? a.group : 1;
      }
    };
    auto advance = [&](Cur& q) {
      if (++q.c == q.nch) {
        q.c = 0;
        if (++q.r == q.nh) start(q, q.n + 1);
      }
    };
    Cur cc, nc;
    start(cc, 0);
    if (cc.valid) load(cur, cc.b, cc.hd, cc.t, cc.r, cc.c);
    nc = cc;
    if (nc.valid) advance(nc);
    while (ok && cc.valid) {
      if (nc.valid) load(nxt, nc.b, nc.hd, nc.t, nc.r, nc.c);
      const int s = static_cast<int>(u % C::NS);
      if (u >= C::NS) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_EMPTY + s), static_cast<uint32_t>((u / C::NS - 1) & 1), w));
        if (!ok) break;
      }
      const uint32_t xb = sbase + s * C::STAGE;
#pragma unroll
      for (int v = 0; v < C::SEG; ++v) {
        const int sg = ct + C::CONV_THREADS * v;
        uint32_t off;
        if constexpr (TRANS) {
          // MN-major: row = K (query within chunk), 64 M elements per 128-byte row, M panels 8 KB apart.
          const int kr = sg >> 5, m = 4 * (sg & 31);
          off = (m >> 6) * 8192 + kr * 128 + ((((m & 63) >> 3) ^ (kr & 7)) << 4) + ((m & 7) << 1);
        } else {
          // K-major: row = M (query row), 64 K elements per 128-byte row.
          const int mr = sg >> 4, kk = 4 * (sg & 15);
          off = mr * 128 + (((kk >> 3) ^ (mr & 7)) << 4) + ((kk & 7) << 1);
        }
        uint32_t h01, l01, h23, l23;
        split_bf16x2(cur[v].x, cur[v].y, h01, l01);
        split_bf16x2(cur[v].z, cur[v].w, h23, l23);
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(xb + off), "r"(h01), "r"(h23) : "memory");
        asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(xb + C::XPART + off), "r"(l01), "r"(l23) : "memory");
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_FULL + s));
      ++u;
      cc = nc;
#pragma unroll
      for (int v = 0; v < C::SEG; ++v) cur[v] = nxt[v];
      if (nc.valid) advance(nc);
    }
  } else if (warp >= 4) {
    // ---------------- epilogue: TMEM -> output rows ----------------
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    for (int n = 0; n < n_mine; ++n) {
      int b, hd, t;
      reduce_item<TRANS>(a, reduce_deal(blockIdx.x, n, G), b, hd, t);
      const int acc = n & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_ACCF + acc), static_cast<uint32_t>((n >> 1) & 1), w))) break;
      tc_fence_after();
      const int pos = 128 * t + row;
      const int H = TRANS ? a.Hkv : a.Hq;
      const size_t obase = ((static_cast<size_t>(b) * a.T + pos) * H + hd) * a.Dh;
#pragma unroll
      for (int c = 0; c < DHP / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + acc * DHP + 32 * c, r);
        if (c == DHP / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_ACCE + acc));
        }
        const int nc = a.Dh - 32 * c;  // valid head columns in this block
        if (pos < a.T && nc > 0) {
          if (a.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + obase + 32 * c);
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4)
              if (4 * u4 < nc)
                dst[u4] = make_float4(__uint_as_float(r[4 * u4]), __uint_as_float(r[4 * u4 + 1]),
                                      __uint_as_float(r[4 * u4 + 2]), __uint_as_float(r[4 * u4 + 3]));
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + obase + 32 * c);
#pragma unroll
            for (int u8 = 0; u8 < 4; ++u8)
              if (8 * u8 < nc)
                dst[u8] = make_uint4(
                    pack_bf16(__uint_as_float(r[8 * u8]), __uint_as_float(r[8 * u8 + 1])),
                    pack_bf16(__uint_as_float(r[8 * u8 + 2]), __uint_as_float(r[8 * u8 + 3])),
                    pack_bf16(__uint_as_float(r[8 * u8 + 4]), __uint_as_float(r[8 * u8 + 5])),
                    pack_bf16(__uint_as_float(r[8 * u8 + 6]), __uint_as_float(r[8 * u8 + 7])));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace mat
}  // namespace rca
