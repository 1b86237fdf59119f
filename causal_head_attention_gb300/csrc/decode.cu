// Paged decode attention for sm_103a.
//
// One query token per request attends over every position the request has
// cached, each key and value fetched through the request's page table
// ("Execution Backends and the Python ABI", section "Incremental attention":
// query/output viewed as [H, d_h]; key and value pools laid out
// [physical_page, H, page_offset, d_h]; a request-local table of physical page
// IDs). Per request b, query head h, KV head kv = h / (Hq / Hkv):
//   s_t = scale * q . K[t],  O = sum_t softmax(s)_t V[t],  LSE = ln sum_t exp(s_t)
// over t = 0 .. L_b - 1. No K/V is gathered into a contiguous copy.
//
// The work is HBM-bound: every cached K/V byte is read once, and a KV head
// group holds only G query rows. What bounds it in practice is how many
// loads are in flight, which on this pattern (page blocks of a few KB at a
// stride of Hkv blocks) takes many resident warps:
//  * Work items are (request, chunk of kDecodeChunk positions, KV head group of
//    G query heads). Persistent CTAs take items i, i + grid, ... from the list
//    of non-empty items, which every CTA rebuilds from the lengths (a prefix
//    sum over the requests in shared memory), so no CTA is launched empty and
//    every CTA gets the same number of items to within one.
//  * A position's head_dim row is spread over LP = Dh * bytes / 16 lanes (one
//    16-byte vector each). A block of RUN = (32 / LP) * U consecutive positions
//    is one warp's load: when a page holds at least RUN positions the block
//    lies in one page, so the warp reads one page-table entry per block and the
//    rest are pointer offsets. Loads go straight to registers; the register
//    budget is capped (launch bounds) so that enough warps stay resident to
//    keep HBM busy while others compute.
//  * Scores: packed fp32x2 products, then a reduce-scatter over the LP lanes
//    (each lane ends up owning one of the G*U scores instead of all of them).
//    Softmax in base 2 (the query is pre-scaled by scale * log2 e) against a
//    running maximum that is raised only when a score passes it by more than
//    2^8 (so probabilities stay <= 256): each lane then takes one exponential
//    per block and the probabilities are broadcast for the fp32x2 P * V update.
//  * A request whose length fits one chunk writes O and LSE directly; longer
//    requests leave (max, sum, unnormalised O) per chunk and a combine kernel
//    merges them.
// Device-side inputs are checked as they are read: a page ID outside
// [0, num_pages) is never dereferenced (its positions read as zeros) and a
// length outside [1, max_pages * page_size] makes that request's outputs NaN;
// both record kStatusBadInput in the status word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "decode.h"
#include "tc.cuh"

namespace rca {
namespace dec {

constexpr int NW = 4;  // warps per CTA (decode and combine kernels)
constexpr int NT = NW * 32;
constexpr unsigned FULL = 0xffffffffu;
constexpr float kRaise = 8.f;  // raise the running max when a score passes it by more (base 2)
#ifndef DEC_U_SMALL_G
#define DEC_U_SMALL_G 4
#endif
#ifndef DEC_U_LARGE_G
#define DEC_U_LARGE_G 2
#endif
// Resident CTAs per SM the register budget is sized for (one query head per
// KV head or two; four or more).
#ifndef DEC_MINB_SMALL_G
#define DEC_MINB_SMALL_G 6
#endif
#ifndef DEC_MINB_LARGE_G
#define DEC_MINB_LARGE_G 4
#endif

struct Args {
  const char* q;
  const char* kp;
  const char* vp;
  const int32_t* table;
  const int32_t* lens;
  char* out;
  float* lse;
  float* part_ml;
  float* part_acc;
  int* status;
  int B, Hq, Hkv, g, ngc, page_shift, max_pages, num_pages, maxch;
  float qscale;  // scale * log2(e)
  unsigned long long timeout_ns;
};

template <bool BF16, int DH, int G>
struct Cfg {
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr int EPV = 16 / ESZ;   // elements per 16-byte vector
  static constexpr int NPAIR = EPV / 2;  // fp32x2 pairs per vector
  static constexpr int LP = DH / EPV;    // lanes per position
  static constexpr int PPW = 32 / LP;    // positions per warp and load step
  static constexpr int U = G >= 4 ? DEC_U_LARGE_G : DEC_U_SMALL_G;  // load steps per stage
  static constexpr int NV = G * U;                    // scores per lane group per stage
  static constexpr int NF = NV > LP ? NV / LP : 1;    // scores a lane owns after the reduce-scatter
  static constexpr int RUN = PPW * U;                 // positions per compute block of a warp
  static constexpr int MINB = G >= 8 ? 2 : G >= 4 ? DEC_MINB_LARGE_G : G >= 2 ? DEC_MINB_SMALL_G - 1 : DEC_MINB_SMALL_G;
  static constexpr int ROW = DH * ESZ;                // bytes of one position's row
  static_assert(LP >= 2 && LP <= 32 && (32 % LP) == 0, "head width");
  static_assert((NV & (NV - 1)) == 0, "scores per block must be a power of two");
  static_assert(kDecodeChunk % RUN == 0, "a chunk is a whole number of blocks");
  static constexpr int ROUNDS = 31 - __builtin_clz(LP);  // log2(LP)

  // Reduce-scatter bookkeeping: in round r (partner distance LP >> (r + 1))
  // a lane holding cur = NV >> r >= 2 scores keeps the upper half if its lane
  // bit is set, else the lower half. holder(v) is a lane (in the group) that
  // owns score v afterwards and slot(v) the index it keeps it under.
  __host__ __device__ static constexpr int rounds() {
    int r = 0;
    while ((LP >> (r + 1)) >= 1) ++r;
    return r;
  }
  __host__ __device__ static constexpr int holder(int v) {
    int li = 0, off = 0;
    for (int r = 0; r < rounds(); ++r) {
      const int cur = NV >> r;
      if (cur < 2) break;
      const int d = LP >> (r + 1);
      if (v - off >= cur / 2) {
        li |= d;
        off += cur / 2;
      }
    }
    return li;
  }
  __host__ __device__ static constexpr int slot(int v) {
    int off = 0;
    for (int r = 0; r < rounds(); ++r) {
      const int cur = NV >> r;
      if (cur < 2) break;
      if (v - off >= cur / 2) off += cur / 2;
    }
    return v - off;
  }
};

// 16-byte load of data read exactly once (not kept in L1).
__device__ __forceinline__ uint4 ld_once(const char* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16 bytes of storage -> fp32 pairs (exact: bf16 is the high half of an fp32).
template <bool BF16>
__device__ __forceinline__ void to_pairs(const uint4& r, uint64_t (&p)[BF16 ? 4 : 2]) {
  if constexpr (BF16) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      p[j] = f2pack(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xffff0000u));
  } else {
    p[0] = f2pack(__uint_as_float(r.x), __uint_as_float(r.y));
    p[1] = f2pack(__uint_as_float(r.z), __uint_as_float(r.w));
  }
}

template <bool BF16>
__device__ __forceinline__ void store_elem(char* base, int64_t idx, float v) {
  if constexpr (BF16)
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(base)[idx] = v;
}

__device__ __forceinline__ bool len_ok(int L, const Args& a) {
  return L >= 1 && L <= (a.max_pages << a.page_shift);
}

__device__ __forceinline__ int n_chunks(int L) { return (L + kDecodeChunk - 1) / kDecodeChunk; }

// Exclusive prefix sums of the per-request chunk counts into pre[0..B]
// (pre[B] = total). CTA 0 also writes NaN outputs for requests whose length is
// out of range and records the bad input.
template <bool BF16, int NTHR>
__device__ void build_prefix(const Args& a, int* pre, int* warp_tot, int dh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (a.B + NTHR - 1) / NTHR;
  const int i0 = min(a.B, tid * seg), i1 = min(a.B, i0 + seg);
  int sum = 0;
  for (int i = i0; i < i1; ++i) {
    const int L = __ldg(a.lens + i);
    int n = 0;
    if (len_ok(L, a)) {
      n = n_chunks(L);
    } else if (blockIdx.x == 0) {
      atomicExch(a.status, kStatusBadInput);
      for (int h = 0; h < a.Hq; ++h) {
        for (int d = 0; d < dh; ++d)
          store_elem<BF16>(a.out, (int64_t(i) * a.Hq + h) * dh + d, __int_as_float(0x7fc00000));
        a.lse[int64_t(i) * a.Hq + h] = __int_as_float(0x7fc00000);
      }
    }
    pre[i + 1] = n;
    sum += n;
  }
  // Block-wide exclusive scan of the per-thread sums.
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(FULL, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += warp_tot[w];
  int run = base + incl - sum;
  for (int i = i0; i < i1; ++i) {
    run += pre[i + 1];
    pre[i + 1] = run;
  }
  if (tid == 0) pre[0] = 0;
  __syncthreads();
}

// Largest b with pre[b] <= ci (pre is non-decreasing, pre[0] = 0 <= ci < pre[B]).
__device__ __forceinline__ int find_request(const int* pre, int B, int ci) {
  int lo = 0, hi = B;  // invariant: pre[lo] <= ci < pre[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= ci) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Item ci*upb + u_ -> (request b, chunk c, KV head kv, first query head h0) and
// its positions [s0, s1).
struct Item {
  int b, c, nch, kv, h0, s0, s1;
};
template <int G>
__device__ __forceinline__ Item item_of(const Args& a, const int* pre, int upb, int item) {
  Item it;
  const int ci = item / upb, u_ = item - ci * upb;
  it.b = find_request(pre, a.B, ci);
  it.c = ci - pre[it.b];
  it.nch = pre[it.b + 1] - pre[it.b];
  it.kv = u_ / a.ngc;
  it.h0 = it.kv * a.g + (u_ - it.kv * a.ngc) * G;
  const int L = __ldg(a.lens + it.b);
  it.s0 = it.c * kDecodeChunk;
  it.s1 = min(L, it.s0 + kDecodeChunk);
  return it;
}

// Warp w of a CTA takes blocks j = w, w + NW, ... of an item; block j covers
// positions [s0 + j*RUN, s0 + (j+1)*RUN) (masked at s1), PPW positions per
// load step, U steps. Loads go straight from the pools to registers; many
// resident warps (a small register budget) keep enough of them in flight.
template <bool BF16, int DH, int G>
__global__ void __launch_bounds__(NT, (Cfg<BF16, DH, G>::MINB)) decode_kernel(Args a) {
  using C = Cfg<BF16, DH, G>;
  constexpr int EPV = C::EPV, NPAIR = C::NPAIR, LP = C::LP, PPW = C::PPW, U = C::U;
  constexpr int NV = C::NV, NF = C::NF, RUN = C::RUN, ROW = C::ROW, ESZ = C::ESZ;

  __shared__ float red_acc[NW][G][DH];
  __shared__ float red_m[NW][G], red_l[NW][G];
  __shared__ int warp_tot[NW];
  extern __shared__ int pre[];  // [B + 1]

  build_prefix<BF16, NT>(a, pre, warp_tot, DH);  // ends with __syncthreads
  const int upb = a.Hkv * a.ngc;  // items per request chunk
  const int total = pre[a.B] * upb;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lg = lane / LP, li = lane % LP, gbase = lg * LP;
  const int pmask = (1 << a.page_shift) - 1;
  const bool one_page = (1 << a.page_shift) >= RUN;  // a block lies in one page
  bool bad_page = false;
  int own0 = 0;  // this lane owns scores own0 .. own0 + NF - 1 of a block after the reduce-scatter
#pragma unroll
  for (int r = 0; r < C::ROUNDS; ++r) {
    const int cur = NV >> r;
    if (cur >= 2 && (li & (LP >> (r + 1)))) own0 += cur / 2;
  }

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const Item it = item_of<G>(a, pre, upb, item);
    const int nblk = (it.s1 - it.s0 + RUN - 1) / RUN;
    const int32_t* trow = a.table + int64_t(it.b) * a.max_pages;
    const int64_t head_off = int64_t(it.kv) << a.page_shift;

    // This lane's slice of the G query rows, pre-scaled to base-2 scores.
    uint64_t qf[G][NPAIR];
    {
      const uint64_t sc = f2pack(a.qscale, a.qscale);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(
            a.q + ((int64_t(it.b) * a.Hq + it.h0 + h) * DH + li * EPV) * ESZ));
        to_pairs<BF16>(r, qf[h]);
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) qf[h][q] = fmul2(qf[h][q], sc);
      }
    }
    // Running state of this lane group: max per head (the same in all its
    // lanes; mown[f] = the max of the head of owned score f), partial sums of
    // the probabilities of the owned scores, this lane's output columns.
    float m[G], mown[NF], lown[NF];
    uint64_t acc[G][NPAIR];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -1e30f;  // finite: a lane group that sees only masked positions keeps finite state
#pragma unroll
      for (int q = 0; q < NPAIR; ++q) acc[h][q] = 0;
    }
#pragma unroll
    for (int f = 0; f < NF; ++f) {
      lown[f] = 0.f;
      mown[f] = -1e30f;
    }

    for (int j = warp; j < nblk; j += NW) {
      const int p0 = it.s0 + j * RUN;
      uint4 kr[U], vr[U];
#pragma unroll
      for (int u = 0; u < U; ++u) kr[u] = vr[u] = make_uint4(0, 0, 0, 0);
      if (one_page) {
        const int pg = __ldg(trow + (p0 >> a.page_shift));
        if (static_cast<unsigned>(pg) < static_cast<unsigned>(a.num_pages)) {
          const int64_t off = (((int64_t(pg) * a.Hkv) << a.page_shift) + head_off + (p0 & pmask) + lg) * ROW + li * 16;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            if (p0 + u * PPW + lg < it.s1) {
              kr[u] = ld_once(a.kp + off + u * PPW * ROW);
              vr[u] = ld_once(a.vp + off + u * PPW * ROW);
            }
          }
        } else {
          bad_page = true;
        }
      } else {
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int t = p0 + u * PPW + lg;
          if (t < it.s1) {
            const int pg = __ldg(trow + (t >> a.page_shift));
            if (static_cast<unsigned>(pg) < static_cast<unsigned>(a.num_pages)) {
              const int64_t off = (((int64_t(pg) * a.Hkv) << a.page_shift) + head_off + (t & pmask)) * ROW + li * 16;
              kr[u] = ld_once(a.kp + off);
              vr[u] = ld_once(a.vp + off);
            } else {
              bad_page = true;
            }
          }
        }
      }
      // Partial dot products of this lane's 16 bytes; score index v = u * G + h.
      float sv[NV];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint64_t kk[NPAIR];
        to_pairs<BF16>(kr[u], kk);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          uint64_t d2 = fmul2(qf[h][0], kk[0]);
#pragma unroll
          for (int q = 1; q < NPAIR; ++q) d2 = ffma2(qf[h][q], kk[q], d2);
          float x, y;
          f2unpack(d2, x, y);
          sv[u * G + h] = x + y;
        }
      }
      // Reduce-scatter over the LP lanes of the group.
#pragma unroll
      for (int r = 0; r < C::ROUNDS; ++r) {
        const int d = LP >> (r + 1);
        const int cur = NV >> r;
        if (cur >= 2) {
          const bool up = (li & d) != 0;
#pragma unroll
          for (int i = 0; i < cur / 2; ++i) {
            const float send = up ? sv[i] : sv[i + cur / 2];
            const float keep = up ? sv[i + cur / 2] : sv[i];
            sv[i] = keep + __shfl_xor_sync(FULL, send, d);
          }
        } else {
          sv[0] += __shfl_xor_sync(FULL, sv[0], d);
        }
      }
      float s_own[NF];
#pragma unroll
      for (int f = 0; f < NF; ++f) {
        const int u = (own0 + f) / G;
        s_own[f] = p0 + u * PPW + lg < it.s1 ? sv[f] : -INFINITY;
      }
      // Raise the running max (rare: the first block of an item, or a score
      // more than 2^8 above it): every lane gathers all scores of its group.
      bool raise = false;
#pragma unroll
      for (int f = 0; f < NF; ++f) raise |= s_own[f] > mown[f] + kRaise;
      if (__any_sync(FULL, raise)) {
        float mn[G];
#pragma unroll
        for (int h = 0; h < G; ++h) mn[h] = m[h];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
          const float sb = __shfl_sync(FULL, s_own[C::slot(v)], gbase + C::holder(v));
          mn[v % G] = fmaxf(mn[v % G], sb);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float al = ex2(m[h] - mn[h]);
          const uint64_t al2 = f2pack(al, al);
#pragma unroll
          for (int q = 0; q < NPAIR; ++q) acc[h][q] = fmul2(acc[h][q], al2);
#pragma unroll
          for (int f = 0; f < NF; ++f) {
            if ((own0 + f) % G == h) {
              lown[f] *= al;
              mown[f] = mn[h];
            }
          }
          m[h] = mn[h];
        }
      }
      // Probabilities of the owned scores, then P * V with every probability.
      float p_own[NF];
#pragma unroll
      for (int f = 0; f < NF; ++f) {
        p_own[f] = ex2(s_own[f] - mown[f]);
        lown[f] += p_own[f];
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint64_t vv[NPAIR];
        to_pairs<BF16>(vr[u], vv);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const int v = u * G + h;
          const float p = __shfl_sync(FULL, p_own[C::slot(v)], gbase + C::holder(v));
          const uint64_t p2 = f2pack(p, p);
#pragma unroll
          for (int q = 0; q < NPAIR; ++q) acc[h][q] = ffma2(p2, vv[q], acc[h][q]);
        }
      }
    }

    // Row sums per head: each score slot's sum taken once, from its owner.
    float l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) l[h] = 0.f;
#pragma unroll
    for (int v = 0; v < NV; ++v) l[v % G] += __shfl_sync(FULL, lown[C::slot(v)], gbase + C::holder(v));

    // Merge the lane groups of the warp (each saw other positions).
#pragma unroll
    for (int off = LP; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mo = __shfl_xor_sync(FULL, m[h], off);
        const float lo = __shfl_xor_sync(FULL, l[h], off);
        const float mn = fmaxf(m[h], mo);
        const float wa = ex2(m[h] - mn), wb = ex2(mo - mn);
        l[h] = l[h] * wa + lo * wb;
        m[h] = mn;
        const uint64_t wa2 = f2pack(wa, wa), wb2 = f2pack(wb, wb);
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          const uint64_t o = __shfl_xor_sync(FULL, acc[h][q], off);
          acc[h][q] = ffma2(o, wb2, fmul2(acc[h][q], wa2));
        }
      }
    }
    if (lg == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int q = 0; q < NPAIR; ++q) {
          float x, y;
          f2unpack(acc[h][q], x, y);
          red_acc[warp][h][li * EPV + 2 * q] = x;
          red_acc[warp][h][li * EPV + 2 * q + 1] = y;
        }
        if (li == 0) {
          red_m[warp][h] = m[h];
          red_l[warp][h] = l[h];
        }
      }
    }
    __syncthreads();
    // Merge the warps; one thread per (head, column).
    for (int idx = tid; idx < G * DH; idx += NT) {
      const int h = idx / DH, d = idx - h * DH;
      float M = red_m[0][h];
#pragma unroll
      for (int q = 1; q < NW; ++q) M = fmaxf(M, red_m[q][h]);
      float Ls = 0.f, A = 0.f;
#pragma unroll
      for (int q = 0; q < NW; ++q) {
        const float wt = ex2(red_m[q][h] - M);
        Ls += red_l[q][h] * wt;
        A += red_acc[q][h][d] * wt;
      }
      const int64_t row = int64_t(it.b) * a.Hq + it.h0 + h;
      if (it.nch == 1) {
        store_elem<BF16>(a.out, row * DH + d, A / Ls);
        if (d == 0) a.lse[row] = 0.69314718055994531f * (M + lg2(Ls));
      } else {
        const int64_t pr = row * a.maxch + it.c;
        a.part_acc[pr * DH + d] = A;
        if (d == 0) {
          a.part_ml[pr * 2] = M;
          a.part_ml[pr * 2 + 1] = Ls;
        }
      }
    }
    __syncthreads();
  }
  if (bad_page) atomicExch(a.status, kStatusBadInput);
}

// Merges the chunk partials of requests longer than one chunk. One warp per
// (request, query head, 32-column slice): lane c of a 32-chunk window weighs
// chunk c once (2^(m_c - M)), the weights are broadcast, and each lane sums
// its column over the chunks with the loads of several chunks in flight.
template <bool BF16, int DH>
__global__ void __launch_bounds__(NT) decode_combine_kernel(Args a) {
  constexpr int NS = (DH + 31) / 32;  // column slices per row
  const int lane = threadIdx.x & 31;
  const int64_t wid = int64_t(blockIdx.x) * NW + (threadIdx.x >> 5);
  if (wid >= int64_t(a.B) * a.Hq * NS) return;
  const int64_t row = wid / NS;
  const int d = int(wid - row * NS) * 32 + lane;
  const int b = int(row / a.Hq);
  const int L = __ldg(a.lens + b);
  if (!len_ok(L, a)) return;  // written as NaN by the decode kernel
  const int nch = n_chunks(L);
  if (nch == 1) return;       // written by the decode kernel
  const float* ml = a.part_ml + row * a.maxch * 2;
  const float* pa = a.part_acc + row * a.maxch * DH;
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, __ldg(ml + 2 * c));
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, off));
  float Ls = 0.f, o = 0.f;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    float wc = 0.f;
    if (c < nch) {
      wc = ex2(__ldg(ml + 2 * c) - M);
      Ls += __ldg(ml + 2 * c + 1) * wc;
    }
    const int n = min(32, nch - c0);
#pragma unroll 8
    for (int i = 0; i < n; ++i) {
      const float w = __shfl_sync(FULL, wc, i);
      if (d < DH) o += __ldg(pa + int64_t(c0 + i) * DH + d) * w;
    }
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) Ls += __shfl_xor_sync(FULL, Ls, off);
  if (d < DH) store_elem<BF16>(a.out, row * DH + d, o / Ls);
  if (d == 0) a.lse[row] = 0.69314718055994531f * (M + lg2(Ls));
}

template <bool BF16, int DH, int G>
cudaError_t launch(const DecodeParams& p, const Args& a, cudaStream_t st) {
  auto k = decode_kernel<BF16, DH, G>;
  using C = Cfg<BF16, DH, G>;
  const size_t dyn = size_t(p.B + 1) * sizeof(int);
  // Opt in once per device to the largest dynamic size any batch needs.
  static std::atomic<unsigned long long> opted{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (!(opted.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int((kDecodeMaxBatch + 1) * sizeof(int)));
    if (e != cudaSuccess) return e;
    opted.fetch_or(bit, std::memory_order_acq_rel);
  }
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, NT, dyn);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const int64_t upper = p.B * int64_t(a.maxch) * a.Hkv * a.ngc;
  const int64_t grid = std::min<int64_t>(upper, int64_t(p.sms) * per_sm);
  k<<<dim3(unsigned(grid)), NT, dyn, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess || a.maxch <= 1) return e;
  const int64_t warps = p.B * p.Hq * ((DH + 31) / 32);
  decode_combine_kernel<BF16, DH><<<dim3(unsigned((warps + NW - 1) / NW)), NT, 0, st>>>(a);
  return cudaGetLastError();
}

template <bool BF16, int DH>
cudaError_t launch_g(const DecodeParams& p, const Args& a, cudaStream_t st, int G) {
  switch (G) {
    case 8: return launch<BF16, DH, 8>(p, a, st);
    case 4: return launch<BF16, DH, 4>(p, a, st);
    case 2: return launch<BF16, DH, 2>(p, a, st);
    default: return launch<BF16, DH, 1>(p, a, st);
  }
}

template <bool BF16>
cudaError_t launch_dh(const DecodeParams& p, const Args& a, cudaStream_t st, int G) {
  switch (p.Dh) {
    case 16: return launch_g<BF16, 16>(p, a, st, G);
    case 32: return launch_g<BF16, 32>(p, a, st, G);
    case 64: return launch_g<BF16, 64>(p, a, st, G);
    default: return launch_g<BF16, 128>(p, a, st, G);
  }
}

}  // namespace dec

cudaError_t launch_paged_decode(const DecodeParams& p, cudaStream_t st) {
  dec::Args a{};
  a.q = static_cast<const char*>(p.q);
  a.kp = static_cast<const char*>(p.k_pool);
  a.vp = static_cast<const char*>(p.v_pool);
  a.table = p.page_table;
  a.lens = p.seq_lens;
  a.out = static_cast<char*>(p.out);
  a.lse = p.lse;
  a.part_ml = p.part_ml;
  a.part_acc = p.part_acc;
  a.status = p.status;
  a.B = int(p.B);
  a.Hq = int(p.Hq);
  a.Hkv = int(p.Hkv);
  a.g = int(p.Hq / p.Hkv);
  // Query heads per item: the largest of 8, 4, 2, 1 that divides the group.
  const int G = a.g % 8 == 0 ? 8 : a.g % 4 == 0 ? 4 : a.g % 2 == 0 ? 2 : 1;
  a.ngc = a.g / G;
  int shift = 0;
  while ((int64_t(1) << shift) < p.page_size) ++shift;
  a.page_shift = shift;
  a.max_pages = int(p.max_pages);
  a.num_pages = int(p.num_pages);
  a.maxch = int(decode_max_chunks(p.page_size, p.max_pages));
  a.qscale = float(1.4426950408889634 / __builtin_sqrt(double(p.Dh)));
  a.timeout_ns = p.timeout_ns;
  return p.bf16 ? dec::launch_dh<true>(p, a, st, G) : dec::launch_dh<false>(p, a, st, G);
}

}  // namespace rca
