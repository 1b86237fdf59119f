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
//    requests leave (max, sum, unnormalised O) per chunk and a combine kernel,
//    launched as a programmatic dependent (its launch overlaps the decode
//    kernel's tail), merges them.
//  * bf16 storage with two or more query heads per KV head runs the group's
//    two products on the tensor cores instead (decode_mma_kernel below): the
//    same items, loads and softmax, with the dot products and P * V as
//    warp-level MMAs fed straight from the loaded registers.
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

constexpr int NW = 4;  // warps per CTA (decode kernels); the combine kernel has NT threads too
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

// Merges the NW warps' partial states of one item (written to shared memory by
// every warp before the call) and writes the output rows and LSE, or the
// item's partial when the request spans several chunks. One thread per
// (head, column); ends with the block synchronised so the buffers can be
// reused.
template <bool BF16, int DH, int G>
__device__ __forceinline__ void finish_item(const Args& a, const Item& it, const float (&red_acc)[NW][G][DH],
                                            const float (&red_m)[NW][G], const float (&red_l)[NW][G]) {
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * DH; idx += NT) {
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
    finish_item<BF16, DH, G>(a, it, red_acc, red_m, red_l);
  }
  if (bad_page) atomicExch(a.status, kStatusBadInput);
}

// ---------------------------------------------------------------------------
// Tensor-core variant (bf16 storage). The G query rows of a KV head group
// share every K and V row, so a block of 16 positions is two small dense
// products, run as warp-level m16n8k16 bf16 MMAs with fp32 accumulation and
// the G heads padded to the 8 columns of n:
//   S^T [16 positions x 8 heads]  = K [16 x Dh] . Q^T [Dh x 8]
//   O^T [Dh x 8 heads]           += V^T [Dh x 16] . P^T [16 x 8]
// The operand fragments are filled straight from 16-byte global loads (no
// shared-memory staging, the same load pattern as the CUDA-core kernel):
//  * the order of the head dimension inside q . k is free, so the dims are
//    dealt to the four lanes of a quad such that a lane's share of a K row
//    (and of the query row) is whole vectors, consecutive lanes reading
//    consecutive vectors;
//  * the output dims are dealt to the eight lane groups the same way for V;
//    a V^T fragment register pairs one dim of two positions (one byte permute);
//  * the S^T accumulator becomes the P^T operand after one 8x8 transpose of
//    each half (movmatrix). The probabilities enter as bf16 hi + lo parts
//    (two MMAs), so the output keeps the accuracy of fp32 probabilities.
// Softmax state per lane: the running max and partial sum of its two heads
// (2t, 2t + 1 for quad lane t), the max being the same across the lane groups.
// ---------------------------------------------------------------------------
// Resident CTAs per SM the tensor-core kernel's registers are sized for (one
// 16-position block of K and V per warp in flight; a second block in flight
// at 2 CTAs per SM, or 4 CTAs per SM with spills, both measured slower).
#ifndef DEC_MMA_MINB
#define DEC_MMA_MINB 3
#endif
static_assert(kDecodeChunk / 16 <= 32 * NW, "a warp's block pages fit one lane each");

template <int DH>
struct MmaCfg {
  static constexpr int S = DH / 16;  // k-steps of the score product = m-tiles of the output
  static constexpr int KW = DH / 8;  // 32-bit words of a K (or query) row per quad lane
  static constexpr int KL = KW * 4 < 16 ? KW * 4 : 16;  // bytes per load
  static constexpr int NKL = KW * 4 / KL;
  static constexpr int VW = DH / 16;  // words of a V row per lane group
  static constexpr int VL = VW * 4 < 16 ? VW * 4 : 16;
  static constexpr int NVL = VW * 4 / VL;
  // Word j of quad lane t's share of a K / query row is the row's word
  // kword(j, t); words 2s and 2s + 1 hold the lane's k-step-s operand columns
  // (2t, 2t + 1) and (2t + 8, 2t + 9).
  __host__ __device__ static constexpr int kword(int j, int t) {
    return ((j / (KL / 4)) * 4 + t) * (KL / 4) + j % (KL / 4);
  }
  // Word r of lane group g's share of a V row is the row's word vword(r, g):
  // its low / high halves are output m-tile r's rows g / g + 8.
  __host__ __device__ static constexpr int vword(int r, int g) {
    return ((r / (VL / 4)) * 8 + g) * (VL / 4) + r % (VL / 4);
  }
};

// One warp block's K and V fragments (see MmaCfg): K rows g, g + 8 and V
// rows 2t, 2t + 1, 2t + 8, 2t + 9 of 16 consecutive positions.
template <int DH>
struct MmaBlock {
  uint32_t kw[2][DH / 8];
  uint32_t vw[4][DH / 16];
};

template <int BYTES, bool ONCE>
__device__ __forceinline__ void ld_words(const char* p, uint32_t* w) {
  if constexpr (BYTES == 16) {
    if constexpr (ONCE)
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "l"(p));
    else
      asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "l"(p));
  } else if constexpr (BYTES == 8) {
    asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(w[0]), "=r"(w[1]) : "l"(p));
  } else {
    static_assert(BYTES == 4, "load width");
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(w[0]) : "l"(p));
  }
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit values held one word per lane (row
// lane / 4, columns 2 (lane % 4) and 2 (lane % 4) + 1).
__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

template <int DH, int G>
__global__ void __launch_bounds__(NT, DEC_MMA_MINB) decode_mma_kernel(Args a) {
  using M = MmaCfg<DH>;
  constexpr int S = M::S, KW = M::KW, KL = M::KL, VL = M::VL, ROW = DH * 2;
  static_assert(G >= 1 && G <= 8, "a group fills at most the 8 columns of n");

  __shared__ __align__(16) float red_acc[NW][G][DH];  // float2 stores
  __shared__ float red_m[NW][G], red_l[NW][G];
  __shared__ int warp_tot[NW];
  extern __shared__ int pre[];  // [B + 1]

  build_prefix<true, NT>(a, pre, warp_tot, DH);  // ends with __syncthreads
  const int upb = a.Hkv * a.ngc;
  const int total = pre[a.B] * upb;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;  // lane group (row of a fragment), quad lane
  const int pmask = (1 << a.page_shift) - 1;
  const bool one_page = a.page_shift >= 4;  // a block of 16 aligned positions lies in one page
  bool bad_page = false;

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const Item it = item_of<G>(a, pre, upb, item);
    const int nblk = (it.s1 - it.s0 + 15) >> 4;
    const int32_t* trow = a.table + int64_t(it.b) * a.max_pages;
    const int64_t head_off = int64_t(it.kv) << a.page_shift;

    // Query head g of the group as the score product's n column g (zero
    // columns past the group).
    uint32_t qw[KW];
#pragma unroll
    for (int j = 0; j < KW; ++j) qw[j] = 0;
    if (g < G) {
      const char* qrow = a.q + (int64_t(it.b) * a.Hq + it.h0 + g) * ROW;
#pragma unroll
      for (int i = 0; i < M::NKL; ++i) ld_words<KL, false>(qrow + (i * 4 + t) * KL, qw + i * (KL / 4));
    }
    float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;  // heads 2t, 2t + 1
    float acc[S][4];
#pragma unroll
    for (int r = 0; r < S; ++r) acc[r][0] = acc[r][1] = acc[r][2] = acc[r][3] = 0.f;

    // This warp takes blocks warp, warp + NW, ... of the item; lane i reads
    // the page of its i-th block up front, so a block's K/V loads never wait
    // for a page-table load.
    const int nmy = nblk > warp ? (nblk - warp + NW - 1) / NW : 0;
    int pg_lane = 0;
    if (one_page && lane < nmy) pg_lane = __ldg(trow + ((it.s0 + (warp + lane * NW) * 16) >> a.page_shift));

    // Loads of the warp's i-th block: K rows g, g + 8; V rows 2t, 2t + 1, 2t + 8, 2t + 9.
    auto load_block = [&](MmaBlock<DH>& bk, int i) {
      const int p0 = it.s0 + (warp + i * NW) * 16;
      int64_t blk = -1;  // byte offset of position p0's row when the block lies in one page
      if (one_page) {
        const int pg = __shfl_sync(FULL, pg_lane, i);
        if (static_cast<unsigned>(pg) < static_cast<unsigned>(a.num_pages))
          blk = (((int64_t(pg) * a.Hkv) << a.page_shift) + head_off + (p0 & pmask)) * ROW;
        else
          bad_page = true;
      }
      // Byte offset of position p0 + d's row, or -1 (past the end, or a bad page).
      auto row_of = [&](int d) -> int64_t {
        const int pos = p0 + d;
        if (pos >= it.s1) return -1;
        if (one_page) return blk < 0 ? -1 : blk + int64_t(d) * ROW;
        const int pg = __ldg(trow + (pos >> a.page_shift));
        if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
          bad_page = true;
          return -1;
        }
        return (((int64_t(pg) * a.Hkv) << a.page_shift) + head_off + (pos & pmask)) * ROW;
      };
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t r = row_of(g + 8 * h);
#pragma unroll
        for (int n = 0; n < M::NKL; ++n) {
          if (r >= 0) {
            ld_words<KL, true>(a.kp + r + (n * 4 + t) * KL, bk.kw[h] + n * (KL / 4));
          } else {
#pragma unroll
            for (int w = 0; w < KL / 4; ++w) bk.kw[h][n * (KL / 4) + w] = 0;
          }
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t r = row_of(2 * t + (c & 1) + 8 * (c >> 1));
#pragma unroll
        for (int n = 0; n < M::NVL; ++n) {
          if (r >= 0) {
            ld_words<VL, true>(a.vp + r + (n * 8 + g) * VL, bk.vw[c] + n * (VL / 4));
          } else {
#pragma unroll
            for (int w = 0; w < VL / 4; ++w) bk.vw[c][n * (VL / 4) + w] = 0;
          }
        }
      }
    };

    auto compute_block = [&](const MmaBlock<DH>& bk, int i) {
      const int p0 = it.s0 + (warp + i * NW) * 16;
      // Scores: s[0], s[1] = position g, heads 2t, 2t + 1; s[2], s[3] = position g + 8.
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < S; ++k)
        mma_bf16_16816(s, bk.kw[0][2 * k], bk.kw[1][2 * k], bk.kw[0][2 * k + 1], bk.kw[1][2 * k + 1], qw[2 * k],
                       qw[2 * k + 1]);
      const bool va = p0 + g < it.s1, vb = p0 + g + 8 < it.s1;
      const float x0 = va ? s[0] * a.qscale : -INFINITY, x1 = va ? s[1] * a.qscale : -INFINITY;
      const float x2 = vb ? s[2] * a.qscale : -INFINITY, x3 = vb ? s[3] * a.qscale : -INFINITY;
      // Raise the running max only when a score passes it by more than 2^8.
      const bool raise = fmaxf(x0, x2) > m0 + kRaise || fmaxf(x1, x3) > m1 + kRaise;
      if (__any_sync(FULL, raise)) {
        float n0 = fmax3(m0, x0, x2), n1 = fmax3(m1, x1, x3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          n0 = fmaxf(n0, __shfl_xor_sync(FULL, n0, off));
          n1 = fmaxf(n1, __shfl_xor_sync(FULL, n1, off));
        }
        const float al0 = ex2(m0 - n0), al1 = ex2(m1 - n1);
#pragma unroll
        for (int r = 0; r < S; ++r) {
          acc[r][0] *= al0;
          acc[r][1] *= al1;
          acc[r][2] *= al0;
          acc[r][3] *= al1;
        }
        l0 *= al0;
        l1 *= al1;
        m0 = n0;
        m1 = n1;
      }
      const float pa = ex2(x0 - m0), pb = ex2(x1 - m1), pc = ex2(x2 - m0), pd = ex2(x3 - m1);
      l0 += pa + pc;
      l1 += pb + pd;
      uint32_t hi01, lo01, hi23, lo23;
      split_bf16x2(pa, pb, hi01, lo01);
      split_bf16x2(pc, pd, hi23, lo23);
      const uint32_t bh0 = transpose8x8(hi01), bh1 = transpose8x8(hi23);
      const uint32_t bl0 = transpose8x8(lo01), bl1 = transpose8x8(lo23);
#pragma unroll
      for (int r = 0; r < S; ++r) {
        const uint32_t a0 = __byte_perm(bk.vw[0][r], bk.vw[1][r], 0x5410);
        const uint32_t a1 = __byte_perm(bk.vw[0][r], bk.vw[1][r], 0x7632);
        const uint32_t a2 = __byte_perm(bk.vw[2][r], bk.vw[3][r], 0x5410);
        const uint32_t a3 = __byte_perm(bk.vw[2][r], bk.vw[3][r], 0x7632);
        mma_bf16_16816(acc[r], a0, a1, a2, a3, bh0, bh1);
        mma_bf16_16816(acc[r], a0, a1, a2, a3, bl0, bl1);
      }
    };

    for (int i = 0; i < nmy; ++i) {
      MmaBlock<DH> bk;
      load_block(bk, i);
      compute_block(bk, i);
    }

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(FULL, l0, off);
      l1 += __shfl_xor_sync(FULL, l1, off);
    }
    // acc[r] = O^T rows (dims) of word vword(r, g), columns (heads) 2t, 2t + 1.
    const int ha = 2 * t, hb = 2 * t + 1;
#pragma unroll
    for (int r = 0; r < S; ++r) {
      const int w = M::vword(r, g);
      if (ha < G) *reinterpret_cast<float2*>(&red_acc[warp][ha][2 * w]) = make_float2(acc[r][0], acc[r][2]);
      if (hb < G) *reinterpret_cast<float2*>(&red_acc[warp][hb][2 * w]) = make_float2(acc[r][1], acc[r][3]);
    }
    if (g == 0) {
      if (ha < G) {
        red_m[warp][ha] = m0;
        red_l[warp][ha] = l0;
      }
      if (hb < G) {
        red_m[warp][hb] = m1;
        red_l[warp][hb] = l1;
      }
    }
    finish_item<true, DH, G>(a, it, red_acc, red_m, red_l);
  }
  if (bad_page) atomicExch(a.status, kStatusBadInput);
}

// Folds one partial (max m2, sum l2, unnormalised row v2) into a running
// merge (M, L, o): both are rescaled to the larger max. An empty side (max
// -inf, nothing merged yet) gets weight 0.
__device__ __forceinline__ void merge_partial(float& M, float& L, float4& o, float m2, float l2, const float4& v2) {
  const float Mn = fmaxf(M, m2);
  if (Mn == -INFINITY) return;  // both sides empty
  const float wa = ex2(M - Mn), wb = ex2(m2 - Mn);
  L = L * wa + l2 * wb;
  o.x = o.x * wa + v2.x * wb;
  o.y = o.y * wa + v2.y * wb;
  o.z = o.z * wa + v2.z * wb;
  o.w = o.w * wa + v2.w * wb;
  M = Mn;
}

// Merges the chunk partials of requests longer than one chunk. Each
// (request, query head, 4 columns) is shared by 4 adjacent lanes: lane s folds
// chunks s, s + 4, ... in one online pass, CB chunks' loads in flight at once,
// then the 4 lanes merge by shuffles. Launched as a programmatic dependent of
// the decode kernel, so its launch overlaps the decode kernel's tail;
// griddepcontrol.wait holds it until the decode grid has finished and its
// writes are visible. The partials were written by that grid, so they are read
// through L2 (ld.global.cg).
template <bool BF16, int DH>
__global__ void __launch_bounds__(NT) decode_combine_kernel(Args a) {
  constexpr int NQ = DH / 4, SPLIT = 4, CB = 8;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t id = int64_t(blockIdx.x) * NT + threadIdx.x;
  const int64_t unit = id / SPLIT;  // the 4 lanes of a unit exit together
  const int sub = int(id % SPLIT);
  if (unit >= int64_t(a.B) * a.Hq * NQ) return;
  const int64_t row = unit / NQ;
  const int d = int(unit - row * NQ) * 4;
  const int L = __ldg(a.lens + row / a.Hq);
  if (!len_ok(L, a)) return;  // written as NaN by the decode kernel
  const int nch = n_chunks(L);
  if (nch == 1) return;       // written by the decode kernel
  const float* ml = a.part_ml + row * a.maxch * 2;
  const float* pa = a.part_acc + row * a.maxch * DH + d;
  float M = -INFINITY, Ls = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = sub; c0 < nch; c0 += SPLIT * CB) {
    float2 mc[CB];
    float4 v[CB];
#pragma unroll
    for (int k = 0; k < CB; ++k) {
      const int c = c0 + SPLIT * k;
      if (c < nch) {
        mc[k] = __ldcg(reinterpret_cast<const float2*>(ml + 2 * c));
        v[k] = __ldcg(reinterpret_cast<const float4*>(pa + int64_t(c) * DH));
      } else {
        mc[k] = make_float2(-INFINITY, 0.f);
        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int k = 0; k < CB; ++k) merge_partial(M, Ls, o, mc[k].x, mc[k].y, v[k]);
  }
  const unsigned gmask = 0xfu << (threadIdx.x & 28);
#pragma unroll
  for (int off = 1; off < SPLIT; off <<= 1) {
    float4 vo;
    const float mo = __shfl_xor_sync(gmask, M, off), lo = __shfl_xor_sync(gmask, Ls, off);
    vo.x = __shfl_xor_sync(gmask, o.x, off);
    vo.y = __shfl_xor_sync(gmask, o.y, off);
    vo.z = __shfl_xor_sync(gmask, o.z, off);
    vo.w = __shfl_xor_sync(gmask, o.w, off);
    merge_partial(M, Ls, o, mo, lo, vo);
  }
  if (sub != 0) return;
  const float r = 1.f / Ls;
  store_elem<BF16>(a.out, row * DH + d, o.x * r);
  store_elem<BF16>(a.out, row * DH + d + 1, o.y * r);
  store_elem<BF16>(a.out, row * DH + d + 2, o.z * r);
  store_elem<BF16>(a.out, row * DH + d + 3, o.w * r);
  if (d == 0) a.lse[row] = 0.69314718055994531f * (M + lg2(Ls));
}

// bf16 groups of at least this many query heads take the tensor-core kernel.
#ifndef DEC_MMA_MIN_G
#define DEC_MMA_MIN_G 2
#endif

template <bool BF16, int DH, int G>
constexpr auto decode_entry() {
  if constexpr (BF16 && G >= DEC_MMA_MIN_G)
    return decode_mma_kernel<DH, G>;
  else
    return decode_kernel<BF16, DH, G>;
}

template <bool BF16, int DH, int G>
cudaError_t launch(const DecodeParams& p, const Args& a, cudaStream_t st) {
  const auto k = decode_entry<BF16, DH, G>();
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
  const int64_t threads = p.B * p.Hq * (DH / 4) * 4;  // 4 lanes per (row, 4 columns)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((threads + NT - 1) / NT));
  cfg.blockDim = dim3(NT);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel<BF16, DH>, a);
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
