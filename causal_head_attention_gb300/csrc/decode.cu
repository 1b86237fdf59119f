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
// The work is HBM-bound: every cached K/V byte is read once and there is one
// query row per KV head group, too little reuse for the tensor cores. The design
// streams the pools with 16-byte loads straight into registers:
//  * Work items are (request, chunk of kDecodeChunk positions, KV head group of
//    G query heads). Persistent CTAs take items i, i + grid, ... from the list
//    of non-empty items, which every CTA rebuilds from the lengths (a prefix
//    sum over the requests in shared memory), so no CTA is launched empty and
//    every CTA gets the same number of items to within one.
//  * A position's head_dim row is spread over LP = Dh * bytes / 16 lanes (one
//    16-byte vector each); a warp covers 32 / LP positions per step and each
//    thread keeps U steps of K and V loads in flight.
//  * Scores: packed fp32x2 products, a butterfly over the LP lanes. Softmax:
//    one rescale per block of U positions (running max in base 2, the query is
//    pre-scaled by scale * log2 e), packed fp32x2 accumulation of p * V.
//  * A request whose length fits one chunk writes O and LSE directly; longer
//    requests leave (max, sum, unnormalised O) per chunk and a combine kernel
//    merges them.
// Device-side inputs are checked as they are read: a page ID outside
// [0, num_pages) is never dereferenced (the position is skipped) and a length
// outside [1, max_pages * page_size] makes that request's outputs NaN; both
// record kStatusBadInput in the status word.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "decode.h"
#include "tc.cuh"

namespace rca {
namespace dec {

constexpr int NW = 4;        // warps per CTA
constexpr int NT = NW * 32;  // threads per CTA

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
};

template <bool BF16, int DH, int G>
struct Cfg {
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr int EPV = 16 / ESZ;   // elements per 16-byte vector
  static constexpr int NPAIR = EPV / 2;  // fp32x2 pairs per vector
  static constexpr int LP = DH / EPV;    // lanes per position
  static constexpr int PPW = 32 / LP;    // positions per warp step
  static constexpr int U = G >= 4 ? 2 : 4;
  static constexpr int STEP = NW * PPW * U;  // positions per CTA iteration
  static_assert(LP >= 1 && LP <= 32 && (32 % LP) == 0, "head width");
};

// 16-byte load of data read exactly once (not kept in L1).
__device__ __forceinline__ uint4 ld_once(const char* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
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
template <bool BF16>
__device__ void build_prefix(const Args& a, int* pre, int* warp_tot, int dh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int seg = (a.B + NT - 1) / NT;
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
        for (int d = 0; d < dh; ++d) store_elem<BF16>(a.out, (int64_t(i) * a.Hq + h) * dh + d, __int_as_float(0x7fc00000));
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
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
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

template <bool BF16, int DH, int G>
__global__ void __launch_bounds__(NT) decode_kernel(Args a) {
  using C = Cfg<BF16, DH, G>;
  constexpr int EPV = C::EPV, NPAIR = C::NPAIR, LP = C::LP, PPW = C::PPW, U = C::U, STEP = C::STEP;
  constexpr int ESZ = C::ESZ;

  __shared__ float red_acc[NW][G][DH];
  __shared__ float red_m[NW][G], red_l[NW][G];
  __shared__ int warp_tot[NW];
  extern __shared__ int pre[];  // [B + 1]

  build_prefix<BF16>(a, pre, warp_tot, DH);
  const int upb = a.Hkv * a.ngc;  // items per request chunk
  const int total = pre[a.B] * upb;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int lg = lane / LP, li = lane % LP;
  const int pmask = (1 << a.page_shift) - 1;
  bool bad_page = false;

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const int ci = item / upb, u_ = item - ci * upb;
    const int b = find_request(pre, a.B, ci);
    const int c = ci - pre[b];
    const int nch = pre[b + 1] - pre[b];
    const int kv = u_ / a.ngc, gc = u_ - kv * a.ngc;
    const int h0 = kv * a.g + gc * G;
    const int L = __ldg(a.lens + b);
    const int s0 = c * kDecodeChunk, s1 = min(L, s0 + kDecodeChunk);

    // This lane's slice of the G query rows, pre-scaled to base-2 scores.
    uint64_t qf[G][NPAIR];
    {
      const uint64_t sc = f2pack(a.qscale, a.qscale);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint4 r = *reinterpret_cast<const uint4*>(
            a.q + ((int64_t(b) * a.Hq + h0 + h) * DH + li * EPV) * ESZ);
        to_pairs<BF16>(r, qf[h]);
#pragma unroll
        for (int j = 0; j < NPAIR; ++j) qf[h][j] = fmul2(qf[h][j], sc);
      }
    }

    float m[G], l[G];
    uint64_t acc[G][NPAIR];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -1e30f;  // finite: an all-masked block leaves the state unchanged
      l[h] = 0.f;
#pragma unroll
      for (int j = 0; j < NPAIR; ++j) acc[h][j] = 0;
    }

    const int32_t* trow = a.table + int64_t(b) * a.max_pages;
    for (int base = s0; base < s1; base += STEP) {
      uint4 kr[U], vr[U];
      bool ok[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = base + (u * NW + warp) * PPW + lg;
        ok[u] = t < s1;
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = kr[u];
        if (ok[u]) {
          const int pg = __ldg(trow + (t >> a.page_shift));
          if (static_cast<unsigned>(pg) >= static_cast<unsigned>(a.num_pages)) {
            bad_page = true;
            ok[u] = false;
          } else {
            const int64_t row = ((int64_t(pg) * a.Hkv + kv) << a.page_shift) | (t & pmask);
            const int64_t off = (row * DH + li * EPV) * ESZ;
            kr[u] = ld_once(a.kp + off);
            vr[u] = ld_once(a.vp + off);
          }
        }
      }
      // Scores of the U positions for the G heads (each lane: its 16-byte slice).
      float s[U][G];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint64_t kk[NPAIR];
        to_pairs<BF16>(kr[u], kk);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          uint64_t d2 = fmul2(qf[h][0], kk[0]);
#pragma unroll
          for (int j = 1; j < NPAIR; ++j) d2 = ffma2(qf[h][j], kk[j], d2);
          float x, y;
          f2unpack(d2, x, y);
          s[u][h] = x + y;
        }
      }
#pragma unroll
      for (int off = 1; off < LP; off <<= 1)
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int h = 0; h < G; ++h) s[u][h] += __shfl_xor_sync(0xffffffffu, s[u][h], off);
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int h = 0; h < G; ++h)
          if (!ok[u]) s[u][h] = -INFINITY;

      // One rescale per block, then p = 2^(s - m) and acc += p * V.
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = s[0][h];
#pragma unroll
        for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[u][h]);
        const float mn = fmaxf(m[h], mx);
        const float al = ex2(m[h] - mn);
        m[h] = mn;
        l[h] *= al;
        const uint64_t al2 = f2pack(al, al);
#pragma unroll
        for (int j = 0; j < NPAIR; ++j) acc[h][j] = fmul2(acc[h][j], al2);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint64_t vv[NPAIR];
        to_pairs<BF16>(vr[u], vv);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float p = ex2(s[u][h] - m[h]);
          l[h] += p;
          const uint64_t p2 = f2pack(p, p);
#pragma unroll
          for (int j = 0; j < NPAIR; ++j) acc[h][j] = ffma2(p2, vv[j], acc[h][j]);
        }
      }
    }

    // Merge the lane groups of the warp (each saw other positions).
#pragma unroll
    for (int off = LP; off < 32; off <<= 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float mo = __shfl_xor_sync(0xffffffffu, m[h], off);
        const float lo = __shfl_xor_sync(0xffffffffu, l[h], off);
        const float mn = fmaxf(m[h], mo);
        const float wa = ex2(m[h] - mn), wb = ex2(mo - mn);
        l[h] = l[h] * wa + lo * wb;
        m[h] = mn;
        const uint64_t wa2 = f2pack(wa, wa), wb2 = f2pack(wb, wb);
#pragma unroll
        for (int j = 0; j < NPAIR; ++j) {
          const uint64_t o = __shfl_xor_sync(0xffffffffu, acc[h][j], off);
          acc[h][j] = ffma2(o, wb2, fmul2(acc[h][j], wa2));
        }
      }
    }
    if (lg == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int j = 0; j < NPAIR; ++j) {
          float x, y;
          f2unpack(acc[h][j], x, y);
          red_acc[warp][h][li * EPV + 2 * j] = x;
          red_acc[warp][h][li * EPV + 2 * j + 1] = y;
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
      for (int w = 1; w < NW; ++w) M = fmaxf(M, red_m[w][h]);
      float Ls = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float wt = ex2(red_m[w][h] - M);
        Ls += red_l[w][h] * wt;
        A += red_acc[w][h][d] * wt;
      }
      const int64_t row = int64_t(b) * a.Hq + h0 + h;
      if (nch == 1) {
        store_elem<BF16>(a.out, row * DH + d, A / Ls);
        if (d == 0) a.lse[row] = 0.69314718055994531f * (M + lg2(Ls));
      } else {
        const int64_t pr = row * a.maxch + c;
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

// Merges the chunk partials of requests longer than one chunk: one warp per
// (request, query head).
template <bool BF16, int DH>
__global__ void __launch_bounds__(NT) decode_combine_kernel(Args a) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * NW + (threadIdx.x >> 5);
  if (row >= int64_t(a.B) * a.Hq) return;
  const int b = int(row / a.Hq);
  const int L = __ldg(a.lens + b);
  if (!len_ok(L, a)) return;  // written as NaN by the decode kernel
  const int nch = n_chunks(L);
  if (nch == 1) return;       // written by the decode kernel
  const float* ml = a.part_ml + row * a.maxch * 2;
  const float* pa = a.part_acc + row * a.maxch * DH;
  float M = -INFINITY;
  for (int c = lane; c < nch; c += 32) M = fmaxf(M, ml[2 * c]);
#pragma unroll
  for (int off = 16; off; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float Ls = 0.f;
  for (int c = lane; c < nch; c += 32) Ls += ml[2 * c + 1] * ex2(ml[2 * c] - M);
#pragma unroll
  for (int off = 16; off; off >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, off);
  for (int d = lane; d < DH; d += 32) {
    float o = 0.f;
    for (int c = 0; c < nch; ++c) o += pa[int64_t(c) * DH + d] * ex2(ml[2 * c] - M);
    store_elem<BF16>(a.out, row * DH + d, o / Ls);
  }
  if (lane == 0) a.lse[row] = 0.69314718055994531f * (M + lg2(Ls));
}

template <bool BF16, int DH, int G>
cudaError_t launch(const DecodeParams& p, const Args& a, cudaStream_t st) {
  auto k = decode_kernel<BF16, DH, G>;
  const size_t dyn = size_t(p.B + 1) * sizeof(int);
  cudaError_t e;
  if (dyn > 16384) {  // static (<= 17 KB) + dynamic may pass the 48 KB default
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn));
    if (e != cudaSuccess) return e;
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
  const int64_t rows = p.B * p.Hq;
  decode_combine_kernel<BF16, DH><<<dim3(unsigned((rows + NW - 1) / NW)), NT, 0, st>>>(a);
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
  return p.bf16 ? dec::launch_dh<true>(p, a, st, G) : dec::launch_dh<false>(p, a, st, G);
}

}  // namespace rca
