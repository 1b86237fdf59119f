// Materialized causal attention for sm_103a: the path that returns and keeps
// the probabilities ("Execution Backends and the Python ABI", section "What
// the Metal slice does": the default materialized request returns
// probabilities and context and retains the [batch, heads, time, time]
// probabilities for its VJPs; the probability-returning diagnostic always
// takes it; causal softmax scales, masks and normalises in one kernel).
//
// Per (batch b, query head h), KV head kv = h / (Hq / Hkv):
//   forward   S = Q K^T;  P = causal_softmax(scale * S) (zero above the
//             diagonal);  LSE = ln sum exp(scale * S);  O = P V
//   backward  dP = dO V^T (+ dP_up, the caller's gradient of P);
//             dS = scale * P * (dP - rowsum(P * dP));  dQ = dS K;
//             dK = dS^T Q;  dV = P^T dO  (dK, dV summed over the group)
//
// The five products are this library's tensor-core kernels (mat_gemm.cuh),
// computed over the causal triangle only: score tiles above the diagonal are
// never formed, and the products over T read only the kept triangle of P or
// dS. The fused causal softmax and its VJP are the kernels below (one warp per
// row, bound by HBM traffic of the [T, T] rows). fp32 storage: Q, K, V and dO
// are first split into three bf16 parts each (split3_kernel), so that the
// scores keep fp32 accuracy.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstdio>
#include <mutex>

#include "mat_gemm.cuh"
#include "materialized.h"
#include "tc.cuh"

namespace rca {
namespace mat {

constexpr unsigned FULL = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// fp32 -> three bf16 parts x = x0 + x1 + x2 (x0 = bf16(x), x1 = bf16(x - x0),
// x2 = bf16(x - x0 - x1); both differences are exact in fp32), 4 elements a
// thread; n is a multiple of 4.
__global__ void split3_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ p0,
                              __nv_bfloat16* __restrict__ p1, __nv_bfloat16* __restrict__ p2, int64_t n4) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
    const float4 f = reinterpret_cast<const float4*>(src)[i];
    uint32_t h01, l01, h23, l23;
    split_bf16x2(f.x, f.y, h01, l01);
    split_bf16x2(f.z, f.w, h23, l23);
    // residuals after the first two parts
    const float r0 = f.x - __uint_as_float(h01 << 16) - __uint_as_float(l01 << 16);
    const float r1 = f.y - __uint_as_float(h01 & 0xffff0000u) - __uint_as_float(l01 & 0xffff0000u);
    const float r2 = f.z - __uint_as_float(h23 << 16) - __uint_as_float(l23 << 16);
    const float r3 = f.w - __uint_as_float(h23 & 0xffff0000u) - __uint_as_float(l23 & 0xffff0000u);
    reinterpret_cast<uint2*>(p0)[i] = make_uint2(h01, h23);
    reinterpret_cast<uint2*>(p1)[i] = make_uint2(l01, l23);
    reinterpret_cast<uint2*>(p2)[i] = make_uint2(pack_bf16(r0, r1), pack_bf16(r2, r3));
  }
}

// Fused causal softmax (scale, mask, normalise), in place, one warp per row
// (e, i) of S [E, T, T]: P[i, j] = exp(scale S[i, j] - LSE[i]) for j <= i, 0
// above; LSE[e, i] = ln sum_{j<=i} exp(scale S[i, j]). Pass 1 keeps a running
// (max, sum) per lane in base 2 and merges the lanes; pass 2 reads the row
// again (mostly from L2) and writes the whole row. VEC: T % 4 == 0, 16-byte
// accesses.
template <bool VEC>
__global__ void causal_softmax_kernel(float* __restrict__ s, float* __restrict__ lse, int64_t rows, int T,
                                      float scale) {
  const float c = scale * kLog2e;
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * int64_t(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    float* row = s + r * T;
    const int n = int(r % T) + 1;  // kept entries of this row
    float m = -INFINITY, l = 0.f;
    if constexpr (VEC) {
      for (int j = lane * 4; j < n; j += 128) {
        const float4 x = *reinterpret_cast<const float4*>(row + j);
        const float a0 = x.x * c;
        const float a1 = j + 1 < n ? x.y * c : -INFINITY;
        const float a2 = j + 2 < n ? x.z * c : -INFINITY;
        const float a3 = j + 3 < n ? x.w * c : -INFINITY;
        const float mn = fmaxf(m, fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)));
        l = l * ex2(m - mn) + ex2(a0 - mn) + ex2(a1 - mn) + ex2(a2 - mn) + ex2(a3 - mn);
        m = mn;
      }
    } else {
      for (int j = lane; j < n; j += 32) {
        const float a = row[j] * c;
        const float mn = fmaxf(m, a);
        l = l * ex2(m - mn) + ex2(a - mn);
        m = mn;
      }
    }
    // Merge the lanes (a lane that saw nothing has m = -inf, l = 0).
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float mo = __shfl_xor_sync(FULL, m, off), lo = __shfl_xor_sync(FULL, l, off);
      const float mn = fmaxf(m, mo);
      l = (m == -INFINITY ? 0.f : l * ex2(m - mn)) + (mo == -INFINITY ? 0.f : lo * ex2(mo - mn));
      m = mn;
    }
    const float inv = 1.f / l;
    if constexpr (VEC) {
      for (int j = lane * 4; j < T; j += 128) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < n) {
          const float4 y = *reinterpret_cast<const float4*>(row + j);
          x.x = ex2(y.x * c - m) * inv;
          x.y = j + 1 < n ? ex2(y.y * c - m) * inv : 0.f;
          x.z = j + 2 < n ? ex2(y.z * c - m) * inv : 0.f;
          x.w = j + 3 < n ? ex2(y.w * c - m) * inv : 0.f;
        }
        *reinterpret_cast<float4*>(row + j) = x;
      }
    } else {
      for (int j = lane; j < T; j += 32) row[j] = j < n ? ex2(row[j] * c - m) * inv : 0.f;
    }
    if (lane == 0) lse[r] = (m + __log2f(l)) * kLn2;
  }
}

// VJP of the fused causal softmax, in place on dP, one warp per row: with
// dPt = dP + dP_up, dS[i, j] = scale P[i, j] (dPt[i, j] - sum_k P[i, k] dPt[i, k])
// for j <= i, 0 above (the gradient with respect to the unscaled scores),
// written up to the end of row i's diagonal tile of `tile` columns (tile >= T:
// the whole row); dP and dP_up are read for j <= i only.
template <bool VEC>
__global__ void causal_softmax_bwd_kernel(const float* __restrict__ p, float* __restrict__ dp,
                                          const float* __restrict__ dp_up, int64_t rows, int T, int tile,
                                          float scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * int64_t(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const float* prow = p + r * T;
    float* drow = dp + r * T;
    const float* urow = dp_up ? dp_up + r * T : nullptr;
    const int n = int(r % T) + 1;
    // Columns written: the row's causal tiles of `tile` columns (the diagonal
    // one zero past n); tile >= T writes the whole row.
    const int wend = tile >= T ? T : min(T, ((n - 1) / tile + 1) * tile);
    float sum = 0.f;
    if constexpr (VEC) {
      for (int j = lane * 4; j < n; j += 128) {
        const float4 a = *reinterpret_cast<const float4*>(prow + j);  // P is 0 past n
        float4 d = *reinterpret_cast<const float4*>(drow + j);
        if (urow) {
          const float4 u = *reinterpret_cast<const float4*>(urow + j);
          d.x += u.x; d.y += u.y; d.z += u.z; d.w += u.w;
        }
        sum += a.x * d.x + (j + 1 < n ? a.y * d.y : 0.f) + (j + 2 < n ? a.z * d.z : 0.f) +
               (j + 3 < n ? a.w * d.w : 0.f);
      }
    } else {
      for (int j = lane; j < n; j += 32) sum += prow[j] * (drow[j] + (urow ? urow[j] : 0.f));
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(FULL, sum, off);
    if constexpr (VEC) {
      for (int j = lane * 4; j < wend; j += 128) {
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (j < n) {
          const float4 a = *reinterpret_cast<const float4*>(prow + j);
          float4 d = *reinterpret_cast<const float4*>(drow + j);
          if (urow) {
            const float4 u = *reinterpret_cast<const float4*>(urow + j);
            d.x += u.x; d.y += u.y; d.z += u.z; d.w += u.w;
          }
          x.x = scale * a.x * (d.x - sum);
          x.y = j + 1 < n ? scale * a.y * (d.y - sum) : 0.f;
          x.z = j + 2 < n ? scale * a.z * (d.z - sum) : 0.f;
          x.w = j + 3 < n ? scale * a.w * (d.w - sum) : 0.f;
        }
        *reinterpret_cast<float4*>(drow + j) = x;
      }
    } else {
      for (int j = lane; j < wend; j += 32)
        drow[j] = j < n ? scale * prow[j] * (drow[j] + (urow ? urow[j] : 0.f) - sum) : 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Row statistics of the two-pass forward, one warp per row (e, i): the
// (max, sum) pairs, in base 2, of the ngrp column groups of each of the row's
// tiles j <= i / 128 (a group wholly above the diagonal holds -inf) merged into
// LSE2 = m + log2 l (and lse = LSE2 ln 2 for the caller); then the row's
// columns past its diagonal tile, which no tile of the probabilities pass
// writes, are set to 0. VEC: T % 4 == 0, 16-byte stores.
template <bool VEC>
__global__ void probs_rows_kernel(const float2* __restrict__ part, float* __restrict__ lse2, float* __restrict__ lse,
                                  float* __restrict__ probs, int64_t rows, int T, int n_t, int ngrp) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * int64_t(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const int nt = int(r % T) / 128 + 1;  // tiles on or left of the diagonal
    const float2* pr = part + r * n_t * ngrp;
    float m = -INFINITY, l = 0.f;
    for (int j = lane; j < ngrp * nt; j += 32) {
      const float2 x = pr[j];
      if (x.x == -INFINITY) continue;
      const float mn = fmaxf(m, x.x);
      l = (m == -INFINITY ? 0.f : l * ex2(m - mn)) + x.y * ex2(x.x - mn);
      m = mn;
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float mo = __shfl_xor_sync(FULL, m, off), lo = __shfl_xor_sync(FULL, l, off);
      const float mn = fmaxf(m, mo);
      l = (m == -INFINITY ? 0.f : l * ex2(m - mn)) + (mo == -INFINITY ? 0.f : lo * ex2(mo - mn));
      m = mn;
    }
    if (lane == 0) {
      const float v = m + __log2f(l);
      lse2[r] = v;
      lse[r] = v * kLn2;
    }
    float* row = probs + r * T;
    if constexpr (VEC) {
      for (int j = nt * 128 + 4 * lane; j < T; j += 128)
        *reinterpret_cast<float4*>(row + j) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      for (int j = nt * 128 + lane; j < T; j += 32) row[j] = 0.f;
    }
  }
}

// Workspace: [dP (backward) | row statistics, LSE2 (forward) | fp32 storage:
// three bf16 parts each of Q, K, V, dO]
struct Layout {
  size_t dp, parts[4][3], stats, lse2, total;
};
enum { P_Q = 0, P_K = 1, P_V = 2, P_DO = 3 };

Layout layout(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, bool bf16) {
  Layout L{};
  const size_t E = size_t(B) * Hq;
  const size_t nq = size_t(B) * T * Hq * Dh, nkv = size_t(B) * T * Hkv * Dh;
  size_t at = 0;
  L.dp = at;
  at += round256(E * size_t(T) * T * 4);
  // Forward: row statistics per tile and column group [E, T, n_t, <= 4] (max,
  // sum) and the base-2 LSE [E, T].
  L.stats = at;
  at += round256(E * size_t(T) * size_t((T + 127) / 128) * 4 * 8);
  L.lse2 = at;
  at += round256(E * size_t(T) * 4);
  if (!bf16) {
    const size_t n[4] = {nq, nkv, nkv, nq};
    for (int t = 0; t < 4; ++t)
      for (int p = 0; p < 3; ++p) {
        L.parts[t][p] = at;
        at += round256(n[t] * 2);
      }
  }
  L.total = at;
  return L;
}

bool cuda_ok(cudaError_t e, const char* what, std::string& err) {
  if (e == cudaSuccess) return true;
  err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return false;
}

int grid_for(int64_t work, int per_block) {
  const int64_t g = (work + per_block - 1) / per_block;
  return int(g < 1 ? 1 : (g > 65535 * 8 ? 65535 * 8 : g));
}

int g_sms[256] = {};
std::mutex g_mu;

bool sm_count(int* out, std::string& err) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice", err)) return false;
  if (dev < 0 || dev >= 256) {
    err = "device ordinal out of range";
    return false;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] <= 0) {
    int n = 0;
    if (!cuda_ok(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev), "cudaDeviceGetAttribute", err))
      return false;
    g_sms[dev] = n;
  }
  *out = g_sms[dev];
  return true;
}

// Opt a kernel into its dynamic shared memory once per device.
template <typename K>
bool ensure_smem(K kernel, int bytes, std::atomic<unsigned long long>& mask, std::string& err) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice", err)) return false;
  const unsigned long long bit = 1ull << (dev & 63);
  if (mask.load(std::memory_order_acquire) & bit) return true;
  if (!cuda_ok(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes),
               "cudaFuncSetAttribute(materialized)", err))
    return false;
  mask.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

struct Ctx {
  const MatParams& p;
  cudaStream_t st;
  Layout L;
  int E, g, T, Dh, DHP;
  char* ws;
};

const void* part(const Ctx& c, int t, int k) { return c.ws + c.L.parts[t][k]; }

bool split3(const Ctx& c, const void* src, int t, int64_t n, std::string& err) {
  split3_kernel<<<grid_for(n / 4, 256), 256, 0, c.st>>>(
      static_cast<const float*>(src), reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.parts[t][0]),
      reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.parts[t][1]), reinterpret_cast<__nv_bfloat16*>(c.ws + c.L.parts[t][2]),
      n / 4);
  return cuda_ok(cudaGetLastError(), "launch split3_kernel", err);
}

// out[e] (tiles j <= i) = A_e B_e^T: a (tensor ia, query heads) against b
// (tensor ib, KV heads); bf16 storage reads the tensors themselves, fp32
// storage their three bf16 parts.
template <int NP, int DHP, int MODE>
bool launch_scores(const Ctx& c, const void* a_src, int ia, const void* b_src, int ib, float* out, float2* stats,
                   const float* lse2, float cexp, int* status, unsigned long long timeout_ns, std::string& err) {
  using C = ScoresCfg<NP, DHP>;
  const MatParams& p = c.p;
  ScoresMaps maps{};
  for (int k = 0; k < NP; ++k) {
    const void* av = NP == 1 ? a_src : part(c, ia, k);
    const void* bv = NP == 1 ? b_src : part(c, ib, k);
    if (!encode_rows_map(&maps.a[k], av, p.B, p.T, p.Hq, p.Dh, 128, err)) return false;
    if (!encode_rows_map(&maps.b[k], bv, p.B, p.T, p.Hkv, p.Dh, 128, err)) return false;
  }
  ScoresArgs a{};
  a.out = out;
  a.part = stats;
  a.lse2 = lse2;
  a.c = cexp;
  a.status = status;
  a.timeout_ns = timeout_ns;
  a.B = int(p.B); a.Hq = int(p.Hq); a.Hkv = int(p.Hkv); a.T = int(p.T);
  a.group = c.g;
  a.n_t = int((p.T + 127) / 128);
  a.n_tri = (long long)a.n_t * (a.n_t + 1) / 2;
  a.n_items = a.n_tri * c.E;
  int sms = 0;
  if (!sm_count(&sms, err)) return false;
  const unsigned grid = unsigned(a.n_items < sms ? a.n_items : sms);
  static std::atomic<unsigned long long> set[2] = {};
  if (p.T % 4 == 0) {
    auto k = mat_scores_kernel<NP, DHP, true, MODE>;
    if (!ensure_smem(k, C::SMEM_BYTES, set[0], err)) return false;
    k<<<grid, C::NTHREADS, C::SMEM_BYTES, c.st>>>(maps, a);
  } else {
    auto k = mat_scores_kernel<NP, DHP, false, MODE>;
    if (!ensure_smem(k, C::SMEM_BYTES, set[1], err)) return false;
    k<<<grid, C::NTHREADS, C::SMEM_BYTES, c.st>>>(maps, a);
  }
  return cuda_ok(cudaGetLastError(), "launch mat_scores_kernel", err);
}

// out = X Y over the kept triangle (rows) or X^T Y summed over each group
// (columns); Y is tensor iy (KV heads for rows, query heads for columns).
template <bool TRANS, int NPY, int DHP>
bool launch_reduce(const Ctx& c, const float* x, const void* y_src, int iy, void* out, int* status,
                   unsigned long long timeout_ns, std::string& err) {
  using C = ReduceCfg<TRANS, NPY, DHP>;
  const MatParams& p = c.p;
  ReduceMaps maps{};
  const int64_t H = TRANS ? p.Hq : p.Hkv;
  for (int k = 0; k < NPY; ++k) {
    const void* yv = NPY == 1 ? y_src : part(c, iy, k);
    if (!encode_rows_map(&maps.y[k], yv, p.B, p.T, H, p.Dh, 64, err)) return false;
  }
  if (NPY == 1) maps.y[1] = maps.y[0];
  ReduceArgs a{};
  a.x = x;
  a.out = out;
  a.status = status;
  a.timeout_ns = timeout_ns;
  a.B = int(p.B); a.Hq = int(p.Hq); a.Hkv = int(p.Hkv); a.T = int(p.T); a.Dh = int(p.Dh);
  a.group = c.g;
  a.n_t = int((p.T + 127) / 128);
  a.n_items = int((TRANS ? p.B * p.Hkv : p.B * p.Hq) * a.n_t);
  a.out_f32 = p.bf16 ? 0 : 1;
  int sms = 0;
  if (!sm_count(&sms, err)) return false;
  const unsigned grid = unsigned(a.n_items < sms ? a.n_items : sms);
  static std::atomic<unsigned long long> set = {};
  auto k = mat_reduce_kernel<TRANS, NPY, DHP>;
  if (!ensure_smem(k, C::SMEM_BYTES, set, err)) return false;
  k<<<grid, C::NTHREADS, C::SMEM_BYTES, c.st>>>(maps, a);
  return cuda_ok(cudaGetLastError(), "launch mat_reduce_kernel", err);
}

template <int MODE>
bool scores(const Ctx& c, const void* a_src, int ia, const void* b_src, int ib, float* out, float2* stats,
            const float* lse2, float cexp, std::string& err) {
  const MatParams& p = c.p;
  if (p.bf16)
    return c.DHP == 64
               ? launch_scores<1, 64, MODE>(c, a_src, ia, b_src, ib, out, stats, lse2, cexp, p.status, p.timeout_ns, err)
               : launch_scores<1, 128, MODE>(c, a_src, ia, b_src, ib, out, stats, lse2, cexp, p.status, p.timeout_ns,
                                             err);
  return c.DHP == 64
             ? launch_scores<3, 64, MODE>(c, a_src, ia, b_src, ib, out, stats, lse2, cexp, p.status, p.timeout_ns, err)
             : launch_scores<3, 128, MODE>(c, a_src, ia, b_src, ib, out, stats, lse2, cexp, p.status, p.timeout_ns, err);
}

bool launch_probs_rows(const Ctx& c, float* lse, float* probs, std::string& err) {
  const float2* stats = reinterpret_cast<const float2*>(c.ws + c.L.stats);
  float* lse2 = reinterpret_cast<float*>(c.ws + c.L.lse2);
  const int64_t rows = int64_t(c.E) * c.T;
  const int n_t = (c.T + 127) / 128;
  // Column groups per tile of the statistics pass (the scores kernel's epilogue layout).
  const int ngrp = c.p.bf16 ? ScoresCfg<1, 64>::NGRP : ScoresCfg<3, 64>::NGRP;
  static_assert(ScoresCfg<1, 64>::NGRP == ScoresCfg<1, 128>::NGRP && ScoresCfg<3, 64>::NGRP == ScoresCfg<3, 128>::NGRP &&
                    ScoresCfg<1, 64>::NGRP <= 4 && ScoresCfg<3, 64>::NGRP <= 4,
                "column groups per tile: as the workspace sizes them");
  if (c.T % 4 == 0)
    probs_rows_kernel<true><<<grid_for(rows, 8), 256, 0, c.st>>>(stats, lse2, lse, probs, rows, c.T, n_t, ngrp);
  else
    probs_rows_kernel<false><<<grid_for(rows, 8), 256, 0, c.st>>>(stats, lse2, lse, probs, rows, c.T, n_t, ngrp);
  return cuda_ok(cudaGetLastError(), "launch probs_rows_kernel", err);
}

template <bool TRANS>
bool reduce(const Ctx& c, const float* x, const void* y_src, int iy, void* out, std::string& err) {
  const MatParams& p = c.p;
  if (p.bf16)
    return c.DHP == 64 ? launch_reduce<TRANS, 1, 64>(c, x, y_src, iy, out, p.status, p.timeout_ns, err)
                       : launch_reduce<TRANS, 1, 128>(c, x, y_src, iy, out, p.status, p.timeout_ns, err);
  return c.DHP == 64 ? launch_reduce<TRANS, 2, 64>(c, x, y_src, iy, out, p.status, p.timeout_ns, err)
                     : launch_reduce<TRANS, 2, 128>(c, x, y_src, iy, out, p.status, p.timeout_ns, err);
}

bool launch_softmax(float* s, float* lse, int64_t rows, int T, float scale, cudaStream_t st, std::string& err) {
  if (T % 4 == 0)
    causal_softmax_kernel<true><<<grid_for(rows, 8), 256, 0, st>>>(s, lse, rows, T, scale);
  else
    causal_softmax_kernel<false><<<grid_for(rows, 8), 256, 0, st>>>(s, lse, rows, T, scale);
  return cuda_ok(cudaGetLastError(), "launch causal_softmax_kernel", err);
}

bool launch_softmax_bwd(const float* p, float* dp, const float* dp_up, int64_t rows, int T, int tile, float scale,
                        cudaStream_t st, std::string& err) {
  // The vector form writes 4 columns at a time: T and the tile width multiples of 4.
  if (T % 4 == 0 && (tile >= T || tile % 4 == 0))
    causal_softmax_bwd_kernel<true><<<grid_for(rows, 8), 256, 0, st>>>(p, dp, dp_up, rows, T, tile, scale);
  else
    causal_softmax_bwd_kernel<false><<<grid_for(rows, 8), 256, 0, st>>>(p, dp, dp_up, rows, T, tile, scale);
  return cuda_ok(cudaGetLastError(), "launch causal_softmax_bwd_kernel", err);
}

Ctx make_ctx(const MatParams& p, cudaStream_t st) {
  return Ctx{p, st, layout(p.B, p.Hq, p.Hkv, p.T, p.Dh, p.bf16), int(p.B * p.Hq), int(p.Hq / p.Hkv), int(p.T),
             int(p.Dh), p.Dh > 64 ? 128 : 64, static_cast<char*>(p.workspace)};
}

}  // namespace mat

bool causal_softmax_fwd(float* scores, float* lse, int64_t N, int64_t T, float scale, cudaStream_t st,
                        std::string& err) {
  return mat::launch_softmax(scores, lse, N * T, int(T), scale, st, err);
}

bool causal_softmax_bwd(const float* probs, float* grad, const float* grad_extra, int64_t N, int64_t T, int64_t tile,
                        float scale, cudaStream_t st, std::string& err) {
  return mat::launch_softmax_bwd(probs, grad, grad_extra, N * T, int(T), int(tile < T ? tile : T), scale, st, err);
}

size_t materialized_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, bool bf16) {
  return mat::layout(B, Hq, Hkv, T, Dh, bf16).total;
}

bool materialized_fwd(const MatParams& p, cudaStream_t st, std::string& err) {
  using namespace mat;
  const Ctx c = make_ctx(p, st);
  const int64_t nkv = p.B * p.T * p.Hkv * p.Dh, nq = p.B * p.T * p.Hq * p.Dh;
  if (!p.bf16) {
    if (!split3(c, p.q, P_Q, nq, err) || !split3(c, p.k, P_K, nkv, err) || !split3(c, p.v, P_V, nkv, err))
      return false;
  }
  const float scale = float(1.0 / __builtin_sqrt(double(p.Dh)));
  const float cexp = float(double(scale) * 1.4426950408889634);  // scores in base 2
  // Two passes over S = Q K^T (kept tiles), which the tensor cores recompute
  // instead of storing: (1) per-tile row statistics; then each row's LSE and
  // the zero columns past its diagonal tile; (2) P = 2^(c S - LSE2) written
  // into the kept tiles. The probabilities are written once and never read
  // back before O = P V.
  float2* stats = reinterpret_cast<float2*>(c.ws + c.L.stats);
  const float* lse2 = reinterpret_cast<const float*>(c.ws + c.L.lse2);
  if (!scores<kScoresStats>(c, p.q, P_Q, p.k, P_K, nullptr, stats, nullptr, cexp, err)) return false;
  if (!launch_probs_rows(c, p.lse, p.probs, err)) return false;
  if (!scores<kScoresProbs>(c, p.q, P_Q, p.k, P_K, p.probs, nullptr, lse2, cexp, err)) return false;
  // O = P V.
  return reduce<false>(c, p.probs, p.v, P_V, p.out, err);
}

bool materialized_bwd(const MatParams& p, cudaStream_t st, std::string& err) {
  using namespace mat;
  const Ctx c = make_ctx(p, st);
  const int64_t nkv = p.B * p.T * p.Hkv * p.Dh, nq = p.B * p.T * p.Hq * p.Dh;
  if (!p.bf16) {
    if (!split3(c, p.q, P_Q, nq, err) || !split3(c, p.k, P_K, nkv, err) || !split3(c, p.v, P_V, nkv, err) ||
        !split3(c, p.dout, P_DO, nq, err))
      return false;
  }
  const float scale = float(1.0 / __builtin_sqrt(double(p.Dh)));
  float* dp = reinterpret_cast<float*>(c.ws + c.L.dp);
  // dP = dO V^T (kept tiles), then dS (with respect to the unscaled scores) in place.
  if (!scores<kScoresRaw>(c, p.dout, P_DO, p.v, P_V, dp, nullptr, nullptr, 0.f, err)) return false;
  // dS only where the products read it: each row's causal 128-column tiles.
  if (!launch_softmax_bwd(p.probs, dp, p.dprobs, int64_t(c.E) * c.T, c.T, 128, scale, st, err)) return false;
  // dQ = dS K;  dK = dS^T Q;  dV = P^T dO  (the last two summed over each group).
  if (!reduce<false>(c, dp, p.k, P_K, p.dq, err)) return false;
  if (!reduce<true>(c, dp, p.q, P_Q, p.dk, err)) return false;
  return reduce<true>(c, p.probs, p.dout, P_DO, p.dv, err);
}

}  // namespace rca
