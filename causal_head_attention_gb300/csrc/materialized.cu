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
// The five products are plain batched GEMMs and run in cuBLAS, one batch
// entry per (b, h) with pointer arrays built on the device: the two that
// contract over Dh (Q K^T, dO V^T) read the stored operands directly (bf16
// tensor cores with fp32 accumulation, or fp32), the three that contract over
// the T positions take fp32 P or dS and run in full fp32. The fused causal
// softmax and its VJP are the kernels written here (one warp per row, bound by
// HBM traffic of the [T, T] rows), with small conversion and group-sum
// kernels around the GEMMs. The full T x T rows are computed (the masked half
// included): this path exists for the probabilities and as an independent
// check of the memory-linear kernels, not for speed.
#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdio>
#include <mutex>

#include "materialized.h"
#include "tc.cuh"

namespace rca {
namespace mat {

constexpr unsigned FULL = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// Pointer arrays of the batched GEMMs: entry e = b * Hq + h of array a is
// base[a] + b * bstride[a] + (h, or its KV head) * hstride[a] bytes.
enum Arr { A_Q, A_K, A_V, A_DO, A_QF, A_KF, A_VF, A_DOF, A_P, A_DP, A_OF, A_DQF, A_DKH, A_DVH, NARR };
struct PtrBuild {
  const char* base[NARR];
  int64_t bstride[NARR];
  int64_t hstride[NARR];
  int kv[NARR];
};

__global__ void build_ptrs_kernel(PtrBuild pb, void** out, int E, int Hq, int g) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int b = e / Hq, h = e - b * Hq;
  for (int a = 0; a < NARR; ++a) {
    const int hh = pb.kv[a] ? h / g : h;
    out[int64_t(a) * E + e] =
        pb.base[a] ? const_cast<char*>(pb.base[a] + b * pb.bstride[a] + hh * pb.hstride[a]) : nullptr;
  }
}

// bf16 -> fp32, 8 elements a thread (n is a multiple of 8).
__global__ void to_f32_kernel(const __nv_bfloat16* __restrict__ src, float* __restrict__ dst, int64_t n8) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n8; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 w = reinterpret_cast<const uint4*>(src)[i];
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    float4 lo, hi;
    lo.x = __uint_as_float(u[0] << 16); lo.y = __uint_as_float(u[0] & 0xffff0000u);
    lo.z = __uint_as_float(u[1] << 16); lo.w = __uint_as_float(u[1] & 0xffff0000u);
    hi.x = __uint_as_float(u[2] << 16); hi.y = __uint_as_float(u[2] & 0xffff0000u);
    hi.z = __uint_as_float(u[3] << 16); hi.w = __uint_as_float(u[3] & 0xffff0000u);
    reinterpret_cast<float4*>(dst)[2 * i] = lo;
    reinterpret_cast<float4*>(dst)[2 * i + 1] = hi;
  }
}

// fp32 -> bf16 (round to nearest even), 4 elements a thread (n a multiple of 4).
__global__ void to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n4) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
    const float4 f = reinterpret_cast<const float4*>(src)[i];
    uint2 w;
    w.x = pack_bf16(f.x, f.y);
    w.y = pack_bf16(f.z, f.w);
    reinterpret_cast<uint2*>(dst)[i] = w;
  }
}

// dst[b, t, kv, d] = sum over the g query heads of the group of src[b, h, t, d]
// (src per query head [B, Hq, T, Dh] fp32; dst in the storage dtype).
template <bool BF16>
__global__ void group_sum_kernel(const float* __restrict__ src, void* __restrict__ dst, int B, int T, int Hq,
                                 int Hkv, int Dh) {
  const int g = Hq / Hkv;
  const int64_t n4 = int64_t(B) * T * Hkv * Dh / 4;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t o = i * 4;  // element index in [B, T, Hkv, Dh]
    const int d = int(o % Dh);
    const int kv = int((o / Dh) % Hkv);
    const int64_t bt = o / (int64_t(Dh) * Hkv);
    const int t = int(bt % T), b = int(bt / T);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < g; ++r) {
      const float4 x = *reinterpret_cast<const float4*>(src + ((int64_t(b) * Hq + kv * g + r) * T + t) * Dh + d);
      s.x += x.x; s.y += x.y; s.z += x.z; s.w += x.w;
    }
    if constexpr (BF16) {
      uint2 w;
      w.x = pack_bf16(s.x, s.y);
      w.y = pack_bf16(s.z, s.w);
      reinterpret_cast<uint2*>(dst)[i] = w;
    } else {
      reinterpret_cast<float4*>(dst)[i] = s;
    }
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
// for j <= i, 0 above (the gradient with respect to the unscaled scores).
template <bool VEC>
__global__ void causal_softmax_bwd_kernel(const float* __restrict__ p, float* __restrict__ dp,
                                          const float* __restrict__ dp_up, int64_t rows, int T, float scale) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = blockIdx.x * int64_t(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const float* prow = p + r * T;
    float* drow = dp + r * T;
    const float* urow = dp_up ? dp_up + r * T : nullptr;
    const int n = int(r % T) + 1;
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
      for (int j = lane * 4; j < T; j += 128) {
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
      for (int j = lane; j < T; j += 32)
        drow[j] = j < n ? scale * prow[j] * (drow[j] + (urow ? urow[j] : 0.f) - sum) : 0.f;
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

struct Layout {
  size_t ptrs, qf, kf, vf, dof, of, dp, dqf, dkh, dvh, total;
};

// [ptr arrays | Qf Kf Vf dOf Of (bf16 only) | dP | dQf (bf16 only) | dKh | dVh]
Layout layout(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, bool bf16) {
  Layout L{};
  const size_t E = size_t(B) * Hq;
  const size_t nq = size_t(B) * T * Hq * Dh, nkv = size_t(B) * T * Hkv * Dh;
  size_t at = 0;
  L.ptrs = at;
  at += round256(NARR * E * sizeof(void*));
  auto take = [&](size_t bytes) {
    const size_t o = at;
    at += round256(bytes);
    return o;
  };
  L.qf = bf16 ? take(nq * 4) : 0;
  L.kf = bf16 ? take(nkv * 4) : 0;
  L.vf = bf16 ? take(nkv * 4) : 0;
  L.dof = bf16 ? take(nq * 4) : 0;
  L.of = bf16 ? take(nq * 4) : 0;
  L.dp = take(E * size_t(T) * T * 4);
  L.dqf = bf16 ? take(nq * 4) : 0;
  L.dkh = take(E * size_t(T) * Dh * 4);
  L.dvh = take(E * size_t(T) * Dh * 4);
  L.total = at;
  return L;
}

std::mutex g_cublas_mu;
cublasHandle_t g_cublas[256] = {};

bool cuda_ok(cudaError_t e, const char* what, std::string& err) {
  if (e == cudaSuccess) return true;
  err = std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")";
  return false;
}

bool cublas_ok(cublasStatus_t s, const char* what, std::string& err) {
  if (s == CUBLAS_STATUS_SUCCESS) return true;
  char buf[160];
  snprintf(buf, sizeof(buf), "%s: cuBLAS status %d", what, int(s));
  err = buf;
  return false;
}

// One cuBLAS handle per device, used under g_cublas_mu (the stream is set per call).
bool handle_for_device(cublasHandle_t* h, std::string& err) {
  int dev = 0;
  if (!cuda_ok(cudaGetDevice(&dev), "cudaGetDevice", err)) return false;
  if (dev < 0 || dev >= 256) {
    err = "device ordinal out of range";
    return false;
  }
  if (!g_cublas[dev]) {
    if (!cublas_ok(cublasCreate(&g_cublas[dev]), "cublasCreate", err)) return false;
    if (!cublas_ok(cublasSetMathMode(g_cublas[dev], CUBLAS_DEFAULT_MATH), "cublasSetMathMode", err)) return false;
  }
  *h = g_cublas[dev];
  return true;
}

struct Ctx {
  const MatParams& p;
  cudaStream_t st;
  Layout L;
  int E, g, T, Dh;
  void** arr;  // device pointer arrays, NARR x E
  cudaDataType_t st_type;
  size_t es;
};

void** arr_of(const Ctx& c, Arr a) { return c.arr + size_t(a) * c.E; }

// Row-major X[r][c] with leading dimension ld is the column-major X^T: every
// product below is written for the column-major views.
bool gemm(cublasHandle_t h, const Ctx& c, cublasOperation_t ta, cublasOperation_t tb, int m, int n, int k,
          float alpha, Arr a, cudaDataType_t at, int lda, Arr b, cudaDataType_t bt, int ldb, Arr cc, int ldc,
          const char* what, std::string& err) {
  const float beta = 0.f;
  return cublas_ok(cublasGemmBatchedEx(h, ta, tb, m, n, k, &alpha, const_cast<const void* const*>(arr_of(c, a)),
                                       at, lda, const_cast<const void* const*>(arr_of(c, b)), bt, ldb, &beta,
                                       arr_of(c, cc), CUDA_R_32F, ldc, c.E, CUBLAS_COMPUTE_32F,
                                       CUBLAS_GEMM_DEFAULT),
                   what, err);
}

int grid_for(int64_t work, int per_block) {
  const int64_t g = (work + per_block - 1) / per_block;
  return int(g < 1 ? 1 : (g > 65535 * 8 ? 65535 * 8 : g));
}

bool build(Ctx& c, std::string& err) {
  const MatParams& p = c.p;
  char* ws = static_cast<char*>(p.workspace);
  const int64_t es = int64_t(c.es);
  const int64_t Hq = p.Hq, Hkv = p.Hkv, T = p.T, Dh = p.Dh;
  PtrBuild pb{};
  auto set = [&](Arr a, const void* base, int64_t bstride, int64_t hstride, bool kv) {
    pb.base[a] = static_cast<const char*>(base);
    pb.bstride[a] = bstride;
    pb.hstride[a] = hstride;
    pb.kv[a] = kv ? 1 : 0;
  };
  const int64_t qb = T * Hq * Dh, kb = T * Hkv * Dh;  // elements per batch index
  set(A_Q, p.q, qb * es, Dh * es, false);
  set(A_K, p.k, kb * es, Dh * es, true);
  set(A_V, p.v, kb * es, Dh * es, true);
  set(A_DO, p.dout, qb * es, Dh * es, false);
  // fp32 operands: copies for bf16 storage, the caller's tensors for fp32.
  set(A_QF, p.bf16 ? ws + c.L.qf : p.q, qb * 4, Dh * 4, false);
  set(A_KF, p.bf16 ? ws + c.L.kf : p.k, kb * 4, Dh * 4, true);
  set(A_VF, p.bf16 ? ws + c.L.vf : p.v, kb * 4, Dh * 4, true);
  set(A_DOF, p.bf16 ? ws + c.L.dof : p.dout, qb * 4, Dh * 4, false);
  set(A_P, p.probs, Hq * T * T * 4, T * T * 4, false);
  set(A_DP, ws + c.L.dp, Hq * T * T * 4, T * T * 4, false);
  set(A_OF, p.bf16 ? ws + c.L.of : p.out, qb * 4, Dh * 4, false);
  set(A_DQF, p.bf16 ? ws + c.L.dqf : p.dq, qb * 4, Dh * 4, false);
  set(A_DKH, ws + c.L.dkh, Hq * T * Dh * 4, T * Dh * 4, false);
  set(A_DVH, ws + c.L.dvh, Hq * T * Dh * 4, T * Dh * 4, false);
  build_ptrs_kernel<<<(c.E + 127) / 128, 128, 0, c.st>>>(pb, c.arr, c.E, int(Hq), c.g);
  return cuda_ok(cudaGetLastError(), "launch build_ptrs_kernel", err);
}

bool convert(const void* src, size_t off, int64_t n, const Ctx& c, std::string& err) {
  float* dst = reinterpret_cast<float*>(static_cast<char*>(c.p.workspace) + off);
  to_f32_kernel<<<grid_for(n / 8, 256), 256, 0, c.st>>>(static_cast<const __nv_bfloat16*>(src), dst, n / 8);
  return cuda_ok(cudaGetLastError(), "launch to_f32_kernel", err);
}

bool launch_softmax(float* s, float* lse, int64_t rows, int T, float scale, cudaStream_t st, std::string& err) {
  if (T % 4 == 0)
    causal_softmax_kernel<true><<<grid_for(rows, 8), 256, 0, st>>>(s, lse, rows, T, scale);
  else
    causal_softmax_kernel<false><<<grid_for(rows, 8), 256, 0, st>>>(s, lse, rows, T, scale);
  return cuda_ok(cudaGetLastError(), "launch causal_softmax_kernel", err);
}

bool launch_softmax_bwd(const float* p, float* dp, const float* dp_up, int64_t rows, int T, float scale,
                        cudaStream_t st, std::string& err) {
  if (T % 4 == 0)
    causal_softmax_bwd_kernel<true><<<grid_for(rows, 8), 256, 0, st>>>(p, dp, dp_up, rows, T, scale);
  else
    causal_softmax_bwd_kernel<false><<<grid_for(rows, 8), 256, 0, st>>>(p, dp, dp_up, rows, T, scale);
  return cuda_ok(cudaGetLastError(), "launch causal_softmax_bwd_kernel", err);
}

}  // namespace mat

bool causal_softmax_fwd(float* scores, float* lse, int64_t N, int64_t T, float scale, cudaStream_t st,
                        std::string& err) {
  return mat::launch_softmax(scores, lse, N * T, int(T), scale, st, err);
}

bool causal_softmax_bwd(const float* probs, float* grad, const float* grad_extra, int64_t N, int64_t T, float scale,
                        cudaStream_t st, std::string& err) {
  return mat::launch_softmax_bwd(probs, grad, grad_extra, N * T, int(T), scale, st, err);
}

size_t materialized_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, bool bf16) {
  return mat::layout(B, Hq, Hkv, T, Dh, bf16).total;
}

bool materialized_fwd(const MatParams& p, cudaStream_t st, std::string& err) {
  using namespace mat;
  Ctx c{p, st, layout(p.B, p.Hq, p.Hkv, p.T, p.Dh, p.bf16), int(p.B * p.Hq), int(p.Hq / p.Hkv), int(p.T),
        int(p.Dh), nullptr, p.bf16 ? CUDA_R_16BF : CUDA_R_32F, size_t(p.bf16 ? 2 : 4)};
  c.arr = reinterpret_cast<void**>(static_cast<char*>(p.workspace) + c.L.ptrs);
  if (!build(c, err)) return false;
  const int64_t nkv = p.B * p.T * p.Hkv * p.Dh, nq = p.B * p.T * p.Hq * p.Dh;
  if (p.bf16 && !convert(p.v, c.L.vf, nkv, c, err)) return false;
  const int T = c.T, Dh = c.Dh, ldq = int(p.Hq * p.Dh), ldk = int(p.Hkv * p.Dh);
  const float scale = float(1.0 / __builtin_sqrt(double(p.Dh)));
  std::lock_guard<std::mutex> lk(g_cublas_mu);
  cublasHandle_t h;
  if (!handle_for_device(&h, err)) return false;
  if (!cublas_ok(cublasSetStream(h, st), "cublasSetStream", err)) return false;
  // S^T (col-major, = row-major S) = K Q^T: m = n = T, k = Dh.
  if (!gemm(h, c, CUBLAS_OP_T, CUBLAS_OP_N, T, T, Dh, 1.f, A_K, c.st_type, ldk, A_Q, c.st_type, ldq, A_P, T,
            "GEMM S = Q K^T", err))
    return false;
  if (!launch_softmax(p.probs, p.lse, int64_t(c.E) * T, T, scale, st, err)) return false;
  // O^T (col-major view of row-major O) = V^T P^T: m = Dh, n = T, k = T.
  if (!gemm(h, c, CUBLAS_OP_N, CUBLAS_OP_N, Dh, T, T, 1.f, A_VF, CUDA_R_32F, ldk, A_P, CUDA_R_32F, T, A_OF, ldq,
            "GEMM O = P V", err))
    return false;
  if (p.bf16) {
    to_bf16_kernel<<<grid_for(nq / 4, 256), 256, 0, st>>>(
        reinterpret_cast<const float*>(static_cast<char*>(p.workspace) + c.L.of), static_cast<__nv_bfloat16*>(p.out),
        nq / 4);
    if (!cuda_ok(cudaGetLastError(), "launch to_bf16_kernel", err)) return false;
  }
  return true;
}

bool materialized_bwd(const MatParams& p, cudaStream_t st, std::string& err) {
  using namespace mat;
  Ctx c{p, st, layout(p.B, p.Hq, p.Hkv, p.T, p.Dh, p.bf16), int(p.B * p.Hq), int(p.Hq / p.Hkv), int(p.T),
        int(p.Dh), nullptr, p.bf16 ? CUDA_R_16BF : CUDA_R_32F, size_t(p.bf16 ? 2 : 4)};
  c.arr = reinterpret_cast<void**>(static_cast<char*>(p.workspace) + c.L.ptrs);
  if (!build(c, err)) return false;
  const int64_t nkv = p.B * p.T * p.Hkv * p.Dh, nq = p.B * p.T * p.Hq * p.Dh;
  if (p.bf16) {
    if (!convert(p.q, c.L.qf, nq, c, err) || !convert(p.k, c.L.kf, nkv, c, err) ||
        !convert(p.dout, c.L.dof, nq, c, err))
      return false;
  }
  const int T = c.T, Dh = c.Dh, ldq = int(p.Hq * p.Dh), ldk = int(p.Hkv * p.Dh);
  const float scale = float(1.0 / __builtin_sqrt(double(p.Dh)));
  float* dp = reinterpret_cast<float*>(static_cast<char*>(p.workspace) + c.L.dp);
  std::lock_guard<std::mutex> lk(g_cublas_mu);
  cublasHandle_t h;
  if (!handle_for_device(&h, err)) return false;
  if (!cublas_ok(cublasSetStream(h, st), "cublasSetStream", err)) return false;
  // dP^T (col-major) = V dO^T: m = n = T, k = Dh.
  if (!gemm(h, c, CUBLAS_OP_T, CUBLAS_OP_N, T, T, Dh, 1.f, A_V, c.st_type, ldk, A_DO, c.st_type, ldq, A_DP, T,
            "GEMM dP = dO V^T", err))
    return false;
  // dS (with respect to the unscaled scores, so the scale is inside).
  if (!launch_softmax_bwd(p.probs, dp, p.dprobs, int64_t(c.E) * T, T, scale, st, err)) return false;
  // dQ^T = K^T dS^T: m = Dh, n = T, k = T.
  if (!gemm(h, c, CUBLAS_OP_N, CUBLAS_OP_N, Dh, T, T, 1.f, A_KF, CUDA_R_32F, ldk, A_DP, CUDA_R_32F, T, A_DQF, ldq,
            "GEMM dQ = dS K", err))
    return false;
  // dK^T (per query head) = Q^T dS: m = Dh, n = T, k = T.
  if (!gemm(h, c, CUBLAS_OP_N, CUBLAS_OP_T, Dh, T, T, 1.f, A_QF, CUDA_R_32F, ldq, A_DP, CUDA_R_32F, T, A_DKH, Dh,
            "GEMM dK = dS^T Q", err))
    return false;
  // dV^T (per query head) = dO^T P: m = Dh, n = T, k = T.
  if (!gemm(h, c, CUBLAS_OP_N, CUBLAS_OP_T, Dh, T, T, 1.f, A_DOF, CUDA_R_32F, ldq, A_P, CUDA_R_32F, T, A_DVH, Dh,
            "GEMM dV = P^T dO", err))
    return false;
  const float* dkh = reinterpret_cast<const float*>(static_cast<char*>(p.workspace) + c.L.dkh);
  const float* dvh = reinterpret_cast<const float*>(static_cast<char*>(p.workspace) + c.L.dvh);
  const int gs = grid_for(nkv / 4, 256);
  if (p.bf16) {
    group_sum_kernel<true><<<gs, 256, 0, st>>>(dkh, p.dk, int(p.B), T, int(p.Hq), int(p.Hkv), Dh);
    group_sum_kernel<true><<<gs, 256, 0, st>>>(dvh, p.dv, int(p.B), T, int(p.Hq), int(p.Hkv), Dh);
    to_bf16_kernel<<<grid_for(nq / 4, 256), 256, 0, st>>>(
        reinterpret_cast<const float*>(static_cast<char*>(p.workspace) + c.L.dqf), static_cast<__nv_bfloat16*>(p.dq),
        nq / 4);
  } else {
    group_sum_kernel<false><<<gs, 256, 0, st>>>(dkh, p.dk, int(p.B), T, int(p.Hq), int(p.Hkv), Dh);
    group_sum_kernel<false><<<gs, 256, 0, st>>>(dvh, p.dv, int(p.B), T, int(p.Hq), int(p.Hkv), Dh);
  }
  return cuda_ok(cudaGetLastError(), "launch group_sum / to_bf16 kernels", err);
}

}  // namespace rca
