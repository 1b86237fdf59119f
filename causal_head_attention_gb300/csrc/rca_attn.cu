// C ABI of librca_attn.so: argument validation, TMA descriptor encoding and
// kernel launches on the caller's stream. See include/rca_attn.h for the
// contract (layouts, ownership, errors).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>
#include <utility>

#include "rca_attn.h"
#include "bwd.cuh"
#include "bwd_sub.cuh"
#include "decode.h"
#include "fwd.cuh"
#include "materialized.h"
#include "varlen.cuh"

namespace rca {
// Failure-detection self-test: one warp waits, with the same time-bounded wait
// the attention kernels use, on an mbarrier that nothing ever arrives on. The
// wait gives up after the configured limit, records the timeout status and the
// kernel returns; the CUDA context stays usable.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) unsigned long long bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    mbar_init_fence();
  }
  __syncwarp();
  const WaitCtl w{status, &abort_flag, timeout_ns};
  mbar_wait_warp(smem_u32(&bar), 0, w);
}
}  // namespace rca

namespace {

thread_local std::string g_err;

rca_status fail(rca_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

rca_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RCA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

std::atomic<unsigned long long> g_timeout_ns{2000000000ull};

// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// ---------------------------------------------------------------------------
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);
EncodeFn g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

EncodeFn get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                    cudaEnableDefault, &q);
    if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeFn>(fn);
  });
  return g_encode;
}

// [B, T, H, Dh] row-major tensor, tiles of 128 rows (positions) x one 128-byte
// panel of the head dimension, 128-byte swizzle. Positions past T and head
// columns past Dh read as zero.
rca_status make_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t H, int64_t Dh,
                    bool f32, const char* name, unsigned box_rows = 128, int64_t row_stride = 0) {
  // (row_stride: elements between consecutive positions of one head; 0 means
  // H * Dh, a contiguous [B, T, H, Dh] tensor. A fused QKV buffer has a larger one.)
  if (row_stride == 0) row_stride = H * Dh;
  // (f32 selects fp32 elements with 32-element panels; bf16 uses 64-element panels;
  // a box covers box_rows positions of one head)
  EncodeFn enc = get_encode();
  if (!enc) return fail(RCA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (%s)", cudaGetErrorName(g_encode_err));
  const uint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(Dh), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(Dh * es), static_cast<cuuint64_t>(row_stride * es),
                           static_cast<cuuint64_t>(T * row_stride * es)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / es), 1, box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(RCA_ERR_CUDA, "cuTensorMapEncodeTiled(%s) failed with CUresult %d", name, (int)r);
  return RCA_OK;
}

}  // namespace

namespace rca {
bool encode_rows_map(CUtensorMap* m, const void* ptr, int64_t B, int64_t T, int64_t H, int64_t Dh,
                     unsigned box_rows, std::string& err) {
  if (make_map(m, ptr, B, T, H, Dh, false, "materialized operand", box_rows) != RCA_OK) {
    err = g_err;
    return false;
  }
  return true;
}
}  // namespace rca

namespace {

// ---------------------------------------------------------------------------
// Per-device status word (device timeouts), allocated on first use.
// ---------------------------------------------------------------------------
std::mutex g_status_mu;
int* g_status[256] = {};

rca_status status_word(int** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 256) return fail(RCA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status[dev]) {
    int* p = nullptr;
    e = cudaMalloc(&p, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(status word)");
    e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status word)");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    g_status[dev] = p;
  }
  *out = g_status[dev];
  return RCA_OK;
}

// Reads and clears the allocation-free backward's device status word on the
// current device (0 when that entry point was never set up there). Defined
// with the built-in scratch region at the end of this file.
rca_status noalloc_take_status(int* out);

// Streaming-multiprocessor count of the current device (cached per device).
int g_sms[256] = {};
rca_status sm_count(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 256) return fail(RCA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (g_sms[dev] <= 0) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiProcessorCount)");
    if (n <= 0) return fail(RCA_ERR_CUDA, "device reports %d multiprocessors", n);
    g_sms[dev] = n;
  }
  *out = g_sms[dev];
  return RCA_OK;
}

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the kernel before it in the stream is still finishing, which
// hides most of the gap between the kernels of a training step (~4 us each
// otherwise). Every kernel launched this way calls rca::grid_dep_sync() before
// it touches global memory, so it still sees everything earlier in the
// stream. A failed launch is reported through cudaGetLastError() like a
// <<<>>> launch.
template <typename... KA, typename... A>
void launch_dep(void (*kern)(KA...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, A&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  (void)cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

template <typename K>
cudaError_t ensure_smem(K kernel, int bytes, std::atomic<unsigned long long>& mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = 1ull << (dev & 63);
  if (mask.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// ---------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rca_status check_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt) {
  if (B < 1 || Hq < 1 || Hkv < 1)
    return fail(RCA_ERR_INVALID_ARGUMENT, "B, Hq and Hkv must be >= 1 (got B=%lld Hq=%lld Hkv=%lld)",
                (long long)B, (long long)Hq, (long long)Hkv);
  if (T < 1)
    return fail(RCA_ERR_INVALID_ARGUMENT,
                "T must be >= 1 (got %lld): an empty causal row is a fully masked softmax slice",
                (long long)T);
  if (Hq % Hkv != 0)
    return fail(RCA_ERR_INVALID_ARGUMENT, "grouped-query attention needs Hq %% Hkv == 0 (Hq=%lld Hkv=%lld)",
                (long long)Hq, (long long)Hkv);
  if (dt != RCA_BF16 && dt != RCA_F32_TF32)
    return fail(RCA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dt);
  const bool ok_dh = Dh == 16 || Dh == 32 || Dh == 64 || (Dh == 128 && dt == RCA_BF16);
  if (!ok_dh)
    return fail(RCA_ERR_UNSUPPORTED,
                "head width Dh=%lld is not supported for %s (supported: 16, 32, 64%s)", (long long)Dh,
                dt == RCA_BF16 ? "bf16" : "fp32/tf32", dt == RCA_BF16 ? ", 128" : "");
  const int64_t n_t = (T + 127) / 128;
  if (T > (int64_t(1) << 30) || B * Hq * n_t > 0x7fffffffLL || B * T * Hq * Dh > (int64_t(1) << 38))
    return fail(RCA_ERR_INVALID_ARGUMENT, "problem too large (B=%lld T=%lld Hq=%lld Dh=%lld)",
                (long long)B, (long long)T, (long long)Hq, (long long)Dh);
  return RCA_OK;
}

struct WsLayout {
  size_t dq_off, lse2_off, d_off, hl_off, total;
  size_t q_part, kv_part;  // bytes of one bf16 part of Q/dO and of K/V (fp32 storage only)
  int64_t Tpad;
};

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// fp32 accumulator for dQ [B,T,Hq,Dh]; base-2 LSE and D rows [B,Hq,Tpad]; and,
// for fp32 storage, bf16 hi/lo copies of Q, dO [B,T,Hq,Dh] and K, V [B,T,Hkv,Dh].
WsLayout ws_layout(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt) {
  WsLayout w{};
  w.Tpad = (T + 127) / 128 * 128;
  w.dq_off = 0;
  w.lse2_off = round256(size_t(B) * T * Hq * Dh * 4);
  w.d_off = w.lse2_off + round256(size_t(B) * Hq * w.Tpad * 4);
  w.hl_off = w.d_off + round256(size_t(B) * Hq * w.Tpad * 4);
  w.total = w.hl_off;
  if (dt == RCA_F32_TF32) {
    w.q_part = round256(size_t(B) * T * Hq * Dh * 2);
    w.kv_part = round256(size_t(B) * T * Hkv * Dh * 2);
    w.total += 4 * w.q_part + 4 * w.kv_part;  // Qhi, Qlo, dOhi, dOlo, Khi, Klo, Vhi, Vlo
  }
  return w;
}

rca_status check_ws(const void* ws, size_t bytes, const WsLayout& L) {
  if (!ws) return fail(RCA_ERR_INVALID_ARGUMENT, "workspace is null");
  if (reinterpret_cast<uintptr_t>(ws) & 255u)
    return fail(RCA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (bytes < L.total)
    return fail(RCA_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", bytes, L.total);
  return RCA_OK;
}

rca_status check_decode_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t Dh, int64_t page_size,
                              int64_t max_pages, int64_t num_pages, rca_dtype dt) {
  if (B < 1 || Hq < 1 || Hkv < 1 || max_pages < 1 || num_pages < 1)
    return fail(RCA_ERR_INVALID_ARGUMENT,
                "B, Hq, Hkv, max_pages and num_pages must be >= 1 (got B=%lld Hq=%lld Hkv=%lld max_pages=%lld "
                "num_pages=%lld)",
                (long long)B, (long long)Hq, (long long)Hkv, (long long)max_pages, (long long)num_pages);
  if (Hq % Hkv != 0)
    return fail(RCA_ERR_INVALID_ARGUMENT, "grouped-query attention needs Hq %% Hkv == 0 (Hq=%lld Hkv=%lld)",
                (long long)Hq, (long long)Hkv);
  if (dt != RCA_BF16 && dt != RCA_F32_TF32) return fail(RCA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dt);
  if (Dh != 16 && Dh != 32 && Dh != 64 && Dh != 128)
    return fail(RCA_ERR_UNSUPPORTED, "head width Dh=%lld is not supported (supported: 16, 32, 64, 128)",
                (long long)Dh);
  if (page_size < 1 || page_size > 65536 || (page_size & (page_size - 1)) != 0)
    return fail(RCA_ERR_INVALID_ARGUMENT, "page_size must be a power of two in [1, 65536] (got %lld)",
                (long long)page_size);
  if (B > rca::kDecodeMaxBatch)
    return fail(RCA_ERR_UNSUPPORTED, "paged decode takes at most %lld requests per call (got B=%lld)",
                (long long)rca::kDecodeMaxBatch, (long long)B);
  if (max_pages > (int64_t(1) << 30) / page_size)
    return fail(RCA_ERR_INVALID_ARGUMENT, "max_pages * page_size must be <= 2^30");
  if (num_pages > 0x7fffffffLL || Hq > 65536 ||
      B * rca::decode_max_chunks(page_size, max_pages) * Hq > 0x7fffffffLL)
    return fail(RCA_ERR_INVALID_ARGUMENT, "paged decode problem too large");
  return RCA_OK;
}

struct DecodeWs {
  size_t ml_off, acc_off, total;
};

// Per (request, query head, chunk): (max, sum) and the unnormalised output row.
// Used only when a request can span more than one chunk; never less than 256
// bytes so that a valid size is never 0.
DecodeWs decode_ws_layout(int64_t B, int64_t Hq, int64_t Dh, int64_t page_size, int64_t max_pages) {
  DecodeWs w{};
  w.total = 256;
  const int64_t maxch = rca::decode_max_chunks(page_size, max_pages);
  if (maxch <= 1) return w;
  const size_t rows = size_t(B) * Hq * maxch;
  w.ml_off = 0;
  w.acc_off = round256(rows * 2 * 4);
  w.total = w.acc_off + round256(rows * Dh * 4);
  return w;
}

#define RCA_CHECK(x)              \
  do {                            \
    rca_status _s = (x);          \
    if (_s != RCA_OK) return _s;  \
  } while (0)

#define RCA_GUARD_BEGIN try {
#define RCA_GUARD_END                                                  \
  }                                                                    \
  catch (...) {                                                        \
    return fail(RCA_ERR_CUDA, "internal error (C++ exception caught)"); \
  }

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
template <bool TF32, int DHP>
rca_status launch_fwd(const void* q, const void* k, const void* v, int64_t B, int64_t Hq, int64_t Hkv,
                      int64_t T, int64_t Dh, void* out, float* lse, cudaStream_t st, int64_t qs, int64_t kvs,
                      const int* lens, const int4* items, const int* n_items_dev) {
  using C = rca::FwdCfg<TF32, DHP>;
  static std::atomic<unsigned long long> smem_set[2] = {};
  CUtensorMap mq, mk, mv;
  RCA_CHECK(make_map(&mq, q, B, T, Hq, Dh, TF32, "q", 128, qs));
  RCA_CHECK(make_map(&mk, k, B, T, Hkv, Dh, TF32, "k", 128, kvs));
  RCA_CHECK(make_map(&mv, v, B, T, Hkv, Dh, TF32, "v", 128, kvs));
  int* status = nullptr;
  RCA_CHECK(status_word(&status));
  const int li = items ? 1 : 0;  // the work-list instantiation has its own caches
  auto kern = items ? rca::attn_fwd_kernel<TF32, DHP, true> : rca::attn_fwd_kernel<TF32, DHP, false>;
  cudaError_t e = ensure_smem(kern, C::SMEM_BYTES, smem_set[li]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(fwd)");
  // Warpgroup register split (setmaxnreg) out of the launch count: checked
  // before the first launch, as in the backward.
  static std::atomic<int> launch_regs[2] = {};
  if (launch_regs[li].load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(fwd)");
    launch_regs[li].store(fa.numRegs, std::memory_order_release);
  }
  if (launch_regs[li].load(std::memory_order_acquire) != C::LAUNCH_REGS)
    return fail(RCA_ERR_UNSUPPORTED, "forward kernel built with %d registers per thread, its warpgroup split needs %d",
                launch_regs[li].load(), C::LAUNCH_REGS);
  rca::FwdArgs a{};
  a.out = out;
  a.lse = lse;
  a.lens = lens;
  a.items = items;
  a.n_items_dev = n_items_dev;
  a.status = status;
  a.timeout_ns = g_timeout_ns.load();
  a.B = int(B); a.Hq = int(Hq); a.Hkv = int(Hkv); a.T = int(T); a.Dh = int(Dh);
  a.group = int(Hq / Hkv);
  a.n_qt = int((T + 127) / 128);
  a.n_items = int(int64_t(a.n_qt) * B * Hq);
  a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(Dh)));
  // Persistent launch (one CTA per SM walking several work items) where the
  // kernel overlaps one item's epilogue with the next item's first products;
  // otherwise one CTA per work item.
  int grid = a.n_items;
  if (C::EPI_WG) {
    int sms = 0;
    RCA_CHECK(sm_count(&sms));
    if (grid > sms) grid = sms;
  }
  launch_dep(kern, dim3(unsigned(grid)), dim3(C::NTHREADS), C::SMEM_BYTES, st, mq, mk, mv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch attn_fwd_kernel");
  return RCA_OK;
}

// n elements in rows of row_len (all heads of one position); source rows are
// src_row apart (== row_len when contiguous).
rca_status launch_split(const void* src, void* hi, void* lo, size_t n, int64_t row_len, int64_t src_row,
                        cudaStream_t st) {
  const long long n4 = (long long)(n / 4);
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (n4 + 255) / 256, cap = (long long)sms * 8;
  const unsigned grid = unsigned(want < cap ? (want > 0 ? want : 1) : cap);
  if (src_row == row_len)
    launch_dep(rca::split_hilo_kernel<false>, dim3(grid), dim3(256), 0, st, static_cast<const float*>(src), static_cast<__nv_bfloat16*>(hi),
                                                         static_cast<__nv_bfloat16*>(lo), n4, row_len / 4, src_row / 4);
  else
    launch_dep(rca::split_hilo_kernel<true>, dim3(grid), dim3(256), 0, st, static_cast<const float*>(src), static_cast<__nv_bfloat16*>(hi),
                                                        static_cast<__nv_bfloat16*>(lo), n4, row_len / 4, src_row / 4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch split_hilo_kernel");
  return RCA_OK;
}

// bf16 storage, head width 128: the 64-row query sub-tile kernel (bwd_sub.cuh),
// one CTA per work item.
rca_status launch_bwd_sub(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                          int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, void* ws, const WsLayout& L,
                          cudaStream_t st, int* status_override, int64_t qs, int64_t kvs, int64_t dkvs,
                          const int4* items, const int* n_items_dev) {
  using C = rca::BwdSubCfg;
  static std::atomic<unsigned long long> smem_set[2] = {};
  uint8_t* w = static_cast<uint8_t*>(ws);
  rca::BwdMaps maps;
  RCA_CHECK(make_map(&maps.q[0], q, B, T, Hq, Dh, false, "q", 64, qs));
  RCA_CHECK(make_map(&maps.k[0], k, B, T, Hkv, Dh, false, "k", 128, kvs));
  RCA_CHECK(make_map(&maps.v[0], v, B, T, Hkv, Dh, false, "v", 128, kvs));
  RCA_CHECK(make_map(&maps.dO[0], dout, B, T, Hq, Dh, false, "dout", 64));
  maps.q[1] = maps.q[0];
  maps.k[1] = maps.k[0];
  maps.v[1] = maps.v[0];
  maps.dO[1] = maps.dO[0];
  RCA_CHECK(make_map(&maps.dq, w + L.dq_off, B, T, Hq, Dh, true, "dq accumulator", 32));
  int* status = status_override;
  if (!status) RCA_CHECK(status_word(&status));
  const int li = items ? 1 : 0;
  auto kern = items ? rca::attn_bwd_sub_kernel<true> : rca::attn_bwd_sub_kernel<false>;
  cudaError_t e = ensure_smem(kern, C::SMEM_BYTES, smem_set[li]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd sub-tile)");
  static std::atomic<int> launch_regs[2] = {};
  if (launch_regs[li].load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(bwd sub-tile)");
    launch_regs[li].store(fa.numRegs, std::memory_order_release);
  }
  if (launch_regs[li].load(std::memory_order_acquire) != C::LAUNCH_REGS)
    return fail(RCA_ERR_UNSUPPORTED, "backward kernel built with %d registers per thread, its warpgroup split needs %d",
                launch_regs[li].load(), C::LAUNCH_REGS);
  rca::BwdArgs a{};
  a.dk = dk;
  a.dv = dv;
  a.dkv_row = dkvs;
  a.items = items;
  a.n_items_dev = n_items_dev;
  a.lse2 = reinterpret_cast<const float*>(w + L.lse2_off);
  a.dvec = reinterpret_cast<const float*>(w + L.d_off);
  a.status = status;
  a.timeout_ns = g_timeout_ns.load();
  a.B = int(B); a.Hq = int(Hq); a.Hkv = int(Hkv); a.T = int(T); a.Dh = int(Dh);
  a.group = int(Hq / Hkv);
  a.n_t = int((T + 127) / 128);
  a.Tpad = int(L.Tpad);
  a.scale = float(1.0 / std::sqrt(double(Dh)));
  a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(Dh)));
  a.n_items = int(int64_t(a.n_t) * B * Hkv);
  launch_dep(kern, dim3(unsigned(a.n_items)), dim3(C::NTHREADS), C::SMEM_BYTES, st, maps, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch attn_bwd_sub_kernel");
  return RCA_OK;
}

template <bool HL, int DHB>
rca_status launch_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, void* ws,
                           const WsLayout& L, cudaStream_t st, int* status_override, int64_t qs, int64_t kvs,
                           int64_t dkvs, const int4* items, const int* n_items_dev) {
  if constexpr (!HL && DHB == 128)
    return launch_bwd_sub(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, ws, L, st, status_override, qs, kvs, dkvs, items,
                          n_items_dev);
  using C = rca::BwdCfg<HL, DHB>;
  static std::atomic<unsigned long long> smem_set[2] = {};
  uint8_t* w = static_cast<uint8_t*>(ws);
  rca::BwdMaps maps;
  if constexpr (HL) {
    // fp32 storage: bf16 hi/lo copies live in the workspace.
    uint8_t* hl = w + L.hl_off;
    void* qh = hl;
    void* ql = hl + L.q_part;
    void* dh = hl + 2 * L.q_part;
    void* dl = hl + 3 * L.q_part;
    void* kh = hl + 4 * L.q_part;
    void* kl = static_cast<uint8_t*>(kh) + L.kv_part;
    void* vh = static_cast<uint8_t*>(kh) + 2 * L.kv_part;
    void* vl = static_cast<uint8_t*>(kh) + 3 * L.kv_part;
    const size_t nq = size_t(B) * T * Hq * Dh, nkv = size_t(B) * T * Hkv * Dh;
    RCA_CHECK(launch_split(q, qh, ql, nq, Hq * Dh, qs, st));
    RCA_CHECK(launch_split(dout, dh, dl, nq, Hq * Dh, Hq * Dh, st));
    RCA_CHECK(launch_split(k, kh, kl, nkv, Hkv * Dh, kvs, st));
    RCA_CHECK(launch_split(v, vh, vl, nkv, Hkv * Dh, kvs, st));
    RCA_CHECK(make_map(&maps.q[0], qh, B, T, Hq, Dh, false, "q hi"));
    RCA_CHECK(make_map(&maps.q[1], ql, B, T, Hq, Dh, false, "q lo"));
    RCA_CHECK(make_map(&maps.dO[0], dh, B, T, Hq, Dh, false, "dout hi"));
    RCA_CHECK(make_map(&maps.dO[1], dl, B, T, Hq, Dh, false, "dout lo"));
    RCA_CHECK(make_map(&maps.k[0], kh, B, T, Hkv, Dh, false, "k hi"));
    RCA_CHECK(make_map(&maps.k[1], kl, B, T, Hkv, Dh, false, "k lo"));
    RCA_CHECK(make_map(&maps.v[0], vh, B, T, Hkv, Dh, false, "v hi"));
    RCA_CHECK(make_map(&maps.v[1], vl, B, T, Hkv, Dh, false, "v lo"));
  } else {
    RCA_CHECK(make_map(&maps.q[0], q, B, T, Hq, Dh, false, "q", 128, qs));
    RCA_CHECK(make_map(&maps.k[0], k, B, T, Hkv, Dh, false, "k", 128, kvs));
    RCA_CHECK(make_map(&maps.v[0], v, B, T, Hkv, Dh, false, "v", 128, kvs));
    RCA_CHECK(make_map(&maps.dO[0], dout, B, T, Hq, Dh, false, "dout"));
    maps.q[1] = maps.q[0];
    maps.k[1] = maps.k[0];
    maps.v[1] = maps.v[0];
    maps.dO[1] = maps.dO[0];
  }
  // dQ partials are added by each warp for its 32 query rows.
  RCA_CHECK(make_map(&maps.dq, w + L.dq_off, B, T, Hq, Dh, true, "dq accumulator", 32));
  int* status = status_override;
  if (!status) RCA_CHECK(status_word(&status));
  const int li = items ? 1 : 0;  // the work-list instantiation has its own caches
  auto kern = items ? rca::attn_bwd_main_kernel<HL, DHB, true> : rca::attn_bwd_main_kernel<HL, DHB, false>;
  cudaError_t e = ensure_smem(kern, C::SMEM_BYTES, smem_set[li]);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd)");
  // The kernel splits its registers between warpgroups (setmaxnreg) out of the
  // per-thread count it is launched with; a different count would make the
  // split wait forever, so it is checked before the first launch.
  static std::atomic<int> launch_regs[2] = {};
  if (launch_regs[li].load(std::memory_order_acquire) == 0) {
    cudaFuncAttributes fa{};
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return cuda_fail(e, "cudaFuncGetAttributes(bwd)");
    launch_regs[li].store(fa.numRegs, std::memory_order_release);
  }
  if (launch_regs[li].load(std::memory_order_acquire) != C::LAUNCH_REGS)
    return fail(RCA_ERR_UNSUPPORTED, "backward kernel built with %d registers per thread, its warpgroup split needs %d",
                launch_regs[li].load(), C::LAUNCH_REGS);
  rca::BwdArgs a{};
  a.dk = dk;
  a.dv = dv;
  a.dkv_row = dkvs;
  a.items = items;
  a.n_items_dev = n_items_dev;
  a.lse2 = reinterpret_cast<const float*>(w + L.lse2_off);
  a.dvec = reinterpret_cast<const float*>(w + L.d_off);
  a.status = status;
  a.timeout_ns = g_timeout_ns.load();
  a.B = int(B); a.Hq = int(Hq); a.Hkv = int(Hkv); a.T = int(T); a.Dh = int(Dh);
  a.group = int(Hq / Hkv);
  a.n_t = int((T + 127) / 128);
  a.Tpad = int(L.Tpad);
  a.scale = float(1.0 / std::sqrt(double(Dh)));
  a.scale_log2 = float(1.4426950408889634 / std::sqrt(double(Dh)));
  a.n_items = int(int64_t(a.n_t) * B * Hkv);
  // Persistent launch (one CTA per SM walking several work items) where the
  // kernel prefetches across items; otherwise one CTA per work item.
  int grid = a.n_items;
  if (C::PTB) {
    int sms = 0;
    RCA_CHECK(sm_count(&sms));
    if (grid > sms) grid = sms;
  }
  launch_dep(kern, dim3(unsigned(grid)), dim3(C::NTHREADS), C::SMEM_BYTES, st, maps, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch attn_bwd_main_kernel");
  return RCA_OK;
}

// qs, kvs: elements between consecutive positions of Q and of K, V (0 means
// contiguous [B, T, H, Dh]); dkvs the same for the dK, dV outputs.
rca_status do_fwd(const void* q, const void* k, const void* v, int64_t B, int64_t Hq, int64_t Hkv, int64_t T,
                  int64_t Dh, void* out, float* lse, rca_dtype dt, cudaStream_t st, int64_t qs = 0,
                  int64_t kvs = 0, const int* lens = nullptr, const int4* items = nullptr,
                  const int* n_items_dev = nullptr) {
  if (dt == RCA_BF16) {
    if (Dh <= 64)
      return launch_fwd<false, 64>(q, k, v, B, Hq, Hkv, T, Dh, out, lse, st, qs, kvs, lens, items, n_items_dev);
    return launch_fwd<false, 128>(q, k, v, B, Hq, Hkv, T, Dh, out, lse, st, qs, kvs, lens, items, n_items_dev);
  }
  if (Dh <= 32)
    return launch_fwd<true, 32>(q, k, v, B, Hq, Hkv, T, Dh, out, lse, st, qs, kvs, lens, items, n_items_dev);
  return launch_fwd<true, 64>(q, k, v, B, Hq, Hkv, T, Dh, out, lse, st, qs, kvs, lens, items, n_items_dev);
}

rca_status do_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                       int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt, void* ws,
                       const WsLayout& L, cudaStream_t st, int* status_override = nullptr, int64_t qs = 0,
                       int64_t kvs = 0, int64_t dkvs = 0, const int4* items = nullptr,
                       const int* n_items_dev = nullptr) {
  if (qs == 0) qs = Hq * Dh;
  if (kvs == 0) kvs = Hkv * Dh;
  if (dkvs == 0) dkvs = Hkv * Dh;
  if (dt == RCA_BF16) {
    if (Dh <= 64)
      return launch_bwd_main<false, 64>(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, ws, L, st, status_override, qs,
                                        kvs, dkvs, items, n_items_dev);
    return launch_bwd_main<false, 128>(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, ws, L, st, status_override, qs,
                                       kvs, dkvs, items, n_items_dev);
  }
  return launch_bwd_main<true, 64>(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, ws, L, st, status_override, qs, kvs,
                                   dkvs, items, n_items_dev);
}

// ---------------------------------------------------------------------------
// Variable-length batches: planned work lists (after the backward's scratch)
// ---------------------------------------------------------------------------
constexpr int64_t kVarlenMaxBatch = 4096, kVarlenMaxT = 131072;

struct VarlenLayout {
  size_t fwd_items, bwd_items, counts, total;  // offsets past the backward scratch
};

VarlenLayout varlen_layout(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt) {
  VarlenLayout v{};
  const size_t n_qt = size_t((T + 127) / 128);
  v.fwd_items = round256(ws_layout(B, Hq, Hkv, T, Dh, dt).total);
  v.bwd_items = v.fwd_items + round256(size_t(B) * Hq * n_qt * 16);
  v.counts = v.bwd_items + round256(size_t(B) * Hkv * n_qt * 16);
  v.total = v.counts + 256;
  return v;
}

rca_status check_varlen(int64_t B, int64_t T) {
  if (B > kVarlenMaxBatch || T > kVarlenMaxT)
    return fail(RCA_ERR_UNSUPPORTED, "variable-length batches take B <= %lld and T <= %lld (got B=%lld T=%lld)",
                (long long)kVarlenMaxBatch, (long long)kVarlenMaxT, (long long)B, (long long)T);
  return RCA_OK;
}

// Builds both work lists from the lengths; returns their device pointers.
rca_status plan_args(rca::VarlenPlanArgs& a, size_t& smem, const int* lens, int64_t B, int64_t Hq, int64_t Hkv,
                     int64_t T, void* ws, const VarlenLayout& V) {
  char* w = static_cast<char*>(ws);
  a = rca::VarlenPlanArgs{};
  a.lens = lens;
  a.fwd_items = reinterpret_cast<int4*>(w + V.fwd_items);
  a.bwd_items = reinterpret_cast<int4*>(w + V.bwd_items);
  a.fwd_count = reinterpret_cast<int*>(w + V.counts);
  a.bwd_count = a.fwd_count + 1;
  RCA_CHECK(status_word(&a.status));
  a.B = int(B);
  a.Hq = int(Hq);
  a.Hkv = int(Hkv);
  a.T = int(T);
  a.n_qt = int((T + 127) / 128);
  smem = (2 * size_t(B) + 3 * (size_t(a.n_qt) + 1)) * sizeof(int);
  return RCA_OK;
}

rca_status plan_varlen(const int* lens, int64_t B, int64_t Hq, int64_t Hkv, int64_t T, void* ws, const VarlenLayout& V,
                       cudaStream_t st, const int4** fwd_items, const int** fwd_count, const int4** bwd_items,
                       const int** bwd_count) {
  rca::VarlenPlanArgs a{};
  size_t smem = 0;
  RCA_CHECK(plan_args(a, smem, lens, B, Hq, Hkv, T, ws, V));
  launch_dep(rca::varlen_plan_kernel, dim3(1), dim3(rca::kVarlenPlanThreads), smem, st, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch varlen_plan_kernel");
  *fwd_items = a.fwd_items;
  *fwd_count = a.fwd_count;
  *bwd_items = a.bwd_items;
  *bwd_count = a.bwd_count;
  return RCA_OK;
}

// Zero the rows at or past each sequence's length (and -inf LSE) of x [B, T, H, Dh]
// and, if given, of x2 of the same shape: one grid column per sequence (and
// tensor), covering only its padding.
// The variable-length prologue launch (varlen.cuh): the work lists, the zero
// fill of the padding rows of x (and x2; lse -inf with x), and with `pre`
// the backward preprocess, in one launch ahead of the attention kernel. Its
// preprocess part indexes rows with 32 bits: callers check
// varlen_pre_fits() first.
bool varlen_pre_fits(int64_t Hq, int64_t Dh, rca_dtype dt, const WsLayout& L) {
  return L.Tpad * Hq * (Dh / (dt == RCA_BF16 ? 8 : 4)) < (int64_t(1) << 31);
}
rca_status varlen_prologue(const int* lens, int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt,
                           void* ws, const VarlenLayout& V, void* x, void* x2, float* lse, int64_t H,
                           const rca::PreArgs* pre, const WsLayout* L, cudaStream_t st, const int4** fwd_items,
                           const int** fwd_count, const int4** bwd_items, const int** bwd_count) {
  rca::VarlenPrologue p{};
  size_t smem = 0;
  RCA_CHECK(plan_args(p.plan, smem, lens, B, Hq, Hkv, T, ws, V));
  int sms = 0;
  RCA_CHECK(sm_count(&sms));
  const int64_t cap = std::max<int64_t>(1, int64_t(sms) * 8 / B);
  const int64_t per_seq = T * H * Dh * (dt == RCA_BF16 ? 2 : 4) / 16;  // 16-byte vectors
  p.zx = x;
  p.zx2 = x2;
  p.zlse = lse;
  p.zH = int(H);
  p.Dh = int(Dh);
  p.zgx = int(std::max<int64_t>(1, std::min((per_seq + 1023) / 1024, cap)));
  int64_t blocks = 1 + int64_t(p.zgx) * B * (x2 ? 2 : 1);
  if (pre) {
    p.pre = *pre;
    const int64_t lpr = Dh / (dt == RCA_BF16 ? 8 : 4);
    p.pgx = int(std::max<int64_t>(1, std::min((L->Tpad * Hq * lpr + 255) / 256, cap)));
    blocks += int64_t(p.pgx) * B;
  }
  const dim3 grid = dim3(static_cast<unsigned>(blocks));
  if (dt == RCA_BF16) {
    if (pre) launch_dep(rca::varlen_prologue_kernel<2, 1>, grid, dim3(256), smem, st, p);
    else launch_dep(rca::varlen_prologue_kernel<2, 0>, grid, dim3(256), smem, st, p);
  } else {
    if (pre) launch_dep(rca::varlen_prologue_kernel<4, 2>, grid, dim3(256), smem, st, p);
    else launch_dep(rca::varlen_prologue_kernel<4, 0>, grid, dim3(256), smem, st, p);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch varlen_prologue_kernel");
  *fwd_items = p.plan.fwd_items;
  *fwd_count = p.plan.fwd_count;
  *bwd_items = p.plan.bwd_items;
  *bwd_count = p.plan.bwd_count;
  return RCA_OK;
}

rca_status zero_padding(void* x, float* lse, const int* lens, int64_t B, int64_t T, int64_t H, int64_t Dh,
                        rca_dtype dt, cudaStream_t st, void* x2 = nullptr) {
  const int64_t per_seq = T * H * Dh * (dt == RCA_BF16 ? 2 : 4) / 16;  // 16-byte vectors
  int sms = 0;
  RCA_CHECK(sm_count(&sms));
  const int64_t want = (per_seq + 1023) / 1024, cap = std::max<int64_t>(1, int64_t(sms) * 8 / B);
  const dim3 grid(unsigned(std::max<int64_t>(1, std::min(want, cap))), unsigned(B), x2 ? 2u : 1u);
  if (dt == RCA_BF16)
    launch_dep(rca::varlen_zero_kernel<2>, dim3(grid), dim3(256), 0, st, x, x2, lse, lens, int(T), int(H), int(Dh));
  else
    launch_dep(rca::varlen_zero_kernel<4>, dim3(grid), dim3(256), 0, st, x, x2, lse, lens, int(T), int(H), int(Dh));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch varlen_zero_kernel");
  return RCA_OK;
}

// dQ of a variable-length batch: real rows converted from the accumulator,
// padding rows written as zeros.
rca_status varlen_convert(void* dq, const int* lens, int64_t B, int64_t Hq, int64_t T, int64_t Dh, rca_dtype dt,
                          const void* ws, const WsLayout& L, cudaStream_t st) {
  const float* acc = reinterpret_cast<const float*>(static_cast<const uint8_t*>(ws) + L.dq_off);
  const long long row4 = Hq * Dh / 4;
  // One resident wave of blocks looping over four groups per thread (one
  // group per thread measured slower here: most of its blocks cover padding).
  int sms = 0;
  RCA_CHECK(sm_count(&sms));
  const int64_t want = (T * row4 + 1023) / 1024, cap = std::max<int64_t>(1, int64_t(sms) * 8 / B);
  const dim3 grid(unsigned(std::max<int64_t>(1, std::min(want, cap))), unsigned(B));
  const float scale = float(1.0 / std::sqrt(double(Dh)));
  if (dt == RCA_BF16)
    launch_dep(rca::varlen_dq_convert_kernel<false>, dim3(grid), dim3(256), 0, st, acc, dq, lens, int(T), row4, scale);
  else
    launch_dep(rca::varlen_dq_convert_kernel<true>, dim3(grid), dim3(256), 0, st, acc, dq, lens, int(T), row4, scale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch varlen_dq_convert_kernel");
  return RCA_OK;
}

rca_status pre_args(rca::PreArgs& a, const void* out, const float* lse, const void* dout, int64_t B, int64_t Hq,
                    int64_t T, int64_t Dh, rca_dtype dt, void* ws, const WsLayout& L, const int* lens) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  a = rca::PreArgs{};
  a.lens = lens;
  if (lens) RCA_CHECK(status_word(&a.status));
  a.out = out;
  a.lse = lse;
  a.dout = dout;
  a.dq_acc = reinterpret_cast<float*>(w + L.dq_off);
  a.lse2 = reinterpret_cast<float*>(w + L.lse2_off);
  a.dvec = reinterpret_cast<float*>(w + L.d_off);
  a.B = int(B); a.Hq = int(Hq); a.T = int(T); a.Dh = int(Dh); a.Tpad = int(L.Tpad);
  const int64_t lpr = Dh / (dt == RCA_BF16 ? 8 : 4);  // 16-byte segments per row, a power of two
  a.lg_lpr = 0;
  while ((int64_t(1) << a.lg_lpr) < lpr) ++a.lg_lpr;
  // n / Hq for n < 2^31 as a multiply-high (Granlund and Montgomery, 1994):
  // l = ceil(log2 Hq), m = floor(2^32 (2^l - Hq) / Hq) + 1 (below 2^32).
  int l = 0;
  while ((int64_t(1) << l) < Hq) ++l;
  a.hq_l = l;
  a.hq_m = uint32_t(((uint64_t(1) << 32) * ((uint64_t(1) << l) - uint64_t(Hq))) / uint64_t(Hq) + 1);
  return RCA_OK;
}

rca_status do_preprocess(const void* out, const float* lse, const void* dout, int64_t B, int64_t Hq, int64_t T,
                         int64_t Dh, rca_dtype dt, void* ws, const WsLayout& L, cudaStream_t st,
                         const int* lens = nullptr) {
  rca::PreArgs a{};
  RCA_CHECK(pre_args(a, out, lse, dout, B, Hq, T, Dh, dt, ws, L, lens));
  const int64_t seg = (L.Tpad * Hq) << a.lg_lpr;  // 16-byte segments of one batch entry
  const int64_t per_block = 256 * rca::kPreSegs;
  const int64_t bpb = (seg + per_block - 1) / per_block;
  if (bpb * B >= (int64_t(1) << 31))
    return fail(RCA_ERR_UNSUPPORTED, "rca_attn_bwd_preprocess: B x T x Hq x Dh too large for one launch");
  a.bpb = int(bpb);
  const dim3 grid = dim3(static_cast<unsigned>(bpb * B));
  const bool narrow = seg < (int64_t(1) << 31);  // 32-bit segment indices within an entry suffice
  if (dt == RCA_BF16) {
    if (narrow) launch_dep(rca::attn_bwd_preprocess_kernel<false, false>, grid, dim3(256), 0, st, a);
    else launch_dep(rca::attn_bwd_preprocess_kernel<false, true>, grid, dim3(256), 0, st, a);
  } else {
    if (narrow) launch_dep(rca::attn_bwd_preprocess_kernel<true, false>, grid, dim3(256), 0, st, a);
    else launch_dep(rca::attn_bwd_preprocess_kernel<true, true>, grid, dim3(256), 0, st, a);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch attn_bwd_preprocess_kernel");
  return RCA_OK;
}

rca_status do_convert(void* dq, int64_t B, int64_t Hq, int64_t T, int64_t Dh, rca_dtype dt, const void* ws,
                      const WsLayout& L, cudaStream_t st, int64_t dqs = 0) {
  if (dqs == 0) dqs = Hq * Dh;  // elements between consecutive positions of dq
  const float* acc = reinterpret_cast<const float*>(static_cast<const uint8_t*>(ws) + L.dq_off);
  const long long n4 = (long long)(B * T * Hq * Dh / 4);
  // One float4 group per thread, every group in flight at once: inside the
  // training step this measured 7 us faster at B4 H16 T2048 Dh64 than one
  // resident wave of blocks looping over four groups per thread.
  const long long want = (n4 + 255) / 256;
  const long long cap = (1LL << 31) - 1;
  const unsigned grid = unsigned(want < cap ? (want > 0 ? want : 1) : cap);
  const float scale = float(1.0 / std::sqrt(double(Dh)));
  const long long row4 = Hq * Dh / 4, dq_row4 = dqs / 4;
  const bool strided = dqs != Hq * Dh;
  if (dt == RCA_BF16) {
    if (strided) launch_dep(rca::attn_bwd_dq_convert_kernel<false, true>, dim3(grid), dim3(256), 0, st, acc, dq, n4, scale, row4, dq_row4);
    else launch_dep(rca::attn_bwd_dq_convert_kernel<false, false>, dim3(grid), dim3(256), 0, st, acc, dq, n4, scale, row4, dq_row4);
  } else {
    if (strided) launch_dep(rca::attn_bwd_dq_convert_kernel<true, true>, dim3(grid), dim3(256), 0, st, acc, dq, n4, scale, row4, dq_row4);
    else launch_dep(rca::attn_bwd_dq_convert_kernel<true, false>, dim3(grid), dim3(256), 0, st, acc, dq, n4, scale, row4, dq_row4);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch attn_bwd_dq_convert_kernel");
  return RCA_OK;
}

}  // namespace

extern "C" {

uint32_t rca_abi_version(void) { return RCA_ABI_VERSION; }

const char* rca_last_error(void) { return g_err.c_str(); }

uint64_t rca_set_wait_timeout_ns(uint64_t ns) {
  if (ns < 1000000ull) ns = 1000000ull;
  return g_timeout_ns.exchange(ns);
}

rca_status rca_attn_fwd(const void* q, const void* k, const void* v, int64_t B, int64_t Hq, int64_t Hkv,
                        int64_t T, int64_t Dh, void* out, float* lse, rca_dtype dt, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !out || !lse) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_fwd: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_fwd: q, k, v, out and lse must be 16-byte aligned");
  return do_fwd(q, k, v, B, Hq, Hkv, T, Dh, out, lse, dt, static_cast<cudaStream_t>(cuda_stream));
  RCA_GUARD_END
}

size_t rca_attn_bwd_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hkv > Hq || T < 1 || Dh < 1 || T > (int64_t(1) << 30)) return 0;
  if (dt != RCA_BF16 && dt != RCA_F32_TF32) return 0;
  return ws_layout(B, Hq, Hkv, T, Dh, dt).total;
}

rca_status rca_attn_bwd_preprocess(const void* out, const float* lse, const void* dout, int64_t B, int64_t Hq,
                                   int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt, void* workspace,
                                   size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!out || !lse || !dout) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_preprocess: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(out) || !aligned16(dout) || !aligned16(lse))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_preprocess: out, dout and lse must be 16-byte aligned");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  RCA_CHECK(check_ws(workspace, workspace_bytes, L));
  return do_preprocess(out, lse, dout, B, Hq, T, Dh, dt, workspace, L, static_cast<cudaStream_t>(cuda_stream));
  RCA_GUARD_END
}

rca_status rca_attn_bwd_main(const void* q, const void* k, const void* v, const void* dout, void* dk, void* dv,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt,
                             void* workspace, size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !dout || !dk || !dv)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_main: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout) || !aligned16(dk) || !aligned16(dv))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_main: tensors must be 16-byte aligned");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  RCA_CHECK(check_ws(workspace, workspace_bytes, L));
  return do_bwd_main(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, dt, workspace, L,
                     static_cast<cudaStream_t>(cuda_stream));
  RCA_GUARD_END
}

rca_status rca_attn_bwd_dq_convert(void* dq, int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                   rca_dtype dt, const void* workspace, size_t workspace_bytes,
                                   void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!dq) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_dq_convert: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(dq)) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_dq_convert: dq must be 16-byte aligned");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  RCA_CHECK(check_ws(workspace, workspace_bytes, L));
  return do_convert(dq, B, Hq, T, Dh, dt, workspace, L, static_cast<cudaStream_t>(cuda_stream));
  RCA_GUARD_END
}

rca_status rca_attn_bwd(const void* q, const void* k, const void* v, const void* out, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int64_t B, int64_t Hq, int64_t Hkv,
                        int64_t T, int64_t Dh, rca_dtype dt, void* workspace, size_t workspace_bytes,
                        void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd: tensors must be 16-byte aligned");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  RCA_CHECK(check_ws(workspace, workspace_bytes, L));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  RCA_CHECK(do_preprocess(out, lse, dout, B, Hq, T, Dh, dt, workspace, L, st));
  RCA_CHECK(do_bwd_main(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, dt, workspace, L, st));
  return do_convert(dq, B, Hq, T, Dh, dt, workspace, L, st);
  RCA_GUARD_END
}

size_t rca_paged_decode_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t Dh, int64_t page_size,
                                       int64_t max_pages, rca_dtype dt) {
  try {
    if (check_decode_shape(B, Hq, Hkv, Dh, page_size, max_pages, 1, dt) != RCA_OK) return 0;
    return decode_ws_layout(B, Hq, Dh, page_size, max_pages).total;
  } catch (...) {
    return 0;
  }
}

rca_status rca_paged_decode(const void* q, const void* k_pool, const void* v_pool, const int32_t* page_table,
                            const int32_t* seq_lens, int64_t B, int64_t Hq, int64_t Hkv, int64_t Dh,
                            int64_t page_size, int64_t max_pages, int64_t num_pages, void* out, float* lse,
                            rca_dtype dt, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !out || !lse)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_paged_decode: null pointer");
  RCA_CHECK(check_decode_shape(B, Hq, Hkv, Dh, page_size, max_pages, num_pages, dt));
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_paged_decode: q, k_pool and v_pool must be 16-byte aligned");
  const auto a4 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
  const uintptr_t out_mis = reinterpret_cast<uintptr_t>(out) & (dt == RCA_F32_TF32 ? 3u : 1u);
  if (!a4(page_table) || !a4(seq_lens) || !a4(lse) || out_mis)
    return fail(RCA_ERR_INVALID_ARGUMENT,
                "rca_paged_decode: page_table, seq_lens and lse must be 4-byte aligned, out aligned to its element");
  const DecodeWs L = decode_ws_layout(B, Hq, Dh, page_size, max_pages);
  if (!workspace) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_paged_decode: workspace is null");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_paged_decode: workspace must be 256-byte aligned");
  if (workspace_bytes < L.total)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_paged_decode: workspace too small: %zu bytes given, %zu needed",
                workspace_bytes, L.total);
  int* status = nullptr;
  RCA_CHECK(status_word(&status));
  int sms = 0;
  RCA_CHECK(sm_count(&sms));
  rca::DecodeParams p{};
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.lse = lse;
  p.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.ml_off);
  p.part_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.acc_off);
  p.status = status;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Dh = Dh;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.bf16 = dt == RCA_BF16;
  p.sms = sms;
  p.timeout_ns = g_timeout_ns.load();
  cudaError_t e = rca::launch_paged_decode(p, static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "launch paged decode");
  return RCA_OK;
  RCA_GUARD_END
}

// ---------------------------------------------------------------------------
// Materialized path (probabilities returned and kept for the VJP)
// ---------------------------------------------------------------------------
static rca_status check_mat_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt) {
  if (B < 1 || Hq < 1 || Hkv < 1)
    return fail(RCA_ERR_INVALID_ARGUMENT, "B, Hq and Hkv must be >= 1 (got B=%lld Hq=%lld Hkv=%lld)",
                (long long)B, (long long)Hq, (long long)Hkv);
  if (T < 1)
    return fail(RCA_ERR_INVALID_ARGUMENT,
                "T must be >= 1 (got %lld): an empty causal row is a fully masked softmax slice", (long long)T);
  if (Hq % Hkv != 0)
    return fail(RCA_ERR_INVALID_ARGUMENT, "grouped-query attention needs Hq %% Hkv == 0 (Hq=%lld Hkv=%lld)",
                (long long)Hq, (long long)Hkv);
  if (dt != RCA_BF16 && dt != RCA_F32_TF32) return fail(RCA_ERR_INVALID_ARGUMENT, "unknown dtype %d", (int)dt);
  if (Dh != 16 && Dh != 32 && Dh != 64 && Dh != 128)
    return fail(RCA_ERR_UNSUPPORTED, "head width Dh=%lld is not supported (supported: 16, 32, 64, 128)",
                (long long)Dh);
  if (T > 65536 || B * Hq > 0x7fffffffLL || double(B) * Hq * T * T > double(int64_t(1) << 37))
    return fail(RCA_ERR_INVALID_ARGUMENT,
                "materialized attention too large: the probabilities [B,Hq,T,T] need %.1f GB (B=%lld Hq=%lld T=%lld)",
                4.0 * double(B) * Hq * T * T / 1e9, (long long)B, (long long)Hq, (long long)T);
  return RCA_OK;
}

size_t rca_attn_materialized_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                            rca_dtype dt) {
  try {
    if (check_mat_shape(B, Hq, Hkv, T, Dh, dt) != RCA_OK) return 0;
    return rca::materialized_workspace_size(B, Hq, Hkv, T, Dh, dt == RCA_BF16);
  } catch (...) {
    return 0;
  }
}

static rca_status check_mat_ws(const void* ws, size_t bytes, int64_t B, int64_t Hq, int64_t Hkv, int64_t T,
                               int64_t Dh, rca_dtype dt) {
  const size_t need = rca::materialized_workspace_size(B, Hq, Hkv, T, Dh, dt == RCA_BF16);
  if (!ws) return fail(RCA_ERR_INVALID_ARGUMENT, "workspace is null");
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return fail(RCA_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
  if (bytes < need)
    return fail(RCA_ERR_INVALID_ARGUMENT, "workspace too small: %zu bytes given, %zu needed", bytes, need);
  return RCA_OK;
}

rca_status rca_attn_materialized_fwd(const void* q, const void* k, const void* v, int64_t B, int64_t Hq,
                                     int64_t Hkv, int64_t T, int64_t Dh, void* out, float* probs, float* lse,
                                     rca_dtype dt, void* workspace, size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !out || !probs || !lse)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_materialized_fwd: null pointer");
  RCA_CHECK(check_mat_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(probs) || !aligned16(lse))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_materialized_fwd: tensors must be 16-byte aligned");
  RCA_CHECK(check_mat_ws(workspace, workspace_bytes, B, Hq, Hkv, T, Dh, dt));
  rca::MatParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.probs = probs;
  p.lse = lse;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.Dh = Dh;
  p.bf16 = dt == RCA_BF16;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  RCA_CHECK(status_word(&p.status));
  p.timeout_ns = g_timeout_ns.load();
  std::string err;
  if (!rca::materialized_fwd(p, static_cast<cudaStream_t>(cuda_stream), err))
    return fail(RCA_ERR_CUDA, "rca_attn_materialized_fwd: %s", err.c_str());
  return RCA_OK;
  RCA_GUARD_END
}

rca_status rca_attn_materialized_bwd(const void* q, const void* k, const void* v, const float* probs,
                                     const void* dout, const float* dprobs, void* dq, void* dk, void* dv, int64_t B,
                                     int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt, void* workspace,
                                     size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !probs || !dout || !dq || !dk || !dv)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_materialized_bwd: null pointer");
  RCA_CHECK(check_mat_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(probs) || !aligned16(dout) ||
      (dprobs && !aligned16(dprobs)) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_materialized_bwd: tensors must be 16-byte aligned");
  RCA_CHECK(check_mat_ws(workspace, workspace_bytes, B, Hq, Hkv, T, Dh, dt));
  rca::MatParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.probs = const_cast<float*>(probs);
  p.dout = dout;
  p.dprobs = dprobs;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.T = T;
  p.Dh = Dh;
  p.bf16 = dt == RCA_BF16;
  p.workspace = workspace;
  p.workspace_bytes = workspace_bytes;
  RCA_CHECK(status_word(&p.status));
  p.timeout_ns = g_timeout_ns.load();
  std::string err;
  if (!rca::materialized_bwd(p, static_cast<cudaStream_t>(cuda_stream), err))
    return fail(RCA_ERR_CUDA, "rca_attn_materialized_bwd: %s", err.c_str());
  return RCA_OK;
  RCA_GUARD_END
}

static rca_status check_softmax_args(int64_t N, int64_t T, float scale) {
  if (N < 1 || T < 1)
    return fail(RCA_ERR_INVALID_ARGUMENT, "N and T must be >= 1 (got N=%lld T=%lld)", (long long)N, (long long)T);
  if (T > 65536 || double(N) * T * T > double(int64_t(1) << 37))
    return fail(RCA_ERR_INVALID_ARGUMENT, "causal softmax too large (N=%lld T=%lld)", (long long)N, (long long)T);
  if (!(scale == scale) || scale == INFINITY || scale == -INFINITY)
    return fail(RCA_ERR_INVALID_ARGUMENT, "scale must be finite");
  return RCA_OK;
}

rca_status rca_causal_softmax(float* scores, float* lse, int64_t N, int64_t T, float scale, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!scores || !lse) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_causal_softmax: null pointer");
  RCA_CHECK(check_softmax_args(N, T, scale));
  if (!aligned16(scores) || !aligned16(lse))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_causal_softmax: tensors must be 16-byte aligned");
  std::string err;
  if (!rca::causal_softmax_fwd(scores, lse, N, T, scale, static_cast<cudaStream_t>(cuda_stream), err))
    return fail(RCA_ERR_CUDA, "rca_causal_softmax: %s", err.c_str());
  return RCA_OK;
  RCA_GUARD_END
}

static rca_status softmax_bwd_call(const char* name, const float* probs, float* grad, const float* grad_extra,
                                   int64_t N, int64_t T, int64_t tile, float scale, void* cuda_stream) {
  if (!probs || !grad) return fail(RCA_ERR_INVALID_ARGUMENT, "%s: null pointer", name);
  RCA_CHECK(check_softmax_args(N, T, scale));
  if (tile < 1) return fail(RCA_ERR_INVALID_ARGUMENT, "%s: tile must be >= 1 (got %lld)", name, (long long)tile);
  if (!aligned16(probs) || !aligned16(grad) || (grad_extra && !aligned16(grad_extra)))
    return fail(RCA_ERR_INVALID_ARGUMENT, "%s: tensors must be 16-byte aligned", name);
  std::string err;
  if (!rca::causal_softmax_bwd(probs, grad, grad_extra, N, T, tile, scale, static_cast<cudaStream_t>(cuda_stream),
                               err))
    return fail(RCA_ERR_CUDA, "%s: %s", name, err.c_str());
  return RCA_OK;
}

rca_status rca_causal_softmax_bwd(const float* probs, float* grad, const float* grad_extra, int64_t N, int64_t T,
                                  float scale, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  return softmax_bwd_call("rca_causal_softmax_bwd", probs, grad, grad_extra, N, T, T, scale, cuda_stream);
  RCA_GUARD_END
}

rca_status rca_causal_softmax_bwd_tiled(const float* probs, float* grad, const float* grad_extra, int64_t N,
                                        int64_t T, int64_t tile, float scale, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  return softmax_bwd_call("rca_causal_softmax_bwd_tiled", probs, grad, grad_extra, N, T, tile, scale, cuda_stream);
  RCA_GUARD_END
}

// ---------------------------------------------------------------------------
// Fused QKV layout: q, k, v read from one [B, T, (Hq + 2 Hkv) * Dh] projection
// output, dq, dk, dv written into one buffer of the same shape.
// ---------------------------------------------------------------------------
rca_status rca_attn_fwd_qkv(const void* qkv, int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t Dh, void* out,
                            float* lse, rca_dtype dt, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!qkv || !out || !lse) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_fwd_qkv: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(lse))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_fwd_qkv: qkv, out and lse must be 16-byte aligned");
  const int64_t es = dt == RCA_BF16 ? 2 : 4, row = (Hq + 2 * Hkv) * Dh;
  const char* base = static_cast<const char*>(qkv);
  return do_fwd(base, base + Hq * Dh * es, base + (Hq + Hkv) * Dh * es, B, Hq, Hkv, T, Dh, out, lse, dt,
                static_cast<cudaStream_t>(cuda_stream), row, row);
  RCA_GUARD_END
}

rca_status rca_attn_bwd_qkv(const void* qkv, const void* out, const float* lse, const void* dout, void* dqkv,
                            int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t Dh, rca_dtype dt,
                            void* workspace, size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!qkv || !out || !lse || !dout || !dqkv) return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_qkv: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(qkv) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) || !aligned16(dqkv))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_qkv: tensors must be 16-byte aligned");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  RCA_CHECK(check_ws(workspace, workspace_bytes, L));
  const int64_t es = dt == RCA_BF16 ? 2 : 4, row = (Hq + 2 * Hkv) * Dh;
  const char* base = static_cast<const char*>(qkv);
  char* dbase = static_cast<char*>(dqkv);
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  RCA_CHECK(do_preprocess(out, lse, dout, B, Hq, T, Dh, dt, workspace, L, st));
  RCA_CHECK(do_bwd_main(base, base + Hq * Dh * es, base + (Hq + Hkv) * Dh * es, dout, dbase + Hq * Dh * es,
                        dbase + (Hq + Hkv) * Dh * es, B, Hq, Hkv, T, Dh, dt, workspace, L, st, nullptr, row, row,
                        row));
  return do_convert(dbase, B, Hq, T, Dh, dt, workspace, L, st, row);
  RCA_GUARD_END
}

// ---------------------------------------------------------------------------
// Padded / variable-length batches (right padding, lengths on the device)
// ---------------------------------------------------------------------------
size_t rca_attn_varlen_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Hkv > Hq || T < 1 || Dh < 1 || B > kVarlenMaxBatch || T > kVarlenMaxT) return 0;
  if (dt != RCA_BF16 && dt != RCA_F32_TF32) return 0;
  return varlen_layout(B, Hq, Hkv, T, Dh, dt).total;
}

rca_status rca_attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* seq_lens, int64_t B,
                               int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, void* out, float* lse, rca_dtype dt,
                               void* workspace, size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !seq_lens || !out || !lse)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_fwd_varlen: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  RCA_CHECK(check_varlen(B, T));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_fwd_varlen: tensors must be 16-byte aligned, seq_lens 4-byte");
  const VarlenLayout V = varlen_layout(B, Hq, Hkv, T, Dh, dt);
  WsLayout W{};
  W.total = V.total;
  RCA_CHECK(check_ws(workspace, workspace_bytes, W));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int4 *fi = nullptr, *bi = nullptr;
  const int *fc = nullptr, *bc = nullptr;
  // Work lists and the zero fill of tiles made only of padding, then the
  // forward over the listed tiles (which writes its own padding rows too).
  RCA_CHECK(varlen_prologue(seq_lens, B, Hq, Hkv, T, Dh, dt, workspace, V, out, nullptr, lse, Hq, nullptr, nullptr,
                            st, &fi, &fc, &bi, &bc));
  return do_fwd(q, k, v, B, Hq, Hkv, T, Dh, out, lse, dt, st, 0, 0, seq_lens, fi, fc);
  RCA_GUARD_END
}

rca_status rca_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out, const float* lse,
                               const void* dout, const int32_t* seq_lens, void* dq, void* dk, void* dv, int64_t B,
                               int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt, void* workspace,
                               size_t workspace_bytes, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !out || !lse || !dout || !seq_lens || !dq || !dk || !dv)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_varlen: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  RCA_CHECK(check_varlen(B, T));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_varlen: tensors must be 16-byte aligned, seq_lens 4-byte");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  const VarlenLayout V = varlen_layout(B, Hq, Hkv, T, Dh, dt);
  WsLayout W = L;
  W.total = V.total;
  RCA_CHECK(check_ws(workspace, workspace_bytes, W));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  const int4 *fi = nullptr, *bi = nullptr;
  const int *fc = nullptr, *bc = nullptr;
  if (varlen_pre_fits(Hq, Dh, dt, L)) {
    // One prologue launch (work lists, dK / dV padding zeroed, preprocess),
    // the main kernel over the listed items, the dQ conversion.
    rca::PreArgs pa{};
    RCA_CHECK(pre_args(pa, out, lse, dout, B, Hq, T, Dh, dt, workspace, L, seq_lens));
    RCA_CHECK(varlen_prologue(seq_lens, B, Hq, Hkv, T, Dh, dt, workspace, V, dk, dv, nullptr, Hkv, &pa, &L, st, &fi,
                              &fc, &bi, &bc));
    RCA_CHECK(do_bwd_main(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, dt, workspace, L, st, nullptr, 0, 0, 0, bi, bc));
    return varlen_convert(dq, seq_lens, B, Hq, T, Dh, dt, workspace, L, st);
  }
  // Rows past 32-bit indexing: separate launches, the dense preprocess
  // skipping padding rows.
  RCA_CHECK(plan_varlen(seq_lens, B, Hq, Hkv, T, workspace, V, st, &fi, &fc, &bi, &bc));
  RCA_CHECK(do_preprocess(out, lse, dout, B, Hq, T, Dh, dt, workspace, L, st, seq_lens));
  RCA_CHECK(do_bwd_main(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, dt, workspace, L, st, nullptr, 0, 0, 0, bi, bc));
  RCA_CHECK(varlen_convert(dq, seq_lens, B, Hq, T, Dh, dt, workspace, L, st));
  return zero_padding(dk, nullptr, seq_lens, B, T, Hkv, Dh, dt, st, dv);
  RCA_GUARD_END
}

rca_status rca_selftest_device_timeout(void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  int* status = nullptr;
  RCA_CHECK(status_word(&status));
  rca::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(cuda_stream)>>>(status, g_timeout_ns.load());
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch selftest_wait_kernel");
  return RCA_OK;
  RCA_GUARD_END
}

rca_status rca_stream_status(void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "asynchronous CUDA error");
  int* status = nullptr;
  RCA_CHECK(status_word(&status));
  int h = 0;
  e = cudaMemcpy(&h, status, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(status word)");
  if (h != 0) {
    cudaMemset(status, 0, sizeof(int));
    cudaDeviceSynchronize();
  }
  // The allocation-free backward records its device-side failures in a status
  // word of its own built-in region; report (and clear) that one too.
  int hn = 0;
  RCA_CHECK(noalloc_take_status(&hn));
  if (h == 0) h = hn;
  if (h != 0) {
    if (h == rca::kStatusLayout)
      return fail(RCA_ERR_CUDA,
                  "a kernel found its dynamic shared memory not 1024-byte aligned and computed nothing; "
                  "the affected results are invalid");
    if (h == rca::kStatusBadInput)
      return fail(RCA_ERR_DEVICE_INVALID_INPUT,
                  "a kernel read an invalid device-side input (a page ID outside [0, num_pages) or a "
                  "length outside [1, max_pages * page_size]); the affected results are invalid");
    return fail(RCA_ERR_DEVICE_TIMEOUT, "a device-side wait exceeded its time limit (status %d); outputs are invalid", h);
  }
  return RCA_OK;
  RCA_GUARD_END
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward without any device allocation (rca_attn_bwd_noalloc).
//
// Some callers cannot allocate device memory when they call the backward: a
// plugin interface that hands over only the input and output buffers, or a
// latency-bound loop that must never hit cudaMalloc (which can synchronise the
// device and take unbounded time). For them the scratch lives in this file-scope
// device array instead of a caller workspace. It is part of the library image,
// so every GPU that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(40) << 20;  // 40 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
static __device__ __align__(256) int g_noalloc_status;

std::mutex g_noalloc_mu;
void* g_noalloc_scratch_ptr[256] = {};
int* g_noalloc_status_ptr[256] = {};

// Once per device, with that device current: the device addresses of the
// scratch array and of its status word (host code cannot use the symbols'
// names as device addresses).
rca_status noalloc_setup(void** scratch, int** status) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 256) return fail(RCA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    void* ps = nullptr;
    e = cudaGetSymbolAddress(&ps, g_noalloc_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status)");
    g_noalloc_scratch_ptr[dev] = p;
    g_noalloc_status_ptr[dev] = static_cast<int*>(ps);
  }
  *scratch = g_noalloc_scratch_ptr[dev];
  *status = g_noalloc_status_ptr[dev];
  return RCA_OK;
}

// Only a device on which the entry point has been set up can hold a nonzero
// word; on any other device the symbol is never touched, so this never makes
// the driver load the module (and commit the scratch array) on its own.
rca_status noalloc_take_status(int* out) {
  *out = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 256) return RCA_OK;
  int* p = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    p = g_noalloc_status_ptr[dev];
  }
  if (!p) return RCA_OK;
  int h = 0;
  e = cudaMemcpy(&h, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(allocation-free status word)");
  if (h != 0) {
    e = cudaMemset(p, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(allocation-free status word)");
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  }
  *out = h;
  return RCA_OK;
}

}  // namespace

extern "C" rca_status rca_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                           const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                           int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                           rca_dtype dt, void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv)
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_noalloc: null pointer");
  RCA_CHECK(check_shape(B, Hq, Hkv, T, Dh, dt));
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(RCA_ERR_INVALID_ARGUMENT, "rca_attn_bwd_noalloc: tensors must be 16-byte aligned");
  const WsLayout L = ws_layout(B, Hq, Hkv, T, Dh, dt);
  if (L.total > kNoAllocScratchBytes)
    return fail(RCA_ERR_INVALID_ARGUMENT,
                "rca_attn_bwd_noalloc: these sizes need %zu bytes of scratch but the built-in scratch "
                "holds %zu bytes; use rca_attn_bwd with a caller workspace",
                L.total, kNoAllocScratchBytes);
  void* ws = nullptr;
  int* status = nullptr;
  RCA_CHECK(noalloc_setup(&ws, &status));
  cudaStream_t st = static_cast<cudaStream_t>(cuda_stream);
  // The preprocess kernel rewrites every scratch word the later kernels read
  // (it zeroes the dQ accumulator), so leftovers of an earlier call do not matter.
  RCA_CHECK(do_preprocess(out, lse, dout, B, Hq, T, Dh, dt, ws, L, st));
  RCA_CHECK(do_bwd_main(q, k, v, dout, dk, dv, B, Hq, Hkv, T, Dh, dt, ws, L, st, status));
  return do_convert(dq, B, Hq, T, Dh, dt, ws, L, st);
  RCA_GUARD_END
}

// Failure-detection self-test of the allocation-free path: the same bounded
// wait as rca_selftest_device_timeout, recording into the built-in status word.
extern "C" rca_status rca_selftest_noalloc_timeout(void* cuda_stream) {
  RCA_GUARD_BEGIN
  g_err.clear();
  void* ws = nullptr;
  int* status = nullptr;
  RCA_CHECK(noalloc_setup(&ws, &status));
  rca::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(cuda_stream)>>>(status, g_timeout_ns.load());
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch selftest_wait_kernel");
  return RCA_OK;
  RCA_GUARD_END
}
