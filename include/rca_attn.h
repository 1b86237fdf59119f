/*
 * rca_attn.h — C ABI of the GB300 (sm_103a) causal multi-head attention library
 * (librca_attn.so).
 *
 * What it computes. Memory-linear ("Flash") causal self-attention and its
 * vector-Jacobian product, as described by the riftco-transformer pages:
 *   - "Architecture" (docs/concepts/architecture.html), "Tensor conventions":
 *     contiguous row-major storage; scores [B,H,Tq,Tk]; a key at t_k is not
 *     used by a query at t_q when t_k > t_q.
 *   - "Execution Backends and the Python ABI" (docs/internals/backends_and_python.html),
 *     "What the Metal slice does": the Flash path is exact, saves only per-row
 *     [B,H,T] statistics, and its backward recomputes scores and probabilities
 *     from Q, K and those statistics.
 *   - Neural-network page (docs/learn/neural_network.html), "Stable softmax and
 *     cross-entropy": max-subtracted softmax; a fully masked row is rejected.
 *   - algo-v1-codepoint "docs/ARCHITECTURE.md", "config.py": grouped-query
 *     attention requires Hq % Hkv == 0.
 *
 * Per batch b and query head h (KV head kv = h / (Hq/Hkv), consecutive groups):
 *   S[i,j]  = scale * sum_d Q[b,i,h,d] K[b,j,kv,d],   kept for j <= i only
 *   LSE[i]  = ln sum_{j<=i} exp(S[i,j])                 (natural log, fp32)
 *   O[i,:]  = sum_{j<=i} exp(S[i,j] - LSE[i]) V[b,j,kv,:]
 * with scale = 1/sqrt(Dh). The backward, for upstream gradient dO:
 *   D[i]  = sum_d dO[i,d] O[i,d];  P = exp(S - LSE);  dP = dO V^T
 *   dS    = P * (dP - D);  dQ = scale dS K;  dK = scale dS^T Q;  dV = P^T dO
 * dK and dV sum over the query heads that share a KV head.
 *
 * Layouts (all contiguous, row-major, element strides implied by the shape):
 *   q, out, dout, dq : [B, T, Hq,  Dh]   storage dtype
 *   k, v, dk, dv     : [B, T, Hkv, Dh]   storage dtype
 *   lse              : [B, Hq, T]        float32
 * Storage dtype: RCA_BF16 (bfloat16 operands, fp32 accumulation) or
 * RCA_F32_TF32 (float32 storage, fp32 accumulation). In fp32 mode the forward's
 * Q K^T uses TF32 tensor-core operands; the products that contract over key or
 * query positions (P V in the forward, all five backward products) use each
 * fp32 operand split into two bf16 values x = hi + lo and the three products
 * hi.hi + hi.lo + lo.hi, which is at least as accurate as TF32.
 * Supported head widths: Dh in {16, 32, 64, 128} for RCA_BF16 and
 * {16, 32, 64} for RCA_F32_TF32; anything else is RCA_ERR_UNSUPPORTED.
 *
 * Ownership and execution. Every pointer except cuda_stream is a DEVICE pointer
 * owned by the caller (e.g. torch CUDA tensors) that stays valid until the
 * work queued on cuda_stream has finished. Calls only enqueue work on
 * cuda_stream (a cudaStream_t; NULL means the legacy default stream) and
 * return; they never synchronise. Inputs are never written. Outputs are fully
 * overwritten. The library keeps, per device, a small cache of TMA descriptors
 * and one device status word used by the bounded-wait timeout described below.
 * The kernels of the Flash forward and backward (and of the fused-QKV and
 * variable-length calls) are launched with programmatic dependent launch: one
 * may be scheduled onto the GPU while the kernel before it on cuda_stream is
 * still finishing, which hides most of the launch gap between the kernels of a
 * training step. Stream order is unchanged: each such kernel waits, before it
 * reads or writes any memory, until all work queued before it on cuda_stream
 * has completed, and nothing queued after it touches memory before it has
 * completed.
 *
 * Errors. Every argument is validated before anything is launched; on a
 * validation failure nothing is enqueued. No C++ exception crosses this
 * boundary. A failed call returns a non-zero rca_status and records a message
 * retrievable with rca_last_error() on the calling thread. Device-side waits
 * are bounded in time; a kernel that gives up records RCA_ERR_DEVICE_TIMEOUT in
 * the status word, which rca_stream_status() reports.
 *
 * All entry points are thread-safe with respect to one another.
 */
#ifndef RCA_ATTN_H
#define RCA_ATTN_H

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden symbol visibility; the calls declared here
 * are its only exported symbols, so two copies of it (or a program that
 * defines the same internal names) can share a process without interfering. */
#if defined(__GNUC__) && !defined(RCA_API)
#define RCA_API __attribute__((visibility("default")))
#elif !defined(RCA_API)
#define RCA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. Published values are never renumbered. */
typedef enum {
  RCA_OK = 0,
  RCA_ERR_INVALID_ARGUMENT = 1, /* null pointer, bad size, Hq % Hkv != 0, misalignment, small workspace */
  RCA_ERR_UNSUPPORTED = 2,      /* valid request this build does not implement (e.g. Dh = 96) */
  RCA_ERR_CUDA = 3,             /* a CUDA runtime/driver call failed; message holds the CUDA error text */
  RCA_ERR_DEVICE_TIMEOUT = 4,   /* a device-side wait exceeded its time limit; outputs are invalid */
  RCA_ERR_DEVICE_INVALID_INPUT = 5 /* a kernel read an invalid device-side input (page ID, length) */
} rca_status;

/* Storage dtype of q/k/v/out/dout/dq/dk/dv; selects the tensor-core operand type. */
typedef enum { RCA_F32_TF32 = 0, RCA_BF16 = 1 } rca_dtype;

/* ABI version: upper 16 bits major, lower 16 bits minor (0x00010007 = 1.7). */
#define RCA_ABI_VERSION 0x00010008u
RCA_API uint32_t rca_abi_version(void);

/* Message of the last failed call on this thread ("" if none). The pointer is
 * owned by the library and valid until the next call on this thread. */
RCA_API const char* rca_last_error(void);

/*
 * Forward. Writes out [B,T,Hq,Dh] (storage dtype) and lse [B,Hq,T] (float32).
 * Requires B, Hq, Hkv, T >= 1 (T = 0 would be a fully masked row: rejected),
 * Hq % Hkv == 0, and 16-byte aligned q, k, v, out, lse.
 */
RCA_API rca_status rca_attn_fwd(const void* q, const void* k, const void* v,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                        void* out, float* lse, rca_dtype dt, void* cuda_stream);

/*
 * Bytes of device scratch rca_attn_bwd needs for these sizes and dtype: an fp32
 * dQ accumulator [B,T,Hq,Dh], the per-row D and base-2 LSE [B,Hq,Tpad] (Tpad =
 * T rounded up to 128), and for RCA_F32_TF32 bf16 hi/lo copies of Q, dout, K
 * and V. Returns 0 for invalid sizes.
 */
RCA_API size_t rca_attn_bwd_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                   rca_dtype dt);

/*
 * Backward. Given the forward's out and lse and the upstream gradient dout,
 * writes dq [B,T,Hq,Dh], dk and dv [B,T,Hkv,Dh] (storage dtype). workspace is
 * caller-owned device memory of at least rca_attn_bwd_workspace_size(...)
 * bytes, 256-byte aligned; its contents on entry do not matter and are
 * clobbered. Runs rca_attn_bwd_preprocess, rca_attn_bwd_main and
 * rca_attn_bwd_dq_convert in order on cuda_stream.
 */
RCA_API rca_status rca_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                        int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                        rca_dtype dt, void* workspace, size_t workspace_bytes,
                        void* cuda_stream);

/*
 * The three stages of rca_attn_bwd, exposed so a caller can time or schedule
 * them separately. They must run in this order on one stream with the same
 * arguments and workspace.
 *  preprocess: -D = -rowsum(dout * out), -LSE in base 2, zeroes the dQ accumulator
 *              (memory-bound).
 *  main:       recomputes P from Q, K and LSE; accumulates dK, dV per key tile
 *              (written to dk, dv) and adds dQ partials into the workspace.
 *              For RCA_F32_TF32 it first writes the bf16 hi/lo operand copies.
 *  dq_convert: dq = scale * accumulator, cast to the storage dtype.
 */
RCA_API rca_status rca_attn_bwd_preprocess(const void* out, const float* lse, const void* dout,
                                   int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                   rca_dtype dt, void* workspace, size_t workspace_bytes,
                                   void* cuda_stream);
RCA_API rca_status rca_attn_bwd_main(const void* q, const void* k, const void* v, const void* dout,
                             void* dk, void* dv,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                             rca_dtype dt, void* workspace, size_t workspace_bytes,
                             void* cuda_stream);
RCA_API rca_status rca_attn_bwd_dq_convert(void* dq, int64_t B, int64_t Hq, int64_t Hkv, int64_t T,
                                   int64_t Dh, rca_dtype dt, const void* workspace,
                                   size_t workspace_bytes, void* cuda_stream);

/*
 * Backward that allocates nothing (no counterpart on the pages; an addition of
 * this library). Same arguments and results as rca_attn_bwd minus the
 * workspace: its scratch is a 40 MiB array built into the library, for callers
 * that cannot allocate device memory when they call the backward (a plugin
 * interface that passes only input and output buffers, or a latency-bound loop
 * that must never reach cudaMalloc, which can synchronise the device).
 *  - Sizes whose scratch (rca_attn_bwd_workspace_size) exceeds 40 MiB are
 *    rejected with RCA_ERR_INVALID_ARGUMENT before anything is launched.
 *  - The array's 40 MiB are committed on a device when the driver loads this
 *    library's device code there: at context creation with eager module
 *    loading, or, with lazy loading (CUDA's default), at the first launch of
 *    any kernel of this library on that device. A caller that must not see
 *    that happen mid-loop makes one call at initialisation (any accepted size,
 *    e.g. B = Hq = Hkv = T = 1, Dh = 16).
 *  - The first call on a device looks up the array's device address with that
 *    device current; make that first call before any stream capture.
 *  - All calls share the one array and it keeps the last call's contents (each
 *    call rewrites what it reads, so the leftovers never matter). Calls whose
 *    work overlaps on the GPU (other streams, other threads) race on it:
 *    serialise them.
 *  - A device-side timeout in these kernels is recorded in a status word of
 *    the built-in region; rca_stream_status() reports it (and clears it) like
 *    the library's other status word. The kernels end within the wait limit.
 * Never calls cudaMalloc, cudaFree or any allocating routine.
 */
RCA_API rca_status rca_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                rca_dtype dt, void* cuda_stream);

/*
 * Padded / variable-length batches (algo-v1-codepoint "docs/ARCHITECTURE.md",
 * "model.py": rows where no key is allowed are zeroed and must not produce NaN).
 * The batch holds B sequences padded on the right to T positions; sequence b
 * is positions 0 .. seq_lens[b]-1 (0 <= seq_lens[b] <= T; int32, device memory).
 * A padding position is neither a query nor a key:
 *   - real rows (t < seq_lens[b]) equal causal attention over the sequence's
 *     first seq_lens[b] positions (causality alone keeps padding keys out);
 *   - padding rows get out = 0 and lse = -inf; their dq, dk, dv rows are 0;
 *     their dout is ignored; seq_lens[b] = 0 gives an all-zero sequence.
 * Inputs at padding positions are read but cannot affect real outputs as long
 * as they are finite (e.g. zeros): a NaN or Inf there would propagate through
 * the tensor-core products (0 * NaN). A length outside [0, T] is clamped and
 * recorded as RCA_ERR_DEVICE_INVALID_INPUT. Tiles of 128 positions made only of
 * padding are not computed: both calls first plan the work from seq_lens on the
 * device, and the rows of those tiles are written as zeros.
 * workspace: at least rca_attn_varlen_workspace_size(...) bytes for either call
 * (the backward's scratch plus the work lists), 256-byte aligned, contents on
 * entry irrelevant. B <= 4096 and T <= 131072 (else RCA_ERR_UNSUPPORTED). Same
 * layouts, dtypes, head widths and errors as rca_attn_fwd / rca_attn_bwd otherwise.
 */
RCA_API size_t rca_attn_varlen_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt);
RCA_API rca_status rca_attn_fwd_varlen(const void* q, const void* k, const void* v, const int32_t* seq_lens,
                               int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                               void* out, float* lse, rca_dtype dt,
                               void* workspace, size_t workspace_bytes, void* cuda_stream);
RCA_API rca_status rca_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* out, const float* lse,
                               const void* dout, const int32_t* seq_lens, void* dq, void* dk, void* dv,
                               int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh, rca_dtype dt,
                               void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Fused QKV layout (an addition around the pages' operation: the pages project
 * query, key and value with three Linear layers, then split heads, attend,
 * merge heads and apply the output projection — "Neural network" page, "Where
 * attention is"). Here q, k and v are read in place from one fused projection
 * output and the gradients are written in place into one buffer of the same
 * shape, so neither direction needs a split or a concatenation copy:
 *   qkv, dqkv : [B, T, (Hq + 2*Hkv) * Dh], per position q heads 0..Hq-1, then
 *               k heads, then v heads, each Dh wide (storage dtype)
 *   out, dout : [B, T, Hq * Dh]  (= [B, T, Hq, Dh], the merged heads)
 *   lse       : [B, Hq, T] float32
 * Same computation, dtypes, head widths, errors and workspace
 * (rca_attn_bwd_workspace_size) as rca_attn_fwd / rca_attn_bwd. 16-byte aligned.
 */
RCA_API rca_status rca_attn_fwd_qkv(const void* qkv, int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t Dh,
                            void* out, float* lse, rca_dtype dt, void* cuda_stream);
RCA_API rca_status rca_attn_bwd_qkv(const void* qkv, const void* out, const float* lse, const void* dout, void* dqkv,
                            int64_t B, int64_t T, int64_t Hq, int64_t Hkv, int64_t Dh, rca_dtype dt,
                            void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Materialized causal attention and its probability-returning diagnostic
 * ("Execution Backends and the Python ABI", docs/internals/backends_and_python.html,
 * section "What the Metal slice does": the default materialized request
 * returns probabilities and context and keeps the [batch, heads, time, time]
 * probabilities for its VJPs; the diagnostic that returns probabilities always
 * uses it; causal softmax scales, masks and normalises in one operation).
 *
 * Forward, per batch b and query head h (KV head kv = h / (Hq/Hkv)):
 *   S = scale * Q K^T (scale = 1/sqrt(Dh));  probs[b,h,i,j] = exp(S[i,j] - lse[b,h,i])
 *   for j <= i and 0 for j > i;  out = probs V.
 * Backward, for upstream gradients dout of out and dprobs of probs (dprobs may
 * be NULL, meaning zero):
 *   dP = dout V^T + dprobs;  dS = probs * (dP - rowsum(probs * dP));
 *   dq = scale dS K;  dk = scale dS^T Q;  dv = probs^T dout  (dk, dv summed over
 *   the query heads of a KV head). The backward reads the probabilities the
 *   forward stored; it does not recompute them. The forward forms S twice on
 *   the tensor cores instead of storing it (pass 1: row statistics, giving
 *   lse; pass 2: probs written from S and lse), then computes out from the
 *   stored probs.
 *
 * Layouts: q, out, dout, dq [B,T,Hq,Dh] and k, v, dk, dv [B,T,Hkv,Dh] in the
 * storage dtype (as rca_attn_fwd); probs, dprobs [B,Hq,T,T] float32 (4*B*Hq*T*T
 * bytes: 1 GiB for B=4, Hq=16, T=2048); lse [B,Hq,T] float32. Dh in {16, 32, 64,
 * 128} for both dtypes. Only the causal triangle is computed: score tiles
 * above the diagonal are never formed and the products over T read only the
 * kept triangle of probs (or dS). Arithmetic: tensor-core products with fp32
 * accumulation. RCA_BF16: the products over Dh take the stored bf16 values
 * (exact products), those over T take probs or dS as two bf16 parts hi + lo
 * (relative representation error ~2^-17). RCA_F32_TF32: Q, K, V, dO enter as
 * three bf16 parts each (scores to fp32 accuracy), probs or dS as two. All
 * tensors 16-byte aligned. workspace: at least
 * rca_attn_materialized_workspace_size(...) bytes (the same size serves both
 * calls), 256-byte aligned, contents on entry irrelevant. Every pointer is a
 * device pointer owned by the caller; calls validate, then only enqueue work
 * on cuda_stream. Device waits are time-bounded like the other kernels'
 * (RCA_ERR_DEVICE_TIMEOUT through rca_stream_status).
 */
RCA_API size_t rca_attn_materialized_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                            rca_dtype dt);
RCA_API rca_status rca_attn_materialized_fwd(const void* q, const void* k, const void* v,
                                     int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                     void* out, float* probs, float* lse, rca_dtype dt,
                                     void* workspace, size_t workspace_bytes, void* cuda_stream);
RCA_API rca_status rca_attn_materialized_bwd(const void* q, const void* k, const void* v, const float* probs,
                                     const void* dout, const float* dprobs,
                                     void* dq, void* dk, void* dv,
                                     int64_t B, int64_t Hq, int64_t Hkv, int64_t T, int64_t Dh,
                                     rca_dtype dt, void* workspace, size_t workspace_bytes,
                                     void* cuda_stream);

/*
 * The fused causal softmax of the materialized path, and its VJP, on N
 * independent row-major [T, T] float32 score matrices (one per batch and head),
 * in place ("Execution Backends and the Python ABI", "What the Metal slice
 * does": causal softmax combines scaling, masking and normalisation in one
 * kernel; Neural-network page, "Stable softmax and cross-entropy":
 * max-subtracted softmax):
 *   forward   scores[n,i,j] <- exp(scale*scores[n,i,j] - lse[n,i]) for j <= i,
 *             0 for j > i;  lse[n,i] = ln sum_{j<=i} exp(scale*scores[n,i,j])
 *   backward  with G = grad + grad_extra (grad_extra may be NULL):
 *             grad[n,i,j] <- scale * probs[n,i,j] * (G[n,i,j] - sum_k probs[n,i,k] G[n,i,k])
 *             for j <= i, 0 for j > i (the gradient of the unscaled scores).
 * Device pointers, 16-byte aligned; lse is [N, T]; 1 <= T <= 65536; scale finite.
 */
RCA_API rca_status rca_causal_softmax(float* scores, float* lse, int64_t N, int64_t T, float scale, void* cuda_stream);
RCA_API rca_status rca_causal_softmax_bwd(const float* probs, float* grad, const float* grad_extra, int64_t N, int64_t T,
                                  float scale, void* cuda_stream);
/*
 * The same VJP restricted to the causal tiles of a tiled consumer: row i is
 * read and written only for columns j < min(T, tile * (floor(i / tile) + 1)),
 * i.e. its tiles of `tile` columns on or left of the diagonal (entries above
 * the diagonal inside the diagonal tile are written as 0); the rest of the
 * row, in grad and grad_extra, is neither read nor written. tile >= T is
 * rca_causal_softmax_bwd. The materialized backward applies it with tile 128
 * to its dP workspace, whose products read only those tiles. tile >= 1, else
 * RCA_ERR_INVALID_ARGUMENT; other arguments and errors as above. (ABI 1.8)
 */
RCA_API rca_status rca_causal_softmax_bwd_tiled(const float* probs, float* grad, const float* grad_extra, int64_t N,
                                                int64_t T, int64_t tile, float scale, void* cuda_stream);

/*
 * Paged decode attention ("Execution Backends and the Python ABI",
 * docs/internals/backends_and_python.html, section "Incremental attention"):
 * one new query token per request attends over every position the request has
 * cached, each key and value fetched through the request's page table. Query
 * and output are [H, d_h] per request; the key and value pools are
 * [physical_page, H, page_offset, d_h]; a request-local table maps logical page
 * j (positions j*page_size .. j*page_size + page_size - 1) to a physical page
 * ID. The operation is inference-only: it has no backward.
 *
 * Per request b (length L = seq_lens[b]) and query head h, with KV head
 * kv = h / (Hq/Hkv) and K[t] = k_pool[page_table[b][t / page_size], kv,
 * t % page_size, :] (likewise V):
 *   s_t    = scale * q[b,h,:] . K[t],   t = 0 .. L-1,  scale = 1/sqrt(Dh)
 *   lse[b,h] = ln sum_t exp(s_t)                       (natural log, fp32)
 *   out[b,h,:] = sum_t exp(s_t - lse[b,h]) V[t]
 * The new token's own key and value must already be in the cache (position
 * L-1), so every request attends to at least one position.
 *
 * Layouts (contiguous, row-major):
 *   q, out            : [B, Hq, Dh]                          storage dtype
 *   k_pool, v_pool    : [num_pages, Hkv, page_size, Dh]      storage dtype
 *   page_table        : [B, max_pages] int32 physical page IDs (entries past a
 *                       request's last page are never read)
 *   seq_lens          : [B] int32
 *   lse               : [B, Hq] float32
 * RCA_BF16: bfloat16 storage; RCA_F32_TF32: float32 storage. Arithmetic is
 * fp32 on the stored values: float32 storage and bf16 with one query head per
 * KV head on the CUDA cores; bf16 with Hq/Hkv >= 2 on the tensor cores (exact
 * bf16 products with fp32 accumulation, probabilities entering the P*V product
 * as a bf16 hi + lo pair, so still ~fp32-accurate). Dh in {16, 32, 64, 128};
 * page_size a power of two in [1, 65536]; 1 <= B <= 8192;
 * max_pages * page_size <= 2^30. q, k_pool and v_pool 16-byte aligned,
 * page_table, seq_lens and lse 4-byte aligned.
 *
 * Device-side inputs (page_table, seq_lens) are checked by the kernels as they
 * read them: a page ID outside [0, num_pages) is never dereferenced and a length
 * outside [1, max_pages * page_size] makes that request's out and lse NaN; both
 * record RCA_ERR_DEVICE_INVALID_INPUT for rca_stream_status(). Other requests'
 * results are unaffected by a bad length; a bad page ID leaves its request's
 * results invalid.
 *
 * workspace: caller-owned device memory of at least
 * rca_paged_decode_workspace_size(...) bytes (>= 256 for valid sizes, 0 for
 * invalid ones), 256-byte aligned: fp32 partial results of requests longer than
 * 256 positions; contents on entry do not matter. All pointers are device
 * pointers owned by the caller; the call validates its host arguments (nothing
 * is enqueued on failure) and then only enqueues work on cuda_stream.
 */
RCA_API size_t rca_paged_decode_workspace_size(int64_t B, int64_t Hq, int64_t Hkv, int64_t Dh,
                                       int64_t page_size, int64_t max_pages, rca_dtype dt);
RCA_API rca_status rca_paged_decode(const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* page_table, const int32_t* seq_lens,
                            int64_t B, int64_t Hq, int64_t Hkv, int64_t Dh,
                            int64_t page_size, int64_t max_pages, int64_t num_pages,
                            void* out, float* lse, rca_dtype dt,
                            void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Synchronises cuda_stream, then reports (and clears) an asynchronous CUDA
 * error, a device-side timeout (RCA_ERR_DEVICE_TIMEOUT) or an invalid
 * device-side input (RCA_ERR_DEVICE_INVALID_INPUT) recorded by a kernel of this
 * library on the current device, the allocation-free backward's included.
 * RCA_OK if none happened.
 */
RCA_API rca_status rca_stream_status(void* cuda_stream);

/*
 * Failure-detection self-test (no counterpart on the pages). Enqueues a small
 * kernel that waits, with the same time-bounded wait the attention kernels
 * use, on a barrier that nothing ever completes. After the current wait limit
 * (rca_set_wait_timeout_ns) the kernel gives up and records a timeout, so the
 * next rca_stream_status() on this stream returns RCA_ERR_DEVICE_TIMEOUT (and
 * clears it); the CUDA context remains usable. Nothing faults or hangs.
 */
RCA_API rca_status rca_selftest_device_timeout(void* cuda_stream);

/*
 * The same self-test for the allocation-free backward's status word: the
 * waiting kernel records its timeout where rca_attn_bwd_noalloc's kernels do,
 * and the next rca_stream_status() returns RCA_ERR_DEVICE_TIMEOUT. Sets up the
 * built-in region on the current device like a first rca_attn_bwd_noalloc call.
 */
RCA_API rca_status rca_selftest_noalloc_timeout(void* cuda_stream);

/*
 * Sets the device-side wait limit in nanoseconds for subsequent launches from
 * any thread (default 2e9 = 2 s; values < 1e6 are raised to 1e6). Returns the
 * previous value.
 */
RCA_API uint64_t rca_set_wait_timeout_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* RCA_ATTN_H */
