// Causal attention forward for sm_103a.
//
// Computes, per (batch b, query head h, 128-row query tile), the exact
// memory-linear ("Flash") forward described on the riftco-transformer page
// "Execution Backends and the Python ABI", section "What the Metal slice does":
// O and the per-row statistic LSE = m + ln(l) are produced without a [T,T]
// buffer. The mask is the one of the "Architecture" page, "Tensor conventions"
// (key t_k dropped when t_k > t_q); the softmax is max-subtracted as on the
// neural-network page, "Stable softmax and cross-entropy".
//
// Work items are (batch, head, 128-row query tile); key tiles 0..qt are
// visited, tile qt being the diagonal one.
//
// CTA layout (512 threads, four warpgroups with their own register budgets):
//   warp 0        TMA producer: per work item the Q tile, then K_t / V_t into
//                 NSK / NSV-stage rings
//   warp 1        single-thread issuer of S_t = Q K_t^T
//   warp 2        single-thread issuer of the P V products
//   warp 3        TMEM owner
//   warps 4..11   two softmax warpgroups (thread i of a warpgroup owns query row i)
//   warps 12..15  epilogue warpgroup (persistent mode): per work item it merges
//                 the two softmax warpgroups' statistics and partials and
//                 stores O and LSE, while the softmax warpgroups already work
//                 on the next item
// Two issuers on different SM sub-partitions keep the tensor pipe fed: each
// has half the instructions, and neither waits for the other's events.
//
// bf16 storage ("ping-pong"): warpgroup g takes the key tiles t with t % 2 == g
// (t counts key tiles across all of a CTA's work items): it reads the full
// 128-key row of S_t from TMEM S buffer g, and O_g += P_t V_t accumulates its
// tiles. While it works on tile t the scores of tile t + 2 are computed, and
// the other warpgroup works on tile t + 1, so one warpgroup's exponentials
// overlap the other's waits. Each warpgroup keeps its own running max m_g and
// sum l_g (base-2 units); O_g is rescaled only when m_g grows by more than 2^8
// (exact: l_g uses the same reference). The partials are merged once per item:
// O = sum_g 2^(m_g - m) O_g / sum_g 2^(m_g - m) l_g.
// With a head width <= 64, P_t stays in TMEM and the P V product reads it from
// there (A operand in TMEM): shared-memory bandwidth, which the TMA writes,
// register stores and the tensor core's operand reads all share, then carries
// only Q, K and V. Wider heads stage P in shared memory (bf16, K-major,
// 128-byte swizzle, one buffer per warpgroup).
// Persistent launch (bf16 storage): one CTA per SM walks several work items
// in the order that balances the SMs; the next item's K tiles and first
// scores (and, with TMEM-resident P, its query tile) are fetched and computed
// while the current item's epilogue merges and stores its output.
// fp32 storage mode: both warpgroups take every key tile, warpgroup g keys
// 64 g .. 64 g + 63 of it, with O_g accumulated from its half of the keys.
// S = Q K^T runs as kind::tf32 on the fp32 tiles (the head dimension is
// contiguous, so both operands are K-major). P V contracts over
// keys, which needs V as an MN-major operand; kind::tf32 produced no result
// with MN-major operands on this GPU, so P and V are split into bf16 pairs
// x = hi + lo and O_g += Phi Vhi + Phi Vlo + Plo Vhi (relative error ~2^-16,
// below TF32's 2^-11).
#pragma once

#include "tc.cuh"

namespace rca {

template <bool TF32, int DHP>
struct FwdCfg {
  // Warpgroups (4 warps each): 0 = TMA producer (warp 0), S = Q K^T issuer
  // (warp 1), P V issuer (warp 2), TMEM owner (warp 3); 1 and 2 = softmax;
  // 3 = epilogue (persistent mode; idle otherwise). Registers are split per
  // warpgroup from the 128 per thread the CTA is launched with.
  static constexpr int NTHREADS = 512;
  static constexpr int LAUNCH_REGS = 128;
  static constexpr int REG_CTL = 96, REG_SM = 168, REG_EPI = 80;
  static_assert(128 * REG_CTL + 256 * REG_SM + 128 * REG_EPI <= NTHREADS * LAUNCH_REGS, "register split");
  // bf16 storage: the two softmax warpgroups alternate whole key tiles
  // ("ping-pong"); fp32 storage: they split every key tile in halves.
  static constexpr bool PP = !TF32;
  // Head width <= 64 (bf16): P_j stays in tensor memory (P V runs with A read
  // from TMEM), so it costs no shared-memory bandwidth, which on this part is
  // shared by TMA writes, register stores and the tensor core's operand reads.
  static constexpr bool PT = PP && DHP <= 64;
  // bf16 storage: persistent CTAs (one per SM) walk several work items and
  // hand each item's merge and output to the epilogue warpgroup, so the
  // softmax warpgroups go straight on to the next item.
  static constexpr bool EPI_WG = PP;
  static constexpr int ES = TF32 ? 4 : 2;     // storage bytes per element
  static constexpr int PE = 128 / ES;         // elements per 128-byte swizzle row
  static constexpr int BM = 128, BN = 128;    // query rows, keys per tile
  static constexpr int PANEL = 128 * 128;     // one 128-row x 128-byte panel
  static constexpr int DPANELS = DHP / PE;    // panels across the head width
  static constexpr int Q_BYTES = DPANELS * PANEL;
  // Persistent CTAs with TMEM-resident P double-buffer Q so the next work
  // item's query tile loads while the current one is still in use; at head
  // width 128 (P staged in shared memory) only one Q buffer fits beside two
  // K/V stages, and the next item's Q loads once the last S of the current
  // item is done.
  static constexpr int QB = PT ? 2 : 1;
  static constexpr int KV_BYTES = DPANELS * PANEL;
  static constexpr int KSTEP = TF32 ? 8 : 16;  // K of one QK^T MMA instruction
  static constexpr int SPP = PE / KSTEP;       // QK^T k-steps per panel
  // P.V operands. bf16 mode: P (bf16) and the V stage itself. fp32 mode: P and
  // V as bf16 hi/lo pairs (x = hi + lo), V converted from its fp32 stage into
  // a DHB-column bf16 tile (zero-padded past the head width).
  static constexpr int DHB = TF32 ? (DHP > 64 ? DHP : 64) : DHP;
  static constexpr int VB_PANELS = DHB / 64;
  static constexpr int VHL_BYTES = TF32 ? 2 * VB_PANELS * PANEL : 0;
  static constexpr int P_HALF = 2 * PANEL;                    // 128 x 128 bf16
  // bf16 mode: one P buffer per warpgroup (full 128 keys); fp32 mode (hi + lo)
  // keeps one buffer shared by the two key halves.
  static constexpr int P_BUFS = TF32 ? 1 : 2;
  static constexpr int P_BUF = TF32 ? 2 * P_HALF : P_HALF;    // one buffer: hi (+ lo)
  static constexpr int P_BYTES = PT ? 0 : P_BUFS * P_BUF;
  // Merge statistics m[2][128], l[2][128] (2 KB per set). Persistent CTAs keep
  // them in a region of their own: two sets (by work-item parity) with
  // TMEM-resident P, one at head width 128; otherwise they reuse the P buffer,
  // dead once the CTA's only work item is finished.
  static constexpr int STAT_SETS = PT ? 2 : 1;
  static constexpr int STATX_BYTES = EPI_WG ? 2048 * STAT_SETS : 0;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int BAR_BYTES = EPI_WG && !PT ? 512 : 1024;
  // The dynamic shared memory of a block starts 1024-aligned (the first 1 KB
  // of a block's shared memory is reserved by the hardware); the persistent
  // head-width-128 layout uses the alignment slack the others keep, and the
  // kernel checks the alignment at run time instead (error, no access).
  static constexpr int SLACK = EPI_WG && !PT ? 0 : 1024;
  static constexpr int AVAIL = SMEM_LIMIT - SLACK - BAR_BYTES - QB * Q_BYTES - P_BYTES - VHL_BYTES - STATX_BYTES;
  static constexpr int NS_BF = AVAIL / (2 * KV_BYTES) > 4 ? 4 : AVAIL / (2 * KV_BYTES);
  static constexpr int NSV = TF32 ? (AVAIL >= 4 * KV_BYTES ? 2 : 1) : NS_BF;
  static constexpr int NSK_FIT = TF32 ? (AVAIL - NSV * KV_BYTES) / KV_BYTES : NS_BF;
  static constexpr int NSK = NSK_FIT > 4 ? 4 : NSK_FIT;
  static_assert(NSK >= 2 && NSV >= 1, "forward needs at least two K stages and one V stage");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + QB * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NSV * KV_BYTES;
  static constexpr int OFF_VHL = OFF_P + P_BYTES;
  static constexpr int OFF_STATX = OFF_VHL + VHL_BYTES;
  static constexpr int OFF_BAR = OFF_STATX + STATX_BYTES;
  static constexpr int OFF_STAT = EPI_WG ? OFF_STATX : OFF_P;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + SLACK;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  static constexpr int TMEM_S = 0;          // two buffers: columns [0,128) and [128,256)
  static constexpr int TMEM_O = 256;        // O_0 at [256, 256+DHB), O_1 after it
  static constexpr int TMEM_P = TMEM_O + 2 * DHB;  // PT: P buffer g (64 columns of bf16 pairs)
  static constexpr int TMEM_COLS = 512;
  static_assert(TMEM_O + 2 * DHB + (PT ? 128 : 0) <= TMEM_COLS, "TMEM budget");
  static constexpr uint32_t IDESC_QK = make_idesc(TF32, 128, 128, false, false);
  static constexpr uint32_t IDESC_PV = make_idesc(false, 128, DHB, false, true);  // bf16 operands
  // barrier slots
  static constexpr int B_QF = 0;            // [QB] query tile landed
  static constexpr int B_QE = B_QF + QB;    // [QB] query buffer free (last S of its item done)
  static constexpr int B_KF = B_QE + QB;
  static constexpr int B_KE = B_KF + NSK;
  static constexpr int B_VF = B_KE + NSK;
  static constexpr int B_VE = B_VF + NSV;
  static constexpr int B_SF = B_VE + NSV;   // [2] S buffer full
  static constexpr int B_SFREE = B_SF + 2;  // [2] S buffer read by both warpgroups
  // [2 halves][2 tile parities] P half g written. One barrier per tile parity:
  // a softmax warpgroup may finish tile j+1 before the MMA thread has consumed
  // tile j's arrival, and a single barrier would then be two phases ahead.
  static constexpr int B_PF = B_SFREE + 2;
  static constexpr int B_OD = B_PF + 4;     // [2 halves][2 parities] P V half done
  static constexpr int B_ITEMD = B_OD + 4;  // every P V product of a work item done
  static constexpr int B_OFREE = B_ITEMD + 1;  // O partials read by the epilogue
  // [2 item parities] merge statistics written (256 softmax arrivals) / read by
  // the epilogue warpgroup (128 arrivals). One barrier per parity: on short
  // items a side may run a whole item ahead of the other.
  static constexpr int B_STAT = B_OFREE + 1;
  static constexpr int B_STATFREE = B_STAT + 2;
  static constexpr int B_FIN = B_STATFREE + 2;   // [2] exit: S issuer's / P V issuer's MMAs done
  static constexpr int NBAR = B_FIN + 2;
  static_assert(8 * NBAR + 8 <= BAR_BYTES, "barrier area");
};

struct FwdArgs {
  void* out;
  float* lse;
  const int* lens;  // per-sequence lengths (right padding), or null: rows t >= lens[b] are padding
  const int4* items;     // variable-length batches: work list {b, h, qt, -} (null: all items)
  const int* n_items_dev;  // its length (device)
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, Dh, group, n_qt;
  int n_items;       // B * Hq * n_qt work items (one query tile of one head each)
  float scale_log2;  // (1/sqrt(Dh)) * log2(e)
};

// Work item k (k = 0, 1, ...) of this CTA. Items are ordered by decreasing
// key-tile count (the last query tile of every head first) and dealt out in a
// snake over the grid: round k gives item k G + c (k even) or k G + G - 1 - c
// (k odd), G CTAs, c this CTA. With one CTA per item the loop runs once.
struct FwdItem {
  int b, h, kvh, qt, nkv;
};

// Length of sequence b of a variable-length batch, clamped to [0, T]; a value
// outside that range is recorded as a bad device-side input.
__device__ __forceinline__ int seq_len(const FwdArgs& a, int b) {
  const int L = __ldg(a.lens + b);
  if (L >= 0 && L <= a.T) return L;
  atomicExch(a.status, kStatusBadInput);
  return L < 0 ? 0 : a.T;
}
template <bool LIST>
__device__ __forceinline__ bool fwd_item(const FwdArgs& a, int k, FwdItem& it) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const long long idx = static_cast<long long>(k) * G + ((k & 1) ? (G - 1 - c) : c);
  if constexpr (LIST) {  // variable-length batch: the planned list (tiles of padding left out)
    if (idx >= __ldg(a.n_items_dev)) return false;
    const int4 e = __ldg(a.items + idx);
    it.b = e.x;
    it.h = e.y;
    it.qt = e.z;
    it.nkv = it.qt + 1;
    it.kvh = it.h / a.group;
    return true;
  }
  if (idx >= a.n_items) return false;
  const int bh_count = a.B * a.Hq;
  const int level = static_cast<int>(idx / bh_count), bh = static_cast<int>(idx % bh_count);
  it.qt = a.n_qt - 1 - level;
  it.nkv = it.qt + 1;
  it.b = bh / a.Hq;
  it.h = bh % a.Hq;
  it.kvh = it.h / a.group;
  return true;
}

// fp32 mode: split rows [64 g, 64 g + 64) of the fp32 V stage (MN-major,
// 32-element panels) into bf16 hi/lo tiles (MN-major, 64-element panels). Two
// threads per key row, each taking every other 8-column group; head columns
// past DHP are written as zeros.
template <class C>
__device__ __forceinline__ void split_v_half(uint32_t vsrc, uint32_t vhi, uint32_t vlo, int g, int t) {
  const int row = 64 * g + (t & 63);
  const uint32_t sw = row & 7;
#pragma unroll
  for (int gg = 0; gg < C::DHB / 16; ++gg) {
    const int grp = 2 * gg + (t >> 6);
    const uint32_t dst = (grp >> 3) * C::PANEL + row * 128 + (((grp & 7) ^ sw) << 4);
    if (grp < C::DPANELS * 4) {
      const uint32_t pf = grp >> 2;  // fp32 panel
      const uint32_t c0 = (2 * grp) & 7, c1 = c0 + 1;
      const uint32_t base = vsrc + pf * C::PANEL + row * 128;
      float x[8];
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]) : "r"(base + ((c0 ^ sw) << 4)));
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(x[4]), "=f"(x[5]), "=f"(x[6]), "=f"(x[7]) : "r"(base + ((c1 ^ sw) << 4)));
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) split_bf16x2(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
      st_shared_v4(vhi + dst, hi[0], hi[1], hi[2], hi[3]);
      st_shared_v4(vlo + dst, lo[0], lo[1], lo[2], lo[3]);
    } else {
      st_shared_v4(vhi + dst, 0u, 0u, 0u, 0u);
      st_shared_v4(vlo + dst, 0u, 0u, 0u, 0u);
    }
  }
}

template <bool TF32, int DHP, bool LIST>
__global__ void __launch_bounds__(512, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<TF32, DHP>;
  grid_dep_sync();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  if constexpr (C::SLACK == 0) {
    // No alignment slack in this layout: a misaligned base is reported, never used.
    if (raw & 1023u) {
      if (threadIdx.x == 0) atomicExch(a.status, kStatusLayout);
      return;
    }
  }
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // A CTA past the end of a planned work list has no item at all.
  if constexpr (LIST) {
    if (static_cast<int>(blockIdx.x) >= __ldg(a.n_items_dev)) return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::QB; ++i) {
      mbar_init(bar(C::B_QF + i), 1);
      mbar_init(bar(C::B_QE + i), 1);
    }
    for (int s = 0; s < C::NSK; ++s) {
      mbar_init(bar(C::B_KF + s), 1);
      mbar_init(bar(C::B_KE + s), 1);
    }
    for (int s = 0; s < C::NSV; ++s) {
      mbar_init(bar(C::B_VF + s), 1);
      mbar_init(bar(C::B_VE + s), TF32 ? 256 : 1);  // fp32: released by the converting warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_SF + i), 1);
      mbar_init(bar(C::B_SFREE + i), C::PP ? 128 : 256);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(C::B_PF + i), 128);
      mbar_init(bar(C::B_OD + i), 1);
    }
    mbar_init(bar(C::B_ITEMD), 1);
    mbar_init(bar(C::B_OFREE), C::EPI_WG ? 128 : 256);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_STAT + i), 256);
      mbar_init(bar(C::B_STATFREE + i), 128);
    }
    mbar_init(bar(C::B_FIN), 1);
    mbar_init(bar(C::B_FIN + 1), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 3) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{a.status, abort_flag, a.timeout_ns};
  // Every role ends in end_role(): the TMEM owner (warp 3) waits until all
  // 512 threads have finished with TMEM and releases it; the others only
  // arrive. No code follows the role branches (each warpgroup runs with its
  // own register budget).
  auto end_role = [&]() {
    tc_fence_before();
    if (warp == 3) {
      named_bar(1, C::NTHREADS);
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    } else {
      named_bar_arrive(1, C::NTHREADS);
    }
  };

  // Every role walks the same sequence of work items; key tiles are numbered
  // t = 0, 1, ... across all of this CTA's items, and every ring position and
  // barrier phase below is a function of t (or of the item number n).
  if (warp < 4) {
   reg_dealloc<C::REG_CTL>();
   if (warp == 0) {
    // ---------------- TMA producer (one elected thread) ----------------
    if (elect_one()) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      // Loads follow the order in which the MMA issuer consumes them: with
      // ping-pong (bf16) S_t is issued right after P_{t-3} V_{t-3}, so K runs
      // three tiles ahead of V; otherwise K_t and V_t alternate. A work item's
      // query tile is loaded just before its first K tile.
      constexpr int KLEAD = C::PP ? 3 : 1;
      FwdItem ik{}, iv{};
      int kn = 0, kj = 0, tk = 0;  // K cursor: item, tile within it, tiles loaded
      int vn = 0, vj = 0, tv = 0;  // V cursor
      int nq = 0;                  // query tiles loaded
      bool khave = fwd_item<LIST>(a, 0, ik), vhave = fwd_item<LIST>(a, 0, iv);
      bool ok = true;
      auto load_k = [&]() -> bool {
        if (kj == 0) {
          const int qb = kn % C::QB;
          if (kn >= C::QB && !mbar_wait(bar(C::B_QE + qb), ((kn / C::QB) - 1) & 1, w)) return false;
          mbar_expect_tx(bar(C::B_QF + qb), C::Q_BYTES);
          for (int p = 0; p < C::DPANELS; ++p)
            tma_load_4d(sbase + C::OFF_Q + qb * C::Q_BYTES + p * C::PANEL, &tmQ, bar(C::B_QF + qb), p * C::PE,
                        ik.h, ik.qt * C::BM, ik.b);
          ++nq;
        }
        const int sk = tk % C::NSK;
        if (tk >= C::NSK && !mbar_wait(bar(C::B_KE + sk), ((tk / C::NSK) - 1) & 1, w)) return false;
        mbar_expect_tx(bar(C::B_KF + sk), C::KV_BYTES);
        for (int p = 0; p < C::DPANELS; ++p)
          tma_load_4d(sbase + C::OFF_K + sk * C::KV_BYTES + p * C::PANEL, &tmK, bar(C::B_KF + sk), p * C::PE,
                      ik.kvh, kj * C::BN, ik.b);
        ++tk;
        if (++kj == ik.nkv) {
          kj = 0;
          khave = fwd_item<LIST>(a, ++kn, ik);
        }
        return true;
      };
      while (ok && khave && tk < KLEAD) ok = load_k();
      while (ok && vhave) {
        const int sv = tv % C::NSV;
        if (tv >= C::NSV && !mbar_wait(bar(C::B_VE + sv), ((tv / C::NSV) - 1) & 1, w)) break;
        mbar_expect_tx(bar(C::B_VF + sv), C::KV_BYTES);
        for (int p = 0; p < C::DPANELS; ++p)
          tma_load_4d(sbase + C::OFF_V + sv * C::KV_BYTES + p * C::PANEL, &tmV, bar(C::B_VF + sv), p * C::PE,
                      iv.kvh, vj * C::BN, iv.b);
        ++tv;
        if (++vj == iv.nkv) {
          vj = 0;
          vhave = fwd_item<LIST>(a, ++vn, iv);
        }
        if (khave) ok = load_k();
      }
      // Exit path: every load issued has landed before shared memory is
      // released (immediate unless a wait above gave up).
      for (int s = 0; s < C::QB && s < nq; ++s) {
        const int last = s + ((nq - 1 - s) / C::QB) * C::QB;
        mbar_drain(bar(C::B_QF + s), (last / C::QB) & 1, a.timeout_ns);
      }
      for (int s = 0; s < C::NSK && s < tk; ++s) {
        const int last = s + ((tk - 1 - s) / C::NSK) * C::NSK;
        mbar_drain(bar(C::B_KF + s), (last / C::NSK) & 1, a.timeout_ns);
      }
      for (int s = 0; s < C::NSV && s < tv; ++s) {
        const int last = s + ((tv - 1 - s) / C::NSV) * C::NSV;
        mbar_drain(bar(C::B_VF + s), (last / C::NSV) & 1, a.timeout_ns);
      }
    }
    __syncwarp();
   } else if (warp == 1) {
    // ---------------- S = Q K^T issuer (one elected thread) ----------------
    // Shared-memory descriptors are built once and advanced by constant
    // offsets (the address field holds address / 16; every address here stays
    // below 256 KB, so the addition never carries out of the field). S_t goes
    // to S buffer t % 2 as soon as K_t has landed and the buffer's previous
    // scores (tile t - 2) have been read by the softmax warps.
    if (elect_one()) {
      bool ok = true;
      const uint64_t dq0 = make_sdesc(sbase + C::OFF_Q, 16, 1024);
      const uint64_t dk0 = make_sdesc(sbase + C::OFF_K, 16, 1024);
      FwdItem is{};
      int sn = 0, sj = 0, ts = 0;  // item, tile within it, global tile
      bool shave = fwd_item<LIST>(a, 0, is);
      while (ok && shave) {
        const int qb = sn % C::QB;
        const int sk = ts % C::NSK;
        const int sb = ts & 1;
        if (sj == 0 && !mbar_wait(bar(C::B_QF + qb), (sn / C::QB) & 1, w)) break;
        if (!mbar_wait(bar(C::B_KF + sk), (ts / C::NSK) & 1, w)) break;
        if (ts >= 2 && !mbar_wait(bar(C::B_SFREE + sb), ((ts - 2) >> 1) & 1, w)) break;
        tc_fence_after();
        const uint64_t dq = dq0 + qb * (C::Q_BYTES >> 4);
        const uint64_t dk = dk0 + sk * (C::KV_BYTES >> 4);
        const uint32_t dst = tmem + C::TMEM_S + sb * 128;
#pragma unroll
        for (int k = 0; k < DHP / C::KSTEP; ++k) {
          const uint32_t off = ((k / C::SPP) * C::PANEL + (k % C::SPP) * 32) >> 4;
          mma_ss<TF32>(dst, dq + off, dk + off, C::IDESC_QK, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF + sb));
        tc_commit(bar(C::B_KE + sk));
        ++ts;
        if (++sj == is.nkv) {
          tc_commit(bar(C::B_QE + qb));  // last S of the item: its query buffer is free
          sj = 0;
          shave = fwd_item<LIST>(a, ++sn, is);
        }
      }
      // Exit path: all issued MMAs finish before TMEM is released.
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
    __syncwarp();
   } else if (warp == 2) {
    // ---------------- P V issuer (one elected thread) ----------------
    if (elect_one()) {
      bool ok = true;
      const uint64_t dv0 = make_sdesc(sbase + C::OFF_V, C::PANEL, 1024);
      const uint64_t dp0 = make_sdesc(sbase + C::OFF_P, 16, 1024);
      FwdItem ip{};
      int pn = 0, pj = 0, tp = 0;  // item, tile within it, global tile
      bool phave = fwd_item<LIST>(a, 0, ip);
      while (ok && phave) {
        // Before the first product of work item n >= 1 the epilogue of item
        // n - 1 must have read the O partials.
        if (pj == 0 && pn >= 1 && !mbar_wait(bar(C::B_OFREE), (pn - 1) & 1, w)) break;
        if constexpr (C::PP) {
          // O_{t%2} += P_t V_t over all 128 keys of tile t (8 k-steps of 16 keys).
          const int sv = tp % C::NSV, pg = tp & 1;
          if (!mbar_wait(bar(C::B_VF + sv), (tp / C::NSV) & 1, w)) break;
          if (!mbar_wait(bar(C::B_PF + pg), (tp >> 1) & 1, w)) break;
          tc_fence_after();
          const uint64_t dv = dv0 + sv * (C::KV_BYTES >> 4);
          const uint32_t od = tmem + C::TMEM_O + pg * C::DHB;
          const uint32_t acc0 = pj >= 2 ? 1u : 0u;  // tiles 0 and 1 of an item start O_0 / O_1
          if constexpr (C::PT) {
            const uint32_t pt = tmem + C::TMEM_P + pg * 64;  // 16 keys = 8 columns per k-step
            mma_ts(od, pt, dv, C::IDESC_PV, acc0);
#pragma unroll
            for (int k = 1; k < 8; ++k) mma_ts(od, pt + 8 * k, dv + ((16 * k * 128) >> 4), C::IDESC_PV, 1u);
          } else {
            const uint64_t dp = dp0 + pg * (C::P_BUF >> 4);
            mma_ss<false>(od, dp, dv, C::IDESC_PV, acc0);
#pragma unroll
            for (int k = 1; k < 8; ++k)
              mma_ss<false>(od, dp + (((k >> 2) * C::PANEL + (k & 3) * 32) >> 4), dv + ((16 * k * 128) >> 4),
                            C::IDESC_PV, 1u);
          }
          tc_commit(bar(C::B_OD + pg));
          tc_commit(bar(C::B_VE + sv));
        } else {
          // O_g += P[:, 64g .. 64g+63] V[64g .. 64g+63, :] for both key halves
          // g (4 k-steps of 16 keys each), as hi/lo bf16 pairs.
          const uint64_t dvh = make_sdesc(sbase + C::OFF_VHL, C::PANEL, 1024);
          const uint64_t dvl = dvh + ((C::VB_PANELS * C::PANEL) >> 4);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (!mbar_wait(bar(C::B_PF + 2 * g + (tp & 1)), (tp >> 1) & 1, w)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t od = tmem + C::TMEM_O + g * C::DHB;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint32_t aoff = (g * C::PANEL + k * 32) >> 4;
              const uint32_t boff = ((64 * g + 16 * k) * 128) >> 4;
              mma_ss<false>(od, dp0 + aoff, dvh + boff, C::IDESC_PV, (pj > 0 || k > 0) ? 1u : 0u);
              mma_ss<false>(od, dp0 + aoff, dvl + boff, C::IDESC_PV, 1u);
              mma_ss<false>(od, dp0 + (C::P_HALF >> 4) + aoff, dvh + boff, C::IDESC_PV, 1u);
            }
            tc_commit(bar(C::B_OD + 2 * g + (tp & 1)));
          }
          if (!ok) break;
        }
        ++tp;
        if (++pj == ip.nkv) {
          tc_commit(bar(C::B_ITEMD));  // every product of the item issued: done when they complete
          pj = 0;
          phave = fwd_item<LIST>(a, ++pn, ip);
        }
      }
      tc_commit(bar(C::B_FIN + 1));
      mbar_drain(bar(C::B_FIN + 1), 0, a.timeout_ns);
    }
    __syncwarp();
   }
   end_role();  // warp 3: TMEM owner
  } else if (warp < 12) {
    reg_alloc<C::REG_SM>();
    // ---------------- softmax warpgroups ----------------
    const int g = (warp - 4) >> 2;               // warpgroup
    const int tq = threadIdx.x - 128 - 128 * g;  // 0..127 within the warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_col = C::TMEM_O + g * C::DHB;
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    bool ok = true;
    // O_g *= alpha (this thread's row), in place in TMEM.
    auto rescale_o = [&](float alpha) {
      if constexpr (DHP == 64) {
        uint32_t r[64];
        tmem_ld64(tl + o_col, r);
#pragma unroll
        for (int i = 0; i < 64; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st64(tl + o_col, r);
      } else if constexpr (DHP > 64) {
#pragma unroll 1
        for (int c = 0; c < DHP / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tl + o_col + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tl + o_col + c * 32, r);
        }
      } else {
        uint32_t r[32];
        tmem_ld32(tl + o_col, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(tl + o_col, r);
      }
    };
    int tb = 0;  // global number of this work item's first key tile
    for (int n = 0; ok; ++n) {
      FwdItem it{};
      if (!fwd_item<LIST>(a, n, it)) break;
      const int q_idx = it.qt * C::BM + row;
      float m = -INFINITY, l = 0.f;
      if constexpr (C::PP) {
        // Warpgroup g takes the key tiles t = tb + j with t % 2 == g: the full
        // 128-key row of S_t from S buffer g, P_t into P buffer g, and
        // O_g += P_t V_t.
        const uint32_t s_col = C::TMEM_S + g * 128;
        const uint32_t prow = sbase + C::OFF_P + g * C::P_BUF + row * 128;
        const uint32_t sw = row & 7;
        for (int j = (g ^ tb) & 1; j < it.nkv; j += 2) {
          const int t = tb + j;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SF + g), (t >> 1) & 1, w));
          if (!ok) break;
          tc_fence_after();
          float s[128];
          {
            uint32_t r0[64], r1[64];
            tmem_ld64x2(tl + s_col, tl + s_col + 64, r0, r1);
#pragma unroll
            for (int i = 0; i < 64; ++i) {
              s[i] = __uint_as_float(r0[i]);
              s[64 + i] = __uint_as_float(r1[i]);
            }
          }
          tc_fence_before();
          mbar_arrive(bar(C::B_SFREE + g));
          if (j == it.nkv - 1) {  // diagonal tile: drop keys after this row's query
            const int lim = q_idx - j * C::BN;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c > lim) s[c] = -INFINITY;
          }
          float mp[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) mp[u] = fmax3(s[u], s[u + 4], s[u + 8]);
#pragma unroll
          for (int c = 12; c < 124; c += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u) mp[u] = fmax3(mp[u], s[c + u], s[c + 4 + u]);
#pragma unroll
          for (int u = 0; u < 4; ++u) mp[u] = fmaxf(mp[u], s[124 + u]);
          const float m_cand = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])) * a.scale_log2;
          const bool grow = m_cand > m + 8.0f;  // true on this warpgroup's first tile (m = -inf)
          // P buffer g and O_g were last used by P_{t-2} V_{t-2}.
          if (t >= 2) {
            ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_OD + g), ((t - 2) >> 1) & 1, w));
            if (!ok) break;
            tc_fence_after();
          }
          float alpha = 1.f;
          if (grow) {
            alpha = ex2(m - m_cand);
            l *= alpha;
            m = m_cand;
          }
          const float mref = (m == -INFINITY) ? 0.f : m;
          const uint64_t negm = f2pack(-mref, -mref);
          uint64_t acc2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int c = 0; c < 128; c += 2) {
            float x0, x1;
            f2unpack(ffma2(f2pack(s[c], s[c + 1]), sl2x2, negm), x0, x1);
            s[c] = ex2(x0);
            s[c + 1] = ex2(x1);
            acc2[(c >> 1) & 3] = fadd2(acc2[(c >> 1) & 3], f2pack(s[c], s[c + 1]));
          }
          float sa, sb2;
          f2unpack(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), sa, sb2);
          l += sa + sb2;
          if constexpr (C::PT) {
            // P row -> TMEM P buffer g: key pair (2c, 2c + 1) in column c,
            // written 16 columns at a time (small register blocks).
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) {
              uint32_t pk[16];
#pragma unroll
              for (int c = 0; c < 16; ++c) pk[c] = pack_bf16(s[32 * hh + 2 * c], s[32 * hh + 2 * c + 1]);
              tmem_st16(tl + C::TMEM_P + g * 64 + 16 * hh, pk);
            }
          } else {
            // P row -> panels (keys 0..63, 64..127) of P buffer g, bf16,
            // K-major, 128-byte swizzle.
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const uint32_t addr = prow + (c >> 3) * C::PANEL + (((c & 7) ^ sw) << 4);
              st_shared_v4(addr, pack_bf16(s[8 * c], s[8 * c + 1]), pack_bf16(s[8 * c + 2], s[8 * c + 3]),
                           pack_bf16(s[8 * c + 4], s[8 * c + 5]), pack_bf16(s[8 * c + 6], s[8 * c + 7]));
            }
          }
          // O_g is rescaled after the scores are dead (register budget); it
          // only has to happen before P_t V_t, which waits for the arrival
          // below. Tiles j = 0, 1 start O_0 / O_1 afresh.
          if (j >= 2 && __any_sync(0xffffffffu, grow)) rescale_o(alpha);
          if constexpr (!C::PT) fence_async_smem();
          tc_fence_before();
          mbar_arrive(bar(C::B_PF + g));
        }
      } else {
        // Both warpgroups take every key tile t = tb + j, warpgroup g keys
        // 64 g .. 64 g + 63 of it; one P buffer, V converted to hi/lo pairs.
        for (int j = 0; j < it.nkv; ++j) {
          const int t = tb + j;
          const int sb = t & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SF + sb), (t >> 1) & 1, w));
          if (!ok) break;
          tc_fence_after();
          float s[64];
          {
            uint32_t r[64];
            tmem_ld64(tl + C::TMEM_S + sb * 128 + 64 * g, r);
#pragma unroll
            for (int i = 0; i < 64; ++i) s[i] = __uint_as_float(r[i]);
          }
          tc_fence_before();
          mbar_arrive(bar(C::B_SFREE + sb));
          if (j == it.nkv - 1) {  // diagonal tile: drop keys after this row's query
            const int lim = q_idx - j * C::BN - 64 * g;
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c > lim) s[c] = -INFINITY;
          }
          float mp[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) mp[u] = fmax3(s[u], s[u + 4], s[u + 8]);
#pragma unroll
          for (int c = 12; c < 60; c += 8)
#pragma unroll
            for (int u = 0; u < 4; ++u) mp[u] = fmax3(mp[u], s[c + u], s[c + 4 + u]);
#pragma unroll
          for (int u = 0; u < 4; ++u) mp[u] = fmaxf(mp[u], s[60 + u]);
          const float mx = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3]));
          // A half that is fully masked (diagonal tile, upper rows of half 1)
          // has mx = -inf: it adds nothing and keeps the reference max.
          const float m_cand = mx * a.scale_log2;
          const bool grow = m_cand > m + 8.0f;  // also true on the first finite tile (m = -inf)
          // The P buffer and the V hi/lo tiles were last read by P_{t-1} V_{t-1}
          // (possibly of the previous work item); a rescale of O_g also needs it.
          if (t > 0) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(C::B_OD + 2 * g + ((t - 1) & 1)), ((t - 1) >> 1) & 1, w));
            if (!ok) break;
            tc_fence_after();
          }
          float alpha = 1.f;
          if (grow) {
            alpha = ex2(m - m_cand);
            l *= alpha;
            m = m_cand;
          }
          if (j > 0 && __any_sync(0xffffffffu, grow)) rescale_o(alpha);
          // p = 2^(s * scale_log2 - m); while the reference is still -inf
          // (every key so far masked) every p is exactly 0.
          const float mref = (m == -INFINITY) ? 0.f : m;
          const uint64_t negm = f2pack(-mref, -mref);
          uint64_t acc2[4] = {0, 0, 0, 0};
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float x0, x1;
            f2unpack(ffma2(f2pack(s[c], s[c + 1]), sl2x2, negm), x0, x1);
            s[c] = ex2(x0);
            s[c + 1] = ex2(x1);
            acc2[(c >> 1) & 3] = fadd2(acc2[(c >> 1) & 3], f2pack(s[c], s[c + 1]));
          }
          float sa, sb2;
          f2unpack(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), sa, sb2);
          l += sa + sb2;
          // V_t: fp32 stage -> bf16 hi/lo rows of this half, then release the stage.
          const int sv = t % C::NSV;
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_VF + sv), (t / C::NSV) & 1, w));
          if (!ok) break;
          const uint32_t vh = sbase + C::OFF_VHL;
          split_v_half<C>(sbase + C::OFF_V + sv * C::KV_BYTES, vh, vh + C::VB_PANELS * C::PANEL, g, tq);
          mbar_arrive(bar(C::B_VE + sv));
          // P row half -> shared memory panel g as hi and lo bf16 parts,
          // K-major with the 128-byte swizzle the MMA expects.
          const uint32_t prow = sbase + C::OFF_P + g * C::PANEL + row * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t addr = prow + ((c ^ (row & 7)) << 4);
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) split_bf16x2(s[8 * c + 2 * i], s[8 * c + 2 * i + 1], hi[i], lo[i]);
            st_shared_v4(addr, hi[0], hi[1], hi[2], hi[3]);
            st_shared_v4(addr + C::P_HALF, lo[0], lo[1], lo[2], lo[3]);
          }
          fence_async_smem();
          tc_fence_before();
          mbar_arrive(bar(C::B_PF + 2 * g + (t & 1)));
        }
      }
      if (!ok) break;
      if constexpr (C::EPI_WG) {
        // Publish this warpgroup's statistics of item n (set n % S, free once
        // the epilogue has read those of item n - S) and go on to the next item.
        constexpr int S = C::STAT_SETS;
        const int set = n % S;
        if (n >= S) {
          ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_STATFREE + set), ((n - S) / S) & 1, w));
          if (!ok) break;
        }
        float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT) + set * 512;
        stat[g * 128 + row] = m;
        stat[256 + g * 128 + row] = l;
        mbar_arrive(bar(C::B_STAT + set));
        tb += it.nkv;
        continue;
      }
      // ---- epilogue of work item n (one item per CTA) ----
      // Every product of the item (both warpgroups') is complete before the
      // partials are read.
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ITEMD), n & 1, w));
      if (!ok) break;
      // Merge the two warpgroups' statistics through shared memory.
      float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);
      stat[g * 128 + row] = m;
      stat[256 + g * 128 + row] = l;
      mbar_arrive(bar(C::B_STAT));
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_STAT), 0, w));
      if (!ok) break;
      tc_fence_after();
      const float m0 = stat[row], m1 = stat[128 + row];
      const float l0 = stat[256 + row], l1 = stat[384 + row];
      const float mt = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mt);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mt);
      const float lt = l0 * f0 + l1 * f1;
      const float c0 = f0 / lt, c1 = f1 / lt;
      // In ping-pong mode a warpgroup that had no key tile in this item (a
      // single-tile item) holds a stale partial: it is not read.
      const bool use0 = !C::PP || it.nkv >= 2 || (tb & 1) == 0;
      const bool use1 = !C::PP || it.nkv >= 2 || (tb & 1) == 1;
      // Warpgroup g finalises output columns [g W, g W + W), W = max(32, DHP / 2).
      constexpr int W = DHP / 2 > 32 ? DHP / 2 : 32;
      float o[W];
#pragma unroll
      for (int i = 0; i < W; ++i) o[i] = 0.f;
      if (g * W < DHP) {
        if constexpr (W == 64) {
          uint32_t r[64];
          if (use0) {
            tmem_ld64(tl + C::TMEM_O + g * W, r);
#pragma unroll
            for (int i = 0; i < 64; ++i) o[i] = __uint_as_float(r[i]) * c0;
          }
          if (use1) {
            tmem_ld64(tl + C::TMEM_O + C::DHB + g * W, r);
#pragma unroll
            for (int i = 0; i < 64; ++i) o[i] = fmaf(__uint_as_float(r[i]), c1, o[i]);
          }
        } else {
          uint32_t r[32];
          if (use0) {
            tmem_ld32(tl + C::TMEM_O + g * W, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]) * c0;
          }
          if (use1) {
            tmem_ld32(tl + C::TMEM_O + C::DHB + g * W, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = fmaf(__uint_as_float(r[i]), c1, o[i]);
          }
        }
      }
      // The partials are in registers: the next item's products may start.
      tc_fence_before();
      mbar_arrive(bar(C::B_OFREE));
      const bool valid = q_idx < a.T;
      // Padding rows (variable-length batches) are written as zeros, LSE -inf.
      const bool pad = a.lens && q_idx >= seq_len(a, it.b);
      if (pad) {
#pragma unroll
        for (int i = 0; i < W; ++i) o[i] = 0.f;
      }
      const size_t row_off = ((static_cast<size_t>(it.b) * a.T + q_idx) * a.Hq + it.h) * a.Dh;
      const int ncol = a.Dh - g * W;  // valid columns in this warpgroup's range
      if (valid && ncol > 0) {
        const int nc = ncol < W ? ncol : W;
        if constexpr (TF32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + row_off + g * W);
#pragma unroll
          for (int u = 0; u < W / 4; ++u)
            if (4 * u < nc) dst[u] = make_float4(o[4 * u], o[4 * u + 1], o[4 * u + 2], o[4 * u + 3]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + row_off + g * W);
#pragma unroll
          for (int u = 0; u < W / 8; ++u)
            if (8 * u < nc)
              dst[u] = make_uint4(pack_bf16(o[8 * u], o[8 * u + 1]), pack_bf16(o[8 * u + 2], o[8 * u + 3]),
                                  pack_bf16(o[8 * u + 4], o[8 * u + 5]), pack_bf16(o[8 * u + 6], o[8 * u + 7]));
        }
      }
      if (g == 0 && valid)
        a.lse[(static_cast<size_t>(it.b) * a.Hq + it.h) * a.T + q_idx] =
            pad ? -INFINITY : (mt + __log2f(lt)) * 0.69314718055994531f;
      tb += it.nkv;
    }
    end_role();
  } else {
    reg_dealloc<C::REG_EPI>();
    if constexpr (C::EPI_WG) {
      // ---------------- epilogue warpgroup ----------------
      // Per work item: merge the softmax warpgroups' statistics, wait for the
      // item's last product, read both O partials (32 head columns at a time),
      // release them for the next item and store the output rows and LSE.
      // Warp q owns TMEM lanes (query rows) 32 q .. 32 q + 31.
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;
      const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
      bool ok = true;
      int tb = 0;
      FwdItem it{};
      for (int n = 0; ok && fwd_item<LIST>(a, n, it); ++n) {
        constexpr int S = C::STAT_SETS;
        const int set = n % S;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_STAT + set), (n / S) & 1, w));
        if (!ok) break;
        const float* stat = reinterpret_cast<const float*>(smem + C::OFF_STAT) + set * 512;
        const float m0 = stat[row], m1 = stat[128 + row];
        const float l0 = stat[256 + row], l1 = stat[384 + row];
        mbar_arrive(bar(C::B_STATFREE + set));
        const float mt = fmaxf(m0, m1);
        const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mt);
        const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mt);
        const float lt = l0 * f0 + l1 * f1;
        const float c0 = f0 / lt, c1 = f1 / lt;
        // A warpgroup that had no key tile in this item (a single-tile item)
        // holds a stale partial: it is not read.
        const bool use0 = it.nkv >= 2 || (tb & 1) == 0;
        const bool use1 = it.nkv >= 2 || (tb & 1) == 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ITEMD), n & 1, w));
        if (!ok) break;
        tc_fence_after();
        const int q_idx = it.qt * C::BM + row;
        const bool valid = q_idx < a.T;
        const bool pad = a.lens && q_idx >= seq_len(a, it.b);  // padding row: zeros, LSE -inf
        const size_t row_off = ((static_cast<size_t>(it.b) * a.T + q_idx) * a.Hq + it.h) * a.Dh;
#pragma unroll
        for (int c = 0; c < DHP / 32; ++c) {
          float o[32];
          uint32_t r[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
          if (use0) {
            tmem_ld32(tl + C::TMEM_O + 32 * c, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]) * c0;
          }
          if (use1) {
            tmem_ld32(tl + C::TMEM_O + C::DHB + 32 * c, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = fmaf(__uint_as_float(r[i]), c1, o[i]);
          }
          if (c == DHP / 32 - 1) {
            tc_fence_before();
            mbar_arrive(bar(C::B_OFREE));  // both partials read: the next item's products may start
          }
          if (pad) {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0.f;
          }
          const int nc = a.Dh - 32 * c;  // valid columns in this block
          if (valid && nc > 0) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + row_off + 32 * c);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (8 * u < nc)
                dst[u] = make_uint4(pack_bf16(o[8 * u], o[8 * u + 1]), pack_bf16(o[8 * u + 2], o[8 * u + 3]),
                                    pack_bf16(o[8 * u + 4], o[8 * u + 5]), pack_bf16(o[8 * u + 6], o[8 * u + 7]));
          }
        }
        if (valid)
          a.lse[(static_cast<size_t>(it.b) * a.Hq + it.h) * a.T + q_idx] =
              pad ? -INFINITY : (mt + __log2f(lt)) * 0.69314718055994531f;
        tb += it.nkv;
      }
    }
    end_role();
  }
}

}  // namespace rca
