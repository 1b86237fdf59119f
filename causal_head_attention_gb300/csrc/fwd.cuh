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
// CTA layout (320 threads):
//   warp 0      TMA producer: Q tile once, then K_j / V_j into NSK / NSV-stage rings
//   warp 1      TMEM owner + single-thread tcgen05 MMA issuer
//   warps 2..5  softmax warpgroup 0: keys 0..63 of every key tile
//   warps 6..9  softmax warpgroup 1: keys 64..127 of every key tile
// Thread t of a softmax warpgroup owns query row t. Each warpgroup keeps its
// own running max m_g and sum l_g (base-2 units) and its own output partial
// O_g in TMEM, accumulated from its half of the keys; the two partials are
// merged once at the end (O = sum_g 2^(m_g - m) O_g / sum_g 2^(m_g - m) l_g).
// Per key tile j (only tiles 0..qt are visited; tile qt is the diagonal):
//   S_j = Q K_j^T            tcgen05, into TMEM S[j % 2] (two 128-column buffers)
//   softmax on S_j           registers; O_g is rescaled only when m_g grows by
//                            more than 2^8 (exact: l_g uses the same reference)
//   P_j -> shared memory     bf16, K-major, 128-B swizzle, one panel per half,
//                            two buffers (P_{j+1} is written while P_j V_j runs)
//   O_g += P_j[:, half g] V_j[half g, :]   tcgen05, issued as soon as half g is ready
// S_{j+1} is issued before the P V products of tile j so the tensor core works
// while the softmax warps handle the next tile.
// fp32 storage mode: S = Q K^T runs as kind::tf32 on the fp32 tiles (the head
// dimension is contiguous, so both operands are K-major). P V contracts over
// keys, which needs V as an MN-major operand; kind::tf32 produced no result
// with MN-major operands on this GPU, so P and V are split into bf16 pairs
// x = hi + lo and O_g += Phi Vhi + Phi Vlo + Plo Vhi (relative error ~2^-16,
// below TF32's 2^-11).
#pragma once

#include "tc.cuh"

namespace rca {

template <bool TF32, int DHP>
struct FwdCfg {
  static constexpr int NTHREADS = 320;
  static constexpr int ES = TF32 ? 4 : 2;     // storage bytes per element
  static constexpr int PE = 128 / ES;         // elements per 128-byte swizzle row
  static constexpr int BM = 128, BN = 128;    // query rows, keys per tile
  static constexpr int PANEL = 128 * 128;     // one 128-row x 128-byte panel
  static constexpr int DPANELS = DHP / PE;    // panels across the head width
  static constexpr int Q_BYTES = DPANELS * PANEL;
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
  // bf16 mode double-buffers P so the softmax of tile j+1 never waits for
  // P_j V_j (only a rare O rescale does); fp32 mode (hi + lo) keeps one buffer.
  static constexpr int P_BUFS = TF32 ? 1 : 2;
  static constexpr int P_BUF = TF32 ? 2 * P_HALF : P_HALF;    // one buffer: hi (+ lo)
  static constexpr int P_BYTES = P_BUFS * P_BUF;
  static constexpr int SMEM_LIMIT = 232448;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int AVAIL = SMEM_LIMIT - 1024 - BAR_BYTES - Q_BYTES - P_BYTES - VHL_BYTES;
  static constexpr int NS_BF = AVAIL / (2 * KV_BYTES) > 4 ? 4 : AVAIL / (2 * KV_BYTES);
  static constexpr int NSV = TF32 ? (AVAIL >= 4 * KV_BYTES ? 2 : 1) : NS_BF;
  static constexpr int NSK_FIT = TF32 ? (AVAIL - NSV * KV_BYTES) / KV_BYTES : NS_BF;
  static constexpr int NSK = NSK_FIT > 4 ? 4 : NSK_FIT;
  static_assert(NSK >= 2 && NSV >= 1, "forward needs at least two K stages and one V stage");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + NSK * KV_BYTES;
  static constexpr int OFF_P = OFF_V + NSV * KV_BYTES;
  static constexpr int OFF_VHL = OFF_P + P_BYTES;
  static constexpr int OFF_BAR = OFF_VHL + VHL_BYTES;
  // float m[2][128], l[2][128] for the final merge; reuses the P buffer, which
  // is dead once every P V product has completed.
  static constexpr int OFF_STAT = OFF_P;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  static constexpr int TMEM_S = 0;          // two buffers: columns [0,128) and [128,256)
  static constexpr int TMEM_O = 256;        // O_0 at [256, 256+DHB), O_1 after it
  static constexpr int TMEM_COLS = 512;
  static_assert(TMEM_O + 2 * DHB <= TMEM_COLS, "TMEM budget");
  static constexpr uint32_t IDESC_QK = make_idesc(TF32, 128, 128, false, false);
  static constexpr uint32_t IDESC_PV = make_idesc(false, 128, DHB, false, true);  // bf16 operands
  // barrier slots
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
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
  static constexpr int B_FIN = B_OD + 4;
  static constexpr int NBAR = B_FIN + 1;
  static_assert(8 * NBAR + 8 <= 512, "barrier area");
};

struct FwdArgs {
  void* out;
  float* lse;
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, Dh, group, n_qt;
  float scale_log2;  // (1/sqrt(Dh)) * log2(e)
};

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

template <bool TF32, int DHP>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<TF32, DHP>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);
  float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);  // m[2][128], l[2][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh_count = a.B * a.Hq;
  const int lin = blockIdx.x;
  const int qt = a.n_qt - 1 - lin / bh_count;  // heaviest query tiles first
  const int bh = lin % bh_count;
  const int b = bh / a.Hq, h = bh % a.Hq, kvh = h / a.group;
  const int nkv = qt + 1;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_Q), 1);
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
      mbar_init(bar(C::B_SFREE + i), 256);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(bar(C::B_PF + i), 128);
      mbar_init(bar(C::B_OD + i), 1);
    }
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
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_expect_tx(bar(C::B_Q), C::Q_BYTES);
      for (int p = 0; p < C::DPANELS; ++p)
        tma_load_4d(sbase + C::OFF_Q + p * C::PANEL, &tmQ, bar(C::B_Q), p * C::PE, h, qt * C::BM, b);
    }
    int jk = 0, jv = 0;
    for (; jv < nkv; ++jv) {
      // K_j then V_j; K stages are released after S_j, V stages after the P V
      // products of tile j (bf16) or after the V_j hi/lo split (fp32).
      const int sk = jk % C::NSK;
      if (jk >= C::NSK && !mbar_wait_warp(bar(C::B_KE + sk), ((jk / C::NSK) - 1) & 1, w)) break;
      if (leader) {
        mbar_expect_tx(bar(C::B_KF + sk), C::KV_BYTES);
        for (int p = 0; p < C::DPANELS; ++p)
          tma_load_4d(sbase + C::OFF_K + sk * C::KV_BYTES + p * C::PANEL, &tmK, bar(C::B_KF + sk),
                      p * C::PE, kvh, jk * C::BN, b);
      }
      ++jk;
      const int sv = jv % C::NSV;
      if (jv >= C::NSV && !mbar_wait_warp(bar(C::B_VE + sv), ((jv / C::NSV) - 1) & 1, w)) break;
      if (leader) {
        mbar_expect_tx(bar(C::B_VF + sv), C::KV_BYTES);
        for (int p = 0; p < C::DPANELS; ++p)
          tma_load_4d(sbase + C::OFF_V + sv * C::KV_BYTES + p * C::PANEL, &tmV, bar(C::B_VF + sv),
                      p * C::PE, kvh, jv * C::BN, b);
      }
    }
    // Exit path: every load this warp issued has landed before shared memory
    // is released (immediate unless a wait above gave up).
    if (leader) {
      mbar_drain(bar(C::B_Q), 0, a.timeout_ns);
      for (int s = 0; s < C::NSK && s < jk; ++s) {
        const int last = s + ((jk - 1 - s) / C::NSK) * C::NSK;
        mbar_drain(bar(C::B_KF + s), (last / C::NSK) & 1, a.timeout_ns);
      }
      for (int s = 0; s < C::NSV && s < jv; ++s) {
        const int last = s + ((jv - 1 - s) / C::NSV) * C::NSV;
        mbar_drain(bar(C::B_VF + s), (last / C::NSV) & 1, a.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ---------------- tcgen05 MMA issuer (whole warp; one elected lane issues) ----------------
    const bool leader = elect_one();
    bool ok = mbar_wait_warp(bar(C::B_Q), 0, w);
    const uint32_t qb = sbase + C::OFF_Q;
    const uint32_t pb = sbase + C::OFF_P;
    // O_g += P[:, 64g .. 64g+63] V[64g .. 64g+63, :]  (4 k-steps of 16 keys)
    auto issue_pv = [&](int jj) -> bool {
      const int sv = jj % C::NSV;
      const uint32_t pbj = pb + (jj % C::P_BUFS) * C::P_BUF;
      if constexpr (!TF32) {
        if (!mbar_wait_warp(bar(C::B_VF + sv), (jj / C::NSV) & 1, w)) return false;
      }
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (!mbar_wait_warp(bar(C::B_PF + 2 * g + (jj & 1)), (jj >> 1) & 1, w)) return false;
        tc_fence_after();
        const uint32_t od = tmem + C::TMEM_O + g * C::DHB;
        if constexpr (TF32) {
          const uint32_t vh = sbase + C::OFF_VHL, vl = vh + C::VB_PANELS * C::PANEL;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t aoff = g * C::PANEL + k * 32;
            const uint64_t ah = make_sdesc(pbj + aoff, 16, 1024);
            const uint64_t al = make_sdesc(pbj + C::P_HALF + aoff, 16, 1024);
            const uint32_t boff = (64 * g + 16 * k) * 128;
            const uint64_t bh_ = make_sdesc(vh + boff, C::PANEL, 1024);
            const uint64_t bl = make_sdesc(vl + boff, C::PANEL, 1024);
            if (leader) {
              mma_ss<false>(od, ah, bh_, C::IDESC_PV, (jj > 0 || k > 0) ? 1u : 0u);
              mma_ss<false>(od, ah, bl, C::IDESC_PV, 1u);
              mma_ss<false>(od, al, bh_, C::IDESC_PV, 1u);
            }
          }
        } else {
          const uint32_t vb = sbase + C::OFF_V + sv * C::KV_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t ad = make_sdesc(pbj + g * C::PANEL + k * 32, 16, 1024);
            const uint64_t bd = make_sdesc(vb + (64 * g + 16 * k) * 128, C::PANEL, 1024);
            if (leader) mma_ss<false>(od, ad, bd, C::IDESC_PV, (jj > 0 || k > 0) ? 1u : 0u);
          }
        }
        if (leader) tc_commit(bar(C::B_OD + 2 * g + (jj & 1)));
      }
      if constexpr (!TF32) {
        if (leader) tc_commit(bar(C::B_VE + sv));
      }
      return true;
    };
    for (int j = 0; ok && j < nkv; ++j) {
      const int sk = j % C::NSK;
      const int sb = j & 1;
      if (!mbar_wait_warp(bar(C::B_KF + sk), (j / C::NSK) & 1, w)) { ok = false; break; }
      if (j >= 2 && !mbar_wait_warp(bar(C::B_SFREE + sb), ((j - 2) >> 1) & 1, w)) { ok = false; break; }
      tc_fence_after();
      const uint32_t kb = sbase + C::OFF_K + sk * C::KV_BYTES;
#pragma unroll
      for (int k = 0; k < DHP / C::KSTEP; ++k) {
        const uint32_t off = (k / C::SPP) * C::PANEL + (k % C::SPP) * 32;
        const uint64_t ad = make_sdesc(qb + off, 16, 1024), bd = make_sdesc(kb + off, 16, 1024);
        if (leader) mma_ss<TF32>(tmem + C::TMEM_S + sb * 128, ad, bd, C::IDESC_QK, k > 0 ? 1u : 0u);
      }
      if (leader) {
        tc_commit(bar(C::B_SF + sb));
        tc_commit(bar(C::B_KE + sk));
      }
      if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
    }
    if (ok) issue_pv(nkv - 1);
    // Exit path: all issued MMAs finish before TMEM is released.
    if (leader) {
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
  } else {
    // ---------------- softmax warpgroups ----------------
    const int g = (warp - 2) >> 2;              // key half owned by this warpgroup
    const int t = threadIdx.x - 64 - 128 * g;   // 0..127 within the warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q_idx = qt * C::BM + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t o_col = C::TMEM_O + g * C::DHB;
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // Warpgroup 1 starts about half a tile after warpgroup 0 (it waits until
    // warpgroup 0 has its first scores in registers), so that from then on one
    // warpgroup's exponentials overlap the other's TMEM load and barrier waits
    // instead of both contending for the same units at the same time.
    if (g == 1) named_bar(3, 256);
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SF + sb), (j >> 1) & 1, w));
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
      if (g == 0 && j == 0) named_bar_arrive(3, 256);
      if (j == nkv - 1) {  // diagonal tile: drop keys after this row's query
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
      // A half that is fully masked (diagonal tile, upper rows of half 1) has
      // mx = -inf: it adds nothing and keeps the reference max.
      const float m_cand = mx * a.scale_log2;
      const bool grow = m_cand > m + 8.0f;  // also true on the first finite tile (m = -inf)
      // P buffer j % P_BUFS was last read by P_{j-P_BUFS} V: wait for it. A rescale
      // of O_g needs every earlier product, i.e. P_{j-1} V_{j-1}, to be complete.
      const bool need_prev = (j > 0) && (C::P_BUFS == 1 || __any_sync(0xffffffffu, grow));
      if (need_prev) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bar(C::B_OD + 2 * g + ((j - 1) & 1)), ((j - 1) >> 1) & 1, w));
        if (!ok) break;
        tc_fence_after();
      } else if (j >= C::P_BUFS) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_OD + 2 * g + ((j - C::P_BUFS) & 1)),
                                               ((j - C::P_BUFS) >> 1) & 1, w));
        if (!ok) break;
        tc_fence_after();
      }
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m - m_cand);
        l *= alpha;
        m = m_cand;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
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
      }
      // p = 2^(s * scale_log2 - m); while the reference is still -inf (every
      // key so far masked) every p is exactly 0.
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
      if constexpr (TF32) {
        // V_j: fp32 stage -> bf16 hi/lo rows of this half, then release the stage.
        const int sv = j % C::NSV;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_VF + sv), (j / C::NSV) & 1, w));
        if (!ok) break;
        const uint32_t vh = sbase + C::OFF_VHL;
        split_v_half<C>(sbase + C::OFF_V + sv * C::KV_BYTES, vh, vh + C::VB_PANELS * C::PANEL, g, t);
        mbar_arrive(bar(C::B_VE + sv));
      }
      // P row half -> shared memory panel g (bf16; fp32 mode writes hi and lo),
      // K-major with the 128-byte swizzle the MMA expects.
      const uint32_t prow = sbase + C::OFF_P + (j % C::P_BUFS) * C::P_BUF + g * C::PANEL + row * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = prow + ((c ^ (row & 7)) << 4);
        if constexpr (TF32) {
          uint32_t hi[4], lo[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) split_bf16x2(s[8 * c + 2 * i], s[8 * c + 2 * i + 1], hi[i], lo[i]);
          st_shared_v4(addr, hi[0], hi[1], hi[2], hi[3]);
          st_shared_v4(addr + C::P_HALF, lo[0], lo[1], lo[2], lo[3]);
        } else {
          st_shared_v4(addr, pack_bf16(s[8 * c], s[8 * c + 1]), pack_bf16(s[8 * c + 2], s[8 * c + 3]),
                       pack_bf16(s[8 * c + 4], s[8 * c + 5]), pack_bf16(s[8 * c + 6], s[8 * c + 7]));
        }
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PF + 2 * g + (j & 1)));
    }
    // Both halves' last P V products must be complete before either partial is read.
    const uint32_t last_par = ((nkv - 1) >> 1) & 1;
    if (ok)
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_OD + ((nkv - 1) & 1)), last_par, w) &&
                                       mbar_wait(bar(C::B_OD + 2 + ((nkv - 1) & 1)), last_par, w));
    // Merge the two halves' statistics (both warpgroups always reach this barrier).
    stat[g * 128 + row] = m;
    stat[256 + g * 128 + row] = l;
    named_bar(1, 256);
    if (ok) {
      tc_fence_after();
      const float m0 = stat[row], m1 = stat[128 + row];
      const float l0 = stat[256 + row], l1 = stat[384 + row];
      const float mt = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mt);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mt);
      const float lt = l0 * f0 + l1 * f1;
      const float c0 = f0 / lt, c1 = f1 / lt;
      const bool valid = q_idx < a.T;
      const size_t row_off = ((static_cast<size_t>(b) * a.T + q_idx) * a.Hq + h) * a.Dh;
      // Warpgroup g finalises output columns [g W, g W + W), W = max(32, DHP / 2).
      constexpr int W = DHP / 2 > 32 ? DHP / 2 : 32;
      if (g * W < DHP) {
        float o[W];
        if constexpr (W == 64) {
          uint32_t r[64];
          tmem_ld64(tl + C::TMEM_O + g * W, r);
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = __uint_as_float(r[i]) * c0;
          tmem_ld64(tl + C::TMEM_O + C::DHB + g * W, r);
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = fmaf(__uint_as_float(r[i]), c1, o[i]);
        } else {
          uint32_t r0[32], r1[32];
          tmem_ld32x2(tl + C::TMEM_O + g * W, tl + C::TMEM_O + C::DHB + g * W, r0, r1);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r0[i]) * c0 + __uint_as_float(r1[i]) * c1;
        }
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
      }
      if (g == 0 && valid)
        a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.T + q_idx] = (mt + __log2f(lt)) * 0.69314718055994531f;
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
