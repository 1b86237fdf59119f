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
// CTA layout (192 threads):
//   warp 0      TMA producer: Q tile once, then K_j / V_j into NSK / NSV-stage rings
//   warp 1      TMEM owner + single-thread tcgen05 MMA issuer
//   warps 2..5  softmax warpgroup: thread t owns query row t of the tile
// Per key tile j (only tiles 0..qt are visited; tile qt is the diagonal):
//   S_j = Q K_j^T            tcgen05, into TMEM S[j % 2] (two 128-column buffers)
//   softmax on S_j           registers; running max m and sum l per row, kept in
//                            base-2 units; O is rescaled only when the running
//                            max grows by more than 2^8 (exact: l uses the same
//                            reference max)
//   P_j -> shared memory     bf16, K-major, 128-B swizzle
//   O += P_j V_j             tcgen05, into TMEM O
// fp32 storage mode: S = Q K^T runs as kind::tf32 on the fp32 tiles (the head
// dimension is contiguous, so both operands are K-major). P V contracts over
// keys, which needs V as an MN-major operand; kind::tf32 produced no result
// with MN-major operands on this GPU, so P and V are split into bf16 pairs
// x = hi + lo and O += Phi Vhi + Phi Vlo + Plo Vhi (relative error ~2^-16,
// below TF32's 2^-11).
// S_{j+1} is issued before O += P_j V_j so the tensor core works while the
// softmax warps handle the next tile.
#pragma once

#include "tc.cuh"

namespace rca {

template <bool TF32, int DHP>
struct FwdCfg {
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
  static constexpr int P_BYTES = TF32 ? 2 * P_HALF : P_HALF;  // hi (+ lo)
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
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory budget");
  static constexpr int TMEM_S = 0;          // two buffers: columns [0,128) and [128,256)
  static constexpr int TMEM_O = 256;        // DHB columns
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = make_idesc(TF32, 128, 128, false, false);
  static constexpr uint32_t IDESC_PV = make_idesc(false, 128, DHB, false, true);  // bf16 operands
  // barrier slots
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;
  static constexpr int B_KE = B_KF + NSK;
  static constexpr int B_VF = B_KE + NSK;
  static constexpr int B_VE = B_VF + NSV;
  static constexpr int B_SF = B_VE + NSV;   // 2
  static constexpr int B_SFREE = B_SF + 2;  // 2
  static constexpr int B_PF = B_SFREE + 2;
  static constexpr int B_OD = B_PF + 1;     // 2
  static constexpr int B_FIN = B_OD + 2;
  static constexpr int NBAR = B_FIN + 1;
};

struct FwdArgs {
  void* out;
  float* lse;
  int* status;
  unsigned long long timeout_ns;
  int B, Hq, Hkv, T, Dh, group, n_qt;
  float scale_log2;  // (1/sqrt(Dh)) * log2(e)
};

// fp32 mode: split the fp32 V stage (MN-major, 32-element panels) into bf16
// hi/lo tiles (MN-major, 64-element panels). Thread t converts key row t; head
// columns past DHP are written as zeros.
template <class C>
__device__ __forceinline__ void split_v_row(uint32_t vsrc, uint32_t vhi, uint32_t vlo, int row) {
  const uint32_t sw = row & 7;
#pragma unroll
  for (int g = 0; g < C::DHB / 8; ++g) {
    const uint32_t dst = (g >> 3) * C::PANEL + row * 128 + (((g & 7) ^ sw) << 4);
    if (g < C::DPANELS * 4) {
      const uint32_t pf = g >> 2;                // fp32 panel
      const uint32_t c0 = (2 * g) & 7, c1 = c0 + 1;
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
__global__ void __launch_bounds__(192, 1)
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
      mbar_init(bar(C::B_VE + s), TF32 ? 128 : 1);  // fp32: released by the converting warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(C::B_SF + i), 1);
      mbar_init(bar(C::B_SFREE + i), 128);
      mbar_init(bar(C::B_OD + i), 1);
    }
    mbar_init(bar(C::B_PF), 128);
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
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_expect_tx(bar(C::B_Q), C::Q_BYTES);
      for (int p = 0; p < C::DPANELS; ++p)
        tma_load_4d(sbase + C::OFF_Q + p * C::PANEL, &tmQ, bar(C::B_Q), p * C::PE, h, qt * C::BM, b);
      int jk = 0, jv = 0;
      for (; jv < nkv; ++jv) {
        // K_j then V_j; K stages are released after S_j, V stages after P_j V_j
        // (bf16) or after the V_j hi/lo split (fp32).
        const int sk = jk % C::NSK;
        if (jk >= C::NSK && !mbar_wait(bar(C::B_KE + sk), ((jk / C::NSK) - 1) & 1, w)) break;
        mbar_expect_tx(bar(C::B_KF + sk), C::KV_BYTES);
        for (int p = 0; p < C::DPANELS; ++p)
          tma_load_4d(sbase + C::OFF_K + sk * C::KV_BYTES + p * C::PANEL, &tmK, bar(C::B_KF + sk),
                      p * C::PE, kvh, jk * C::BN, b);
        ++jk;
        const int sv = jv % C::NSV;
        if (jv >= C::NSV && !mbar_wait(bar(C::B_VE + sv), ((jv / C::NSV) - 1) & 1, w)) break;
        mbar_expect_tx(bar(C::B_VF + sv), C::KV_BYTES);
        for (int p = 0; p < C::DPANELS; ++p)
          tma_load_4d(sbase + C::OFF_V + sv * C::KV_BYTES + p * C::PANEL, &tmV, bar(C::B_VF + sv),
                      p * C::PE, kvh, jv * C::BN, b);
      }
      // Exit path: every load this thread issued has landed before shared
      // memory is released (immediate unless a wait above gave up).
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
    // ---------------- tcgen05 MMA issuer ----------------
    if (lane == 0) {
      bool ok = mbar_wait(bar(C::B_Q), 0, w);
      const uint32_t qb = sbase + C::OFF_Q;
      const uint32_t pb = sbase + C::OFF_P;
      auto issue_pv = [&](int jj) -> bool {
        if (!mbar_wait(bar(C::B_PF), jj & 1, w)) return false;
        const int sv = jj % C::NSV;
        if constexpr (!TF32) {
          if (!mbar_wait(bar(C::B_VF + sv), (jj / C::NSV) & 1, w)) return false;
        }
        tc_fence_after();
        if constexpr (TF32) {
          // O += Phi Vhi + Phi Vlo + Plo Vhi  (bf16 products, fp32 accumulate)
          const uint32_t vh = sbase + C::OFF_VHL, vl = vh + C::VB_PANELS * C::PANEL;
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k) {
            const uint32_t aoff = (k / 4) * C::PANEL + (k % 4) * 32;
            const uint64_t ah = make_sdesc(pb + aoff, 16, 1024);
            const uint64_t al = make_sdesc(pb + C::P_HALF + aoff, 16, 1024);
            const uint64_t bh_ = make_sdesc(vh + k * 16 * 128, C::PANEL, 1024);
            const uint64_t bl = make_sdesc(vl + k * 16 * 128, C::PANEL, 1024);
            mma_ss<false>(tmem + C::TMEM_O, ah, bh_, C::IDESC_PV, (jj > 0 || k > 0) ? 1u : 0u);
            mma_ss<false>(tmem + C::TMEM_O, ah, bl, C::IDESC_PV, 1u);
            mma_ss<false>(tmem + C::TMEM_O, al, bh_, C::IDESC_PV, 1u);
          }
          tc_commit(bar(C::B_OD + (jj & 1)));
        } else {
          const uint32_t vb = sbase + C::OFF_V + sv * C::KV_BYTES;
#pragma unroll
          for (int k = 0; k < C::BN / 16; ++k) {
            const uint64_t ad = make_sdesc(pb + (k / 4) * C::PANEL + (k % 4) * 32, 16, 1024);
            const uint64_t bd = make_sdesc(vb + k * 16 * 128, C::PANEL, 1024);
            mma_ss<false>(tmem + C::TMEM_O, ad, bd, C::IDESC_PV, (jj > 0 || k > 0) ? 1u : 0u);
          }
          tc_commit(bar(C::B_OD + (jj & 1)));
          tc_commit(bar(C::B_VE + sv));
        }
        return true;
      };
      for (int j = 0; ok && j < nkv; ++j) {
        const int sk = j % C::NSK;
        const int sb = j & 1;
        if (!mbar_wait(bar(C::B_KF + sk), (j / C::NSK) & 1, w)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(bar(C::B_SFREE + sb), ((j - 2) >> 1) & 1, w)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kb = sbase + C::OFF_K + sk * C::KV_BYTES;
#pragma unroll
        for (int k = 0; k < DHP / C::KSTEP; ++k) {
          const uint32_t off = (k / C::SPP) * C::PANEL + (k % C::SPP) * 32;
          mma_ss<TF32>(tmem + C::TMEM_S + sb * 128, make_sdesc(qb + off, 16, 1024),
                       make_sdesc(kb + off, 16, 1024), C::IDESC_QK, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SF + sb));
        tc_commit(bar(C::B_KE + sk));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok) issue_pv(nkv - 1);
      // Exit path: all issued MMAs finish before TMEM is released.
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
  } else {
    // ---------------- softmax warpgroup ----------------
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q_idx = qt * C::BM + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SF + sb), (j >> 1) & 1, w));
      if (!ok) break;
      tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + C::TMEM_S + sb * 128 + c * 32, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_SFREE + sb));
      if (j == nkv - 1) {  // diagonal tile: drop keys after this row's query
        const int lim = q_idx - j * C::BN;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > lim) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_cand = mx * sl2;
      if (j > 0) {
        // P_{j-1} V_{j-1} is complete: P (and the fp32-mode V hi/lo tile) may be
        // overwritten and O holds every earlier tile.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_OD + ((j - 1) & 1)), ((j - 1) >> 1) & 1, w));
        if (!ok) break;
        tc_fence_after();
      }
      const bool grow = m_cand > m + 8.0f;  // also true on the first tile (m = -inf)
      float alpha = 1.f;
      if (grow) {
        alpha = ex2(m - m_cand);
        l *= alpha;
        m = m_cand;
      }
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < DHP / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(tl + C::TMEM_O + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tl + C::TMEM_O + c * 32, r);
        }
      }
      const float neg_m = -m;
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        s[c] = ex2(fmaf(s[c], sl2, neg_m));
        sum += s[c];
      }
      l += sum;
      if constexpr (TF32) {
        // V_j: fp32 stage -> bf16 hi/lo tile, then release the stage.
        const int sv = j % C::NSV;
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_VF + sv), (j / C::NSV) & 1, w));
        if (!ok) break;
        const uint32_t vh = sbase + C::OFF_VHL;
        split_v_row<C>(sbase + C::OFF_V + sv * C::KV_BYTES, vh, vh + C::VB_PANELS * C::PANEL, row);
        mbar_arrive(bar(C::B_VE + sv));
      }
      // P row -> shared memory (bf16; fp32 mode writes hi and lo), K-major with
      // the 128-byte swizzle the MMA expects.
      const uint32_t prow = sbase + C::OFF_P + row * 128;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint32_t addr = prow + (c >> 3) * C::PANEL + (((c & 7) ^ (row & 7)) << 4);
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
      mbar_arrive(bar(C::B_PF));
    }
    if (ok) {
      ok = __all_sync(0xffffffffu,
                      mbar_wait(bar(C::B_OD + ((nkv - 1) & 1)), ((nkv - 1) >> 1) & 1, w));
    }
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool valid = q_idx < a.T;
      const size_t row_off = ((static_cast<size_t>(b) * a.T + q_idx) * a.Hq + h) * a.Dh;
#pragma unroll
      for (int c = 0; c < DHP / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tl + C::TMEM_O + c * 32, r);  // whole warp, even for padding rows
        const int ncol = a.Dh - c * 32;
        if (!valid || ncol <= 0) continue;
        if constexpr (TF32) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + row_off + c * 32);
          const int nv = (ncol >= 32 ? 32 : ncol) / 4;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (u < nv)
              dst[u] = make_float4(__uint_as_float(r[4 * u]) * inv_l, __uint_as_float(r[4 * u + 1]) * inv_l,
                                   __uint_as_float(r[4 * u + 2]) * inv_l, __uint_as_float(r[4 * u + 3]) * inv_l);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + row_off + c * 32);
          const int nv = (ncol >= 32 ? 32 : ncol) / 8;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (u < nv)
              dst[u] = make_uint4(
                  pack_bf16(__uint_as_float(r[8 * u]) * inv_l, __uint_as_float(r[8 * u + 1]) * inv_l),
                  pack_bf16(__uint_as_float(r[8 * u + 2]) * inv_l, __uint_as_float(r[8 * u + 3]) * inv_l),
                  pack_bf16(__uint_as_float(r[8 * u + 4]) * inv_l, __uint_as_float(r[8 * u + 5]) * inv_l),
                  pack_bf16(__uint_as_float(r[8 * u + 6]) * inv_l, __uint_as_float(r[8 * u + 7]) * inv_l));
        }
      }
      if (valid) a.lse[(static_cast<size_t>(b) * a.Hq + h) * a.T + q_idx] = (m + __log2f(l)) * 0.69314718055994531f;
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
