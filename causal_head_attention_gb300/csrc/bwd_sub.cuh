// Causal attention backward, bf16 storage, head width 128: 64-row query
// sub-tiles.
//
// Same operation and work items as attn_bwd_main_kernel (bwd.cuh): a work item
// is (batch, KV head, 128-key tile j); it loops over every query head of the
// group and every query position at or after the tile, accumulating dK and dV
// in TMEM and adding dQ partials into the fp32 accumulator. At head width 128
// a 128-row Q and dO tile leave room for one stage only, so every iteration
// waited for its loads. Here an iteration takes 64 query rows: a Q + dO stage
// is 32 KB and two of them fit, so the next sub-tile loads while the current
// one is computed. dQ is computed transposed, dQ^T = K^T dS^T (M = head width,
// N = 64 queries), so it has TMEM columns of its own, and the last 64 columns
// hold the item's K tile, copied there once (tcgen05.cp), so that S^T reads
// its A operand from TMEM instead of shared memory every iteration:
//   S^T [0, 64)  dP^T [64, 128)  dV [128, 256)  dK [256, 384)  dQ^T [384, 448)  K [448, 512)
// Products per iteration (M = 128 each): S^T = K Q^T and dP^T = V dO^T
// (N = 64 queries, K = head width), dV += P^T dO and dK += dS^T Q (N = head
// width, K = 64 queries), dQ^T = K^T dS^T (N = 64 queries, K = 128 keys; A and
// B MN-major). P^T and dS^T are [128 keys][64 queries] bf16 tiles, one 128-byte
// swizzled row per key.
// Warps: 0..3 dQ drain (and the item's dK, dV), 4..11 two compute warpgroups
// (warpgroup g owns query columns 32 g .. 32 g + 31), 12 TMA producer, 13 MMA
// issuer and TMEM owner. One CTA per work item.
#pragma once

#include "bwd.cuh"

namespace rca {

struct BwdSubCfg {
  static constexpr int PANEL = 128 * 128;          // 128 rows x 128 bytes
  static constexpr int KV_TILE = 2 * PANEL;        // 128 keys x 128 head columns (two 64-column panels)
  static constexpr int QPANEL = 64 * 128;          // 64 rows x 128 bytes
  static constexpr int QTILE = 2 * QPANEL;         // 64 query rows x 128 head columns
  static constexpr int PT_BYTES = 128 * 128;       // [128 keys][64 queries] bf16
  static constexpr int STG_BYTES = 4 * 8192;       // dQ staging: per drain warp two 32 x 32 fp32 boxes
  static constexpr int NQS = 2;
  static constexpr int STAGE_BYTES = 2 * QTILE + 1024;  // Q, dO, LSE2[64], D[64] (1 KB-aligned)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = KV_TILE;
  static constexpr int OFF_P = 2 * KV_TILE;
  static constexpr int OFF_DS = OFF_P + PT_BYTES;
  static constexpr int OFF_STG = OFF_DS + PT_BYTES;
  static constexpr int OFF_STAGE = OFF_STG + STG_BYTES;
  static constexpr int OFF_BAR = OFF_STAGE + NQS * STAGE_BYTES;
  static constexpr int BAR_BYTES = 1024;
  static constexpr int SMEM_BYTES = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static constexpr int TM_S = 0, TM_DP = 64, TM_DV = 128, TM_DK = 256, TM_DQ = 384, TM_K = 448;
  static constexpr int TMEM_COLS = 512;
  static constexpr uint32_t IDESC_T = make_idesc(false, 128, 64, false, false);   // S^T, dP^T
  static constexpr uint32_t IDESC_KV = make_idesc(false, 128, 128, false, true);  // dV, dK
  static constexpr uint32_t IDESC_QT = make_idesc(false, 128, 64, true, true);    // dQ^T
  static constexpr int NTHREADS = 512;
  static constexpr int LAUNCH_REGS = 128;
  static constexpr int REG_DQ = 64, REG_CTL = 96, REG_CMP = 176;
  static_assert(128 * REG_DQ + 256 * REG_CMP + 128 * REG_CTL <= NTHREADS * LAUNCH_REGS, "register split");
  // barriers
  static constexpr int B_KVF = 0;           // K, V of the item landed
  static constexpr int B_QF = 1;            // [NQS] Q / dO / LSE2 / D stage landed
  static constexpr int B_QE = B_QF + NQS;   // [NQS] stage free (its last product done)
  static constexpr int B_SR = B_QE + NQS;   // S^T(it) in TMEM
  static constexpr int B_DPR = B_SR + 1;    // dP^T(it) in TMEM
  static constexpr int B_SDPF = B_DPR + 1;  // S^T, dP^T of it read by both warpgroups (256)
  static constexpr int B_PR = B_SDPF + 1;   // [2] P^T half g written (128 each)
  static constexpr int B_DVD = B_PR + 2;    // [2] dV half g done: P^T half g free
  static constexpr int B_DSR = B_DVD + 2;   // [2] dS^T half g written
  static constexpr int B_DQF = B_DSR + 2;   // dK(it), dQ^T(it) done: dS^T free, dQ^T ready
  static constexpr int B_ITF = B_DQF + 1;   // dQ^T(it) read by the drain warpgroup (128)
  static constexpr int B_KVD = B_ITF + 1;   // dK, dV of the item final
  static constexpr int B_FIN = B_KVD + 1;
  static constexpr int NBAR = B_FIN + 1;
  static_assert(8 * NBAR + 8 <= BAR_BYTES, "barrier area");
};

// q and dO maps have 64-row boxes here (K, V: 128 rows; dq: 32 x 32 fp32).
template <bool LIST>
__global__ void __launch_bounds__(512, 1)
    attn_bwd_sub_kernel(const __grid_constant__ BwdMaps maps, const BwdArgs a) {
  using C = BwdSubCfg;
  grid_dep_sync();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sbase + C::OFF_BAR + 8u * i; };
  auto stage = [&](int s) -> uint32_t { return sbase + C::OFF_STAGE + s * C::STAGE_BYTES; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + 8 * C::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_BAR + 8 * C::NBAR + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One work item per CTA (a CTA past the end of a planned list has none).
  BwdItem itm{};
  if (!bwd_item<LIST>(a, 0, itm)) return;
  const int n_i2 = 2 * itm.n_i;           // 64-row query sub-tiles from 2 j on
  const int n_it = a.group * n_i2;

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_KVF), 1);
    for (int s = 0; s < C::NQS; ++s) {
      mbar_init(bar(C::B_QF + s), 1);
      mbar_init(bar(C::B_QE + s), 1);
    }
    mbar_init(bar(C::B_SR), 1);
    mbar_init(bar(C::B_DPR), 1);
    mbar_init(bar(C::B_SDPF), 256);
    for (int g = 0; g < 2; ++g) {
      mbar_init(bar(C::B_PR + g), 128);
      mbar_init(bar(C::B_DVD + g), 1);
      mbar_init(bar(C::B_DSR + g), 128);
    }
    mbar_init(bar(C::B_DQF), 1);
    mbar_init(bar(C::B_ITF), 128);
    mbar_init(bar(C::B_KVD), 1);
    mbar_init(bar(C::B_FIN), 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 13) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl w{a.status, abort_flag, a.timeout_ns};
  auto end_role = [&]() {
    tc_fence_before();
    if (warp == 13) {
      named_bar(1, C::NTHREADS);
      tc_fence_after();
      tmem_dealloc(tmem, C::TMEM_COLS);
    } else {
      named_bar_arrive(1, C::NTHREADS);
    }
  };
  // Iteration it: query head and 64-row sub-tile.
  auto head_of = [&](int it) { return itm.kvh * a.group + it / n_i2; };
  auto sub_of = [&](int it) { return 2 * itm.j + it % n_i2; };

  if (warp >= 12) {
   reg_dealloc<C::REG_CTL>();
   if (warp == 12) {
    // ---------------- TMA producer (one elected thread) ----------------
    if (elect_one()) {
      tma_prefetch_desc(&maps.q[0]);
      tma_prefetch_desc(&maps.k[0]);
      tma_prefetch_desc(&maps.v[0]);
      tma_prefetch_desc(&maps.dO[0]);
      mbar_expect_tx(bar(C::B_KVF), 2 * C::KV_TILE);
      for (int p = 0; p < 2; ++p) {
        tma_load_4d(sbase + C::OFF_K + p * C::PANEL, &maps.k[0], bar(C::B_KVF), p * 64, itm.kvh, itm.j * 128, itm.b);
        tma_load_4d(sbase + C::OFF_V + p * C::PANEL, &maps.v[0], bar(C::B_KVF), p * 64, itm.kvh, itm.j * 128, itm.b);
      }
      int it = 0;
      for (; it < n_it; ++it) {
        const int s = it % C::NQS;
        if (it >= C::NQS && !mbar_wait(bar(C::B_QE + s), ((it / C::NQS) - 1) & 1, w)) break;
        const int h = head_of(it), i2 = sub_of(it);
        const uint32_t st = stage(s);
        mbar_expect_tx(bar(C::B_QF + s), 2 * C::QTILE + 512);
        for (int p = 0; p < 2; ++p) {
          tma_load_4d(st + p * C::QPANEL, &maps.q[0], bar(C::B_QF + s), p * 64, h, i2 * 64, itm.b);
          tma_load_4d(st + C::QTILE + p * C::QPANEL, &maps.dO[0], bar(C::B_QF + s), p * 64, h, i2 * 64, itm.b);
        }
        const size_t ro = (static_cast<size_t>(itm.b) * a.Hq + h) * a.Tpad + static_cast<size_t>(i2) * 64;
        bulk_load(st + 2 * C::QTILE, a.lse2 + ro, 256, bar(C::B_QF + s));
        bulk_load(st + 2 * C::QTILE + 256, a.dvec + ro, 256, bar(C::B_QF + s));
      }
      // Exit path: every load issued has landed before shared memory is released.
      mbar_drain(bar(C::B_KVF), 0, a.timeout_ns);
      for (int s = 0; s < C::NQS && s < it; ++s) {
        const int last = s + ((it - 1 - s) / C::NQS) * C::NQS;
        mbar_drain(bar(C::B_QF + s), (last / C::NQS) & 1, a.timeout_ns);
      }
    }
    __syncwarp();
   } else if (warp == 13) {
    // ---------------- tcgen05 MMA issuer (one elected thread) ----------------
    if (elect_one()) {
      const uint64_t k_km = make_sdesc(sbase + C::OFF_K, 16, 1024);            // K: copied to TMEM (A of S^T)
      const uint64_t v_km = make_sdesc(sbase + C::OFF_V, 16, 1024);            // V: A of dP^T
      const uint64_t k_mn = make_sdesc(sbase + C::OFF_K, C::PANEL, 1024);      // K^T: A of dQ^T (MN-major)
      const uint64_t q_km = make_sdesc(stage(0), 16, 1024);                    // Q: B of S^T
      const uint64_t q_mn = make_sdesc(stage(0), C::QPANEL, 1024);             // Q: B of dK
      const uint64_t do_km = make_sdesc(stage(0) + C::QTILE, 16, 1024);        // dO: B of dP^T
      const uint64_t do_mn = make_sdesc(stage(0) + C::QTILE, C::QPANEL, 1024);  // dO: B of dV
      const uint64_t p_km = make_sdesc(sbase + C::OFF_P, 16, 1024);            // P^T: A of dV
      const uint64_t ds_km = make_sdesc(sbase + C::OFF_DS, 16, 1024);          // dS^T: A of dK
      const uint64_t ds_mn = make_sdesc(sbase + C::OFF_DS, C::PANEL, 1024);    // dS^T: B of dQ^T (MN-major)
      auto issue_s_dp = [&](int it2) {
        const uint32_t so = (it2 % C::NQS) * C::STAGE_BYTES;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t qo = so + (k / 4) * C::QPANEL + (k % 4) * 32;
          mma_ts(tmem + C::TM_S, tmem + C::TM_K + 8 * k, desc_add(q_km, qo), C::IDESC_T, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_SR));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t ko = (k / 4) * C::PANEL + (k % 4) * 32, qo = so + (k / 4) * C::QPANEL + (k % 4) * 32;
          mma_ss<false>(tmem + C::TM_DP, desc_add(v_km, ko), desc_add(do_km, qo), C::IDESC_T, k > 0 ? 1u : 0u);
        }
        tc_commit(bar(C::B_DPR));
      };
      bool ok = mbar_wait(bar(C::B_KVF), 0, w) && mbar_wait(bar(C::B_QF), 0, w);
      if (ok) {
        tc_fence_after();
        // K into TMEM: eight K = 16 slices of the K-major tile.
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tmem_cp_128x256b(tmem + C::TM_K + 8 * k, desc_add(k_km, (k / 4) * C::PANEL + (k % 4) * 32));
        issue_s_dp(0);
      }
      for (int it = 0; ok && it < n_it; ++it) {
        const int s = it % C::NQS;
        const uint32_t so = s * C::STAGE_BYTES;
        // The next iteration's S^T / dP^T first: they need this iteration's
        // to have been read and the next stage to have landed.
        if (it + 1 < n_it) {
          if (!mbar_wait(bar(C::B_QF + (it + 1) % C::NQS), ((it + 1) / C::NQS) & 1, w) ||
              !mbar_wait(bar(C::B_SDPF), it & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s_dp(it + 1);
        }
        // dV += P^T dO, one query half per warpgroup as soon as it is written.
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (!mbar_wait(bar(C::B_PR + g), it & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 2 * g; k < 2 * g + 2; ++k)
            mma_ss<false>(tmem + C::TM_DV, desc_add(p_km, k * 32), desc_add(do_mn, so + k * 16 * 128), C::IDESC_KV,
                          (it > 0 || k > 0) ? 1u : 0u);
          tc_commit(bar(C::B_DVD + g));
        }
        if (!ok) break;
        // dK += dS^T Q, one query half per warpgroup.
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (!mbar_wait(bar(C::B_DSR + g), it & 1, w)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 2 * g; k < 2 * g + 2; ++k)
            mma_ss<false>(tmem + C::TM_DK, desc_add(ds_km, k * 32), desc_add(q_mn, so + k * 16 * 128), C::IDESC_KV,
                          (it > 0 || k > 0) ? 1u : 0u);
        }
        if (!ok) break;
        tc_commit(bar(C::B_QE + s));  // the stage is no longer read
        if (it == n_it - 1) tc_commit(bar(C::B_KVD));
        // dQ^T = K^T dS^T (M = head width, N = 64 queries, K = 128 keys): the
        // previous one must have been drained from its columns.
        if (it > 0 && !mbar_wait(bar(C::B_ITF), (it - 1) & 1, w)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss<false>(tmem + C::TM_DQ, desc_add(k_mn, k * 16 * 128), desc_add(ds_mn, k * 16 * 128), C::IDESC_QT,
                        k > 0 ? 1u : 0u);
        tc_commit(bar(C::B_DQF));
      }
      tc_commit(bar(C::B_FIN));
      mbar_drain(bar(C::B_FIN), 0, a.timeout_ns);
    }
    __syncwarp();
   }
   end_role();  // warps 14 and 15 have no role
  } else if (warp < 4) {
    reg_dealloc<C::REG_DQ>();
    // ---------------- dQ drain warpgroup ----------------
    // Warp q reads TMEM lanes 32 q .. 32 q + 31 of dQ^T: head columns
    // 32 q .. 32 q + 31, one per lane, over the 64 query columns, 32 at a time.
    // Each 32 x 32 block is written transposed (query rows, head columns) into
    // one of the warp's two 4 KB 128-byte-swizzled boxes and added to the fp32
    // accumulator with a bulk tensor reduction issued by lane 0; a box is
    // rewritten once that lane's reductions of the previous iteration have
    // read it. It also writes the item's dK and dV once the last dK product is
    // done.
    const int quarter = warp;
    const int rl = quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t stg = sbase + C::OFF_STG + quarter * 8192;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      if (it == n_it - 1) {
        // ---- dK, dV of the item (key row rl), 32 head columns at a time;
        // dK carries the softmax scale.
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_KVD), 0, w));
        if (!ok) break;
        tc_fence_after();
        const int key = itm.j * 128 + rl;
        const bool valid = key < a.T;
        const size_t row_off = (static_cast<size_t>(itm.b) * a.T + key) * a.dkv_row + static_cast<size_t>(itm.kvh) * a.Dh;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t r[32];
            tmem_ld32(tl + (which == 0 ? C::TM_DV : C::TM_DK) + 32 * c, r);
            if (!valid) continue;
            const float mul = which == 0 ? 1.f : a.scale;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(which == 0 ? a.dv : a.dk) + row_off +
                                                  32 * c);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[u] = make_uint4(pack_bf16(__uint_as_float(r[8 * u]) * mul, __uint_as_float(r[8 * u + 1]) * mul),
                                  pack_bf16(__uint_as_float(r[8 * u + 2]) * mul, __uint_as_float(r[8 * u + 3]) * mul),
                                  pack_bf16(__uint_as_float(r[8 * u + 4]) * mul, __uint_as_float(r[8 * u + 5]) * mul),
                                  pack_bf16(__uint_as_float(r[8 * u + 6]) * mul, __uint_as_float(r[8 * u + 7]) * mul));
          }
        }
      }
      const int h = head_of(it), i2 = sub_of(it);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DQF), it & 1, w));
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        uint32_t r[32];
        tmem_ld32(tl + C::TM_DQ + 32 * hb, r);  // queries 32 hb .. 32 hb + 31 of head column rl
        if (hb == 1) {
          tc_fence_before();
          mbar_arrive(bar(C::B_ITF));  // dQ^T(it) read: its columns may be overwritten
        }
        if (hb == 0 && lane == 0) bulk_wait_read0();  // both boxes read by the previous reductions
        __syncwarp();
        const uint32_t box = stg + hb * 4096;
#pragma unroll
        for (int q = 0; q < 32; ++q)
          asm volatile("st.shared.b32 [%0], %1;" ::"r"(box + q * 128 + ((((lane >> 2) ^ (q & 7))) << 4) + (lane & 3) * 4),
                       "r"(r[q])
                       : "memory");
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          // Rows past the tensor's end (a partial last tile) are clipped by the reduction.
          tma_reduce_add_4d(&maps.dq, box, 32 * quarter, h, i2 * 64 + 32 * hb, itm.b);
          bulk_commit();
        }
      }
    }
    if (lane == 0) bulk_wait0();  // every bulk reduction this warp issued has landed
    __syncwarp();
    end_role();
  } else {
    reg_alloc<C::REG_CMP>();
    // ---------------- compute warpgroups ----------------
    // Warpgroup g owns query columns 32 g .. 32 g + 31 of every S^T / dP^T.
    const int g = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int rl = quarter * 32 + lane;  // key row of P^T / dS^T
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint64_t sl2x2 = f2pack(a.scale_log2, a.scale_log2);
    const uint32_t prow = sbase + C::OFF_P + rl * 128, dsrow = sbase + C::OFF_DS + rl * 128;
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % C::NQS;
      const int i2 = sub_of(it);
      ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SR), it & 1, w) &&
                                       mbar_wait(bar(C::B_QF + s), (it / C::NQS) & 1, w) &&
                                       mbar_wait(bar(C::B_DPR), it & 1, w));
      if (!ok) break;
      tc_fence_after();
      float p[32];
      uint32_t dpr[32];
      {
        uint32_t r[32];
        tmem_ld32(tl + C::TM_S + 32 * g, r);
        tmem_ld32(tl + C::TM_DP + 32 * g, dpr);
#pragma unroll
        for (int c = 0; c < 32; ++c) p[c] = __uint_as_float(r[c]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::B_SDPF));
      const float* lse2s = reinterpret_cast<const float*>(smem + (stage(s) - sbase) + 2 * C::QTILE) + 32 * g;
      const float* dvs = lse2s + 64;
      // P^T = 2^(S^T * scale * log2 e - LSE * log2 e) (the stage holds the
      // negated base-2 LSE), two columns per packed FMA.
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 l4 = *reinterpret_cast<const float4*>(lse2s + c);
        float x0, x1, x2, x3;
        f2unpack(ffma2(f2pack(p[c], p[c + 1]), sl2x2, f2pack(l4.x, l4.y)), x0, x1);
        f2unpack(ffma2(f2pack(p[c + 2], p[c + 3]), sl2x2, f2pack(l4.z, l4.w)), x2, x3);
        p[c] = ex2(x0);
        p[c + 1] = ex2(x1);
        p[c + 2] = ex2(x2);
        p[c + 3] = ex2(x3);
      }
      // Causality: key 128 j + rl is dropped for query 64 i2 + 32 g + c when
      // it is later, i.e. c < rl - lim (only the first two sub-tiles).
      const int lim = 64 * i2 + 32 * g - 128 * itm.j;
      if (lim < 128) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (rl > lim + c) p[c] = 0.f;
      }
      // P^T half g (query chunks 4 g .. 4 g + 3 of row rl) was last read by dV(it - 1).
      if (it > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DVD + g), (it - 1) & 1, w));
        if (!ok) break;
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        st_shared_v4(prow + (((4 * g + cc) ^ (rl & 7)) << 4), pack_bf16(p[8 * cc], p[8 * cc + 1]),
                     pack_bf16(p[8 * cc + 2], p[8 * cc + 3]), pack_bf16(p[8 * cc + 4], p[8 * cc + 5]),
                     pack_bf16(p[8 * cc + 6], p[8 * cc + 7]));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_PR + g));
      // dS^T = P^T * (dP^T - D) (the stage holds -D)
#pragma unroll
      for (int c = 0; c < 32; c += 4) {
        const float4 d4 = *reinterpret_cast<const float4*>(dvs + c);
        float y0, y1, y2, y3;
        f2unpack(fmul2(f2pack(p[c], p[c + 1]),
                       fadd2(f2pack(__uint_as_float(dpr[c]), __uint_as_float(dpr[c + 1])), f2pack(d4.x, d4.y))),
                 y0, y1);
        f2unpack(fmul2(f2pack(p[c + 2], p[c + 3]),
                       fadd2(f2pack(__uint_as_float(dpr[c + 2]), __uint_as_float(dpr[c + 3])), f2pack(d4.z, d4.w))),
                 y2, y3);
        p[c] = y0;
        p[c + 1] = y1;
        p[c + 2] = y2;
        p[c + 3] = y3;
      }
      // The dS^T buffer is free once dK(it - 1) and dQ^T(it - 1) are done.
      if (it > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_DQF), (it - 1) & 1, w));
        if (!ok) break;
      }
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        st_shared_v4(dsrow + (((4 * g + cc) ^ (rl & 7)) << 4), pack_bf16(p[8 * cc], p[8 * cc + 1]),
                     pack_bf16(p[8 * cc + 2], p[8 * cc + 3]), pack_bf16(p[8 * cc + 4], p[8 * cc + 5]),
                     pack_bf16(p[8 * cc + 6], p[8 * cc + 7]));
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(C::B_DSR + g));
    }
    end_role();
  }
}

}  // namespace rca
