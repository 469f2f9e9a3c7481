// fa_fwd_fp8.cu -- attention forward with 8-bit (e4m3) Q, K, V on sm_103a.
//
// The same tiled online-softmax forward as fa_fwd.cu ("FlashAttention"
// notes, "Tiling"; "Как работает FlashAttention математически", sections 3,
// 4, 6), with both products on the 8-bit tensor-core path (the same page's
// section 9 names 8-bit tensor-core arithmetic as the FlashAttention-3
// extension):
//   S = (Q8 K8^T) * scale * dq * dk     (kind::f8f6f4, fp32 in tensor memory)
//   P8 = e4m3(exp2(S log2 e - m + 4))   (values in (0, 256], e4m3 max 448)
//   O = (sum P8 V8) * dv / l,  l = sum exp2(S log2 e - m + 4) in fp32,
//   LSE = m - 4 + log2(l) in log2 units
// where dq, dk, dv are per-(batch, head) descale factors (the real inputs are
// Q8 dq, K8 dk, V8 dv).  The reference max m moves only when a tile's max
// exceeds it by more than 2^4 (exp2 units), so the largest P of a row lies in
// [16, 256] and e4m3 keeps about 2^-14 of it.  O is normalised by the exact
// row sum (the one LSE uses); the e4m3 rounding of P (at most 2^-4 relative)
// is the method's only extra error.
//
// Every MMA operand is K-major: S = Q K^T reads Q and K rows; O += P V reads
// P from tensor memory (4 e4m3 per 32-bit column) and V^T from shared
// memory, so V is first transposed to [B*H][128][npad] by a separate
// memory-bound kernel.  One CTA owns two 128-row query tiles of one (b, h);
// 10 warps: 0-3 and 4-7 softmax for the two tiles, 8 MMA issuer, 9 TMA
// producer; tensor memory S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512),
// P_w over the first 32 columns of S_w.
#include <cuda_fp8.h>

#include "fa_common.cuh"
#include "fa_ptx.cuh"

namespace fa {

struct Fp8Layout {
  static constexpr int D = 128;
  static constexpr int TILE_BYTES = TILE * 128;            // 128 rows x 128 bytes: one swizzle chunk
  static constexpr int STAGES = 8;                         // K and V^T slots
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = RING_OFF + STAGES * TILE_BYTES;
  static constexpr int B_Q = 0;                  // 2
  static constexpr int B_FULL = 2;               // STAGES
  static constexpr int B_EMPTY = 2 + STAGES;     // STAGES
  static constexpr int B_S = 2 + 2 * STAGES;     // 2
  static constexpr int B_P = B_S + 2;            // 2
  static constexpr int B_PH = B_P + 2;           // 2: first half of P_w (keys 0-63) in tensor memory
  static constexpr int B_O = B_PH + 2;           // 2
  static constexpr int B_DONE = B_O + 2;         // 1
  static constexpr int B_QFREE = B_DONE + 1;     // 1: an item's S products done, Q may be reloaded
  static constexpr int NBARS = B_QFREE + 1;
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 384;
  static constexpr int THREADS = 320;
};

// e4m3 pair: (lo, hi) -> 16 bits with lo in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ void fp8_drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

__global__ void __launch_bounds__(320, 1) fa_fwd_fp8_kernel(const __grid_constant__ Fp8Params p) {
  using L = Fp8Layout;
  constexpr int D = L::D;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  // Work items: query-tile pairs j of all (batch, head)s, head fastest,
  // longest causal rows first; a persistent grid (at most one CTA per SM)
  // where CTA c takes items c, 2G - 1 - c, 2G + c, ... (G CTAs), as in the
  // bf16 forward.
  const int n_items = p.n_pairs * p.BH;
  auto item_index = [&](int k) {
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int j = k * G + ((k & 1) ? G - 1 - c : c);
    return j < n_items ? j : -1;
  };
  struct Item {
    int bh, qt0, qt1, kt_end, nv0, nv1;
  };
  auto item_info = [&](int j) {
    Item it;
    it.bh = j % p.BH;
    int pair = j / p.BH;
    if (p.causal) pair = p.n_pairs - 1 - pair;             // longest rows first
    it.qt0 = 2 * pair;
    it.qt1 = 2 * pair + 1;
    it.kt_end = p.causal ? min(it.qt1, p.n_qt - 1) + 1 : p.n_qt;
    it.nv0 = it.qt0 < p.n_qt ? (p.causal ? it.qt0 + 1 : p.n_qt) : 0;
    it.nv1 = it.qt1 < p.n_qt ? (p.causal ? it.qt1 + 1 : p.n_qt) : 0;
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_Q + 0), 1);
    mbar_init(bar(L::B_Q + 1), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(L::B_FULL + s), 1);
      mbar_init(bar(L::B_EMPTY + s), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(L::B_S + w), 1);
      mbar_init(bar(L::B_P + w), 4);
      mbar_init(bar(L::B_PH + w), 4);
      mbar_init(bar(L::B_O + w), 1);
    }
    mbar_init(bar(L::B_DONE), 1);
    mbar_init(bar(L::B_QFREE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  auto visible = [&](int qt, int kt) { return qt < p.n_qt && (!p.causal || kt <= qt); };

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_vt);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued[L::STAGES] = {};
      bool ok = true;
      for (int k = 0; ok; ++k) {
      const int j = item_index(k);
      if (j < 0) break;
      const Item it = item_info(j);
      const int bh = it.bh, qt0 = it.qt0, qt1 = it.qt1, kt_end = it.kt_end;
      // the Q buffers are free once the previous item's S products are done
      if (k > 0 && !(ok = mbar_wait(bar(L::B_QFREE), (k - 1) & 1, wc))) break;
      for (int w = 0; w < 2; ++w) {
        const int qt = qt0 + w;
        if (qt >= p.n_qt) {              // no such tile: complete the phase empty
          mbar_arrive(bar(L::B_Q + w));
          continue;
        }
        mbar_arrive_expect_tx(bar(L::B_Q + w), L::TILE_BYTES);
        tma_load_3d(sbase + L::Q_OFF + w * L::TILE_BYTES, &p.tm_q, bar(L::B_Q + w), 0, qt * TILE, bh, pol_q);
      }
      for (int kt = 0; kt < kt_end && ok; ++kt) {
        if (!(visible(qt0, kt) || visible(qt1, kt))) continue;
        for (int which = 0; which < 2; ++which) {          // K_j, then V_j^T
          if (!mbar_wait(bar(L::B_EMPTY + slot), phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = bar(L::B_FULL + slot);
          mbar_arrive_expect_tx(fb, L::TILE_BYTES);
          const uint32_t dst = sbase + L::RING_OFF + slot * L::TILE_BYTES;
          if (which == 0)
            tma_load_3d(dst, &p.tm_k, fb, 0, kt * TILE, bh, pol_kv);
          else
            tma_load_3d(dst, &p.tm_vt, fb, kt * TILE, 0, bh, pol_kv);   // keys kt*128.., all 128 d rows
          ++issued[slot];
          if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }
        }
      }
      }
      if (!ok) {
        for (int s = 0; s < L::STAGES; ++s)
          if (issued[s]) fp8_drain(bar(L::B_FULL + s), (issued[s] - 1) & 1u, 100000000ull);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t IDESC = idesc_e4m3(128, 128);
    bool ok = true;
    const uint64_t dq0 = sdesc_sw128(sbase + L::Q_OFF, 16, 1024);
    const uint64_t dq1 = sdesc_sw128(sbase + L::Q_OFF + L::TILE_BYTES, 16, 1024);
    const uint64_t d_ring = sdesc_sw128(sbase + L::RING_OFF, 16, 1024);   // K and V^T slots, K-major
    constexpr uint32_t SLOT16 = L::TILE_BYTES >> 4;
    // S_w = Q_w K^T: 4 k-steps of 32 e4m3 (32 bytes inside the 128-byte row)
    auto issue_s = [&](uint64_t dq, uint32_t scol, int kslot) {
      const uint64_t dk = d_ring + static_cast<uint64_t>(kslot) * SLOT16;
#pragma unroll
      for (int k = 0; k < D / 32; ++k) mma_ss_f8_elect(tmem + scol, dq + 2 * k, dk + 2 * k, IDESC, k > 0 ? 1u : 0u);
    };
    // O_w += P_w V: 4 k-steps of 32 keys; P from tensor memory (8 columns of
    // 4 e4m3 per step), V^T K-major (32 bytes per step)
    auto issue_pv_half = [&](uint32_t ocol, uint32_t scol, int vslot, bool started, int k0) {
      const uint64_t dv = d_ring + static_cast<uint64_t>(vslot) * SLOT16;
#pragma unroll
      for (int kk = 0; kk < TILE / 64; ++kk) {
        const int k = k0 + kk;
        mma_ts_f8_elect(tmem + ocol, tmem + scol + 8 * k, dv + 2 * k, IDESC, (started || k > 0) ? 1u : 0u);
      }
    };
    // P_w V in two halves: keys 0-63 once the softmax warps have published
    // that half of P, the rest once all of P is in (one phase bit: both
    // barriers complete once per tile)
    auto pv = [&](int w, uint32_t& ph, int vslot, bool started) {
      const uint32_t ocol = w ? L::O_COL1 : L::O_COL0, scol = w ? L::S_COL1 : L::S_COL0;
      if (!mbar_wait_warp(bar(L::B_PH + w), ph, wc)) return false;
      tc_fence_after();
      issue_pv_half(ocol, scol, vslot, started, 0);
      if (!mbar_wait_warp(bar(L::B_P + w), ph, wc)) return false;
      tc_fence_after();
      issue_pv_half(ocol, scol, vslot, started, TILE / 64);
      ph ^= 1u;
      return true;
    };
    int slot = 0;
    uint32_t phase = 0;
    uint32_t pph0 = 0, pph1 = 0;
    for (int k = 0; ok; ++k) {
    const int j = item_index(k);
    if (j < 0) break;
    const Item it = item_info(j);
    const int qt0 = it.qt0, qt1 = it.qt1, kt_end = it.kt_end, nv0 = it.nv0, nv1 = it.nv1;
    // Q of both tiles (a missing tile's phase completes empty); see the bf16
    // forward for why the next item's S and P V need no further barrier
    if (!(ok = mbar_wait_warp(bar(L::B_Q + 0), k & 1, wc))) break;
    if (!(ok = mbar_wait_warp(bar(L::B_Q + 1), k & 1, wc))) break;
    int done0 = 0, done1 = 0;
    bool has_prev = false, pf0 = false, pf1 = false;
    int pvslot = 0;
    uint32_t pvphase = 0;
    for (int kt = 0; kt < kt_end && ok; ++kt) {
      const bool f0 = visible(qt0, kt);
      const bool f1 = visible(qt1, kt);
      if (!(f0 || f1)) continue;
      const int kslot = slot;
      const uint32_t kphase = phase;
      if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }
      const int vslot = slot;
      const uint32_t vphase = phase;
      if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }
      if (!(ok = mbar_wait_warp(bar(L::B_FULL + kslot), kphase, wc))) break;
      tc_fence_after();
      if (has_prev) {
        if (!(ok = mbar_wait_warp(bar(L::B_FULL + pvslot), pvphase, wc))) break;
      }
      if (has_prev && pf0) {
        if (!(ok = pv(0, pph0, pvslot, done0 > 0))) break;
        if (++done0 == nv0) mma_commit_elect(bar(L::B_O + 0));
      }
      if (f0) {
        issue_s(dq0, L::S_COL0, kslot);
        mma_commit_elect(bar(L::B_S + 0));
      }
      if (has_prev && pf1) {
        if (!(ok = pv(1, pph1, pvslot, done1 > 0))) break;
        if (++done1 == nv1) mma_commit_elect(bar(L::B_O + 1));
      }
      if (f1) {
        issue_s(dq1, L::S_COL1, kslot);
        mma_commit_elect(bar(L::B_S + 1));
      }
      mma_commit_elect(bar(L::B_EMPTY + kslot));
      if (has_prev) mma_commit_elect(bar(L::B_EMPTY + pvslot));
      has_prev = true;
      pf0 = f0;
      pf1 = f1;
      pvslot = vslot;
      pvphase = vphase;
    }
    if (ok) mma_commit_elect(bar(L::B_QFREE));   // all S of this item issued: Q may be reloaded
    if (ok && has_prev) {
      ok = mbar_wait_warp(bar(L::B_FULL + pvslot), pvphase, wc);
      if (ok && pf0) {
        ok = pv(0, pph0, pvslot, done0 > 0);   // (the phases continue into the next item)
        if (ok) mma_commit_elect(bar(L::B_O + 0));
      }
      if (ok && pf1) {
        ok = pv(1, pph1, pvslot, done1 > 0);
        if (ok) mma_commit_elect(bar(L::B_O + 1));
      }
      if (ok) mma_commit_elect(bar(L::B_EMPTY + pvslot));
    }
    }
    mma_commit_elect(bar(L::B_DONE));
    if (lane == 0) fp8_drain(bar(L::B_DONE), 0, 1000000000ull);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int w = static_cast<int>(warp >> 2);
    const uint32_t quarter = warp & 3u;
    uint32_t sphase = 0;   // phase of this tile's S barrier, continued across items
    int n_out = 0;         // items whose O this group has read (phase of its O barrier)
    bool ok = true;
    for (int k = 0; ok; ++k) {
    const int j = item_index(k);
    if (j < 0) break;
    const Item it = item_info(j);
    const int bh = it.bh, nv0 = it.nv0, nv1 = it.nv1;
    const int qt = it.qt0 + w;
    if (qt < p.n_qt) {
      const int row = static_cast<int>(quarter * 32 + lane);
      const uint32_t s_addr = tmem_addr(tmem, quarter * 32, w ? L::S_COL1 : L::S_COL0);
      const uint32_t o_addr = tmem_addr(tmem, quarter * 32, w ? L::O_COL1 : L::O_COL0);
      const float dqk = (p.q_descale ? __ldg(p.q_descale + bh) : 1.f) * (p.k_descale ? __ldg(p.k_descale + bh) : 1.f);
      const float sl2 = p.scale_log2 * dqk;
      float m = -INFINITY;   // running max of S * log2 e (exp2 units)
      float l = 0.f;         // sum of exp2(S - m + 8), fp32
      bool has_o = false;
      const int n_vis = w ? nv1 : nv0;
      // only the last visited tile can need a per-element mask (causal
      // diagonal, keys past N)
      const int last_kt = n_vis - 1;
      int last_lim = p.N - last_kt * TILE;
      if (p.causal && last_kt == qt) last_lim = min(last_lim, row + 1);
      for (int rr = 0; rr < n_vis; ++rr) {
        if (!mbar_wait_warp(bar(L::B_S + w), sphase, wc)) { ok = false; break; }
        sphase ^= 1u;
        tc_fence_after();
        uint32_t r[128];
        tmem_ld_x128(s_addr, r);
        float* s = reinterpret_cast<float*>(r);
        if (rr == n_vis - 1 && last_lim < TILE) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= last_lim) s[c] = -INFINITY;
        }
        float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
        for (int c = 4; c < 124; c += 8) {
          mx0 = fmax3(mx0, s[c], s[c + 1]);
          mx1 = fmax3(mx1, s[c + 2], s[c + 3]);
          mx2 = fmax3(mx2, s[c + 4], s[c + 5]);
          mx3 = fmax3(mx3, s[c + 6], s[c + 7]);
        }
        mx0 = fmax3(mx0, s[124], s[125]);
        mx1 = fmax3(mx1, s[126], s[127]);
        const float m_tile = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
        const bool need = m_tile > m + 4.f;
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m - m_tile);                  // 0 when m = -inf
          m = m_tile;
        }
        if (has_o && __any_sync(0xffffffffu, need)) {
          // O rescaled before any of this tile's P is published (the P V
          // halves accumulate onto it); O may be read here: S(j) completing
          // implies the previous PV is done.  16 columns at a time: S is live.
#pragma unroll 1
          for (int c = 0; c < D; c += 16) {
            uint32_t ov[16];
            tmem_ld_x16(o_addr + c, ov);
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st_x16(o_addr + c, ov);
          }
        }
        // P = exp2(S sl2 - m + 8) in (0, 256]; four e4m3 per 32-bit column,
        // 32 columns in all, written over the first 32 columns of S
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 off = make_float2(4.f - m, 4.f - m);
        float2 la = make_float2(0.f, 0.f), lb = la;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = 64 * q + 4 * e;
            const float2 x0 = ffma2(make_float2(s[c], s[c + 1]), sl2v, off);
            const float2 x1 = ffma2(make_float2(s[c + 2], s[c + 3]), sl2v, off);
            const float2 p0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
            const float2 p1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
            la = fadd2(la, p0);
            lb = fadd2(lb, p1);
            pk[e] = pack_e4m3x2(p0.x, p0.y) | (pack_e4m3x2(p1.x, p1.y) << 16);
          }
          if (q == 1) {
            // keys 0-63 of P are stored: publish that half (its store
            // completed while keys 64-127 were computed)
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::B_PH + w));
          }
          tmem_st_x16_async(s_addr + 16 * q, pk);
        }
        l = l * alpha + ((la.x + la.y) + (lb.x + lb.y));
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_P + w));
        has_o = true;
      }
      if (ok) {
        const bool row_ok = qt * TILE + row < p.N;
        const size_t grow = static_cast<size_t>(bh) * p.N + static_cast<size_t>(qt) * TILE + row;
        __nv_bfloat16* orow = p.o + grow * D;
        if (n_vis > 0) {
          ok = mbar_wait_warp(bar(L::B_O + w), n_out & 1, wc);
          ++n_out;
          if (ok) {
            tc_fence_after();
            const float inv = (p.v_descale ? __ldg(p.v_descale + bh) : 1.f) / l;
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t ov[32];
              tmem_ld_x32(o_addr + c, ov);
              uint4 pkd[4];
              uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pw[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv, __uint_as_float(ov[2 * i + 1]) * inv);
              if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = pkd[i];
              }
            }
            if (row_ok) p.lse[grow] = (m - 4.f + __log2f(l)) * 0.69314718055994530942f;
          }
        } else if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          p.lse[grow] = -INFINITY;
        }
      }
    }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

int launch_fwd_fp8(const Fp8Params& p, cudaStream_t stream) {
  using L = Fp8Layout;
  static_assert(L::SMEM_BYTES <= 232448, "shared memory budget");
  static SmemAttrOnce attr;
  if (!attr.ensure(reinterpret_cast<const void*>(fa_fwd_fp8_kernel), L::SMEM_BYTES)) return -4;
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return -4;
  const long long items = static_cast<long long>(p.n_pairs) * p.BH;
  const long long grid = items < sms ? items : sms;      // persistent: at most one CTA per SM
  fa_fwd_fp8_kernel<<<static_cast<unsigned>(grid), L::THREADS, L::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// V [BH][N][128] bytes -> V^T [BH][128][npad] bytes, zeros for keys N..npad-1.
// One CTA per 128-key block of one (b, h): 16-byte loads of the 128 x 128
// byte tile into shared memory, 4 x 4 byte-block transposes (byte_perm),
// 16-byte stores.
__global__ void __launch_bounds__(256) fp8_transpose_v_kernel(const uint8_t* __restrict__ v, uint8_t* __restrict__ vt,
                                                              int N, int npad) {
  __shared__ uint32_t tin[128][33];   // [key][d / 4], padded against bank conflicts
  __shared__ uint32_t tout[128][33];  // [d][key / 4]
  const int bh = blockIdx.y;
  const int k0 = blockIdx.x * 128;
  const uint8_t* src = v + (static_cast<size_t>(bh) * N) * 128;
  for (int i = threadIdx.x; i < 128 * 8; i += 256) {      // 8 x 16 bytes per key row
    const int key = i >> 3, part = i & 7;
    uint4 x = make_uint4(0, 0, 0, 0);
    if (k0 + key < N) x = __ldg(reinterpret_cast<const uint4*>(src + static_cast<size_t>(k0 + key) * 128) + part);
    tin[key][4 * part + 0] = x.x;
    tin[key][4 * part + 1] = x.y;
    tin[key][4 * part + 2] = x.z;
    tin[key][4 * part + 3] = x.w;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < 32 * 32; b += 256) {       // 4 x 4 byte blocks
    const int kb = b >> 5, db = b & 31;                    // keys 4kb.., d bytes 4db..
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = tin[4 * kb + i][db];
    // y[t] = byte t (d = 4 db + t) of keys 4 kb .. 4 kb + 3
    const uint32_t a0 = __byte_perm(w[0], w[1], 0x5140), a1 = __byte_perm(w[0], w[1], 0x7362);
    const uint32_t a2 = __byte_perm(w[2], w[3], 0x5140), a3 = __byte_perm(w[2], w[3], 0x7362);
    tout[4 * db + 0][kb] = __byte_perm(a0, a2, 0x5410);
    tout[4 * db + 1][kb] = __byte_perm(a0, a2, 0x7632);
    tout[4 * db + 2][kb] = __byte_perm(a1, a3, 0x5410);
    tout[4 * db + 3][kb] = __byte_perm(a1, a3, 0x7632);
  }
  __syncthreads();
  uint8_t* dst = vt + static_cast<size_t>(bh) * 128 * npad;
  for (int i = threadIdx.x; i < 128 * 8; i += 256) {      // 128 d rows x 8 x 16 bytes
    const int d = i >> 3, part = i & 7;
    const int key = k0 + 16 * part;
    if (key >= npad) continue;
    const uint4 x = make_uint4(tout[d][4 * part], tout[d][4 * part + 1], tout[d][4 * part + 2], tout[d][4 * part + 3]);
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(d) * npad + key) = x;
  }
}

int launch_fp8_transpose_v(const uint8_t* v, uint8_t* vt, int BH, int N, int npad, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((npad + 127) / 128), static_cast<unsigned>(BH));
  fp8_transpose_v_kernel<<<grid, 256, 0, stream>>>(v, vt, N, npad);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace fa
