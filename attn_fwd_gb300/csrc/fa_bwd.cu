// fa_bwd.cu -- backward main kernel for sm_103a: recompute P from Q, K and
// the saved LSE, then accumulate dK, dV and the fp32 dQ accumulator.
//
// What one CTA computes ("FlashAttention" notes, "Backward Pass of
// flashattention"): for one 128-row key tile K_j, V_j of one (batch, head)
// and every visible query tile Q_i (BQ rows), with the scale's chain rule:
//   S_ij  = scale * Q_i K_j^T,  P_ij = exp(S_ij - LSE_i)      (recompute)
//   dV_j += P_ij^T dO_i
//   dP_ij = dO_i V_j^T,  dS_ij = P_ij o (dP_ij - D_i)           (D_i = dO_i . O_i)
//   dK_j += scale * dS_ij^T Q_i
//   dQ_i += dS_ij K_j   (fp32 reductions into the accumulator; scaled later)
// Masks are regenerated from (i, j) or the block mask, never stored.  K_j and
// V_j stay in shared memory for the whole loop (the key/value-stationary loop
// order of "Transformer 入门", V1), so dK_j and dV_j are written once.
//
// The five products run on the tensor cores (tcgen05, fp32 accumulators in
// tensor memory), computed transposed so that the key index is the
// tensor-memory lane, i.e. one softmax thread per key:
//   S^T  = K_j Q_i^T          (M=128 keys, N=BQ, K=d)   A,B K-major
//   dP^T = V_j dO_i^T         (M=128, N=BQ, K=d)        A,B K-major
//   dV  += P^T dO_i           (M=128, N=d, K=BQ)        A = P^T, B MN-major
//   dK  += dS^T Q_i           (M=128, N=d, K=BQ)        A = dS^T, B MN-major
// (A of dV from tensor memory; A of dK from tensor memory at d=128, from
// shared memory at d=64, where the 512 columns hold P^T but not dS^T too)
//   d=128: dQ^T = K_j^T dS^T  (M=d=128, N=BQ=64, K=128) A,B MN-major
//   d=64:  dQ   = dS K_j      (M=BQ=128, N=d, K=128)    A,B MN-major
// The d=128 form keeps the head-dim index on the lanes, so each warp's fp32
// reduction covers 32 consecutive floats of one dQ row (128-byte coalesced).
//
// Warp roles (14 warps): 0-7 recompute P and dS (thread = key row; warps
// 0-3 take the first half of the step's query columns, 4-7 the second half,
// so two warps per SM sub-partition share the CUDA-core work) and write P^T
// (bf16) to tensor memory and dS^T (bf16, 128-byte swizzle) to a
// double-buffered shared-memory tile (d=128: to tensor memory too); 8-11 drain dQ from
// tensor memory into the fp32 accumulator; 12 issues MMAs; 13 loads K_j, V_j
// once and Q_i, dO_i, LSE_i, D_i per step into a two-stage ring.
#include "fa_common.cuh"
#include "fa_dropout.cuh"
#include "fa_ptx.cuh"

namespace fa {

template <int D>
struct BwdLayout {
  static constexpr int BQ = (D == 128) ? 64 : 128;          // query rows per step
  static constexpr bool DQ_T = (D == 128);                  // dQ computed transposed
  static constexpr int NCH = D / 64;
  static constexpr int KV_CHUNK = TILE * 128;               // [128 rows][128 B]
  static constexpr int KV_BYTES = NCH * KV_CHUNK;           // 128 x D bf16
  static constexpr int Q_CHUNK = BQ * 128;                  // [BQ rows][128 B]
  static constexpr int Q_BYTES = NCH * Q_CHUNK;             // BQ x D bf16
  static constexpr int STAGES = 3;                          // Q_i/dO_i ring: loads run two steps ahead
  static constexpr int ST_Q = 0;
  static constexpr int ST_DO = Q_BYTES;
  static constexpr int ST_LSE = 2 * Q_BYTES;
  static constexpr int ST_DV = 2 * Q_BYTES + BQ * 4;
  static constexpr int STAGE_BYTES = ((2 * Q_BYTES + 2 * BQ * 4) + 1023) / 1024 * 1024;
  static constexpr int PT_CHUNK = TILE * 128;               // [128 key rows][64 queries]
  static constexpr int PT_BYTES = (BQ / 64) * PT_CHUNK;     // 128 x BQ bf16
  // Shared dS^T area (2 x PT_BYTES): dS^T double-buffered there, so step
  // i+1 can write while dQ(i) still reads step i's; P^T lives in tensor
  // memory (and at d=128 a copy of dS^T too).
  static constexpr int PBUFS = 1;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = KV_BYTES;
  static constexpr int RING_OFF = 2 * KV_BYTES;
  static constexpr int PT_OFF = RING_OFF + STAGES * STAGE_BYTES;   // buffer b: P^T at +2b*PT, dS^T at +(2b+1)*PT
  static constexpr int BAR_OFF = PT_OFF + PBUFS * 2 * PT_BYTES;
  // barriers
  static constexpr int B_KV = 0;
  static constexpr int B_FULL = 1;                       // STAGES
  static constexpr int B_EMPTY = B_FULL + STAGES;        // STAGES
  static constexpr int B_SDP = B_EMPTY + STAGES;         // S^T and dP^T of a step in tensor memory
  static constexpr int B_SDP_FREE = B_SDP + 1;           // ... and read out (one arrival per warp)
  static constexpr int B_DS = B_SDP_FREE + 1;            // P^T, dS^T of a step written (one arrival per warp)
  static constexpr int B_PFREE = B_DS + 1;               // dV, dK done reading P^T (d=128: dS^T) in TMEM
  static constexpr int B_DSF = B_PFREE + 1;              // 2: dS^T smem buffer b consumed (dQ; d=64: dK too)
  static constexpr int B_DQ = B_DSF + 2;                 // dQ of a step in tensor memory
  static constexpr int B_DQ_FREE = B_DQ + 1;             // ... and read out (one arrival per warp)
  static constexpr int B_DONE = B_DQ_FREE + 1;
  static constexpr int NBARS = B_DONE + 1;
  // block masks: list of the visible 128-row query blocks of this key tile
  static constexpr int LIST_OFF = BAR_OFF + NBARS * 8 + 16;
  static constexpr int LIST_BYTES = MAX_SPARSE_TILES * 2 + 16;
  static constexpr int SMEM_BYTES = LIST_OFF + LIST_BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t COL_S = 0;
  static constexpr uint32_t COL_DP = BQ;
  static constexpr uint32_t COL_DQ = 2 * BQ;
  static constexpr uint32_t COL_DV = (D == 128) ? 256 : 320;
  static constexpr uint32_t COL_DK = 384;     // dK [384, 384 + d)
  // d=128: P^T and dS^T (bf16 pairs, 32 columns each) also go to tensor
  // memory, so dV and dK read their A operand from there (TS form) instead of
  // shared memory.  Map at d=128: S^T [0,64) dP^T [64,128) dQ^T [128,192)
  // P^T [192,224) dS^T [224,256) dV [256,384) dK [384,512).  d=64 has no room
  // left (S^T and dP^T take 128 columns each).
  static constexpr bool DST_TMEM = (D == 128);   // dS^T also in TMEM (dK as a TS product)
  // P^T: d=128 in the free columns between dQ^T [128,192) and dV [256,384);
  // d=64 in the last 64 columns, after dK [384,448)
  static constexpr uint32_t COL_PT = (D == 128) ? 192 : 448;
  static constexpr uint32_t COL_DST = 224;
  static constexpr int THREADS = 448;
  static constexpr int W_DRAIN = 8;      // first drain warp
  static constexpr int W_MMA = 12;
  static constexpr int W_TMA = 13;
  static constexpr int RECOMPUTE_WARPS = 8;
};

// The query tiles (BQ rows) a key tile visits, in increasing order, as steps
// 0..count-1.  No mask: all; causal: from the first tile that reaches the
// key tile's diagonal; block mask: the 128-row query blocks whose mask byte
// for this key tile is nonzero (with the causal flag, only blocks at or below
// the diagonal), compacted once per CTA by one warp into a shared-memory list,
// each split into 128 / BQ steps.
template <int BQ>
struct StepSched {
  static constexpr int SUB = TILE / BQ;
  const uint16_t* list;
  int mask_kind;
  int first;      // causal: the first visible query tile
  int count;

  __device__ __forceinline__ int qi(int i) const {
    if (mask_kind & MASK_BLOCK) return static_cast<int>(list[i / SUB]) * SUB + i % SUB;
    return first + i;
  }
};

__device__ __forceinline__ int build_sparse_column(const BwdParams& p, int kt, uint16_t* list, uint32_t lane) {
  int n = 0;
  for (int base = 0; base < p.n_kt; base += 32) {
    const int qb = base + static_cast<int>(lane);
    const size_t at = static_cast<size_t>(qb) * p.n_kt + kt;
    const bool v = qb < p.n_kt && (!(p.mask_kind & MASK_CAUSAL) || qb >= kt) &&
                   dcheck(at < static_cast<size_t>(p.n_kt) * p.n_kt, p.status) && __ldg(p.block_mask + at) != 0;
    const uint32_t m = __ballot_sync(0xffffffffu, v);
    if (v) list[n + __popc(m & ((1u << lane) - 1u))] = static_cast<uint16_t>(qb);
    n += __popc(m);
  }
  return n;
}

__device__ __forceinline__ void mbar_drain_b(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

// P^T and dS^T of one key row over 32 query columns c0 .. c0+31 of a step:
// P = exp2(S^T * scale * log2 e - LSE * log2 e), dS = P (dP - D), packed as
// bf16 pairs.  nlse and nd hold -LSE * log2 e and -D per query column.
// MASKED: P = 0 where the query q (q_base + column) is at or past q_end, or,
// causal, where q < key.  DROP: with Z the keep bit of the pair (keep_bit
// layout of `keep`) and c the dropout scale, the dV operand is P Z c and
// dS = P (Z c dP~ - D), dP~ = dO V^T being the gradient of the dropped P.
template <bool MASKED, bool DROP>
__device__ __forceinline__ void recompute32(const uint32_t (&sr)[32], const uint32_t (&dr)[32], const float* nlse,
                                            const float* nd, int c0, float2 sl2v, int q_base, int q_end, int key,
                                            bool causal, uint32_t keep, float dscale, uint32_t (&pt_pk)[16],
                                            uint32_t (&ds_pk)[16]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {                        // 8 queries per group
    const int cq = c0 + 8 * j;
    const float4 l0 = *reinterpret_cast<const float4*>(nlse + cq);
    const float4 l1 = *reinterpret_cast<const float4*>(nlse + cq + 4);
    const float4 d0 = *reinterpret_cast<const float4*>(nd + cq);
    const float4 d1 = *reinterpret_cast<const float4*>(nd + cq + 4);
    const float2 nl[4] = {make_float2(l0.x, l0.y), make_float2(l0.z, l0.w), make_float2(l1.x, l1.y),
                          make_float2(l1.z, l1.w)};
    const float2 ndv[4] = {make_float2(d0.x, d0.y), make_float2(d0.z, d0.w), make_float2(d1.x, d1.y),
                           make_float2(d1.z, d1.w)};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 8 * j + 2 * e;                     // register index within the 32 columns
      const float2 x = ffma2(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), sl2v, nl[e]);
      float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      if constexpr (MASKED) {
        const int q0 = q_base + cq + 2 * e;
        if (!(q0 < q_end && (!causal || q0 >= key))) pv.x = 0.f;
        if (!(q0 + 1 < q_end && (!causal || q0 + 1 >= key))) pv.y = 0.f;
      }
      const float2 dpv = make_float2(__uint_as_float(dr[k]), __uint_as_float(dr[k + 1]));
      if constexpr (DROP) {
        const uint32_t f = keep >> keep_bit(k);             // columns k, k + 1: adjacent bits
        const float2 zc = make_float2((f & 1u) ? dscale : 0.f, (f & 2u) ? dscale : 0.f);
        const float2 ptv = fmul2(pv, zc);
        const float2 ds = fmul2(pv, ffma2(zc, dpv, ndv[e]));
        pt_pk[4 * j + e] = pack_bf16x2(ptv.x, ptv.y);
        ds_pk[4 * j + e] = pack_bf16x2(ds.x, ds.y);
      } else {
        const float2 ds = fmul2(pv, fadd2(dpv, ndv[e]));
        pt_pk[4 * j + e] = pack_bf16x2(pv.x, pv.y);
        ds_pk[4 * j + e] = pack_bf16x2(ds.x, ds.y);
      }
    }
  }
}

template <int D, bool DROP>
__global__ void __launch_bounds__(448, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
  using L = BwdLayout<D>;
  constexpr int BQ = L::BQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  // CTA order: bands of up to 8 heads; within a band key tile outer, head
  // inner.  A band's Q, dO and dQ accumulator stay L2-resident while its key
  // tiles run, and causal key tiles with the most query tiles start first.
  const int band_heads = p.BH < 8 ? p.BH : 8;
  const int band = blockIdx.x / (band_heads * p.n_kt);
  const int in_band = blockIdx.x % (band_heads * p.n_kt);
  const int heads_here = min(band_heads, p.BH - band * band_heads);
  const int kt = in_band / heads_here;
  const int bh = band * band_heads + in_band % heads_here;
  const int n_qi = (p.N + BQ - 1) / BQ;
  const int qi_begin = (p.mask_kind == MASK_CAUSAL) ? (kt * TILE) / BQ : 0;
  uint16_t* list = reinterpret_cast<uint16_t*>(smem + L::LIST_OFF);
  int* list_count = reinterpret_cast<int*>(smem + L::LIST_OFF + MAX_SPARSE_TILES * 2);
  if ((p.mask_kind & MASK_BLOCK) && warp == 0) {
    const int n = build_sparse_column(p, kt, list, lane);
    if (lane == 0) *list_count = n;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(L::B_KV), 1);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(L::B_FULL + s), 1);
      mbar_init(bar(L::B_EMPTY + s), 1);
    }
    mbar_init(bar(L::B_SDP), 1);
    mbar_init(bar(L::B_SDP_FREE), L::RECOMPUTE_WARPS);   // one arrival per warp
    mbar_init(bar(L::B_DS), L::RECOMPUTE_WARPS);
    mbar_init(bar(L::B_PFREE), 1);
    mbar_init(bar(L::B_DSF + 0), 1);
    mbar_init(bar(L::B_DSF + 1), 1);
    mbar_init(bar(L::B_DQ), 1);
    mbar_init(bar(L::B_DQ_FREE), 4);
    mbar_init(bar(L::B_DONE), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == L::W_MMA) {
    tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};

  const int n_steps = (p.mask_kind & MASK_BLOCK) ? *list_count * StepSched<BQ>::SUB : n_qi - qi_begin;
  const StepSched<BQ> sched{list, p.mask_kind, qi_begin, n_steps};

  if (warp == L::W_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_do);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      const uint64_t pol_first = l2_policy_evict_first();
      const uint64_t pol_last = l2_policy_evict_last();
      uint32_t issued[L::STAGES] = {};
      bool ok = true;
      bool kv_issued = false;
      if (n_steps > 0) {
        mbar_arrive_expect_tx(bar(L::B_KV), 2 * L::KV_BYTES);
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_3d(sbase + L::K_OFF + c * L::KV_CHUNK, &p.tm_k, bar(L::B_KV), c * 64, kt * TILE, bh, pol_first);
          tma_load_3d(sbase + L::V_OFF + c * L::KV_CHUNK, &p.tm_v, bar(L::B_KV), c * 64, kt * TILE, bh, pol_first);
        }
        kv_issued = true;
      }
      for (int step = 0; step < n_steps && ok; ++step) {
        const int qi = sched.qi(step);
        const int st = step % L::STAGES;
        if (!mbar_wait(bar(L::B_EMPTY + st), ((step / L::STAGES) & 1) ^ 1, wc)) { ok = false; break; }
        const uint32_t fb = bar(L::B_FULL + st);
        const uint32_t sb = sbase + L::RING_OFF + st * L::STAGE_BYTES;
        // -LSE * log2 e and -D of the step's query rows (rows past N are zero;
        // each head's row is padded to a multiple of 128, so the copy stays in
        // bounds and 16-byte aligned)
        const size_t row0 = static_cast<size_t>(bh) * p.npad + static_cast<size_t>(qi) * BQ;
        const bool vec_ok = dcheck(row0 + BQ <= static_cast<size_t>(p.BH) * p.npad, p.status);
        mbar_arrive_expect_tx(fb, 2 * L::Q_BYTES + (vec_ok ? 2 * BQ * 4 : 0));
        for (int c = 0; c < L::NCH; ++c) {
          tma_load_3d(sb + L::ST_Q + c * L::Q_CHUNK, &p.tm_q, fb, c * 64, qi * BQ, bh, pol_last);
          tma_load_3d(sb + L::ST_DO + c * L::Q_CHUNK, &p.tm_do, fb, c * 64, qi * BQ, bh, pol_last);
        }
        if (vec_ok) {
          bulk_load(sb + L::ST_LSE, p.nlse + row0, BQ * 4, fb);
          bulk_load(sb + L::ST_DV, p.nd + row0, BQ * 4, fb);
        }
        ++issued[st];
      }
      if (!ok) {
        if (kv_issued) mbar_drain_b(bar(L::B_KV), 0, 100000000ull);
        for (int s = 0; s < L::STAGES; ++s)
          if (issued[s]) mbar_drain_b(bar(L::B_FULL + s), (issued[s] - 1) & 1u, 100000000ull);
      }
    }
  } else if (warp == L::W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // Warp-uniform schedule; one elected lane issues each tcgen05 instruction.
    // Descriptors are a base plus a compile-time offset (16-byte units).
    if (n_steps > 0) {
      constexpr uint32_t ID_S = idesc_bf16(128, BQ, false, false);     // S^T, dP^T
      constexpr uint32_t ID_G = idesc_bf16(128, D, false, true);       // dV, dK
      constexpr uint32_t ID_Q = L::DQ_T ? idesc_bf16(128, BQ, true, true) : idesc_bf16(128, D, true, true);
      constexpr uint32_t STAGE16 = L::STAGE_BYTES >> 4;
      const uint64_t dK_kmaj = sdesc_sw128(sbase + L::K_OFF, 16, 1024);             // K as A of S^T
      const uint64_t dV_kmaj = sdesc_sw128(sbase + L::V_OFF, 16, 1024);             // V as A of dP^T
      const uint64_t dK_mn = sdesc_sw128(sbase + L::K_OFF, L::KV_CHUNK, 1024);      // K^T (d=128) / K (d=64), MN-major
      const uint64_t dQ_kmaj = sdesc_sw128(sbase + L::RING_OFF + L::ST_Q, 16, 1024);    // stage 0 Q, K-major
      const uint64_t dO_kmaj = sdesc_sw128(sbase + L::RING_OFF + L::ST_DO, 16, 1024);   // stage 0 dO, K-major
      const uint64_t dQ_mn = sdesc_sw128(sbase + L::RING_OFF + L::ST_Q, L::Q_CHUNK, 1024);   // stage 0 Q, MN-major
      const uint64_t dO_mn = sdesc_sw128(sbase + L::RING_OFF + L::ST_DO, L::Q_CHUNK, 1024);  // stage 0 dO, MN-major
      const uint32_t pt = sbase + L::PT_OFF;                                         // dS^T buffers
      // dS^T, step i in buffer i % 2: K-major as the A operand of dK (d=64),
      // MN-major as the B (d=128) or A (d=64) operand of the dQ product
      const uint64_t dDS_kmaj0 = sdesc_sw128(pt, 16, 1024);
      const uint64_t dDS_mn0 = sdesc_sw128(pt, L::PT_CHUNK, 1024);
      constexpr uint32_t PT16 = L::PT_BYTES >> 4;
      bool ok = mbar_wait_warp(bar(L::B_KV), 0, wc);

      // S^T = K Q_i^T and dP^T = V dO_i^T for the step held in ring stage st
      auto issue_sdp = [&](int st) {
        const uint64_t so = static_cast<uint64_t>(st) * STAGE16;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ao = ((k >> 2) * L::KV_CHUNK + (k & 3) * 32) >> 4;
          const uint32_t bo = ((k >> 2) * L::Q_CHUNK + (k & 3) * 32) >> 4;
          mma_ss_elect(tmem + L::COL_S, dK_kmaj + ao, dQ_kmaj + so + bo, ID_S, k > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t ao = ((k >> 2) * L::KV_CHUNK + (k & 3) * 32) >> 4;
          const uint32_t bo = ((k >> 2) * L::Q_CHUNK + (k & 3) * 32) >> 4;
          mma_ss_elect(tmem + L::COL_DP, dV_kmaj + ao, dO_kmaj + so + bo, ID_S, k > 0 ? 1u : 0u);
        }
        mma_commit_elect(bar(L::B_SDP));
      };

      if (ok) {
        ok = mbar_wait_warp(bar(L::B_FULL + 0), 0, wc);
        if (ok) {
          tc_fence_after();
          issue_sdp(0);
        }
      }
      for (int i = 0; i < n_steps && ok; ++i) {
        const int st = i % L::STAGES;
        if (i + 1 < n_steps) {
          // the next S^T, dP^T may overwrite tensor memory once step i's are read out
          const int st1 = (i + 1) % L::STAGES;
          if (!(ok = mbar_wait_warp(bar(L::B_SDP_FREE), i & 1, wc))) break;
          if (!(ok = mbar_wait_warp(bar(L::B_FULL + st1), ((i + 1) / L::STAGES) & 1, wc))) break;
          tc_fence_after();
          issue_sdp(st1);
        }
        if (!(ok = mbar_wait_warp(bar(L::B_DS), i & 1, wc))) break;
        tc_fence_after();
        const uint64_t so = static_cast<uint64_t>(st) * STAGE16;
        // dV += P^T dO_i ; dK += dS^T Q_i   (K = BQ queries, 16 per step)
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k) {
          const uint64_t bd = dO_mn + so + ((k * 2048) >> 4);
          mma_ts_elect(tmem + L::COL_DV, tmem + L::COL_PT + 8 * k, bd, ID_G, (i > 0 || k > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int k = 0; k < BQ / 16; ++k) {
          const uint32_t ao = ((k >> 2) * L::PT_CHUNK + (k & 3) * 32) >> 4;
          const uint64_t bd = dQ_mn + so + ((k * 2048) >> 4);
          if constexpr (L::DST_TMEM)
            mma_ts_elect(tmem + L::COL_DK, tmem + L::COL_DST + 8 * k, bd, ID_G, (i > 0 || k > 0) ? 1u : 0u);
          else
            mma_ss_elect(tmem + L::COL_DK, dDS_kmaj0 + static_cast<uint64_t>(i & 1) * PT16 + ao, bd, ID_G,
                         (i > 0 || k > 0) ? 1u : 0u);
        }
        mma_commit_elect(bar(L::B_EMPTY + st));     // Q_i, dO_i are no longer needed after dV, dK
        mma_commit_elect(bar(L::B_PFREE));          // P^T (d=128: and dS^T) in TMEM consumed
        // dQ for this step, once the drain warps have read the previous one
        if (i > 0) {
          if (!(ok = mbar_wait_warp(bar(L::B_DQ_FREE), (i - 1) & 1, wc))) break;
          tc_fence_after();
        }
        const uint64_t dDS_mn = dDS_mn0 + static_cast<uint64_t>(i & 1) * PT16;
#pragma unroll
        for (int k = 0; k < TILE / 16; ++k) {
          const uint32_t o = (k * 2048) >> 4;
          if constexpr (L::DQ_T) {
            // A = K^T: MN-major over d (two 64-wide blocks 16 KB apart), 16 keys per step
            // B = dS^T seen as [queries][keys]: MN-major over the 64 queries
            mma_ss_elect(tmem + L::COL_DQ, dK_mn + o, dDS_mn + o, ID_Q, k > 0 ? 1u : 0u);
          } else {
            // A = dS: MN-major over queries (two 64-wide blocks 16 KB apart)
            // B = K: MN-major over d (one 64-wide block)
            mma_ss_elect(tmem + L::COL_DQ, dDS_mn + o, dK_mn + o, ID_Q, k > 0 ? 1u : 0u);
          }
        }
        mma_commit_elect(bar(L::B_DQ));
        mma_commit_elect(bar(L::B_DSF + (i & 1)));     // dS^T buffer i % 2 consumed (dK, dQ)
      }
      mma_commit_elect(bar(L::B_DONE));
      if (lane == 0) mbar_drain_b(bar(L::B_DONE), 0, 1000000000ull);
    }
    __syncwarp();
  } else if (warp < L::W_DRAIN) {
    // ------------------------------------------------- recompute P and dS
    const uint32_t quarter = warp & 3u;
    const int half = static_cast<int>(warp >> 2);           // which half of the query columns
    const int r = static_cast<int>(quarter * 32 + lane);    // key row in the tile == lane
    const int key = kt * TILE + r;
    const uint32_t lane_base = quarter * 32;
    const float2 sl2v = make_float2(p.scale_log2, p.scale_log2);
    const uint32_t hd = static_cast<uint32_t>(bh % p.H), bd = static_cast<uint32_t>(bh / p.H);
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i) {
      const int qi = sched.qi(i);
      const int st = i % L::STAGES;
      constexpr int COLS = BQ / 2;                           // query columns of this warp
      // dropout keep bits of this key row for the warp's query columns, made
      // before S^T and dP^T are waited for
      uint32_t keep[COLS / 32];
      if constexpr (DROP) {
#pragma unroll
        for (int cc = 0; cc < COLS / 32; ++cc)
          keep[cc] = keep_bits_col(key, qi * BQ + half * COLS + 32 * cc, hd, bd, p.drop.seed_lo, p.drop.seed_hi,
                                   p.drop.add, lane & 3u);
      } else {
#pragma unroll
        for (int cc = 0; cc < COLS / 32; ++cc) keep[cc] = 0;
      }
      if (!(ok = mbar_wait_warp(bar(L::B_SDP), i & 1, wc))) break;
      tc_fence_after();
      const uint8_t* stage = smem + L::RING_OFF + st * L::STAGE_BYTES;
      const float* lse = reinterpret_cast<const float*>(stage + L::ST_LSE);
      const float* dvec = reinterpret_cast<const float*>(stage + L::ST_DV);
      // dS^T of step i into shared buffer i % 2
      uint8_t* const dsT = smem + L::PT_OFF + (i & 1) * L::PT_BYTES;
      const bool causal = (p.mask_kind & MASK_CAUSAL) != 0;
      const bool key_ok = key < p.N;
      const bool need_mask = (causal && qi * BQ < kt * TILE + TILE) || !key_ok || qi * BQ + BQ > p.N;
#pragma unroll 1
      for (int c0 = half * COLS; c0 < (half + 1) * COLS; c0 += 32) {
        uint32_t sr[32], dr[32];
        tmem_ld_x32(tmem_addr(tmem, lane_base, L::COL_S + c0), sr);
        tmem_ld_x32(tmem_addr(tmem, lane_base, L::COL_DP + c0), dr);
        if (c0 + 32 == (half + 1) * COLS) {                  // this warp's last read of S^T, dP^T
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(L::B_SDP_FREE));
        }
        // pass 1: P and dS for these 32 query columns, in registers only (no
        // shared-memory stores in between, so the LSE/D loads can be hoisted);
        // the masked form only for steps that need it (causal diagonal, past N)
        uint32_t pt_pk[16], ds_pk[16];
        const uint32_t kp = keep[(c0 - half * COLS) / 32];
        if (need_mask)
          recompute32<true, DROP>(sr, dr, lse, dvec, c0, sl2v, qi * BQ, key_ok ? p.N : -1, key, causal, kp,
                                  p.drop.scale, pt_pk, ds_pk);
        else
          recompute32<false, DROP>(sr, dr, lse, dvec, c0, sl2v, 0, 0, 0, false, kp, p.drop.scale, pt_pk, ds_pk);
        // pass 2: stores, once the buffers they overwrite have been consumed
        // the dS^T buffer is free once dK(i-2), dQ(i-2) have read it
        if (c0 == half * COLS && i >= 2 &&
            !(ok = mbar_wait_warp(bar(L::B_DSF + (i & 1)), ((i >> 1) - 1) & 1, wc)))
          break;
        uint8_t* drow = dsT + (c0 >> 6) * L::PT_CHUNK + r * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int sw = ((((c0 & 63) >> 3) + j) ^ (r & 7)) << 4;   // 128-byte swizzle of the 16-byte chunk
          *reinterpret_cast<uint4*>(drow + sw) = make_uint4(ds_pk[4 * j], ds_pk[4 * j + 1], ds_pk[4 * j + 2], ds_pk[4 * j + 3]);
        }
        // P^T (d=128: and dS^T) in tensor memory are free once dV(i-1), dK(i-1) are done
        if (i >= 1 && !(ok = mbar_wait_warp(bar(L::B_PFREE), (i - 1) & 1, wc))) break;
        // 32 query columns = 16 bf16-pair columns
        tmem_st_x16_async(tmem_addr(tmem, lane_base, L::COL_PT + c0 / 2), pt_pk);
        if constexpr (L::DST_TMEM) tmem_st_x16_async(tmem_addr(tmem, lane_base, L::COL_DST + c0 / 2), ds_pk);
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_DS));
    }
    // ------------------------------------------------- epilogue: dV rows, half the columns each
    const bool key_ok = key < p.N && dcheck(bh < p.BH, p.status);   // rows past N are not stored
    if (ok) {
      constexpr int DC = D / 2;
      __nv_bfloat16* out = p.dv + (static_cast<size_t>(bh) * p.N + static_cast<size_t>(kt) * TILE + r) * D + half * DC;
      if (n_steps > 0 && mbar_wait_warp(bar(L::B_DONE), 0, wc)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < DC; c += 32) {
          uint32_t v[32];
          tmem_ld_x32(tmem_addr(tmem, lane_base, L::COL_DV + half * DC + c), v);
          uint4 o4[4];
          uint32_t* ow = reinterpret_cast<uint32_t*>(o4);
#pragma unroll
          for (int e = 0; e < 16; ++e) ow[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          uint4* dst = reinterpret_cast<uint4*>(out + c);
          if (key_ok)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = o4[e];
        }
      } else if (n_steps == 0 && key_ok) {
        uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
        for (int e = 0; e < DC / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
      }
    }
  } else {
    // ------------------------------------------------- drain dQ; dK epilogue
    const uint32_t quarter = warp & 3u;
    const uint32_t lane_base = quarter * 32;
    const int t = static_cast<int>(quarter * 32 + lane);
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i) {
      const int qi = sched.qi(i);
      if (!(ok = mbar_wait_warp(bar(L::B_DQ), i & 1, wc))) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_x64(tmem_addr(tmem, lane_base, L::COL_DQ), v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(L::B_DQ_FREE));
      const size_t row0 = static_cast<size_t>(bh) * p.N + static_cast<size_t>(qi) * BQ;
      if constexpr (L::DQ_T) {
        // lane t holds head-dim column t of dQ for the BQ = 64 queries of the step
        float* dst = p.dq_acc + row0 * D + t;
        int c_lim = p.N - qi * BQ;                // query rows of the step inside N
        if (!dcheck(row0 + (c_lim < 64 ? c_lim : 64) <= static_cast<size_t>(p.BH) * p.N, p.status)) c_lim = 0;
        if (c_lim >= 64) {
#pragma unroll
          for (int c = 0; c < 64; ++c) atomicAdd(dst + static_cast<size_t>(c) * D, __uint_as_float(v[c]));
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c < c_lim) atomicAdd(dst + static_cast<size_t>(c) * D, __uint_as_float(v[c]));
        }
      } else {
        // lane t holds query row t of the step, 64 head-dim columns
        float4* dst = reinterpret_cast<float4*>(p.dq_acc + (row0 + t) * D);
        if (qi * BQ + t < p.N && dcheck(row0 + t < static_cast<size_t>(p.BH) * p.N, p.status))
#pragma unroll
        for (int c = 0; c < 16; ++c)
          atomicAdd(dst + c, make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                         __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3])));
      }
    }
    // dK rows (lane = key row), scaled by the chain-rule factor
    const bool key_ok = kt * TILE + t < p.N && dcheck(bh < p.BH, p.status);   // rows past N are not stored
    if (ok) {
      __nv_bfloat16* out = p.dk + (static_cast<size_t>(bh) * p.N + static_cast<size_t>(kt) * TILE + t) * D;
      if (n_steps > 0 && mbar_wait_warp(bar(L::B_DONE), 0, wc)) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t v[32];
          tmem_ld_x32(tmem_addr(tmem, lane_base, L::COL_DK + c), v);
          uint4 o4[4];
          uint32_t* ow = reinterpret_cast<uint32_t*>(o4);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            ow[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * p.scale, __uint_as_float(v[2 * e + 1]) * p.scale);
          uint4* dst = reinterpret_cast<uint4*>(out + c);
          if (key_ok)
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = o4[e];
        }
      } else if (n_steps == 0 && key_ok) {
        uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == L::W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool DROP>
static int launch_bwd_t(const BwdParams& p, cudaStream_t stream) {
  using L = BwdLayout<D>;
  static_assert(L::SMEM_BYTES <= 232448, "shared memory budget");
  static SmemAttrOnce attr;
  if (!attr.ensure(reinterpret_cast<const void*>(fa_bwd_kernel<D, DROP>), L::SMEM_BYTES)) return -4;
  const unsigned grid = static_cast<unsigned>(p.n_kt) * static_cast<unsigned>(p.BH);
  fa_bwd_kernel<D, DROP><<<grid, L::THREADS, L::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream) {
  const bool drop = p.drop.t != 0;
  if (d == 128) return drop ? launch_bwd_t<128, true>(p, stream) : launch_bwd_t<128, false>(p, stream);
  if (d == 64) return drop ? launch_bwd_t<64, true>(p, stream) : launch_bwd_t<64, false>(p, stream);
  return -2;
}

}  // namespace fa
