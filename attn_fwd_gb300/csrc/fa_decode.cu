// fa_decode.cu -- attention of the newest query tokens against a key/value
// cache, split over the cache ("Как работает FlashAttention математически",
// section 9: FlashDecoding -- K and V are cached, Q is the newest token).
//
// The work is bound by reading K and V once from HBM, so it runs on CUDA
// cores: one CTA per (batch, head, chunk of the cache); a producer lane
// streams 64-key tiles of K and V with 1-D bulk copies (each tile is a
// contiguous run of rows) into a shared-memory ring; two consumer warps take
// 32 keys of each tile.  For S = scale * q k^T lane j owns key j: it reads
// its key row once, in 16-byte chunks taken in a lane-rotated order (so the
// 32 rows hit different banks), and forms every query's dot product against
// q kept in shared memory as fp32, two products per packed FMA.  The online
// softmax ("FlashAttention" notes, "Tiling"; the aivaro.ru page, sections
// 3-4) keeps the running max m, the row sum l and the output per query; for
// O += p V lane t owns d/32 columns, reads each V row once and updates two
// queries per packed FMA with their p broadcast by shuffle.  Each chunk writes its
// normalised O and its LSE; a second kernel merges the chunks with the
// statistics merge of "FlashAttention" notes, "Tiling":
// M = max LSE_c, w_c = exp(LSE_c - M), O = sum w_c O_c / sum w_c,
// LSE = M + ln sum w_c.  With a single chunk the first kernel writes O and
// LSE itself.
#include "fa_common.cuh"
#include "fa_ptx.cuh"

namespace fa {

template <int D, int NQ>
struct DecLayout {
  static constexpr int KT = DEC_TILE;                      // keys per stage
  static constexpr int ROW = D * 2;                        // bytes per key row
  static constexpr int TILE_BYTES = KT * ROW;              // K (or V) of one stage
  // 3 stages: 96 KB (d=128) / 48 KB (d=64) of K/V, 2 / 4 CTAs per SM; with
  // several query tokens at d=128, 2 stages and 3 CTAs per SM, so more
  // consumer warps hide the per-key latency of the longer score loop
  static constexpr int STAGES = (D == 128 && NQ > 1) ? 2 : 3;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = STAGES * TILE_BYTES;
  static constexpr int MERGE_OFF = 2 * STAGES * TILE_BYTES;            // warp 1's state
  static constexpr int MERGE_BYTES = DEC_MAX_Q * (D + 2) * 4;
  static constexpr int QS_OFF = MERGE_OFF + MERGE_BYTES;               // q, fp32, pre-scaled
  static constexpr int QS_BYTES = DEC_MAX_Q * D * 4;
  static constexpr int BAR_OFF = QS_OFF + QS_BYTES;
  static constexpr int B_FULL = 0;
  static constexpr int B_EMPTY = STAGES;
  static constexpr int NBARS = 2 * STAGES;
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 128;   // + abort flag, + alignment slack
  static constexpr int THREADS = 96;                       // warps 0-1 consume, warp 2 loads
  static constexpr int E = D / 32;                         // head-dim columns per lane
};

// Sum over the 32 lanes of v[j] for each j, leaving the total of entry `lane`
// in v[0]: at each step a lane keeps the half of its entries selected by its
// lane bit and adds the partner's copy of that half (31 shuffles in all).
template <int OFF>
__device__ __forceinline__ void xpose_step(float (&v)[32], uint32_t lane) {
  const bool up = (lane & OFF) != 0;
#pragma unroll
  for (int t = 0; t < OFF; ++t) {
    const float send = up ? v[t] : v[t + OFF];
    const float keep = up ? v[t + OFF] : v[t];
    v[t] = keep + __shfl_xor_sync(0xffffffffu, send, OFF);
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// E consecutive bf16 of a row as floats (E = 2 or 4).
template <int E>
__device__ __forceinline__ void load_bf16(const uint8_t* p, float (&f)[E]) {
  if constexpr (E == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = __uint_as_float(w.x << 16);
    f[1] = __uint_as_float(w.x & 0xffff0000u);
    f[2] = __uint_as_float(w.y << 16);
    f[3] = __uint_as_float(w.y & 0xffff0000u);
  } else {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = __uint_as_float(w << 16);
    f[1] = __uint_as_float(w & 0xffff0000u);
  }
}

__device__ __forceinline__ void dec_drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

// One query token: lane t holds d/32 columns of q and of O; scores by a
// transposing butterfly reduction over the lanes.
template <int D, int NQ>
__device__ __forceinline__ void consume_one(const DecParams& p, uint8_t* smem, uint64_t* bars, const WaitCtx& wc,
                                        uint32_t warp, uint32_t lane, int bh, int len, int k_begin, int k_end,
                                        int n_tiles, float (&o)[NQ][D / 32], float (&m)[NQ], float (&l)[NQ],
                                        bool& ok) {
  using L = DecLayout<D, NQ>;
  constexpr int E = L::E;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  // q pre-scaled by scale * log2(e): scores come out in exp2 units
  float qf[NQ][E];
  const int nq = p.Nq;
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    if (i < nq) {
      load_bf16<E>(reinterpret_cast<const uint8_t*>(p.q + (static_cast<size_t>(bh) * nq + i) * D + lane * E), qf[i]);
#pragma unroll
      for (int e = 0; e < E; ++e) qf[i][e] *= p.scale_log2;
    }
  }
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[i][e] = 0.f;
  }
  // the last key query i may see (bottom-right causal alignment)
  const int last_key0 = p.causal ? len - nq : len - 1;
  ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % L::STAGES;
    if (!(ok = mbar_wait_warp(bar(L::B_FULL + s), (t / L::STAGES) & 1, wc))) break;
    const int kb = k_begin + t * L::KT + 32 * static_cast<int>(warp);   // this warp's first key
    const int nv = min(max(k_end - kb, 0), 32);                         // its valid keys
    const uint8_t* ks = smem + L::K_OFF + s * L::TILE_BYTES + (32 * warp) * L::ROW + lane * E * 2;
    const uint8_t* vs = smem + L::V_OFF + s * L::TILE_BYTES + (32 * warp) * L::ROW + lane * E * 2;
    if (nv > 0) {
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        if (i >= nq) break;
        float part[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float kf[E];
          load_bf16<E>(ks + j * L::ROW, kf);
          float acc = qf[i][0] * kf[0];
#pragma unroll
          for (int e = 1; e < E; ++e) acc = fmaf(qf[i][e], kf[e], acc);
          part[j] = acc;
        }
        xpose_step<16>(part, lane);
        xpose_step<8>(part, lane);
        xpose_step<4>(part, lane);
        xpose_step<2>(part, lane);
        xpose_step<1>(part, lane);
        const int key = kb + static_cast<int>(lane);
        const bool vis = static_cast<int>(lane) < nv && key <= last_key0 + (p.causal ? i : 0);
        const float sc = vis ? part[0] : -INFINITY;
        const float m_new = fmaxf(m[i], warp_max(sc));
        if (m_new == -INFINITY) continue;                  // nothing visible yet (warp-uniform)
        const float alpha = ex2_approx(m[i] - m_new);      // 0 when m was -inf
        const float pj = ex2_approx(sc - m_new);           // 0 for masked keys
        m[i] = m_new;
        l[i] = l[i] * alpha + pj;
#pragma unroll
        for (int e = 0; e < E; ++e) o[i][e] *= alpha;
        // O += p V over this warp's keys; rows past nv are stale and never read
        if (nv == 32) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float w = __shfl_sync(0xffffffffu, pj, j);
            float vf[E];
            load_bf16<E>(vs + j * L::ROW, vf);
#pragma unroll
            for (int e = 0; e < E; ++e) o[i][e] = fmaf(w, vf[e], o[i][e]);
          }
        } else {
          for (int j = 0; j < nv; ++j) {
            const float w = __shfl_sync(0xffffffffu, pj, j);
            float vf[E];
            load_bf16<E>(vs + j * L::ROW, vf);
#pragma unroll
            for (int e = 0; e < E; ++e) o[i][e] = fmaf(w, vf[e], o[i][e]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::B_EMPTY + s));
  }
}

// Several query tokens: lane j scores key j against every query; O columns
// per lane, two queries per packed FMA.
template <int D, int NQ>
__device__ __forceinline__ void consume_many(const DecParams& p, uint8_t* smem, uint64_t* bars, const WaitCtx& wc,
                                        uint32_t warp, uint32_t lane, int bh, int len, int k_begin, int k_end,
                                        int n_tiles, float (&o)[NQ][D / 32], float (&m)[NQ], float (&l)[NQ],
                                        bool& ok) {
  using L = DecLayout<D, NQ>;
  constexpr int E = L::E;
  auto bar = [&](int i) { return smem_u32(bars + i); };
  // q pre-scaled by scale * log2(e) (scores come out in exp2 units), fp32 in
  // shared memory: [query][d]
  const int nq = p.Nq;
  float* qs = reinterpret_cast<float*>(smem + L::QS_OFF);
  for (int x = static_cast<int>(threadIdx.x); x < nq * D; x += 64) {
    const float f = __bfloat162float(p.q[static_cast<size_t>(bh) * nq * D + x]);
    qs[x] = f * p.scale_log2;
  }
  named_bar_sync(2, 64);
  constexpr int NP = NQ > 1 ? NQ / 2 : 1;                 // query pairs
  float2 o2[NP][E];                                       // (query 2r, query 2r+1) per column
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }
#pragma unroll
  for (int r = 0; r < NP; ++r)
#pragma unroll
    for (int e = 0; e < E; ++e) o2[r][e] = make_float2(0.f, 0.f);
  // the last key query i may see (bottom-right causal alignment)
  const int last_key0 = p.causal ? len - nq : len - 1;
  constexpr int CH = D / 8;                                // 16-byte chunks per key row
  ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % L::STAGES;
    if (!(ok = mbar_wait_warp(bar(L::B_FULL + s), (t / L::STAGES) & 1, wc))) break;
    const int kb = k_begin + t * L::KT + 32 * static_cast<int>(warp);   // this warp's first key
    const int nv = min(max(k_end - kb, 0), 32);                         // its valid keys
    const uint8_t* krow = smem + L::K_OFF + s * L::TILE_BYTES + (32 * warp + lane) * L::ROW;
    const uint8_t* vs = smem + L::V_OFF + s * L::TILE_BYTES + (32 * warp) * L::ROW + lane * E * 2;
    if (nv > 0) {
      // scores: lane = key; rows past nv are stale, their scores are masked below
      float2 acc[NQ];
#pragma unroll
      for (int i = 0; i < NQ; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        const int cc = (c + static_cast<int>(lane)) & (CH - 1);
        const uint4 kw = *reinterpret_cast<const uint4*>(krow + cc * 16);
        const float2 k0 = make_float2(__uint_as_float(kw.x << 16), __uint_as_float(kw.x & 0xffff0000u));
        const float2 k1 = make_float2(__uint_as_float(kw.y << 16), __uint_as_float(kw.y & 0xffff0000u));
        const float2 k2 = make_float2(__uint_as_float(kw.z << 16), __uint_as_float(kw.z & 0xffff0000u));
        const float2 k3 = make_float2(__uint_as_float(kw.w << 16), __uint_as_float(kw.w & 0xffff0000u));
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
          if (i < nq) {
            const float4 qa = *reinterpret_cast<const float4*>(qs + i * D + cc * 8);
            const float4 qb = *reinterpret_cast<const float4*>(qs + i * D + cc * 8 + 4);
            acc[i] = ffma2(make_float2(qa.x, qa.y), k0, acc[i]);
            acc[i] = ffma2(make_float2(qa.z, qa.w), k1, acc[i]);
            acc[i] = ffma2(make_float2(qb.x, qb.y), k2, acc[i]);
            acc[i] = ffma2(make_float2(qb.z, qb.w), k3, acc[i]);
          }
        }
      }
      // online softmax per query; pj = this lane's key weight
      const int key = kb + static_cast<int>(lane);
      float pj[NQ], alpha[NQ];
#pragma unroll
      for (int i = 0; i < NQ; ++i) {
        pj[i] = 0.f;
        alpha[i] = 1.f;
        if (i < nq) {
          const bool vis = static_cast<int>(lane) < nv && key <= last_key0 + (p.causal ? i : 0);
          const float sc = vis ? acc[i].x + acc[i].y : -INFINITY;
          const float m_new = fmaxf(m[i], warp_max(sc));
          if (m_new != -INFINITY) {                        // warp-uniform
            alpha[i] = ex2_approx(m[i] - m_new);           // 0 when m was -inf
            pj[i] = ex2_approx(sc - m_new);                // 0 for masked keys
            m[i] = m_new;
            l[i] = l[i] * alpha[i] + pj[i];
          }
        }
      }
#pragma unroll
      for (int r = 0; r < NP; ++r) {
        const float2 a2 = make_float2(alpha[2 * r], NQ > 1 ? alpha[2 * r + 1] : 1.f);
#pragma unroll
        for (int e = 0; e < E; ++e) o2[r][e] = fmul2(o2[r][e], a2);
      }
      // O += p V over this warp's keys; rows past nv are stale and never read
      auto pv_row = [&](int j) {
        float vf[E];
        load_bf16<E>(vs + j * L::ROW, vf);
#pragma unroll
        for (int r = 0; r < NP; ++r) {
          const float wa = __shfl_sync(0xffffffffu, pj[2 * r], j);
          const float wb = NQ > 1 ? __shfl_sync(0xffffffffu, pj[2 * r + 1], j) : 0.f;
          const float2 w2 = make_float2(wa, wb);
#pragma unroll
          for (int e = 0; e < E; ++e) o2[r][e] = ffma2(w2, make_float2(vf[e], vf[e]), o2[r][e]);
        }
      };
      if (nv == 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) pv_row(j);
      } else {
        for (int j = 0; j < nv; ++j) pv_row(j);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::B_EMPTY + s));
  }
#pragma unroll
  for (int i = 0; i < NQ; ++i)
#pragma unroll
    for (int e = 0; e < E; ++e) o[i][e] = (i & 1) ? o2[i / 2][e].y : o2[i / 2][e].x;
}

template <int D, int NQ>
__global__ void __launch_bounds__(96) fa_decode_kernel(const __grid_constant__ DecParams p) {
  using L = DecLayout<D, NQ>;
  constexpr int E = L::E;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + L::NBARS);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const int bh = blockIdx.x / p.splits;
  const int split = blockIdx.x % p.splits;
  const int b = bh / p.H;
  int len = p.Nk;                                            // valid cache rows of this batch
  if (p.seqlens) len = min(max(__ldg(p.seqlens + b), 0), p.Nk);
  const int k_begin = split * p.chunk;
  const int k_end = min(k_begin + p.chunk, len);
  const int n_tiles = k_end > k_begin ? (k_end - k_begin + L::KT - 1) / L::KT : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(L::B_FULL + s), 1);
      mbar_init(bar(L::B_EMPTY + s), 2);                   // one arrival per consumer warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{abort_flag, p.status, p.timeout_ns};
  const size_t head_rows = static_cast<size_t>(bh) * p.Nk;

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t issued[L::STAGES] = {};
      bool ok = true;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % L::STAGES;
        if (!mbar_wait(bar(L::B_EMPTY + s), ((t / L::STAGES) & 1) ^ 1, wc)) { ok = false; break; }
        const int k0 = k_begin + t * L::KT;
        const int rows = min(L::KT, k_end - k0);
        const uint32_t bytes = static_cast<uint32_t>(rows * L::ROW);    // a multiple of 128
        const size_t off = (head_rows + static_cast<size_t>(k0)) * D;
        mbar_arrive_expect_tx(bar(L::B_FULL + s), 2 * bytes);
        bulk_load(smem_u32(smem + L::K_OFF + s * L::TILE_BYTES), p.k + off, bytes, bar(L::B_FULL + s));
        bulk_load(smem_u32(smem + L::V_OFF + s * L::TILE_BYTES), p.v + off, bytes, bar(L::B_FULL + s));
        ++issued[s];
      }
      if (!ok) {
        for (int s = 0; s < L::STAGES; ++s)
          if (issued[s]) dec_drain(bar(L::B_FULL + s), (issued[s] - 1) & 1u, 100000000ull);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  // One token: the transposing-reduction form (its loop is short enough for
  // one consumer warp per SM sub-partition to keep up with HBM).  Several
  // tokens: lane-per-key scores with shared K and V reads.
  float o[NQ][E], m[NQ], l[NQ];
  bool ok = true;
  const int nq = p.Nq;
  if constexpr (NQ == 1) {
    consume_one<D, NQ>(p, smem, bars, wc, warp, lane, bh, len, k_begin, k_end, n_tiles, o, m, l, ok);
  } else {
    consume_many<D, NQ>(p, smem, bars, wc, warp, lane, bh, len, k_begin, k_end, n_tiles, o, m, l, ok);
  }
  // ------------------------------------------ merge the two warps' states
  float* mg = reinterpret_cast<float*>(smem + L::MERGE_OFF);   // [DEC_MAX_Q][D + 2]
#pragma unroll
  for (int i = 0; i < NQ; ++i) l[i] = warp_sum(l[i]);
  if (warp == 1) {
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
      if (i < nq) {
        float* r = mg + i * (D + 2);
#pragma unroll
        for (int e = 0; e < E; ++e) r[lane * E + e] = o[i][e];
        if (lane == 0) {
          r[D] = m[i];
          r[D + 1] = l[i];
        }
      }
    }
  }
  named_bar_sync(1, 64);
  if (warp != 0) return;
  const bool failed = !ok || *abort_flag;
  if (failed) return;                                      // the status word says why
  const size_t out_q = static_cast<size_t>(bh) * nq;
#pragma unroll
  for (int i = 0; i < NQ; ++i) {
    if (i >= nq) break;
    const float* r = mg + i * (D + 2);
    const float m1 = r[D], l1 = r[D + 1];
    const float M = fmaxf(m[i], m1);
    float lsum = 0.f, ov[E];
    if (M == -INFINITY) {
#pragma unroll
      for (int e = 0; e < E; ++e) ov[e] = 0.f;
    } else {
      const float a0 = ex2_approx(m[i] - M), a1 = ex2_approx(m1 - M);
      lsum = a0 * l[i] + a1 * l1;
      const float inv = 1.f / lsum;
#pragma unroll
      for (int e = 0; e < E; ++e) ov[e] = (a0 * o[i][e] + a1 * r[lane * E + e]) * inv;
    }
    const float lse2 = M == -INFINITY ? -INFINITY : M + __log2f(lsum);   // log2 units
    if (p.splits == 1) {
      __nv_bfloat16* dst = p.o + (out_q + i) * D + lane * E;
      if constexpr (E == 4) {
        uint2 w;
        w.x = pack_bf16x2(ov[0], ov[1]);
        w.y = pack_bf16x2(ov[2], ov[3]);
        *reinterpret_cast<uint2*>(dst) = w;
      } else {
        *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(ov[0], ov[1]);
      }
      if (lane == 0) p.lse[out_q + i] = lse2 * 0.69314718055994530942f;
    } else {
      const size_t part_row = (static_cast<size_t>(bh) * p.splits + split) * nq + i;
      float* dst = p.o_part + part_row * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) dst[e] = ov[e];
      if (lane == 0) p.lse_part[part_row] = lse2;
    }
  }
}

// One warp per (batch * head, query): merge the chunks' outputs.
template <int D>
__global__ void __launch_bounds__(128) fa_decode_combine_kernel(const __grid_constant__ DecParams p) {
  constexpr int E = D / 32;
  const uint32_t lane = lane_id();
  const long long row = static_cast<long long>(blockIdx.x) * 4 + (threadIdx.x >> 5);   // bh * Nq + i
  const long long rows = static_cast<long long>(p.BH) * p.Nq;
  if (row >= rows) return;
  const long long bh = row / p.Nq;
  const int i = static_cast<int>(row % p.Nq);
  const float* lp = p.lse_part + static_cast<size_t>(bh) * p.splits * p.Nq + i;      // stride Nq
  float M = -INFINITY;
  for (int c = lane; c < p.splits; c += 32) M = fmaxf(M, lp[static_cast<size_t>(c) * p.Nq]);
  M = warp_max(M);
  float acc[E] = {}, W = 0.f;
  if (M != -INFINITY) {
    for (int c = 0; c < p.splits; ++c) {
      const float lc = lp[static_cast<size_t>(c) * p.Nq];
      if (lc == -INFINITY) continue;                       // a chunk with no visible key
      const float w = ex2_approx(lc - M);
      W += w;
      const float* oc = p.o_part + ((static_cast<size_t>(bh) * p.splits + c) * p.Nq + i) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(w, oc[e], acc[e]);
    }
  }
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __nv_bfloat16* dst = p.o + static_cast<size_t>(row) * D + lane * E;
  if constexpr (E == 4) {
    uint2 w;
    w.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    w.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0) p.lse[row] = W > 0.f ? (M + __log2f(W)) * 0.69314718055994530942f : -INFINITY;
}

template <int D, int NQ>
int launch_decode_t(const DecParams& p, cudaStream_t stream) {
  using L = DecLayout<D, NQ>;
  static SmemAttrOnce attr;
  if (!attr.ensure(reinterpret_cast<const void*>(fa_decode_kernel<D, NQ>), L::SMEM_BYTES)) return -4;
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.splits);
  fa_decode_kernel<D, NQ><<<grid, L::THREADS, L::SMEM_BYTES, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return -4;
  if (p.splits > 1) {
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    fa_decode_combine_kernel<D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -4;
  }
  return 0;
}

template <int D>
int launch_decode_d(const DecParams& p, cudaStream_t stream) {
  if (p.Nq <= 1) return launch_decode_t<D, 1>(p, stream);
  if (p.Nq <= 2) return launch_decode_t<D, 2>(p, stream);
  if (p.Nq <= 4) return launch_decode_t<D, 4>(p, stream);
  return launch_decode_t<D, 8>(p, stream);
}

int launch_decode(const DecParams& p, int d, cudaStream_t stream) {
  if (d == 128) return launch_decode_d<128>(p, stream);
  if (d == 64) return launch_decode_d<64>(p, stream);
  return -2;
}

}  // namespace fa
