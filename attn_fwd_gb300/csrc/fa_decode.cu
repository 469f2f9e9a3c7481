// fa_decode.cu -- attention of the newest query tokens against a key/value
// cache, split over the cache ("Как работает FlashAttention математически",
// section 9: FlashDecoding -- K and V are cached, Q is the newest token).
//
// The work is bound by reading K and V once from HBM.  One CTA per (batch,
// head, chunk of the cache): a producer lane streams 64-key tiles of K and V
// by TMA into a shared-memory ring; two consumer warps take 32 keys of each
// tile and keep the online softmax per query token ("FlashAttention" notes,
// "Tiling"; the aivaro.ru page, sections 3-4): running max m, row sum l and
// the output.  For 1 to 8 tokens the scores S^T = K q^T (keys x tokens) and
// the output O^T += V^T P^T (head dim x tokens) are matrix products with a
// short side; they go to warp-level m16n8k16 tensor-core MMAs with the keys
// (or head-dim rows) in M and the tokens in N = 8, which leaves CUDA cores
// only the softmax, so the kernel runs at the HBM bound for any token count.
// K and V tiles arrive with 128-byte swizzle (boxes of 64 keys x 64
// columns), so the fragment loads hit 8 different bank groups.
//
// Each chunk writes its normalised O and its LSE; a second kernel merges the
// chunks with the statistics merge of "FlashAttention" notes, "Tiling":
// M = max LSE_c, w_c = exp(LSE_c - M), O = sum w_c O_c / sum w_c,
// LSE = M + ln sum w_c.  With a single chunk the first kernel writes O and
// LSE itself.
#include "fa_common.cuh"
#include "fa_ptx.cuh"

namespace fa {

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ void dec_drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

template <int D>
struct DecLayout {
  static constexpr int KT = DEC_TILE;                      // keys per stage
  static constexpr int BOX_BYTES = KT * 128;               // 64 keys x 64 columns
  static constexpr int TILE_BYTES = KT * D * 2;            // K (or V) of one stage
  static constexpr int STAGES = 3;                         // 96 KB (d=128) / 48 KB (d=64)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = STAGES * TILE_BYTES;
  static constexpr int MS = D + 4;                         // merge row stride (floats)
  static constexpr int MERGE_OFF = 2 * STAGES * TILE_BYTES;
  static constexpr int MERGE_BYTES = (DEC_MAX_Q * MS + 2 * DEC_MAX_Q) * 4;   // O, then m, l
  static constexpr int BAR_OFF = MERGE_OFF + MERGE_BYTES;
  static constexpr int B_FULL = 0;
  static constexpr int B_EMPTY = STAGES;
  static constexpr int NBARS = 2 * STAGES;
  static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;  // + abort flag, + 1 KB alignment slack
  static constexpr int THREADS = 96;                       // warps 0-1 consume, warp 2 loads
};

// Byte offset of 16-byte chunk j (columns 8j..8j+7) of key row r in a tile
// stored as D/64 boxes of [64 rows][128 B] with 128-byte swizzle.
template <int D>
__device__ __forceinline__ uint32_t sw_chunk(int r, int j) {
  return static_cast<uint32_t>((j >> 3) * DecLayout<D>::BOX_BYTES + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(96) fa_decode_kernel(const __grid_constant__ DecParams p) {
  using L = DecLayout<D>;
  constexpr int KS = D / 16;                               // 16-column steps of the head dim
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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

  if (warp == 2) {
    // ------------------------------------------------------------ producer
    // Whole 64-key boxes: rows past the cache's end (Nk) are zero-filled;
    // rows past this batch's length are read and masked by the consumers.
    if (lane == 0) {
      uint32_t issued[L::STAGES] = {};
      bool ok = true;
      const uint64_t pol = l2_policy_evict_first();          // K and V are read once
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % L::STAGES;
        if (!mbar_wait(bar(L::B_EMPTY + s), ((t / L::STAGES) & 1) ^ 1, wc)) { ok = false; break; }
        const int k0 = k_begin + t * L::KT;
        mbar_arrive_expect_tx(bar(L::B_FULL + s), 2 * L::TILE_BYTES);
#pragma unroll
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(smem_u32(smem + L::K_OFF + s * L::TILE_BYTES + h * L::BOX_BYTES), &p.tm_k, bar(L::B_FULL + s),
                      64 * h, k0, bh, pol);
          tma_load_3d(smem_u32(smem + L::V_OFF + s * L::TILE_BYTES + h * L::BOX_BYTES), &p.tm_v, bar(L::B_FULL + s),
                      64 * h, k0, bh, pol);
        }
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
  // Warp w takes keys 32w..32w+31 of every tile.  Fragment coordinates:
  // g = lane / 4 (a row of M), tq = lane % 4 (query columns 2tq, 2tq+1).
  const int nq = p.Nq;
  const int g = static_cast<int>(lane >> 2), tq = static_cast<int>(lane & 3);
  // q^T as the B operand of S^T = K q^T, for every 16-column step kk:
  // (q[g][16kk + 2tq, +1], q[g][16kk + 8 + 2tq, +1]); zero for absent tokens
  uint32_t qb[KS][2];
  {
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(p.q + (static_cast<size_t>(bh) * nq + g) * D);
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qb[kk][0] = g < nq ? __ldg(qrow + 8 * kk + tq) : 0u;
      qb[kk][1] = g < nq ? __ldg(qrow + 8 * kk + 4 + tq) : 0u;
    }
  }
  // running max (exp2 units), this lane's part of the row sum, and O^T
  // fragments: oacc[dm] holds O^T[16dm + g (+8)][2tq, 2tq+1]
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float oacc[KS][4];
#pragma unroll
  for (int dm = 0; dm < KS; ++dm)
#pragma unroll
    for (int e = 0; e < 4; ++e) oacc[dm][e] = 0.f;
  // the last key each of this lane's two queries may see (bottom-right causal
  // alignment); query columns past nq compute on zeros and are never stored
  const int last_key0 = p.causal ? len - nq : len - 1;
  const int lim0 = last_key0 + (p.causal ? 2 * tq : 0);
  const int lim1 = last_key0 + (p.causal ? 2 * tq + 1 : 0);
  const uint32_t sk0 = smem_u32(smem + L::K_OFF), sv0 = smem_u32(smem + L::V_OFF);
  const int rw = 32 * static_cast<int>(warp);                // this warp's first row in a tile
  bool ok = true;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % L::STAGES;
    if (!(ok = mbar_wait_warp(bar(L::B_FULL + s), (t / L::STAGES) & 1, wc))) break;
    const int kb = k_begin + t * L::KT + rw;                 // this warp's first key
    const int nv = min(max(k_end - kb, 0), 32);              // its valid keys
    if (nv > 0) {
      const uint32_t kt = sk0 + s * L::TILE_BYTES, vt = sv0 + s * L::TILE_BYTES;
      if (nv < 32) {
        // rows past the batch's length hold whatever the cache holds there:
        // zero this warp's V rows past nv (P is 0 there, but 0 * NaN is not)
        uint8_t* vrow = smem + L::V_OFF + s * L::TILE_BYTES;
        for (int x = static_cast<int>(lane); x < (32 - nv) * (D / 8); x += 32) {
          const int r = rw + nv + x / (D / 8), j = x % (D / 8);
          *reinterpret_cast<uint4*>(vrow + (j >> 3) * L::BOX_BYTES + r * 128 + ((j & 7) << 4)) =
              make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S^T for the warp's two 16-key row blocks
      float sacc[2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[mt][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          // matrices: rows +0 / +8 of the block, columns 16kk / 16kk + 8
          const int r = rw + 16 * mt + static_cast<int>(lane & 7) + static_cast<int>((lane >> 3) & 1) * 8;
          const int j = 2 * kk + static_cast<int>(lane >> 4);
          uint32_t a[4];
          ldsm_x4(kt + sw_chunk<D>(r, j), a);
          mma_16816(sacc[mt], a, qb[kk][0], qb[kk][1]);
        }
      }
      // online softmax per query column: mask, max over the 32 keys (this
      // lane's 4 rows, then the 8 lanes sharing tq), exp2
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int kr = 16 * mt + 8 * hh + g;               // key row within the warp's 32
          const bool in = kr < nv;
          const int key = kb + kr;
          sacc[mt][2 * hh] = (in && key <= lim0) ? sacc[mt][2 * hh] * p.scale_log2 : -INFINITY;
          sacc[mt][2 * hh + 1] = (in && key <= lim1) ? sacc[mt][2 * hh + 1] * p.scale_log2 : -INFINITY;
          mx0 = fmaxf(mx0, sacc[mt][2 * hh]);
          mx1 = fmaxf(mx1, sacc[mt][2 * hh + 1]);
        }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      // a column with nothing visible yet keeps m = -inf, p = 0, alpha = 1
      const float al0 = mn0 == -INFINITY ? 1.f : ex2_approx(m[0] - mn0);
      const float al1 = mn1 == -INFINITY ? 1.f : ex2_approx(m[1] - mn1);
      const float mb0 = mn0 == -INFINITY ? 0.f : mn0, mb1 = mn1 == -INFINITY ? 0.f : mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          sacc[mt][2 * hh] = ex2_approx(sacc[mt][2 * hh] - mb0);          // 0 where masked
          sacc[mt][2 * hh + 1] = ex2_approx(sacc[mt][2 * hh + 1] - mb1);
          ps0 += sacc[mt][2 * hh];
          ps1 += sacc[mt][2 * hh + 1];
        }
      }
      m[0] = mn0;
      m[1] = mn1;
      l[0] = l[0] * al0 + ps0;
      l[1] = l[1] * al1 + ps1;
#pragma unroll
      for (int dm = 0; dm < KS; ++dm) {
        oacc[dm][0] *= al0;
        oacc[dm][1] *= al1;
        oacc[dm][2] *= al0;
        oacc[dm][3] *= al1;
      }
      // O^T += V^T P^T: per 16-key step mt, P^T as the B operand is the
      // transpose of the score fragments (keys x queries -> queries x keys)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint32_t b0 = movm_t(pack_bf16x2(sacc[mt][0], sacc[mt][1]));
        const uint32_t b1 = movm_t(pack_bf16x2(sacc[mt][2], sacc[mt][3]));
#pragma unroll
        for (int dm = 0; dm < KS; ++dm) {
          // matrices (transposed): keys +0 / +8 of the step, columns 16dm / 16dm + 8
          const int r = rw + 16 * mt + static_cast<int>(lane & 7) + static_cast<int>((lane >> 4) & 1) * 8;
          const int j = 2 * dm + static_cast<int>((lane >> 3) & 1);
          uint32_t a[4];
          ldsm_x4_t(vt + sw_chunk<D>(r, j), a);
          mma_16816(oacc[dm], a, b0, b1);
        }
      }
      // the generic zero stores above precede the stage's next TMA refill
      if (nv < 32) fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::B_EMPTY + s));
  }
  // ------------------------------------------ merge the two warps' states
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
  }
  float* mg = reinterpret_cast<float*>(smem + L::MERGE_OFF);   // [DEC_MAX_Q][MS] O, then m, l
  float* mm = mg + DEC_MAX_Q * L::MS;
  const int q0 = 2 * tq, q1 = 2 * tq + 1;
  if (warp == 1) {
#pragma unroll
    for (int dm = 0; dm < KS; ++dm) {
      mg[q0 * L::MS + 16 * dm + g] = oacc[dm][0];
      mg[q1 * L::MS + 16 * dm + g] = oacc[dm][1];
      mg[q0 * L::MS + 16 * dm + g + 8] = oacc[dm][2];
      mg[q1 * L::MS + 16 * dm + g + 8] = oacc[dm][3];
    }
    if (g == 0) {
      mm[q0] = m[0];
      mm[q1] = m[1];
      mm[DEC_MAX_Q + q0] = l[0];
      mm[DEC_MAX_Q + q1] = l[1];
    }
  }
  named_bar_sync(1, 64);
  if (warp != 0) return;
  if (!ok || *abort_flag) return;                          // the status word says why
  // combined and normalised O^T back into the merge buffer (each position
  // is read and written by one lane), then stored row by row
  float lse2[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const int qc = 2 * tq + c;
    const float m1 = mm[qc], l1 = mm[DEC_MAX_Q + qc];
    const float M = fmaxf(m[c], m1);
    float a0 = 0.f, a1 = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
      a0 = ex2_approx(m[c] - M);
      a1 = ex2_approx(m1 - M);
      lsum = a0 * l[c] + a1 * l1;
    }
    const float iv = lsum > 0.f ? 1.f / lsum : 0.f;
    lse2[c] = M == -INFINITY ? -INFINITY : M + __log2f(lsum);          // log2 units
    // scale factors for this warp's and the other warp's parts
    m[c] = a0 * iv;
    l[c] = a1 * iv;
  }
#pragma unroll
  for (int dm = 0; dm < KS; ++dm) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int qc = 2 * tq + (e & 1);
      float* x = mg + qc * L::MS + 16 * dm + g + 8 * (e >> 1);
      *x = oacc[dm][e] * m[e & 1] + *x * l[e & 1];
    }
  }
  __syncwarp();
  const size_t out_q = static_cast<size_t>(bh) * nq;
  if (g == 0) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int qc = 2 * tq + c;
      if (qc < nq) {
        if (p.splits == 1) {
          p.lse[out_q + qc] = lse2[c] * 0.69314718055994530942f;
        } else {
          p.lse_part[(static_cast<size_t>(bh) * p.splits + split) * nq + qc] = lse2[c];
        }
      }
    }
  }
  // rows of O: lane x covers 4 consecutive columns
  for (int x = static_cast<int>(lane); x < nq * (D / 4); x += 32) {
    const int qc = x / (D / 4), c4 = (x % (D / 4)) * 4;
    const float4 v = *reinterpret_cast<const float4*>(mg + qc * L::MS + c4);
    if (p.splits == 1) {
      uint2 w;
      w.x = pack_bf16x2(v.x, v.y);
      w.y = pack_bf16x2(v.z, v.w);
      *reinterpret_cast<uint2*>(p.o + (out_q + qc) * D + c4) = w;
    } else {
      const size_t part_row = (static_cast<size_t>(bh) * p.splits + split) * nq + qc;
      *reinterpret_cast<float4*>(p.o_part + part_row * D + c4) = v;
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

template <int D>
int launch_decode_combine(const DecParams& p, cudaStream_t stream) {
  if (p.splits > 1) {
    const long long rows = static_cast<long long>(p.BH) * p.Nq;
    fa_decode_combine_kernel<D><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return -4;
  }
  return 0;
}

template <int D>
int launch_decode_d(const DecParams& p, cudaStream_t stream) {
  using L = DecLayout<D>;
  static SmemAttrOnce attr;
  if (!attr.ensure(reinterpret_cast<const void*>(fa_decode_kernel<D>), L::SMEM_BYTES)) return -4;
  const unsigned grid = static_cast<unsigned>(p.BH) * static_cast<unsigned>(p.splits);
  fa_decode_kernel<D><<<grid, L::THREADS, L::SMEM_BYTES, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return -4;
  return launch_decode_combine<D>(p, stream);
}

int launch_decode(const DecParams& p, int d, cudaStream_t stream) {
  if (d == 128) return launch_decode_d<128>(p, stream);
  if (d == 64) return launch_decode_d<64>(p, stream);
  return -2;
}

}  // namespace fa
