// fa_fwd.cu -- fused attention forward for sm_103a.
//
// What one CTA computes: two 128-row query tiles Q_i (i = 2t, 2t+1) of one
// (batch, head), each against every visible 128-row key/value tile K_j, V_j,
// with the online-softmax recurrence ("FlashAttention" notes, "Tiling" and
// Theorem 1; "Как работает FlashAttention математически", sections 3, 4, 6):
//   S_ij = scale * Q_i K_j^T;  m_new = max(m, rowmax S_ij);
//   P~_ij = exp(S_ij - m_new); l = exp(m - m_new) l + rowsum P~_ij;
//   O_i = exp(m - m_new) O_i + P~_ij V_j;  finally O_i /= l, LSE = m + ln l.
// O is kept un-normalised and divided once at the end (the same page's
// section 4 notes that implementations do this).  S and P live only in
// tensor memory.  The loop runs query-tile outer, key-tile inner (the V2
// order of "Transformer 入门"), so O is written once per tile.
//
// GB300 mapping (warp specialisation, 10 warps):
//   warp 9      TMA producer: Q tiles once, then K_j and V_j into a ring of
//               shared-memory slots (128-byte swizzle), L2 evict-last for K/V.
//   warp 8      MMA issuer (warp-uniform, one elected lane issues):
//               S_w = Q_w K_j^T (SS form) and
//               O_w += P_w V_j (A operand P_w read from tensor memory).
//   warps 0-3   softmax for query tile 0, warps 4-7 for tile 1: one thread
//               per query row reads its S row from tensor memory, computes the
//               masked row max, exp2, row sum, writes P (bf16) back over S,
//               and rescales its O row in tensor memory when needed.
// The MMA order S0(j) S1(j) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ... lets the
// softmax of one tile overlap the tensor-core work of the other.
//
// Rescaling is lazy: the reference max m only moves when the tile max
// exceeds it by more than 2^8 in exp2 units.  exp(S - m) then stays <= 256,
// and because O and l always share the same m the result is unchanged
// (every term carries the same factor exp(-m)).
//
// Tensor memory (512 columns x 128 lanes): S0 [0,128) S1 [128,256)
// O0 [256,256+d) O1 [256+d,256+2d); P_w (bf16 pairs) overwrites the first 64
// columns of S_w.  tcgen05 MMAs issued by one thread execute in order, so the
// next S_w(j+1) never overwrites P_w(j) before O_w += P_w(j) V_j has read it.
#include "fa_common.cuh"
#include "fa_dropout.cuh"
#include "fa_ptx.cuh"

namespace fa {

template <int D, bool SPARSE, bool DROP = false>
struct FwdLayout {
  static constexpr int NCH = D / 64;                      // 64-column (128-byte) chunks
  static constexpr int CHUNK_BYTES = TILE * 128;          // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = NCH * CHUNK_BYTES;    // one 128 x D bf16 tile
  // K/V ring slots.  A block-sparse round can need two K and two V tiles,
  // so it gets a fifth slot at d=128 to keep one load in flight ahead.
  static constexpr int STAGES = (D == 128) ? (SPARSE ? 5 : 4) : 6;
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = RING_OFF + STAGES * TILE_BYTES;
  // barrier indices
  static constexpr int B_Q = 0;                  // 2
  static constexpr int B_FULL = 2;               // STAGES
  static constexpr int B_EMPTY = 2 + STAGES;     // STAGES
  static constexpr int B_S = 2 + 2 * STAGES;     // 2
  static constexpr int B_P = B_S + 2;            // 2: all of P_w in tensor memory
  static constexpr int B_PH = B_P + 2;           // 2: its first half (keys 0-63)
  static constexpr int B_O = B_PH + 2;           // 2
  static constexpr int B_DONE = B_O + 2;         // 1
  static constexpr int B_QFREE = B_DONE + 1;     // 1: an item's S products done, Q may be reloaded
  static constexpr int NBARS = B_QFREE + 1;
  // block-sparse: one bit per key tile for each of the two query tiles, and
  // the two counts
  static constexpr int BITS_OFF = BAR_OFF + NBARS * 8 + 16;
  static constexpr int BITS_WORDS = MAX_SPARSE_TILES / 32;
  static constexpr int BITS_BYTES = SPARSE ? 2 * BITS_WORDS * 4 + 16 : 0;
  // block-sparse: one bit per round, set where both query tiles take the
  // same key tile (written and read by the MMA warp only)
  static constexpr int SHR_OFF = BITS_OFF + BITS_BYTES;
  static constexpr int SHR_BYTES = SPARSE ? BITS_WORDS * 4 : 0;
  // Dense and causal masks: the epilogue stages each softmax warp's 32 rows
  // of O, one 64-column chunk (4 KB, 128-byte swizzle) at a time, for a TMA
  // store.  Block masks keep per-thread stores (their 5-slot ring leaves no
  // room), and so does dropout (measured slower: its softmax spills, and the
  // staging tiles take shared memory from the L1 that holds the spills).
  static constexpr bool TMA_EPI = !SPARSE && !DROP;
  static constexpr int STG_OFF = (SHR_OFF + SHR_BYTES + 1023) / 1024 * 1024;
  static constexpr int STG_BYTES = TMA_EPI ? 8 * 4096 : 0;
  static constexpr int SMEM_BYTES = STG_OFF + STG_BYTES + 1024;      // + 1 KB alignment slack
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128;
  static constexpr uint32_t O_COL0 = 256, O_COL1 = 256 + D;
  static constexpr int THREADS = 320;
};

// Groups of MMAs into one accumulator under a single elect.sync: the k-steps
// of one product.  The first accumulates onto D when `acc_first` is nonzero,
// the rest always do.  Same operands as mma_ss_elect / mma_ts_elect.
__device__ __forceinline__ void mma_ss_x8_elect(uint32_t d_tmem, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                                uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %18, 0;\n\t"
      "setp.eq.b32 t, %18, %18;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, t;\n\t}" ::"r"(d_tmem),
      "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
      "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]),
      "r"(idesc), "r"(acc_first)
      : "memory");
}
__device__ __forceinline__ void mma_ts_x4_elect(uint32_t d_tmem, const uint32_t (&a)[4], const uint64_t (&b)[4],
                                                uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred e, p, t;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %10, 0;\n\t"
      "setp.eq.b32 t, %10, %10;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %9, p;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %9, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %9, t;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %9, t;\n\t}" ::"r"(d_tmem),
      "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
      "r"(idesc), "r"(acc_first)
      : "memory");
}

// TMA stores of shared memory to a tensor (bulk-group completion): the
// epilogue's O.  x (c0) is 0 or 64 here, a multiple of 8 bf16 elements.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the staged source has been read (the buffer may be rewritten)
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every store of the thread is complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Reference-max threshold for lazy rescaling, in exp2 units (factor 256).
constexpr float RESCALE_THRESHOLD = 8.0f;

// Block-sparse masks: which key tiles a query tile visits, as one bit per key
// tile, copied once per CTA from the mask row into shared memory by one warp
// (a ballot per 32 tiles); with the causal flag, tiles above the diagonal are
// dropped too.  Roles walk the set bits in increasing order.
__device__ __forceinline__ void build_sparse_bits(const FwdParams& p, int qt, uint32_t* bits, int* count,
                                                  uint32_t lane) {
  int n = 0;
  const int nw = (p.n_qt + 31) / 32;
  for (int wd = 0; wd < nw; ++wd) {
    const int kt = wd * 32 + static_cast<int>(lane);
    const size_t at = static_cast<size_t>(qt) * p.n_qt + kt;
    const bool v = qt < p.n_qt && kt < p.n_qt && (!(p.mask_kind & MASK_CAUSAL) || kt <= qt) &&
                   dcheck(at < static_cast<size_t>(p.n_qt) * p.n_qt, p.status) && __ldg(p.block_mask + at) != 0;
    const uint32_t m = __ballot_sync(0xffffffffu, v);
    if (lane == 0) bits[wd] = m;
    n += __popc(m);
  }
  if (lane == 0) *count = n;
}

// The first visible key tile at or after `from`, or -1.
__device__ __forceinline__ int next_visible(const uint32_t* bits, int from, int n_kt) {
  if (from >= n_kt) return -1;
  int wd = from >> 5;
  uint32_t m = bits[wd] & (0xffffffffu << (from & 31));
  const int nw = (n_kt + 31) >> 5;
  while (m == 0) {
    if (++wd >= nw) return -1;
    m = bits[wd];
  }
  return wd * 32 + __ffs(m) - 1;
}

// Key tiles of a CTA's two query tiles by class: mode 0 those only tile 0
// visits (x and not y), mode 1 only tile 1 (y and not x), mode 2 both; the
// first one at or after `from`, or -1.
__device__ __forceinline__ int next_in_class(const uint32_t* x, const uint32_t* y, int mode, int from, int n_kt) {
  if (from >= n_kt) return -1;
  auto word = [&](int wd) {
    const uint32_t a = x[wd], b = y[wd];
    return mode == 0 ? (a & ~b) : (mode == 1 ? (b & ~a) : (a & b));
  };
  int wd = from >> 5;
  uint32_t m = word(wd) & (0xffffffffu << (from & 31));
  const int nw = (n_kt + 31) >> 5;
  while (m == 0) {
    if (++wd >= nw) return -1;
    m = word(wd);
  }
  return wd * 32 + __ffs(m) - 1;
}

// Round schedule of a block-sparse CTA.  When the two query tiles share at
// least as many key tiles as either visits alone (sliding windows: all but
// one), the rounds take first the tiles only one query tile visits, tile 0's
// r-th paired with tile 1's r-th (rounds 0 .. split-1), then the shared tiles
// in increasing order, where one K and one V load serve both.  Otherwise
// (scattered masks, where reordering only loses L2 locality) round r pairs
// the r-th visible tile of each, in increasing order.  Every role walks the
// same schedule.
struct SparsePlan {
  int na, nb, nc;        // tiles only tile 0 / only tile 1 / both visit
  bool shared_first;
};

__device__ __forceinline__ SparsePlan sparse_plan(const uint32_t* x, const uint32_t* y, int n_kt) {
  SparsePlan pl{0, 0, 0, false};
  for (int wd = 0; wd < (n_kt + 31) / 32; ++wd) {
    pl.na += __popc(x[wd] & ~y[wd]);
    pl.nb += __popc(y[wd] & ~x[wd]);
    pl.nc += __popc(x[wd] & y[wd]);
  }
  pl.shared_first = pl.nc >= (pl.na > pl.nb ? pl.na : pl.nb);
  return pl;
}

struct SparseRounds {
  const uint32_t* x;
  const uint32_t* y;
  int n_kt, split, ca, cb, cc;
  bool shared_first;
  __device__ __forceinline__ SparseRounds(const uint32_t* x_, const uint32_t* y_, int n) : x(x_), y(y_), n_kt(n) {
    const SparsePlan pl = sparse_plan(x, y, n);
    shared_first = pl.shared_first;
    split = pl.na > pl.nb ? pl.na : pl.nb;
    ca = cb = cc = 0;
  }
  // the key tiles (a for query tile 0, b for tile 1; -1 for none) of round r,
  // called once per round in increasing r
  __device__ __forceinline__ void next(int r, int& a, int& b) {
    if (!shared_first) {
      a = next_visible(x, ca, n_kt);
      b = next_visible(y, cb, n_kt);
      if (a >= 0) ca = a + 1;
      if (b >= 0) cb = b + 1;
    } else if (r < split) {
      a = next_in_class(x, y, 0, ca, n_kt);
      b = next_in_class(x, y, 1, cb, n_kt);
      if (a >= 0) ca = a + 1;
      if (b >= 0) cb = b + 1;
    } else {
      a = b = next_in_class(x, y, 2, cc, n_kt);
      if (a >= 0) cc = a + 1;
    }
  }
};

// Query tile w's key tiles in the order of SparseRounds (for dropout, which
// needs each round's tile index): class w, then class 2 when shared-first;
// mode 3 (all of tile w's tiles, increasing) otherwise.  x, y: the bits of
// query tiles 0 and 1.
struct SparseTileSeq {
  int mode, cur;
  __device__ __forceinline__ int next(const uint32_t* x, const uint32_t* y, int w, int n_kt) {
    if (mode == 3) {
      const int kt = next_visible(w ? y : x, cur, n_kt);
      cur = kt + 1;
      return kt;
    }
    for (;;) {
      const int kt = next_in_class(x, y, mode, cur, n_kt);
      if (kt >= 0 || mode == 2) {
        cur = kt + 1;
        return kt;
      }
      mode = 2;
      cur = 0;
    }
  }
};

// The last visible key tile, or -1.
__device__ __forceinline__ int last_visible(const uint32_t* bits, int n_kt) {
  for (int wd = (n_kt + 31) / 32 - 1; wd >= 0; --wd)
    if (bits[wd]) return wd * 32 + 31 - __clz(bits[wd]);
  return -1;
}

// No mask or causal: the two query tiles of a CTA share one key-tile
// sequence 0..kt_end-1 (causal: a tile skips the tiles above its diagonal).
__device__ __forceinline__ bool dense_visible(const FwdParams& p, int qt, int kt) {
  if (qt >= p.n_qt) return false;
  return p.mask_kind != MASK_CAUSAL || kt <= qt;
}

// Banded item order (dense and causal masks whose heads' K and V outgrow
// L2).  The items -- pairs of query tiles of one (batch, head) -- are cut
// into bands of `band_heads` heads, so that the items of one band run
// together and its heads' K and V stay in L2 while they do.  Within a band
// the positions go pair-major (decreasing length when causal), heads
// fastest.  CTA c of G takes band positions c, 2G-1-c, 2G+c, 4G-1-c, ...
// (a zig-zag: long and short causal pairs even out), band after band;
// successive bands mirror the CTA index and every second band rotates it, so
// that a CTA drawing the heavier end of one band's partial last round draws
// the lighter end of the next.  Item k of CTA c, encoded as
// j = bh + BH * position, or -1 when c has fewer items.
__device__ __forceinline__ int banded_item(const FwdParams& p, int c, int k) {
  const int G = static_cast<int>(gridDim.x);
  const int bhd = p.band_heads;
  const int nb = (p.BH + bhd - 1) / bhd;
  const int half = nb >= 2 ? nb / 2 : 1;
  for (int b = 0; b < nb; ++b) {
    const int heads = min(bhd, p.BH - b * bhd);
    const int m = heads * p.n_pairs;
    const int x = (c + (b >> 1) * (G / half)) % G;
    const int cc = (b & 1) ? G - 1 - x : x;
    // rounds 0 .. m / G - 1 give the CTA one position each; the partial
    // round m / G gives one when the CTA's position falls inside the band
    const int full = m / G;
    const int jp = full * G + ((full & 1) ? G - 1 - cc : cc);
    const int count = full + (jp < m ? 1 : 0);
    if (k < count) {
      const int jj = k * G + ((k & 1) ? G - 1 - cc : cc);
      return b * bhd + jj % heads + p.BH * (jj / heads);
    }
    k -= count;
  }
  return -1;
}

// Bounded wait used only while tearing down after a failure: ignores the
// abort flag, gives up after `ns`.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

template <int D, bool SPARSE, bool DROP, bool BANDED>
__global__ void __launch_bounds__(320, 1) fa_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = FwdLayout<D, SPARSE, DROP>;
  // P V of a tile issued in two halves (the first once half of P is stored)
  // where the softmax outweighs the products: with dropout, and at d = 64
  // without a block mask
  constexpr bool SPLIT_PV = DROP || (D == 64 && !SPARSE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  // Work items: the query-tile pairs j = 0 .. n_items - 1 of all (batch,
  // head)s, head fastest, pairs in decreasing length when causal.  The grid
  // is persistent for dense and causal masks (at most one CTA per SM): CTA c
  // takes items c, 2G - 1 - c, 2G + c, ... (G CTAs), so the long and short
  // causal pairs even out; one item per CTA with a block mask.  BANDED: the
  // order of banded_item (the heads cut into bands that fit L2).
  const int n_items = p.n_pairs * p.BH;
  auto item_index = [&](int k) {
    if constexpr (BANDED) return banded_item(p, static_cast<int>(blockIdx.x), k);
    const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    const int j = k * G + ((k & 1) ? G - 1 - c : c);
    return (SPARSE && k > 0) || j >= n_items ? -1 : j;
  };
  uint32_t* bits = reinterpret_cast<uint32_t*>(smem + L::BITS_OFF);   // [2][BITS_WORDS], then 2 counts
  int* bit_counts = reinterpret_cast<int*>(bits + 2 * L::BITS_WORDS);
  // item j: (batch, head) bh, query tiles qt0 and qt1 = qt0 + 1, the key-tile
  // range of the dense schedule, visible key tiles per query tile (a block
  // mask's bits describe this CTA's single item)
  struct Item {
    int bh, qt0, qt1, kt_end, nv0, nv1;
  };
  auto item_info = [&](int j) {
    Item it;
    it.bh = j % p.BH;
    int pair = j / p.BH;
    if (p.mask_kind & MASK_CAUSAL) pair = p.n_pairs - 1 - pair;  // longest rows first
    it.qt0 = 2 * pair;
    it.qt1 = 2 * pair + 1;
    it.kt_end = (p.mask_kind == MASK_CAUSAL) ? min(it.qt1, p.n_qt - 1) + 1 : p.n_qt;
    if constexpr (SPARSE) {
      it.nv0 = bit_counts[0];
      it.nv1 = bit_counts[1];
    } else {
      it.nv0 = it.qt0 < p.n_qt ? (p.mask_kind == MASK_CAUSAL ? it.qt0 + 1 : p.n_qt) : 0;
      it.nv1 = it.qt1 < p.n_qt ? (p.mask_kind == MASK_CAUSAL ? it.qt1 + 1 : p.n_qt) : 0;
    }
    return it;
  };
  if constexpr (SPARSE) {
    const int pair0 = (p.mask_kind & MASK_CAUSAL) ? p.n_pairs - 1 - static_cast<int>(blockIdx.x) / p.BH
                                                  : static_cast<int>(blockIdx.x) / p.BH;
    if (warp < 2) build_sparse_bits(p, 2 * pair0 + static_cast<int>(warp), bits + warp * L::BITS_WORDS,
                                    bit_counts + warp, lane);
  }

  // Q of the CTA's first item is requested by the producer warp before the
  // rest of the set-up, so its copies land while the barriers, tensor memory
  // and mask bits are prepared (it initialises the two Q barriers itself).
  if (warp == 9 && lane == 0) {
    mbar_init(bar(L::B_Q + 0), 1);
    mbar_init(bar(L::B_Q + 1), 1);
    fence_mbar_init();
    const int j0 = item_index(0);
    if (j0 >= 0) {
      prefetch_tmap(&p.tm_q);
      const uint64_t pol_q = l2_policy_evict_first();
      const int bh0 = j0 % p.BH;
      int pair = j0 / p.BH;
      if (p.mask_kind & MASK_CAUSAL) pair = p.n_pairs - 1 - pair;   // as item_info
      for (int w = 0; w < 2; ++w) {
        const int qt = 2 * pair + w;
        if (qt >= p.n_qt) {
          mbar_arrive(bar(L::B_Q + w));
          continue;
        }
        mbar_arrive_expect_tx(bar(L::B_Q + w), L::TILE_BYTES);
        for (int c = 0; c < L::NCH; ++c)
          tma_load_3d(sbase + L::Q_OFF + w * L::TILE_BYTES + c * L::CHUNK_BYTES, &p.tm_q, bar(L::B_Q + w), c * 64,
                      qt * TILE, bh0, pol_q);
      }
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(bar(L::B_FULL + s), 1);
      mbar_init(bar(L::B_EMPTY + s), 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(bar(L::B_S + w), 1);
      mbar_init(bar(L::B_P + w), 4);      // the four warps of softmax group w
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
  const uint32_t* bits0 = bits;
  const uint32_t* bits1 = bits + L::BITS_WORDS;
  // Block-sparse: round r pairs key tile a_r of query tile 0 with b_r of tile
  // 1 (-1 when a tile has none), in the order of SparseRounds.  The producer
  // loads, per round, K(a) K(b) V(a) V(b) into consecutive ring slots, once
  // when a_r == b_r; the MMA issuer walks the same sequence.

  if (warp == 9) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      prefetch_tmap(&p.tm_k);
      prefetch_tmap(&p.tm_v);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      int slot = 0;
      uint32_t phase = 0;
      uint32_t issued[L::STAGES];
      for (int s = 0; s < L::STAGES; ++s) issued[s] = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
      const int j = item_index(k);
      if (j < 0) break;
      const Item it = item_info(j);
      const int bh = it.bh, qt0 = it.qt0, qt1 = it.qt1, kt_end = it.kt_end;
      const int rounds = it.nv0 > it.nv1 ? it.nv0 : it.nv1;
      // the Q buffers are free once the previous item's S products are done
      // (the first item's Q was requested before the set-up)
      if (k > 0 && !(ok = mbar_wait(bar(L::B_QFREE), (k - 1) & 1, wc))) break;
      for (int w = 0; w < 2 && k > 0; ++w) {
        const int qt = qt0 + w;
        if (qt >= p.n_qt) {              // no such tile: complete the phase empty
          mbar_arrive(bar(L::B_Q + w));
          continue;
        }
        mbar_arrive_expect_tx(bar(L::B_Q + w), L::TILE_BYTES);
        for (int c = 0; c < L::NCH; ++c)
          tma_load_3d(sbase + L::Q_OFF + w * L::TILE_BYTES + c * L::CHUNK_BYTES, &p.tm_q,
                      bar(L::B_Q + w), c * 64, qt * TILE, bh, pol_q);
      }
      if constexpr (!SPARSE) {
      for (int kt = 0; kt < kt_end && ok; ++kt) {
        if (!(dense_visible(p, qt0, kt) || dense_visible(p, qt1, kt))) continue;
        for (int which = 0; which < 2; ++which) {  // K_j, then V_j
          if (!mbar_wait(bar(L::B_EMPTY + slot), phase ^ 1u, wc)) { ok = false; break; }
          const uint32_t fb = bar(L::B_FULL + slot);
          mbar_arrive_expect_tx(fb, L::TILE_BYTES);
          const CUtensorMap* m = which ? &p.tm_v : &p.tm_k;
          for (int c = 0; c < L::NCH; ++c)
            tma_load_3d(sbase + L::RING_OFF + slot * L::TILE_BYTES + c * L::CHUNK_BYTES, m, fb,
                        c * 64, kt * TILE, bh, pol_kv);
          ++issued[slot];
          if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }
        }
      }
      } else {
      auto load = [&](const CUtensorMap* m, int kt) {
        if (!mbar_wait(bar(L::B_EMPTY + slot), phase ^ 1u, wc)) return false;
        const uint32_t fb = bar(L::B_FULL + slot);
        mbar_arrive_expect_tx(fb, L::TILE_BYTES);
        for (int c = 0; c < L::NCH; ++c)
          tma_load_3d(sbase + L::RING_OFF + slot * L::TILE_BYTES + c * L::CHUNK_BYTES, m, fb, c * 64, kt * TILE,
                      bh, pol_kv);
        ++issued[slot];
        if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }
        return true;
      };
      // Loads go in the order the MMAs consume them, so a FIFO ring of
      // STAGES slots keeps STAGES - 1 tiles in flight ahead: per round r,
      // V(a_{r-1}), K(a_r), V(b_{r-1}), K(b_r) -- a tile both query tiles
      // use is loaded once -- and after the last round the last V tiles.
      SparseRounds sched(bits0, bits1, p.n_qt);
      int pa = -1, pb = -1;                 // previous round's key tiles
      for (int r = 0; r <= rounds && ok; ++r) {
        int a = -1, b = -1;
        if (r < rounds) sched.next(r, a, b);
        if (pa >= 0) ok = load(&p.tm_v, pa);
        if (ok && a >= 0) ok = load(&p.tm_k, a);
        if (ok && pb >= 0 && pb != pa) ok = load(&p.tm_v, pb);
        if (ok && b >= 0 && b != a) ok = load(&p.tm_k, b);
        pa = a;
        pb = b;
      }
      }
      if constexpr (SPARSE) break;       // one item per CTA
      }
      if (!ok) {  // let copies already in flight land before the CTA exits
        for (int s = 0; s < L::STAGES; ++s)
          if (issued[s]) mbar_drain(bar(L::B_FULL + s), (issued[s] - 1) & 1u, 100000000ull);
      }
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this schedule (warp-uniform); one elected lane
    // issues each tcgen05 instruction.  Descriptors are a base plus a
    // compile-time offset (start-address field, in 16-byte units).
    constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
    constexpr uint32_t IDESC_O = idesc_bf16(128, D, false, true);
    bool ok = true;
    const uint64_t dq0 = sdesc_sw128(sbase + L::Q_OFF, 16, 1024);                 // Q tile 0, K-major
    const uint64_t dq1 = sdesc_sw128(sbase + L::Q_OFF + L::TILE_BYTES, 16, 1024);  // Q tile 1
    const uint64_t dk_ring = sdesc_sw128(sbase + L::RING_OFF, 16, 1024);           // ring slot 0 as K (K-major)
    const uint64_t dv_ring = sdesc_sw128(sbase + L::RING_OFF, L::CHUNK_BYTES, 1024);  // ring slot 0 as V (MN-major)
    constexpr uint32_t SLOT16 = L::TILE_BYTES >> 4;

    // S_w = Q_w K^T: D/16 k-steps of 16 (32 bytes inside a 128-byte swizzle
    // row; a new 16 KB chunk every 64 columns).
    auto issue_s = [&](uint64_t dq, uint32_t scol, int kslot) {
      const uint64_t dk = dk_ring + static_cast<uint64_t>(kslot) * SLOT16;
      if constexpr (D == 128 && SPARSE) {   // the eight k-steps under one elect (measured:
                                            // faster with block masks, slower without)
        uint64_t da[8], db[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = ((k >> 2) * L::CHUNK_BYTES + (k & 3) * 32) >> 4;
          da[k] = dq + off;
          db[k] = dk + off;
        }
        mma_ss_x8_elect(tmem + scol, da, db, IDESC_S, 0u);
      } else {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = ((k >> 2) * L::CHUNK_BYTES + (k & 3) * 32) >> 4;
          mma_ss_elect(tmem + scol, dq + off, dk + off, IDESC_S, k > 0 ? 1u : 0u);
        }
      }
    };
    // O_w += P_w V: 128/16 k-steps; P from tensor memory (8 columns of bf16
    // pairs per step), V MN-major (16 key rows of 128 bytes per step; the
    // second 64-column half of d sits 16 KB further).
    auto issue_pv_half = [&](uint32_t ocol, uint32_t scol, int vslot, bool started, int k0) {
      const uint64_t dv = dv_ring + static_cast<uint64_t>(vslot) * SLOT16;
      if constexpr (SPARSE) {          // four k-steps under one elect (as for S)
        uint32_t ta[4];
        uint64_t db[4];
#pragma unroll
        for (int kk = 0; kk < TILE / 32; ++kk) {
          const int k = k0 + kk;
          ta[kk] = tmem + scol + 8 * k;
          db[kk] = dv + ((k * 2048) >> 4);
        }
        mma_ts_x4_elect(tmem + ocol, ta, db, IDESC_O, (started || k0 > 0) ? 1u : 0u);
      } else {
#pragma unroll
        for (int kk = 0; kk < TILE / 32; ++kk) {
          const int k = k0 + kk;
          mma_ts_elect(tmem + ocol, tmem + scol + 8 * k, dv + ((k * 2048) >> 4), IDESC_O,
                       (started || k > 0) ? 1u : 0u);
        }
      }
    };
    // P_w V.  Where the softmax outweighs the products (SPLIT_PV: dropout,
    // and d = 64 without a block mask) the first half (keys 0-63) is issued
    // once the softmax warps have published that half of P and the rest once
    // all of P is in; both barriers complete once per tile, so one phase bit
    // serves both.  Otherwise all of it waits for all of P (splitting
    // measured neutral with a dense mask at d = 128 and slower with block
    // masks).
    auto pv = [&](int w, uint32_t& ph, int vslot, bool started) {
      const uint32_t ocol = w ? L::O_COL1 : L::O_COL0, scol = w ? L::S_COL1 : L::S_COL0;
      if constexpr (SPLIT_PV) {
        if (!mbar_wait_warp(bar(L::B_PH + w), ph, wc)) return false;
        tc_fence_after();
        issue_pv_half(ocol, scol, vslot, started, 0);
      }
      if (!mbar_wait_warp(bar(L::B_P + w), ph, wc)) return false;
      tc_fence_after();
      if constexpr (!SPLIT_PV) issue_pv_half(ocol, scol, vslot, started, 0);
      issue_pv_half(ocol, scol, vslot, started, TILE / 32);
      ph ^= 1u;
      return true;
    };

    if constexpr (!SPARSE) {
    int slot = 0;
    uint32_t phase = 0;
    uint32_t pph0 = 0, pph1 = 0;       // phases of the P barriers
    for (int k = 0; ok; ++k) {
    const int j = item_index(k);
    if (j < 0) break;
    const Item it = item_info(j);
    const int qt0 = it.qt0, qt1 = it.qt1, kt_end = it.kt_end, nv0 = it.nv0, nv1 = it.nv1;
    // Q of both tiles (a missing tile's phase completes empty).  The first
    // S of this item overwrites the P that the previous item's last P V
    // reads: issued after it, it runs after it.  Its first P V waits for P
    // of this item, which its softmax warps publish only after they have
    // read out the previous item's O.
    if (!(ok = mbar_wait_warp(bar(L::B_Q + 0), k & 1, wc))) break;
    if (!(ok = mbar_wait_warp(bar(L::B_Q + 1), k & 1, wc))) break;
    int done0 = 0, done1 = 0;          // PV products issued per tile
    bool has_prev = false, pf0 = false, pf1 = false;
    int pvslot = 0;
    uint32_t pvphase = 0;
    for (int kt = 0; kt < kt_end && ok; ++kt) {
      const bool f0 = dense_visible(p, qt0, kt);
      const bool f1 = dense_visible(p, qt1, kt);
      if (!(f0 || f1)) continue;
      const int kslot = slot;
      const uint32_t kphase = phase;
      if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }
      const int vslot = slot;
      const uint32_t vphase = phase;
      if (++slot == L::STAGES) { slot = 0; phase ^= 1u; }

      // tile 0: PV(prev), then S(this).  Unsplit P V: K(this) is waited for
      // after PV(prev) is issued, so that check overlaps the product instead
      // of delaying it (with the split P V, measured slower).
      if constexpr (SPLIT_PV) {
        if (!(ok = mbar_wait_warp(bar(L::B_FULL + kslot), kphase, wc))) break;
        tc_fence_after();
      }
      if (has_prev) {
        if (!(ok = mbar_wait_warp(bar(L::B_FULL + pvslot), pvphase, wc))) break;
      }
      if (has_prev && pf0) {
        if (!(ok = pv(0, pph0, pvslot, done0 > 0))) break;
        if (++done0 == nv0) mma_commit_elect(bar(L::B_O + 0));
      }
      if constexpr (!SPLIT_PV) {
        if (!(ok = mbar_wait_warp(bar(L::B_FULL + kslot), kphase, wc))) break;
        tc_fence_after();
      }
      if (f0) {
        issue_s(dq0, L::S_COL0, kslot);
        mma_commit_elect(bar(L::B_S + 0));
      }
      // tile 1
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
    } else {
    const Item it = item_info(static_cast<int>(blockIdx.x));
    const int nv0 = it.nv0, nv1 = it.nv1;
    const int rounds = nv0 > nv1 ? nv0 : nv1;
    if (nv0 > 0) ok = mbar_wait_warp(bar(L::B_Q + 0), 0, wc);
    if (ok && nv1 > 0) ok = mbar_wait_warp(bar(L::B_Q + 1), 0, wc);
    // The MMA warp needs, per round of SparseRounds' schedule, only which
    // query tiles take a key tile and whether they take the same one (then
    // one K and one V load serve both); not the tile indices themselves.
    // Shared-first: rounds 0 .. split-1 give tile 0 a tile while r < na and
    // tile 1 while r < nb, never the same; the nc rounds after split are all
    // shared.  Otherwise round r takes the r-th visible tile of each, and it
    // is the same tile exactly where a key tile t visible to both has equal
    // rank (number of visible tiles before it) in both lists: one bit per
    // round, set here with one lane per 32-tile word.
    const SparsePlan pl = sparse_plan(bits0, bits1, p.n_qt);
    const int split = pl.na > pl.nb ? pl.na : pl.nb;
    uint32_t* shr = reinterpret_cast<uint32_t*>(smem + L::SHR_OFF);
    if (!pl.shared_first) {
      const int nw = (p.n_qt + 31) / 32;
      const uint32_t x = lane < static_cast<uint32_t>(nw) ? bits0[lane] : 0u;
      const uint32_t y = lane < static_cast<uint32_t>(nw) ? bits1[lane] : 0u;
      int ex = __popc(x), ey = __popc(y);       // exclusive prefix counts over the words
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int tx = __shfl_up_sync(0xffffffffu, ex, o), ty = __shfl_up_sync(0xffffffffu, ey, o);
        if (lane >= static_cast<uint32_t>(o)) { ex += tx; ey += ty; }
      }
      ex -= __popc(x);
      ey -= __popc(y);
      if (lane < static_cast<uint32_t>(nw)) shr[lane] = 0u;
      __syncwarp();
      for (uint32_t m = x & y; m != 0u; m &= m - 1u) {
        const uint32_t below = (1u << (__ffs(m) - 1)) - 1u;
        const int rx = ex + __popc(x & below), ry = ey + __popc(y & below);
        if (rx == ry) atomicOr(shr + (rx >> 5), 1u << (rx & 31));
      }
      __syncwarp();
    }
    auto takes0 = [&](int r) { return r < rounds && (pl.shared_first ? (r < pl.na || r >= split) : r < nv0); };
    auto takes1 = [&](int r) { return r < rounds && (pl.shared_first ? (r < pl.nb || r >= split) : r < nv1); };
    auto same = [&](int r) { return pl.shared_first ? r >= split : ((shr[r >> 5] >> (r & 31)) & 1u) != 0u; };
    // Ring slots in load order (the producer's sequence: per round V(a_{r-1}),
    // K(a_r), V(b_{r-1}), K(b_r), a tile both use once): the running slot and
    // phase of the next fill.  Each slot is released right after the MMAs
    // that read it.
    int cslot = 0;
    uint32_t cphase = 0;
    auto take = [&](int& sl, uint32_t& ph) {
      sl = cslot;
      ph = cphase;
      if (++cslot == L::STAGES) { cslot = 0; cphase ^= 1u; }
    };
    uint32_t pph0 = 0, pph1 = 0;       // phases of the P barriers
    int done0 = 0, done1 = 0;          // PV products issued per tile
    bool pa = false, pb = false, pshared = false;   // the previous round's takes
    for (int r = 0; r <= rounds && ok; ++r) {
      const bool a = takes0(r), b = takes1(r);
      const bool kshared = a && b && same(r);     // tile 1 takes tile 0's K of this round
      const bool vshared = pshared;               // and took its V of the previous round
      int sva = 0, ska = 0, svb = 0, skb = 0;
      uint32_t hva = 0, hka = 0, hvb = 0, hkb = 0;
      if (pa) take(sva, hva);
      if (a) take(ska, hka);
      if (pb) {
        if (vshared) { svb = sva; hvb = hva; } else { take(svb, hvb); }
      }
      if (b) {
        if (kshared) { skb = ska; hkb = hka; } else { take(skb, hkb); }
      }
      // tile 0: PV of the previous round, then S of this round
      if (pa) {
        if (!(ok = mbar_wait_warp(bar(L::B_FULL + sva), hva, wc))) break;
        if (!(ok = pv(0, pph0, sva, done0 > 0))) break;
        if (++done0 == nv0) mma_commit_elect(bar(L::B_O + 0));
        if (!vshared) mma_commit_elect(bar(L::B_EMPTY + sva));
      }
      if (a) {
        if (!(ok = mbar_wait_warp(bar(L::B_FULL + ska), hka, wc))) break;
        tc_fence_after();
        issue_s(dq0, L::S_COL0, ska);
        mma_commit_elect(bar(L::B_S + 0));
        if (!kshared) mma_commit_elect(bar(L::B_EMPTY + ska));
      }
      // tile 1
      if (pb) {
        if (!vshared && !(ok = mbar_wait_warp(bar(L::B_FULL + svb), hvb, wc))) break;
        if (!(ok = pv(1, pph1, svb, done1 > 0))) break;
        if (++done1 == nv1) mma_commit_elect(bar(L::B_O + 1));
        mma_commit_elect(bar(L::B_EMPTY + svb));
      }
      if (b) {
        if (!kshared && !(ok = mbar_wait_warp(bar(L::B_FULL + skb), hkb, wc))) break;
        tc_fence_after();
        issue_s(dq1, L::S_COL1, skb);
        mma_commit_elect(bar(L::B_S + 1));
        mma_commit_elect(bar(L::B_EMPTY + skb));
      }
      pa = a;
      pb = b;
      pshared = kshared;
    }
    }
    // nothing may be in flight when tensor memory is released
    mma_commit_elect(bar(L::B_DONE));
    if (lane == 0) mbar_drain(bar(L::B_DONE), 0, 1000000000ull);
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
      const int row = static_cast<int>(quarter * 32 + lane);      // row in tile == TMEM lane
      const uint32_t s_addr = tmem_addr(tmem, quarter * 32, w ? L::S_COL1 : L::S_COL0);
      const uint32_t o_addr = tmem_addr(tmem, quarter * 32, w ? L::O_COL1 : L::O_COL0);
      const float sl2 = p.scale_log2;
      float m = -INFINITY;  // reference max, in exp2 units of scaled scores
      float l = 0.f;    // row sum of exp2(S - m), fp32
      bool has_o = false;
      const int n_vis = w ? nv1 : nv0;
      // Only the highest visible key tile can need a per-element mask: the
      // causal diagonal and the ragged tile holding key N-1.  Keys at or past
      // last_lim (a column in that tile) are masked to -inf.  Dense: the
      // tiles come in increasing order, so that is the last round; sparse:
      // the round whose tile is last_kt (SparseRounds' order).
      const int last_kt = SPARSE ? last_visible(w ? bits1 : bits0, p.n_qt) : n_vis - 1;
      int last_lim = p.N - last_kt * TILE;
      if ((p.mask_kind & MASK_CAUSAL) && last_kt == qt) last_lim = min(last_lim, row + 1);
      // the round (of this tile's own) that holds last_kt: the last one, or,
      // shared-first, the last of its own tiles when the other tile does not
      // visit last_kt
      int mask_rr = n_vis - 1;
      const uint32_t* other = w ? bits0 : bits1;
      SparseTileSeq seq{3, 0};
      if constexpr (SPARSE) {
        const SparsePlan pl = sparse_plan(bits0, bits1, p.n_qt);
        if (pl.shared_first) {
          seq.mode = w;
          if (last_kt >= 0 && !((other[last_kt >> 5] >> (last_kt & 31)) & 1u)) mask_rr = (w ? pl.nb : pl.na) - 1;
        }
      }
      const uint32_t bh_u = static_cast<uint32_t>(bh);
      const uint32_t hd = bh_u % static_cast<uint32_t>(p.H), bd = bh_u / static_cast<uint32_t>(p.H);
      for (int rr = 0; rr < n_vis; ++rr) {
        uint32_t dbits[4];
        if constexpr (DROP) {
          // keep bits of this row's 128 columns for this round's key tile,
          // made before S is waited for
          const int kt = SPARSE ? seq.next(bits0, bits1, w, p.n_qt) : rr;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dbits[q] = keep_bits_row(qt * TILE + row, kt * TILE + 32 * q, hd, bd, p.drop.seed_lo, p.drop.seed_hi,
                                     p.drop.add, lane & 3u);
        }
        if (!mbar_wait_warp(bar(L::B_S + w), sphase, wc)) { ok = false; break; }
        sphase ^= 1u;
        tc_fence_after();
        uint32_t r[128];
        tmem_ld_x128(s_addr, r);
        float* s = reinterpret_cast<float*>(r);
        if (rr == mask_rr && last_lim < TILE) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= last_lim) s[c] = -INFINITY;
        }
        // row max: 3-input max over four independent chains
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
        const bool need = m_tile > m + RESCALE_THRESHOLD;   // always true on the first tile
        float alpha = 1.f;
        if (need) {
          alpha = ex2_approx(m - m_tile);                  // 0 when m = -inf
          m = m_tile;
        }
        // P = exp2(S * scale * log2e - m), two columns per packed FMA; the
        // bf16 pairs go to tensor memory 32 columns at a time while the next
        // 32 are computed.  l sums the fp32 values: it gives the LSE and
        // normalises O (P V multiplies the bf16-rounded values, whose sum
        // differs from l by the rounding only, within the bf16 error of O).
        // Dropout zeroes the dropped pairs of the P V operand only: l is the
        // softmax's own sum.
        if (SPLIT_PV && has_o && __any_sync(0xffffffffu, need)) {
          // With dropout, O is rescaled before any of this tile's P is
          // published (the P V halves accumulate onto it).  O may be read
          // here: S(j) completing implies the previous P V is done.
#pragma unroll 1
          for (int c = 0; c < D; c += 16) {   // 16 columns at a time: S is live in registers here
            uint32_t ov[16];
            tmem_ld_x16(o_addr + c, ov);
#pragma unroll
            for (int i = 0; i < 16; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st_x16(o_addr + c, ov);
          }
        }
        const float2 sl2v = make_float2(sl2, sl2);
        const float2 negm = make_float2(-m, -m);
        float2 la = make_float2(0.f, 0.f), lb = la;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float2 x = ffma2(make_float2(s[32 * q + 2 * e], s[32 * q + 2 * e + 1]), sl2v, negm);
            const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            const uint32_t pku = pack_bf16x2(pv.x, pv.y);
            if (e & 1)
              lb = fadd2(lb, pv);
            else
              la = fadd2(la, pv);
            if constexpr (DROP) {
              const uint32_t f = dbits[q] >> keep_bit(2 * e);   // columns 2e, 2e+1: adjacent bits
              pk[e] = pku & (((f & 1u) ? 0x0000FFFFu : 0u) | ((f & 2u) ? 0xFFFF0000u : 0u));
            } else {
              pk[e] = pku;
            }
          }
          if (SPLIT_PV && q == 2) {
            // keys 0-63 of P are stored: publish that half (the stores of
            // chunks 0 and 1 completed while chunk 2 was computed)
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::B_PH + w));
          }
          tmem_st_x16_async(s_addr + 16 * q, pk);
        }
        l = l * alpha + ((la.x + la.y) + (lb.x + lb.y));
        if (!SPLIT_PV && has_o && __any_sync(0xffffffffu, need)) {
          // O may be read here: S(j) completing implies the previous PV is done.
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tmem_ld_x32(o_addr + c, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
            tmem_st_x32(o_addr + c, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(L::B_P + w));   // one arrival per warp
        has_o = true;
      }
      // ---------------------------------------------------------- epilogue
      if (ok) {
        // rows beyond N (ragged last query tile) are computed but not stored
        // (banded order: the item recomputed here instead of kept in
        // registers across the row loop)
        const int qt_e = BANDED ? item_info(item_index(k)).qt0 + w : qt;
        const int bh_e = BANDED ? item_index(k) % p.BH : bh;
        const bool row_ok = qt_e * TILE + row < p.N &&
                            dcheck(bh_e < p.BH && qt_e * TILE + row >= 0, p.status);
        const size_t grow = static_cast<size_t>(bh_e) * p.N + static_cast<size_t>(qt_e) * TILE + row;
        __nv_bfloat16* orow = p.o + grow * D;
        if (n_vis > 0) {
          ok = mbar_wait_warp(bar(L::B_O + w), n_out & 1, wc);
          ++n_out;
          if (ok) {
            tc_fence_after();
            const float inv_l = DROP ? p.drop.scale / l : 1.f / l;
            if constexpr (L::TMA_EPI) {
              // this warp's 32 rows, a 64-column chunk at a time: bf16 into the
              // warp's 4 KB staging tile (row = lane, 16-byte unit u of the
              // 128-byte row at u ^ (row % 8)), then one TMA store, whose
              // copies skip rows past N
              uint8_t* stg = smem + L::STG_OFF + warp * 4096;
#pragma unroll 1
              for (int h = 0; h < D / 64; ++h) {
                if (h > 0) {           // the previous chunk's store has read the tile
                  if (lane == 0) bulk_wait_read_all();
                  __syncwarp();
                }
#pragma unroll
                for (int c2 = 0; c2 < 64; c2 += 32) {
                  uint32_t ov[32];
                  tmem_ld_x32(o_addr + h * 64 + c2, ov);
                  uint4 pkd[4];
                  uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
                  for (int i = 0; i < 16; ++i)
                    pw[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const uint32_t u = static_cast<uint32_t>(c2 / 8 + e) ^ (lane & 7u);
                    *reinterpret_cast<uint4*>(stg + lane * 128 + u * 16) = pkd[e];
                  }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                  tma_store_3d(&p.tm_o, smem_u32(stg), h * 64, qt_e * TILE + static_cast<int>(quarter) * 32, bh_e);
                  bulk_commit();
                }
              }
              if (lane == 0) bulk_wait_read_all();   // the tile is free for the next item
              __syncwarp();
            } else {
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t ov[32];
              tmem_ld_x32(o_addr + c, ov);
              uint4 pkd[4];
              uint32_t* pw = reinterpret_cast<uint32_t*>(pkd);
#pragma unroll
              for (int i = 0; i < 16; ++i)
                pw[i] = pack_bf16x2(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
              if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = pkd[i];
              }
            }
            }
            if (row_ok) p.lse[grow] = (m + __log2f(l)) * 0.69314718055994530942f;
          }
        } else if (row_ok) {
          // no visible key: O = 0, LSE = -inf
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          p.lse[grow] = -INFINITY;
        }
      }
    }
    if constexpr (SPARSE) break;         // one item per CTA
    }
    if constexpr (L::TMA_EPI) {          // every O store of this warp complete
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

template <int D, bool SPARSE, bool DROP, bool BANDED = false>
static int launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  using L = FwdLayout<D, SPARSE, DROP>;
  static_assert(L::SMEM_BYTES <= 232448, "shared memory budget");
  static SmemAttrOnce attr;
  if (!attr.ensure(reinterpret_cast<const void*>(fa_fwd_kernel<D, SPARSE, DROP, BANDED>), L::SMEM_BYTES)) return -4;
  const long long items = static_cast<long long>(p.n_pairs) * p.BH;
  const long long grid = SPARSE ? items : (items < p.max_ctas ? items : p.max_ctas);
  fa_fwd_kernel<D, SPARSE, DROP, BANDED><<<static_cast<unsigned>(grid), L::THREADS, L::SMEM_BYTES, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_fwd(const FwdParams& p, int d, cudaStream_t stream) {
  const bool sparse = (p.mask_kind & MASK_BLOCK) != 0;
  const bool drop = p.drop.t != 0;
  // the banded order only where it was asked for (dense and causal masks
  // without dropout whose heads' K and V outgrow L2)
  const bool banded = !sparse && !drop && p.band_heads < p.BH;
  if (d == 128) {
    if (drop) return sparse ? launch_fwd_t<128, true, true>(p, stream) : launch_fwd_t<128, false, true>(p, stream);
    if (banded) return launch_fwd_t<128, false, false, true>(p, stream);
    return sparse ? launch_fwd_t<128, true, false>(p, stream) : launch_fwd_t<128, false, false>(p, stream);
  }
  if (d == 64) {
    if (drop) return sparse ? launch_fwd_t<64, true, true>(p, stream) : launch_fwd_t<64, false, true>(p, stream);
    if (banded) return launch_fwd_t<64, false, false, true>(p, stream);
    return sparse ? launch_fwd_t<64, true, false>(p, stream) : launch_fwd_t<64, false, false>(p, stream);
  }
  return -2;
}

}  // namespace fa
