// fa_api.cu -- the C ABI of libfa.so (declared in include/fa.h): argument
// validation, device checks, TMA tensor-map encoding, the device status word
// and the launches of the attention kernels.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/fa.h"
#include "fa_common.cuh"
#include "fa_ptx.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kVersion = 100;  // 0.1.0

// One status word per device; kernels record FA_ERR_TIMEOUT here.
__device__ int g_fa_status;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};

struct DeviceState {
  std::once_flag once;
  int arch_ok = 0;      // 1 when compute capability is 10.3
  int sms = 0;          // multiprocessors
  int* status = nullptr;
  cudaError_t err = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool log_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("FA_LOG");
    return e && e[0] == '1';
  }();
  return on;
}

// Current device, checked once per device: compute capability 10.3 and the
// device address of its status word.
int device_ready(int** status_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&] {
    int major = 0, minor = 0;
    st.err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (st.err == cudaSuccess) st.err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    st.arch_ok = (major == 10 && minor == 3) ? 1 : 0;
    if (st.err == cudaSuccess) st.err = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
    if (st.err == cudaSuccess && st.arch_ok) {
      void* a = nullptr;
      st.err = cudaGetSymbolAddress(&a, g_fa_status);
      st.status = static_cast<int*>(a);
    }
  });
  if (st.err != cudaSuccess) return FA_ERR_CUDA;
  if (!st.arch_ok) return FA_ERR_ARCH;
  *status_out = st.status;
  return FA_OK;
}

// Multiprocessors of the current device (after device_ready succeeded).
int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  return g_dev[dev].sms > 0 ? g_dev[dev].sms : 1;
}

int encoder_ready() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? FA_OK : FA_ERR_CUDA;
}

// Encoded tensor maps are a pure function of (address, sizes, box), so a
// direct-mapped table of recent ones saves the host the encoding on repeated
// calls over the same buffers (a training loop's steady state).
struct MapKey {
  const void* ptr;
  int BH, N, d, box_rows;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && BH == o.BH && N == o.N && d == o.d && box_rows == o.box_rows;
  }
};
struct MapSlot {
  MapKey key;
  CUtensorMap map;
  bool valid;
};
constexpr int kMapSlots = 256;
MapSlot g_map_slots[kMapSlots];
std::mutex g_map_mu;

int map_slot(const MapKey& k) {
  uint64_t h = reinterpret_cast<uintptr_t>(k.ptr) >> 8;
  h = h * 0x9E3779B97F4A7C15ull ^ (static_cast<uint64_t>(k.N) << 20) ^ (static_cast<uint64_t>(k.BH) << 4) ^
      static_cast<uint64_t>(k.d + k.box_rows);
  return static_cast<int>((h ^ (h >> 29)) % kMapSlots);
}

// 3-D map over a bf16 array [BH][N][d]: box {64, box_rows, 1}, 128-byte
// swizzle, zero fill outside the array.
int make_map_bf16(CUtensorMap* m, const void* ptr, int BH, int N, int d, int box_rows) {
  const MapKey key{ptr, BH, N, d, box_rows};
  const int slot = map_slot(key);
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_map_slots[slot].valid && g_map_slots[slot].key == key) {
      *m = g_map_slots[slot].map;
      return FA_OK;
    }
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_map_mu);
  g_map_slots[slot] = MapSlot{key, *m, true};
  return FA_OK;
}

// 3-D map over a byte array [BH][rows][cols]: box {128, 128, 1}, 128-byte swizzle.
int make_map_u8(CUtensorMap* m, const void* ptr, int BH, int rows, int cols) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows) * cols};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FA_OK : FA_ERR_CUDA;
}

// 128-row tiles covering N rows (the last one may be ragged).
int tiles(int N) { return (N + fa::TILE - 1) / fa::TILE; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and scalar checks shared by every compute entry point.
int check_shape(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID;
  const long long elems = static_cast<long long>(B) * H * N * d;
  if (elems >= (1ll << 31)) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

int check_scale(float scale) { return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID; }

int check_dropout(float p) { return (std::isfinite(p) && p >= 0.f && p < 1.f) ? FA_OK : FA_ERR_INVALID; }

// Byte threshold t = round(256 p) (at most 255), and the keep scale 256 / (256 - t).
fa::Dropout make_dropout(float p, unsigned long long seed) {
  fa::Dropout d;
  const double t = std::floor(256.0 * static_cast<double>(p) + 0.5);
  d.t = static_cast<uint32_t>(t > 255.0 ? 255.0 : t);
  d.add = (256u - d.t) * 0x00010001u;
  d.scale = static_cast<float>(256.0 / (256.0 - d.t));
  d.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFull);
  d.seed_hi = static_cast<uint32_t>(seed >> 32);
  return d;
}

int check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p == nullptr || !aligned16(p)) return FA_ERR_INVALID;
  return FA_OK;
}

// Backward workspace: the fp32 dQ accumulator [B*H][N][d], then -D and
// -LSE * log2(e), each [B*H][npad] with every head's row padded to a multiple
// of 128 (zeros past N), each region 256-byte aligned.
struct Workspace {
  float* dq_acc;
  float* nd;
  float* nlse;
  int npad;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int padded(int N) { return tiles(N) * fa::TILE; }

size_t workspace_bytes(int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t prows = static_cast<size_t>(B) * H * padded(N);
  return align256(rows * d * sizeof(float)) + 2 * align256(prows * sizeof(float));
}

Workspace carve(void* ws, int B, int H, int N, int d) {
  const size_t rows = static_cast<size_t>(B) * H * N;
  const size_t prows = static_cast<size_t>(B) * H * padded(N);
  char* base = static_cast<char*>(ws);
  Workspace w;
  w.npad = padded(N);
  w.dq_acc = reinterpret_cast<float*>(base);
  base += align256(rows * d * sizeof(float));
  w.nd = reinterpret_cast<float*>(base);
  base += align256(prows * sizeof(float));
  w.nlse = reinterpret_cast<float*>(base);
  return w;
}

// Heads per band of the forward's item order (dense and causal masks).  Every
// item streams its head's K and V, and while a band's items run its heads' K
// and V should stay in L2: measured on B1 H16 d128 without a mask, 16 heads'
// K and V of 34 MB (N = 4096) are read from DRAM once, of 67 MB (N = 8192)
// 2.3 times.  So all heads form one band while their K and V take at most
// 48 MB (half that counted for a causal mask, whose pairs read half of them
// on average); beyond, a band is the largest power of two of heads whose K
// and V, twice over (bands overlap at their ends), take at most 48 MB.
int fwd_band_heads(int BH, int N, int d, int mask_kind) {
  constexpr double kBudget = 48.0 * 1024 * 1024;
  const double kv = 4.0 * N * d;                        // K and V of one head, bf16
  const double eff = (mask_kind == fa::MASK_CAUSAL) ? kv / 2 : kv;
  if (BH * eff <= kBudget) return BH;
  int band = 1;
  while (band * 2 < BH && 2.0 * (band * 2) * eff <= kBudget) band *= 2;
  return band;
}

int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const uint8_t* block_mask,
             int B, int H, int N, int d, float scale, int mask_kind, float dropout_p, unsigned long long seed,
             fa_stream_t stream) {
  int rc;
  if ((rc = check_dropout(dropout_p)) != FA_OK) return rc;
  if ((rc = check_ptrs({q, k, v, o, lse})) != FA_OK) return rc;
  if ((mask_kind & fa::MASK_BLOCK) && block_mask == nullptr) return FA_ERR_INVALID;
  if ((rc = check_shape(B, H, N, d)) != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if ((mask_kind & fa::MASK_BLOCK) && tiles(N) > fa::MAX_SPARSE_TILES) return FA_ERR_UNSUPPORTED;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  if ((rc = encoder_ready()) != FA_OK) return rc;

  fa::FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int BH = B * H;
  if (make_map_bf16(&p.tm_q, q, BH, N, d, fa::TILE) != FA_OK || make_map_bf16(&p.tm_k, k, BH, N, d, fa::TILE) != FA_OK ||
      make_map_bf16(&p.tm_v, v, BH, N, d, fa::TILE) != FA_OK || make_map_bf16(&p.tm_o, o, BH, N, d, 32) != FA_OK)
    return FA_ERR_CUDA;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.block_mask = block_mask;
  p.status = status;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.N = N;
  p.BH = BH;
  p.n_qt = tiles(N);
  p.n_pairs = (p.n_qt + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = mask_kind;
  p.H = H;
  p.drop = make_dropout(dropout_p, seed);
  p.max_ctas = device_sms();
  p.band_heads = (mask_kind & fa::MASK_BLOCK) || dropout_p > 0.f ? BH : fwd_band_heads(BH, N, d, mask_kind);
  if (log_enabled())
    std::fprintf(stderr, "[fa] fwd B=%d H=%d N=%d d=%d mask=%d items=%d band=%d\n", B, H, N, d, mask_kind,
                 p.n_pairs * BH, p.band_heads);
  return fa::launch_fwd(p, d, reinterpret_cast<cudaStream_t>(stream));
}

int bwd_main_impl(const void* q, const void* k, const void* v, const void* dout, const uint8_t* block_mask,
                  void* dk, void* dv, void* workspace, int B, int H, int N, int d, float scale, int mask_kind,
                  float dropout_p, unsigned long long seed, fa_stream_t stream) {
  int rc;
  if ((rc = check_dropout(dropout_p)) != FA_OK) return rc;
  if ((rc = check_ptrs({q, k, v, dout, dk, dv, workspace})) != FA_OK) return rc;
  if (mask_kind < 0 || mask_kind > 3) return FA_ERR_INVALID;
  if ((mask_kind & fa::MASK_BLOCK) && block_mask == nullptr) return FA_ERR_INVALID;
  if ((rc = check_shape(B, H, N, d)) != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  if ((mask_kind & fa::MASK_BLOCK) && tiles(N) > fa::MAX_SPARSE_TILES) return FA_ERR_UNSUPPORTED;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  if ((rc = encoder_ready()) != FA_OK) return rc;

  const int BH = B * H;
  const int bq = (d == 128) ? 64 : 128;  // query rows per backward step
  fa::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  if (make_map_bf16(&p.tm_q, q, BH, N, d, bq) != FA_OK || make_map_bf16(&p.tm_do, dout, BH, N, d, bq) != FA_OK ||
      make_map_bf16(&p.tm_k, k, BH, N, d, fa::TILE) != FA_OK || make_map_bf16(&p.tm_v, v, BH, N, d, fa::TILE) != FA_OK)
    return FA_ERR_CUDA;
  Workspace w = carve(workspace, B, H, N, d);
  p.nlse = w.nlse;
  p.nd = w.nd;
  p.dq_acc = w.dq_acc;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.block_mask = block_mask;
  p.status = status;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.N = N;
  p.npad = w.npad;
  p.BH = BH;
  p.n_kt = tiles(N);
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.mask_kind = mask_kind;
  p.H = H;
  p.drop = make_dropout(dropout_p, seed);
  if (log_enabled())
    std::fprintf(stderr, "[fa] bwd B=%d H=%d N=%d d=%d mask=%d bq=%d\n", B, H, N, d, mask_kind, bq);
  return fa::launch_bwd_main(p, d, reinterpret_cast<cudaStream_t>(stream));
}

int preprocess_impl(const void* o, const void* dout, const float* lse, void* workspace, int B, int H, int N, int d,
                    fa_stream_t stream) {
  int rc;
  if ((rc = check_ptrs({o, dout, lse, workspace})) != FA_OK) return rc;
  if ((rc = check_shape(B, H, N, d)) != FA_OK) return rc;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  Workspace w = carve(workspace, B, H, N, d);
  return fa::launch_bwd_preprocess(static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout),
                                   lse, w.nd, w.nlse, w.dq_acc, B * H, N, w.npad, d,
                                   reinterpret_cast<cudaStream_t>(stream));
}

int convert_impl(const void* workspace, void* dq, int B, int H, int N, int d, float scale, fa_stream_t stream) {
  int rc;
  if ((rc = check_ptrs({workspace, dq})) != FA_OK) return rc;
  if ((rc = check_shape(B, H, N, d)) != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  Workspace w = carve(const_cast<void*>(workspace), B, H, N, d);
  return fa::launch_bwd_dq_convert(w.dq_acc, static_cast<__nv_bfloat16*>(dq),
                                   static_cast<long long>(B) * H * N * d, scale,
                                   reinterpret_cast<cudaStream_t>(stream));
}

int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             const uint8_t* block_mask, void* dq, void* dk, void* dv, void* workspace, int B, int H, int N, int d,
             float scale, int mask_kind, float dropout_p, unsigned long long seed, fa_stream_t stream) {
  int rc;
  if ((rc = check_dropout(dropout_p)) != FA_OK) return rc;
  // validate everything first so that nothing is enqueued on a bad call
  if ((rc = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv, workspace})) != FA_OK) return rc;
  if ((mask_kind & fa::MASK_BLOCK) && block_mask == nullptr) return FA_ERR_INVALID;
  if ((rc = check_shape(B, H, N, d)) != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  if ((mask_kind & fa::MASK_BLOCK) && tiles(N) > fa::MAX_SPARSE_TILES) return FA_ERR_UNSUPPORTED;
  if ((rc = preprocess_impl(o, dout, lse, workspace, B, H, N, d, stream)) != FA_OK) return rc;
  if ((rc = bwd_main_impl(q, k, v, dout, block_mask, dk, dv, workspace, B, H, N, d, scale, mask_kind, dropout_p,
                          seed, stream)) != FA_OK)
    return rc;
  return convert_impl(workspace, dq, B, H, N, d, scale, stream);
}

// Decoding: split the cache into chunks of a whole number of 64-key tiles.
// The split kernel keeps fa::dec_ctas_per_sm CTAs on an SM (its shared
// memory), so 152 SMs run `slots` CTAs at once; the chunk size (1..64 tiles) minimises
// waves * (tiles per chunk + 1), the +1 standing for a CTA's pipeline ramp,
// and prefers fewer chunks on ties.  The plan depends only on the sizes, so
// the workspace query and the call agree.
constexpr long long kPlanSMs = 152;

struct DecodePlan {
  int splits;
  int chunk;
};

DecodePlan decode_plan(int B, int H, int Nq, int Nk, int d) {
  const long long tiles = (static_cast<long long>(Nk) + fa::DEC_TILE - 1) / fa::DEC_TILE;
  const long long slots = kPlanSMs * fa::dec_ctas_per_sm(d);
  const long long bh = static_cast<long long>(B) * H;
  long long best_per = 1, best_cost = -1;
  for (long long per = 1; per <= 64 && per <= tiles; ++per) {
    const long long splits = (tiles + per - 1) / per;
    const long long waves = (bh * splits + slots - 1) / slots;
    const long long cost = waves * (per + 1);
    if (best_cost < 0 || cost <= best_cost) {
      best_cost = cost;
      best_per = per;
    }
  }
  const int chunk = static_cast<int>(best_per) * fa::DEC_TILE;
  return {static_cast<int>((static_cast<long long>(Nk) + chunk - 1) / chunk), chunk};
}

int check_decode_shape(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID;
  if (static_cast<long long>(B) * H * Nk * d >= (1ll << 31)) return FA_ERR_INVALID;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (Nq > fa::DEC_MAX_Q) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t decode_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  const DecodePlan plan = decode_plan(B, H, Nq, Nk, d);
  if (plan.splits == 1) return 0;
  const size_t rows = static_cast<size_t>(B) * H * plan.splits * Nq;
  return align256(rows * d * sizeof(float)) + align256(rows * sizeof(float));
}

int decode_impl(const void* q, const void* k, const void* v, void* o, float* lse, const int* seqlens, int B, int H,
                int Nq, int Nk, int d, float scale, int causal, void* workspace, fa_stream_t stream) {
  int rc;
  if ((rc = check_ptrs({q, k, v, o, lse})) != FA_OK) return rc;
  if (seqlens != nullptr && (reinterpret_cast<uintptr_t>(seqlens) & 3u) != 0) return FA_ERR_INVALID;
  if ((rc = check_decode_shape(B, H, Nq, Nk, d)) != FA_OK) return rc;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  const DecodePlan plan = decode_plan(B, H, Nq, Nk, d);
  if (plan.splits > 1 && (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return FA_ERR_INVALID;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  fa::DecParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  if (plan.splits > 1) {
    const size_t rows = static_cast<size_t>(B) * H * plan.splits * Nq;
    char* base = static_cast<char*>(workspace);
    p.o_part = reinterpret_cast<float*>(base);
    p.lse_part = reinterpret_cast<float*>(base + align256(rows * d * sizeof(float)));
  }
  p.seqlens = seqlens;
  p.status = status;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.BH = B * H;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.splits = plan.splits;
  p.chunk = plan.chunk;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  // the cache tiles go through TMA with 128-byte swizzle
  if ((rc = encoder_ready()) != FA_OK) return rc;
  if ((rc = make_map_bf16(&p.tm_k, k, B * H, Nk, d, fa::DEC_TILE)) != FA_OK) return rc;
  if ((rc = make_map_bf16(&p.tm_v, v, B * H, Nk, d, fa::DEC_TILE)) != FA_OK) return rc;
  if (log_enabled())
    std::fprintf(stderr, "[fa] decode B=%d H=%d Nq=%d Nk=%d d=%d splits=%d chunk=%d\n", B, H, Nq, Nk, d, plan.splits,
                 plan.chunk);
  return fa::launch_decode(p, d, reinterpret_cast<cudaStream_t>(stream));
}

// FP8 forward: V^T workspace [B*H][128][npad] bytes, npad = N rounded up to 16
// (the row pitch of a TMA map must be a multiple of 16 bytes).
int fp8_npad(int N) { return (N + 15) / 16 * 16; }

size_t fp8_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d != 128) return 0;
  if (static_cast<long long>(B) * H * N * d >= (1ll << 31)) return 0;
  return align256(static_cast<size_t>(B) * H * 128 * fp8_npad(N));
}

int fwd_fp8_impl(const void* q, const void* k, const void* v, void* o, float* lse, const float* qd, const float* kd,
                 const float* vd, int B, int H, int N, int d, float scale, int causal, void* workspace,
                 fa_stream_t stream) {
  int rc;
  if ((rc = check_ptrs({q, k, v, o, lse, workspace})) != FA_OK) return rc;
  for (const float* x : {qd, kd, vd})
    if (x != nullptr && (reinterpret_cast<uintptr_t>(x) & 3u) != 0) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  if ((rc = check_shape(B, H, N, d)) != FA_OK) return rc;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if ((rc = check_scale(scale)) != FA_OK) return rc;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  if ((rc = encoder_ready()) != FA_OK) return rc;
  const int BH = B * H;
  const int npad = fp8_npad(N);
  uint8_t* vt = static_cast<uint8_t*>(workspace);
  fa::Fp8Params p;
  std::memset(&p, 0, sizeof(p));
  if (make_map_u8(&p.tm_q, q, BH, N, 128) != FA_OK || make_map_u8(&p.tm_k, k, BH, N, 128) != FA_OK ||
      make_map_u8(&p.tm_vt, vt, BH, 128, npad) != FA_OK)
    return FA_ERR_CUDA;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.q_descale = qd;
  p.k_descale = kd;
  p.v_descale = vd;
  p.status = status;
  p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
  p.N = N;
  p.BH = BH;
  p.n_qt = tiles(N);
  p.n_pairs = (p.n_qt + 1) / 2;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (fa::launch_fp8_transpose_v(static_cast<const uint8_t*>(v), vt, BH, N, npad, st) != 0) return FA_ERR_LAUNCH;
  return fa::launch_fwd_fp8(p, st) == 0 ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

// --------------------------------------------------------------------------
// the timeout self-test kernel: waits on a barrier that nothing completes
// --------------------------------------------------------------------------
namespace fa {
__global__ void wait_timeout_probe_kernel(int* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t b;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&b), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtx wc{&abort_flag, status, timeout_ns};
  if (threadIdx.x < 32) (void)mbar_wait_warp(smem_u32(&b), 0, wc);
  __syncthreads();
}

int launch_wait_timeout_probe(int* status, uint64_t timeout_ns, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 64, 0, stream>>>(status, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}
}  // namespace fa

// --------------------------------------------------------------------------
// exported C ABI
// --------------------------------------------------------------------------
extern "C" {

int fa_version(void) { return kVersion; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID: return "FA_ERR_INVALID: invalid argument";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim must be 64 or 128 (block masks: N <= 131072)";
    case FA_ERR_ARCH: return "FA_ERR_ARCH: device is not compute capability 10.3";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: kernel launch failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel wait exceeded the wait timeout";
    case FA_ERR_CUDA: return "FA_ERR_CUDA: CUDA runtime error";
    case FA_ERR_SCRATCH: return "FA_ERR_SCRATCH: the backward workspace would exceed the static scratch of fa_bwd_noalloc";
    case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS: a device index check of the debug build failed (access skipped)";
    default: return "unknown fa_status";
  }
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
           float scale, int causal, fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, nullptr, B, H, N, d, scale, causal ? fa::MASK_CAUSAL : fa::MASK_NONE, 0.f, 0,
                  stream);
}

int fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, const uint8_t* block_mask,
                       int B, int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, block_mask, B, H, N, d, scale, causal ? fa::MASK_BLOCK_CAUSAL : fa::MASK_BLOCK,
                  0.f, 0, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
  if (static_cast<long long>(B) * H * N * d >= (1ll << 31)) return 0;
  return workspace_bytes(B, H, N, d);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse, void* dq,
           void* dk, void* dv, void* workspace, int B, int H, int N, int d, float scale, int causal,
           fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, nullptr, dq, dk, dv, workspace, B, H, N, d, scale,
                  causal ? fa::MASK_CAUSAL : fa::MASK_NONE, 0.f, 0, stream);
}

int fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, const uint8_t* block_mask, void* dq, void* dk, void* dv, void* workspace,
                       int B, int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, block_mask, dq, dk, dv, workspace, B, H, N, d, scale,
                  causal ? fa::MASK_BLOCK_CAUSAL : fa::MASK_BLOCK, 0.f, 0, stream);
}

int fa_bwd_preprocess(const void* o, const void* dout, const float* lse, void* workspace, int B, int H, int N, int d,
                      fa_stream_t stream) {
  return preprocess_impl(o, dout, lse, workspace, B, H, N, d, stream);
}

int fa_bwd_main(const void* q, const void* k, const void* v, const void* dout, const uint8_t* block_mask, void* dk,
                void* dv, void* workspace, int B, int H, int N, int d, float scale, int mask_kind, float dropout_p,
                unsigned long long seed, fa_stream_t stream) {
  return bwd_main_impl(q, k, v, dout, block_mask, dk, dv, workspace, B, H, N, d, scale, mask_kind, dropout_p, seed,
                       stream);
}

float fa_dropout_effective_p(float dropout_p) {
  if (check_dropout(dropout_p) != FA_OK) return -1.f;
  return static_cast<float>(make_dropout(dropout_p, 0).t) / 256.f;
}

int fa_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, const uint8_t* block_mask, int B,
                   int H, int N, int d, float scale, int causal, float dropout_p, unsigned long long seed,
                   fa_stream_t stream) {
  const int kind = (block_mask ? fa::MASK_BLOCK : 0) | (causal ? fa::MASK_CAUSAL : 0);
  return fwd_impl(q, k, v, o, lse, block_mask, B, H, N, d, scale, kind, dropout_p, seed, stream);
}

int fa_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   const uint8_t* block_mask, void* dq, void* dk, void* dv, void* workspace, int B, int H, int N, int d,
                   float scale, int causal, float dropout_p, unsigned long long seed, fa_stream_t stream) {
  const int kind = (block_mask ? fa::MASK_BLOCK : 0) | (causal ? fa::MASK_CAUSAL : 0);
  return bwd_impl(q, k, v, o, dout, lse, block_mask, dq, dk, dv, workspace, B, H, N, d, scale, kind, dropout_p, seed,
                  stream);
}

int fa_bwd_dq_convert(const void* workspace, void* dq, int B, int H, int N, int d, float scale, fa_stream_t stream) {
  return convert_impl(workspace, dq, B, H, N, d, scale, stream);
}

size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (check_decode_shape(B, H, Nq, Nk, d) != FA_OK) return 0;
  return decode_workspace_bytes(B, H, Nq, Nk, d);
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, const int* seqlens_k, int B, int H,
              int Nq, int Nk, int d, float scale, int causal, void* workspace, fa_stream_t stream) {
  return decode_impl(q, k, v, o, lse, seqlens_k, B, H, Nq, Nk, d, scale, causal, workspace, stream);
}

size_t fa_fwd_fp8_workspace_bytes(int B, int H, int N, int d) { return fp8_workspace_bytes(B, H, N, d); }

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, const float* q_descale,
               const float* k_descale, const float* v_descale, int B, int H, int N, int d, float scale, int causal,
               void* workspace, fa_stream_t stream) {
  return fwd_fp8_impl(q, k, v, o, lse, q_descale, k_descale, v_descale, B, H, N, d, scale, causal, workspace,
                      stream);
}

int fa_block_mask_window(uint8_t* mask, int N, int left, int right) {
  if (mask == nullptr || N < 1 || left < 0 || right < 0) return FA_ERR_INVALID;
  const int nb = tiles(N);
  if (nb > fa::MAX_SPARSE_TILES) return FA_ERR_UNSUPPORTED;
  for (int i = 0; i < nb; ++i)
    for (int j = 0; j < nb; ++j) mask[static_cast<size_t>(i) * nb + j] = (j - i <= right && i - j <= left) ? 1 : 0;
  return FA_OK;
}

int fa_block_mask_dilated(uint8_t* mask, int N, int window, int dilation, int causal) {
  if (mask == nullptr || N < 1 || window < 0 || dilation < 1) return FA_ERR_INVALID;
  const int nb = tiles(N);
  if (nb > fa::MAX_SPARSE_TILES) return FA_ERR_UNSUPPORTED;
  const long long reach = static_cast<long long>(window) * dilation;
  for (int i = 0; i < nb; ++i)
    for (int j = 0; j < nb; ++j) {
      const int delta = i - j;  // query block minus key block
      const bool keep = delta % dilation == 0 && (delta < 0 ? -delta : delta) <= reach && (!causal || delta >= 0);
      mask[static_cast<size_t>(i) * nb + j] = keep ? 1 : 0;
    }
  return FA_OK;
}

int fa_get_device_error(fa_stream_t stream) {
  int* status = nullptr;
  int rc = device_ready(&status);
  if (rc != FA_OK) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return v;
}

int fa_set_wait_timeout_ns(uint64_t ns) {
  if (ns == 0) return FA_ERR_INVALID;
  g_timeout_ns.store(ns, std::memory_order_relaxed);
  return FA_OK;
}

int fa_debug_wait_timeout(uint64_t timeout_ns, fa_stream_t stream) {
  if (timeout_ns == 0 || timeout_ns > 1000000000ull) return FA_ERR_INVALID;
  int* status = nullptr;
  int rc = device_ready(&status);
  if (rc != FA_OK) return rc;
  if (fa::launch_wait_timeout_probe(status, timeout_ns, reinterpret_cast<cudaStream_t>(stream)) != 0)
    return FA_ERR_LAUNCH;
  return fa_get_device_error(stream);
}

}  // extern "C"

// --------------------------------------------------------------------------
// the steps of fa_bwd, for entry points in other translation units that
// supply the workspace themselves (fa_noalloc.cu)
// --------------------------------------------------------------------------
namespace fa {

int api_check_shape(int B, int H, int N, int d) { return check_shape(B, H, N, d); }

int api_check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, const void* dq, const void* dk, const void* dv, float scale) {
  int rc;
  if ((rc = check_ptrs({q, k, v, o, dout, lse, dq, dk, dv})) != FA_OK) return rc;
  return check_scale(scale);
}

int api_device_ready() {
  int* status = nullptr;
  return device_ready(&status);
}

int api_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, void* workspace, int B, int H, int N, int d, float scale, int causal,
            cudaStream_t stream) {
  return bwd_impl(q, k, v, o, dout, lse, nullptr, dq, dk, dv, workspace, B, H, N, d, scale,
                  causal ? MASK_CAUSAL : MASK_NONE, 0.f, 0, reinterpret_cast<fa_stream_t>(stream));
}

}  // namespace fa

// --------------------------------------------------------------------------
// fa_fwd_bwd_host: forward and backward of tensors in (pinned) host memory,
// streamed through the device in chunks of heads.  Three library-owned
// streams per device overlap the copies in of chunk c + 1, the kernels of
// chunk c and the copies out of chunk c - 1 (the link carries both
// directions at once); two device buffer sets alternate between chunks.
// --------------------------------------------------------------------------
namespace {

// Heads per chunk: enough CTAs for two waves on 152 SMs (the backward runs
// one CTA per key tile, the forward one per pair of query tiles), so a
// chunk's kernels run near full speed; at most 8 chunks; the heads spread
// evenly over the chunks.  (Measured on B2 H16 N4096 d128, forward and
// backward: chunks of 8 heads beat chunks of 16, whose longer first copy in
// and last copy back are not overlapped, and chunks of 4, whose kernels run
// half empty.)
long long host_chunk_heads(int B, int H, int N, bool backward) {
  const long long bh = static_cast<long long>(B) * H;
  const long long per_head = backward ? tiles(N) : (tiles(N) + 1) / 2;
  const long long waves = (2 * kPlanSMs + per_head - 1) / per_head;
  long long g = waves > (bh + 7) / 8 ? waves : (bh + 7) / 8;
  if (g > bh) g = bh;
  const long long chunks = (bh + g - 1) / g;
  return (bh + chunks - 1) / chunks;
}

// One device buffer set for G heads: the bf16 [G][N][d] tensors (forward:
// q, k, v, O; with the backward: q, k, v, dO, O, dQ, dK, dV), LSE [G][N]
// fp32, then (backward) the backward workspace of G heads.
struct HostSet {
  char* t[8];
  float* lse;
  void* ws;
};

int host_tensors(bool backward) { return backward ? 8 : 4; }

size_t host_set_bytes(long long G, int N, int d, bool backward) {
  const size_t t = align256(static_cast<size_t>(G) * N * d * 2);
  return host_tensors(backward) * t + align256(static_cast<size_t>(G) * N * sizeof(float)) +
         (backward ? align256(workspace_bytes(1, static_cast<int>(G), N, d)) : 0);
}

HostSet host_carve(char* base, long long G, int N, int d, bool backward) {
  const size_t t = align256(static_cast<size_t>(G) * N * d * 2);
  const int nt = host_tensors(backward);
  HostSet s{};
  for (int i = 0; i < nt; ++i) s.t[i] = base + i * t;
  s.lse = reinterpret_cast<float*>(base + nt * t);
  s.ws = backward ? base + nt * t + align256(static_cast<size_t>(G) * N * sizeof(float)) : nullptr;
  return s;
}

struct HostStreams {
  std::once_flag once;
  std::mutex mu;                // one caller enqueues at a time on a device
  cudaStream_t in = nullptr, cmp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_done[2] = {}, cmp_done[2] = {}, out_done[2] = {}, join[3] = {};
  cudaError_t err = cudaSuccess;
};
HostStreams g_host[kMaxDevices];

int host_streams(HostStreams** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_CUDA;
  HostStreams& h = g_host[dev];
  std::call_once(h.once, [&] {
    cudaError_t e = cudaSuccess;
    for (cudaStream_t* s : {&h.in, &h.cmp, &h.out})
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&h.start, &h.in_done[0], &h.in_done[1], &h.cmp_done[0], &h.cmp_done[1],
                            &h.out_done[0], &h.out_done[1], &h.join[0], &h.join[1], &h.join[2]})
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    h.err = e;
  });
  if (h.err != cudaSuccess) return FA_ERR_CUDA;
  *out = &h;
  return FA_OK;
}

}  // namespace

namespace {

// One host-streamed call: the forward alone, or the forward and the
// backward, of host-resident tensors.
struct HostJob {
  bool backward;
  const void* in[4];            // q, k, v (, dO)
  void* out[4];                 // O (, dQ, dK, dV)
  float* lse;
  const uint8_t* block_mask;
  int B, H, N, d;
  float scale;
  int mask_kind;
};

size_t host_workspace_bytes(int B, int H, int N, int d, bool backward) {
  if (check_shape(B, H, N, d) != FA_OK) return 0;
  return 2 * host_set_bytes(host_chunk_heads(B, H, N, backward), N, d, backward);
}

int host_stream(const HostJob& j, void* workspace, size_t workspace_size, fa_stream_t stream) {
  int rc;
  const int n_in = j.backward ? 4 : 3, n_out = j.backward ? 4 : 1;
  for (int i = 0; i < n_in; ++i)
    if (j.in[i] == nullptr) return FA_ERR_INVALID;
  for (int i = 0; i < n_out; ++i)
    if (j.out[i] == nullptr) return FA_ERR_INVALID;
  if (j.lse == nullptr || workspace == nullptr) return FA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID;
  if ((rc = check_shape(j.B, j.H, j.N, j.d)) != FA_OK) return rc;
  if ((rc = check_scale(j.scale)) != FA_OK) return rc;
  if ((j.mask_kind & fa::MASK_BLOCK) && tiles(j.N) > fa::MAX_SPARSE_TILES) return FA_ERR_UNSUPPORTED;
  if (workspace_size < host_workspace_bytes(j.B, j.H, j.N, j.d, j.backward)) return FA_ERR_INVALID;
  int* status = nullptr;
  if ((rc = device_ready(&status)) != FA_OK) return rc;
  HostStreams* hs = nullptr;
  if ((rc = host_streams(&hs)) != FA_OK) return rc;
  std::lock_guard<std::mutex> lk(hs->mu);
  const cudaStream_t caller = reinterpret_cast<cudaStream_t>(stream);
  const int N = j.N, d = j.d;
  const long long BH = static_cast<long long>(j.B) * j.H;
  const long long G = host_chunk_heads(j.B, j.H, N, j.backward);
  const size_t set_bytes = host_set_bytes(G, N, d, j.backward);
  const size_t head_elems = static_cast<size_t>(N) * d;
  auto cu = [](cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; };
  // everything starts after the work already queued on the caller's stream
  if ((rc = cu(cudaEventRecord(hs->start, caller))) != FA_OK) return rc;
  auto enqueue = [&]() -> int {
    int rc;
    for (cudaStream_t s : {hs->in, hs->cmp, hs->out})
      if ((rc = cu(cudaStreamWaitEvent(s, hs->start, 0))) != FA_OK) return rc;
    // chunks of G heads, except a first chunk of G / 2 when there are several
    // (the pipeline fills and drains faster); the last takes the rest
    long long c = 0;
    for (long long h0 = 0; h0 < BH; ++c) {
      const int b = static_cast<int>(c & 1);
      long long gc = (c == 0 && BH > G) ? (G + 1) / 2 : G;
      if (gc > BH - h0) gc = BH - h0;
      const int g = static_cast<int>(gc);
      const HostSet s = host_carve(static_cast<char*>(workspace) + b * set_bytes, G, N, d, j.backward);
      const size_t bytes = static_cast<size_t>(g) * head_elems * 2;
      const size_t off = static_cast<size_t>(h0) * head_elems * 2;
      // copies in, once the kernels of chunk c - 2 are done with this set's
      // inputs (its outputs may still be on their way out)
      if (c >= 2 && (rc = cu(cudaStreamWaitEvent(hs->in, hs->cmp_done[b], 0))) != FA_OK) return rc;
      for (int i = 0; i < n_in; ++i)
        if ((rc = cu(cudaMemcpyAsync(s.t[i], static_cast<const char*>(j.in[i]) + off, bytes,
                                     cudaMemcpyHostToDevice, hs->in))) != FA_OK)
          return rc;
      if ((rc = cu(cudaEventRecord(hs->in_done[b], hs->in))) != FA_OK) return rc;
      // kernels, once the inputs are in and chunk c - 2's outputs have left
      // this set: the forward (O, LSE), then the backward stages
      if ((rc = cu(cudaStreamWaitEvent(hs->cmp, hs->in_done[b], 0))) != FA_OK) return rc;
      if (c >= 2 && (rc = cu(cudaStreamWaitEvent(hs->cmp, hs->out_done[b], 0))) != FA_OK) return rc;
      const fa_stream_t cs = reinterpret_cast<fa_stream_t>(hs->cmp);
      char* const o_dev = s.t[n_in];                      // O follows the inputs
      if ((rc = fwd_impl(s.t[0], s.t[1], s.t[2], o_dev, s.lse, j.block_mask, 1, g, N, d, j.scale, j.mask_kind,
                         0.f, 0, cs)) != FA_OK)
        return rc;
      if (j.backward &&
          (rc = bwd_impl(s.t[0], s.t[1], s.t[2], o_dev, s.t[3], s.lse, j.block_mask, s.t[5], s.t[6], s.t[7], s.ws,
                         1, g, N, d, j.scale, j.mask_kind, 0.f, 0, cs)) != FA_OK)
        return rc;
      if ((rc = cu(cudaEventRecord(hs->cmp_done[b], hs->cmp))) != FA_OK) return rc;
      // copies out
      if ((rc = cu(cudaStreamWaitEvent(hs->out, hs->cmp_done[b], 0))) != FA_OK) return rc;
      for (int i = 0; i < n_out; ++i)
        if ((rc = cu(cudaMemcpyAsync(static_cast<char*>(j.out[i]) + off, s.t[n_in + i], bytes,
                                     cudaMemcpyDeviceToHost, hs->out))) != FA_OK)
          return rc;
      if ((rc = cu(cudaMemcpyAsync(j.lse + h0 * N, s.lse, static_cast<size_t>(g) * N * sizeof(float),
                                   cudaMemcpyDeviceToHost, hs->out))) != FA_OK)
        return rc;
      if ((rc = cu(cudaEventRecord(hs->out_done[b], hs->out))) != FA_OK) return rc;
      h0 += gc;
    }
    return FA_OK;
  };
  rc = enqueue();
  // The caller's stream continues once everything enqueued on the three
  // streams is done -- also after a failed enqueue, so that no copy or
  // kernel of this call still runs when the caller reuses its buffers.
  const cudaStream_t own[3] = {hs->in, hs->cmp, hs->out};
  for (int i = 0; i < 3; ++i) {
    const int rj = cu(cudaEventRecord(hs->join[i], own[i]));
    const int rw = rj == FA_OK ? cu(cudaStreamWaitEvent(caller, hs->join[i], 0)) : rj;
    if (rc == FA_OK) rc = rw;
  }
  return rc;
}

}  // namespace

extern "C" size_t fa_fwd_bwd_host_workspace_bytes(int B, int H, int N, int d) {
  return host_workspace_bytes(B, H, N, d, true);
}

extern "C" int fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dout, void* o, float* lse,
                               void* dq, void* dk, void* dv, const uint8_t* block_mask, void* workspace,
                               size_t workspace_size, int B, int H, int N, int d, float scale, int causal,
                               fa_stream_t stream) {
  const HostJob j{true, {q, k, v, dout}, {o, dq, dk, dv}, lse, block_mask, B, H, N, d, scale,
                  (block_mask ? fa::MASK_BLOCK : 0) | (causal ? fa::MASK_CAUSAL : 0)};
  return host_stream(j, workspace, workspace_size, stream);
}

extern "C" size_t fa_fwd_host_workspace_bytes(int B, int H, int N, int d) {
  return host_workspace_bytes(B, H, N, d, false);
}

extern "C" int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                           const uint8_t* block_mask, void* workspace, size_t workspace_size, int B, int H, int N,
                           int d, float scale, int causal, fa_stream_t stream) {
  const HostJob j{false, {q, k, v, nullptr}, {o, nullptr, nullptr, nullptr}, lse, block_mask, B, H, N, d, scale,
                  (block_mask ? fa::MASK_BLOCK : 0) | (causal ? fa::MASK_CAUSAL : 0)};
  return host_stream(j, workspace, workspace_size, stream);
}
