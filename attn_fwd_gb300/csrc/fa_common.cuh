// fa_common.cuh -- launch parameters shared by the host launchers and the
// kernels of libfa.so.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace fa {

// Mask kinds are bit flags: causal (key j visible to query i iff j <= i) and
// block (a 128 x 128 block mask); both together keep what both keep.
enum MaskKind : int { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_BLOCK = 2, MASK_BLOCK_CAUSAL = 3 };

// Tile sizes along the sequence: B_r = B_c = 128 (one tensor-memory lane per
// query row, one 128-byte swizzle span per 64 head-dim columns).
constexpr int TILE = 128;

// Block-sparse masks: each CTA keeps the mask bits of its tiles in shared
// memory, one bit per 128-row tile, for at most this many tiles per row
// (N <= 131072).
constexpr int MAX_SPARSE_TILES = 1024;

// Dropout with regenerated masks (fa_dropout.cuh): kept iff the pair's random
// byte >= t, values scaled by 256 / (256 - t).  t = 0 switches it off.
struct Dropout {
  uint32_t t;                // byte threshold, 0..255
  uint32_t add;              // (256 - t) in both 16-bit halves
  float scale;               // 256 / (256 - t)
  uint32_t seed_lo;
  uint32_t seed_hi;
};

// Forward launch parameters.  Tensor maps describe Q, K, V as 3-D bf16
// arrays [B*H][N][d] with a {64, 128, 1} box and 128-byte swizzle.
struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;          // O, {64, 32, 1} box: the epilogue's stores (dense and causal masks)
  __nv_bfloat16* o;          // [B*H][N][d]
  float* lse;                // [B*H][N]
  const uint8_t* block_mask; // [N/128][N/128] or null
  int* status;               // device status word
  uint64_t timeout_ns;
  int N;
  int BH;
  int n_qt;                  // N / 128
  int n_pairs;               // ceil(n_qt / 2): each CTA owns two query tiles
  float scale_log2;          // scale * log2(e)
  int mask_kind;
  int H;                     // heads: (b, h) = divmod(bh, H) keys the dropout generator
  Dropout drop;
  int max_ctas;              // persistent grid size (one CTA per SM)
  int band_heads;            // dense and causal masks: heads per band of the item order (BH: one band)
};


// Backward main-kernel parameters.  Q and dO use a {64, BQ, 1} box, K and V a
// {64, 128, 1} box.
struct BwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  const float* nlse;         // [B*H][npad]: -LSE_i * log2(e), zero past N
  const float* nd;           // [B*H][npad]: -D_i = -dO_i . O_i, zero past N
  float* dq_acc;             // [B*H][N][d] fp32 accumulator
  __nv_bfloat16* dk;         // [B*H][N][d]
  __nv_bfloat16* dv;         // [B*H][N][d]
  const uint8_t* block_mask; // [N/128][N/128] or null
  int* status;
  uint64_t timeout_ns;
  int N;
  int npad;                  // N rounded up to a multiple of 128
  int BH;
  int n_kt;                  // ceil(N / 128) key tiles
  float scale;
  float scale_log2;
  int mask_kind;
  int H;
  Dropout drop;
};

// Decoding against a key/value cache: keys per shared-memory stage, and the
// largest number of query tokens per (batch, head).
constexpr int DEC_TILE = 64;
constexpr int DEC_MAX_Q = 8;

// CTAs of the decode split kernel that fit on one SM (shared memory: a
// 3-stage ring of 64-key K and V tiles, 101 KB at d = 128, 53 KB at d = 64);
// the host-side planner sizes its chunks with the same number.
__host__ __device__ constexpr int dec_ctas_per_sm(int d) { return d == 128 ? 2 : 4; }

struct DecParams {
  CUtensorMap tm_k;          // K, V as [B*H][Nk][d], box {64, 64, 1}, 128-byte swizzle
  CUtensorMap tm_v;
  const __nv_bfloat16* q;    // [B*H][Nq][d]
  __nv_bfloat16* o;          // [B*H][Nq][d]
  float* lse;                // [B*H][Nq], natural log
  float* o_part;             // [B*H][splits][Nq][d] fp32, normalised per chunk (splits > 1)
  float* lse_part;           // [B*H][splits][Nq], log2 units (splits > 1)
  const int* seqlens;        // [B] valid cache rows, or null for all Nk
  int* status;
  uint64_t timeout_ns;
  int BH;
  int H;
  int Nq;
  int Nk;
  int splits;                // chunks of the cache per (batch, head)
  int chunk;                 // keys per chunk, a multiple of DEC_TILE
  float scale_log2;
  int causal;
};

// Raises a kernel's dynamic shared-memory limit once per device (the
// attribute is per device context), instead of on every launch.
struct SmemAttrOnce {
  std::atomic<uint64_t> done{0};   // bit per device ordinal below 64
  bool ensure(const void* kernel, int bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    done.fetch_or(bit, std::memory_order_release);
    return true;
  }
};

// FP8 (e4m3) forward, d = 128: Q, K as 3-D byte arrays [B*H][N][128] with a
// {128, 128, 1} box, V transposed to [B*H][128][npad] with the same box.
struct Fp8Params {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_vt;
  __nv_bfloat16* o;          // [B*H][N][128]
  float* lse;                // [B*H][N]
  const float* q_descale;    // [B*H] or null (1)
  const float* k_descale;
  const float* v_descale;
  int* status;
  uint64_t timeout_ns;
  int N;
  int BH;
  int n_qt;
  int n_pairs;
  float scale_log2;          // scale * log2(e), before the descales
  int causal;
};

int launch_fwd(const FwdParams& p, int d, cudaStream_t stream);
int launch_fwd_fp8(const Fp8Params& p, cudaStream_t stream);
int launch_fp8_transpose_v(const uint8_t* v, uint8_t* vt, int BH, int N, int npad, cudaStream_t stream);
int launch_decode(const DecParams& p, int d, cudaStream_t stream);
int launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dout, const float* lse, float* nd,
                          float* nlse, float* dq_acc, int BH, int N, int npad, int d, cudaStream_t stream);
int launch_bwd_main(const BwdParams& p, int d, cudaStream_t stream);
int launch_bwd_dq_convert(const float* dq_acc, __nv_bfloat16* dq, long long n, float scale,
                          cudaStream_t stream);
int launch_wait_timeout_probe(int* status, uint64_t timeout_ns, cudaStream_t stream);

// Steps of fa_bwd (fa_api.cu) for entry points that supply the workspace
// themselves: the shape check, the pointer and scale checks, the device check
// (compute capability 10.3), and the three backward stages on `workspace`.
// Each returns FA_OK (0) or an fa_status code.
int api_check_shape(int B, int H, int N, int d);
int api_check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dout,
                       const float* lse, const void* dq, const void* dk, const void* dv, float scale);
int api_device_ready();
int api_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
            void* dq, void* dk, void* dv, void* workspace, int B, int H, int N, int d, float scale, int causal,
            cudaStream_t stream);

}  // namespace fa
