// fa_bwd_aux.cu -- the two memory-bound stages around the backward main
// kernel.
//
// Preprocess: D_i = sum_c dO[i,c] O[i,c] in fp32 ("FlashAttention" notes,
// "Backward Pass of flashattention": D_i = do_i^T o_i replaces
// rowsum(P o dP), which would need a whole row of P), stored as -D_i next to
// -LSE_i * log2(e) in the workspace, and the fp32 dQ accumulator set to zero.
// Convert: dQ = bf16(scale * accumulator), the scale being the chain-rule
// factor of S = scale * Q K^T.
#include "fa_common.cuh"

namespace fa {

// One thread per 8 head-dim elements (16-byte loads); d/8 threads per row.
// Rows are walked per head padded to npad (a multiple of 128): row n < N
// writes -D_n and -LSE_n * log2(e) (the form the main kernel consumes) and
// zeroes its dQ accumulator row; rows N..npad-1 write zeros, so every
// 64- or 128-row step of the main kernel reads finite values.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const uint4* __restrict__ o,
                                                             const uint4* __restrict__ dout,
                                                             const float* __restrict__ lse,
                                                             float* __restrict__ nd, float* __restrict__ nlse,
                                                             float4* __restrict__ dq_acc, int BH, int N, int npad) {
  constexpr int TPR = D / 8;  // threads per row (8 or 16), a power of two within a warp
  const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long prow = t / TPR;                        // padded row: bh * npad + n
  const int part = static_cast<int>(t % TPR);
  const long long bh = prow / npad;
  const int n = static_cast<int>(prow % npad);
  const bool live = bh < BH && n < N;
  const long long row = bh * N + n;                      // row in the [BH][N] tensors
  float acc = 0.f;
  if (live) {
    const uint4 a = __ldg(o + row * TPR + part);
    const uint4 b = __ldg(dout + row * TPR + part);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(a2[i]);
      const float2 y = __bfloat1622float2(b2[i]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    float4* z = dq_acc + (row * D + part * 8) / 4;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (bh < BH && part == 0) {
    if (live) {
      const float l = __ldg(lse + row);
      nd[prow] = -acc;
      // a row with no visible key (LSE = -inf) is never visited; keep it finite
      nlse[prow] = isinf(l) ? 0.f : -l * 1.4426950408889634f;
    } else {
      nd[prow] = 0.f;
      nlse[prow] = 0.f;
    }
  }
}

int launch_bwd_preprocess(const __nv_bfloat16* o, const __nv_bfloat16* dout, const float* lse, float* nd,
                          float* nlse, float* dq_acc, int BH, int N, int npad, int d, cudaStream_t stream) {
  const long long threads = static_cast<long long>(BH) * npad * (d / 8);
  const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
  if (d == 128)
    bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(o),
                                                         reinterpret_cast<const uint4*>(dout), lse, nd, nlse,
                                                         reinterpret_cast<float4*>(dq_acc), BH, N, npad);
  else if (d == 64)
    bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(reinterpret_cast<const uint4*>(o),
                                                        reinterpret_cast<const uint4*>(dout), lse, nd, nlse,
                                                        reinterpret_cast<float4*>(dq_acc), BH, N, npad);
  else
    return -2;
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// Eight elements per thread: two 16-byte loads, one 16-byte store.
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                             uint4* __restrict__ dq, long long n8, float scale) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(acc + 2 * i);
    const float4 b = __ldg(acc + 2 * i + 1);
    uint4 r;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(a.x * scale, a.y * scale); r.x = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(a.z * scale, a.w * scale); r.y = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(b.x * scale, b.y * scale); r.z = *reinterpret_cast<uint32_t*>(&h);
    h = __floats2bfloat162_rn(b.z * scale, b.w * scale); r.w = *reinterpret_cast<uint32_t*>(&h);
    dq[i] = r;
  }
}

int launch_bwd_dq_convert(const float* dq_acc, __nv_bfloat16* dq, long long n, float scale, cudaStream_t stream) {
  const long long n8 = n / 8;  // d is 64 or 128, so n is a multiple of 8
  long long blocks = (n8 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;  // a few resident waves on 152 SMs; the loop strides the rest
  if (blocks < 1) blocks = 1;
  bwd_dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint4*>(dq), n8, scale);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace fa
