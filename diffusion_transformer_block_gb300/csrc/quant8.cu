// e4m3 casts of GEMM operands for the 8-bit block ("训练 › 预训练" / Training › Pretraining:
// 8-bit GEMMs with tensor-wise or row-wise scaling).
//
// A group (one row, or the whole tensor) with largest magnitude amax is multiplied by the
// power of two 2^k, k the largest integer with amax 2^k <= 448, and cast to e4m3 (nearest,
// ties to even, saturating); 2^-k dequantises it. Both kernels are HBM-bound streams with
// 16-byte accesses.
#include "common.cuh"
#include "internal.h"

namespace kd {
namespace {

constexpr int QT = 256;  // threads per CTA

// q[r, :] = e4m3(src[r, :] * 2^k_r); dq[r] = 2^-k_r (per_row) or one k for all rows.
__global__ void __launch_bounds__(QT) quant_e4m3_kernel(const bf16* __restrict__ src, int R, int K,
                                                        const float* __restrict__ rowamax, int per_row,
                                                        uint8_t* __restrict__ q, float* __restrict__ dq) {
  __shared__ float red[QT / 32];
  __shared__ float tensor_scale;
  if (!per_row) {
    float m = 0.0f;
    for (int i = threadIdx.x; i < R; i += QT) m = fmaxf(m, rowamax[i]);
    m = warp_max(m);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < QT / 32; ++w) t = fmaxf(t, red[w]);
      const int k = e4m3_scale_exp(t);
      tensor_scale = pow2f(k);
      if (blockIdx.x == 0) dq[0] = pow2f(-k);
    }
    __syncthreads();
  }
  const size_t chunks = static_cast<size_t>(R) * (K / 16);
  for (size_t c = static_cast<size_t>(blockIdx.x) * QT + threadIdx.x; c < chunks;
       c += static_cast<size_t>(gridDim.x) * QT) {
    const size_t e0 = c * 16;
    const int r = static_cast<int>(e0 / K);
    float scale;
    if (per_row) {
      const int k = e4m3_scale_exp(rowamax[r]);
      scale = pow2f(k);
      if (e0 == static_cast<size_t>(r) * K) dq[r] = pow2f(-k);
    } else {
      scale = tensor_scale;
    }
    const uint4* s4 = reinterpret_cast<const uint4*>(src + e0);
    const uint4 u0 = s4[0], u1 = s4[1];
    const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float lo[8], hi[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 a = unpack_bf16x2(w[i]), b = unpack_bf16x2(w[4 + i]);
      lo[2 * i] = a.x * scale;
      lo[2 * i + 1] = a.y * scale;
      hi[2 * i] = b.x * scale;
      hi[2 * i + 1] = b.y * scale;
    }
    const uint2 a8 = cvt_e4m3x8(lo), b8 = cvt_e4m3x8(hi);
    *reinterpret_cast<uint4*>(q + e0) = make_uint4(a8.x, a8.y, b8.x, b8.y);
  }
}

// rowamax[r] = max |src[r, :]|, one warp per row
__global__ void __launch_bounds__(QT) row_amax_kernel(const bf16* __restrict__ src, int R, int K,
                                                      float* __restrict__ rowamax) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (QT / 32);
  for (int r = blockIdx.x * (QT / 32) + (threadIdx.x >> 5); r < R; r += warps) {
    const bf16* row = src + static_cast<size_t>(r) * K;
    float m = 0.0f;
    for (int k = lane * 8; k < K; k += 256) {
      const uint4 u = *reinterpret_cast<const uint4*>(row + k);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v = unpack_bf16x2(w[i]);
        m = fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
      }
    }
    m = warp_max(m);
    if (lane == 0) rowamax[r] = m;
  }
}

}  // namespace

cudaError_t launch_quant_e4m3(const void* src, int R, int K, const float* rowamax, int per_row, void* q, float* dq,
                              int num_sms, cudaStream_t st) {
  if (R <= 0 || K <= 0) return cudaSuccess;
  if (K % 16) return cudaErrorInvalidValue;
  const long long chunks = static_cast<long long>(R) * (K / 16);
  long long grid = (chunks + QT - 1) / QT;
  const long long cap = 4LL * num_sms;  // 4 CTAs per SM, grid-stride beyond
  if (grid > cap) grid = cap;
  quant_e4m3_kernel<<<static_cast<unsigned>(grid), QT, 0, st>>>(reinterpret_cast<const bf16*>(src), R, K, rowamax,
                                                                 per_row, reinterpret_cast<uint8_t*>(q), dq);
  return cudaGetLastError();
}

cudaError_t launch_row_amax(const void* src, int R, int K, float* rowamax, int num_sms, cudaStream_t st) {
  if (R <= 0) return cudaSuccess;
  if (K % 8) return cudaErrorInvalidValue;
  long long grid = (R + QT / 32 - 1) / (QT / 32);
  const long long cap = 4LL * num_sms;
  if (grid > cap) grid = cap;
  row_amax_kernel<<<static_cast<unsigned>(grid), QT, 0, st>>>(reinterpret_cast<const bf16*>(src), R, K, rowamax);
  return cudaGetLastError();
}

}  // namespace kd
