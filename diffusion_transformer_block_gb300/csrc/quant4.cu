// NVFP4 casts of GEMM operands (Krea 2 Technical Report, "讨论与未来工作" / Discussion and
// future work: NVFP4 pretraining as a next step).
//
// An operand [R, K] (K a multiple of 64) becomes E2M1 codes, two per byte (element 2i in
// the low nibble), with one E4M3 scale per 16 consecutive elements of a row and one
// power-of-two tensor scale s_t = 2^j, j the smallest integer with amax <= 448 * 6 * 2^j:
//   s_b = E4M3(amax_b / (6 s_t)),  q_i = E2M1(x_i / (s_b s_t))  (q = 0 where s_b = 0),
// both casts rounding to nearest even and saturating. Every division is by an exact value
// (6 s_t, s_b s_t), so fp32 takes the same rounding decisions as exact arithmetic.
//
// The scales are stored in the order the tensor core's scale copy reads them: for each
// 128-row block rb and each 64-element step ks of K, a 512-byte atom whose byte
// (r % 32) * 16 + (r / 32) * 4 + j holds the scale of row r (of the block) for elements
// 16 j .. 16 j + 15 of the step. Rows of the last block past R get scale 0.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace kd {
namespace {

constexpr int Q4T = 256;  // threads per CTA of the cast

// the power-of-two tensor scale of a tensor with largest magnitude amax
__device__ __forceinline__ float nvfp4_tensor_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  int e = 0;
  const float m0 = frexpf(amax / 2688.0f, &e);  // amax / (448 * 6) = m0 2^e, 0.5 <= m0 < 1
  return pow2f(m0 == 0.5f ? e - 1 : e);
}

// One 16-element block (two 16-byte units u0, u1 of bf16) of a row: returns its scale
// byte and writes its eight code bytes to lo, hi.
__device__ __forceinline__ uint32_t nvfp4_block(const uint4& u0, const uint4& u1, float six_ts, float ts,
                                                uint32_t& lo, uint32_t& hi) {
  const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
  float v[16];
  float amax = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float2 f = unpack_bf16x2(w[q]);
    v[2 * q] = f.x;
    v[2 * q + 1] = f.y;
    amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
  }
  const uint32_t sbyte = cvt_e4m3x2(amax / six_ts, 0.0f) & 0xFFu;  // block scale code
  __nv_fp8_e4m3 sb8;
  sb8.__x = static_cast<__nv_fp8_storage_t>(sbyte);
  const float den = static_cast<float>(sb8) * ts;  // exact: an E4M3 value times a power of two
  lo = 0;
  hi = 0;
  if (den > 0.0f) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      lo |= cvt_e2m1x2(v[2 * q] / den, v[2 * q + 1] / den) << (8 * q);
      hi |= cvt_e2m1x2(v[8 + 2 * q] / den, v[8 + 2 * q + 1] / den) << (8 * q);
    }
  }
  return sbyte;
}

// Persistent, one thread per (row, 64-element step): it reads the step's 128 bytes of the
// row, writes their 32 code bytes with two 16-byte stores and the row's four scale bytes
// of the step with one 4-byte store. Items run through the scale atoms in order, 128 rows
// of one atom after another, so a warp covers 32 rows of one atom and its scale stores
// fall into one 512-byte atom. Every CTA first reduces the row amaxes to the tensor scale
// (block 0 also stores it).
__global__ void __launch_bounds__(Q4T, 3) nvfp4_cast_kernel(const bf16* __restrict__ src, int R, int K,
                                                            const float* __restrict__ rowamax,
                                                            float* __restrict__ ts_out, uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ sf) {
  __shared__ float red[Q4T / 32];
  __shared__ float ts_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  {
    float m = 0.0f;
#pragma unroll 8
    for (int i = threadIdx.x; i < R; i += Q4T) m = fmaxf(m, rowamax[i]);
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float amax = 0.0f;
      for (int w = 0; w < Q4T / 32; ++w) amax = fmaxf(amax, red[w]);
      ts_sh = nvfp4_tensor_scale(amax);
      if (blockIdx.x == 0) ts_out[0] = ts_sh;
    }
    __syncthreads();
  }
  const float ts = ts_sh;
  const float six_ts = 6.0f * ts;
  const int KS = K / 64;
  const int items = (R + 127) / 128 * 128 * KS;  // the launcher checks that this fits an int
  for (int i = blockIdx.x * Q4T + threadIdx.x; i < items; i += gridDim.x * Q4T) {
    const int a = i >> 7, rr = i & 127;  // scale atom, row inside its 128-row block
    const int rb = a / KS, ks = a - rb * KS;
    const int r = rb * 128 + rr;
    uint32_t bytes = 0;
    if (r < R) {
      const uint4* p = reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * K + ks * 64);
      uint4 u[8];
#pragma unroll
      for (int t = 0; t < 8; ++t) u[t] = p[t];
      uint32_t c[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) bytes |= nvfp4_block(u[2 * j], u[2 * j + 1], six_ts, ts, c[2 * j], c[2 * j + 1]) << (8 * j);
      uint4* o = reinterpret_cast<uint4*>(codes + static_cast<size_t>(r) * (K / 2) + ks * 32);
      o[0] = make_uint4(c[0], c[1], c[2], c[3]);
      o[1] = make_uint4(c[4], c[5], c[6], c[7]);
    }
    *reinterpret_cast<uint32_t*>(sf + static_cast<size_t>(a) * 512 + (rr & 31) * 16 + (rr >> 5) * 4) = bytes;
  }
}

}  // namespace

size_t nvfp4_scale_bytes(long long rows, long long cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return static_cast<size_t>((rows + 127) / 128 * 128) * static_cast<size_t>(cols / 16);
}

cudaError_t launch_nvfp4_cast(const void* src, int R, int K, const float* rowamax, float* ts, void* codes, void* sf,
                              int num_sms, cudaStream_t st) {
  if (R <= 0 || K <= 0) return cudaSuccess;
  if (K % 64) return cudaErrorInvalidValue;
  const long long items = (static_cast<long long>(R) + 127) / 128 * 128 * (K / 64);
  if (items > (1LL << 30)) return cudaErrorInvalidValue;
  long long grid = (items + Q4T - 1) / Q4T;
  const long long cap = 3LL * num_sms;  // resident CTAs, each paying the amax reduction once
  if (grid > cap) grid = cap;
  nvfp4_cast_kernel<<<static_cast<unsigned>(grid), Q4T, 0, st>>>(reinterpret_cast<const bf16*>(src), R, K, rowamax,
                                                                  ts, reinterpret_cast<uint8_t*>(codes),
                                                                  reinterpret_cast<uint8_t*>(sf));
  return cudaGetLastError();
}

}  // namespace kd
