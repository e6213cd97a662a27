// CUDA-core kernels of the block backward (bf16 storage, fp32 arithmetic): transposes
// that turn activations and weights into K-major GEMM operands, and the elementwise and
// reduction steps between the backward's tensor-core products (Krea 2 Technical Report,
// "训练" / Training: the gradients of the single-stream block of "架构" / Architecture).
// The products themselves run on gemm_tc's plain epilogue.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace kd {
namespace {

constexpr int TB = 64;  // transpose tile (64 x 64 bf16), 256 threads

// dst[z][c, r] = src[z][r, c] for r < R, 0 for R <= r < Rp (bf16). Loads and stores move
// 8 elements (16 bytes) per thread where the row lies inside the matrix and the address is
// 16-byte aligned, else element by element.
__global__ void __launch_bounds__(256) transpose_kernel(const bf16* __restrict__ src, int R, int C, long long lds,
                                                        long long src_bs, bf16* __restrict__ dst, int Rp,
                                                        long long ldd, long long dst_bs) {
  __shared__ uint16_t tile[TB][TB + 2];  // +2: a column read walks the banks
  const uint16_t* s = reinterpret_cast<const uint16_t*>(src) + blockIdx.z * src_bs;
  uint16_t* d = reinterpret_cast<uint16_t*>(dst) + blockIdx.z * dst_bs;
  const int r0 = blockIdx.y * TB, c0 = blockIdx.x * TB;
  const int t = threadIdx.x, chunk = t & 7;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int k = (t >> 3) + 32 * h;  // tile row
    const int r = r0 + k, c = c0 + 8 * chunk;
    uint16_t v[8];
    const uint16_t* p = s + static_cast<long long>(r) * lds + c;
    if (r < R && c + 8 <= C && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[2 * i] = static_cast<uint16_t>(w[i] & 0xFFFFu);
        v[2 * i + 1] = static_cast<uint16_t>(w[i] >> 16);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = (r < R && c + i < C) ? p[i] : static_cast<uint16_t>(0);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) tile[k][8 * chunk + i] = v[i];
  }
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int k = (t >> 3) + 32 * h;  // tile column = destination row
    const int c = c0 + k, r = r0 + 8 * chunk;
    if (c >= C) continue;
    uint16_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = tile[8 * chunk + i][k];
    uint16_t* q = d + static_cast<long long>(c) * ldd + r;
    if (r + 8 <= Rp && (reinterpret_cast<uintptr_t>(q) & 15) == 0) {
      *reinterpret_cast<uint4*>(q) = make_uint4(v[0] | (static_cast<uint32_t>(v[1]) << 16),
                                                v[2] | (static_cast<uint32_t>(v[3]) << 16),
                                                v[4] | (static_cast<uint32_t>(v[5]) << 16),
                                                v[6] | (static_cast<uint32_t>(v[7]) << 16));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (r + i < Rp) q[i] = v[i];
    }
  }
}

__device__ __forceinline__ float ld_any(const void* p, long long i, int f32) {
  return f32 ? reinterpret_cast<const float*>(p)[i] : __bfloat162float(reinterpret_cast<const bf16*>(p)[i]);
}

// Gated residual, backward: y = res + gate * f. d_f = dy * gate (bf16); the gate's
// gradient sum_l dy * f is added to d_mod[b, chunk] and d_bias[chunk]. Block = 256
// consecutive columns x one chunk of rows of one batch element.
__global__ void gated_bwd_kernel(Fwd f, const void* __restrict__ dy, int dy_f32, const float* __restrict__ fv,
                                 const float* __restrict__ mod_shared, const float* __restrict__ mod_bias,
                                 int chunk, int rows_per, bf16* __restrict__ d_f, float* __restrict__ d_mod,
                                 float* __restrict__ d_bias) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.z;
  const int l0 = blockIdx.y * rows_per, l1 = min(l0 + rows_per, f.L);
  if (c >= f.d || l0 >= l1) return;
  const float gate = mod_shared[(b * 6 + chunk) * f.d + c] + mod_bias[chunk * f.d + c];
  float acc = 0.0f;
  for (int l = l0; l < l1; ++l) {
    const long long i = (static_cast<long long>(b) * f.L + l) * f.d + c;
    const float g = ld_any(dy, i, dy_f32);
    acc = fmaf(g, fv[i], acc);
    d_f[i] = __float2bfloat16_rn(g * gate);
  }
  atomicAdd(&d_mod[(b * 6 + chunk) * f.d + c], acc);
  atomicAdd(&d_bias[chunk * f.d + c], acc);
}

// block-wide sum (blockDim.x multiple of 32, <= 1024)
__device__ __forceinline__ float block_sum(float v, float* red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.0f;
  for (int i = 0; i < (blockDim.x >> 5); ++i) t += red[i];
  return t;
}

// Norm + modulation, backward, rows: y = n (1 + w)(1 + scale) + shift, n = x r,
// r = (mean(x^2) + eps)^(-1/2). dx = r dn - r^3 x mean(dn x) + d_res, dn = dy (1 + w)(1 + scale).
// One block per row; writes r to rstd[t] for the column pass. dx goes to a joint fp32 buffer
// (dx_f32) or, as the storage dtype, to split text / image buffers (dx_src).
__device__ __forceinline__ float4 ld4_any(const void* p, long long i, int f32) {
  if (f32) return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
  const uint2 u = *reinterpret_cast<const uint2*>(reinterpret_cast<const bf16*>(p) + i);
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y);
  return make_float4(a.x, a.y, b.x, b.y);
}

__global__ void __launch_bounds__(256) norm_bwd_rows_kernel(Fwd f, RowSrc xs, int x_f32, const float* __restrict__ dy,
                                                            const float* __restrict__ gain_w,
                                                            const float* __restrict__ mod_shared,
                                                            const float* __restrict__ mod_bias, int chunk_scale,
                                                            const void* __restrict__ d_res, int res_f32,
                                                            float* __restrict__ dx_f32, RowSrc dx_bf16,
                                                            float* __restrict__ rstd) {
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int b = t / f.L;
  const int d = f.d;  // a multiple of 64: four columns per access
  const void* x = x_f32 ? static_cast<const void*>(row_src_ptr<float>(xs, t, f.L, f.n_txt, f.n_img, d))
                        : static_cast<const void*>(row_src_ptr<bf16>(xs, t, f.L, f.n_txt, f.n_img, d));
  const float* ms = mod_shared + (static_cast<size_t>(b) * 6 + chunk_scale) * d;
  const float* mb = mod_bias + static_cast<size_t>(chunk_scale) * d;
  const float* dyr = dy + static_cast<long long>(t) * d;
  auto coef = [&](int c) {  // (1 + w)(1 + scale) for columns c .. c+3
    const float4 w = *reinterpret_cast<const float4*>(gain_w + c);
    const float4 s0 = *reinterpret_cast<const float4*>(ms + c);
    const float4 s1 = *reinterpret_cast<const float4*>(mb + c);
    return make_float4((1.0f + w.x) * (1.0f + s0.x + s1.x), (1.0f + w.y) * (1.0f + s0.y + s1.y),
                       (1.0f + w.z) * (1.0f + s0.z + s1.z), (1.0f + w.w) * (1.0f + s0.w + s1.w));
  };
  float ss = 0.0f, sdx = 0.0f;
  for (int c = 4 * threadIdx.x; c < d; c += 4 * blockDim.x) {
    const float4 xv = ld4_any(x, c, x_f32);
    const float4 A = coef(c);
    const float4 g = *reinterpret_cast<const float4*>(dyr + c);
    ss += xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
    sdx += g.x * A.x * xv.x + g.y * A.y * xv.y + g.z * A.z * xv.z + g.w * A.w * xv.w;
  }
  ss = block_sum(ss, red);
  sdx = block_sum(sdx, red);
  const float r = rsqrtf(ss / d + f.eps);
  const float k = r * r * r * (sdx / d);
  if (threadIdx.x == 0) rstd[t] = r;
  bf16* ob = dx_f32 ? nullptr : const_cast<bf16*>(row_src_ptr<bf16>(dx_bf16, t, f.L, f.n_txt, f.n_img, d));
  for (int c = 4 * threadIdx.x; c < d; c += 4 * blockDim.x) {
    const long long i = static_cast<long long>(t) * d + c;
    const float4 xv = ld4_any(x, c, x_f32);
    const float4 A = coef(c);
    const float4 g = *reinterpret_cast<const float4*>(dyr + c);
    const float4 rs = ld4_any(d_res, i, res_f32);
    const float4 o = make_float4(r * g.x * A.x - k * xv.x + rs.x, r * g.y * A.y - k * xv.y + rs.y,
                                 r * g.z * A.z - k * xv.z + rs.z, r * g.w * A.w - k * xv.w + rs.w);
    if (dx_f32) *reinterpret_cast<float4*>(dx_f32 + i) = o;
    else *reinterpret_cast<uint2*>(ob + c) = make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
  }
}

// Norm + modulation, backward, columns: per batch element b and column c,
// d_shift += sum_l dy, d_scale += (1 + w) sum_l dy n, d_w += (1 + scale_b) sum_l dy n.
__global__ void norm_bwd_cols_kernel(Fwd f, RowSrc xs, int x_f32, const float* __restrict__ rstd,
                                     const float* __restrict__ dy, const float* __restrict__ gain_w,
                                     const float* __restrict__ mod_shared, const float* __restrict__ mod_bias,
                                     int chunk_shift, int chunk_scale, int rows_per, float* __restrict__ d_mod,
                                     float* __restrict__ d_bias, float* __restrict__ d_gain) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  const int b = blockIdx.z;
  const int l0 = blockIdx.y * rows_per, l1 = min(l0 + rows_per, f.L);
  if (c >= f.d || l0 >= l1) return;
  float s_dy = 0.0f, s_dyn = 0.0f;
  for (int l = l0; l < l1; ++l) {
    const int t = b * f.L + l;
    const void* x = x_f32 ? static_cast<const void*>(row_src_ptr<float>(xs, t, f.L, f.n_txt, f.n_img, f.d))
                          : static_cast<const void*>(row_src_ptr<bf16>(xs, t, f.L, f.n_txt, f.n_img, f.d));
    const float g = dy[static_cast<long long>(t) * f.d + c];
    s_dy += g;
    s_dyn = fmaf(g, ld_any(x, c, x_f32) * rstd[t], s_dyn);
  }
  const float scale = mod_shared[(b * 6 + chunk_scale) * f.d + c] + mod_bias[chunk_scale * f.d + c];
  const float dsc = s_dyn * (1.0f + gain_w[c]);
  atomicAdd(&d_mod[(b * 6 + chunk_shift) * f.d + c], s_dy);
  atomicAdd(&d_bias[chunk_shift * f.d + c], s_dy);
  atomicAdd(&d_mod[(b * 6 + chunk_scale) * f.d + c], dsc);
  atomicAdd(&d_bias[chunk_scale * f.d + c], dsc);
  atomicAdd(&d_gain[c], s_dyn * (1.0f + scale));
}

// QK-RMSNorm + RoPE, backward, and the V gradient, into d_P (bf16 [T, ldp]). Block = 8
// warps over a chunk of rows of one head slot (blockIdx.y: q heads, then k heads, then v
// heads); a warp takes one row at a time, lane i the head-dim elements 4i .. 4i+3 (two
// rotation pairs). For q / k: d_n = rotation by -angle of d (fp32 gradient of the
// rotated, normalised head), dx = r dn (1 + w) - r^3 x mean(dn (1 + w) x) with x the raw
// projection (fp32 [T, ldr]) and r its rstd over hd; the gain's gradient sum d_n x r is
// added to d_gain. For v: d_P takes d_v.
__global__ void __launch_bounds__(256) qkv_bwd_kernel(Fwd f, const float* __restrict__ raw, int ldr,
                                                      const float* __restrict__ dq, const float* __restrict__ dk,
                                                      const float* __restrict__ dv,
                                                      const float* __restrict__ q_norm_w,
                                                      const float* __restrict__ k_norm_w,
                                                      const float2* __restrict__ rope, int rows_per,
                                                      bf16* __restrict__ d_P, int ldp, float* __restrict__ d_qw,
                                                      float* __restrict__ d_kw) {
  constexpr int HD = 128;
  __shared__ float red[8][HD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slot = blockIdx.y;
  const int kind = slot < f.n_q ? 0 : (slot < f.n_q + f.n_kv ? 1 : 2);
  const int head = kind == 0 ? slot : (kind == 1 ? slot - f.n_q : slot - f.n_q - f.n_kv);
  const int nh = kind == 0 ? f.n_q : f.n_kv;
  const float* dsrc = kind == 0 ? dq : (kind == 1 ? dk : dv);
  const int j0 = 4 * lane;
  const int col = (kind == 0 ? 0 : (kind == 1 ? f.n_q * HD : (f.n_q + f.n_kv) * HD)) + head * HD + j0;
  float w1[4] = {1.f, 1.f, 1.f, 1.f};
  if (kind < 2) {
    const float4 w4 = *reinterpret_cast<const float4*>((kind == 0 ? q_norm_w : k_norm_w) + j0);
    w1[0] = 1.0f + w4.x; w1[1] = 1.0f + w4.y; w1[2] = 1.0f + w4.z; w1[3] = 1.0f + w4.w;
  }
  const int t0 = blockIdx.x * rows_per, t1 = min(t0 + rows_per, f.T);
  float gacc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int t = t0 + warp; t < t1; t += 8) {
    const int b = t / f.L, l = t - b * f.L;
    const float4 g4 = *reinterpret_cast<const float4*>(dsrc + ((static_cast<long long>(b) * nh + head) * f.L + l) * HD + j0);
    bf16* out = d_P + static_cast<long long>(t) * ldp + col;
    if (kind == 2) {
      *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(g4.x, g4.y), pack_bf16x2(g4.z, g4.w));
      continue;
    }
    float dn[4] = {g4.x, g4.y, g4.z, g4.w};
    if (l >= f.n_txt) {  // rotation by the negative angle, pairs (j0, j0+1) and (j0+2, j0+3)
      const int n = l - f.n_txt, pr = n / f.img_w, pc = n - pr * f.img_w;
      const float2* tab = rope + (j0 < 64 ? pr : pc) * (HD / 4) + ((j0 & 63) >> 1);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float2 cs = tab[e];
        const float a = dn[2 * e], bb = dn[2 * e + 1];
        dn[2 * e] = a * cs.x + bb * cs.y;
        dn[2 * e + 1] = -a * cs.y + bb * cs.x;
      }
    }
    const float4 x4 = *reinterpret_cast<const float4*>(raw + static_cast<long long>(t) * ldr + col);
    const float x[4] = {x4.x, x4.y, x4.z, x4.w};
    const float ss = warp_sum(x[0] * x[0] + x[1] * x[1] + x[2] * x[2] + x[3] * x[3]);
    const float r = rsqrtf(ss / HD + f.eps);
    float dnw[4], md = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      dnw[e] = dn[e] * w1[e];
      md = fmaf(dnw[e], x[e], md);
      gacc[e] = fmaf(dn[e], x[e] * r, gacc[e]);
    }
    const float m = warp_sum(md) / HD;
    const float r3m = r * r * r * m;
    float o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = r * dnw[e] - r3m * x[e];
    *reinterpret_cast<uint2*>(out) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
  }
  if (kind < 2) {
#pragma unroll
    for (int e = 0; e < 4; ++e) red[warp][j0 + e] = gacc[e];
    __syncthreads();
    if (threadIdx.x < HD) {
      float s = 0.0f;
#pragma unroll
      for (int w = 0; w < 8; ++w) s += red[w][threadIdx.x];
      atomicAdd(kind == 0 ? &d_qw[threadIdx.x] : &d_kw[threadIdx.x], s);
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_transpose_bf16(const void* src, int R, int C, long long lds, long long src_bs, void* dst, int Rp,
                                  long long ldd, long long dst_bs, int batch, cudaStream_t st) {
  if (R <= 0 || C <= 0 || batch <= 0) return cudaSuccess;
  dim3 grid((C + TB - 1) / TB, (Rp + TB - 1) / TB, batch), block(256);
  transpose_kernel<<<grid, block, 0, st>>>(reinterpret_cast<const bf16*>(src), R, C, lds, src_bs,
                                           reinterpret_cast<bf16*>(dst), Rp, ldd, dst_bs);
  return cudaGetLastError();
}

cudaError_t launch_gated_bwd(const Fwd& f, const void* dy, int dy_f32, const float* fv, const float* mod_shared,
                             const float* mod_bias, int chunk, void* d_f, float* d_mod, float* d_bias,
                             cudaStream_t st) {
  const int rows_per = 64;
  dim3 grid((f.d + 255) / 256, (f.L + rows_per - 1) / rows_per, f.B);
  gated_bwd_kernel<<<grid, 256, 0, st>>>(f, dy, dy_f32, fv, mod_shared, mod_bias, chunk, rows_per,
                                         reinterpret_cast<bf16*>(d_f), d_mod, d_bias);
  return cudaGetLastError();
}

cudaError_t launch_norm_bwd(const Fwd& f, RowSrc xs, int x_f32, const float* dy, const float* gain_w,
                            const float* mod_shared, const float* mod_bias, int chunk_shift, int chunk_scale,
                            const void* d_res, int res_f32, float* dx_f32, RowSrc dx_bf16, float* rstd,
                            float* d_mod, float* d_bias, float* d_gain, cudaStream_t st) {
  if (f.T == 0) return cudaSuccess;
  norm_bwd_rows_kernel<<<f.T, 256, 0, st>>>(f, xs, x_f32, dy, gain_w, mod_shared, mod_bias, chunk_scale, d_res,
                                            res_f32, dx_f32, dx_bf16, rstd);
  const int rows_per = 64;
  dim3 grid((f.d + 255) / 256, (f.L + rows_per - 1) / rows_per, f.B);
  norm_bwd_cols_kernel<<<grid, 256, 0, st>>>(f, xs, x_f32, rstd, dy, gain_w, mod_shared, mod_bias, chunk_shift,
                                             chunk_scale, rows_per, d_mod, d_bias, d_gain);
  return cudaGetLastError();
}

cudaError_t launch_qkv_bwd(const Fwd& f, const float* raw, int ldr, const float* dq, const float* dk, const float* dv,
                           const float* q_norm_w, const float* k_norm_w, const float2* rope, void* d_P, int ldp,
                           float* d_qw, float* d_kw, cudaStream_t st) {
  if (f.T == 0) return cudaSuccess;
  const int rows_per = 64;
  dim3 grid((f.T + rows_per - 1) / rows_per, f.n_q + 2 * f.n_kv);
  qkv_bwd_kernel<<<grid, 256, 0, st>>>(f, raw, ldr, dq, dk, dv, q_norm_w, k_norm_w, rope, rows_per,
                                       reinterpret_cast<bf16*>(d_P), ldp, d_qw, d_kw);
  return cudaGetLastError();
}

}  // namespace kd
