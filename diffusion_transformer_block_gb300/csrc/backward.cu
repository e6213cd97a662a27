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

constexpr int TB = 32;  // transpose tile

// dst[z][c, r] = src[z][r, c] for r < R, 0 for R <= r < Rp (bf16).
__global__ void transpose_kernel(const bf16* __restrict__ src, int R, int C, long long lds, long long src_bs,
                                 bf16* __restrict__ dst, int Rp, long long ldd, long long dst_bs) {
  __shared__ bf16 tile[TB][TB + 2];
  const bf16* s = src + blockIdx.z * src_bs;
  bf16* d = dst + blockIdx.z * dst_bs;
  const int r0 = blockIdx.y * TB, c0 = blockIdx.x * TB;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  for (int k = ty; k < TB; k += 8) {
    const int r = r0 + k, c = c0 + tx;
    tile[k][tx] = (r < R && c < C) ? s[r * lds + c] : __float2bfloat16_rn(0.0f);
  }
  __syncthreads();
  for (int k = ty; k < TB; k += 8) {
    const int c = c0 + k, r = r0 + tx;
    if (c < C && r < Rp) d[c * ldd + r] = tile[tx][k];
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

// SwiGLU, backward: hmid = silu(a) u. d_au[t, 0:F] = d_hmid u silu'(a), d_au[t, F:2F] =
// d_hmid silu(a), silu'(a) = sigma(a) (1 + a (1 - sigma(a))).
__global__ void swiglu_bwd_kernel(const float* __restrict__ d_hmid, const float* __restrict__ a,
                                  const float* __restrict__ u, long long T, int F, bf16* __restrict__ d_au) {
  const long long n = T * F;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / F;
    const int j = static_cast<int>(i - t * F);
    const float av = a[i], sg = 1.0f / (1.0f + __expf(-av));
    const float dh = d_hmid[i];
    d_au[t * 2 * F + j] = __float2bfloat16_rn(dh * u[i] * sg * (1.0f + av * (1.0f - sg)));
    d_au[t * 2 * F + F + j] = __float2bfloat16_rn(dh * av * sg);
  }
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
__global__ void norm_bwd_rows_kernel(Fwd f, RowSrc xs, int x_f32, const float* __restrict__ dy,
                                     const float* __restrict__ gain_w, const float* __restrict__ mod_shared,
                                     const float* __restrict__ mod_bias, int chunk_scale, const void* __restrict__ d_res,
                                     int res_f32, float* __restrict__ dx_f32, RowSrc dx_bf16,
                                     float* __restrict__ rstd) {
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int b = t / f.L;
  const int d = f.d;
  const void* x = x_f32 ? static_cast<const void*>(row_src_ptr<float>(xs, t, f.L, f.n_txt, f.n_img, d))
                        : static_cast<const void*>(row_src_ptr<bf16>(xs, t, f.L, f.n_txt, f.n_img, d));
  float ss = 0.0f, sdx = 0.0f;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float xv = ld_any(x, c, x_f32);
    const float A = (1.0f + gain_w[c]) * (1.0f + mod_shared[(b * 6 + chunk_scale) * d + c] +
                                          mod_bias[chunk_scale * d + c]);
    ss = fmaf(xv, xv, ss);
    sdx = fmaf(dy[static_cast<long long>(t) * d + c] * A, xv, sdx);
  }
  ss = block_sum(ss, red);
  sdx = block_sum(sdx, red);
  const float r = rsqrtf(ss / d + f.eps);
  const float k = r * r * r * (sdx / d);
  if (threadIdx.x == 0) rstd[t] = r;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const long long i = static_cast<long long>(t) * d + c;
    const float xv = ld_any(x, c, x_f32);
    const float A = (1.0f + gain_w[c]) * (1.0f + mod_shared[(b * 6 + chunk_scale) * d + c] +
                                          mod_bias[chunk_scale * d + c]);
    const float g = r * dy[i] * A - k * xv + ld_any(d_res, i, res_f32);
    if (dx_f32) {
      dx_f32[i] = g;
    } else {
      bf16* o = const_cast<bf16*>(row_src_ptr<bf16>(dx_bf16, t, f.L, f.n_txt, f.n_img, d));
      o[c] = __float2bfloat16_rn(g);
    }
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

// Output gate, backward: og = o sigmoid(g). d_o = d_og sigmoid(g), stored head-major (bf16
// [B, n_q, L, 128], so that a KV group's heads are one contiguous block of rows); the
// gate's gradient d_og o sigmoid(g)(1 - sigmoid(g)) goes to d_P's g columns (bf16).
__global__ void gate_bwd_kernel(const float* __restrict__ d_og, const float* __restrict__ o,
                                const bf16* __restrict__ g, long long T, int L, int n_q, int gate_on,
                                bf16* __restrict__ d_o, bf16* __restrict__ d_P, int ldp, int goff) {
  const int nq = n_q * 128;
  const long long n = T * nq;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long t = i / nq;
    const int col = static_cast<int>(i - t * nq);
    const long long b = t / L, l = t - b * L;
    const long long hm = ((b * n_q + (col >> 7)) * L + l) * 128 + (col & 127);
    const float dv = d_og[i];
    if (gate_on) {
      const float sg = 1.0f / (1.0f + __expf(-__bfloat162float(g[i])));
      d_o[hm] = __float2bfloat16_rn(dv * sg);
      d_P[t * ldp + goff + col] = __float2bfloat16_rn(dv * o[i] * sg * (1.0f - sg));
    } else {
      d_o[hm] = __float2bfloat16_rn(dv);
    }
  }
}

// QK-RMSNorm + RoPE, backward, and the V gradient, into d_P (bf16 [T, ldp]). Block = one
// head slot (blockIdx.y: q heads, then k heads, then v heads) over a chunk of rows;
// thread j = head-dim element. For q / k: d_n = rotation by -angle of d (fp32 gradient
// of the rotated, normalised head), dx = r dn (1 + w) - r^3 x mean(dn (1 + w) x) with x the
// raw projection (fp32 [T, ldr]) and r its rstd over hd; the gain's gradient
// sum d_n x r is added to d_gain. For v: d_P takes d_v.
__global__ void qkv_bwd_kernel(Fwd f, const float* __restrict__ raw, int ldr, const float* __restrict__ dq,
                               const float* __restrict__ dk, const float* __restrict__ dv,
                               const float* __restrict__ q_norm_w, const float* __restrict__ k_norm_w,
                               const float2* __restrict__ rope, int rows_per, bf16* __restrict__ d_P, int ldp,
                               float* __restrict__ d_qw, float* __restrict__ d_kw) {
  __shared__ float red[32];
  const int HD = 128;
  const int j = threadIdx.x;  // 0..127
  const int slot = blockIdx.y;
  const int kind = slot < f.n_q ? 0 : (slot < f.n_q + f.n_kv ? 1 : 2);
  const int head = kind == 0 ? slot : (kind == 1 ? slot - f.n_q : slot - f.n_q - f.n_kv);
  const int nh = kind == 0 ? f.n_q : f.n_kv;
  const float* dsrc = kind == 0 ? dq : (kind == 1 ? dk : dv);
  const int col = (kind == 0 ? 0 : (kind == 1 ? f.n_q * HD : (f.n_q + f.n_kv) * HD)) + head * HD + j;
  const float wj = kind == 0 ? q_norm_w[j] : (kind == 1 ? k_norm_w[j] : 0.0f);
  const int t0 = blockIdx.x * rows_per, t1 = min(t0 + rows_per, f.T);
  float gacc = 0.0f;
  for (int t = t0; t < t1; ++t) {
    const int b = t / f.L, l = t - b * f.L;
    const float g = dsrc[((static_cast<long long>(b) * nh + head) * f.L + l) * HD + j];
    if (kind == 2) {
      d_P[static_cast<long long>(t) * ldp + col] = __float2bfloat16_rn(g);
      continue;
    }
    // rotation by the negative angle: pair (2p, 2p+1) of this element
    float dn = g;
    if (l >= f.n_txt) {
      const int n = l - f.n_txt, pr = n / f.img_w, pc = n - pr * f.img_w;
      const float2 cs = rope[(j < 64 ? pr : pc) * (HD / 4) + ((j & 63) >> 1)];
      const float other = __shfl_xor_sync(0xffffffffu, g, 1);
      dn = (j & 1) == 0 ? g * cs.x + other * cs.y : -other * cs.y + g * cs.x;
    }
    const float x = raw[static_cast<long long>(t) * ldr + col];
    const float ss = block_sum(x * x, red);
    const float r = rsqrtf(ss / HD + f.eps);
    const float dnw = dn * (1.0f + wj);
    const float m = block_sum(dnw * x, red) / HD;
    gacc = fmaf(dn, x * r, gacc);
    d_P[static_cast<long long>(t) * ldp + col] = __float2bfloat16_rn(r * dnw - r * r * r * x * m);
  }
  if (kind < 2) atomicAdd(kind == 0 ? &d_qw[j] : &d_kw[j], gacc);
}

// D[b, h, l] = sum_j d_o[b, h, l, j] o[t, h hd + j] (t = b L + l, hd = 128; d_o head-major):
// the row term of the softmax gradient, rowsum(P dP) = rowsum(dO O). One warp per (row, head).
__global__ void attn_rowdot_kernel(const bf16* __restrict__ d_o, const float* __restrict__ o, int T, int L, int Lp,
                                   int n_q, float* __restrict__ D) {
  const long long wid = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= static_cast<long long>(T) * n_q) return;
  const int t = static_cast<int>(wid / n_q), h = static_cast<int>(wid - static_cast<long long>(t) * n_q);
  const int b = t / L, l = t - b * L;
  const long long base = static_cast<long long>(t) * n_q * 128 + h * 128 + lane * 4;
  const long long hm = ((static_cast<long long>(b) * n_q + h) * L + l) * 128 + lane * 4;
  const uint2 u = *reinterpret_cast<const uint2*>(d_o + hm);
  const float4 ov = *reinterpret_cast<const float4*>(o + base);
  const float2 a = unpack_bf16x2(u.x), b2 = unpack_bf16x2(u.y);
  float s = a.x * ov.x + a.y * ov.y + b2.x * ov.z + b2.y * ov.w;
  s = warp_sum(s);
  if (lane == 0) D[(static_cast<long long>(b) * n_q + h) * Lp + l] = s;
}

}  // namespace

// ------------------------------------------------------------------ launchers
cudaError_t launch_attn_rowdot(const void* d_o, const float* o, int T, int L, int Lp, int n_q, float* D,
                               cudaStream_t st) {
  const long long warps = static_cast<long long>(T) * n_q;
  if (warps == 0) return cudaSuccess;
  const long long blocks = (warps * 32 + 255) / 256;
  attn_rowdot_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(reinterpret_cast<const bf16*>(d_o), o, T, L, Lp,
                                                                   n_q, D);
  return cudaGetLastError();
}
cudaError_t launch_transpose_bf16(const void* src, int R, int C, long long lds, long long src_bs, void* dst, int Rp,
                                  long long ldd, long long dst_bs, int batch, cudaStream_t st) {
  if (R <= 0 || C <= 0 || batch <= 0) return cudaSuccess;
  dim3 grid((C + TB - 1) / TB, (Rp + TB - 1) / TB, batch), block(TB, 8);
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

cudaError_t launch_swiglu_bwd(const float* d_hmid, const float* a, const float* u, long long T, int F, void* d_au,
                              int num_sms, cudaStream_t st) {
  swiglu_bwd_kernel<<<num_sms * 8, 256, 0, st>>>(d_hmid, a, u, T, F, reinterpret_cast<bf16*>(d_au));
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

cudaError_t launch_gate_bwd(const float* d_og, const float* o, const void* g, long long T, int L, int n_q, int gate_on,
                            void* d_o, void* d_P, int ldp, int goff, int num_sms, cudaStream_t st) {
  gate_bwd_kernel<<<num_sms * 8, 256, 0, st>>>(d_og, o, reinterpret_cast<const bf16*>(g), T, L, n_q, gate_on,
                                               reinterpret_cast<bf16*>(d_o), reinterpret_cast<bf16*>(d_P), ldp, goff);
  return cudaGetLastError();
}

cudaError_t launch_qkv_bwd(const Fwd& f, const float* raw, int ldr, const float* dq, const float* dk, const float* dv,
                           const float* q_norm_w, const float* k_norm_w, const float2* rope, void* d_P, int ldp,
                           float* d_qw, float* d_kw, cudaStream_t st) {
  if (f.T == 0) return cudaSuccess;
  const int rows_per = 64;
  dim3 grid((f.T + rows_per - 1) / rows_per, f.n_q + 2 * f.n_kv);
  qkv_bwd_kernel<<<grid, 128, 0, st>>>(f, raw, ldr, dq, dk, dv, q_norm_w, k_norm_w, rope, rows_per,
                                       reinterpret_cast<bf16*>(d_P), ldp, d_qw, d_kw);
  return cudaGetLastError();
}

}  // namespace kd
