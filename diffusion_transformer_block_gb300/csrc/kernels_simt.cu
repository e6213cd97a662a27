// CUDA-core kernels of the DiT block library (the norm kernel lives in norm.cu).
//
//  * temb_sinusoid  (both modes): the sinusoidal timestep embedding ("Timestep
//    conditioning"), argument and sin/cos in fp64 then rounded to fp32.
//  * fp32 check mode: a plain tiled fp32 GEMM, the QK-norm + RoPE scatter, the GQA
//    attention with the sigmoid gate ("Transformer block"), the gated residual and the
//    SwiGLU product, as separate simple kernels with fp32 arithmetic (no tensor cores).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace kd {

// ============================================================== timestep sinusoid
// e[b] = [cos(1000 t w_i) | sin(1000 t w_i)], w_i = 10000^(-i/128), i < 128.
__global__ void temb_sinusoid_kernel(const float* __restrict__ t, int B, float* __restrict__ e) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * 128) return;
  const int b = idx / 128, i = idx - b * 128;
  const double w = exp(-log(10000.0) * static_cast<double>(i) / 128.0);
  const double arg = 1000.0 * static_cast<double>(t[b]) * w;
  double s, c;
  sincos(arg, &s, &c);
  e[b * 256 + i] = static_cast<float>(c);
  e[b * 256 + 128 + i] = static_cast<float>(s);
}

cudaError_t launch_temb_sinusoid(const float* t, int B, float* e, cudaStream_t st) {
  const int n = B * 128;
  temb_sinusoid_kernel<<<(n + 127) / 128, 128, 0, st>>>(t, B, e);
  return cudaGetLastError();
}

// ============================================================== fp32 SIMT GEMM
// C[M,N] = act(A[M,K] W[N,K]^T + bias). 64x64 tile, BK = 16, 256 threads, 4x4 per thread.
constexpr int SG_BM = 64, SG_BN = 64, SG_BK = 16;
__global__ void __launch_bounds__(256) gemm_simt_f32_kernel(const float* __restrict__ A, const float* __restrict__ W,
                                                            float* __restrict__ C, int M, int N, int K,
                                                            const float* __restrict__ bias, int act) {
  __shared__ float As[SG_BK][SG_BM + 4];
  __shared__ float Ws[SG_BK][SG_BN + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * SG_BM, n0 = blockIdx.x * SG_BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += SG_BK) {
    for (int i = threadIdx.x; i < SG_BM * SG_BK; i += 256) {
      const int r = i / SG_BK, c = i % SG_BK;
      const int gm = m0 + r, gk = k0 + c;
      As[c][r] = (gm < M && gk < K) ? A[static_cast<size_t>(gm) * K + gk] : 0.f;
      const int gn = n0 + r;
      Ws[c][r] = (gn < N && gk < K) ? W[static_cast<size_t>(gn) * K + gk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SG_BK; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int gm = m0 + ty * 4 + i;
    if (gm >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int gn = n0 + tx * 4 + j;
      if (gn >= N) continue;
      float v = acc[i][j] + (bias ? bias[gn] : 0.f);
      if (act == 1) v = v / (1.0f + expf(-v));
      C[static_cast<size_t>(gm) * N + gn] = v;
    }
  }
}

cudaError_t launch_gemm_simt_f32(const float* A, const float* W, float* C, int M, int N, int K, const float* bias,
                                 int act, cudaStream_t st) {
  dim3 grid((N + SG_BN - 1) / SG_BN, (M + SG_BM - 1) / SG_BM);
  gemm_simt_f32_kernel<<<grid, 256, 0, st>>>(A, W, C, M, N, K, bias, act);
  return cudaGetLastError();
}

// ============================================================== fp32: QK-norm + RoPE + scatter
// One warp per (row, head segment). Segments: n_q query heads, n_kv key heads, n_kv
// value heads, then n_q gate heads. Lane owns hd/32 consecutive channels (whole pairs).
template <int E>
__global__ void qkvg_post_f32_kernel(Fwd f, const float* __restrict__ raw, QkvgDst dst) {
  const int nseg = (f.gate_on ? 2 * f.n_q : f.n_q) + 2 * f.n_kv;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= f.T * nseg) return;
  const int m = warp / nseg, s = warp - m * nseg;
  const int b = m / f.L, l = m - b * f.L;
  const int hd = f.hd, N = nseg * hd;
  float v[E];
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = raw[static_cast<size_t>(m) * N + s * hd + lane * E + i];

  int kind, head;  // 0 q, 1 k, 2 v, 3 g
  if (s < f.n_q) { kind = 0; head = s; }
  else if (s < f.n_q + f.n_kv) { kind = 1; head = s - f.n_q; }
  else if (s < f.n_q + 2 * f.n_kv) { kind = 2; head = s - f.n_q - f.n_kv; }
  else { kind = 3; head = s - f.n_q - 2 * f.n_kv; }

  if (kind <= 1) {
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) ss = fmaf(v[i], v[i], ss);
    ss = warp_sum(ss);
    const float rstd = 1.0f / sqrtf(ss / static_cast<float>(hd) + f.eps);
    const float* w = kind == 0 ? dst.q_norm_w : dst.k_norm_w;
#pragma unroll
    for (int i = 0; i < E; ++i) v[i] = v[i] * rstd * (1.0f + w[lane * E + i]);
    if (l >= f.n_txt) {  // image token: rotate pairs by (row, col) position
      const int n = l - f.n_txt, r = n / f.img_w, c = n - r * f.img_w;
      const int quarter = hd / 4;
#pragma unroll
      for (int i = 0; i < E; i += 2) {
        const int p = (lane * E + i) / 2;  // pair index in [0, hd/2)
        const int half = p / quarter, j = p - half * quarter;
        const float2 cs = dst.rope[(half == 0 ? r : c) * quarter + j];
        const float a = v[i], bb = v[i + 1];
        v[i] = a * cs.x - bb * cs.y;
        v[i + 1] = a * cs.y + bb * cs.x;
      }
    }
    float* out = reinterpret_cast<float*>(kind == 0 ? dst.q : dst.k);
    const int nh = kind == 0 ? f.n_q : f.n_kv;
#pragma unroll
    for (int i = 0; i < E; ++i)
      out[((static_cast<size_t>(b) * nh + head) * f.L + l) * hd + lane * E + i] = v[i];
  } else if (kind == 2) {
    float* vt = reinterpret_cast<float*>(dst.vt);
#pragma unroll
    for (int i = 0; i < E; ++i)
      vt[((static_cast<size_t>(b) * f.n_kv + head) * hd + lane * E + i) * f.Lp + l] = v[i];
  } else {
    float* g = reinterpret_cast<float*>(dst.g);
#pragma unroll
    for (int i = 0; i < E; ++i) g[static_cast<size_t>(m) * f.n_q * hd + head * hd + lane * E + i] = sigmoidf_(v[i]);
  }
}

cudaError_t launch_qkvg_post_f32(const Fwd& f, const float* raw, QkvgDst dst, cudaStream_t st) {
  const int nseg = (f.gate_on ? 2 * f.n_q : f.n_q) + 2 * f.n_kv;
  const long long warps = static_cast<long long>(f.T) * nseg;
  const int grid = static_cast<int>((warps * 32 + 255) / 256);
  if (f.hd == 64)
    qkvg_post_f32_kernel<2><<<grid, 256, 0, st>>>(f, raw, dst);
  else
    qkvg_post_f32_kernel<4><<<grid, 256, 0, st>>>(f, raw, dst);
  return cudaGetLastError();
}

// ============================================================== SIMT attention (+ gate)
// One warp per (b, h, query row l). Lane owns E = hd/32 channels. Online softmax in the
// base-2 domain: p = 2^(s*log2e/sqrt(hd) - m).
template <class T, int E>
__global__ void __launch_bounds__(128) attn_simt_kernel(Fwd f, const T* __restrict__ q, const T* __restrict__ k,
                                                        const T* __restrict__ vt, const T* __restrict__ g,
                                                        T* __restrict__ og) {
  const int lane = threadIdx.x & 31;
  const int l = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int h = blockIdx.y, b = blockIdx.z;
  if (l >= f.L) return;
  const int hd = f.hd, G = f.n_q / f.n_kv, kvh = h / G;
  const float scale = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
  const T* qr = q + ((static_cast<size_t>(b) * f.n_q + h) * f.L + l) * hd + lane * E;
  float qv[E], acc[E];
#pragma unroll
  for (int i = 0; i < E; ++i) {
    qv[i] = Conv<T>::to_f(qr[i]) * scale;
    acc[i] = 0.f;
  }
  const T* kb = k + (static_cast<size_t>(b) * f.n_kv + kvh) * f.L * hd + lane * E;
  const T* vb = vt + ((static_cast<size_t>(b) * f.n_kv + kvh) * hd + lane * E) * f.Lp;
  float mx = -INFINITY, den = 0.f;
  for (int j = 0; j < f.L; ++j) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i) s = fmaf(qv[i], Conv<T>::to_f(kb[static_cast<size_t>(j) * hd + i]), s);
    s = warp_sum(s);
    const float mn = fmaxf(mx, s);
    const float corr = exp2f(mx - mn);
    const float p = exp2f(s - mn);
    den = den * corr + p;
#pragma unroll
    for (int i = 0; i < E; ++i) acc[i] = fmaf(p, Conv<T>::to_f(vb[static_cast<size_t>(i) * f.Lp + j]), acc[i] * corr);
    mx = mn;
  }
  const int m = b * f.L + l;
  const size_t o_off = static_cast<size_t>(m) * f.n_q * hd + h * hd + lane * E;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    float o = acc[i] / den;
    if (f.gate_on) o *= Conv<T>::to_f(g[o_off + i]);  // g holds the gate value
    og[o_off + i] = Conv<T>::from_f(o);
  }
}

cudaError_t launch_attn_simt(bool bf16_mode, const Fwd& f, const void* q, const void* k, const void* vt,
                             const void* g, void* og, cudaStream_t st) {
  dim3 grid((f.L + 3) / 4, f.n_q, f.B);
#define KD_ATTN(T, E)                                                                                       \
  attn_simt_kernel<T, E><<<grid, 128, 0, st>>>(f, reinterpret_cast<const T*>(q), reinterpret_cast<const T*>(k), \
                                               reinterpret_cast<const T*>(vt), reinterpret_cast<const T*>(g),   \
                                               reinterpret_cast<T*>(og))
  if (bf16_mode) {
    if (f.hd == 64) KD_ATTN(bf16, 2); else KD_ATTN(bf16, 4);
  } else {
    if (f.hd == 64) KD_ATTN(float, 2); else KD_ATTN(float, 4);
  }
#undef KD_ATTN
  return cudaGetLastError();
}

// ============================================================== fp32: gated residual, SwiGLU
__global__ void residual_f32_kernel(Fwd f, RowSrc res, const float* __restrict__ acc,
                                    const float* __restrict__ mod_shared, const float* __restrict__ mod_bias,
                                    int chunk_gate, float* __restrict__ out) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(f.T) * f.d) return;
  const int m = static_cast<int>(idx / f.d), c = static_cast<int>(idx % f.d);
  const int b = m / f.L;
  const float* x = row_src_ptr<float>(res, m, f.L, f.n_txt, f.n_img, f.d);
  const float gate = mod_shared[(static_cast<size_t>(b) * 6 + chunk_gate) * f.d + c] +
                     mod_bias[static_cast<size_t>(chunk_gate) * f.d + c];
  out[idx] = x[c] + gate * acc[idx];
}

cudaError_t launch_residual_f32(const Fwd& f, RowSrc res, const float* acc, const float* mod_shared,
                                const float* mod_bias, int chunk_gate, float* out, cudaStream_t st) {
  const size_t n = static_cast<size_t>(f.T) * f.d;
  residual_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(f, res, acc, mod_shared, mod_bias,
                                                                              chunk_gate, out);
  return cudaGetLastError();
}

__global__ void swiglu_f32_kernel(size_t n, const float* __restrict__ a, const float* __restrict__ u,
                                  float* __restrict__ hmid) {
  const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const float x = a[i];
  hmid[i] = x / (1.0f + expf(-x)) * u[i];
}

cudaError_t launch_swiglu_f32(const Fwd& f, const float* a, const float* u, float* hmid, cudaStream_t st) {
  const size_t n = static_cast<size_t>(f.T) * f.F;
  swiglu_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(n, a, u, hmid);
  return cudaGetLastError();
}

}  // namespace kd
