// CUDA-core kernels of the DiT block library.
//
//  * norm_modulate  (both modes): zero-centred RMSNorm + shift/scale modulation with the
//    per-block bias (Krea 2 Technical Report, "Normalisation" and "Timestep
//    conditioning"). HBM-bound: 16-byte vector loads/stores, fp32 math.
//  * temb_sinusoid  (both modes): the sinusoidal timestep embedding ("Timestep
//    conditioning"), argument and sin/cos in fp64 then rounded to fp32.
//  * fp32 check mode: a plain tiled fp32 GEMM, the QK-norm + RoPE scatter, the GQA
//    attention with the sigmoid gate ("Transformer block"), the gated residual and the
//    SwiGLU product, as separate simple kernels with fp32 arithmetic (no tensor cores).
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace kd {

// ============================================================== norm + modulate
// y = x / sqrt(mean(x^2) + eps) * (1 + w) * (1 + scale) + shift,
// scale/shift = mod_shared[b, chunk] + mod_bias[chunk].
//
// One warp per row: lane l holds columns 8(l + 32c) .. +7 for c < NV, so all of a row's
// 16-byte loads are in flight at once and the sum of squares is a warp reduction. A CTA
// owns a contiguous range of rows; the per-column factors A = (1 + w)(1 + scale) and
// S = shift of the batch elements it meets are computed once into shared memory (two
// sets, refreshed when the rows move to a batch element not in them).
template <class T>
__device__ __forceinline__ void store8(T* p, const float (&v)[8]);
template <>
__device__ __forceinline__ void store8<bf16>(bf16* p, const float (&v)[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                            pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

constexpr int NM_WARPS = 16;

// A row chunk of 8 values kept as loaded (packed bf16 or fp32) between the two passes.
template <class T>
struct Raw8;
template <>
struct Raw8<bf16> {
  uint4 u;
  __device__ __forceinline__ void load(const bf16* p) { u = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), e = unpack_bf16x2(u.w);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y; v[4] = c.x; v[5] = c.y; v[6] = e.x; v[7] = e.y;
  }
};
template <>
struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

template <class Tin, class Tout, int NV>
__global__ void __launch_bounds__(NM_WARPS * 32, 1) norm_modulate_kernel(
    Fwd f, RowSrc src, const float* __restrict__ gain_w, const float* __restrict__ mod_shared,
    const float* __restrict__ mod_bias, int chunk_shift, int chunk_scale, int rows_per_cta, Tout* __restrict__ out) {
  extern __shared__ float nm_smem[];  // [2 sets][A | S][d]
  __shared__ int set_b[2];
  const int d = f.d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * rows_per_cta;
  const int r1 = min(r0 + rows_per_cta, f.T);
  auto fill = [&](int set, int b) {  // A, S of batch element b into set (all threads)
    float* A = nm_smem + set * 2 * d;
    float* S = A + d;
    const float* sc_s = mod_shared + (static_cast<size_t>(b) * 6 + chunk_scale) * d;
    const float* sh_s = mod_shared + (static_cast<size_t>(b) * 6 + chunk_shift) * d;
    const float* sc_b = mod_bias + static_cast<size_t>(chunk_scale) * d;
    const float* sh_b = mod_bias + static_cast<size_t>(chunk_shift) * d;
    for (int c = threadIdx.x; c < d; c += blockDim.x) {
      A[c] = (1.0f + gain_w[c]) * (1.0f + (sc_s[c] + sc_b[c]));
      S[c] = sh_s[c] + sh_b[c];
    }
  };
  if (threadIdx.x == 0) {
    set_b[0] = -1;
    set_b[1] = -1;
  }
  __syncthreads();
  for (int g0 = r0; g0 < r1; g0 += NM_WARPS) {
    // batch elements of this group's rows: [g0 / L, (g1 - 1) / L]
    const int g1 = min(g0 + NM_WARPS, r1);
    const int blo = g0 / f.L, bhi = (g1 - 1) / f.L;
    if (set_b[0] != blo || (bhi != blo && set_b[1] != bhi)) {
      __syncthreads();  // every warp is done with the old sets
      if (set_b[0] != blo) fill(0, blo);
      if (bhi != blo && set_b[1] != bhi) fill(1, bhi);
      __syncthreads();
      if (threadIdx.x == 0) {
        set_b[0] = blo;
        if (bhi != blo) set_b[1] = bhi;
      }
      __syncthreads();
    }
    const int m = g0 + warp;
    if (m >= g1) continue;
    const int b = m / f.L;
    const Tin* x = row_src_ptr<Tin>(src, m, f.L, f.n_txt, f.n_img, d);
    Raw8<Tin> raw[NV];
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < NV; ++c) {
      const int col = (lane + 32 * c) * 8;
      if (col < d) raw[c].load(x + col);
      else raw[c].zero();
    }
#pragma unroll
    for (int c = 0; c < NV; ++c) {
      float v[8];
      raw[c].get(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
    }
    ss = warp_sum(ss);
    const float rstd = 1.0f / sqrtf(ss / static_cast<float>(d) + f.eps);
    const bool in_sets = b == set_b[0] || b == set_b[1];  // false only when L < 8 (a group spans 3+ batch elements)
    const float* A = nm_smem + (b == set_b[0] ? 0 : 2 * d);
    const float* S = A + d;
    Tout* y = out + static_cast<size_t>(m) * d;
#pragma unroll
    for (int c = 0; c < NV; ++c) {
      const int col = (lane + 32 * c) * 8;
      if (col < d) {
        float av[8], sv[8];
        if (in_sets) {
          const float4 a0 = *reinterpret_cast<const float4*>(A + col), a1 = *reinterpret_cast<const float4*>(A + col + 4);
          const float4 s0 = *reinterpret_cast<const float4*>(S + col), s1 = *reinterpret_cast<const float4*>(S + col + 4);
          av[0] = a0.x; av[1] = a0.y; av[2] = a0.z; av[3] = a0.w; av[4] = a1.x; av[5] = a1.y; av[6] = a1.z; av[7] = a1.w;
          sv[0] = s0.x; sv[1] = s0.y; sv[2] = s0.z; sv[3] = s0.w; sv[4] = s1.x; sv[5] = s1.y; sv[6] = s1.z; sv[7] = s1.w;
        } else {
          const float* sc_s = mod_shared + (static_cast<size_t>(b) * 6 + chunk_scale) * d;
          const float* sh_s = mod_shared + (static_cast<size_t>(b) * 6 + chunk_shift) * d;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            av[i] = (1.0f + gain_w[col + i]) * (1.0f + (sc_s[col + i] + mod_bias[chunk_scale * d + col + i]));
            sv[i] = sh_s[col + i] + mod_bias[chunk_shift * d + col + i];
          }
        }
        float v[8], o[8];
        raw[c].get(v);
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = fmaf(v[i] * rstd, av[i], sv[i]);
        store8<Tout>(y + col, o);
      }
    }
  }
}

template <class Tin, class Tout, int NV>
cudaError_t launch_nm(const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared, const float* mod_bias,
                      int chunk_shift, int chunk_scale, Tout* out, int num_sms, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(4) * f.d * sizeof(float);  // limit set by norm_init
  const int ctas = num_sms;  // one CTA (16 warps) per SM: the parameter fill is paid once per SM
  int rows = (f.T + ctas - 1) / ctas;
  rows = (rows + NM_WARPS - 1) / NM_WARPS * NM_WARPS;
  const int grid = (f.T + rows - 1) / rows;
  norm_modulate_kernel<Tin, Tout, NV><<<grid, NM_WARPS * 32, smem, st>>>(f, src, gain_w, mod_shared, mod_bias,
                                                                        chunk_shift, chunk_scale, rows, out);
  return cudaGetLastError();
}

template <class Tin, class Tout, int NV>
cudaError_t init_nm(int d) {
  return cudaFuncSetAttribute(norm_modulate_kernel<Tin, Tout, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              4 * d * static_cast<int>(sizeof(float)));
}

template <class Tin, class Tout>
cudaError_t init_nm_all(int d) {
  const int nv = (d / 8 + 31) / 32;
#define KD_NMI(N) \
  if (nv <= N) return init_nm<Tin, Tout, N>(d)
  KD_NMI(1);
  KD_NMI(2);
  KD_NMI(3);
  KD_NMI(4);
  KD_NMI(6);
  KD_NMI(8);
  KD_NMI(12);
  KD_NMI(16);
  KD_NMI(24);
  KD_NMI(32);
#undef KD_NMI
  return cudaErrorInvalidValue;
}

cudaError_t norm_init(int d) {
  cudaError_t e;
  if ((e = init_nm_all<bf16, bf16>(d)) != cudaSuccess) return e;
  if ((e = init_nm_all<float, bf16>(d)) != cudaSuccess) return e;
  return init_nm_all<float, float>(d);
}

template <class Tin, class Tout>
cudaError_t dispatch_nm(const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared, const float* mod_bias,
                        int chunk_shift, int chunk_scale, Tout* out, int num_sms, cudaStream_t st) {
  const int nv = (f.d / 8 + 31) / 32;  // 8-column chunks per lane
#define KD_NM(N) \
  if (nv <= N) return launch_nm<Tin, Tout, N>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, num_sms, st)
  KD_NM(1);
  KD_NM(2);
  KD_NM(3);
  KD_NM(4);
  KD_NM(6);
  KD_NM(8);
  KD_NM(12);
  KD_NM(16);
  KD_NM(24);
  KD_NM(32);
#undef KD_NM
  return cudaErrorInvalidValue;
}

cudaError_t launch_norm_modulate(NormIO io, const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared,
                                 const float* mod_bias, int chunk_shift, int chunk_scale, void* out, int num_sms,
                                 cudaStream_t st) {
  switch (io) {
    case NormIO::BF16_BF16:
      return dispatch_nm<bf16, bf16>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale,
                                     reinterpret_cast<bf16*>(out), num_sms, st);
    case NormIO::F32_BF16:
      return dispatch_nm<float, bf16>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale,
                                      reinterpret_cast<bf16*>(out), num_sms, st);
    case NormIO::F32_F32:
      return dispatch_nm<float, float>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale,
                                       reinterpret_cast<float*>(out), num_sms, st);
  }
  return cudaErrorInvalidValue;
}

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
    for (int i = 0; i < E; ++i) g[static_cast<size_t>(m) * f.n_q * hd + head * hd + lane * E + i] = v[i];
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
    if (f.gate_on) o *= sigmoidf_(Conv<T>::to_f(g[o_off + i]));
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
