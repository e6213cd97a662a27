// Norm + modulate kernel of the DiT block library (all modes): zero-centred RMSNorm +
// shift/scale modulation with the per-block bias (Krea 2 Technical Report, "Normalisation"
// and "Timestep conditioning"), optionally with an e4m3 output for an 8-bit GEMM.
// HBM-bound: 16-byte vector loads/stores, fp32 math.
#include <math.h>

#include <type_traits>

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

// Shared-memory order of the per-column factors: within each 256-column chunk, the lane
// that owns columns 8l .. 8l+7 finds the first four at 4l and the last four at 128 + 4l,
// so that a warp's 16-byte reads of either half are 512 contiguous bytes (no bank
// conflicts; in column order the 32-byte stride between lanes made every read two-way).
__host__ __device__ __forceinline__ int nm_pos(int col) {
  const int r = col & 255;
  return (col & ~255) + ((r & 4) << 5) + ((r >> 3) << 2) + (r & 3);
}
__host__ __device__ __forceinline__ int nm_padded(int d) { return (d + 255) / 256 * 256; }

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

// QM = output mode (NormQ): 0 plain store of Tout; 1 e4m3 codes with one power-of-two
// scale per row; 2 row amax only; 3 e4m3 codes with one scale for the whole tensor, from
// the row amax of a preceding mode-2 pass; 4 plain store plus the row's amax (of the
// stored bf16 values), for a cast that follows. The e4m3 modes cast the row as a bf16 store
// would keep it ("训练 › 预训练" / Training › Pretraining: 8-bit GEMM operands).
template <class Tin, class Tout, int NV, int QM>
__global__ void __launch_bounds__(NM_WARPS * 32, 1) norm_modulate_kernel(
    Fwd f, RowSrc src, const float* __restrict__ gain_w, const float* __restrict__ mod_shared,
    const float* __restrict__ mod_bias, int chunk_shift, int chunk_scale, int rows_per_cta, Tout* __restrict__ out,
    uint8_t* __restrict__ q8, float* __restrict__ dq, float* __restrict__ rowamax) {
  extern __shared__ float nm_smem[];  // [2 sets][A | S][dp], in nm_pos order
  __shared__ int set_b[2];
  __shared__ float red[NM_WARPS];
  __shared__ float tensor_scale;
  const int d = f.d, dp = nm_padded(d);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r0 = blockIdx.x * rows_per_cta;
  const int r1 = min(r0 + rows_per_cta, f.T);
  auto fill = [&](int set, int b) {  // A, S of batch element b into set (all threads)
    float* A = nm_smem + set * 2 * dp;
    float* S = A + dp;
    const float* sc_s = mod_shared + (static_cast<size_t>(b) * 6 + chunk_scale) * d;
    const float* sh_s = mod_shared + (static_cast<size_t>(b) * 6 + chunk_shift) * d;
    const float* sc_b = mod_bias + static_cast<size_t>(chunk_scale) * d;
    const float* sh_b = mod_bias + static_cast<size_t>(chunk_shift) * d;
    // four columns per thread per pass, so that their twenty loads are in flight together
    for (int c0 = threadIdx.x; c0 < d; c0 += 4 * blockDim.x) {
      float g[4], ss_[4], sb_[4], hs[4], hb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + k * blockDim.x;
        const bool in = c < d;
        g[k] = in ? gain_w[c] : 0.f;
        ss_[k] = in ? sc_s[c] : 0.f;
        sb_[k] = in ? sc_b[c] : 0.f;
        hs[k] = in ? sh_s[c] : 0.f;
        hb[k] = in ? sh_b[c] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = c0 + k * blockDim.x;
        if (c < d) {
          A[nm_pos(c)] = (1.0f + g[k]) * (1.0f + (ss_[k] + sb_[k]));
          S[nm_pos(c)] = hs[k] + hb[k];
        }
      }
    }
  };
  if (threadIdx.x == 0) {
    set_b[0] = -1;
    set_b[1] = -1;
  }
  if constexpr (QM == 3) {  // the tensor's scale from every row's amax
    float m = 0.0f;
    for (int i = threadIdx.x; i < f.T; i += blockDim.x) m = fmaxf(m, rowamax[i]);
    m = warp_max(m);
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.0f;
      for (int w = 0; w < NM_WARPS; ++w) t = fmaxf(t, red[w]);
      const int k = e4m3_scale_exp(t);
      tensor_scale = pow2f(k);
      if (blockIdx.x == 0) dq[0] = pow2f(-k);
    }
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
#pragma unroll
    for (int c = 0; c < NV; ++c) {
      const int col = (lane + 32 * c) * 8;
      if (col < d) raw[c].load(x + col);
      else raw[c].zero();
    }
    float ss4[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains
#pragma unroll
    for (int c = 0; c < NV; ++c) {
      float v[8];
      raw[c].get(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss4[i & 3] = fmaf(v[i], v[i], ss4[i & 3]);
    }
    const float ss = warp_sum((ss4[0] + ss4[1]) + (ss4[2] + ss4[3]));
    const float rstd = 1.0f / sqrtf(ss / static_cast<float>(d) + f.eps);
    const bool in_sets = b == set_b[0] || b == set_b[1];  // false only when L < 8 (a group spans 3+ batch elements)
    const float* A = nm_smem + (b == set_b[0] ? 0 : 2 * dp);
    const float* S = A + dp;
    // the 8 outputs of chunk c (columns col .. col+7) in fp32
    auto chunk_out = [&](int c, int col, float (&o)[8]) {
      float av[8], sv[8];
      if (in_sets) {
        const int p = nm_pos(col);  // columns col .. col+3 at p, col+4 .. col+7 at p + 128
        const float4 a0 = *reinterpret_cast<const float4*>(A + p), a1 = *reinterpret_cast<const float4*>(A + p + 128);
        const float4 s0 = *reinterpret_cast<const float4*>(S + p), s1 = *reinterpret_cast<const float4*>(S + p + 128);
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
      float v[8];
      raw[c].get(v);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = fmaf(v[i] * rstd, av[i], sv[i]);
    };
    if constexpr (QM == 0 || QM == 4) {
      Tout* y = out + static_cast<size_t>(m) * d;
      float amax = 0.0f;
#pragma unroll
      for (int c = 0; c < NV; ++c) {
        const int col = (lane + 32 * c) * 8;
        if (col < d) {
          float o[8];
          chunk_out(c, col, o);
          store8<Tout>(y + col, o);
          if constexpr (QM == 4) {
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(o[i]));
          }
        }
      }
      if constexpr (QM == 4) {
        amax = round_bf16(warp_max(amax));  // the largest magnitude of the stored row
        if (lane == 0) rowamax[m] = amax;
      }
    } else {
      float scale;
      if constexpr (QM == 3) {
        scale = tensor_scale;
      } else {
        float amax = 0.0f;
#pragma unroll
        for (int c = 0; c < NV; ++c) {
          const int col = (lane + 32 * c) * 8;
          if (col < d) {
            float o[8];
            chunk_out(c, col, o);
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(o[i]));
          }
        }
        amax = round_bf16(warp_max(amax));  // the largest magnitude a bf16 store keeps
        if constexpr (QM == 2) {
          if (lane == 0) rowamax[m] = amax;
          continue;
        }
        const int k = e4m3_scale_exp(amax);
        scale = pow2f(k);
        if (lane == 0) dq[m] = pow2f(-k);
      }
      uint8_t* y8 = q8 + static_cast<size_t>(m) * d;
#pragma unroll
      for (int c = 0; c < NV; ++c) {
        const int col = (lane + 32 * c) * 8;
        if (col < d) {
          float o[8];
          chunk_out(c, col, o);
#pragma unroll
          for (int i = 0; i < 8; ++i) o[i] = round_bf16(o[i]) * scale;
          *reinterpret_cast<uint2*>(y8 + col) = cvt_e4m3x8(o);
        }
      }
    }
  }
}

template <class Tin, class Tout, int NV, int QM>
cudaError_t launch_nm(const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared, const float* mod_bias,
                      int chunk_shift, int chunk_scale, Tout* out, const NormQOut& q, int num_sms, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(4) * nm_padded(f.d) * sizeof(float);  // limit set by norm_init
  const int ctas = num_sms;  // one CTA (16 warps) per SM: the parameter fill is paid once per SM
  int rows = (f.T + ctas - 1) / ctas;
  rows = (rows + NM_WARPS - 1) / NM_WARPS * NM_WARPS;
  const int grid = (f.T + rows - 1) / rows;
  norm_modulate_kernel<Tin, Tout, NV, QM><<<grid, NM_WARPS * 32, smem, st>>>(
      f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, rows, out, reinterpret_cast<uint8_t*>(q.q8),
      q.dq, q.rowamax);
  return cudaGetLastError();
}

template <class Tin, class Tout, int NV, int QM>
cudaError_t init_nm(int d) {
  return cudaFuncSetAttribute(norm_modulate_kernel<Tin, Tout, NV, QM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              4 * nm_padded(d) * static_cast<int>(sizeof(float)));
}

// The e4m3 output modes exist for bf16 outputs and rows of up to NM_Q_MAX_NV * 256 columns.
constexpr int NM_Q_MAX_NV = 12;

template <class Tin, class Tout, int NV>
cudaError_t init_nm_modes(int d) {
  cudaError_t e = init_nm<Tin, Tout, NV, 0>(d);
  if constexpr (std::is_same<Tout, bf16>::value && NV <= NM_Q_MAX_NV) {
    if (e != cudaSuccess) return e;
    if ((e = init_nm<Tin, Tout, NV, 1>(d)) != cudaSuccess) return e;
    if ((e = init_nm<Tin, Tout, NV, 2>(d)) != cudaSuccess) return e;
    if ((e = init_nm<Tin, Tout, NV, 3>(d)) != cudaSuccess) return e;
    return init_nm<Tin, Tout, NV, 4>(d);
  }
  return e;
}

template <class Tin, class Tout>
cudaError_t init_nm_all(int d) {
  const int nv = (d / 8 + 31) / 32;
#define KD_NMI(N) \
  if (nv <= N) return init_nm_modes<Tin, Tout, N>(d)
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

template <class Tin, class Tout, int NV>
cudaError_t launch_nm_mode(const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared,
                           const float* mod_bias, int chunk_shift, int chunk_scale, Tout* out, const NormQOut& q,
                           int num_sms, cudaStream_t st) {
  if constexpr (std::is_same<Tout, bf16>::value && NV <= NM_Q_MAX_NV) {
    switch (q.mode) {
      case NormQ::NONE:
        break;
      case NormQ::ROW:
        return launch_nm<Tin, Tout, NV, 1>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, q,
                                           num_sms, st);
      case NormQ::AMAX:
        return launch_nm<Tin, Tout, NV, 2>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, q,
                                           num_sms, st);
      case NormQ::TENSOR:
        return launch_nm<Tin, Tout, NV, 3>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, q,
                                           num_sms, st);
      case NormQ::STORE_AMAX:
        return launch_nm<Tin, Tout, NV, 4>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, q,
                                           num_sms, st);
    }
  } else {
    if (q.mode != NormQ::NONE) return cudaErrorInvalidValue;
  }
  return launch_nm<Tin, Tout, NV, 0>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, q, num_sms,
                                     st);
}

template <class Tin, class Tout>
cudaError_t dispatch_nm(const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared, const float* mod_bias,
                        int chunk_shift, int chunk_scale, Tout* out, const NormQOut& q, int num_sms,
                        cudaStream_t st) {
  const int nv = (f.d / 8 + 31) / 32;  // 8-column chunks per lane
#define KD_NM(N)                                                                                                 \
  if (nv <= N)                                                                                                   \
  return launch_nm_mode<Tin, Tout, N>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale, out, q, \
                                      num_sms, st)
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
                                 cudaStream_t st, const NormQOut* q8) {
  const NormQOut q = q8 ? *q8 : NormQOut{NormQ::NONE, nullptr, nullptr, nullptr};
  switch (io) {
    case NormIO::BF16_BF16:
      return dispatch_nm<bf16, bf16>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale,
                                     reinterpret_cast<bf16*>(out), q, num_sms, st);
    case NormIO::F32_BF16:
      return dispatch_nm<float, bf16>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale,
                                      reinterpret_cast<bf16*>(out), q, num_sms, st);
    case NormIO::F32_F32:
      return dispatch_nm<float, float>(f, src, gain_w, mod_shared, mod_bias, chunk_shift, chunk_scale,
                                       reinterpret_cast<float*>(out), q, num_sms, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kd
