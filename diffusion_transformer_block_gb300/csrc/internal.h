// Internal launcher interface between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kd {

// Shape of one forward call plus the block hyper-parameters.
struct Fwd {
  int B, L, n_txt, n_img, img_w, T, Lp;  // T = B*L joint rows, Lp = L rounded up to 64
  int d, n_q, n_kv, hd, F, gate_on;
  float eps;
};

// Where row m (joint order, m = b*L + l) of a block input lives: the split caller
// buffers (text rows l < n_txt, image rows after) or one joint [T, d] buffer.
struct RowSrc {
  const void* x_txt;  // [B, n_txt, d]
  const void* x_img;  // [B, n_img, d]
  const void* joint;  // [T, d]; used when non-null
};

// Destination buffers of the fused QKV+gate projection.
struct QkvgDst {
  void* q;   // [B, n_q, L, hd]
  void* k;   // [B, n_kv, L, hd]
  void* vt;  // [B, n_kv, hd, Lp]
  void* g;   // [T, n_q*hd]
  const float* q_norm_w;
  const float* k_norm_w;
  const float2* rope;  // [pos][hd/4] (cos, sin)
  float* raw = nullptr;  // optional [T, ldr] fp32: the Q and K columns of the projection
  int ldr = 0;           // before the norm (for the backward)
};

// Dequantisation factors of an 8-bit GEMM (powers of two): row m, column n of the
// product is scaled by a[m] * b[n] (per_row) or a[0] * b[0] (per tensor).
struct Deq {
  const float* a;   // A (activation) factors: [M] or [1]
  const float* b;   // B (weight) factors: [N] or [1]
  const float* b2;  // second B of the SwiGLU GEMM (W_up)
  int per_row;
};

#ifdef __CUDACC__
// Pointer to row m of a block input (see RowSrc).
template <class T>
__device__ __forceinline__ const T* row_src_ptr(const RowSrc& s, int m, int L, int n_txt, int n_img, int d) {
  if (s.joint) return reinterpret_cast<const T*>(s.joint) + static_cast<size_t>(m) * d;
  const int b = m / L, l = m - b * L;
  if (l < n_txt) return reinterpret_cast<const T*>(s.x_txt) + (static_cast<size_t>(b) * n_txt + l) * d;
  return reinterpret_cast<const T*>(s.x_img) + (static_cast<size_t>(b) * n_img + (l - n_txt)) * d;
}
#endif

// ---- kernels_simt.cu (both modes: norm; fp32 mode: everything else) ----
// sets the norm kernels' shared-memory limit for width d (once per handle, before capture)
cudaError_t norm_init(int d);
// input -> output storage types of a norm+modulate launch
enum class NormIO { BF16_BF16, F32_BF16, F32_F32 };
// e4m3 output of a norm+modulate launch (the bf16-rounded row cast to e4m3):
//   NONE   : plain output (`out`, type from NormIO)
//   ROW    : row-wise scaled codes -> q8 [T, d], dq [T]
//   AMAX   : no output; rowamax[m] = largest |bf16 row value|
//   TENSOR : codes with one scale from max(rowamax[0..T)) -> q8, dq [1]
enum class NormQ { NONE, ROW, AMAX, TENSOR, STORE_AMAX };
struct NormQOut {
  NormQ mode;
  void* q8;
  float* dq;
  float* rowamax;
};
// requires d % 8 == 0 and d <= 8192 (a warp holds a row in registers); e4m3 modes need
// NormIO::BF16_BF16 or F32_BF16 (the row is rounded to bf16 before the cast) and d <= 3072
cudaError_t launch_norm_modulate(NormIO io, const Fwd& f, RowSrc src, const float* gain_w, const float* mod_shared,
                                 const float* mod_bias, int chunk_shift, int chunk_scale, void* out, int num_sms,
                                 cudaStream_t st, const NormQOut* q8 = nullptr);
cudaError_t launch_temb_sinusoid(const float* t, int B, float* e, cudaStream_t st);
// C[M,N] = act(A[M,K] * W[N,K]^T + bias), fp32, act = 1 -> silu
cudaError_t launch_gemm_simt_f32(const float* A, const float* W, float* C, int M, int N, int K, const float* bias,
                                 int act, cudaStream_t st);
// fp32 mode: raw [T, Nqkvg] -> QK-norm + RoPE + scatter
cudaError_t launch_qkvg_post_f32(const Fwd& f, const float* raw, QkvgDst dst, cudaStream_t st);
// attention with gate epilogue, SIMT, both dtypes (bf16: stand-in until the tensor-core kernel)
cudaError_t launch_attn_simt(bool bf16, const Fwd& f, const void* q, const void* k, const void* vt, const void* g,
                             void* og, cudaStream_t st);
// fp32 mode: out = res + gate_chunk * acc
cudaError_t launch_residual_f32(const Fwd& f, RowSrc res, const float* acc, const float* mod_shared,
                                const float* mod_bias, int chunk_gate, float* out, cudaStream_t st);
// fp32 mode: hmid = silu(a) * u
cudaError_t launch_swiglu_f32(const Fwd& f, const float* a, const float* u, float* hmid, cudaStream_t st);

// ---- gemm_tc.cu (bf16 and e4m3 operands, tcgen05 + TMA) ----
// Every launcher takes `dq`: nullptr = bf16 operands (tensor maps of bf16), otherwise
// e4m3 operands (tensor maps of bytes) whose products are dequantised by dq.
int gemm_tc_smem_bytes();
// sets the kernels' dynamic shared-memory limit and queries co-resident CTA pairs (once per
// handle, before any stream capture)
cudaError_t gemm_tc_init(int num_sms);
// xn[T,d] x W_qkvg^T -> QK-norm, RoPE, scatter to Q / K / V^T / G
cudaError_t launch_gemm_qkvg(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int N,
                             const QkvgDst& dst, const Deq* dq, int num_sms, int* err, cudaStream_t st);
// h1[T,d] (fp32) = x (bf16, split buffers) + gate_a * (A W^T), stored through tm_h1 (fp32
// [T, d], box 32 x 32, 128-byte swizzle); pre (optional, bf16 mode, fp32 [T,d]) gets A W^T
cudaError_t launch_gemm_resid_attn(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K, RowSrc x,
                                   const float* mod_shared, const float* mod_bias, const CUtensorMap* tm_h1,
                                   const Deq* dq, float* pre, int num_sms, int* err, cudaStream_t st);
// out[T,d] (bf16) = h1 (fp32) + gate_m * (A W^T), stored through tm_out (bf16 [T, d], box
// 64 x 32, 128-byte swizzle); pre as above
cudaError_t launch_gemm_resid_mlp(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K,
                                  const float* h1, const float* mod_shared, const float* mod_bias,
                                  const CUtensorMap* tm_out, const Deq* dq, float* pre, int num_sms, int* err,
                                  cudaStream_t st);
// hmid[T,F] = silu(hn W_gate^T) * (hn W_up^T); rowamax (optional, pre-zeroed [T]) gets
// each row's largest |hmid| as stored (bf16); pre_a / pre_u (optional, bf16 mode, fp32
// [T,F]) get the two products
cudaError_t launch_gemm_swiglu(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_gate,
                               const CUtensorMap* tm_up, void* hmid, float* rowamax, const Deq* dq, float* pre_a,
                               float* pre_u, int num_sms, int* err, cudaStream_t st);

// the output-gate backward and the softmax row term in the epilogue of d_og = A[T,K] W_o^T
// (B = W_o^T as a K-major [n_q*128, K] map): d_o (bf16, head-major [B, n_q, L, 128]), the
// gate's gradient into d_P columns goff.. (bf16, row pitch ldp), D = rowsum(d_o o) per head
// ([B, n_q, Lp]); o fp32 [T, n_q*128], g bf16 [T, n_q*128]
cudaError_t launch_gemm_gate_bwd(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K, const float* o,
                                 const void* g, void* d_o, void* d_P, int ldp, int goff, float* D, int num_sms,
                                 int* err, cudaStream_t st);
// d_au [M, 2F] (bf16) = SwiGLU backward of d_hmid = A[M,K] B[F,K]^T with the forward's
// fp32 pre-activations a, u [M, F]: d_a = d_hmid u silu'(a), d_u = d_hmid silu(a) (F % 8 == 0)
cudaError_t launch_gemm_swiglu_bwd(const CUtensorMap* tm_a, const CUtensorMap* tm_b, int M, int F, int K,
                                   const float* a, const float* u, void* d_au, int num_sms, int* err,
                                   cudaStream_t st);
// C[M,N] (fp32, row pitch ldc % 4 == 0) = alpha * A[M,K] B[N,K]^T (+ C if accumulate);
// A and B bf16 K-major tensor maps (box 64 x 128)
cudaError_t launch_gemm_plain(const CUtensorMap* tm_a, const CUtensorMap* tm_b, int M, int N, int K, float* C,
                              long long ldc, float alpha, int accumulate, int num_sms, int* err, cudaStream_t st);

// ---- attn_tc.cu (bf16 mode, tcgen05 + TMA) ----
cudaError_t attn_tc_init();
// og = softmax(q k^T / sqrt(hd)) v * s with s = sigmoid(xn W_g^T) as stored by the QKV+G
// projection; s is read through tm_g and og written
// through tm_og, both 3D bf16 maps over [B, L, n_q*hd] with the 128-byte swizzle (box 64 x
// 128 rows for g, 64 x 32 rows for og; tm_g unused without the gate); rowamax (optional,
// pre-zeroed [T]) gets each row's largest |og| as stored (bf16)
// lse (optional, [B, n_q, Lp]: row pitch Lp) gets m + log2(l) per row in the scores'
// scaled-log2 units, o_raw (optional, fp32 [T, n_q*hd]) the output before the gate; both
// for the backward
cudaError_t launch_attn_tc(const Fwd& f, const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_vt,
                           const CUtensorMap* tm_g, const CUtensorMap* tm_og, float* rowamax, float* lse, float* o_raw,
                           int num_sms, int* err, cudaStream_t st);

// ---- attn_bwd.cu (flash-style attention backward, tcgen05 + TMA) ----
cudaError_t attn_bwd_init();
// dq [B n_q, L, hd], dk and dv [B n_kv, L, hd] (fp32) from d_o (head-major bf16, the
// gradient of the ungated output), the forward's lse and D = rowsum(d_o o) (both
// [B n_q, Lp]). Maps (bf16, 128 x 64 boxes, 128-byte swizzle): tm_q / tm_do over
// [B n_q, L, hd], tm_k / tm_v over [B n_kv, L, hd] (row-major V), tm_qt / tm_dot over
// [B n_q, hd, L] (pitch Lp), tm_kt over [B n_kv, hd, L] (pitch Lp). Two launches.
cudaError_t launch_attn_bwd(const Fwd& f, const CUtensorMap* tm_q, const CUtensorMap* tm_do, const CUtensorMap* tm_k,
                            const CUtensorMap* tm_v, const CUtensorMap* tm_qt, const CUtensorMap* tm_dot,
                            const CUtensorMap* tm_kt, const float* lse, const float* D, float* dq, float* dk,
                            float* dv, int* err, cudaStream_t st);

// ---- quant8.cu (e4m3 casts of GEMM operands) ----
// Scaled e4m3 cast of a bf16 matrix src [R, K] (K % 16 == 0) into codes q [R, K]:
// per_row: row r uses rowamax[r], per tensor: the largest rowamax over all rows. dq gets
// the dequantisation factors 2^-k ([R] or [1]).
cudaError_t launch_quant_e4m3(const void* src, int R, int K, const float* rowamax, int per_row, void* q, float* dq,
                              int num_sms, cudaStream_t st);
// rowamax[r] = max_k |src[r, k]| of a bf16 matrix [R, K] (K % 8 == 0)
cudaError_t launch_row_amax(const void* src, int R, int K, float* rowamax, int num_sms, cudaStream_t st);

// ---- backward.cu (block backward: transposes, elementwise and reduction steps) ----
// dst[z][c, r] = src[z][r, c] (bf16), r < R; columns R .. Rp-1 of dst are zeroed
cudaError_t launch_transpose_bf16(const void* src, int R, int C, long long lds, long long src_bs, void* dst, int Rp,
                                  long long ldd, long long dst_bs, int batch, cudaStream_t st);
// y = res + gate_chunk * f: d_f = dy * gate (bf16 [T, d]); sum_l dy f -> d_mod[b, chunk], d_bias[chunk]
cudaError_t launch_gated_bwd(const Fwd& f, const void* dy, int dy_f32, const float* fv, const float* mod_shared,
                             const float* mod_bias, int chunk, void* d_f, float* d_mod, float* d_bias, cudaStream_t st);
// norm + modulation backward: dx (fp32 joint, or bf16 into the split buffers of dx_bf16)
// = d_res + RMSNorm gradient of dy (1 + w)(1 + scale); column sums into d_mod / d_bias / d_gain
cudaError_t launch_norm_bwd(const Fwd& f, RowSrc xs, int x_f32, const float* dy, const float* gain_w,
                            const float* mod_shared, const float* mod_bias, int chunk_shift, int chunk_scale,
                            const void* d_res, int res_f32, float* dx_f32, RowSrc dx_bf16, float* rstd,
                            float* d_mod, float* d_bias, float* d_gain, cudaStream_t st);
// QK-norm + RoPE backward and the V gradient into d_P (bf16); gain gradients into d_qw / d_kw
cudaError_t launch_qkv_bwd(const Fwd& f, const float* raw, int ldr, const float* dq, const float* dk, const float* dv,
                           const float* q_norm_w, const float* k_norm_w, const float2* rope, void* d_P, int ldp,
                           float* d_qw, float* d_kw, cudaStream_t st);

// ---- NVFP4 (quant4.cu casts, gemm_tc.cu GEMMs) ----
// one NVFP4 GEMM operand: a byte tensor map over its E2M1 codes ([rows, K/2], 128-byte
// boxes, 128-byte swizzle) and its scale atoms (see quant4.cu)
struct Op4 {
  const CUtensorMap* map;
  const uint8_t* sf;
};
// bytes of the scale atoms of a [rows, cols] operand (rows padded to 128)
size_t nvfp4_scale_bytes(long long rows, long long cols);
// codes / scale atoms of a bf16 [R, K] operand (K % 64 == 0); the tensor scale comes from
// rowamax[0..R) (reduced by every CTA) and is stored to ts[0]
cudaError_t launch_nvfp4_cast(const void* src, int R, int K, const float* rowamax, float* ts, void* codes, void* sf,
                              int num_sms, cudaStream_t st);
// sets the NVFP4 GEMM kernels' shared-memory limits (once per handle, before any capture)
cudaError_t gemm_fp4_init();
cudaError_t launch_gemm_qkvg_fp4(const Fwd& f, const Op4& a, const Op4& b, int N, const QkvgDst& dst, const Deq& dq,
                                 int num_sms, int* err, cudaStream_t st);
cudaError_t launch_gemm_resid_attn_fp4(const Fwd& f, const Op4& a, const Op4& b, int K, RowSrc x,
                                       const float* mod_shared, const float* mod_bias, const CUtensorMap* tm_h1,
                                       const Deq& dq, int num_sms, int* err, cudaStream_t st);
cudaError_t launch_gemm_resid_mlp_fp4(const Fwd& f, const Op4& a, const Op4& b, int K, const float* h1,
                                      const float* mod_shared, const float* mod_bias, const CUtensorMap* tm_out,
                                      const Deq& dq, int num_sms, int* err, cudaStream_t st);
cudaError_t launch_gemm_swiglu_fp4(const Fwd& f, const Op4& a, const Op4& gate, const Op4& up, void* hmid,
                                   float* rowamax, const Deq& dq, int num_sms, int* err, cudaStream_t st);

// ---- selftest.cu ----
// one CTA per SM waits (bounded by limit_ns) on an mbarrier nothing arrives at, records
// `site` in *err, frees its tensor memory and returns
cudaError_t launch_wait_selftest(int* err, int site, unsigned long long limit_ns, int num_sms, cudaStream_t st);

}  // namespace kd
