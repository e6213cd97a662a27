// Tensor-core GEMMs of the DiT block (bf16 or scaled e4m3 in, fp32 accumulate), tcgen05 +
// TMA, sm_103a.
//
// One persistent, warp-specialised kernel template with three fused epilogues:
//   * QKVG  : xn W_qkvg^T -> per-head QK-RMSNorm, 2D axial RoPE, scatter to Q, K, V^T, G
//             (Krea 2 Technical Report, "Transformer block", "Positional encoding",
//             "Normalisation")
//   * RESID : out = res + gate * (A W^T)   -- attention output projection and the MLP
//             down projection, each with its gated residual ("Residual design",
//             "Timestep conditioning"); the residual stream between them is fp32
//   * SWIGLU: silu(hn W_gate^T) * (hn W_up^T), both products in one 128x256 accumulator
//             ("Transformer block": SwiGLU MLP)
//
// CTAs run in clusters of two; the pair computes one 256 x 256 output tile (m-blocks 2p and
// 2p + 1 of one N-block) with pair MMAs (tcgen05 cta_group::2, M = 256, N = 256): each CTA
// holds its 128 rows of A and one 128-row half of the B tile, and receives its 128 rows of
// the accumulator in its own tensor memory. A k-step is 128-byte operand rows (64 bf16 or
// 128 e4m3 of K): 16 KB of A + 16 KB of B per CTA per stage, 6 stages in shared memory
// written by TMA with the 128-byte swizzle; one stage is four MMAs of 32 bytes of K
// (kind::f16, K = 16, or kind::f8f6f4, K = 32), issued by one thread of the even CTA. The 8-bit GEMMs ("训练 › 预训练" / Training › Pretraining: 8-bit
// training with tensor-wise or row-wise scaling) multiply e4m3 codes and dequantise each
// accumulator by the power-of-two factors of its row and column in the epilogue. The accumulator is double-buffered in TMEM
// (2 x 256 columns), so the epilogue of one tile overlaps the main loop of the next.
// Warp roles: warp 0 = TMA producer (one thread), warp 1 = TMEM allocator + MMA issuer
// (one thread), warps 2..9 = epilogue (two warpgroups, one per 128-column half).
//
// Both CTAs' TMA loads of a stage complete on the even CTA's "full" barrier (one expected
// byte count for the pair), the MMA commit frees the stage in both CTAs, each accumulator
// is announced to both CTAs' epilogues, and both CTAs' epilogue warps release it on the
// even CTA's barrier. Against one CTA per tile (the pair sharing B by multicast), a stage
// takes 32 KB of shared memory instead of 48 KB, so six stages fit instead of four and
// cover half as much again of the L2 latency.
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace kd {
namespace {

#ifndef KD_GEMM_STAGES
#define KD_GEMM_STAGES 6
#endif
constexpr int BM = 128, BN = 256, BK_BYTES = 128, STAGES = KD_GEMM_STAGES;
constexpr int A_BYTES = BM * BK_BYTES;             // this CTA's 128 rows of A
constexpr int BH_BYTES = (BN / 2) * BK_BYTES;      // this CTA's 128-row half of the B tile
constexpr int STAGE_BYTES = A_BYTES + BH_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + NUM_EPI_WARPS * 32;
// shared-memory staging per epilogue warp (epilogues that store through TMA declare kStgBytes)
template <class E, class = void>
struct StgOf {
  static constexpr int value = 0;
};
template <class E>
struct StgOf<E, std::void_t<decltype(E::kStgBytes)>> {
  static constexpr int value = E::kStgBytes;
};
template <class Epi>
constexpr int smem_bytes() {
  return STAGES * STAGE_BYTES + NUM_EPI_WARPS * StgOf<Epi>::value + 1024 /*alignment slack*/ + 256 /*barriers*/;
}
// Tile raster. Tiles are ordered in groups of `group` m-block pairs: within a group the
// m-pairs vary fastest, then the n-blocks (tile t of a group -> m-pair t % group, n-block
// t / group). group = 1 is n-fastest order, group >= the m-pairs of the call is m-fastest
// order over all of M. See raster_group for the choice.
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int group, int& mb, int& nb) {
  const int per_group = group * num_n;
  const int g = tile / per_group;
  const int first_m = g * group;
  const int gsize = min(num_m - first_m, group);
  const int r = tile - g * per_group;
  mb = first_m + r % gsize;
  nb = r / gsize;
}

// Wait used while tearing down: ignores the abort flag, still bounded.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err, int site) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, site);
      return;
    }
  }
}

__device__ __forceinline__ float u2f(uint32_t u) { return __uint_as_float(u); }

// Dequantise 32 accumulator columns col .. col+31 of one row (8-bit GEMMs only):
// fa = the row's factor, bp = the column factors. Products of powers of two: exact.
template <bool S8>
__device__ __forceinline__ void deq32(uint32_t (&r)[32], const Deq& dq, float fa, const float* bp, int col) {
  if constexpr (S8) {
    if (dq.per_row) {
      const float4* b4 = reinterpret_cast<const float4*>(bp + col);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 b = __ldg(b4 + q);
        r[4 * q + 0] = __float_as_uint(u2f(r[4 * q + 0]) * (fa * b.x));
        r[4 * q + 1] = __float_as_uint(u2f(r[4 * q + 1]) * (fa * b.y));
        r[4 * q + 2] = __float_as_uint(u2f(r[4 * q + 2]) * (fa * b.z));
        r[4 * q + 3] = __float_as_uint(u2f(r[4 * q + 3]) * (fa * b.w));
      }
    } else {
      const float s = fa * __ldg(bp);
#pragma unroll
      for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(u2f(r[i]) * s);
    }
  }
}
// the row's factor (0 for rows past M, whose results are discarded)
template <bool S8>
__device__ __forceinline__ float deq_row(const Deq& dq, int row, bool ok) {
  if constexpr (S8) return ok ? __ldg(dq.a + (dq.per_row ? row : 0)) : 0.0f;
  return 1.0f;
}

// ------------------------------------------------------------------ epilogues
// apply(): called by one epilogue warp for its 32 rows (one per lane) and one 128-column
// half of the 256-column accumulator. `taddr` = TMEM address of the lane's row at
// accumulator column 0. TMEM loads are warp-collective; stores are masked by row < M.
//
// The QKV+G, residual and SwiGLU epilogues read their warp's 128 accumulator columns
// through a source, in their own logical order (logical columns [0, 64) at lo, [64, 128)
// at hi): TmemAcc loads each 32-column chunk from tensor memory when it is needed (chunk
// loops rolled); RegAcc reads the chunks from registers that the whole share was copied
// into beforehand (chunk loops unrolled, so every register index is a constant), which
// lets a kernel hand the accumulator back to its MMAs before the epilogue's work.
struct TmemAcc {
  static constexpr int kUnroll = 1;
  uint32_t lo, hi;
  __device__ __forceinline__ uint32_t at(int l) const { return l < 64 ? lo + l : hi + (l - 64); }
  __device__ __forceinline__ void ld32(int l, uint32_t (&r)[32]) const { tmem_ld32(at(l), r); }
  __device__ __forceinline__ void ld32x2(int l1, int l2, uint32_t (&r)[32], uint32_t (&q)[32]) const {
    tmem_ld32x2(at(l1), at(l2), r, q);
  }
};
struct RegAcc {
  static constexpr int kUnroll = 4;
  const uint32_t (&c0)[32];
  const uint32_t (&c1)[32];
  const uint32_t (&c2)[32];
  const uint32_t (&c3)[32];
  __device__ __forceinline__ void ld32(int l, uint32_t (&r)[32]) const {
    const uint32_t(&c)[32] = l < 32 ? c0 : (l < 64 ? c1 : (l < 96 ? c2 : c3));
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = c[i];
  }
  __device__ __forceinline__ void ld32x2(int l1, int l2, uint32_t (&r)[32], uint32_t (&q)[32]) const {
    ld32(l1, r);
    ld32(l2, q);
  }
};

template <bool S8>
struct EpiQKVGT {
  static constexpr bool kS8 = S8;
  Fwd f;
  QkvgDst dst;
  int N;  // rows of W_qkvg
  Deq dq;
  // logical columns = accumulator columns half * 128 .. + 127 (one head)
  static __device__ __forceinline__ TmemAcc tmem_acc(uint32_t taddr, int half) {
    return TmemAcc{taddr + half * 128, taddr + half * 128 + 64};
  }
  __device__ __forceinline__ void apply(int row, int nb, int half, uint32_t taddr, int M) const {
    apply_acc(row, nb, half, tmem_acc(taddr, half), M);
  }
  template <class A>
  __device__ __forceinline__ void apply_acc(int row, int nb, int half, const A& acc, int M) const {
    constexpr int HD = 128;
    const int n0 = nb * BN + half * HD;
    if (n0 >= N) return;
    const bool ok = row < M;
    const int seg = n0 / HD;
    int kind, head;
    if (seg < f.n_q) { kind = 0; head = seg; }
    else if (seg < f.n_q + f.n_kv) { kind = 1; head = seg - f.n_q; }
    else if (seg < f.n_q + 2 * f.n_kv) { kind = 2; head = seg - f.n_q - f.n_kv; }
    else { kind = 3; head = seg - f.n_q - 2 * f.n_kv; }
    const int b = ok ? row / f.L : 0;
    const int l = ok ? row - b * f.L : 0;
    const float fa = deq_row<S8>(dq, row, ok);
    uint32_t r[32];

    if (kind <= 1) {
      float ss = 0.f;
#pragma unroll(A::kUnroll)
      for (int c = 0; c < 4; ++c) {
        acc.ld32(c * 32, r);
        deq32<S8>(r, dq, fa, dq.b, n0 + c * 32);
#pragma unroll
        for (int i = 0; i < 32; ++i) ss = fmaf(u2f(r[i]), u2f(r[i]), ss);
      }
      const float rstd = 1.0f / sqrtf(ss * (1.0f / HD) + f.eps);
      const float* w = kind == 0 ? dst.q_norm_w : dst.k_norm_w;
      const bool img = ok && l >= f.n_txt;
      int pr = 0, pc = 0;
      if (img) {
        const int n = l - f.n_txt;
        pr = n / f.img_w;
        pc = n - pr * f.img_w;
      }
      const int nh = kind == 0 ? f.n_q : f.n_kv;
      bf16* out = reinterpret_cast<bf16*>(kind == 0 ? dst.q : dst.k) +
                  ((static_cast<size_t>(b) * nh + head) * f.L + l) * HD;
#pragma unroll(A::kUnroll)
      for (int c = 0; c < 4; ++c) {
        acc.ld32(c * 32, r);
        deq32<S8>(r, dq, fa, dq.b, n0 + c * 32);
        if (dst.raw && ok) {  // the projection before the norm, for the backward
          float4* o4 = reinterpret_cast<float4*>(dst.raw + static_cast<size_t>(row) * dst.ldr + n0 + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) o4[q] = make_float4(u2f(r[4 * q]), u2f(r[4 * q + 1]), u2f(r[4 * q + 2]), u2f(r[4 * q + 3]));
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = u2f(r[i]) * rstd * (1.0f + __ldg(w + c * 32 + i));
        if (img) {
          // chunk c holds pairs 16c .. 16c+15; pairs 0..31 turn with the row, 32..63 with the column
          const float2* tab = dst.rope + (c < 2 ? pr : pc) * (HD / 4) + (c & 1) * 16;
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            const float2 cs = __ldg(tab + p);
            const float a = v[2 * p], bb = v[2 * p + 1];
            v[2 * p] = a * cs.x - bb * cs.y;
            v[2 * p + 1] = a * cs.y + bb * cs.x;
          }
        }
        if (ok) {
          uint4* o4 = reinterpret_cast<uint4*>(out + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            o4[q4] = make_uint4(pack_bf16x2(v[8 * q4 + 0], v[8 * q4 + 1]), pack_bf16x2(v[8 * q4 + 2], v[8 * q4 + 3]),
                                pack_bf16x2(v[8 * q4 + 4], v[8 * q4 + 5]), pack_bf16x2(v[8 * q4 + 6], v[8 * q4 + 7]));
        }
      }
    } else if (kind == 2) {
      // V^T [B, n_kv, hd, Lp]: lanes hold consecutive tokens, so each channel's 32 values
      // from a warp land in one contiguous 64-byte run.
      bf16* vt = reinterpret_cast<bf16*>(dst.vt) + (static_cast<size_t>(b) * f.n_kv + head) * HD * f.Lp + l;
#pragma unroll(A::kUnroll)
      for (int c = 0; c < 4; ++c) {
        acc.ld32(c * 32, r);
        deq32<S8>(r, dq, fa, dq.b, n0 + c * 32);
        if (ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i) vt[static_cast<size_t>(c * 32 + i) * f.Lp] = __float2bfloat16_rn(u2f(r[i]));
        }
      }
    } else {
      bf16* g = reinterpret_cast<bf16*>(dst.g) + static_cast<size_t>(row) * (f.n_q * HD) + head * HD;
#pragma unroll(A::kUnroll)
      for (int c = 0; c < 4; ++c) {
        acc.ld32(c * 32, r);
        deq32<S8>(r, dq, fa, dq.b, n0 + c * 32);
        if (ok) {
          // the gate value sigmoid(xn W_g^T) itself: the attention epilogue and the gate
          // backward only multiply by it
          float sg[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) sg[i] = sigmoid_fast(u2f(r[i]));
          uint4* o4 = reinterpret_cast<uint4*>(g + c * 32);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            o4[q4] = make_uint4(pack_bf16x2(sg[8 * q4 + 0], sg[8 * q4 + 1]), pack_bf16x2(sg[8 * q4 + 2], sg[8 * q4 + 3]),
                                pack_bf16x2(sg[8 * q4 + 4], sg[8 * q4 + 5]), pack_bf16x2(sg[8 * q4 + 6], sg[8 * q4 + 7]));
        }
      }
    }
  }
};

// 32 consecutive residual values of one row (one accumulator chunk), loaded one chunk
// ahead of their use so that the load's DRAM latency overlaps the previous chunk's work
template <class T>
struct Res32;
template <>
struct Res32<bf16> {
  uint4 v[4];
  __device__ __forceinline__ void load(const bf16* p) {
    const uint4* p4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(p4 + i);
  }
  __device__ __forceinline__ void get8(int q4, float (&o)[8]) const {
    const float2 a = unpack_bf16x2(v[q4].x), b = unpack_bf16x2(v[q4].y), c = unpack_bf16x2(v[q4].z),
                 e = unpack_bf16x2(v[q4].w);
    o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y; o[4] = c.x; o[5] = c.y; o[6] = e.x; o[7] = e.y;
  }
};
template <>
struct Res32<float> {
  float4 v[8];
  __device__ __forceinline__ void load(const float* p) {
    const float4* p4 = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(p4 + i);
  }
  __device__ __forceinline__ void get8(int q4, float (&o)[8]) const {
    const float4 a = v[2 * q4], b = v[2 * q4 + 1];
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
  }
};

// 8 consecutive residual values of one row (zeros for a row past M)
__device__ __forceinline__ void res8(const bf16* p, bool ok, float (&o)[8]) {
  const uint4 u = ok ? __ldg(reinterpret_cast<const uint4*>(p)) : make_uint4(0, 0, 0, 0);
  const float2 a = unpack_bf16x2(u.x), b = unpack_bf16x2(u.y), c = unpack_bf16x2(u.z), e = unpack_bf16x2(u.w);
  o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y; o[4] = c.x; o[5] = c.y; o[6] = e.x; o[7] = e.y;
}
__device__ __forceinline__ void res8(const float* p, bool ok, float (&o)[8]) {
  const float4 a = ok ? __ldg(reinterpret_cast<const float4*>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 b = ok ? __ldg(reinterpret_cast<const float4*>(p) + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

// out = res + gate * acc. The attention residual reads the bf16 block input from the
// caller's split text/image buffers and writes the fp32 residual stream h1; the MLP
// residual reads h1 and writes the bf16 block output. d is a multiple of 64, so a
// 128-column half holds 2 or 4 whole 32-column chunks.
// The result leaves through shared memory: each epilogue warp owns a 4 KB box (32 rows x
// 128 bytes, laid out in the 128-byte swizzle), every lane writes its row into it and one
// lane hands the box to a TMA store, so the output reaches L2 as whole lines rather than as
// 32 scattered 16-byte pieces per store instruction. Rows past M are clipped by the store.
template <class TRes, class TOut, bool S8>
struct EpiResid {
  static constexpr bool kS8 = S8;
  static constexpr int kStgBytes = 4096;  // per epilogue warp
  static constexpr int kPerBox = sizeof(TOut) == 4 ? 1 : 2;  // 32-column chunks per box
  Fwd f;
  RowSrc res;
  const float* mod_shared;
  const float* mod_bias;
  int chunk;   // modulation chunk of the gate (2 = gate_a, 5 = gate_m)
  Deq dq;
  float* pre = nullptr;  // optional [T, d] fp32: the product before the gate (for the backward)
  // stg: this warp's box (1024-byte aligned); tm_out: the output [T, d] with a box of 128
  // bytes x 32 rows and the 128-byte swizzle
  // logical columns = accumulator columns half * 128 .. + 127
  static __device__ __forceinline__ TmemAcc tmem_acc(uint32_t taddr, int half) {
    return TmemAcc{taddr + half * 128, taddr + half * 128 + 64};
  }
  __device__ __forceinline__ void apply(int row, int nb, int half, uint32_t taddr, int M, uint8_t* stg, int lane,
                                        const CUtensorMap* tm_out) const {
    apply_acc(row, nb, half, tmem_acc(taddr, half), M, stg, lane, tm_out);
  }
  template <class A>
  __device__ __forceinline__ void apply_acc(int row, int nb, int half, const A& acc, int M, uint8_t* stg, int lane,
                                            const CUtensorMap* tm_out) const {
    const int N = f.d;
    const int n0 = nb * BN + half * 128;
    if (n0 >= N) return;
    const bool ok = row < M;
    const int b = ok ? row / f.L : 0;
    const TRes* x = ok ? row_src_ptr<TRes>(res, row, f.L, f.n_txt, f.n_img, f.d) : nullptr;
    const float* gs = mod_shared + (static_cast<size_t>(b) * 6 + chunk) * N;
    const float* gb = mod_bias + static_cast<size_t>(chunk) * N;
    const float fa = deq_row<S8>(dq, row, ok);
    const int nc = min(4, (N - n0) >> 5);
    uint8_t* srow = stg + lane * 128;
    const int sw = lane & 7;  // the swizzle of this row: 16-byte unit j sits at j ^ sw
    // From tensor memory the residual chunk after the current one is loaded ahead; from
    // registers (which already hold the accumulator, and where the epilogue overlaps the
    // next tile's products) each chunk is loaded where it is used.
    constexpr bool kAhead = A::kUnroll == 1;
    Res32<TRes> cur, nxt;
    if (ok && kAhead) cur.load(x + n0);
    uint32_t r[32];
#pragma unroll(A::kUnroll)
    for (int c = 0; c < (A::kUnroll == 1 ? nc : 4); ++c) {  // a constant trip count when unrolled
      if (c < nc) {
      const int col = n0 + c * 32;
      if constexpr (kAhead) {
        if (ok && c + 1 < nc) nxt.load(x + col + 32);
      }
      acc.ld32(c * 32, r);
      deq32<S8>(r, dq, fa, dq.b, col);
      if (ok && pre) {
        float4* p4 = reinterpret_cast<float4*>(pre + static_cast<size_t>(row) * N + col);
#pragma unroll
        for (int q = 0; q < 8; ++q) p4[q] = make_float4(u2f(r[4 * q]), u2f(r[4 * q + 1]), u2f(r[4 * q + 2]), u2f(r[4 * q + 3]));
      }
      if (c % kPerBox == 0) {  // the previous box has left shared memory before it is rewritten
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
      }
      const float4* gs4 = reinterpret_cast<const float4*>(gs + col);
      const float4* gb4 = reinterpret_cast<const float4*>(gb + col);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float xv[8];
        if constexpr (kAhead) cur.get8(q4, xv);
        else res8(x + col + 8 * q4, ok, xv);
        const float4 s0 = __ldg(gs4 + 2 * q4), s1 = __ldg(gs4 + 2 * q4 + 1);
        const float4 b0 = __ldg(gb4 + 2 * q4), b1 = __ldg(gb4 + 2 * q4 + 1);
        const float gt[8] = {s0.x + b0.x, s0.y + b0.y, s0.z + b0.z, s0.w + b0.w,
                             s1.x + b1.x, s1.y + b1.y, s1.z + b1.z, s1.w + b1.w};
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = fmaf(gt[i], u2f(r[8 * q4 + i]), xv[i]);
        if constexpr (sizeof(TOut) == 4) {
          const int j = 2 * q4;
          *reinterpret_cast<float4*>(srow + ((j ^ sw) << 4)) = make_float4(y[0], y[1], y[2], y[3]);
          *reinterpret_cast<float4*>(srow + (((j + 1) ^ sw) << 4)) = make_float4(y[4], y[5], y[6], y[7]);
        } else {
          const int j = (c & 1) * 4 + q4;
          *reinterpret_cast<uint4*>(srow + ((j ^ sw) << 4)) =
              make_uint4(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]), pack_bf16x2(y[4], y[5]),
                         pack_bf16x2(y[6], y[7]));
        }
      }
      if (c % kPerBox == kPerBox - 1) {
        fence_proxy_async_smem();  // the lanes' writes are visible to the TMA engine
        __syncwarp();
        if (lane == 0 && row < M) {  // lane 0's row is the box's first: a box wholly past M is skipped
          tma_store_2d(tm_out, stg, col - (kPerBox - 1) * 32, row);
          bulk_commit();
        }
      }
      }
      if constexpr (kAhead) cur = nxt;
    }
  }
};
template <bool S8>
using EpiResidAttnT = EpiResid<bf16, float, S8>;
template <bool S8>
using EpiResidMlpT = EpiResid<float, bf16, S8>;

template <bool S8>
struct EpiSwiGLUT {
  static constexpr bool kS8 = S8;
  int F;
  bf16* hmid;      // [T, F]
  float* rowamax;  // optional [T] (8-bit GEMMs only): largest |hmid| of each row, as stored
  Deq dq;
  float* pre_a = nullptr;  // optional [T, F] fp32: hn W_gate^T and hn W_up^T (for the backward)
  float* pre_u = nullptr;
  // accumulator columns [0,128) = hn W_gate^T, [128,256) = hn W_up^T for F-columns nb*128 ..;
  // logical columns: [0, 64) = gate columns half * 64 .., [64, 128) = the same columns of up
  static __device__ __forceinline__ TmemAcc tmem_acc(uint32_t taddr, int half) {
    return TmemAcc{taddr + half * 64, taddr + 128 + half * 64};
  }
  __device__ __forceinline__ void apply(int row, int nb, int half, uint32_t taddr, int M) const {
    apply_acc(row, nb, half, tmem_acc(taddr, half), M);
  }
  template <class A>
  __device__ __forceinline__ void apply_acc(int row, int nb, int half, const A& acc, int M) const {
    const int f0 = nb * 128 + half * 64;
    if (f0 >= F) return;
    const bool ok = row < M;
    const float fa = deq_row<S8>(dq, row, ok);
    float amax = 0.0f;
    uint32_t rg[32], ru[32];
#pragma unroll(A::kUnroll)
    for (int c = 0; c < 2; ++c) {
      acc.ld32x2(c * 32, 64 + c * 32, rg, ru);
      deq32<S8>(rg, dq, fa, dq.b, f0 + c * 32);
      deq32<S8>(ru, dq, fa, dq.b2, f0 + c * 32);
      if (ok && pre_a) {
        float4* a4 = reinterpret_cast<float4*>(pre_a + static_cast<size_t>(row) * F + f0 + c * 32);
        float4* u4 = reinterpret_cast<float4*>(pre_u + static_cast<size_t>(row) * F + f0 + c * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          a4[q] = make_float4(u2f(rg[4 * q]), u2f(rg[4 * q + 1]), u2f(rg[4 * q + 2]), u2f(rg[4 * q + 3]));
          u4[q] = make_float4(u2f(ru[4 * q]), u2f(ru[4 * q + 1]), u2f(ru[4 * q + 2]), u2f(ru[4 * q + 3]));
        }
      }
      if (ok) {
        uint4* o4 = reinterpret_cast<uint4*>(hmid + static_cast<size_t>(row) * F + f0 + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float h[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            h[i] = u2f(rg[8 * q4 + i]) * sigmoid_fast(u2f(rg[8 * q4 + i])) * u2f(ru[8 * q4 + i]);
            if constexpr (S8) amax = fmaxf(amax, fabsf(h[i]));
          }
          o4[q4] = make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]), pack_bf16x2(h[4], h[5]),
                              pack_bf16x2(h[6], h[7]));
        }
      }
    }
    // bf16 rounding is monotone, so the largest stored magnitude is the rounded largest
    if constexpr (S8) {
      if (rowamax && ok) atomic_max_nonneg(rowamax + row, round_bf16(amax));
    }
  }
};

// SwiGLU backward finished in the epilogue of d_hmid = d_fm W_down: with hmid = silu(a) u,
// d_a = d_hmid u silu'(a) and d_u = d_hmid silu(a) go as bf16 into d_au [T, 2F] (columns
// [0, F) and [F, 2F)); a and u are the forward's fp32 pre-activations [T, F].
struct EpiSwiGLUBwd {
  static constexpr bool kS8 = false;
  const float* a;
  const float* u;
  bf16* d_au;
  int F;
  __device__ __forceinline__ void apply(int row, int nb, int half, uint32_t taddr, int M) const {
    const int n0 = nb * BN + half * 128;
    if (n0 >= F) return;
    const bool ok = row < M;
    uint32_t r[32];
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = n0 + c * 32;
      if (col >= F) break;
      tmem_ld32(taddr + half * 128 + c * 32, r);
      if (!ok) continue;
      const size_t off = static_cast<size_t>(row) * F + col;
      bf16* da = d_au + static_cast<size_t>(row) * 2 * F + col;
      if (col + 32 <= F) {
        const float4* a4 = reinterpret_cast<const float4*>(a + off);
        const float4* u4 = reinterpret_cast<const float4*>(u + off);
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // 8 columns per step
          const float4 a0 = __ldg(a4 + 2 * q), a1 = __ldg(a4 + 2 * q + 1);
          const float4 u0 = __ldg(u4 + 2 * q), u1 = __ldg(u4 + 2 * q + 1);
          const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          float ga[8], gu[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float dh = u2f(r[8 * q + i]);
            const float sg = sigmoid_fast(av[i]);
            ga[i] = dh * uv[i] * sg * (1.0f + av[i] * (1.0f - sg));
            gu[i] = dh * av[i] * sg;
          }
          reinterpret_cast<uint4*>(da)[q] = make_uint4(pack_bf16x2(ga[0], ga[1]), pack_bf16x2(ga[2], ga[3]),
                                                       pack_bf16x2(ga[4], ga[5]), pack_bf16x2(ga[6], ga[7]));
          reinterpret_cast<uint4*>(da + F)[q] = make_uint4(pack_bf16x2(gu[0], gu[1]), pack_bf16x2(gu[2], gu[3]),
                                                           pack_bf16x2(gu[4], gu[5]), pack_bf16x2(gu[6], gu[7]));
        }
      } else {
        for (int i = 0; i < F - col; ++i) {
          const float dh = u2f(r[i]), av = a[off + i], sg = sigmoid_fast(av);
          da[i] = __float2bfloat16_rn(dh * u[off + i] * sg * (1.0f + av * (1.0f - sg)));
          da[F + i] = __float2bfloat16_rn(dh * av * sg);
        }
      }
    }
  }
};

// Output-gate backward finished in the epilogue of d_og = d_fa W_o (one 128-column half of
// a tile is one head): with og = o s, s = sigmoid(g) as the forward stored it, d_o = d_og s
// goes as bf16 to the head-major [B, n_q, L, 128] buffer the attention backward reads,
// the gradient of the pre-activation d_og o s (1 - s) to d_P's g columns (bf16, from
// column goff), and the
// softmax row term D = sum over the head of d_o (as stored) times o to D[b, head, l] (row
// pitch Lp). Without the gate, d_o = d_og.
struct EpiGateBwd {
  static constexpr bool kS8 = false;
  Fwd f;
  const float* o;    // [T, n_q*128] fp32, the ungated attention output
  const bf16* g;     // [T, n_q*128] the gate value sigmoid(xn W_g^T)
  bf16* d_o;         // [B, n_q, L, 128]
  bf16* d_P;         // [T, ldp]
  int ldp, goff;
  float* D;          // [B, n_q, Lp]
  __device__ __forceinline__ void apply(int row, int nb, int half, uint32_t taddr, int M) const {
    constexpr int HD = 128;
    const int nq = f.n_q * HD;
    const int n0 = nb * BN + half * HD;
    if (n0 >= nq) return;
    const bool ok = row < M;
    const int head = n0 / HD;
    const int b = ok ? row / f.L : 0, l = ok ? row - b * f.L : 0;
    bf16* dst = d_o + ((static_cast<size_t>(b) * f.n_q + head) * f.L + l) * HD;
    const size_t off = static_cast<size_t>(row) * nq + n0;
    float dsum = 0.0f;
    uint32_t r[32];
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      tmem_ld32(taddr + half * HD + c * 32, r);
      if (!ok) continue;
      const float4* o4 = reinterpret_cast<const float4*>(o + off + c * 32);
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // 8 columns per step
        const float4 oa = __ldg(o4 + 2 * q), ob = __ldg(o4 + 2 * q + 1);
        const float ov[8] = {oa.x, oa.y, oa.z, oa.w, ob.x, ob.y, ob.z, ob.w};
        float dov[8], dg[8];
        if (f.gate_on) {
          const uint4 gu = __ldg(reinterpret_cast<const uint4*>(g + off + c * 32) + q);
          const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 gg = unpack_bf16x2(gw[e]);
            const float s0 = gg.x, s1 = gg.y;  // the stored gate values
            const float a0 = u2f(r[8 * q + 2 * e]), a1 = u2f(r[8 * q + 2 * e + 1]);
            dov[2 * e] = a0 * s0;
            dov[2 * e + 1] = a1 * s1;
            dg[2 * e] = a0 * ov[2 * e] * s0 * (1.0f - s0);
            dg[2 * e + 1] = a1 * ov[2 * e + 1] * s1 * (1.0f - s1);
          }
          reinterpret_cast<uint4*>(d_P + static_cast<size_t>(row) * ldp + goff + n0 + c * 32)[q] =
              make_uint4(pack_bf16x2(dg[0], dg[1]), pack_bf16x2(dg[2], dg[3]), pack_bf16x2(dg[4], dg[5]),
                         pack_bf16x2(dg[6], dg[7]));
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) dov[e] = u2f(r[8 * q + e]);
        }
        const uint4 pk = make_uint4(pack_bf16x2(dov[0], dov[1]), pack_bf16x2(dov[2], dov[3]),
                                    pack_bf16x2(dov[4], dov[5]), pack_bf16x2(dov[6], dov[7]));
        reinterpret_cast<uint4*>(dst + c * 32)[q] = pk;
        const uint32_t pw[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 dd = unpack_bf16x2(pw[e]);
          dsum = fmaf(dd.x, ov[2 * e], dsum);
          dsum = fmaf(dd.y, ov[2 * e + 1], dsum);
        }
      }
    }
    if (ok) D[(static_cast<size_t>(b) * f.n_q + head) * f.Lp + l] = dsum;
  }
};

// C = alpha * (A B^T) (+ C when accumulating), fp32 row-major with row pitch ldc (a
// multiple of 4): the plain product the block backward is built from.
struct EpiPlain {
  static constexpr bool kS8 = false;
  float* C;
  long long ldc;
  int N;
  int accumulate;
  float alpha;
  __device__ __forceinline__ void apply(int row, int nb, int half, uint32_t taddr, int M) const {
    const int n0 = nb * BN + half * 128;
    if (n0 >= N) return;
    const bool ok = row < M;
    uint32_t r[32];
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      const int col = n0 + c * 32;
      if (col >= N) break;
      tmem_ld32(taddr + half * 128 + c * 32, r);
      if (!ok) continue;
      float* o = C + static_cast<long long>(row) * ldc + col;
      if (col + 32 <= N) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 v = make_float4(alpha * u2f(r[4 * q]), alpha * u2f(r[4 * q + 1]), alpha * u2f(r[4 * q + 2]),
                                 alpha * u2f(r[4 * q + 3]));
          float4* p4 = reinterpret_cast<float4*>(o + 4 * q);
          if (accumulate) {
            const float4 w = *p4;
            v.x += w.x;
            v.y += w.y;
            v.z += w.z;
            v.w += w.w;
          }
          *p4 = v;
        }
      } else {
        for (int i = 0; i < N - col; ++i) o[i] = alpha * u2f(r[i]) + (accumulate ? o[i] : 0.0f);
      }
    }
  }
};

// ------------------------------------------------------------------ the kernel
template <class Epi, bool DUAL>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_b2, const __grid_constant__ CUtensorMap tm_c, int M,
                   int num_n, int K, int group, Epi epi, int* err) {
  constexpr bool FP8 = Epi::kS8;
  constexpr int BK = FP8 ? 128 : 64;  // K elements per stage (128 bytes of each operand row)
  constexpr int STG = StgOf<Epi>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = smem + STAGES * STAGE_BYTES;  // epilogue staging boxes (1024-byte aligned)
  uint64_t* full = reinterpret_cast<uint64_t*>(stg_base + NUM_EPI_WARPS * STG);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = static_cast<int>(cluster_ctarank());  // 0 or 1 inside the CTA pair
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int num_m = (M + BM - 1) / BM;
  const int num_mp = (num_m + 1) / 2;                    // pairs of m-blocks
  const int num_tiles = num_mp * num_n;                  // pair tiles (256 x 256)
  const int num_kb = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);   // even CTA: its producer's arrive + both CTAs' bytes
      mbar_init(&empty[s], 1);  // the pair MMA's commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * NUM_EPI_WARPS);  // even CTA: both CTAs' epilogue warps
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers are initialised before the peer signals any of them
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx wc{abort_flag, err};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      if (DUAL) tma_prefetch_desc(&tm_b2);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      // B half of this CTA: rows [128 rank, 128 rank + 128) of the 256-row B tile (for the
      // SwiGLU GEMM: W_gate rows for rank 0, W_up rows for rank 1)
      const CUtensorMap* map_b = (DUAL && rank == 1) ? &tm_b2 : &tm_b;
      const uint32_t full0 = mapa_shared(smem_u32(full), 0);  // the even CTA's full barriers
      for (int tile = pair; ok && tile < num_tiles; tile += npairs) {
        int mp, nb;
        tile_coords(tile, num_mp, num_n, group, mp, nb);
        const int mb = 2 * mp + rank;
        const int yb = DUAL ? nb * (BN / 2) : nb * BN + rank * (BN / 2);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wc, SITE_GEMM_PRODUCER)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * STAGE_BYTES;
          uint8_t* sb = sa + A_BYTES;
          // own A (16 KB) + own B half (16 KB), completing on the even CTA's barrier, which
          // expects both CTAs' bytes
          if (rank == 0) mbar_arrive_expect_tx(&full[stage], 2 * STAGE_BYTES);
          const uint32_t fb = full0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
          tma_load_2d_pair(sa, &tm_a, fb, kb * BK, mb * BM);
          tma_load_2d_pair(sb, map_b, fb, kb * BK, yb);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every copy this thread started has landed before the CTA exits: on the even CTA
      // its full barriers count both CTAs' bytes; the odd CTA sees its stages freed by the
      // MMA, which reads them only after they landed
      for (long long i = (issued > STAGES ? issued - STAGES : 0); i < issued; ++i)
        drain_wait(rank == 0 ? &full[i % STAGES] : &empty[i % STAGES], static_cast<uint32_t>((i / STAGES) & 1),
                   err, SITE_GEMM_TEARDOWN);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (even CTA): pair MMAs, M = 256 across the two CTAs
      constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(2 * BM, BN) : idesc_bf16_f32(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int tile = pair; ok && tile < num_tiles; tile += npairs) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, wc, SITE_GEMM_MMA)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, wc, SITE_GEMM_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // 32 bytes of K per MMA
            if constexpr (FP8)
              mma_e4m3_ss_pair(d_tmem, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32), idesc,
                               (kb | k) != 0 ? 1u : 0u);
            else
              mma_bf16_ss_pair(d_tmem, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32), idesc,
                               (kb | k) != 0 ? 1u : 0u);
          }
          mma_commit_pair_mc(&empty[stage], 0x3);  // frees the stage in both CTAs once these MMAs read it
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_mc(&tfull[acc], 0x3);  // accumulator ready for both CTAs' epilogues
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      mma_commit_pair_mc(done, 0x1);  // completes when every MMA issued above has finished
      drain_wait(done, 0, err, SITE_GEMM_TEARDOWN);
    }
  } else {
    // ---------------- epilogue warps
    const int quad = warp & 3;                 // TMEM lanes this warp may access: 32*quad ..
    const int half = (warp - 2) / 4;           // 128-column half of the accumulator
    int acc = 0;
    uint32_t acc_phase = 0;
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);  // the even CTA's tempty barriers
    for (int tile = pair; tile < num_tiles; tile += npairs) {
      int mp, nb;
      tile_coords(tile, num_mp, num_n, group, mp, nb);
      const int mb = 2 * mp + rank;
      const bool got = mbar_wait(&tfull[acc], acc_phase, wc, SITE_GEMM_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int row = mb * BM + quad * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * BN);
      if constexpr (STG > 0)
        epi.apply(row, nb, half, taddr, M, stg_base + (warp - 2) * STG, lane, &tm_c);
      else
        epi.apply(row, nb, half, taddr, M);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty0 + static_cast<uint32_t>(acc * sizeof(uint64_t)));
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
    if constexpr (STG > 0) {  // this warp's TMA stores have completed
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  __syncthreads();
  cluster_sync();  // no CTA leaves while the pair's MMAs, copies or arrivals may still reach it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ NVFP4 GEMM
// Operands are E2M1 codes (two per byte) with E4M3 scales per 16 elements of K (see
// quant4.cu for the formats) and one power-of-two tensor scale each; the tensor scales
// reach the epilogue as the per-tensor factors of an 8-bit epilogue (Deq).
//
// One CTA per 128 x 256 output tile (no CTA pairs), persistent over the tiles. A stage
// covers 256 elements of K (128 bytes of each operand row): A 128 x 128 B and the two
// 128-row halves of B by TMA with the 128-byte swizzle, and the stage's scale atoms of A
// and of both B halves by 1D bulk copies (54 KB). The scale atoms go into tensor memory
// by tcgen05.cp, split over three threads because a copy occupies its issuing thread far
// longer than an MMA does: two copy warps take the atoms of the two B halves, the MMA
// thread those of A, each stage into one of two 48-column slots. The MMA thread waits for
// the copy warps' copies, then issues one kind::mxf4nvf4 MMA (M = 128, N = 256, K = 64) per
// 64-element step into the 256-column accumulator, which has the layout the bf16 kernel's
// epilogues read, and frees the slot with a commit. The B halves are two TMA boxes of 128
// rows stacked in shared memory (so the SwiGLU GEMM's W_gate and W_up rows form one 256-row
// operand) and their scale atoms two adjacent 4-column groups in tensor memory. The
// accumulator is single-buffered (the scale slots take tensor-memory columns 256 .. 351);
// each epilogue warp copies its 128 columns into registers and hands the accumulator back
// at once, so the epilogue's work overlaps the next tile's main loop. Warp roles: 0 TMA,
// 1 TMEM + A scale copies + MMA, 2..9 epilogue, 10 and 11 B scale copies.
constexpr int F4_BM = 128, F4_BN = 256;
constexpr int F4_A_BYTES = F4_BM * 128;
constexpr int F4_BH_BYTES = (F4_BN / 2) * 128;
constexpr int F4_ATOM = 512;                       // scales of 128 rows x 64 elements
constexpr int F4_SF_BYTES = 3 * 4 * F4_ATOM;       // A, B half 0, B half 1; four 64-element steps
constexpr int F4_STAGE = F4_A_BYTES + 2 * F4_BH_BYTES + F4_SF_BYTES;
constexpr int F4_SF_TMEM = 256;                    // first TMEM column of the scale copies
template <class Epi>
__host__ __device__ constexpr int f4_stages() {
  return StgOf<Epi>::value > 0 ? 3 : 4;
}
// Two more warps than the bf16 kernel copy the B operand's scale atoms (one warp per
// 128-row half); 12 warps keep the 168-register cap of 10 (3 warps per SM sub-partition).
constexpr int F4_THREADS = NUM_THREADS + 64;
constexpr int F4_SF_SLOT = 48;  // TMEM columns of one stage's scales; two slots
template <class Epi>
__host__ __device__ constexpr int f4_smem_bytes() {
  return f4_stages<Epi>() * F4_STAGE + NUM_EPI_WARPS * StgOf<Epi>::value + 1024 + 256;
}

template <class Epi, bool DUAL>
__global__ void __launch_bounds__(F4_THREADS, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_b2, const __grid_constant__ CUtensorMap tm_c, int M,
                    int num_n, int K, int group, int b_blocks, const uint8_t* __restrict__ sf_a,
                    const uint8_t* __restrict__ sf_b, const uint8_t* __restrict__ sf_b2, Epi epi, int* err) {
  constexpr int NST = f4_stages<Epi>();
  constexpr int STG = StgOf<Epi>::value;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg_base = smem + NST * F4_STAGE;
  uint64_t* full = reinterpret_cast<uint64_t*>(stg_base + NUM_EPI_WARPS * STG);
  uint64_t* empty = full + NST;
  uint64_t* tfull = empty + NST;
  uint64_t* tempty = tfull + 1;
  uint64_t* done = tempty + 1;
  uint64_t* sf_ready = done + 1;     // [2] the B scale copies of a slot have landed (2 arrivals)
  uint64_t* sf_free = sf_ready + 2;  // [2] the MMAs that read a slot have finished
  uint64_t* done_cp = sf_free + 2;   // every copy of the two copy warps has finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_cp + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (M + F4_BM - 1) / F4_BM;
  const int num_tiles = num_m * num_n;
  const int KS = K / 64;                  // 64-element steps (scale atoms per 128-row block)
  const int num_kb = (KS + 3) / 4;        // stages of 256 elements

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, NUM_EPI_WARPS);
    mbar_init(done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sf_ready[i], 2);
      mbar_init(&sf_free[i], 1);
    }
    mbar_init(done_cp, 2);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  // zero every stage's scale area: a B half past the matrix's last 128-row block is not
  // copied (its codes arrive as TMA zero fill), so its scales must be finite
  for (int i = threadIdx.x; i < NST * (F4_SF_BYTES / 16); i += blockDim.x) {
    const int st = i / (F4_SF_BYTES / 16), u = i % (F4_SF_BYTES / 16);
    reinterpret_cast<uint4*>(smem + st * F4_STAGE + F4_A_BYTES + 2 * F4_BH_BYTES)[u] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitCtx wc{abort_flag, err};

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA / bulk-copy producer
      tma_prefetch_desc(&tm_a);
      tma_prefetch_desc(&tm_b);
      if (DUAL) tma_prefetch_desc(&tm_b2);
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int mb, nb;
        tile_coords(tile, num_m, num_n, group, mb, nb);
        // B halves: rows of W (or of W_gate / W_up for the SwiGLU GEMM) and their scale blocks
        const CUtensorMap* map_b1 = DUAL ? &tm_b2 : &tm_b;
        const int yb0 = DUAL ? nb * 128 : nb * F4_BN, yb1 = DUAL ? nb * 128 : nb * F4_BN + 128;
        const int rb0 = DUAL ? nb : 2 * nb, rb1 = DUAL ? nb : 2 * nb + 1;  // scale blocks of the halves
        const bool has1 = rb1 < b_blocks;  // the second half lies (partly) inside the matrix
        const uint8_t* sfb0 = sf_b + static_cast<size_t>(rb0) * KS * F4_ATOM;
        const uint8_t* sfb1 = (DUAL ? sf_b2 : sf_b) + static_cast<size_t>(has1 ? rb1 : rb0) * KS * F4_ATOM;
        const uint8_t* sfa = sf_a + static_cast<size_t>(mb) * KS * F4_ATOM;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wc, SITE_GEMM_PRODUCER)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * F4_STAGE;
          uint8_t* sb = sa + F4_A_BYTES;
          uint8_t* ssf = sb + 2 * F4_BH_BYTES;
          const int nks = min(4, KS - 4 * kb);
          const uint32_t sf_bytes = static_cast<uint32_t>(nks) * F4_ATOM;
          mbar_arrive_expect_tx(&full[stage], F4_A_BYTES + 2 * F4_BH_BYTES + (has1 ? 3 : 2) * sf_bytes);
          tma_load_2d(sa, &tm_a, &full[stage], kb * 128, mb * F4_BM);
          tma_load_2d(sb, &tm_b, &full[stage], kb * 128, yb0);
          tma_load_2d(sb + F4_BH_BYTES, map_b1, &full[stage], kb * 128, yb1);
          bulk_load(ssf, sfa + static_cast<size_t>(4 * kb) * F4_ATOM, sf_bytes, &full[stage]);
          bulk_load(ssf + 4 * F4_ATOM, sfb0 + static_cast<size_t>(4 * kb) * F4_ATOM, sf_bytes, &full[stage]);
          if (has1)
            bulk_load(ssf + 8 * F4_ATOM, sfb1 + static_cast<size_t>(4 * kb) * F4_ATOM, sf_bytes, &full[stage]);
          ++issued;
          if (++stage == NST) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // every copy this thread started has landed before the CTA exits
      for (long long i = (issued > NST ? issued - NST : 0); i < issued; ++i)
        drain_wait(&full[i % NST], static_cast<uint32_t>((i / NST) & 1), err, SITE_GEMM_TEARDOWN);
    }
  } else if (warp == 1) {
    // ---------------- A scale copies + MMA issue. The whole warp runs the loop (waits,
    // addresses and descriptors computed warp-uniformly); lane 0 issues every tcgen05
    // instruction and commit. The B scale atoms of a stage are copied by warps 10 and 11
    // into the stage's TMEM slot (two slots of 48 columns, alternating by stage): the MMA
    // thread waits for their copies to land and frees the slot with a commit after the
    // stage's MMAs.
    constexpr uint32_t idesc = idesc_nvf4_f32(F4_BM, F4_BN);
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t slot_phase = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      if (!__all_sync(0xffffffffu, mbar_wait(tempty, acc_phase ^ 1, wc, SITE_GEMM_MMA))) break;
      tc_fence_after();
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, wc, SITE_GEMM_MMA)) ||
            !__all_sync(0xffffffffu, mbar_wait(&sf_ready[slot], slot_phase, wc, SITE_GEMM_MMA))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * F4_STAGE);
        const uint32_t sb = sa + F4_A_BYTES;
        const uint32_t ssf = sb + 2 * F4_BH_BYTES;
        const uint32_t t_sf0 = tmem_base + F4_SF_TMEM + slot * F4_SF_SLOT;
        const uint32_t acc = (kb != 0) ? 1u : 0u;
        // per 64-element step: A's scale atom (TMEM columns +0..3 of the step's group of
        // 12), then one M = 128, N = 256 MMA; B row n (0 .. 255) takes its scales from
        // column +4 + n / 32 of the group, where the copy warps put the two halves' atoms
        if (lane == 0) {
          if (4 * kb + 4 <= KS) {
#pragma unroll
            for (int k = 0; k < 4; ++k) tmem_cp_scales(t_sf0 + k * 12, sdesc_rows16(ssf + k * F4_ATOM));
#pragma unroll
            for (int k = 0; k < 4; ++k)  // 64 elements = 32 bytes of each row per step
              mma_nvf4(tmem_base, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32), idesc,
                       t_sf0 + k * 12, t_sf0 + k * 12 + 4, (acc | k) != 0 ? 1u : 0u);
          } else {  // a last stage of fewer than four steps
            const int nks = KS - 4 * kb;
            for (int k = 0; k < nks; ++k) tmem_cp_scales(t_sf0 + k * 12, sdesc_rows16(ssf + k * F4_ATOM));
            for (int k = 0; k < nks; ++k)
              mma_nvf4(tmem_base, sdesc_kmajor_sw128(sa + k * 32), sdesc_kmajor_sw128(sb + k * 32), idesc,
                       t_sf0 + k * 12, t_sf0 + k * 12 + 4, (acc | k) != 0 ? 1u : 0u);
          }
          mma_commit(&empty[stage]);    // frees the stage once these MMAs (and copies) have read it
          mma_commit(&sf_free[slot]);   // and the scale slot once the MMAs have read it
        }
        __syncwarp();
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
        if (++slot == 2) {
          slot = 0;
          slot_phase ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(tfull);  // accumulator ready for the epilogue
      __syncwarp();
      acc_phase ^= 1;
    }
    if (lane == 0) {
      mma_commit(done);  // completes when every MMA and copy issued above has finished
      drain_wait(done, 0, err, SITE_GEMM_TEARDOWN);
    }
    __syncwarp();
  } else if (warp >= 2 + NUM_EPI_WARPS) {
    // ---------------- B scale copies: warp 10 the atoms of B rows 0..127, warp 11 of rows
    // 128..255, into TMEM columns +4..7 / +8..11 of each step's group in the stage's slot.
    const int bh = warp - (2 + NUM_EPI_WARPS);
    int stage = 0;
    uint32_t phase = 0;
    int slot = 0;
    uint32_t slot_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, wc, SITE_GEMM_MMA)) ||
            !__all_sync(0xffffffffu, mbar_wait(&sf_free[slot], slot_phase ^ 1, wc, SITE_GEMM_MMA))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ssf = smem_u32(smem + stage * F4_STAGE) + F4_A_BYTES + 2 * F4_BH_BYTES;
        const uint32_t t_sf0 = tmem_base + F4_SF_TMEM + slot * F4_SF_SLOT + 4 + 4 * bh;
        if (lane == 0) {
          if (4 * kb + 4 <= KS) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tmem_cp_scales(t_sf0 + k * 12, sdesc_rows16(ssf + (4 + 4 * bh + k) * F4_ATOM));
          } else {
            const int nks = KS - 4 * kb;
            for (int k = 0; k < nks; ++k)
              tmem_cp_scales(t_sf0 + k * 12, sdesc_rows16(ssf + (4 + 4 * bh + k) * F4_ATOM));
          }
          mma_commit(&sf_ready[slot]);  // one of the slot's two arrivals, when the copies land
        }
        __syncwarp();
        if (++stage == NST) {
          stage = 0;
          phase ^= 1;
        }
        if (++slot == 2) {
          slot = 0;
          slot_phase ^= 1;
        }
      }
    }
    if (lane == 0) {
      mma_commit(done_cp);  // completes when every copy issued above has finished
      drain_wait(done_cp, 0, err, SITE_GEMM_TEARDOWN);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps
    const int quad = warp & 3;        // TMEM lanes this warp may access: 32*quad ..
    const int half = (warp - 2) / 4;  // 128-column half of the accumulator
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int mb, nb;
      tile_coords(tile, num_m, num_n, group, mb, nb);
      const bool got = mbar_wait(tfull, acc_phase, wc, SITE_GEMM_EPILOGUE);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      const int row = mb * F4_BM + quad * 32 + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
      // this warp's 128 accumulator columns into registers, then the accumulator goes back
      // to the MMA warp, so that the epilogue's work overlaps the next tile's products
      uint32_t a0[32], a1[32], a2[32], a3[32];
      const TmemAcc ta = Epi::tmem_acc(taddr, half);
      ta.ld32x2(0, 32, a0, a1);
      ta.ld32x2(64, 96, a2, a3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      const RegAcc ra{a0, a1, a2, a3};
      if constexpr (STG > 0)
        epi.apply_acc(row, nb, half, ra, M, stg_base + (warp - 2) * STG, lane, &tm_c);
      else
        epi.apply_acc(row, nb, half, ra, M);
      acc_phase ^= 1;
    }
    if constexpr (STG > 0) {  // this warp's TMA stores have completed
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

template <class Epi, bool DUAL>
cudaError_t set_smem_attr_fp4() {
  static_assert(f4_smem_bytes<Epi>() <= 232448, "shared memory per CTA");
  return cudaFuncSetAttribute(gemm_fp4_kernel<Epi, DUAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              f4_smem_bytes<Epi>());
}

// NVFP4 operands: tm_a / tm_b / tm_b2 are byte maps over the codes ([rows, K/2], 128-byte
// boxes); sf_* the scale atoms; K in elements (a multiple of 64).
template <class Epi, bool DUAL>
cudaError_t launch_fp4(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* b2, const uint8_t* sf_a,
                       const uint8_t* sf_b, const uint8_t* sf_b2, int M, int N, int num_n, int K, const Epi& epi,
                       int num_sms, int* err, cudaStream_t st, const CUtensorMap* c = nullptr) {
  if (StgOf<Epi>::value > 0 && !c) return cudaErrorInvalidValue;
  if (K % 64 || !sf_a || !sf_b || (DUAL && !sf_b2)) return cudaErrorInvalidValue;
  const int num_m = (M + F4_BM - 1) / F4_BM;
  const int tiles = num_m * num_n;
  if (tiles == 0) return cudaSuccess;
  // tile raster: B resident (n-fastest) when all of it fits and is no larger than A
  const long long a_all = static_cast<long long>(num_m) * F4_BM * (K / 2);
  const long long b_all = static_cast<long long>(num_n) * F4_BN * (K / 2);
  const int group = (b_all <= a_all && b_all <= (80ll << 20)) ? 1 : 16;
  const int grid = tiles < num_sms ? tiles : num_sms;  // persistent: one CTA per SM
  const int b_blocks = (N + 127) / 128;  // 128-row scale blocks of B (of W_gate / W_up for the SwiGLU GEMM)
  gemm_fp4_kernel<Epi, DUAL><<<grid, F4_THREADS, f4_smem_bytes<Epi>(), st>>>(
      *a, *b, *b2, c ? *c : *a, M, num_n, K, group, b_blocks, sf_a, sf_b, DUAL ? sf_b2 : sf_b, epi, err);
  return cudaGetLastError();
}

// Co-resident CTA pairs per instantiation, queried once by gemm_tc_init.
template <class Epi, bool DUAL>
struct MaxClusters {
  static int value;
};
template <class Epi, bool DUAL>
int MaxClusters<Epi, DUAL>::value = 0;

template <class Epi, bool DUAL>
cudaError_t set_smem_attr(int num_sms) {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<Epi, DUAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       smem_bytes<Epi>());
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * (num_sms / 2));
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes<Epi>();
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<Epi, DUAL>, &cfg);
  if (e != cudaSuccess) return e;
  MaxClusters<Epi, DUAL>::value = n;
  return cudaSuccess;
}

// Raster group for a call (see tile_coords). A pair tile reads a 256-row panel of A and a
// 256-row panel of B over all of K. When all of B fits the budget and is no larger than
// A, n-fastest order: the tiles that read one A panel run at about the same time and B
// stays in L2 (at 1024px this cut the DRAM reads of the down projection from 710 to 579
// MB and of the attention output projection from 187 to 136 MB). Otherwise groups of 16
// m-pairs, each group's A panels shared by its sweep over N (m-fastest order over all
// of M, to keep A resident instead, read more: 383 against 362 MB for the SwiGLU GEMM).
// The budget leaves room in the 126 MB L2 for the streamed operand and the epilogue.
int raster_group(int num_mp, int num_n, long long k_bytes) {
  constexpr long long kResident = 80ll << 20;
  const long long panel = 256ll * k_bytes;
  const long long a_all = num_mp * panel, b_all = num_n * panel;
  return (b_all <= a_all && b_all <= kResident) ? 1 : 16;
}

template <class Epi, bool DUAL>
cudaError_t launch(const CUtensorMap* a, const CUtensorMap* b, const CUtensorMap* b2, int M, int num_n, int K,
                   const Epi& epi, int num_sms, int* err, cudaStream_t st, const CUtensorMap* c = nullptr) {
  static_assert(smem_bytes<Epi>() <= 232448, "shared memory per CTA");
  if (StgOf<Epi>::value > 0 && !c) return cudaErrorInvalidValue;
  const int num_m = (M + BM - 1) / BM;
  const int tiles = ((num_m + 1) / 2) * num_n;  // pair tiles
  if (tiles == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem_bytes<Epi>();
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent grid: as many CTA pairs as fit on the device at once (queried at init)
  const int max_clusters = MaxClusters<Epi, DUAL>::value > 0 ? MaxClusters<Epi, DUAL>::value : num_sms / 2;
  const int pairs = tiles < max_clusters ? tiles : max_clusters;
  cfg.gridDim = dim3(2 * pairs);
  const int group = raster_group((num_m + 1) / 2, num_n, static_cast<long long>(K) * (Epi::kS8 ? 1 : 2));
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<Epi, DUAL>, *a, *b, *b2, c ? *c : *a, M, num_n, K, group, epi,
                            err);
}

}  // namespace

int gemm_tc_smem_bytes() { return smem_bytes<EpiResidAttnT<false>>(); }

template <bool S8>
cudaError_t gemm_tc_init_set(int num_sms) {
  cudaError_t e;
  if ((e = set_smem_attr<EpiQKVGT<S8>, false>(num_sms)) != cudaSuccess) return e;
  if ((e = set_smem_attr<EpiResidAttnT<S8>, false>(num_sms)) != cudaSuccess) return e;
  if ((e = set_smem_attr<EpiResidMlpT<S8>, false>(num_sms)) != cudaSuccess) return e;
  return set_smem_attr<EpiSwiGLUT<S8>, true>(num_sms);
}

cudaError_t gemm_fp4_init() {
  cudaError_t e;
  if ((e = set_smem_attr_fp4<EpiQKVGT<true>, false>()) != cudaSuccess) return e;
  if ((e = set_smem_attr_fp4<EpiResidAttnT<true>, false>()) != cudaSuccess) return e;
  if ((e = set_smem_attr_fp4<EpiResidMlpT<true>, false>()) != cudaSuccess) return e;
  return set_smem_attr_fp4<EpiSwiGLUT<true>, true>();
}

cudaError_t gemm_tc_init(int num_sms) {
  cudaError_t e = gemm_tc_init_set<false>(num_sms);
  if (e == cudaSuccess) e = gemm_tc_init_set<true>(num_sms);
  if (e == cudaSuccess) e = set_smem_attr<EpiSwiGLUBwd, false>(num_sms);
  if (e == cudaSuccess) e = set_smem_attr<EpiGateBwd, false>(num_sms);
  return e != cudaSuccess ? e : set_smem_attr<EpiPlain, false>(num_sms);
}

cudaError_t launch_gemm_gate_bwd(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K, const float* o,
                                 const void* g, void* d_o, void* d_P, int ldp, int goff, float* D, int num_sms,
                                 int* err, cudaStream_t st) {
  const int nq = f.n_q * 128;
  if (f.T <= 0) return cudaSuccess;
  if (ldp % 8 || goff % 8) return cudaErrorInvalidValue;
  EpiGateBwd epi{f, o, reinterpret_cast<const bf16*>(g), reinterpret_cast<bf16*>(d_o), reinterpret_cast<bf16*>(d_P),
                 ldp, goff, D};
  return launch<EpiGateBwd, false>(tm_a, tm_b, tm_b, f.T, (nq + BN - 1) / BN, K, epi, num_sms, err, st);
}

cudaError_t launch_gemm_swiglu_bwd(const CUtensorMap* tm_a, const CUtensorMap* tm_b, int M, int F, int K,
                                   const float* a, const float* u, void* d_au, int num_sms, int* err,
                                   cudaStream_t st) {
  if (M <= 0 || F <= 0) return cudaSuccess;
  if (F % 8) return cudaErrorInvalidValue;
  EpiSwiGLUBwd epi{a, u, reinterpret_cast<bf16*>(d_au), F};
  return launch<EpiSwiGLUBwd, false>(tm_a, tm_b, tm_b, M, (F + BN - 1) / BN, K, epi, num_sms, err, st);
}

cudaError_t launch_gemm_plain(const CUtensorMap* tm_a, const CUtensorMap* tm_b, int M, int N, int K, float* C,
                              long long ldc, float alpha, int accumulate, int num_sms, int* err, cudaStream_t st) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  if (ldc % 4 || ldc < N) return cudaErrorInvalidValue;
  EpiPlain epi{C, ldc, N, accumulate, alpha};
  return launch<EpiPlain, false>(tm_a, tm_b, tm_b, M, (N + BN - 1) / BN, K, epi, num_sms, err, st);
}

cudaError_t launch_gemm_qkvg(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int N,
                             const QkvgDst& dst, const Deq* dq, int num_sms, int* err, cudaStream_t st) {
  const int num_n = (N + BN - 1) / BN;
  if (dq) {
    EpiQKVGT<true> epi{f, dst, N, *dq};
    return launch<EpiQKVGT<true>, false>(tm_a, tm_b, tm_b, f.T, num_n, f.d, epi, num_sms, err, st);
  }
  EpiQKVGT<false> epi{f, dst, N, Deq{}};
  return launch<EpiQKVGT<false>, false>(tm_a, tm_b, tm_b, f.T, num_n, f.d, epi, num_sms, err, st);
}

cudaError_t launch_gemm_resid_attn(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K, RowSrc x,
                                   const float* mod_shared, const float* mod_bias, const CUtensorMap* tm_h1,
                                   const Deq* dq, float* pre, int num_sms, int* err, cudaStream_t st) {
  const int num_n = (f.d + BN - 1) / BN;
  if (dq) {
    EpiResidAttnT<true> epi{f, x, mod_shared, mod_bias, 2, *dq};
    return launch<EpiResidAttnT<true>, false>(tm_a, tm_b, tm_b, f.T, num_n, K, epi, num_sms, err, st, tm_h1);
  }
  EpiResidAttnT<false> epi{f, x, mod_shared, mod_bias, 2, Deq{}, pre};
  return launch<EpiResidAttnT<false>, false>(tm_a, tm_b, tm_b, f.T, num_n, K, epi, num_sms, err, st, tm_h1);
}

cudaError_t launch_gemm_resid_mlp(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_b, int K,
                                  const float* h1, const float* mod_shared, const float* mod_bias,
                                  const CUtensorMap* tm_out, const Deq* dq, float* pre, int num_sms, int* err,
                                  cudaStream_t st) {
  const int num_n = (f.d + BN - 1) / BN;
  const RowSrc res{nullptr, nullptr, h1};
  if (dq) {
    EpiResidMlpT<true> epi{f, res, mod_shared, mod_bias, 5, *dq};
    return launch<EpiResidMlpT<true>, false>(tm_a, tm_b, tm_b, f.T, num_n, K, epi, num_sms, err, st, tm_out);
  }
  EpiResidMlpT<false> epi{f, res, mod_shared, mod_bias, 5, Deq{}, pre};
  return launch<EpiResidMlpT<false>, false>(tm_a, tm_b, tm_b, f.T, num_n, K, epi, num_sms, err, st, tm_out);
}

cudaError_t launch_gemm_swiglu(const Fwd& f, const CUtensorMap* tm_a, const CUtensorMap* tm_gate,
                               const CUtensorMap* tm_up, void* hmid, float* rowamax, const Deq* dq, float* pre_a,
                               float* pre_u, int num_sms, int* err, cudaStream_t st) {
  const int num_n = (f.F + 127) / 128;
  if (dq) {
    EpiSwiGLUT<true> epi{f.F, reinterpret_cast<bf16*>(hmid), rowamax, *dq};
    return launch<EpiSwiGLUT<true>, true>(tm_a, tm_gate, tm_up, f.T, num_n, f.d, epi, num_sms, err, st);
  }
  EpiSwiGLUT<false> epi{f.F, reinterpret_cast<bf16*>(hmid), rowamax, Deq{}, pre_a, pre_u};
  return launch<EpiSwiGLUT<false>, true>(tm_a, tm_gate, tm_up, f.T, num_n, f.d, epi, num_sms, err, st);
}

// ---- NVFP4 launchers (Op4: codes' tensor map, scale atoms; dq: the tensor scales)
cudaError_t launch_gemm_qkvg_fp4(const Fwd& f, const Op4& a, const Op4& b, int N, const QkvgDst& dst, const Deq& dq,
                                 int num_sms, int* err, cudaStream_t st) {
  const int num_n = (N + BN - 1) / BN;
  EpiQKVGT<true> epi{f, dst, N, dq};
  return launch_fp4<EpiQKVGT<true>, false>(a.map, b.map, b.map, a.sf, b.sf, b.sf, f.T, N, num_n, f.d, epi, num_sms,
                                           err, st);
}

cudaError_t launch_gemm_resid_attn_fp4(const Fwd& f, const Op4& a, const Op4& b, int K, RowSrc x,
                                       const float* mod_shared, const float* mod_bias, const CUtensorMap* tm_h1,
                                       const Deq& dq, int num_sms, int* err, cudaStream_t st) {
  const int num_n = (f.d + BN - 1) / BN;
  EpiResidAttnT<true> epi{f, x, mod_shared, mod_bias, 2, dq};
  return launch_fp4<EpiResidAttnT<true>, false>(a.map, b.map, b.map, a.sf, b.sf, b.sf, f.T, f.d, num_n, K, epi,
                                                num_sms, err, st, tm_h1);
}

cudaError_t launch_gemm_resid_mlp_fp4(const Fwd& f, const Op4& a, const Op4& b, int K, const float* h1,
                                      const float* mod_shared, const float* mod_bias, const CUtensorMap* tm_out,
                                      const Deq& dq, int num_sms, int* err, cudaStream_t st) {
  const int num_n = (f.d + BN - 1) / BN;
  const RowSrc res{nullptr, nullptr, h1};
  EpiResidMlpT<true> epi{f, res, mod_shared, mod_bias, 5, dq};
  return launch_fp4<EpiResidMlpT<true>, false>(a.map, b.map, b.map, a.sf, b.sf, b.sf, f.T, f.d, num_n, K, epi,
                                               num_sms, err, st, tm_out);
}

cudaError_t launch_gemm_swiglu_fp4(const Fwd& f, const Op4& a, const Op4& gate, const Op4& up, void* hmid,
                                   float* rowamax, const Deq& dq, int num_sms, int* err, cudaStream_t st) {
  const int num_n = (f.F + 127) / 128;
  EpiSwiGLUT<true> epi{f.F, reinterpret_cast<bf16*>(hmid), rowamax, dq};
  return launch_fp4<EpiSwiGLUT<true>, true>(a.map, gate.map, up.map, a.sf, gate.sf, up.sf, f.T, f.F, num_n, f.d,
                                            epi, num_sms, err, st);
}

}  // namespace kd
