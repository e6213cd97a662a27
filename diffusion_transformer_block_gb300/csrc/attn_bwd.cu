// Flash-style backward of the gated GQA attention, tcgen05 + TMA, sm_103a (Krea 2
// Technical Report, "Transformer block": GQA attention whose output is scaled by a
// sigmoid gate; the gate's own gradient is taken before these kernels, which start from
// d_o, the gradient of the ungated attention output).
//
// With S = Q K^T (raw scores), c = log2(e)/sqrt(hd), the forward's per-row normaliser
// lse = m + log2(l) (scaled-log2 units) and D = rowsum(d_o * o):
//   P  = exp2(c S - lse)           (the forward's softmax, recomputed tile by tile)
//   dP = d_o V^T
//   dS = P (dP - D)                 (gradient of the raw scores, times sqrt(hd))
//   dV = P^T d_o,   dK = dS^T Q / sqrt(hd),   dQ = dS K / sqrt(hd)
// Nothing of size L x L reaches memory: each 128 x 128 score tile lives in TMEM.
//
// attn_bwd_kv_kernel — one CTA per (batch, KV head, 128-key tile); it walks every query
// tile of the KV group's G heads:
//   S^T  = K Q^T        (tensor core, smem x smem, fp32 in TMEM)
//   dP^T = V d_o^T
//   P^T  = exp2(c S^T - lse), dS^T = P^T (dP^T - D)   (8 warps, one key row per thread and
//                        64 query columns per warp; P^T and dS^T go back into TMEM as bf16
//                        over the columns they were computed from)
//   dV  += P^T (d_o^T)^T  and  dK += dS^T (Q^T)^T     (A operand from TMEM; d_o^T and Q^T,
//                        head-dim-major copies, are the K-major B operands)
// The tensor core runs one CTA's MMAs in issue order, and the issue order
// S^T(n), dK(n-1), dP^T(n), dV(n), S^T(n+1), ... gives the element warps the time of two
// products for each half of their work: P^T(n) while dK(n-1) and dP^T(n) run, dS^T(n)
// while dV(n) and S^T(n+1) run.
//
// attn_bwd_q_kernel — one CTA per (batch, query head, 128-query tile); it walks the key
// tiles: S = Q K^T (two TMEM buffers), dP = d_o V^T, dS = P (dP - D) back into S's
// buffer as bf16, dQ += dS (K^T)^T. Issue order S(j+1), dQ(j), dP(j+1), ...
//
// Shared memory: two fixed 32 KB tiles (K and V, or Q and d_o) and a 5-slot ring of
// 32 KB tiles streamed in the order the MMA thread consumes them. Warps 0-7: element
// work and epilogue, warp 8: TMA, warp 9: TMEM allocation + MMA issue.
#include "common.cuh"
#include "internal.h"

namespace kd {
namespace {

constexpr int HD = 128;   // head dim
constexpr int BT = 128;   // rows of a query or key tile
constexpr int TILE_BYTES = 128 * 128 * 2;
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr int NSLOT = 5;
constexpr int NUM_THREADS = 320;
constexpr int SMEM_FIX = 0;
constexpr int SMEM_RING = SMEM_FIX + 2 * TILE_BYTES;
constexpr int SMEM_BAR = SMEM_RING + NSLOT * TILE_BYTES;
constexpr int SMEM_BYTES = SMEM_BAR + 256 + 1024;
constexpr int N_ELEM_THREADS = 256;

struct BwdArgs {
  int B, L, Lp, n_q, n_kv, G, nqt, nkt;
  float scale_log2;  // log2(e) / sqrt(hd)
  float scale;       // 1 / sqrt(hd)
  const float* lse;  // [B n_q, Lp]
  const float* D;    // [B n_q, Lp]
  float* dq;         // [B n_q, L, hd]
  float* dk;         // [B n_kv, L, hd]
  float* dv;         // [B n_kv, L, hd]
  int* err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err, int site) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, site);
      return;
    }
  }
}

// D (+)= A B^T over K = 128: A and B are 128-row K-major tiles in shared memory, each two
// 64-column swizzled halves.
__device__ __forceinline__ void mma_ss_tile(uint32_t d, uint32_t sa, uint32_t sb, uint32_t idesc, bool acc) {
#pragma unroll
  for (int kh = 0; kh < 2; ++kh)
#pragma unroll
    for (int ks = 0; ks < 4; ++ks)
      mma_bf16_ss(d, sdesc_kmajor_sw128(sa + kh * HALF_BYTES + ks * 32), sdesc_kmajor_sw128(sb + kh * HALF_BYTES + ks * 32),
                  idesc, (acc || (kh | ks) != 0) ? 1u : 0u);
}

// D (+)= A B^T over K = 128 with A = 128 x 128 bf16 in TMEM, packed two per column: K
// elements 0-63 in columns ta .. ta+31, 64-127 in columns ta+64 .. ta+95 (each element
// warp packs its 64 columns over the first half of them). B: K-major tile in smem.
__device__ __forceinline__ void mma_ts_tile(uint32_t d, uint32_t ta, uint32_t sb, uint32_t idesc, bool acc) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_bf16_ts(d, ta + (ks >> 2) * 64 + (ks & 3) * 8,
                sdesc_kmajor_sw128(sb + (ks >> 2) * HALF_BYTES + (ks & 3) * 32), idesc,
                (acc || ks != 0) ? 1u : 0u);
}

// Packs 64 fp32 values to bf16 pairs and stores them over the first 32 of the thread's 64
// TMEM columns at taddr (warp-collective), then waits for the store.
__device__ __forceinline__ void store_packed(uint32_t taddr, const float (&v)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  tmem_st32(taddr, pk);
  tmem_st_wait();
}

// 64 consecutive fp32 TMEM columns of this thread's lane
__device__ __forceinline__ void load64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[32], q[32];
  tmem_ld32x2(taddr, taddr + 32, r, q);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = __uint_as_float(r[i]);
    v[32 + i] = __uint_as_float(q[i]);
  }
}

// Writes 64 fp32 values (times s) to a 16-byte aligned row segment.
__device__ __forceinline__ void store_row64(float* dst, const float (&v)[64], float s) {
  float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 16; ++i) d4[i] = make_float4(v[4 * i] * s, v[4 * i + 1] * s, v[4 * i + 2] * s, v[4 * i + 3] * s);
}

// ====================================================================== dK, dV
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_qt, const __grid_constant__ CUtensorMap tm_dot,
                       BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SMEM_BAR);
  uint64_t* bar_kv = bar + 0;             // K and V landed
  uint64_t* full = bar + 1;               // [NSLOT]
  uint64_t* empty = full + NSLOT;         // [NSLOT]
  uint64_t* s_full = empty + NSLOT;       // S^T(n) landed
  uint64_t* dp_full = s_full + 1;         // dP^T(n) landed
  uint64_t* p_full = dp_full + 1;         // P^T(n) in TMEM (256 arrivals)
  uint64_t* ds_full = p_full + 1;         // dS^T(n) in TMEM (256 arrivals)
  uint64_t* acc_done = ds_full + 1;       // the last dK / dV product landed
  uint64_t* done = acc_done + 1;          // every MMA issued has finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kt = blockIdx.x % a.nkt;
  const int bk = blockIdx.x / a.nkt;  // b * n_kv + kv
  const int b = bk / a.n_kv, kvh = bk - b * a.n_kv;
  const int NT = a.G * a.nqt;          // query tiles of the group
  auto plane_of = [&](int n) { return b * a.n_q + kvh * a.G + n / a.nqt; };
  auto qt_of = [&](int n) { return n % a.nqt; };

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(dp_full, 1);
    mbar_init(p_full, N_ELEM_THREADS);
    mbar_init(ds_full, N_ELEM_THREADS);
    mbar_init(acc_done, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, a.err};
  // ring tiles, in the order the MMA thread consumes them:
  //   Q(0), dO(0), dO^T(0), then per n >= 1: Q(n), Q^T(n-1), dO(n), dO^T(n); finally Q^T(NT-1)
  enum Kind { KQ = 0, KDO = 1, KDOT = 2, KQT = 3 };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA loads
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_qt);
      tma_prefetch_desc(&tm_dot);
      mbar_arrive_expect_tx(bar_kv, 2 * TILE_BYTES);
      for (int h2 = 0; h2 < 2; ++h2) {
        tma_load_3d(smem + SMEM_FIX + h2 * HALF_BYTES, &tm_k, bar_kv, h2 * 64, kt * BT, bk);
        tma_load_3d(smem + SMEM_FIX + TILE_BYTES + h2 * HALF_BYTES, &tm_v, bar_kv, h2 * 64, kt * BT, bk);
      }
      int ld = 0;
      auto load = [&](int kind, int n) -> bool {
        const int slot = ld % NSLOT;
        if (!mbar_wait(&empty[slot], static_cast<uint32_t>(((ld / NSLOT) & 1) ^ 1), wc, SITE_ATTN_LOAD)) return false;
        uint8_t* dst = smem + SMEM_RING + slot * TILE_BYTES;
        mbar_arrive_expect_tx(&full[slot], TILE_BYTES);
        const int pl = plane_of(n), q0 = qt_of(n) * BT;
        for (int h2 = 0; h2 < 2; ++h2) {
          if (kind == KQ) tma_load_3d(dst + h2 * HALF_BYTES, &tm_q, &full[slot], h2 * 64, q0, pl);
          else if (kind == KDO) tma_load_3d(dst + h2 * HALF_BYTES, &tm_do, &full[slot], h2 * 64, q0, pl);
          else if (kind == KDOT) tma_load_3d(dst + h2 * HALF_BYTES, &tm_dot, &full[slot], q0 + h2 * 64, 0, pl);
          else tma_load_3d(dst + h2 * HALF_BYTES, &tm_qt, &full[slot], q0 + h2 * 64, 0, pl);
        }
        ++ld;
        return true;
      };
      bool ok = load(KQ, 0) && load(KDO, 0) && load(KDOT, 0);
      for (int n = 1; ok && n < NT; ++n) ok = load(KQ, n) && load(KQT, n - 1) && load(KDO, n) && load(KDOT, n);
      if (ok) load(KQT, NT - 1);
      // every copy started here has landed before the CTA exits
      drain_wait(bar_kv, 0, a.err, SITE_ATTN_TEARDOWN);
      for (int i = (ld > NSLOT ? ld - NSLOT : 0); i < ld; ++i)
        drain_wait(&full[i % NSLOT], static_cast<uint32_t>((i / NSLOT) & 1), a.err, SITE_ATTN_TEARDOWN);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t sK = smem_u32(smem + SMEM_FIX), sV = sK + TILE_BYTES, sRing = smem_u32(smem + SMEM_RING);
      const uint32_t tS = tmem, tdP = tmem + 128, tdV = tmem + 256, tdK = tmem + 384;
      int cs = 0;  // ring tiles consumed
      int slot = 0;
      auto acquire = [&](uint32_t& s_addr) -> bool {
        slot = cs % NSLOT;
        if (!mbar_wait(&full[slot], static_cast<uint32_t>((cs / NSLOT) & 1), wc, SITE_ATTN_MMA)) return false;
        s_addr = sRing + slot * TILE_BYTES;
        ++cs;
        return true;
      };
      bool ok = mbar_wait(bar_kv, 0, wc, SITE_ATTN_MMA);
      uint32_t sA = 0;
      for (int n = 0; ok && n < NT; ++n) {
        // S^T(n) = K Q(n)^T over the columns of P^T(n-1): dV(n-1), issued before, read them
        if (!(ok = acquire(sA))) break;
        tc_fence_after();
        mma_ss_tile(tS, sK, sA, idesc, false);
        mma_commit(s_full);
        mma_commit(&empty[slot]);
        if (n > 0) {  // dK += dS^T(n-1) Q^T(n-1)
          if (!(ok = acquire(sA))) break;
          if (!(ok = mbar_wait(ds_full, static_cast<uint32_t>((n - 1) & 1), wc, SITE_ATTN_MMA))) break;
          tc_fence_after();
          mma_ts_tile(tdK, tdP, sA, idesc, n > 1);
          mma_commit(&empty[slot]);
        }
        // dP^T(n) = V dO(n)^T over the columns of dS^T(n-1): dK(n-1) was issued before
        if (!(ok = acquire(sA))) break;
        tc_fence_after();
        mma_ss_tile(tdP, sV, sA, idesc, false);
        mma_commit(dp_full);
        mma_commit(&empty[slot]);
        // dV += P^T(n) dO^T(n)
        if (!(ok = acquire(sA))) break;
        if (!(ok = mbar_wait(p_full, static_cast<uint32_t>(n & 1), wc, SITE_ATTN_MMA))) break;
        tc_fence_after();
        mma_ts_tile(tdV, tS, sA, idesc, n > 0);
        mma_commit(&empty[slot]);
      }
      if (ok && (ok = acquire(sA)) && (ok = mbar_wait(ds_full, static_cast<uint32_t>((NT - 1) & 1), wc, SITE_ATTN_MMA))) {
        tc_fence_after();
        mma_ts_tile(tdK, tdP, sA, idesc, NT > 1);
        mma_commit(&empty[slot]);
        mma_commit(acc_done);
      }
      mma_commit(done);
      drain_wait(done, 0, a.err, SITE_ATTN_TEARDOWN);
    }
  } else {
    // ------------------------------------------------------------ P^T, dS^T; epilogue
    const int quad = warp & 3, half = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + half * 64;
    const uint32_t tdP = tmem + lane_off + 128 + half * 64;
    bool ok = true;
    for (int n = 0; n < NT; ++n) {
      const int pl = plane_of(n), q0 = qt_of(n) * BT + half * 64;
      const int qvalid = a.L - q0;  // query columns of this warp's half inside the sequence
      const float4* lse4 = reinterpret_cast<const float4*>(a.lse + static_cast<size_t>(pl) * a.Lp + q0);
      const float4* D4 = reinterpret_cast<const float4*>(a.D + static_cast<size_t>(pl) * a.Lp + q0);
      const bool got = mbar_wait(s_full, static_cast<uint32_t>(n & 1), wc, SITE_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      float p[64];
      load64(tS, p);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 l4 = 4 * j < qvalid ? __ldg(lse4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int i = 4 * j + e;
          p[i] = i < qvalid ? ex2(fmaf(p[i], a.scale_log2, -lv[e])) : 0.0f;
        }
      }
      store_packed(tS, p);
      tc_fence_before();
      mbar_arrive(p_full);
      const bool got2 = mbar_wait(dp_full, static_cast<uint32_t>(n & 1), wc, SITE_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, got2)) { ok = false; break; }
      tc_fence_after();
      float dp[64];
      load64(tdP, dp);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 d4 = 4 * j < qvalid ? __ldg(D4 + j) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) dp[4 * j + e] = p[4 * j + e] * (dp[4 * j + e] - dv[e]);
      }
      store_packed(tdP, dp);
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (ok) {
      const bool w = mbar_wait(acc_done, 0, wc, SITE_ATTN_SOFTMAX);
      ok = __all_sync(0xffffffffu, w);
    }
    if (ok) {
      tc_fence_after();
      const int key = kt * BT + quad * 32 + lane;
      float v[64];
      load64(tmem + lane_off + 256 + half * 64, v);
      if (key < a.L) store_row64(a.dv + (static_cast<size_t>(bk) * a.L + key) * HD + half * 64, v, 1.0f);
      load64(tmem + lane_off + 384 + half * 64, v);
      if (key < a.L) store_row64(a.dk + (static_cast<size_t>(bk) * a.L + key) * HD + half * 64, v, a.scale);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ====================================================================== dQ
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_kt, BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SMEM_BAR);
  uint64_t* bar_q = bar + 0;              // Q and dO landed
  uint64_t* full = bar + 1;               // [NSLOT]
  uint64_t* empty = full + NSLOT;         // [NSLOT]
  uint64_t* s_full = empty + NSLOT;       // [2] S(j) landed in buffer j & 1
  uint64_t* dp_full = s_full + 2;         // dP(j) landed
  uint64_t* ds_full = dp_full + 1;        // dS(j) in TMEM (256 arrivals)
  uint64_t* acc_done = ds_full + 1;       // the last dQ product landed
  uint64_t* done = acc_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_group = a.G * a.nqt;
  const int bk = blockIdx.x / per_group;  // b * n_kv + kv
  const int r = blockIdx.x - bk * per_group;
  const int b = bk / a.n_kv, kvh = bk - b * a.n_kv;
  const int plane = b * a.n_q + kvh * a.G + r / a.nqt;
  const int qt = r % a.nqt;
  const int nkt = a.nkt;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&s_full[0], 1);
    mbar_init(&s_full[1], 1);
    mbar_init(dp_full, 1);
    mbar_init(ds_full, N_ELEM_THREADS);
    mbar_init(acc_done, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, a.err};
  // ring tiles in consumption order: K(0), V(0), then per j: K(j+1), K^T(j), V(j+1)
  // (K(j+1) and V(j+1) only while j + 1 < nkt)
  enum Kind { KK = 0, KV = 1, KKT = 2 };

  if (warp == 8) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_kt);
      mbar_arrive_expect_tx(bar_q, 2 * TILE_BYTES);
      for (int h2 = 0; h2 < 2; ++h2) {
        tma_load_3d(smem + SMEM_FIX + h2 * HALF_BYTES, &tm_q, bar_q, h2 * 64, qt * BT, plane);
        tma_load_3d(smem + SMEM_FIX + TILE_BYTES + h2 * HALF_BYTES, &tm_do, bar_q, h2 * 64, qt * BT, plane);
      }
      int ld = 0;
      auto load = [&](int kind, int j) -> bool {
        const int slot = ld % NSLOT;
        if (!mbar_wait(&empty[slot], static_cast<uint32_t>(((ld / NSLOT) & 1) ^ 1), wc, SITE_ATTN_LOAD)) return false;
        uint8_t* dst = smem + SMEM_RING + slot * TILE_BYTES;
        mbar_arrive_expect_tx(&full[slot], TILE_BYTES);
        for (int h2 = 0; h2 < 2; ++h2) {
          if (kind == KK) tma_load_3d(dst + h2 * HALF_BYTES, &tm_k, &full[slot], h2 * 64, j * BT, bk);
          else if (kind == KV) tma_load_3d(dst + h2 * HALF_BYTES, &tm_v, &full[slot], h2 * 64, j * BT, bk);
          else tma_load_3d(dst + h2 * HALF_BYTES, &tm_kt, &full[slot], j * BT + h2 * 64, 0, bk);
        }
        ++ld;
        return true;
      };
      bool ok = load(KK, 0) && load(KV, 0);
      for (int j = 0; ok && j < nkt; ++j) {
        const bool more = j + 1 < nkt;
        if (more) ok = load(KK, j + 1);
        if (ok) ok = load(KKT, j);
        if (ok && more) ok = load(KV, j + 1);
      }
      drain_wait(bar_q, 0, a.err, SITE_ATTN_TEARDOWN);
      for (int i = (ld > NSLOT ? ld - NSLOT : 0); i < ld; ++i)
        drain_wait(&full[i % NSLOT], static_cast<uint32_t>((i / NSLOT) & 1), a.err, SITE_ATTN_TEARDOWN);
    }
  } else if (warp == 9) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t sQ = smem_u32(smem + SMEM_FIX), sdO = sQ + TILE_BYTES, sRing = smem_u32(smem + SMEM_RING);
      const uint32_t tdP = tmem + 256, tdQ = tmem + 384;
      int cs = 0;
      int slot = 0;
      auto acquire = [&](uint32_t& s_addr) -> bool {
        slot = cs % NSLOT;
        if (!mbar_wait(&full[slot], static_cast<uint32_t>((cs / NSLOT) & 1), wc, SITE_ATTN_MMA)) return false;
        s_addr = sRing + slot * TILE_BYTES;
        ++cs;
        return true;
      };
      uint32_t sA = 0;
      bool ok = mbar_wait(bar_q, 0, wc, SITE_ATTN_MMA) && acquire(sA);
      if (ok) {  // S(0) = Q K(0)^T
        tc_fence_after();
        mma_ss_tile(tmem, sQ, sA, idesc, false);
        mma_commit(&s_full[0]);
        mma_commit(&empty[slot]);
        ok = acquire(sA);
      }
      if (ok) {  // dP(0) = dO V(0)^T
        tc_fence_after();
        mma_ss_tile(tdP, sdO, sA, idesc, false);
        mma_commit(dp_full);
        mma_commit(&empty[slot]);
      }
      for (int j = 0; ok && j < nkt; ++j) {
        const bool more = j + 1 < nkt;
        if (more) {  // S(j+1) into the other buffer: dQ(j-1), issued before, read its dS
          if (!(ok = acquire(sA))) break;
          tc_fence_after();
          mma_ss_tile(tmem + ((j + 1) & 1) * 128, sQ, sA, idesc, false);
          mma_commit(&s_full[(j + 1) & 1]);
          mma_commit(&empty[slot]);
        }
        // dQ += dS(j) K^T(j)
        if (!(ok = acquire(sA))) break;
        if (!(ok = mbar_wait(ds_full, static_cast<uint32_t>(j & 1), wc, SITE_ATTN_MMA))) break;
        tc_fence_after();
        mma_ts_tile(tdQ, tmem + (j & 1) * 128, sA, idesc, j > 0);
        mma_commit(&empty[slot]);
        if (more) {  // dP(j+1): the element warps read dP(j) before they signalled dS(j)
          if (!(ok = acquire(sA))) break;
          tc_fence_after();
          mma_ss_tile(tdP, sdO, sA, idesc, false);
          mma_commit(dp_full);
          mma_commit(&empty[slot]);
        }
      }
      if (ok) mma_commit(acc_done);
      mma_commit(done);
      drain_wait(done, 0, a.err, SITE_ATTN_TEARDOWN);
    }
  } else {
    // ------------------------------------------------------------ P, dS; epilogue
    const int quad = warp & 3, half = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int q = qt * BT + quad * 32 + lane;
    const bool qv = q < a.L;
    const float lse_r = qv ? a.lse[static_cast<size_t>(plane) * a.Lp + q] : 0.0f;
    const float D_r = qv ? a.D[static_cast<size_t>(plane) * a.Lp + q] : 0.0f;
    const uint32_t tdP = tmem + lane_off + 256 + half * 64;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const uint32_t tS = tmem + lane_off + (j & 1) * 128 + half * 64;
      const int kvalid = a.L - j * BT - half * 64;  // key columns of this half inside the sequence
      const bool got = mbar_wait(&s_full[j & 1], static_cast<uint32_t>((j >> 1) & 1), wc, SITE_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      tc_fence_after();
      float p[64];
      load64(tS, p);
#pragma unroll
      for (int i = 0; i < 64; ++i) p[i] = i < kvalid ? ex2(fmaf(p[i], a.scale_log2, -lse_r)) : 0.0f;
      const bool got2 = mbar_wait(dp_full, static_cast<uint32_t>(j & 1), wc, SITE_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, got2)) { ok = false; break; }
      tc_fence_after();
      float dp[64];
      load64(tdP, dp);
#pragma unroll
      for (int i = 0; i < 64; ++i) dp[i] = p[i] * (dp[i] - D_r);
      store_packed(tS, dp);
      tc_fence_before();
      mbar_arrive(ds_full);
    }
    if (ok) {
      const bool w = mbar_wait(acc_done, 0, wc, SITE_ATTN_SOFTMAX);
      ok = __all_sync(0xffffffffu, w);
    }
    if (ok) {
      tc_fence_after();
      float v[64];
      load64(tmem + lane_off + 384 + half * 64, v);
      if (qv) store_row64(a.dq + (static_cast<size_t>(plane) * a.L + q) * HD + half * 64, v, a.scale);
    }
    tc_fence_before();
  }
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t attn_bwd_init() {
  cudaError_t e = cudaFuncSetAttribute(attn_bwd_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(attn_bwd_q_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  return e;
}

cudaError_t launch_attn_bwd(const Fwd& f, const CUtensorMap* tm_q, const CUtensorMap* tm_do, const CUtensorMap* tm_k,
                            const CUtensorMap* tm_v, const CUtensorMap* tm_qt, const CUtensorMap* tm_dot,
                            const CUtensorMap* tm_kt, const float* lse, const float* D, float* dq, float* dk,
                            float* dv, int* err, cudaStream_t st) {
  BwdArgs a;
  a.B = f.B;
  a.L = f.L;
  a.Lp = f.Lp;
  a.n_q = f.n_q;
  a.n_kv = f.n_kv;
  a.G = f.n_q / f.n_kv;
  a.nqt = (f.L + BT - 1) / BT;
  a.nkt = (f.L + BT - 1) / BT;
  a.scale = 1.0f / sqrtf(static_cast<float>(HD));
  a.scale_log2 = 1.4426950408889634f * a.scale;
  a.lse = lse;
  a.D = D;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.err = err;
  const long long kv_units = static_cast<long long>(f.B) * f.n_kv * a.nkt;
  const long long q_units = static_cast<long long>(f.B) * f.n_q * a.nqt;
  if (kv_units == 0) return cudaSuccess;
  attn_bwd_kv_kernel<<<static_cast<unsigned>(kv_units), NUM_THREADS, SMEM_BYTES, st>>>(*tm_k, *tm_v, *tm_q, *tm_do,
                                                                                     *tm_qt, *tm_dot, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  attn_bwd_q_kernel<<<static_cast<unsigned>(q_units), NUM_THREADS, SMEM_BYTES, st>>>(*tm_q, *tm_do, *tm_k, *tm_v,
                                                                                    *tm_kt, a);
  return cudaGetLastError();
}

}  // namespace kd
