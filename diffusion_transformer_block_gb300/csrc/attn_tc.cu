// Flash-style GQA attention with the sigmoid output gate, tcgen05 + TMA, sm_103a
// (Krea 2 Technical Report, "Transformer block": GQA with gated attention output; the
// pass is pure prefill, so there is no mask and no KV cache).
//
// Work unit = two 128-row query tiles of the same (batch, KV group): both tiles read the
// same K/V tiles from shared memory, so every K/V tile loaded is used by two query
// tiles; the other query tiles of the group re-read the group's K/V from L2.
//
// Per unit, for each 128-key K/V tile j and query tile t = 0, 1:
//   S_t  = Q_t K_j^T        tensor core, both operands in shared memory, fp32 in TMEM
//   P_t  = exp2(S_t * log2(e)/sqrt(hd) - m_t)
//                           softmax warpgroup t, one thread per row: S read from TMEM,
//                           P written back as bf16 over the first 64 columns of S_t
//   O_t += P_t V_j          tensor core, A operand (P) from TMEM, V^T from shared memory
// The tensor core runs one CTA's MMAs in issue order, so S_t(j+1) (issued after
// O_t += P_t(j) V_j) overwrites P_t only after it was read, and S_t(j+1) landing means
// O_t is idle: the softmax may rescale it in TMEM without another wait. The running max
// is raised only when a row's tile max exceeds it by more than 2^8, so most tiles skip
// the rescale. The two tiles ping-pong: the tensor core runs one tile's products while
// the other tile's softmax runs.
// Epilogue: O_t / l_t * s -> bf16 [T, n_q*hd], s = sigmoid(xn W_g^T) as the QKV+G
// projection stored it (so no exponential is left here). The softmax warps read O_t into
// registers and hand it back (the next unit's first P V may overwrite it); the gate tile
// arrives by TMA in a ring slot after the unit's last V, each thread overwrites its row
// of it with the gated output, and every warp TMA-stores its 32 rows. The slot goes back
// to the loader once that store has read it, checked after the next unit's first softmax.
//
// Persistent: one CTA per SM walks the units u = blockIdx.x, + gridDim.x, ... with one
// TMEM allocation and one set of barriers, and every barrier phase is counted across
// units. The loader fetches the next unit's Q_t as soon as the current unit's last S_t has
// read the buffer, and its first K/V tiles as ring slots free up, so a unit's start-up
// overlaps the previous unit's last products and epilogue instead of following them.
//
// Warps 0-3: softmax/epilogue for tile 0, warps 4-7: tile 1, warp 8: TMA loads,
// warp 9: TMEM allocation + MMA issue for tile 0, warp 10: MMA issue for tile 1. The
// tensor core's instruction queue is shallow and every barrier wait costs the issuing
// thread ~100+ cycles, so each tile has its own issuing thread, which does its K/V
// waits ahead of time. The two issuers hand a turn back and forth, so their MMA groups
// strictly alternate (S_0 | S_1 | P_0 V, S_0 | P_1 V, S_1 | ...): the tiles settle in
// anti-phase, one tile's softmax running under the other tile's MMAs. TMEM: S_0/P_0, S_1/P_1, O_0, O_1 (4 x 128 columns). Shared memory:
// Q_0, Q_1 (32 KB each) and a 5-slot ring of 32 KB tiles (K, V^T, gate/output staging).
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace kd {
namespace {

constexpr int HD = 128;            // head dim
constexpr int BQ = 128;            // query rows per tile
constexpr int BKV = 128;           // keys per K/V tile
constexpr int TILE_BYTES = 128 * 128 * 2;  // one 128 x 128 bf16 operand (two 64-col swizzled halves)
constexpr int HALF_BYTES = TILE_BYTES / 2;
constexpr int NSLOT = 5;
constexpr int NUM_THREADS = 352;
constexpr int SMEM_Q = 0;
constexpr int SMEM_KV = SMEM_Q + 2 * TILE_BYTES;
constexpr int SMEM_BAR = SMEM_KV + NSLOT * TILE_BYTES;
constexpr int SMEM_BYTES = SMEM_BAR + 256 + 1024;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units: rescale O only if the max grows by > 2^8

struct AttnArgs {
  int B, L, Lp, n_q, n_kv, G, nqt, nkt, npairs, units, gate_on;
  float scale_log2;  // log2(e) / sqrt(hd)
  float* rowamax;    // optional [T]: largest |og| of each row, as stored (for an 8-bit o_proj)
  float* lse;        // optional [B, n_q, Lp]: log2 of each row's softmax normaliser, in the
                     // scaled-log2 units of the scores (for the backward)
  float* o_raw;      // optional [T, n_q*hd] fp32: the attention output before the gate (backward)
  int* err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3f(float x, float y, float z) {
  float m;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(m) : "f"(x), "f"(y), "f"(z));
  return m;
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

// Work unit u of a launch: (b, kv group, pair of query tiles 2p, 2p + 1 of the group).
struct Unit {
  int b, bk, kvh, p, nt;  // nt: query tiles of the unit (1 for the last pair of an odd count)
};
__device__ __forceinline__ Unit unit_of(const AttnArgs& a, int u) {
  Unit w;
  w.p = u % a.npairs;
  w.bk = u / a.npairs;  // b * n_kv + kv
  w.b = w.bk / a.n_kv;
  w.kvh = w.bk - w.b * a.n_kv;
  w.nt = 2 * w.p + 1 < a.G * a.nqt ? 2 : 1;
  return w;
}
// query tile t of a unit = (head, query-tile index) of group tile 2p + t
__device__ __forceinline__ int tile_head(const AttnArgs& a, const Unit& w, int t) {
  return w.kvh * a.G + (2 * w.p + t) / a.nqt;
}
__device__ __forceinline__ int tile_qt(const AttnArgs& a, const Unit& w, int t) { return (2 * w.p + t) % a.nqt; }

// 352 threads x at most 168 registers per thread: with 178 the launch is refused for lack
// of registers (allocation granularity), so the cap stays where the kernel fits today
__global__ void __maxnreg__(168)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_g,
                   const __grid_constant__ CUtensorMap tm_og, AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + SMEM_BAR);
  uint64_t* kv_full = bar;               // [NSLOT] a ring tile landed (K, V^T, gate, or an empty staging slot)
  uint64_t* kv_empty = kv_full + NSLOT;  // [NSLOT] 4 arrivals: the slot may be refilled
  uint64_t* q_full = kv_empty + NSLOT;   // [2] Q_t of the current unit landed
  uint64_t* q_free = q_full + 2;         // [2] the unit's last S_t was issued and has read Q_t
  uint64_t* s_full = q_free + 2;         // [2] S_t(j) landed (and every earlier MMA of its issuer)
  uint64_t* p_full = s_full + 2;         // [2] P_t(j) written to TMEM by all 128 rows
  uint64_t* o_done = p_full + 2;         // [2] the unit's last O_t += P_t V landed
  uint64_t* o_free = o_done + 2;         // [2] the epilogue has read O_t (4 warps)
  uint64_t* turn = o_free + 2;           // [2] turn[t]: the other issuer passed the turn
  uint64_t* done = turn + 2;             // [2] every MMA of issuing thread t finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkt = a.nkt;
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 4);  // K/V: 4 commits by the issuers; gate slot: the tile's 4 epilogue warps
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_free[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], 128);
      mbar_init(&o_done[t], 1);
      mbar_init(&o_free[t], 4);
      mbar_init(&turn[t], 1);
      mbar_init(&done[t], 1);
    }
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
  auto ring_ph = [](int n) { return static_cast<uint32_t>((n / NSLOT) & 1); };

  if (warp == 8) {
    // ------------------------------------------------------------ TMA loads
    // Per unit: Q_0, Q_1 (each once the previous unit's last S of that tile has read its
    // buffer), then through the ring K_0, V_0, ..., K_{nkt-1}, V_{nkt-1} and one slot per
    // query tile for the epilogue: the gate tile by TMA, or (without the gate) just
    // handed over empty. The next unit's Q and first K/V tiles therefore load while the
    // current unit's last products and epilogues run.
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_vt);
      if (a.gate_on) tma_prefetch_desc(&tm_g);
      tma_prefetch_desc(&tm_og);
      int n = 0;             // ring loads issued
      int qn[2] = {0, 0};    // Q loads issued per tile
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
        const Unit w = unit_of(a, u);
        for (int t = 0; t < w.nt; ++t) {
          if (qn[t] > 0 && !mbar_wait(&q_free[t], static_cast<uint32_t>((qn[t] - 1) & 1), wc, SITE_ATTN_LOAD)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&q_full[t], TILE_BYTES);
          for (int kh = 0; kh < 2; ++kh)
            tma_load_3d(smem + SMEM_Q + t * TILE_BYTES + kh * HALF_BYTES, &tm_q, &q_full[t], kh * 64,
                        tile_qt(a, w, t) * BQ, w.b * a.n_q + tile_head(a, w, t));
          ++qn[t];
        }
        const int nl = 2 * nkt + w.nt;
        for (int i = 0; ok && i < nl; ++i, ++n) {
          const int slot = n % NSLOT;
          if (!mbar_wait(&kv_empty[slot], ring_ph(n) ^ 1, wc, SITE_ATTN_LOAD)) {
            ok = false;
            break;
          }
          uint8_t* dst = smem + SMEM_KV + slot * TILE_BYTES;
          if (i < 2 * nkt) {
            const int m = i >> 1;
            mbar_arrive_expect_tx(&kv_full[slot], TILE_BYTES);
            for (int h2 = 0; h2 < 2; ++h2) {
              if ((i & 1) == 0)
                tma_load_3d(dst + h2 * HALF_BYTES, &tm_k, &kv_full[slot], h2 * 64, m * BKV, w.bk);
              else
                tma_load_3d(dst + h2 * HALF_BYTES, &tm_vt, &kv_full[slot], m * BKV + h2 * 64, 0, w.bk);
            }
          } else if (a.gate_on) {  // the gate tile of query tile i - 2 nkt
            const int t = i - 2 * nkt;
            mbar_arrive_expect_tx(&kv_full[slot], TILE_BYTES);
            for (int kh = 0; kh < 2; ++kh)
              tma_load_3d(dst + kh * HALF_BYTES, &tm_g, &kv_full[slot], tile_head(a, w, t) * HD + kh * 64,
                          tile_qt(a, w, t) * BQ, w.b);
          } else {
            mbar_arrive(&kv_full[slot]);  // staging for the output of query tile i - 2 nkt
          }
        }
      }
      // every copy started here has landed before the CTA exits
      for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) drain_wait(&q_full[t], static_cast<uint32_t>((qn[t] - 1) & 1), a.err, SITE_ATTN_TEARDOWN);
      for (int i = (n > NSLOT ? n - NSLOT : 0); i < n; ++i)
        drain_wait(&kv_full[i % NSLOT], ring_ph(i), a.err, SITE_ATTN_TEARDOWN);
    }
  } else if (warp == 9 || warp == 10) {
    // ------------------------------------------------------------ MMA issue, tile t
    const int t = warp - 9;
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      const uint32_t sQ = smem_u32(smem + SMEM_Q + t * TILE_BYTES), sKV = smem_u32(smem + SMEM_KV);
      const uint32_t dS = tmem + t * 128;        // S_t, and P_t over its first 64 columns
      const uint32_t dO = tmem + 256 + t * 128;  // O_t
      int n0 = 0;        // ring index of the current unit's K_0
      int uq = 0;        // units of this tile so far (q_full, o_done, o_free phases)
      uint32_t tk = 0;   // turn phases consumed
      uint32_t sp = 0;   // p_full phases consumed
      bool ok = true;
      for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
        const Unit w = unit_of(a, u);
        const int nl = 2 * nkt + w.nt;
        if (t >= w.nt) {  // a one-tile unit: issuer 1 sits it out
          n0 += nl;
          continue;
        }
        // Turns (two-tile units): issuer 0 runs group g = 0, 1, 2, ... after issuer 1
        // finished its group g - 1; issuer 1 runs group g after issuer 0 finished group g.
        // Group 0 is S_t(0), group j + 1 is P_t(j) V_j followed by S_t(j + 1). Each issuer
        // passes the turn once per group; issuer 0 takes one extra turn after its last
        // group so that both turn barriers end every unit with all phases consumed.
        const bool two = w.nt == 2;
        const int rel = two ? 2 : 4;  // commits per consumed ring slot (4 arrivals free it)
        auto take_turn = [&](bool first) {
          if (!two || (t == 0 && first)) return true;
          const bool r = mbar_wait(&turn[t], tk & 1, wc, SITE_ATTN_MMA);
          ++tk;
          return r;
        };
        auto pass_turn = [&]() {
          if (two) mbar_arrive(&turn[1 - t]);
        };
        auto release = [&](int slot) {
          for (int r = 0; r < rel; ++r) mma_commit(&kv_empty[slot]);
        };
        // pass_turn() is called inside a group before its final 4 MMAs: the hand-over
        // (commit, arrive, the other issuer waking up) then overlaps the tail of this group
        // instead of leaving the shallow MMA queue empty. The turns only steer scheduling;
        // the two tiles never share TMEM, so no ordering between them is needed.
        auto issue_s = [&](int slot) {  // S_t = Q_t K^T (both operands in shared memory)
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              if (kh == 1 && ks == 0) pass_turn();
              mma_bf16_ss(dS, sdesc_kmajor_sw128(sQ + kh * HALF_BYTES + ks * 32),
                          sdesc_kmajor_sw128(sKV + slot * TILE_BYTES + kh * HALF_BYTES + ks * 32), idesc,
                          (kh | ks) != 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int slot, bool acc, bool pass) {  // O_t += P_t V (P from TMEM)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {  // 16 keys per step: 8 TMEM columns of P
            if (pass && ks == 4) pass_turn();
            mma_bf16_ts(dO, dS + ks * 8,
                        sdesc_kmajor_sw128(sKV + slot * TILE_BYTES + (ks >> 2) * HALF_BYTES + (ks & 3) * 32), idesc,
                        (acc || ks != 0) ? 1u : 0u);
          }
        };
        const int s0 = n0 % NSLOT;
        ok = mbar_wait(&q_full[t], static_cast<uint32_t>(uq & 1), wc, SITE_ATTN_MMA);
        if (ok) ok = mbar_wait(&kv_full[s0], ring_ph(n0), wc, SITE_ATTN_MMA);  // K_0
        if (ok) ok = take_turn(true);
        if (!ok) break;
        // S_t(0) may run while the previous unit's epilogue still reads O_t: it writes S_t,
        // whose P the previous unit's last P V (issued before it) has already consumed
        tc_fence_after();
        issue_s(s0);
        mma_commit(&s_full[t]);
        release(s0);
        if (nkt == 1) mma_commit(&q_free[t]);
        for (int j = 0; j < nkt; ++j) {
          const int nv = n0 + 2 * j + 1, nk = n0 + 2 * j + 2;  // ring indices of V_j, K_{j+1}
          const int sv = nv % NSLOT, sk = nk % NSLOT;
          const bool more = j + 1 < nkt;
          // operands first (normally long landed), then the real dependencies
          if (!mbar_wait(&kv_full[sv], ring_ph(nv), wc, SITE_ATTN_MMA)) { ok = false; break; }
          if (more && !mbar_wait(&kv_full[sk], ring_ph(nk), wc, SITE_ATTN_MMA)) { ok = false; break; }
          if (!mbar_wait(&p_full[t], sp & 1, wc, SITE_ATTN_MMA)) { ok = false; break; }
          ++sp;
          // the first P V overwrites O_t: the previous unit's epilogue must have read it
          if (j == 0 && uq > 0 && !mbar_wait(&o_free[t], static_cast<uint32_t>((uq - 1) & 1), wc, SITE_ATTN_MMA)) {
            ok = false;
            break;
          }
          if (!take_turn(false)) { ok = false; break; }
          tc_fence_after();
          issue_pv(sv, j > 0, !more);
          release(sv);
          if (!more) {
            mma_commit(&o_done[t]);
            break;
          }
          issue_s(sk);  // after the P V above: it overwrites P_t only once P_t was read
          mma_commit(&s_full[t]);
          release(sk);
          if (j + 2 == nkt) mma_commit(&q_free[t]);  // that was the unit's last S_t
        }
        if (!ok) break;
        if (two && t == 0 && !take_turn(false)) break;
        ++uq;
        n0 += nl;
      }
      mma_commit(&done[t]);
      drain_wait(&done[t], 0, a.err, SITE_ATTN_TEARDOWN);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;           // query tile of this warpgroup
    const int quad = warp & 3;         // TMEM lane quadrant
    const int row = quad * 32 + lane;  // row inside the query tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t tS = tmem + lane_off + t * 128;
    const uint32_t tO = tmem + lane_off + 256 + t * 128;
    int n0 = 0;        // ring index of the current unit's K_0
    int uq = 0;        // units of this tile so far (o_done phases)
    // Ring slot of this warp's last output store. It is released (the store has read it)
    // only after the next unit's first P is written, so that the store's completion does
    // not sit between a unit's epilogue and the next unit's first softmax.
    int pend = -1;
    auto release_pend = [&]() {
      if (pend < 0) return;
      if (lane == 0) {
        bulk_wait_read_all();
        mbar_arrive(&kv_empty[pend]);
      }
      pend = -1;
    };
    uint32_t sp = 0;   // s_full phases consumed
    bool ok = true;
    for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
      const Unit w = unit_of(a, u);
      const int nl = 2 * nkt + w.nt;
      if (t >= w.nt) {
        release_pend();
        n0 += nl;
        continue;
      }
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkt; ++j) {
        const bool got = mbar_wait(&s_full[t], sp & 1, wc, SITE_ATTN_SOFTMAX);
        ++sp;
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[128];
        tmem_ld128(tS, sv);
        const int kvalid = a.L - j * BKV;  // keys of this tile inside the sequence (>= 1)
        if (kvalid < BKV) {  // ragged last tile (same for the whole warp): keys past L get -inf
#pragma unroll
          for (int i = 0; i < 128; ++i)
            if (i >= kvalid) sv[i] = __float_as_uint(-INFINITY);
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // 4 independent chains
#pragma unroll
        for (int i = 0; i < 128; i += 8)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            mq[q] = max3f(mq[q], __uint_as_float(sv[i + 2 * q]), __uint_as_float(sv[i + 2 * q + 1]));
        const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * a.scale_log2;
        // Lazy rescale: raise the running max only when some row's tile max exceeds it by
        // more than 2^8. The decision is warp-uniform because the O rescale uses
        // warp-collective TMEM accesses; each row moves to its own new max (alpha = 1 for
        // a row whose max did not grow).
        bool rescale = false;
        float m_new = m_run;
        if (j == 0) {
          m_new = mx;
        } else if (__any_sync(0xffffffffu, mx > m_run + RESCALE_THRESHOLD)) {
          rescale = true;
          m_new = fmaxf(m_run, mx);
        }
        // P = exp2(s * scale - m), bf16 pairs; row sum in fp32
        const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
        const float2 nm2 = make_float2(-m_new, -m_new);
        float2 sum2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};  // 4 independent chains
        uint32_t pk[64];
#pragma unroll
        for (int i2 = 0; i2 < 64; ++i2) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sv[2 * i2]), __uint_as_float(sv[2 * i2 + 1])),
                                      sc2, nm2);
          const float2 pr = make_float2(ex2(x.x), ex2(x.y));
          sum2[i2 & 3] = __fadd2_rn(sum2[i2 & 3], pr);
          pk[i2] = pack_bf16x2(pr.x, pr.y);
        }
        tmem_st64(tS, pk);  // P_t over the first 64 columns of S_t
        const float2 s01 = __fadd2_rn(sum2[0], sum2[1]), s23 = __fadd2_rn(sum2[2], sum2[3]);
        const float sum = (s01.x + s01.y) + (s23.x + s23.y);
        if (rescale) {  // O_t is idle: S_t(j) landing means O_t += P_t(j-1) V landed too
          const float alpha = ex2(m_run - m_new);
          l_run *= alpha;
          uint32_t r[32];
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            tmem_ld32(tO + c * 32, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(tO + c * 32, r);
          }
        }
        m_run = m_new;
        l_run += sum;
        tmem_st_wait();   // P (and any O rescale) written
        tc_fence_before();
        mbar_arrive(&p_full[t]);
        release_pend();
      }
      if (!ok) break;
      // ---- epilogue: O_t / l * s -> og (s: the stored gate). O_t is handed back once it is all in
      // registers; the gate tile (or an empty staging slot) is the ring slot after this
      // unit's last V.
      const bool w4 = mbar_wait(&o_done[t], static_cast<uint32_t>(uq & 1), wc, SITE_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, w4)) { ok = false; break; }
      const int ng = n0 + 2 * nkt + t;
      const int gsl = ng % NSLOT;
      const bool wg = mbar_wait(&kv_full[gsl], ring_ph(ng), wc, SITE_ATTN_SOFTMAX);
      if (!__all_sync(0xffffffffu, wg)) { ok = false; break; }
      tc_fence_after();
      const int head = tile_head(a, w, t), qt = tile_qt(a, w, t);
      const int ql = qt * BQ + row;  // query position in the sequence
      const bool valid = ql < a.L;
      const float inv_l = 1.0f / l_run;
      const size_t off = (static_cast<size_t>(w.b) * a.L + (valid ? ql : 0)) * (a.n_q * HD) + head * HD;
      uint8_t* buf = smem + SMEM_KV + gsl * TILE_BYTES;
      // this row in the two 64-column halves of the tile (128-byte swizzle: unit u of row r
      // sits at u ^ (r & 7))
      uint8_t* rb = buf + row * 128;
      const int sw = row & 7;
      float amax = 0.0f;
      // one 32-column chunk c of O (in r): scale, gate, write back over the gate in place
      auto chunk = [&](const uint32_t (&r)[32], int c) {
        float o[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(r[i]) * inv_l;
        if (a.o_raw && valid) {
          float4* w4p = reinterpret_cast<float4*>(a.o_raw + off + c * 32);
#pragma unroll
          for (int q = 0; q < 8; ++q) w4p[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
        uint8_t* hb = rb + (c >> 1) * HALF_BYTES;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4* p16 = reinterpret_cast<uint4*>(hb + ((((c & 1) * 4 + q4) ^ sw) << 4));
          if (a.gate_on) {
            const uint4 gu = *p16;
            const uint32_t gw[4] = {gu.x, gu.y, gu.z, gu.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 gg = unpack_bf16x2(gw[e]);
              o[8 * q4 + 2 * e] *= gg.x;
              o[8 * q4 + 2 * e + 1] *= gg.y;
            }
          }
          *p16 = make_uint4(pack_bf16x2(o[8 * q4 + 0], o[8 * q4 + 1]), pack_bf16x2(o[8 * q4 + 2], o[8 * q4 + 3]),
                            pack_bf16x2(o[8 * q4 + 4], o[8 * q4 + 5]), pack_bf16x2(o[8 * q4 + 6], o[8 * q4 + 7]));
        }
        if (a.rowamax && valid) {
#pragma unroll
          for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(o[i]));
        }
      };
#pragma unroll 1
      for (int cc = 0; cc < 2; ++cc) {  // two TMEM round trips of 64 columns
        uint32_t ra[32], rb2[32];
        tmem_ld32x2(tO + cc * 64, tO + cc * 64 + 32, ra, rb2);
        if (cc == 1) {  // all of O_t is in registers: the next unit's first P V may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_free[t]);
        }
        chunk(ra, 2 * cc);
        chunk(rb2, 2 * cc + 1);
      }
      fence_proxy_async_smem();  // the rows are visible to the TMA engine
      __syncwarp();
      const int r0 = qt * BQ + quad * 32;  // first sequence row of this warp's 32 rows
      if (lane == 0) {
        if (r0 < a.L) {  // rows past L are clipped by the store (3D map over [B, L, .])
          for (int kh = 0; kh < 2; ++kh)
            tma_store_3d(&tm_og, buf + kh * HALF_BYTES + quad * 32 * 128, head * HD + kh * 64, r0, w.b);
          bulk_commit();
        }
      }
      pend = gsl;
      // bf16 rounding is monotone, so the largest stored magnitude is the rounded largest
      if (a.lse && valid) a.lse[(static_cast<size_t>(w.b) * a.n_q + head) * a.Lp + ql] = m_run + log2f(l_run);
      if (a.rowamax && valid)
        atomic_max_nonneg(a.rowamax + static_cast<size_t>(w.b) * a.L + ql, round_bf16(amax));
      ++uq;
      n0 += nl;
    }
    release_pend();
    // this warp's output stores have completed before exit
    if (lane == 0) bulk_wait_all();
    __syncwarp();
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

cudaError_t attn_tc_init() {
  return cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t launch_attn_tc(const Fwd& f, const CUtensorMap* tm_q, const CUtensorMap* tm_k, const CUtensorMap* tm_vt,
                           const CUtensorMap* tm_g, const CUtensorMap* tm_og, float* rowamax, float* lse, float* o_raw,
                           int num_sms, int* err, cudaStream_t st) {
  AttnArgs a;
  a.B = f.B;
  a.L = f.L;
  a.Lp = f.Lp;
  a.n_q = f.n_q;
  a.n_kv = f.n_kv;
  a.G = f.n_q / f.n_kv;
  a.nqt = (f.L + BQ - 1) / BQ;
  a.nkt = (f.L + BKV - 1) / BKV;
  a.npairs = (a.G * a.nqt + 1) / 2;
  a.gate_on = f.gate_on;
  a.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  a.rowamax = rowamax;
  a.lse = lse;
  a.o_raw = o_raw;
  a.err = err;
  const long long units = static_cast<long long>(f.B) * f.n_kv * a.npairs;
  if (units == 0) return cudaSuccess;
  if (units > INT_MAX || num_sms <= 0) return cudaErrorInvalidValue;
  a.units = static_cast<int>(units);
  const int grid = static_cast<int>(units < num_sms ? units : num_sms);  // persistent: one CTA per SM
  if (!tm_og || (f.gate_on && !tm_g)) return cudaErrorInvalidValue;
  attn_tc_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(*tm_q, *tm_k, *tm_vt,
                                                                                f.gate_on ? *tm_g : *tm_q, *tm_og, a);
  return cudaGetLastError();
}

}  // namespace kd
