// C ABI of the DiT block library: argument validation, workspace, TMA tensor maps,
// kernel sequencing, per-kernel timing and device-side failure reporting.
// The operation and every argument are documented in include/krea_dit.h.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "internal.h"
#include "krea_dit.h"

using kd::Fwd;
using kd::QkvgDst;
using kd::RowSrc;

namespace {

// ---- kernel slots (one per logical kernel the library launches) --------------------
enum Slot {
  S_NORM1,
  S_QKVG_TC,
  S_ATTN,
  S_OPROJ_TC,
  S_NORM2,
  S_UPGATE_TC,
  S_DOWN_TC,
  S_QKVG_F32,
  S_QKVG_POST_F32,
  S_OPROJ_F32,
  S_RESID_ATTN_F32,
  S_GATE_F32,
  S_UP_F32,
  S_SWIGLU_F32,
  S_DOWN_F32,
  S_RESID_MLP_F32,
  S_TEMB_SIN,
  S_TEMB_MLP1,
  S_TEMB_MLP2,
  S_NORM1_AMAX,
  S_QUANT_OG,
  S_NORM2_AMAX,
  S_QUANT_HMID,
  S_W8_AMAX,
  S_W8_QUANT,
  S_BWD_GEMM,
  S_BWD_TRANSPOSE,
  S_BWD_POINTWISE,
  S_BWD_ATTN,
  S_Q4_AMAX,
  S_Q4_CAST,
  S_COUNT
};
const char* const kSlotNames[S_COUNT] = {
    "norm1_modulate",       "qkvg_gemm_qknorm_rope", "attention_gate",  "oproj_gemm_residual",
    "norm2_modulate",       "upgate_gemm_swiglu",    "down_gemm_residual", "qkvg_gemm_f32",
    "qkvg_qknorm_rope_f32", "oproj_gemm_f32",        "residual_attn_f32", "gate_gemm_f32",
    "up_gemm_f32",          "swiglu_f32",            "down_gemm_f32",   "residual_mlp_f32",
    "temb_sinusoid",        "temb_mlp1",             "temb_mlp2",       "norm1_amax",
    "quant_og_e4m3",        "norm2_amax",            "quant_hmid_e4m3", "weights8_row_amax",
    "weights8_quant_e4m3",  "bwd_gemm",              "bwd_transpose",   "bwd_pointwise",
    "bwd_attention",        "nvfp4_row_amax",        "nvfp4_cast"};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 2D bf16 tensor map over a row-major [rows, cols] matrix with pitch `pitch_elems`,
// box = box_cols x box_rows, 128-byte swizzle, zero fill outside the matrix.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch_elems,
               uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D fp32 tensor map over a row-major [rows, cols] matrix (pitch = cols), box = 32 x 32
// (128-byte rows, matching the 128-byte swizzle): the residual epilogue's store target.
bool encode_2d_f32(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D bf16 tensor map over [planes, rows, cols] (cols contiguous, pitch `pitch_elems`).
bool encode_3d(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t planes,
               uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows) {
  cuuint64_t dims[3] = {cols, rows, planes};
  cuuint64_t strides[2] = {pitch_elems * 2, pitch_elems * 2 * rows};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2D tensor map of bytes (e4m3 codes) over a row-major [rows, cols] matrix, pitch = cols,
// box = 128 x box_rows (128-byte rows, matching the 128-byte swizzle).
bool encode_2d_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (!a || !b || !na || !nb) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

struct GraphBox {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

struct TimedLaunch {
  int slot;
  cudaEvent_t begin, end;
};

}  // namespace

struct krea_dit_block_s {
  krea_dit_config cfg{};
  int device = 0, num_sms = 0;
  bool bf16 = true;  // bf16 storage (also in the 8-bit modes)
  int mode8 = 0;     // 0: no 8-bit GEMMs, 1: tensor-wise scaling, 2: row-wise scaling
  size_t esz = 2;
  size_t max_T = 0;
  int n_qkvg = 0;
  int rope_rows = 0;
  // one device allocation, carved into the buffers below
  char* ws = nullptr;
  size_t ws_bytes = 0;
  void *xn = nullptr, *q = nullptr, *k = nullptr, *vt = nullptr, *g = nullptr, *og = nullptr, *h1 = nullptr,
       *hn = nullptr, *hmid = nullptr;
  size_t sz_xn = 0, sz_q = 0, sz_k = 0, sz_vt = 0, sz_g = 0, sz_og = 0, sz_h1 = 0, sz_hn = 0, sz_hmid = 0;
  float *raw_qkvg = nullptr, *raw_o = nullptr, *raw_a = nullptr, *raw_u = nullptr, *raw_down = nullptr;
  float *temb_e = nullptr, *temb_h = nullptr;
  // 8-bit modes: e4m3 GEMM operands, their dequantisation factors, row amax accumulators
  void *xn8 = nullptr, *og8 = nullptr, *hn8 = nullptr, *hmid8 = nullptr;
  float *dq_xn = nullptr, *dq_og = nullptr, *dq_hn = nullptr, *dq_hmid = nullptr;
  float *am_xn = nullptr, *am_og = nullptr, *am_hn = nullptr, *am_hmid = nullptr, *am_w = nullptr;
  // NVFP4 mode: E2M1 GEMM operands, their block scales and tensor scales
  bool mode4 = false;
  void *xn4 = nullptr, *og4 = nullptr, *hn4 = nullptr, *hmid4 = nullptr;
  void *sf_xn4 = nullptr, *sf_og4 = nullptr, *sf_hn4 = nullptr, *sf_hmid4 = nullptr;
  float* ts4 = nullptr;  // [4]: xn, og, hn, hmid
  // backward workspace (krea_dit_block_enable_backward): one allocation, carved below
  char* bw = nullptr;
  size_t bw_Tp = 0, bw_Lp = 0;
  bool bw_stats = false;  // the next forward also writes the attention's lse and ungated output
  float* f_lse = nullptr;
  float* f_D = nullptr;
  void *bw_out = nullptr, *wT_down = nullptr, *wT_gu = nullptr, *wT_o = nullptr, *wT_qkvg = nullptr;
  float *f_td = nullptr, *f_fa = nullptr, *f_a = nullptr, *f_u = nullptr, *f_dn = nullptr, *f_dh1 = nullptr,
        *f_o = nullptr, *f_raw = nullptr, *f_dq = nullptr, *f_dk = nullptr, *f_dv = nullptr,
        *f_rstd = nullptr;
  void *b_dfm = nullptr, *b_dau = nullptr, *b_dfa = nullptr, *b_do = nullptr, *b_dP = nullptr, *b_vrow = nullptr,
       *b_kT = nullptr, *b_qT = nullptr, *b_doT = nullptr;
  void *t_dfm = nullptr, *t_hmid = nullptr, *t_dau = nullptr, *t_hn = nullptr, *t_dfa = nullptr, *t_og = nullptr,
       *t_dP = nullptr, *t_xn = nullptr;
  float2* rope = nullptr;
  int* err = nullptr;
  Fwd last{};
  bool have_last = false;
  // timing
  bool timing = false;
  std::vector<cudaEvent_t> free_events;
  std::vector<TimedLaunch> pending;
  double total_ms[S_COUNT] = {};
  int launches[S_COUNT] = {};
  int inject = 0;
  // host-buffer path: two staging sets, upload / download streams, events per set
  bool host_io = false;
  char* stage = nullptr;
  size_t stage_in_bytes = 0, stage_out_bytes = 0;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
  bool set_used[2] = {};
  int next_set = 0;
};

namespace {

int harvest(krea_dit_block_s* h) {
  for (auto& t : h->pending) {
    if (cudaEventSynchronize(t.end) != cudaSuccess) return KREA_DIT_ERR_CUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.begin, t.end) != cudaSuccess) return KREA_DIT_ERR_CUDA;
    h->total_ms[t.slot] += ms;
    h->launches[t.slot] += 1;
    h->free_events.push_back(t.begin);
    h->free_events.push_back(t.end);
  }
  h->pending.clear();
  return KREA_DIT_OK;
}

cudaEvent_t take_event(krea_dit_block_s* h) {
  if (h->free_events.empty()) {
    if (h->pending.size() >= 4096) harvest(h);  // bound the number of live events
  }
  if (!h->free_events.empty()) {
    cudaEvent_t e = h->free_events.back();
    h->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
  return e;
}

// Runs one launch; when timing is on, brackets it with events on `st`.
// Host-side NVTX range for the lifetime of the object (header-only NVTX v3).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

template <class F>
cudaError_t timed(krea_dit_block_s* h, int slot, cudaStream_t st, F&& launch) {
  // Every launch sits in an NVTX range named after its kernel slot, so a profiler can
  // select one kernel of the block by name (ncu --nvtx --nvtx-include "<slot>/"). With no
  // tool attached an NVTX call returns at once.
  NvtxRange range(kSlotNames[slot]);
  if (!h->timing) return launch();
  cudaEvent_t b = take_event(h), e = take_event(h);
  if (!b || !e) return cudaErrorMemoryAllocation;
  cudaEventRecord(b, st);
  cudaError_t r = launch();
  cudaEventRecord(e, st);
  h->pending.push_back({slot, b, e});
  return r;
}

bool sm103_current(int* dev, int* sms) {
  if (cudaGetDevice(dev) != cudaSuccess) return false;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess) return false;
  return major == 10 && minor == 3;
}

}  // namespace

extern "C" {

const char* krea_dit_status_string(int s) {
  switch (s) {
    case KREA_DIT_OK: return "ok";
    case KREA_DIT_ERR_INVALID_ARG: return "invalid argument";
    case KREA_DIT_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case KREA_DIT_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS: return "call exceeds the limits the handle was created with";
    case KREA_DIT_ERR_CUDA: return "CUDA runtime or driver error";
    case KREA_DIT_ERR_NO_DEVICE: return "current device is not an sm_103 GPU";
    case KREA_DIT_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait expired";
    case KREA_DIT_ERR_INJECTED: return "injected fault";
    case KREA_DIT_ERR_SCRATCH_TOO_SMALL: return "call needs more than the no-alloc entry point's fixed scratch";
    default: return "unknown status";
  }
}

int krea_dit_kernel_names(const char** names, int cap) {
  for (int i = 0; i < S_COUNT && i < cap; ++i)
    if (names) names[i] = kSlotNames[i];
  return S_COUNT;
}

int krea_dit_block_create(const krea_dit_config* c, krea_dit_block_t* out) {
  if (!out) return KREA_DIT_ERR_INVALID_ARG;
  *out = nullptr;
  if (!c) return KREA_DIT_ERR_INVALID_ARG;
  if (c->mode != KREA_DIT_BF16 && c->mode != KREA_DIT_FP32 && c->mode != KREA_DIT_FP8_TENSOR &&
      c->mode != KREA_DIT_FP8_ROW && c->mode != KREA_DIT_NVFP4)
    return KREA_DIT_ERR_INVALID_ARG;
  if (c->max_batch < 1 || c->max_seq < 1 || c->img_h_max < 0 || c->img_w_max < 0) return KREA_DIT_ERR_INVALID_ARG;
  if (!(c->eps > 0.f) || !(c->rope_base > 0.f) || (c->gate_on != 0 && c->gate_on != 1))
    return KREA_DIT_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->n_q <= 0 || c->n_kv <= 0 || c->ffn <= 0) return KREA_DIT_ERR_INVALID_ARG;
  if (c->d_model % 64 || c->ffn % 64 || c->n_q % c->n_kv) return KREA_DIT_ERR_UNSUPPORTED_SHAPE;
  if (c->d_model > 8192) return KREA_DIT_ERR_UNSUPPORTED_SHAPE;  // norm kernel: one thread per 8 columns
  if (c->head_dim != 64 && c->head_dim != 128) return KREA_DIT_ERR_UNSUPPORTED_SHAPE;
  if (c->mode != KREA_DIT_FP32 && c->head_dim != 128) return KREA_DIT_ERR_UNSUPPORTED_SHAPE;
  // the norm kernel's e4m3 output holds rows of up to 3072 columns
  if ((c->mode == KREA_DIT_FP8_TENSOR || c->mode == KREA_DIT_FP8_ROW) && c->d_model > 3072)
    return KREA_DIT_ERR_UNSUPPORTED_SHAPE;
  // 32-bit index arithmetic inside the kernels
  const double big = static_cast<double>(c->max_batch) * c->max_seq *
                     (c->ffn > (2 * c->n_q + 2 * c->n_kv) * c->head_dim ? c->ffn
                                                                          : (2 * c->n_q + 2 * c->n_kv) * c->head_dim);
  if (static_cast<double>(c->max_batch) * c->max_seq > 2147483647.0 || big > 9.0e15)
    return KREA_DIT_ERR_UNSUPPORTED_SHAPE;

  int dev = 0, sms = 0;
  if (!sm103_current(&dev, &sms)) return KREA_DIT_ERR_NO_DEVICE;

  krea_dit_block_s* h = new (std::nothrow) krea_dit_block_s();
  if (!h) return KREA_DIT_ERR_CUDA;
  h->cfg = *c;
  h->device = dev;
  h->num_sms = sms;
  h->bf16 = c->mode != KREA_DIT_FP32;
  h->mode8 = c->mode == KREA_DIT_FP8_TENSOR ? 1 : (c->mode == KREA_DIT_FP8_ROW ? 2 : 0);
  h->mode4 = c->mode == KREA_DIT_NVFP4;
  h->esz = h->bf16 ? 2 : 4;
  h->max_T = static_cast<size_t>(c->max_batch) * c->max_seq;
  h->n_qkvg = ((c->gate_on ? 2 : 1) * c->n_q + 2 * c->n_kv) * c->head_dim;
  h->rope_rows = c->img_h_max > c->img_w_max ? c->img_h_max : c->img_w_max;
  if (h->rope_rows < 1) h->rope_rows = 1;

  const size_t T = h->max_T, d = c->d_model, hd = c->head_dim, F = c->ffn, es = h->esz;
  const size_t Lp = round_up(static_cast<size_t>(c->max_seq), 64);
  struct Item {
    void** p;
    size_t bytes;
    size_t* sz;
  };
  h->sz_xn = T * d * es;
  h->sz_q = T * c->n_q * hd * es;
  h->sz_k = T * c->n_kv * hd * es;
  h->sz_vt = static_cast<size_t>(c->max_batch) * c->n_kv * hd * Lp * es;
  h->sz_g = T * c->n_q * hd * es;
  h->sz_og = T * c->n_q * hd * es;
  h->sz_h1 = T * d * 4;  // the residual stream between the two residual adds is fp32 in both modes
  h->sz_hn = T * d * es;
  h->sz_hmid = T * F * es;
  std::vector<Item> items = {
      {&h->xn, h->sz_xn, nullptr},  {&h->q, h->sz_q, nullptr},   {&h->k, h->sz_k, nullptr},
      {&h->vt, h->sz_vt, nullptr},  {&h->g, h->sz_g, nullptr},   {&h->og, h->sz_og, nullptr},
      {&h->h1, h->sz_h1, nullptr},  {&h->hn, h->sz_hn, nullptr}, {&h->hmid, h->sz_hmid, nullptr},
  };
  if (!h->bf16) {
    items.push_back({reinterpret_cast<void**>(&h->raw_qkvg), T * h->n_qkvg * 4, nullptr});
    items.push_back({reinterpret_cast<void**>(&h->raw_o), T * d * 4, nullptr});
    items.push_back({reinterpret_cast<void**>(&h->raw_a), T * F * 4, nullptr});
    items.push_back({reinterpret_cast<void**>(&h->raw_u), T * F * 4, nullptr});
    items.push_back({reinterpret_cast<void**>(&h->raw_down), T * d * 4, nullptr});
  }
  if (h->mode8) {
    const size_t nqhd = static_cast<size_t>(c->n_q) * hd;
    size_t wrows = static_cast<size_t>(h->n_qkvg);
    if (d > wrows) wrows = d;
    if (F > wrows) wrows = F;
    items.push_back({&h->xn8, T * d, nullptr});
    items.push_back({&h->og8, T * nqhd, nullptr});
    items.push_back({&h->hn8, T * d, nullptr});
    items.push_back({&h->hmid8, T * F, nullptr});
    for (float** p : {&h->dq_xn, &h->dq_og, &h->dq_hn, &h->dq_hmid, &h->am_xn, &h->am_og, &h->am_hn, &h->am_hmid})
      items.push_back({reinterpret_cast<void**>(p), T * 4, nullptr});
    items.push_back({reinterpret_cast<void**>(&h->am_w), wrows * 4, nullptr});
  }
  if (h->mode4) {
    const size_t nqhd = static_cast<size_t>(c->n_q) * hd;
    size_t wrows = static_cast<size_t>(h->n_qkvg);
    if (d > wrows) wrows = d;
    if (F > wrows) wrows = F;
    items.push_back({&h->xn4, T * d / 2, nullptr});
    items.push_back({&h->og4, T * nqhd / 2, nullptr});
    items.push_back({&h->hn4, T * d / 2, nullptr});
    items.push_back({&h->hmid4, T * F / 2, nullptr});
    items.push_back({&h->sf_xn4, kd::nvfp4_scale_bytes(static_cast<long long>(T), d), nullptr});
    items.push_back({&h->sf_og4, kd::nvfp4_scale_bytes(static_cast<long long>(T), nqhd), nullptr});
    items.push_back({&h->sf_hn4, kd::nvfp4_scale_bytes(static_cast<long long>(T), d), nullptr});
    items.push_back({&h->sf_hmid4, kd::nvfp4_scale_bytes(static_cast<long long>(T), F), nullptr});
    items.push_back({reinterpret_cast<void**>(&h->ts4), 4 * sizeof(float), nullptr});
    for (float** p : {&h->am_xn, &h->am_og, &h->am_hn, &h->am_hmid})
      items.push_back({reinterpret_cast<void**>(p), T * 4, nullptr});
    items.push_back({reinterpret_cast<void**>(&h->am_w), wrows * 4, nullptr});
  }
  items.push_back({reinterpret_cast<void**>(&h->temb_e), static_cast<size_t>(c->max_batch) * 256 * 4, nullptr});
  items.push_back({reinterpret_cast<void**>(&h->temb_h), static_cast<size_t>(c->max_batch) * d * 4, nullptr});
  items.push_back({reinterpret_cast<void**>(&h->rope), static_cast<size_t>(h->rope_rows) * (hd / 4) * 8, nullptr});
  items.push_back({reinterpret_cast<void**>(&h->err), 256, nullptr});
  size_t total = 0;
  for (auto& it : items) total += round_up(it.bytes, 256);
  if (cudaMalloc(&h->ws, total) != cudaSuccess) {
    delete h;
    return KREA_DIT_ERR_CUDA;
  }
  h->ws_bytes = total;
  size_t off = 0;
  for (auto& it : items) {
    *it.p = h->ws + off;
    off += round_up(it.bytes, 256);
  }
  // zero the workspace once so padded V^T columns are finite from the first call
  if (cudaMemset(h->ws, 0, total) != cudaSuccess) {
    cudaFree(h->ws);
    delete h;
    return KREA_DIT_ERR_CUDA;
  }
  // RoPE table: (cos, sin) of pos * base^(-2j/D), D = hd/2, j < hd/4, computed in double.
  {
    const int Q = c->head_dim / 4;
    const double D = c->head_dim / 2;
    std::vector<float2> tab(static_cast<size_t>(h->rope_rows) * Q);
    for (int p = 0; p < h->rope_rows; ++p)
      for (int j = 0; j < Q; ++j) {
        const double ang = p * pow(static_cast<double>(c->rope_base), -2.0 * j / D);
        tab[static_cast<size_t>(p) * Q + j] = make_float2(static_cast<float>(cos(ang)), static_cast<float>(sin(ang)));
      }
    if (cudaMemcpy(h->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
      cudaFree(h->ws);
      delete h;
      return KREA_DIT_ERR_CUDA;
    }
  }
  if (kd::norm_init(c->d_model) != cudaSuccess ||
      (h->mode4 && kd::gemm_fp4_init() != cudaSuccess) ||
      (h->bf16 && (!get_encode() || kd::gemm_tc_init(sms) != cudaSuccess || kd::attn_tc_init() != cudaSuccess ||
                      kd::attn_bwd_init() != cudaSuccess))) {
    cudaFree(h->ws);
    delete h;
    return KREA_DIT_ERR_CUDA;
  }
  *out = h;
  return KREA_DIT_OK;
}

int krea_dit_block_destroy(krea_dit_block_t h) {
  if (!h) return KREA_DIT_OK;
  cudaDeviceSynchronize();
  harvest(h);
  for (auto e : h->free_events) cudaEventDestroy(e);
  if (h->host_io) {
    for (int i = 0; i < 2; ++i) {
      cudaEventDestroy(h->ev_in[i]);
      cudaEventDestroy(h->ev_comp[i]);
      cudaEventDestroy(h->ev_out[i]);
    }
    cudaStreamDestroy(h->up);
    cudaStreamDestroy(h->down);
    cudaFree(h->stage);
  }
  if (h->bw) cudaFree(h->bw);
  cudaError_t r = cudaFree(h->ws);
  delete h;
  return r == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

int krea_dit_timestep_embed(krea_dit_block_t h, const float* t, int B, const krea_dit_temb_weights* w,
                            float* mod_shared, krea_dit_stream_t stream) {
  if (!h || !t || !w || !mod_shared || !w->w1 || !w->b1 || !w->w2 || !w->b2) return KREA_DIT_ERR_INVALID_ARG;
  if (B < 0) return KREA_DIT_ERR_INVALID_ARG;
  if (B > h->cfg.max_batch) return KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS;
  if (!aligned16(t) || !aligned16(mod_shared) || !aligned16(w->w1) || !aligned16(w->b1) || !aligned16(w->w2) ||
      !aligned16(w->b2))
    return KREA_DIT_ERR_MISALIGNED;
  if (B == 0) return KREA_DIT_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int d = h->cfg.d_model;
  cudaError_t e;
  e = timed(h, S_TEMB_SIN, st, [&] { return kd::launch_temb_sinusoid(t, B, h->temb_e, st); });
  if (e == cudaSuccess)
    e = timed(h, S_TEMB_MLP1, st,
              [&] { return kd::launch_gemm_simt_f32(h->temb_e, w->w1, h->temb_h, B, d, 256, w->b1, 1, st); });
  if (e == cudaSuccess)
    e = timed(h, S_TEMB_MLP2, st,
              [&] { return kd::launch_gemm_simt_f32(h->temb_h, w->w2, mod_shared, B, 6 * d, d, w->b2, 0, st); });
  return e == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

}  // extern "C"

namespace {
// Shared body of the split-input and joint-input forwards. `x_joint` non-null selects
// the joint input [B, L, d] (then x_img / x_txt are ignored) and allows out == x_joint.
// 3D maps over [B, L, n_q*hd] of the gate value (box 64 x 128 rows: the attention
// epilogue loads a query tile's gate with it; only with the gate) and of the attention
// output (box 64 x 32 rows: the epilogue's stores)
bool encode_attn_gate_out(CUtensorMap* tm_g, CUtensorMap* tm_og, krea_dit_block_t h, int B, int L) {
  const uint64_t nq = static_cast<uint64_t>(h->cfg.n_q) * h->cfg.head_dim;
  if (h->cfg.gate_on && !encode_3d(tm_g, h->g, nq, L, B, nq, 64, 128)) return false;
  return encode_3d(tm_og, h->og, nq, L, B, nq, 64, 32);
}

int forward_impl(krea_dit_block_t h, const void* x_img, const void* x_txt, const void* x_joint, int B, int img_h,
                 int img_w, int n_txt, const float* t_emb, const krea_dit_weights* w, const krea_dit_weights8* w8,
                 void* out, krea_dit_stream_t stream, const krea_dit_weights4* w4 = nullptr) {
  if (!h || !w || !t_emb || !out) return KREA_DIT_ERR_INVALID_ARG;
  if ((h->mode8 != 0) != (w8 != nullptr)) return KREA_DIT_ERR_INVALID_ARG;  // 8-bit handles need forward8
  if (h->mode4 != (w4 != nullptr)) return KREA_DIT_ERR_INVALID_ARG;        // NVFP4 handles need forward4
  if (B < 0 || img_h < 0 || img_w < 0 || n_txt < 0) return KREA_DIT_ERR_INVALID_ARG;
  if (!w->norm1_w || !w->norm2_w || !w->q_norm_w || !w->k_norm_w || !w->mod_bias) return KREA_DIT_ERR_INVALID_ARG;
  if (w8) {
    const void* p8[] = {w8->w_qkvg, w8->w_o,    w8->w_gate, w8->w_up,    w8->w_down,
                        w8->dq_qkvg, w8->dq_o, w8->dq_gate, w8->dq_up, w8->dq_down};
    for (const void* p : p8) {
      if (!p) return KREA_DIT_ERR_INVALID_ARG;
      if (!aligned16(p)) return KREA_DIT_ERR_MISALIGNED;
    }
  } else if (w4) {
    const void* p4[] = {w4->w_qkvg,  w4->w_o,  w4->w_gate,  w4->w_up,  w4->w_down,  w4->sf_qkvg, w4->sf_o, w4->sf_gate,
                        w4->sf_up, w4->sf_down, w4->ts_qkvg, w4->ts_o, w4->ts_gate, w4->ts_up, w4->ts_down};
    for (const void* p : p4) {
      if (!p) return KREA_DIT_ERR_INVALID_ARG;
      if (!aligned16(p)) return KREA_DIT_ERR_MISALIGNED;
    }
  } else if (!w->w_qkvg || !w->w_o || !w->w_gate || !w->w_up || !w->w_down) {
    return KREA_DIT_ERR_INVALID_ARG;
  }
  const krea_dit_config& c = h->cfg;
  const long long n_img_ll = static_cast<long long>(img_h) * img_w;
  const long long L_ll = n_img_ll + n_txt;
  if (B > c.max_batch || L_ll > c.max_seq || (n_img_ll > 0 && (img_h > c.img_h_max || img_w > c.img_w_max)))
    return KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS;
  const int n_img = static_cast<int>(n_img_ll), L = static_cast<int>(L_ll);
  if (x_joint) {
    x_img = x_txt = nullptr;
  } else if ((n_img > 0 && !x_img) || (n_txt > 0 && !x_txt)) {
    return KREA_DIT_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {w->w_qkvg, w->w_o,     w->w_gate,   w->w_up,     w->w_down, w->norm1_w, w->norm2_w,
                        w->q_norm_w, w->k_norm_w, w->mod_bias, t_emb, out};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return KREA_DIT_ERR_MISALIGNED;
  if ((x_img && !aligned16(x_img)) || (x_txt && !aligned16(x_txt)) || (x_joint && !aligned16(x_joint)))
    return KREA_DIT_ERR_MISALIGNED;
  const size_t es = h->esz, d = c.d_model;
  const size_t out_bytes = static_cast<size_t>(B) * L * d * es;
  if (overlaps(out, out_bytes, x_img, static_cast<size_t>(B) * n_img * d * es) ||
      overlaps(out, out_bytes, x_txt, static_cast<size_t>(B) * n_txt * d * es) ||
      overlaps(out, out_bytes, t_emb, static_cast<size_t>(B) * 6 * d * 4) ||
      (x_joint && out != x_joint && overlaps(out, out_bytes, x_joint, out_bytes)))
    return KREA_DIT_ERR_INVALID_ARG;
  if (B == 0 || L == 0) return KREA_DIT_OK;
  if (h->inject > 0) {
    --h->inject;
    return KREA_DIT_ERR_INJECTED;
  }

  Fwd f{};
  f.B = B;
  f.L = L;
  f.n_txt = n_txt;
  f.n_img = n_img;
  f.img_w = img_w > 0 ? img_w : 1;
  f.T = B * L;
  f.Lp = static_cast<int>(round_up(static_cast<size_t>(L), 64));
  f.d = c.d_model;
  f.n_q = c.n_q;
  f.n_kv = c.n_kv;
  f.hd = c.head_dim;
  f.F = c.ffn;
  f.gate_on = c.gate_on;
  f.eps = c.eps;
  h->last = f;
  h->have_last = true;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const RowSrc xsrc{x_txt, x_img, x_joint};
  const RowSrc h1src{nullptr, nullptr, h->h1};
  QkvgDst dst{h->q, h->k, h->vt, h->g, w->q_norm_w, w->k_norm_w, h->rope};
  if (h->bw_stats) {  // the backward's recomputed forward keeps its pre-activations
    dst.raw = h->f_raw;
    dst.ldr = h->n_qkvg;
  }
  const int nqhd = c.n_q * c.head_dim;
  cudaError_t e = cudaSuccess;
#define KD_RUN(slot, expr)                                 \
  do {                                                     \
    if (e == cudaSuccess) e = timed(h, slot, st, [&] { return (expr); }); \
  } while (0)

  if (h->mode4) {
    const uint64_t T = static_cast<uint64_t>(f.T);
    const uint64_t F = static_cast<uint64_t>(c.ffn), nq = static_cast<uint64_t>(nqhd);
    CUtensorMap tm_xn4, tm_wqkvg4, tm_og4, tm_wo4, tm_hn4, tm_wgate4, tm_wup4, tm_hmid4, tm_wdown4, tm_q, tm_k, tm_vt,
        tm_h1, tm_out, tm_g, tm_og;
    bool ok = encode_2d_u8(&tm_xn4, h->xn4, d / 2, T, 128) &&
              encode_2d_u8(&tm_wqkvg4, w4->w_qkvg, d / 2, h->n_qkvg, 128) &&
              encode_2d_u8(&tm_og4, h->og4, nq / 2, T, 128) && encode_2d_u8(&tm_wo4, w4->w_o, nq / 2, d, 128) &&
              encode_2d_u8(&tm_hn4, h->hn4, d / 2, T, 128) && encode_2d_u8(&tm_wgate4, w4->w_gate, d / 2, F, 128) &&
              encode_2d_u8(&tm_wup4, w4->w_up, d / 2, F, 128) && encode_2d_u8(&tm_hmid4, h->hmid4, F / 2, T, 128) &&
              encode_2d_u8(&tm_wdown4, w4->w_down, F / 2, d, 128) &&
              encode_3d(&tm_q, h->q, c.head_dim, L, static_cast<uint64_t>(B) * c.n_q, c.head_dim, 64, 128) &&
              encode_3d(&tm_k, h->k, c.head_dim, L, static_cast<uint64_t>(B) * c.n_kv, c.head_dim, 64, 128) &&
              encode_3d(&tm_vt, h->vt, L, c.head_dim, static_cast<uint64_t>(B) * c.n_kv, f.Lp, 64, 128) &&
              encode_2d_f32(&tm_h1, h->h1, d, T) && encode_2d(&tm_out, out, d, T, d, 64, 32) &&
              encode_attn_gate_out(&tm_g, &tm_og, h, B, L);
    if (!ok) return KREA_DIT_ERR_CUDA;
    const int sms = h->num_sms;
    const auto u8 = [](const void* p) { return static_cast<const uint8_t*>(p); };
    const kd::Op4 a_xn{&tm_xn4, u8(h->sf_xn4)}, a_og{&tm_og4, u8(h->sf_og4)}, a_hn{&tm_hn4, u8(h->sf_hn4)},
        a_hmid{&tm_hmid4, u8(h->sf_hmid4)};
    const kd::Op4 b_qkvg{&tm_wqkvg4, u8(w4->sf_qkvg)}, b_o{&tm_wo4, u8(w4->sf_o)}, b_gate{&tm_wgate4, u8(w4->sf_gate)},
        b_up{&tm_wup4, u8(w4->sf_up)}, b_down{&tm_wdown4, u8(w4->sf_down)};
    const kd::Deq dq_qkvg{h->ts4 + 0, w4->ts_qkvg, nullptr, 0};
    const kd::Deq dq_o{h->ts4 + 1, w4->ts_o, nullptr, 0};
    const kd::Deq dq_ff{h->ts4 + 2, w4->ts_gate, w4->ts_up, 0};
    const kd::Deq dq_down{h->ts4 + 3, w4->ts_down, nullptr, 0};
    // NVFP4 cast of a bf16 activation [T, K] whose row amaxes are in am: tensor scale, codes
    const auto cast4 = [&](const void* src, int K, float* am, float* ts, void* codes, void* sf) {
      KD_RUN(S_Q4_CAST, kd::launch_nvfp4_cast(src, f.T, K, am, ts, codes, sf, sms, st));
    };
    // row amax accumulators of the attention and SwiGLU outputs (atomic max from zero)
    e = cudaMemsetAsync(h->am_og, 0, T * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->am_hmid, 0, T * sizeof(float), st);
    // the norms store bf16 and each row's amax; the casts reduce those to the tensor scale
    const kd::NormQOut nq_xn{kd::NormQ::STORE_AMAX, nullptr, nullptr, h->am_xn};
    const kd::NormQOut nq_hn{kd::NormQ::STORE_AMAX, nullptr, nullptr, h->am_hn};
    KD_RUN(S_NORM1, kd::launch_norm_modulate(kd::NormIO::BF16_BF16, f, xsrc, w->norm1_w, t_emb, w->mod_bias, 0, 1,
                                             h->xn, sms, st, &nq_xn));
    cast4(h->xn, c.d_model, h->am_xn, h->ts4 + 0, h->xn4, h->sf_xn4);
    KD_RUN(S_QKVG_TC, kd::launch_gemm_qkvg_fp4(f, a_xn, b_qkvg, h->n_qkvg, dst, dq_qkvg, sms, h->err, st));
    KD_RUN(S_ATTN, kd::launch_attn_tc(f, &tm_q, &tm_k, &tm_vt, &tm_g, &tm_og, h->am_og, nullptr, nullptr, sms, h->err,
                                        st));
    cast4(h->og, nqhd, h->am_og, h->ts4 + 1, h->og4, h->sf_og4);
    KD_RUN(S_OPROJ_TC, kd::launch_gemm_resid_attn_fp4(f, a_og, b_o, nqhd, xsrc, t_emb, w->mod_bias, &tm_h1, dq_o, sms,
                                                      h->err, st));
    KD_RUN(S_NORM2, kd::launch_norm_modulate(kd::NormIO::F32_BF16, f, h1src, w->norm2_w, t_emb, w->mod_bias, 3, 4,
                                             h->hn, sms, st, &nq_hn));
    cast4(h->hn, c.d_model, h->am_hn, h->ts4 + 2, h->hn4, h->sf_hn4);
    KD_RUN(S_UPGATE_TC, kd::launch_gemm_swiglu_fp4(f, a_hn, b_gate, b_up, h->hmid, h->am_hmid, dq_ff, sms, h->err,
                                                   st));
    cast4(h->hmid, c.ffn, h->am_hmid, h->ts4 + 3, h->hmid4, h->sf_hmid4);
    KD_RUN(S_DOWN_TC, kd::launch_gemm_resid_mlp_fp4(f, a_hmid, b_down, c.ffn, static_cast<const float*>(h->h1), t_emb,
                                                    w->mod_bias, &tm_out, dq_down, sms, h->err, st));
  } else if (h->mode8) {
    const int per_row = h->mode8 == 2;
    const uint64_t T = static_cast<uint64_t>(f.T);
    CUtensorMap tm_xn8, tm_wqkvg, tm_og8, tm_wo, tm_hn8, tm_wgate, tm_wup, tm_hmid8, tm_wdown, tm_q, tm_k, tm_vt,
        tm_h1, tm_out, tm_g, tm_og;
    bool ok = encode_2d_u8(&tm_xn8, h->xn8, d, T, 128) && encode_2d_u8(&tm_wqkvg, w8->w_qkvg, d, h->n_qkvg, 128) &&
              encode_2d_u8(&tm_og8, h->og8, nqhd, T, 128) && encode_2d_u8(&tm_wo, w8->w_o, nqhd, d, 128) &&
              encode_2d_u8(&tm_hn8, h->hn8, d, T, 128) && encode_2d_u8(&tm_wgate, w8->w_gate, d, c.ffn, 128) &&
              encode_2d_u8(&tm_wup, w8->w_up, d, c.ffn, 128) && encode_2d_u8(&tm_hmid8, h->hmid8, c.ffn, T, 128) &&
              encode_2d_u8(&tm_wdown, w8->w_down, c.ffn, d, 128) &&
              encode_3d(&tm_q, h->q, c.head_dim, L, static_cast<uint64_t>(B) * c.n_q, c.head_dim, 64, 128) &&
              encode_3d(&tm_k, h->k, c.head_dim, L, static_cast<uint64_t>(B) * c.n_kv, c.head_dim, 64, 128) &&
              encode_3d(&tm_vt, h->vt, L, c.head_dim, static_cast<uint64_t>(B) * c.n_kv, f.Lp, 64, 128) &&
              encode_2d_f32(&tm_h1, h->h1, d, T) && encode_2d(&tm_out, out, d, T, d, 64, 32) &&
              encode_attn_gate_out(&tm_g, &tm_og, h, B, L);
    if (!ok) return KREA_DIT_ERR_CUDA;
    const int sms = h->num_sms;
    // row amax accumulators of the attention and SwiGLU outputs (atomic max from zero)
    e = cudaMemsetAsync(h->am_og, 0, T * sizeof(float), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(h->am_hmid, 0, T * sizeof(float), st);
    const kd::NormQ qmode = per_row ? kd::NormQ::ROW : kd::NormQ::TENSOR;
    const kd::NormQOut q_amax1{kd::NormQ::AMAX, nullptr, nullptr, h->am_xn};
    const kd::NormQOut q_xn{qmode, h->xn8, h->dq_xn, h->am_xn};
    const kd::NormQOut q_amax2{kd::NormQ::AMAX, nullptr, nullptr, h->am_hn};
    const kd::NormQOut q_hn{qmode, h->hn8, h->dq_hn, h->am_hn};
    const kd::Deq dq_qkvg{h->dq_xn, w8->dq_qkvg, nullptr, per_row};
    const kd::Deq dq_o{h->dq_og, w8->dq_o, nullptr, per_row};
    const kd::Deq dq_ff{h->dq_hn, w8->dq_gate, w8->dq_up, per_row};
    const kd::Deq dq_down{h->dq_hmid, w8->dq_down, nullptr, per_row};
    if (!per_row)
      KD_RUN(S_NORM1_AMAX, kd::launch_norm_modulate(kd::NormIO::BF16_BF16, f, xsrc, w->norm1_w, t_emb, w->mod_bias, 0,
                                                    1, nullptr, sms, st, &q_amax1));
    KD_RUN(S_NORM1, kd::launch_norm_modulate(kd::NormIO::BF16_BF16, f, xsrc, w->norm1_w, t_emb, w->mod_bias, 0, 1,
                                             nullptr, sms, st, &q_xn));
    KD_RUN(S_QKVG_TC, kd::launch_gemm_qkvg(f, &tm_xn8, &tm_wqkvg, h->n_qkvg, dst, &dq_qkvg, sms, h->err, st));
    KD_RUN(S_ATTN, kd::launch_attn_tc(f, &tm_q, &tm_k, &tm_vt, &tm_g, &tm_og, h->am_og, nullptr, nullptr, sms, h->err,
                                        st));
    KD_RUN(S_QUANT_OG, kd::launch_quant_e4m3(h->og, f.T, nqhd, h->am_og, per_row, h->og8, h->dq_og, sms, st));
    KD_RUN(S_OPROJ_TC, kd::launch_gemm_resid_attn(f, &tm_og8, &tm_wo, nqhd, xsrc, t_emb, w->mod_bias, &tm_h1, &dq_o,
                                                  nullptr, sms, h->err, st));
    if (!per_row)
      KD_RUN(S_NORM2_AMAX, kd::launch_norm_modulate(kd::NormIO::F32_BF16, f, h1src, w->norm2_w, t_emb, w->mod_bias, 3,
                                                    4, nullptr, sms, st, &q_amax2));
    KD_RUN(S_NORM2, kd::launch_norm_modulate(kd::NormIO::F32_BF16, f, h1src, w->norm2_w, t_emb, w->mod_bias, 3, 4,
                                             nullptr, sms, st, &q_hn));
    KD_RUN(S_UPGATE_TC, kd::launch_gemm_swiglu(f, &tm_hn8, &tm_wgate, &tm_wup, h->hmid, h->am_hmid, &dq_ff, nullptr,
                                               nullptr, sms, h->err, st));
    KD_RUN(S_QUANT_HMID,
           kd::launch_quant_e4m3(h->hmid, f.T, c.ffn, h->am_hmid, per_row, h->hmid8, h->dq_hmid, sms, st));
    KD_RUN(S_DOWN_TC, kd::launch_gemm_resid_mlp(f, &tm_hmid8, &tm_wdown, c.ffn, static_cast<const float*>(h->h1),
                                                t_emb, w->mod_bias, &tm_out, &dq_down, nullptr, sms, h->err, st));
  } else if (h->bf16) {
    CUtensorMap tm_xn, tm_wqkvg, tm_og, tm_wo, tm_hn, tm_wgate, tm_wup, tm_hmid, tm_wdown, tm_q, tm_k, tm_vt, tm_h1,
        tm_out, tm_g, tm_og_st;
    const uint64_t T = static_cast<uint64_t>(f.T);
    bool ok = encode_2d(&tm_xn, h->xn, d, T, d, 64, 128) &&
              encode_2d(&tm_wqkvg, w->w_qkvg, d, h->n_qkvg, d, 64, 128) &&
              encode_2d(&tm_og, h->og, nqhd, T, nqhd, 64, 128) &&
              encode_2d(&tm_wo, w->w_o, nqhd, d, nqhd, 64, 128) && encode_2d(&tm_hn, h->hn, d, T, d, 64, 128) &&
              encode_2d(&tm_wgate, w->w_gate, d, c.ffn, d, 64, 128) &&
              encode_2d(&tm_wup, w->w_up, d, c.ffn, d, 64, 128) &&
              encode_2d(&tm_hmid, h->hmid, c.ffn, T, c.ffn, 64, 128) &&
              encode_2d(&tm_wdown, w->w_down, c.ffn, d, c.ffn, 64, 128) &&
              encode_3d(&tm_q, h->q, c.head_dim, L, static_cast<uint64_t>(B) * c.n_q, c.head_dim, 64, 128) &&
              encode_3d(&tm_k, h->k, c.head_dim, L, static_cast<uint64_t>(B) * c.n_kv, c.head_dim, 64, 128) &&
              encode_3d(&tm_vt, h->vt, L, c.head_dim, static_cast<uint64_t>(B) * c.n_kv, f.Lp, 64, 128) &&
              encode_2d_f32(&tm_h1, h->h1, d, T) && encode_2d(&tm_out, out, d, T, d, 64, 32) &&
              encode_attn_gate_out(&tm_g, &tm_og_st, h, B, L);
    if (!ok) return KREA_DIT_ERR_CUDA;
    const int sms = h->num_sms;
    KD_RUN(S_NORM1, kd::launch_norm_modulate(kd::NormIO::BF16_BF16, f, xsrc, w->norm1_w, t_emb, w->mod_bias, 0, 1,
                                             h->xn, sms, st));
    KD_RUN(S_QKVG_TC, kd::launch_gemm_qkvg(f, &tm_xn, &tm_wqkvg, h->n_qkvg, dst, nullptr, sms, h->err, st));
    KD_RUN(S_ATTN, kd::launch_attn_tc(f, &tm_q, &tm_k, &tm_vt, &tm_g, &tm_og_st, nullptr, h->bw_stats ? h->f_lse : nullptr,
                                        h->bw_stats ? h->f_o : nullptr, sms, h->err, st));
    KD_RUN(S_OPROJ_TC, kd::launch_gemm_resid_attn(f, &tm_og, &tm_wo, nqhd, xsrc, t_emb, w->mod_bias, &tm_h1, nullptr,
                                                  h->bw_stats ? h->f_fa : nullptr, sms, h->err, st));
    KD_RUN(S_NORM2, kd::launch_norm_modulate(kd::NormIO::F32_BF16, f, h1src, w->norm2_w, t_emb, w->mod_bias, 3, 4,
                                             h->hn, sms, st));
    KD_RUN(S_UPGATE_TC, kd::launch_gemm_swiglu(f, &tm_hn, &tm_wgate, &tm_wup, h->hmid, nullptr, nullptr,
                                               h->bw_stats ? h->f_a : nullptr, h->bw_stats ? h->f_u : nullptr,
                                               sms, h->err, st));
    KD_RUN(S_DOWN_TC, kd::launch_gemm_resid_mlp(f, &tm_hmid, &tm_wdown, c.ffn, static_cast<const float*>(h->h1),
                                                t_emb, w->mod_bias, &tm_out, nullptr, h->bw_stats ? h->f_td : nullptr,
                                                sms, h->err, st));
  } else {
    const int T = f.T;
    const float* wq = static_cast<const float*>(w->w_qkvg);
    KD_RUN(S_NORM1, kd::launch_norm_modulate(kd::NormIO::F32_F32, f, xsrc, w->norm1_w, t_emb, w->mod_bias, 0, 1,
                                             h->xn, h->num_sms, st));
    KD_RUN(S_QKVG_F32, kd::launch_gemm_simt_f32(static_cast<const float*>(h->xn), wq, h->raw_qkvg, T, h->n_qkvg,
                                                c.d_model, nullptr, 0, st));
    KD_RUN(S_QKVG_POST_F32, kd::launch_qkvg_post_f32(f, h->raw_qkvg, dst, st));
    KD_RUN(S_ATTN, kd::launch_attn_simt(false, f, h->q, h->k, h->vt, h->g, h->og, st));
    KD_RUN(S_OPROJ_F32, kd::launch_gemm_simt_f32(static_cast<const float*>(h->og), static_cast<const float*>(w->w_o),
                                                 h->raw_o, T, c.d_model, nqhd, nullptr, 0, st));
    KD_RUN(S_RESID_ATTN_F32, kd::launch_residual_f32(f, xsrc, h->raw_o, t_emb, w->mod_bias, 2,
                                                     static_cast<float*>(h->h1), st));
    KD_RUN(S_NORM2, kd::launch_norm_modulate(kd::NormIO::F32_F32, f, h1src, w->norm2_w, t_emb, w->mod_bias, 3, 4,
                                             h->hn, h->num_sms, st));
    KD_RUN(S_GATE_F32, kd::launch_gemm_simt_f32(static_cast<const float*>(h->hn),
                                                static_cast<const float*>(w->w_gate), h->raw_a, T, c.ffn, c.d_model,
                                                nullptr, 0, st));
    KD_RUN(S_UP_F32, kd::launch_gemm_simt_f32(static_cast<const float*>(h->hn), static_cast<const float*>(w->w_up),
                                              h->raw_u, T, c.ffn, c.d_model, nullptr, 0, st));
    KD_RUN(S_SWIGLU_F32, kd::launch_swiglu_f32(f, h->raw_a, h->raw_u, static_cast<float*>(h->hmid), st));
    KD_RUN(S_DOWN_F32, kd::launch_gemm_simt_f32(static_cast<const float*>(h->hmid),
                                                static_cast<const float*>(w->w_down), h->raw_down, T, c.d_model,
                                                c.ffn, nullptr, 0, st));
    KD_RUN(S_RESID_MLP_F32,
           kd::launch_residual_f32(f, h1src, h->raw_down, t_emb, w->mod_bias, 5, static_cast<float*>(out), st));
  }
#undef KD_RUN
  return e == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

}  // namespace

extern "C" {

int krea_dit_block_forward(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                           int n_txt, const float* t_emb, const krea_dit_weights* w, void* out,
                           krea_dit_stream_t stream) {
  return forward_impl(h, x_img, x_txt, nullptr, B, img_h, img_w, n_txt, t_emb, w, nullptr, out, stream);
}

int krea_dit_block_forward8(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                            int n_txt, const float* t_emb, const krea_dit_weights* w, const krea_dit_weights8* q,
                            void* out, krea_dit_stream_t stream) {
  if (!q) return KREA_DIT_ERR_INVALID_ARG;
  return forward_impl(h, x_img, x_txt, nullptr, B, img_h, img_w, n_txt, t_emb, w, q, out, stream);
}

size_t krea_dit_nvfp4_scale_bytes(int rows, int cols) { return kd::nvfp4_scale_bytes(rows, cols); }

int krea_dit_block_forward4(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                            int n_txt, const float* t_emb, const krea_dit_weights* w, const krea_dit_weights4* q,
                            void* out, krea_dit_stream_t stream) {
  if (!q) return KREA_DIT_ERR_INVALID_ARG;
  return forward_impl(h, x_img, x_txt, nullptr, B, img_h, img_w, n_txt, t_emb, w, nullptr, out, stream, q);
}

int krea_dit_weights4_quantize(krea_dit_block_t h, const krea_dit_weights* w, const krea_dit_weights4* q,
                               krea_dit_stream_t stream) {
  if (!h || !w || !q || !h->mode4) return KREA_DIT_ERR_INVALID_ARG;
  const krea_dit_config& c = h->cfg;
  const int d = c.d_model, F = c.ffn, nqhd = c.n_q * c.head_dim;
  struct Mat {
    const void* src;
    int rows, cols;
    void* codes;
    void* sf;
    float* ts;
  };
  const Mat mats[5] = {{w->w_qkvg, h->n_qkvg, d, q->w_qkvg, q->sf_qkvg, q->ts_qkvg},
                       {w->w_o, d, nqhd, q->w_o, q->sf_o, q->ts_o},
                       {w->w_gate, F, d, q->w_gate, q->sf_gate, q->ts_gate},
                       {w->w_up, F, d, q->w_up, q->sf_up, q->ts_up},
                       {w->w_down, d, F, q->w_down, q->sf_down, q->ts_down}};
  for (const Mat& m : mats) {
    if (!m.src || !m.codes || !m.sf || !m.ts) return KREA_DIT_ERR_INVALID_ARG;
    if (!aligned16(m.src) || !aligned16(m.codes) || !aligned16(m.sf) || !aligned16(m.ts))
      return KREA_DIT_ERR_MISALIGNED;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  for (const Mat& m : mats) {
    if (e == cudaSuccess)
      e = timed(h, S_Q4_AMAX, st, [&] { return kd::launch_row_amax(m.src, m.rows, m.cols, h->am_w, h->num_sms, st); });
    if (e == cudaSuccess)
      e = timed(h, S_Q4_CAST, st, [&] {
        return kd::launch_nvfp4_cast(m.src, m.rows, m.cols, h->am_w, m.ts, m.codes, m.sf, h->num_sms, st);
      });
  }
  return e == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

int krea_dit_weights8_quantize(krea_dit_block_t h, const krea_dit_weights* w, const krea_dit_weights8* q,
                               krea_dit_stream_t stream) {
  if (!h || !w || !q || !h->mode8) return KREA_DIT_ERR_INVALID_ARG;
  const krea_dit_config& c = h->cfg;
  const int d = c.d_model, F = c.ffn, nqhd = c.n_q * c.head_dim;
  struct Mat {
    const void* src;
    int rows, cols;
    void* codes;
    float* dq;
  };
  const Mat mats[5] = {{w->w_qkvg, h->n_qkvg, d, q->w_qkvg, q->dq_qkvg},
                       {w->w_o, d, nqhd, q->w_o, q->dq_o},
                       {w->w_gate, F, d, q->w_gate, q->dq_gate},
                       {w->w_up, F, d, q->w_up, q->dq_up},
                       {w->w_down, d, F, q->w_down, q->dq_down}};
  for (const Mat& m : mats) {
    if (!m.src || !m.codes || !m.dq) return KREA_DIT_ERR_INVALID_ARG;
    if (!aligned16(m.src) || !aligned16(m.codes) || !aligned16(m.dq)) return KREA_DIT_ERR_MISALIGNED;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int per_row = h->mode8 == 2;
  cudaError_t e = cudaSuccess;
  for (const Mat& m : mats) {
    if (e == cudaSuccess)
      e = timed(h, S_W8_AMAX, st, [&] { return kd::launch_row_amax(m.src, m.rows, m.cols, h->am_w, h->num_sms, st); });
    if (e == cudaSuccess)
      e = timed(h, S_W8_QUANT, st, [&] {
        return kd::launch_quant_e4m3(m.src, m.rows, m.cols, h->am_w, per_row, m.codes, m.dq, h->num_sms, st);
      });
  }
  return e == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

int krea_dit_block_forward_joint(krea_dit_block_t h, const void* x, int B, int img_h, int img_w, int n_txt,
                                 const float* t_emb, const krea_dit_weights* w, void* out,
                                 krea_dit_stream_t stream) {
  if (!x) return KREA_DIT_ERR_INVALID_ARG;
  return forward_impl(h, nullptr, nullptr, x, B, img_h, img_w, n_txt, t_emb, w, nullptr, out, stream);
}

int krea_dit_stack_forward(krea_dit_block_t h, void* x, int B, int img_h, int img_w, int n_txt, const float* t_emb,
                           const krea_dit_weights* w, int n_blocks, krea_dit_stream_t stream) {
  if (!h || !x || n_blocks < 0 || (n_blocks > 0 && !w)) return KREA_DIT_ERR_INVALID_ARG;
  for (int i = 0; i < n_blocks; ++i) {
    const int r = forward_impl(h, nullptr, nullptr, x, B, img_h, img_w, n_txt, t_emb, &w[i], nullptr, x, stream);
    if (r != KREA_DIT_OK) return r;
  }
  return KREA_DIT_OK;
}

}  // extern "C"

struct krea_dit_graph_s : GraphBox {};

extern "C" {

int krea_dit_stack_graph_create(krea_dit_block_t h, void* x, int B, int img_h, int img_w, int n_txt,
                                const float* t_emb, const krea_dit_weights* w, int n_blocks, krea_dit_stream_t stream,
                                krea_dit_graph_t* out) {
  if (!out) return KREA_DIT_ERR_INVALID_ARG;
  *out = nullptr;
  if (!h || !x || n_blocks < 0 || (n_blocks > 0 && !w) || !stream) return KREA_DIT_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return KREA_DIT_ERR_INVALID_ARG;
  const bool timing = h->timing;
  h->timing = false;  // no event records inside the graph
  if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    h->timing = timing;
    return KREA_DIT_ERR_CUDA;
  }
  const int r = krea_dit_stack_forward(h, x, B, img_h, img_w, n_txt, t_emb, w, n_blocks, stream);
  cudaGraph_t graph = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(st, &graph);
  h->timing = timing;
  if (r != KREA_DIT_OK || ec != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    return r != KREA_DIT_OK ? r : KREA_DIT_ERR_CUDA;
  }
  krea_dit_graph_s* g = new (std::nothrow) krea_dit_graph_s();
  if (!g || cudaGraphInstantiate(&g->exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    delete g;
    return KREA_DIT_ERR_CUDA;
  }
  g->graph = graph;
  *out = g;
  return KREA_DIT_OK;
}

int krea_dit_graph_launch(krea_dit_graph_t g, krea_dit_stream_t stream) {
  if (!g) return KREA_DIT_ERR_INVALID_ARG;
  return cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KREA_DIT_OK
                                                                                           : KREA_DIT_ERR_CUDA;
}

int krea_dit_graph_destroy(krea_dit_graph_t g) {
  if (!g) return KREA_DIT_OK;
  cudaGraphExecDestroy(g->exec);
  cudaGraphDestroy(g->graph);
  delete g;
  return KREA_DIT_OK;
}

int krea_dit_block_enable_backward(krea_dit_block_t h) {
  if (!h) return KREA_DIT_ERR_INVALID_ARG;
  if (!h->bf16 || h->mode8 || h->mode4) return KREA_DIT_ERR_INVALID_ARG;  // bf16 mode only
  if (h->bw) return KREA_DIT_OK;
  const krea_dit_config& c = h->cfg;
  const size_t T = h->max_T, d = c.d_model, F = c.ffn, hd = c.head_dim;
  const size_t nq = static_cast<size_t>(c.n_q) * hd, nkv = static_cast<size_t>(c.n_kv) * hd, nqkvg = h->n_qkvg;
  const size_t Tp = round_up(T, 64), Lp = round_up(static_cast<size_t>(c.max_seq), 64);
  struct Item {
    void** p;
    size_t bytes;
  };
  std::vector<Item> items = {
      {&h->bw_out, T * d * 2},
      {&h->wT_down, F * d * 2},
      {&h->wT_gu, d * 2 * F * 2},
      {&h->wT_o, nq * d * 2},
      {&h->wT_qkvg, d * nqkvg * 2},
      {reinterpret_cast<void**>(&h->f_td), T * d * 4},
      {reinterpret_cast<void**>(&h->f_fa), T * d * 4},
      {reinterpret_cast<void**>(&h->f_a), T * F * 4},
      {reinterpret_cast<void**>(&h->f_u), T * F * 4},
      {reinterpret_cast<void**>(&h->f_dn), T * d * 4},
      {reinterpret_cast<void**>(&h->f_dh1), T * d * 4},
      {reinterpret_cast<void**>(&h->f_o), T * nq * 4},
      {reinterpret_cast<void**>(&h->f_raw), T * nqkvg * 4},
      {reinterpret_cast<void**>(&h->f_dq), T * nq * 4},
      {reinterpret_cast<void**>(&h->f_dk), T * nkv * 4},
      {reinterpret_cast<void**>(&h->f_dv), T * nkv * 4},
      {reinterpret_cast<void**>(&h->f_rstd), T * 4},
      {reinterpret_cast<void**>(&h->f_lse), static_cast<size_t>(c.max_batch) * c.n_q * Lp * 4},
      {reinterpret_cast<void**>(&h->f_D), static_cast<size_t>(c.max_batch) * c.n_q * Lp * 4},
      {&h->b_dfm, T * d * 2},
      {&h->b_dau, T * 2 * F * 2},
      {&h->b_dfa, T * d * 2},
      {&h->b_do, T * nq * 2},
      {&h->b_dP, T * nqkvg * 2},
      {&h->b_vrow, static_cast<size_t>(c.max_batch) * c.n_kv * c.max_seq * hd * 2},
      {&h->b_kT, static_cast<size_t>(c.max_batch) * c.n_kv * hd * Lp * 2},
      {&h->b_qT, static_cast<size_t>(c.max_batch) * c.n_q * hd * Lp * 2},
      {&h->b_doT, static_cast<size_t>(c.max_batch) * c.n_q * hd * Lp * 2},
      {&h->t_dfm, d * Tp * 2},
      {&h->t_hmid, F * Tp * 2},
      {&h->t_dau, 2 * F * Tp * 2},
      {&h->t_hn, d * Tp * 2},
      {&h->t_dfa, d * Tp * 2},
      {&h->t_og, nq * Tp * 2},
      {&h->t_dP, nqkvg * Tp * 2},
      {&h->t_xn, d * Tp * 2},
  };
  size_t total = 0;
  for (auto& it : items) total += round_up(it.bytes, 256);
  char* base = nullptr;
  if (cudaMalloc(&base, total) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  if (cudaMemset(base, 0, total) != cudaSuccess) {
    cudaFree(base);
    return KREA_DIT_ERR_CUDA;
  }
  size_t off = 0;
  for (auto& it : items) {
    *it.p = base + off;
    off += round_up(it.bytes, 256);
  }
  h->bw = base;
  h->bw_Tp = Tp;
  h->bw_Lp = Lp;
  return KREA_DIT_OK;
}

int krea_dit_block_backward(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                            int n_txt, const float* t_emb, const krea_dit_weights* w, const void* d_out,
                            const krea_dit_grads* g, krea_dit_stream_t stream) {
  if (!h || !w || !g || !d_out || !t_emb) return KREA_DIT_ERR_INVALID_ARG;
  if (!h->bw) return KREA_DIT_ERR_INVALID_ARG;  // krea_dit_block_enable_backward first
  const float* gp[] = {g->d_w_qkvg, g->d_w_o, g->d_w_gate, g->d_w_up, g->d_w_down, g->d_norm1_w, g->d_norm2_w,
                       g->d_q_norm_w, g->d_k_norm_w, g->d_mod_bias, g->d_mod_shared};
  for (const float* p : gp) {
    if (!p) return KREA_DIT_ERR_INVALID_ARG;
    if (!aligned16(p)) return KREA_DIT_ERR_MISALIGNED;
  }
  const int n_img = img_h * img_w;
  if ((n_img > 0 && !g->d_x_img) || (n_txt > 0 && !g->d_x_txt)) return KREA_DIT_ERR_INVALID_ARG;
  if (!aligned16(d_out) || (g->d_x_img && !aligned16(g->d_x_img)) || (g->d_x_txt && !aligned16(g->d_x_txt)))
    return KREA_DIT_ERR_MISALIGNED;
  // the forward, recomputed: fills the workspace (xn, Q, K, V^T, G, O_g, h1, hn, hmid)
  h->bw_stats = true;  // the attention also leaves lse and the ungated output
  int r = forward_impl(h, x_img, x_txt, nullptr, B, img_h, img_w, n_txt, t_emb, w, nullptr, h->bw_out, stream);
  h->bw_stats = false;
  if (r != KREA_DIT_OK) return r;
  const Fwd f = h->last;
  if (f.T == 0) return KREA_DIT_OK;
  const krea_dit_config& c = h->cfg;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int sms = h->num_sms;
  const int T = f.T, d = c.d_model, F = c.ffn, hd = c.head_dim, L = f.L;
  const int nq = c.n_q * hd, nkv = c.n_kv * hd, nqkvg = h->n_qkvg;
  const int Tp = static_cast<int>(round_up(static_cast<size_t>(T), 64));
  const int Lp = static_cast<int>(round_up(static_cast<size_t>(L), 64));
  const float scale = 1.0f / sqrtf(static_cast<float>(hd));
  float* d_mod = g->d_mod_shared;
  float* d_bias = g->d_mod_bias;
  cudaError_t e = cudaSuccess;
  auto run = [&](int slot, auto&& fn) {
    if (e == cudaSuccess) e = timed(h, slot, st, fn);
  };
  // C[M,N] (+)= alpha * A[M,K] B[N,K]^T, A / B bf16 row-major with pitches (elements)
  auto gemm = [&](const void* A, int a_rows, long long a_pitch, const void* Bm, int b_rows, long long b_pitch, int K,
                  float* C, long long ldc, int M, int N, float alpha, int acc) {
    run(S_BWD_GEMM, [&]() -> cudaError_t {
      CUtensorMap ta, tb;
      if (!encode_2d(&ta, A, K, a_rows, a_pitch, 64, 128) || !encode_2d(&tb, Bm, K, b_rows, b_pitch, 64, 128))
        return cudaErrorInvalidValue;
      return kd::launch_gemm_plain(&ta, &tb, M, N, K, C, ldc, alpha, acc, sms, h->err, st);
    });
  };
  auto transpose = [&](const void* src, int R, int C, long long lds, long long sbs, void* dst, int Rp, long long ldd,
                       long long dbs, int batch) {
    run(S_BWD_TRANSPOSE, [&] { return kd::launch_transpose_bf16(src, R, C, lds, sbs, dst, Rp, ldd, dbs, batch, st); });
  };
  // element offsets into bf16 buffers (2 bytes per element)
  auto bf = [](const void* p, long long off) { return static_cast<const void*>(static_cast<const char*>(p) + 2 * off); };
  auto bfw = [](void* p, long long off) { return static_cast<void*>(static_cast<char*>(p) + 2 * off); };

  // accumulators
  if (e == cudaSuccess) e = cudaMemsetAsync(d_mod, 0, static_cast<size_t>(B) * 6 * d * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(d_bias, 0, static_cast<size_t>(6) * d * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(g->d_norm1_w, 0, static_cast<size_t>(d) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(g->d_norm2_w, 0, static_cast<size_t>(d) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(g->d_q_norm_w, 0, static_cast<size_t>(hd) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(g->d_k_norm_w, 0, static_cast<size_t>(hd) * 4, st);
  // weights as K-major operands of the data-gradient products
  transpose(w->w_down, d, F, F, 0, h->wT_down, d, d, 0, 1);                    // [F, d]
  transpose(w->w_gate, F, d, d, 0, h->wT_gu, F, 2LL * F, 0, 1);                // [d, 0:F]
  transpose(w->w_up, F, d, d, 0, bfw(h->wT_gu, F), F, 2LL * F, 0, 1);          // [d, F:2F]
  transpose(w->w_o, d, nq, nq, 0, h->wT_o, d, d, 0, 1);                        // [nq, d]
  transpose(w->w_qkvg, nqkvg, d, d, 0, h->wT_qkvg, nqkvg, nqkvg, 0, 1);        // [d, nqkvg]

  // ---- MLP residual: out = h1 + gate_m * fm,  fm = hmid W_down^T (kept by the forward in f_td)
  run(S_BWD_POINTWISE, [&] {
    return kd::launch_gated_bwd(f, d_out, 0, h->f_td, t_emb, w->mod_bias, 5, h->b_dfm, d_mod, d_bias, st);
  });
  // ---- d_hmid = d_fm W_down and the SwiGLU backward in its epilogue (a, u kept by the forward)
  run(S_BWD_GEMM, [&]() -> cudaError_t {
    CUtensorMap ta, tb;
    if (!encode_2d(&ta, h->b_dfm, d, T, d, 64, 128) || !encode_2d(&tb, h->wT_down, d, F, d, 64, 128))
      return cudaErrorInvalidValue;
    return kd::launch_gemm_swiglu_bwd(&ta, &tb, T, F, d, h->f_a, h->f_u, h->b_dau, sms, h->err, st);
  });
  gemm(h->b_dau, T, 2LL * F, h->wT_gu, d, 2LL * F, 2 * F, h->f_dn, d, T, d, 1.0f, 0);  // d_hn
  // ---- norm2 + modulation; the residual adds d_out
  const RowSrc h1src{nullptr, nullptr, h->h1};
  run(S_BWD_POINTWISE, [&] {
    return kd::launch_norm_bwd(f, h1src, 1, h->f_dn, w->norm2_w, t_emb, w->mod_bias, 3, 4, d_out, 0, h->f_dh1,
                               RowSrc{}, h->f_rstd, d_mod, d_bias, g->d_norm2_w, st);
  });
  // ---- attention residual: h1 = x + gate_a * fa,  fa = og W_o^T (kept by the forward)
  run(S_BWD_POINTWISE, [&] {
    return kd::launch_gated_bwd(f, h->f_dh1, 1, h->f_fa, t_emb, w->mod_bias, 2, h->b_dfa, d_mod, d_bias, st);
  });
  // d_og = d_fa W_o, with the gate backward and D = rowsum(d_o o) in its epilogue
  run(S_BWD_GEMM, [&]() -> cudaError_t {
    CUtensorMap ta, tb;
    if (!encode_2d(&ta, h->b_dfa, d, T, d, 64, 128) || !encode_2d(&tb, h->wT_o, d, nq, d, 64, 128))
      return cudaErrorInvalidValue;
    return kd::launch_gemm_gate_bwd(f, &ta, &tb, d, h->f_o, h->g, h->b_do, h->b_dP, nqkvg, nq + 2 * nkv, h->f_D, sms,
                                    h->err, st);
  });
  // ---- attention: the forward left each row's log2 normaliser (lse) and the ungated
  // output o; two flash-style kernels recompute P and dP tile by tile in TMEM (no L x L
  // array in memory) and give dQ, dK, dV in fp32.
  const long long qh = static_cast<long long>(L) * hd;  // one head of Q / K (elements)
  // head-dim-major copies (B operands of dQ, dK, dV) and row-major V [B n_kv, L, hd]
  transpose(h->vt, hd, L, f.Lp, static_cast<long long>(hd) * f.Lp, h->b_vrow, hd, hd, qh, B * c.n_kv);
  transpose(h->k, L, hd, hd, qh, h->b_kT, Lp, Lp, static_cast<long long>(hd) * Lp, B * c.n_kv);
  transpose(h->q, L, hd, hd, qh, h->b_qT, Lp, Lp, static_cast<long long>(hd) * Lp, B * c.n_q);
  transpose(h->b_do, L, hd, hd, qh, h->b_doT, Lp, Lp, static_cast<long long>(hd) * Lp, B * c.n_q);
  run(S_BWD_ATTN, [&]() -> cudaError_t {
    const uint64_t pq = static_cast<uint64_t>(B) * c.n_q, pkv = static_cast<uint64_t>(B) * c.n_kv;
    CUtensorMap tm_q, tm_do, tm_k, tm_v, tm_qt, tm_dot, tm_kt;
    if (!encode_3d(&tm_q, h->q, hd, L, pq, hd, 64, 128) || !encode_3d(&tm_do, h->b_do, hd, L, pq, hd, 64, 128) ||
        !encode_3d(&tm_k, h->k, hd, L, pkv, hd, 64, 128) || !encode_3d(&tm_v, h->b_vrow, hd, L, pkv, hd, 64, 128) ||
        !encode_3d(&tm_qt, h->b_qT, L, hd, pq, Lp, 64, 128) || !encode_3d(&tm_dot, h->b_doT, L, hd, pq, Lp, 64, 128) ||
        !encode_3d(&tm_kt, h->b_kT, L, hd, pkv, Lp, 64, 128))
      return cudaErrorInvalidValue;
    return kd::launch_attn_bwd(f, &tm_q, &tm_do, &tm_k, &tm_v, &tm_qt, &tm_dot, &tm_kt, h->f_lse, h->f_D, h->f_dq,
                               h->f_dk, h->f_dv, h->err, st);
  });
  // ---- QK-norm + RoPE and V into d_P (the Q, K projections before the norm kept by the forward)
  run(S_BWD_POINTWISE, [&] {
    return kd::launch_qkv_bwd(f, h->f_raw, nqkvg, h->f_dq, h->f_dk, h->f_dv, w->q_norm_w, w->k_norm_w, h->rope,
                              h->b_dP, nqkvg, g->d_q_norm_w, g->d_k_norm_w, st);
  });
  gemm(h->b_dP, T, nqkvg, h->wT_qkvg, d, nqkvg, nqkvg, h->f_dn, d, T, d, 1.0f, 0);  // d_xn
  // ---- norm1 + modulation; the residual adds d_h1; d_x in the storage dtype, split
  const RowSrc xsrc{x_txt, x_img, nullptr};
  const RowSrc dxs{g->d_x_txt, g->d_x_img, nullptr};
  run(S_BWD_POINTWISE, [&] {
    return kd::launch_norm_bwd(f, xsrc, 0, h->f_dn, w->norm1_w, t_emb, w->mod_bias, 0, 1, h->f_dh1, 1, nullptr, dxs,
                               h->f_rstd, d_mod, d_bias, g->d_norm1_w, st);
  });
  // ---- weight gradients: dW = dY^T X over the T rows (both operands transposed, K = Tp)
  transpose(h->b_dfm, T, d, d, 0, h->t_dfm, Tp, Tp, 0, 1);
  transpose(h->hmid, T, F, F, 0, h->t_hmid, Tp, Tp, 0, 1);
  gemm(h->t_dfm, d, Tp, h->t_hmid, F, Tp, Tp, g->d_w_down, F, d, F, 1.0f, 0);
  transpose(h->b_dau, T, 2 * F, 2LL * F, 0, h->t_dau, Tp, Tp, 0, 1);
  transpose(h->hn, T, d, d, 0, h->t_hn, Tp, Tp, 0, 1);
  gemm(h->t_dau, F, Tp, h->t_hn, d, Tp, Tp, g->d_w_gate, d, F, d, 1.0f, 0);
  gemm(bf(h->t_dau, static_cast<long long>(F) * Tp), F, Tp, h->t_hn, d, Tp, Tp, g->d_w_up, d, F, d, 1.0f, 0);
  transpose(h->b_dfa, T, d, d, 0, h->t_dfa, Tp, Tp, 0, 1);
  transpose(h->og, T, nq, nq, 0, h->t_og, Tp, Tp, 0, 1);
  gemm(h->t_dfa, d, Tp, h->t_og, nq, Tp, Tp, g->d_w_o, nq, d, nq, 1.0f, 0);
  transpose(h->b_dP, T, nqkvg, nqkvg, 0, h->t_dP, Tp, Tp, 0, 1);
  transpose(h->xn, T, d, d, 0, h->t_xn, Tp, Tp, 0, 1);
  gemm(h->t_dP, nqkvg, Tp, h->t_xn, d, Tp, Tp, g->d_w_qkvg, d, nqkvg, d, 1.0f, 0);
  return e == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

int krea_dit_block_enable_host_io(krea_dit_block_t h) {
  if (!h) return KREA_DIT_ERR_INVALID_ARG;
  if (h->host_io) return KREA_DIT_OK;
  const size_t tokens = static_cast<size_t>(h->cfg.max_batch) * h->cfg.max_seq;
  h->stage_in_bytes = round_up(tokens * h->cfg.d_model * h->esz, 256);
  h->stage_out_bytes = h->stage_in_bytes;
  if (cudaMalloc(&h->stage, 2 * (h->stage_in_bytes + h->stage_out_bytes)) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  bool ok = cudaStreamCreateWithFlags(&h->up, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&h->down, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < 2; ++i)
    ok = cudaEventCreateWithFlags(&h->ev_in[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&h->ev_comp[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&h->ev_out[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) return KREA_DIT_ERR_CUDA;
  h->host_io = true;
  return KREA_DIT_OK;
}

int krea_dit_block_forward_host(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                                int n_txt, const float* t_emb, const krea_dit_weights* w, void* out,
                                krea_dit_stream_t stream) {
  if (!h || !out) return KREA_DIT_ERR_INVALID_ARG;
  if (!h->host_io) return KREA_DIT_ERR_INVALID_ARG;
  if (B < 0 || img_h < 0 || img_w < 0 || n_txt < 0) return KREA_DIT_ERR_INVALID_ARG;
  const long long n_img = static_cast<long long>(img_h) * img_w, L = n_img + n_txt;
  if (B > h->cfg.max_batch || L > h->cfg.max_seq) return KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS;
  if ((n_img > 0 && !x_img) || (n_txt > 0 && !x_txt)) return KREA_DIT_ERR_INVALID_ARG;
  if (B == 0 || L == 0) return KREA_DIT_OK;
  const size_t row = static_cast<size_t>(h->cfg.d_model) * h->esz;
  const size_t img_bytes = static_cast<size_t>(B) * n_img * row, txt_bytes = static_cast<size_t>(B) * n_txt * row;
  const size_t out_bytes = static_cast<size_t>(B) * L * row;
  const int k = h->next_set;
  char* base = h->stage + k * (h->stage_in_bytes + h->stage_out_bytes);
  char* d_img = base;
  char* d_txt = base + round_up(img_bytes, 256);
  char* d_out = base + h->stage_in_bytes;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // upload: the set's previous forward must have finished reading its inputs
  if (h->set_used[k] && cudaStreamWaitEvent(h->up, h->ev_comp[k], 0) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  if (img_bytes && cudaMemcpyAsync(d_img, x_img, img_bytes, cudaMemcpyHostToDevice, h->up) != cudaSuccess)
    return KREA_DIT_ERR_CUDA;
  if (txt_bytes && cudaMemcpyAsync(d_txt, x_txt, txt_bytes, cudaMemcpyHostToDevice, h->up) != cudaSuccess)
    return KREA_DIT_ERR_CUDA;
  if (cudaEventRecord(h->ev_in[k], h->up) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  // compute: inputs landed, and the set's previous download has read the output staging
  if (cudaStreamWaitEvent(st, h->ev_in[k], 0) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  if (h->set_used[k] && cudaStreamWaitEvent(st, h->ev_out[k], 0) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  const int r = krea_dit_block_forward(h, n_img ? d_img : nullptr, n_txt ? d_txt : nullptr, B, img_h, img_w, n_txt,
                                       t_emb, w, d_out, stream);
  if (r != KREA_DIT_OK) return r;
  if (cudaEventRecord(h->ev_comp[k], st) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  // download
  if (cudaStreamWaitEvent(h->down, h->ev_comp[k], 0) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  if (cudaMemcpyAsync(out, d_out, out_bytes, cudaMemcpyDeviceToHost, h->down) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  if (cudaEventRecord(h->ev_out[k], h->down) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  h->set_used[k] = true;
  h->next_set = 1 - k;
  return KREA_DIT_OK;
}

int krea_dit_block_host_sync(krea_dit_block_t h) {
  if (!h) return KREA_DIT_ERR_INVALID_ARG;
  if (!h->host_io) return KREA_DIT_OK;
  if (cudaStreamSynchronize(h->up) != cudaSuccess || cudaStreamSynchronize(h->down) != cudaSuccess)
    return KREA_DIT_ERR_CUDA;
  return KREA_DIT_OK;
}

int krea_dit_block_workspace(krea_dit_block_t h, int which, void** dev_ptr, size_t* bytes) {
  if (!h || !dev_ptr || !bytes) return KREA_DIT_ERR_INVALID_ARG;
  const Fwd& f = h->last;
  const size_t es = h->esz;
  const size_t T = h->have_last ? static_cast<size_t>(f.T) : 0;
  const size_t hd = h->cfg.head_dim;
  switch (which) {
    case KREA_DIT_BUF_XN: *dev_ptr = h->xn; *bytes = T * h->cfg.d_model * es; break;
    case KREA_DIT_BUF_Q: *dev_ptr = h->q; *bytes = T * h->cfg.n_q * hd * es; break;
    case KREA_DIT_BUF_K: *dev_ptr = h->k; *bytes = T * h->cfg.n_kv * hd * es; break;
    case KREA_DIT_BUF_VT:
      *dev_ptr = h->vt;
      *bytes = h->have_last ? static_cast<size_t>(f.B) * h->cfg.n_kv * hd * f.Lp * es : 0;
      break;
    case KREA_DIT_BUF_G: *dev_ptr = h->g; *bytes = T * h->cfg.n_q * hd * es; break;
    case KREA_DIT_BUF_OG: *dev_ptr = h->og; *bytes = T * h->cfg.n_q * hd * es; break;
    case KREA_DIT_BUF_H1: *dev_ptr = h->h1; *bytes = T * h->cfg.d_model * 4; break;
    case KREA_DIT_BUF_HN: *dev_ptr = h->hn; *bytes = T * h->cfg.d_model * es; break;
    case KREA_DIT_BUF_HMID: *dev_ptr = h->hmid; *bytes = T * h->cfg.ffn * es; break;
    case KREA_DIT_BUF_XN8: *dev_ptr = h->xn8; *bytes = h->mode8 ? T * h->cfg.d_model : 0; break;
    case KREA_DIT_BUF_OG8: *dev_ptr = h->og8; *bytes = h->mode8 ? T * h->cfg.n_q * hd : 0; break;
    case KREA_DIT_BUF_HN8: *dev_ptr = h->hn8; *bytes = h->mode8 ? T * h->cfg.d_model : 0; break;
    case KREA_DIT_BUF_HMID8: *dev_ptr = h->hmid8; *bytes = h->mode8 ? T * h->cfg.ffn : 0; break;
    case KREA_DIT_BUF_XN4:
    case KREA_DIT_BUF_OG4:
    case KREA_DIT_BUF_HN4:
    case KREA_DIT_BUF_HMID4:
    case KREA_DIT_BUF_SF_XN4:
    case KREA_DIT_BUF_SF_OG4:
    case KREA_DIT_BUF_SF_HN4:
    case KREA_DIT_BUF_SF_HMID4:
    case KREA_DIT_BUF_TS_XN4:
    case KREA_DIT_BUF_TS_OG4:
    case KREA_DIT_BUF_TS_HN4:
    case KREA_DIT_BUF_TS_HMID4: {
      const size_t nq = static_cast<size_t>(h->cfg.n_q) * hd;
      const size_t K[4] = {static_cast<size_t>(h->cfg.d_model), nq, static_cast<size_t>(h->cfg.d_model),
                           static_cast<size_t>(h->cfg.ffn)};
      void* const codes[4] = {h->xn4, h->og4, h->hn4, h->hmid4};
      void* const sfs[4] = {h->sf_xn4, h->sf_og4, h->sf_hn4, h->sf_hmid4};
      const int which4 = (which - KREA_DIT_BUF_XN4) % 4, kind = (which - KREA_DIT_BUF_XN4) / 4;
      if (!h->mode4) {
        *dev_ptr = nullptr;
        *bytes = 0;
      } else if (kind == 0) {
        *dev_ptr = codes[which4];
        *bytes = T * K[which4] / 2;
      } else if (kind == 1) {
        *dev_ptr = sfs[which4];
        *bytes = kd::nvfp4_scale_bytes(static_cast<long long>(T), static_cast<long long>(K[which4]));
      } else {
        *dev_ptr = h->ts4 + which4;
        *bytes = T ? sizeof(float) : 0;
      }
      break;
    }
    case KREA_DIT_BUF_DQ_XN:
    case KREA_DIT_BUF_DQ_OG:
    case KREA_DIT_BUF_DQ_HN:
    case KREA_DIT_BUF_DQ_HMID: {
      float* const dqs[4] = {h->dq_xn, h->dq_og, h->dq_hn, h->dq_hmid};
      *dev_ptr = dqs[which - KREA_DIT_BUF_DQ_XN];
      *bytes = h->mode8 ? (h->mode8 == 2 ? T : (T ? 1 : 0)) * sizeof(float) : 0;
      break;
    }
    default: return KREA_DIT_ERR_INVALID_ARG;
  }
  return KREA_DIT_OK;
}

int krea_dit_block_set_timing(krea_dit_block_t h, int enable) {
  if (!h) return KREA_DIT_ERR_INVALID_ARG;
  h->timing = enable != 0;
  return KREA_DIT_OK;
}

int krea_dit_block_timing_reset(krea_dit_block_t h) {
  if (!h) return KREA_DIT_ERR_INVALID_ARG;
  int r = harvest(h);
  for (int i = 0; i < S_COUNT; ++i) {
    h->total_ms[i] = 0.0;
    h->launches[i] = 0;
  }
  return r;
}

int krea_dit_block_kernel_times(krea_dit_block_t h, const char** names, double* total_ms, int* launches, int cap,
                                int* n) {
  if (!h || !n) return KREA_DIT_ERR_INVALID_ARG;
  int r = harvest(h);
  for (int i = 0; i < S_COUNT && i < cap; ++i) {
    if (names) names[i] = kSlotNames[i];
    if (total_ms) total_ms[i] = h->total_ms[i];
    if (launches) launches[i] = h->launches[i];
  }
  *n = S_COUNT;
  return r;
}

int krea_dit_block_device_status(krea_dit_block_t h, krea_dit_stream_t stream, int* site) {
  if (!h || !site) return KREA_DIT_ERR_INVALID_ARG;
  *site = 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, h->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return KREA_DIT_ERR_CUDA;
  if (word) {
    *site = word;
    if (cudaMemset(h->err, 0, sizeof(int)) != cudaSuccess) return KREA_DIT_ERR_CUDA;
    return KREA_DIT_ERR_DEVICE_TIMEOUT;
  }
  return KREA_DIT_OK;
}

int krea_dit_block_selftest_wait(krea_dit_block_t h, int site, long long limit_ns, krea_dit_stream_t stream) {
  if (!h || site == 0 || (site & ~0xFF) != 0) return KREA_DIT_ERR_INVALID_ARG;
  if (limit_ns < 1000 || limit_ns > 1000000000LL) return KREA_DIT_ERR_INVALID_ARG;
  const cudaError_t e = kd::launch_wait_selftest(h->err, site, static_cast<unsigned long long>(limit_ns), h->num_sms,
                                                 reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}

int krea_dit_block_inject_fault(krea_dit_block_t h, int count) {
  if (!h || count < 0) return KREA_DIT_ERR_INVALID_ARG;
  h->inject = count;
  return KREA_DIT_OK;
}

}  // extern "C"
