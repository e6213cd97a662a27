/*
 * krea_dit.h -- C ABI of the GB300 (sm_103a) Krea 2 single-stream DiT block forward.
 *
 * The operation (Krea 2 Technical Report, section "Architecture": "Transformer block",
 * "Modality streams", "Timestep conditioning", "Positional encoding", "Normalisation"):
 * one transformer block over the joint [text; image] token sequence, with weights shared
 * by both modalities.
 *
 *   mod    = mod_shared[b] + mod_bias              (shift_a, scale_a, gate_a, shift_m, scale_m, gate_m)
 *   X      = [x_txt[b]; x_img[b]]                  (text rows first, image rows row-major over (r, c))
 *   xn     = rms(X) * (1 + norm1_w) * (1 + scale_a) + shift_a
 *   q,k,v,g= xn W_q^T, xn W_k^T, xn W_v^T, xn W_g^T
 *   q,k    = rms_hd(.) * (1 + q_norm_w / k_norm_w), then 2D axial RoPE on image rows
 *   o_h    = softmax(q_h k_{h/G}^T / sqrt(hd)) v_{h/G}            (GQA, no mask)
 *   o_g    = o * sigmoid(g)                        (omitted when gate_on = 0)
 *   h1     = X + gate_a * (o_g W_o^T)
 *   hn     = rms(h1) * (1 + norm2_w) * (1 + scale_m) + shift_m
 *   out    = h1 + gate_m * ((silu(hn W_gate^T) * (hn W_up^T)) W_down^T)
 *
 * rms(v) = v / sqrt(mean(v^2) + eps). RoPE: head_dim is split in halves, [0, hd/2) turns
 * with the row r and [hd/2, hd) with the column c; pair (2j, 2j+1) of a half of size
 * D = hd/2 turns by pos * rope_base^(-2j/D). Text tokens sit at position 0 (identity).
 *
 * Conventions shared by every call:
 *  - Pointers marked "device" are CUDA device (or managed) memory owned by the caller;
 *    the library never frees them. Pointers marked "host" are host memory.
 *  - Matrices are row-major; weights are nn.Linear-style [out_features, in_features].
 *  - Storage dtype: KREA_DIT_BF16 mode stores weights, token activations and outputs as
 *    bf16 (fp32 accumulation); KREA_DIT_FP32 mode stores them as fp32 (a check mode with
 *    fp32 arithmetic and no tensor cores). Gains, modulation and timestep weights are fp32
 *    in both modes.
 *  - Every device pointer must be 16-byte aligned (tensor-memory-accelerator rule).
 *  - Return value: KREA_DIT_OK (0) or a negative KREA_DIT_ERR_* code. All argument checks
 *    happen on the host before anything is enqueued; a failed check enqueues nothing.
 *  - Calls that take a stream only enqueue work on it: they do not allocate device
 *    memory and do not synchronise. A handle's workspace is shared by its calls, so one
 *    handle must not run on two streams at once.
 */
#ifndef KREA_DIT_H
#define KREA_DIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------------------ */
#define KREA_DIT_OK 0
#define KREA_DIT_ERR_INVALID_ARG (-1)          /* null pointer, negative size, bad enum */
#define KREA_DIT_ERR_UNSUPPORTED_SHAPE (-2)    /* shape outside what the kernels implement */
#define KREA_DIT_ERR_MISALIGNED (-3)           /* a device pointer is not 16-byte aligned */
#define KREA_DIT_ERR_EXCEEDS_CREATE_LIMITS (-4) /* call larger than the handle was created for */
#define KREA_DIT_ERR_CUDA (-5)                 /* a CUDA runtime/driver call failed */
#define KREA_DIT_ERR_NO_DEVICE (-6)            /* current device is not an sm_103 GPU */
#define KREA_DIT_ERR_DEVICE_TIMEOUT (-7)       /* a bounded on-device wait expired (see krea_dit_block_device_status) */
#define KREA_DIT_ERR_INJECTED (-8)             /* host-side fault injection fired (testing aid) */
#define KREA_DIT_ERR_SCRATCH_TOO_SMALL (-9)    /* call needs more than the no-alloc entry point's fixed scratch */

/* ---- modes -------------------------------------------------------------------------- */
#define KREA_DIT_BF16 0
#define KREA_DIT_FP32 1
/* 8-bit GEMM modes (Krea 2 Technical Report, "Training" > "Pretraining": the 256px stage
 * trains with 8-bit matrix multiplications under tensor-wise scaling, the 512px stage
 * under row-wise scaling). Activations, outputs and the non-GEMM steps are as in
 * KREA_DIT_BF16; the four GEMMs (fused QKV+gate, attention output, SwiGLU gate/up, down)
 * take e4m3 operands, see krea_dit_block_forward8. */
#define KREA_DIT_FP8_TENSOR 2
#define KREA_DIT_FP8_ROW 3
/* NVFP4 GEMM mode (Krea 2 Technical Report, "Discussion and future work": pretraining at
 * NVFP4 precision). Activations, outputs and the non-GEMM steps are as in KREA_DIT_BF16;
 * the four GEMMs take NVFP4 operands (E2M1 elements with an E4M3 scale per 16 elements
 * along K and a power-of-two scale per tensor), see krea_dit_block_forward4. */
#define KREA_DIT_NVFP4 4

typedef struct krea_dit_block_s* krea_dit_block_t;
/* Same object as cudaStream_t / CUstream. NULL means the legacy default stream. */
typedef struct CUstream_st* krea_dit_stream_t;

/* Block hyper-parameters and the largest call a handle must serve.
 *  max_batch, max_seq  : largest B and L = n_txt + img_h*img_w a forward may use
 *  d_model             : width d (multiple of 64)
 *  n_q, n_kv, head_dim : query heads, key/value heads (n_q % n_kv == 0), hd (64 or 128;
 *                        BF16 mode needs 128)
 *  ffn                 : SwiGLU hidden size F (multiple of 64)
 *  img_h_max, img_w_max: largest image grid (sizes the RoPE table)
 *  eps                 : RMSNorm epsilon (the block uses 1e-6)
 *  rope_base           : RoPE base (10000)
 *  gate_on             : 1 = sigmoid output gate on attention, 0 = off (then w_qkvg has no g rows)
 *  mode                : KREA_DIT_BF16, KREA_DIT_FP32, KREA_DIT_FP8_TENSOR,
 *                        KREA_DIT_FP8_ROW or KREA_DIT_NVFP4 (the 8-bit and NVFP4 modes
 *                        need head_dim 128, like BF16; the 8-bit modes d_model <= 3072) */
typedef struct {
  int max_batch, max_seq;
  int d_model, n_q, n_kv, head_dim, ffn;
  int img_h_max, img_w_max;
  float eps, rope_base;
  int gate_on;
  int mode;
} krea_dit_config;

/* Block weights, all device memory, caller-owned. "dtype" = the mode's storage dtype.
 *  w_qkvg  [(2 n_q + 2 n_kv) hd, d] dtype, rows ordered q | k | v | g (heads contiguous
 *          inside each part); [(n_q + 2 n_kv) hd, d] when gate_on = 0
 *  w_o     [d, n_q hd] dtype
 *  w_gate  [F, d] dtype ; w_up [F, d] dtype ; w_down [d, F] dtype
 *  norm1_w, norm2_w [d] fp32 : zero-centred gain offsets (gain = 1 + w)
 *  q_norm_w, k_norm_w [hd] fp32 : QK-RMSNorm gain offsets (gain = 1 + w)
 *  mod_bias [6, d] fp32 : this block's modulation bias, chunk order
 *          shift_a, scale_a, gate_a, shift_m, scale_m, gate_m */
typedef struct {
  const void* w_qkvg;
  const void* w_o;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const float* norm1_w;
  const float* norm2_w;
  const float* q_norm_w;
  const float* k_norm_w;
  const float* mod_bias;
} krea_dit_weights;

/* 8-bit GEMM weights of one block (modes KREA_DIT_FP8_TENSOR / KREA_DIT_FP8_ROW), all
 * device memory, caller-owned, filled by krea_dit_weights8_quantize.
 *  w_qkvg, w_o, w_gate, w_up, w_down : e4m3 codes (one byte each), same shapes and row
 *          order as the bf16 matrices of krea_dit_weights
 *  dq_*    fp32 dequantisation factors 2^-k: one per matrix row (FP8_ROW: [rows] floats)
 *          or one per matrix (FP8_TENSOR: [1] float); matrix row r is codes * dq[r].
 * Scaling rule: a group (row or matrix) with largest magnitude amax is multiplied by 2^k,
 * k the largest integer with amax * 2^k <= 448 (k = 0 if amax = 0, k <= 125), then cast
 * to e4m3 (round to nearest, ties to even, saturating at +-448). */
typedef struct {
  void* w_qkvg;
  void* w_o;
  void* w_gate;
  void* w_up;
  void* w_down;
  float* dq_qkvg;
  float* dq_o;
  float* dq_gate;
  float* dq_up;
  float* dq_down;
} krea_dit_weights8;

/* NVFP4 GEMM weights of one block (mode KREA_DIT_NVFP4), all device memory, caller-owned,
 * filled by krea_dit_weights4_quantize. For a bf16 matrix W [rows, cols] of
 * krea_dit_weights (cols = K, a multiple of 64):
 *  w_*   E2M1 codes [rows, cols / 2] bytes, element 2i of a row in the low nibble of byte i
 *  sf_*  E4M3 block scales, krea_dit_nvfp4_scale_bytes(rows, cols) bytes: for each 128-row
 *        block rb (rows padded to 128) and each 64-element step ks of K a 512-byte atom
 *        at offset (rb * cols / 64 + ks) * 512 whose byte (r % 32) * 16 + (r / 32) * 4 + j
 *        scales elements 16j .. 16j + 15 of the step in row r of the block (padding rows 0)
 *  ts_*  fp32 [1]: the tensor scale s_t
 * Rule: s_t = 2^j, j the smallest integer with amax <= 448 * 6 * 2^j (1 when amax = 0);
 * a block of 16 with largest magnitude a_b gets s_b = E4M3(a_b / (6 s_t)) and its elements
 * q = E2M1(x / (s_b s_t)) (0 where s_b = 0); casts round to nearest even and saturate.
 * W is approximated by q * s_b * s_t. */
typedef struct {
  void* w_qkvg;
  void* w_o;
  void* w_gate;
  void* w_up;
  void* w_down;
  void* sf_qkvg;
  void* sf_o;
  void* sf_gate;
  void* sf_up;
  void* sf_down;
  float* ts_qkvg;
  float* ts_o;
  float* ts_gate;
  float* ts_up;
  float* ts_down;
} krea_dit_weights4;

/* Shared timestep-MLP weights, fp32 device memory: w1 [d, 256], b1 [d], w2 [6d, d], b2 [6d]. */
typedef struct {
  const float* w1;
  const float* b1;
  const float* w2;
  const float* b2;
} krea_dit_temb_weights;

/* Create a handle on the current CUDA device. Validates the config, checks the device is
 * sm_103, allocates the workspace for max_batch x max_seq tokens (the only allocation
 * the library makes) and uploads the RoPE table. Synchronous. On error *out is NULL. */
int krea_dit_block_create(const krea_dit_config* cfg, krea_dit_block_t* out);

/* Free the handle and its workspace. Synchronises the device first. NULL is a no-op. */
int krea_dit_block_destroy(krea_dit_block_t h);

/* Shared timestep embedding (Krea 2 Technical Report, "Timestep conditioning"):
 * e = [cos(1000 t w_i) | sin(1000 t w_i)], w_i = 10000^(-i/128), i < 128;
 * mod_shared = W2 silu(W1 e + b1) + b2, written as [B, 6, d].
 *  t          device fp32 [B], t in [0, 1]
 *  B          1 .. max_batch
 *  mod_shared device fp32 [B, 6, d], written. */
int krea_dit_timestep_embed(krea_dit_block_t h, const float* t, int B, const krea_dit_temb_weights* w,
                            float* mod_shared, krea_dit_stream_t stream);

/* One block forward (operation at the top of this file).
 *  x_img      device dtype [B, img_h*img_w, d] (may be NULL when img_h*img_w == 0)
 *  x_txt      device dtype [B, n_txt, d]       (may be NULL when n_txt == 0)
 *  B, img_h, img_w, n_txt : B <= max_batch, img_h <= img_h_max, img_w <= img_w_max,
 *               L = n_txt + img_h*img_w <= max_seq; B == 0 or L == 0 enqueues nothing
 *  t_emb      device fp32 [B, 6, d]: mod_shared from krea_dit_timestep_embed
 *  out        device dtype [B, L, d], text rows first; must not alias any input. */
int krea_dit_block_forward(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h,
                           int img_w, int n_txt, const float* t_emb, const krea_dit_weights* w, void* out,
                           krea_dit_stream_t stream);

/* Timestep embedding that allocates nothing (no counterpart in the Krea 2 report: it
 * exists for callers, not for the method). For callers that cannot call cudaMalloc, e.g.
 * a serving runtime that reserves all device memory for its own pool and forbids
 * allocations after start-up, or a latency-critical loop where an allocation could
 * block behind other streams. It needs no handle and computes the same mod_shared as
 * krea_dit_timestep_embed.
 *  t          device fp32 [B]
 *  B, d_model B >= 0, d_model > 0, and B * (256 + d_model) <= KREA_DIT_NOALLOC_SCRATCH_FLOATS,
 *             else KREA_DIT_ERR_SCRATCH_TOO_SMALL (e.g. d = 3072 allows B <= 78)
 *  w          timestep-MLP weights as for krea_dit_timestep_embed
 *  mod_shared device fp32 [B, 6, d_model], written
 * Scratch lives in one fixed file-scope device array of KREA_DIT_NOALLOC_SCRATCH_FLOATS
 * floats (1 MiB). The first call on a device looks up the array's device address (with
 * that device current) and caches it; under CUDA's lazy module loading (the default) that
 * first call is also when the device gets its copy of the array, which it then holds
 * until the process exits. So make one call on each device at start-up, before reserving
 * the device's memory for a pool and before any stream capture. Every call
 * shares the array and writes all scratch it reads, so nothing carries over between
 * calls, but calls that overlap on the GPU (two streams, two threads) race. It calls
 * no cudaMalloc, cudaFree or allocating library routine. */
#define KREA_DIT_NOALLOC_SCRATCH_FLOATS 262144
int krea_dit_timestep_embed_noalloc(const float* t, int B, int d_model, const krea_dit_temb_weights* w,
                                    float* mod_shared, krea_dit_stream_t stream);

/* ---- 8-bit GEMM forward (modes KREA_DIT_FP8_TENSOR, KREA_DIT_FP8_ROW) ----------------- */

/* Cast the bf16 GEMM weights of w (w_qkvg, w_o, w_gate, w_up, w_down) to e4m3 codes with
 * the handle's scaling (per row, or one scale per matrix) into the caller's buffers of q.
 * Enqueued on `stream`; the other fields of w are not read. Errors: INVALID_ARG for a
 * NULL pointer or a handle not in an 8-bit mode, MISALIGNED for an unaligned pointer. */
int krea_dit_weights8_quantize(krea_dit_block_t h, const krea_dit_weights* w, const krea_dit_weights8* q,
                               krea_dit_stream_t stream);

/* krea_dit_block_forward with 8-bit GEMM operands. Each of the four GEMMs casts its
 * activation operand (the bf16 value the BF16 mode stores there: xn, o_g, hn, hmid) to
 * e4m3 with the handle's scaling (FP8_ROW: one scale per token row; FP8_TENSOR: one
 * scale for the whole [B L, K] activation of the call) and multiplies it by the e4m3
 * weight codes of q; each product is dequantised by its row and column factors and
 * accumulated in fp32. x_img, x_txt, t_emb, out and every other argument are as in
 * krea_dit_block_forward; from w only norm1_w, norm2_w, q_norm_w, k_norm_w and mod_bias
 * are read (its matrix pointers may be NULL). Errors as krea_dit_block_forward, plus
 * INVALID_ARG when the handle is not in an 8-bit mode or q has a NULL pointer. A handle
 * in an 8-bit mode rejects krea_dit_block_forward and the joint / stack calls
 * (INVALID_ARG). */
int krea_dit_block_forward8(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                            int n_txt, const float* t_emb, const krea_dit_weights* w, const krea_dit_weights8* q,
                            void* out, krea_dit_stream_t stream);

/* ---- NVFP4 GEMM forward (mode KREA_DIT_NVFP4) ---------------------------------------- */

/* Bytes of the block scales of a [rows, cols] matrix (cols a multiple of 64; rows padded to
 * a multiple of 128): ceil(rows / 128) * 128 * cols / 16. 0 for rows <= 0 or cols <= 0. */
size_t krea_dit_nvfp4_scale_bytes(int rows, int cols);

/* Cast the bf16 GEMM weights of w to NVFP4 into the caller's buffers of q (layout and rule
 * at krea_dit_weights4). Enqueued on `stream`; the other fields of w are not read. Errors:
 * INVALID_ARG for a NULL pointer or a handle not in KREA_DIT_NVFP4 mode, MISALIGNED. */
int krea_dit_weights4_quantize(krea_dit_block_t h, const krea_dit_weights* w, const krea_dit_weights4* q,
                               krea_dit_stream_t stream);

/* krea_dit_block_forward with NVFP4 GEMM operands. Each of the four GEMMs casts its
 * activation operand (the bf16 value the BF16 mode stores there: xn, o_g, hn, hmid) to
 * NVFP4 with one tensor scale for the whole [B L, K] activation of the call, and
 * multiplies it by the weight codes of q on the tensor core (block-scaled E2M1 MMA, fp32
 * accumulation); the tensor scales multiply the products in the epilogue. Arguments and
 * errors as krea_dit_block_forward8, with q the NVFP4 weights. A handle in this mode
 * rejects every other forward (INVALID_ARG). */
int krea_dit_block_forward4(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                            int n_txt, const float* t_emb, const krea_dit_weights* w, const krea_dit_weights4* q,
                            void* out, krea_dit_stream_t stream);

/* ---- block backward (KREA_DIT_BF16 mode) -------------------------------------------- */

/* Gradients of one block forward (Krea 2 Technical Report, "Training": the block is
 * trained, so its forward has a backward). Device memory, caller-owned; every buffer is
 * overwritten by krea_dit_block_backward.
 *  d_x_txt, d_x_img  bf16 [B, n_txt, d], [B, img_h*img_w, d]: gradient of the block input
 *  d_w_*             fp32, the shapes of the matching weights of krea_dit_weights
 *  d_norm1_w, d_norm2_w fp32 [d]; d_q_norm_w, d_k_norm_w fp32 [hd]
 *  d_mod_bias        fp32 [6, d]: gradient of the block's modulation bias
 *  d_mod_shared      fp32 [B, 6, d]: gradient of the shared modulation (chain it through
 *                    the timestep MLP outside the block) */
typedef struct {
  void* d_x_txt;
  void* d_x_img;
  float* d_w_qkvg;
  float* d_w_o;
  float* d_w_gate;
  float* d_w_up;
  float* d_w_down;
  float* d_norm1_w;
  float* d_norm2_w;
  float* d_q_norm_w;
  float* d_k_norm_w;
  float* d_mod_bias;
  float* d_mod_shared;
} krea_dit_grads;

/* Allocate the backward workspace of a KREA_DIT_BF16 handle (transposed operands and the
 * recomputed activations for max_batch x max_seq tokens; about 3.5 GB at d = 3072,
 * F = 8192, 9216 tokens). Synchronous; INVALID_ARG for another mode. Idempotent. */
int krea_dit_block_enable_backward(krea_dit_block_t h);

/* Gradients of krea_dit_block_forward for the upstream gradient d_out (bf16 [B, L, d],
 * joint order, text rows first) at inputs x_img, x_txt, t_emb and weights w (the same
 * arguments as the forward). Recomputes the forward into the handle's workspace, then
 * runs the chain rule in reverse: the data gradients of the four projections and the
 * attention products on the tensor cores (bf16 operands, fp32 accumulation), the
 * attention's probabilities recomputed per head, the weight gradients as products over
 * the token rows. Needs krea_dit_block_enable_backward (INVALID_ARG otherwise). Errors as
 * krea_dit_block_forward, plus INVALID_ARG / MISALIGNED for the gradient buffers. */
int krea_dit_block_backward(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h, int img_w,
                            int n_txt, const float* t_emb, const krea_dit_weights* w, const void* d_out,
                            const krea_dit_grads* g, krea_dit_stream_t stream);

/* ---- joint-layout forward and stacks of blocks ------------------------------------ */

/* One block forward whose input is the joint sequence itself (Krea 2 Technical Report,
 * "Modality streams": text and image tokens form one sequence through every block).
 *  x    device dtype [B, L, d], L = n_txt + img_h*img_w, text rows first (the layout
 *       krea_dit_block_forward writes)
 *  out  device dtype [B, L, d]; may be x itself (the block reads x only before writing
 *       out), otherwise must not overlap it.
 * Other arguments and errors as krea_dit_block_forward. */
int krea_dit_block_forward_joint(krea_dit_block_t h, const void* x, int B, int img_h, int img_w, int n_txt,
                                 const float* t_emb, const krea_dit_weights* w, void* out, krea_dit_stream_t stream);

/* A stack of n_blocks blocks applied in place to the joint sequence x [B, L, d]: block i
 * uses weights w[i] (host array of n_blocks structs, read during the call only; may be NULL
 * when n_blocks is 0) and the shared t_emb (each block adds its own mod_bias). One handle's
 * workspace serves every block in turn. Enqueues 7 * n_blocks kernels (bf16 mode) and
 * stops at the first block whose arguments fail a check, returning that block's status
 * (earlier blocks stay enqueued). Capturable in a CUDA graph (krea_dit_stack_graph_create). */
int krea_dit_stack_forward(krea_dit_block_t h, void* x, int B, int img_h, int img_w, int n_txt, const float* t_emb,
                           const krea_dit_weights* w, int n_blocks, krea_dit_stream_t stream);

/* Capture krea_dit_stack_forward with these exact arguments into a CUDA graph and
 * instantiate it, so that a whole stack replays with one launch call.
 *  stream  a created (non-default) stream that is not capturing already; the capture is
 *          thread-local, and per-kernel timing is suspended while it runs.
 *  out     receives the graph; set to NULL on any error.
 * The graph records device pointers only: x, t_emb, every weight buffer and the handle
 * (its workspace) must outlive it, and each launch reruns the stack in place on whatever
 * those buffers hold then. Launches on one handle must not overlap another forward on the
 * same handle (they share its workspace). Argument errors are those of
 * krea_dit_stack_forward, plus KREA_DIT_ERR_INVALID_ARG for a NULL or capturing stream;
 * KREA_DIT_ERR_CUDA if capture or instantiation fails.
 * krea_dit_graph_launch enqueues the graph on `stream` (any stream, NULL = legacy default).
 * krea_dit_graph_destroy frees it (NULL is a no-op). */
typedef struct krea_dit_graph_s* krea_dit_graph_t;
int krea_dit_stack_graph_create(krea_dit_block_t h, void* x, int B, int img_h, int img_w, int n_txt,
                                const float* t_emb, const krea_dit_weights* w, int n_blocks, krea_dit_stream_t stream,
                                krea_dit_graph_t* out);
int krea_dit_graph_launch(krea_dit_graph_t g, krea_dit_stream_t stream);
int krea_dit_graph_destroy(krea_dit_graph_t g);

/* Static text for a status code. Never NULL. */
const char* krea_dit_status_string(int status);

/* ---- host-buffer forward (end-to-end path) ----------------------------------------- */

/* Prepare the handle for krea_dit_block_forward_host: allocates two device staging sets
 * (inputs and output for max_batch x max_seq tokens each), two copy streams and their
 * events. Synchronous; call once, before any stream capture. */
int krea_dit_block_enable_host_io(krea_dit_block_t h);

/* One block forward from and to host memory. Same operation and arguments as
 * krea_dit_block_forward except that x_img, x_txt and out are HOST pointers (pinned memory
 * gives full copy bandwidth); t_emb and the weights stay in device memory. The inputs are
 * copied into a staging set on the handle's upload stream, the forward runs on `stream`,
 * and the output is copied back on the handle's download stream. Staging sets alternate
 * between calls, so the upload of call i+1 and the download of call i-1 overlap the
 * compute of call i. Returns after enqueueing; the host buffers of a call must stay
 * valid and untouched until krea_dit_block_host_sync returns. */
int krea_dit_block_forward_host(krea_dit_block_t h, const void* x_img, const void* x_txt, int B, int img_h,
                                int img_w, int n_txt, const float* t_emb, const krea_dit_weights* w, void* out,
                                krea_dit_stream_t stream);

/* Wait until every krea_dit_block_forward_host call enqueued so far has finished,
 * including its download. */
int krea_dit_block_host_sync(krea_dit_block_t h);

/* ---- inspection, timing and failure reporting ------------------------------------- */

/* Workspace buffers written by the most recent forward (read-only views, owned by the
 * handle, valid until the next forward or destroy). T = B L rows in joint order.
 *  XN   [T, d] dtype       normed+modulated input of the attention branch
 *  Q    [B, n_q, L, hd]    dtype, after QK-norm and RoPE
 *  K    [B, n_kv, L, hd]   dtype, after QK-norm and RoPE
 *  VT   [B, n_kv, hd, Lp]  dtype, values transposed, Lp = L rounded up to 64
 *  G    [T, n_q hd]        dtype, the gate sigmoid(xn W_g^T) (unused when gate_on = 0)
 *  OG   [T, n_q hd]        dtype, o * sigmoid(g)
 *  H1   [T, d]             fp32 in both modes, block state after the attention residual
 *                          (the residual stream between the two residual adds)
 *  HN   [T, d]             dtype, normed+modulated input of the MLP
 *  HMID [T, F]             dtype, silu(hn W_gate^T) * (hn W_up^T) */
#define KREA_DIT_BUF_XN 0
#define KREA_DIT_BUF_Q 1
#define KREA_DIT_BUF_K 2
#define KREA_DIT_BUF_VT 3
#define KREA_DIT_BUF_G 4
#define KREA_DIT_BUF_OG 5
#define KREA_DIT_BUF_H1 6
#define KREA_DIT_BUF_HN 7
#define KREA_DIT_BUF_HMID 8
/* 8-bit modes: the e4m3 GEMM operands (codes) and their dequantisation factors (fp32,
 * [T] row-wise or [1] tensor-wise) of the last forward */
#define KREA_DIT_BUF_XN8 9
#define KREA_DIT_BUF_OG8 10
#define KREA_DIT_BUF_HN8 11
#define KREA_DIT_BUF_HMID8 12
#define KREA_DIT_BUF_DQ_XN 13
#define KREA_DIT_BUF_DQ_OG 14
#define KREA_DIT_BUF_DQ_HN 15
#define KREA_DIT_BUF_DQ_HMID 16
/* NVFP4 mode: the GEMM operands of the last forward: E2M1 codes ([T, K/2] bytes), block
 * scales (the atom layout of krea_dit_weights4) and tensor scales (fp32 [1]) */
#define KREA_DIT_BUF_XN4 17
#define KREA_DIT_BUF_OG4 18
#define KREA_DIT_BUF_HN4 19
#define KREA_DIT_BUF_HMID4 20
#define KREA_DIT_BUF_SF_XN4 21
#define KREA_DIT_BUF_SF_OG4 22
#define KREA_DIT_BUF_SF_HN4 23
#define KREA_DIT_BUF_SF_HMID4 24
#define KREA_DIT_BUF_TS_XN4 25
#define KREA_DIT_BUF_TS_OG4 26
#define KREA_DIT_BUF_TS_HN4 27
#define KREA_DIT_BUF_TS_HMID4 28
int krea_dit_block_workspace(krea_dit_block_t h, int which, void** dev_ptr, size_t* bytes);

/* Per-kernel timing. When enabled, each forward records a CUDA event before and after
 * every kernel it launches, on the forward's stream. krea_dit_block_kernel_times waits
 * for those events and returns, per kernel slot, the summed milliseconds and the number
 * of launches since the last reset (names: host strings owned by the library).
 * cap = capacity of the arrays; *n = number of slots. Timing adds one event record per
 * kernel and nothing else. */
int krea_dit_block_set_timing(krea_dit_block_t h, int enable);
int krea_dit_block_kernel_times(krea_dit_block_t h, const char** names, double* total_ms, int* launches,
                                int cap, int* n);
int krea_dit_block_timing_reset(krea_dit_block_t h);

/* Every wait inside the tensor-core kernels (on a TMA arrival or an MMA commit) gives up
 * after about one second, records which wait it was in a device-side error word, and the
 * kernel returns. This call synchronises `stream`, reads the word, clears it, and returns
 * KREA_DIT_OK or KREA_DIT_ERR_DEVICE_TIMEOUT (*site = the first wait that gave up, a
 * bit mask of sites otherwise 0). */
int krea_dit_block_device_status(krea_dit_block_t h, krea_dit_stream_t stream, int* site);

/* Sites reported by krea_dit_block_device_status: which kind of wait gave up. */
#define KREA_DIT_SITE_GEMM_PRODUCER 0x01 /* GEMM TMA-load warp waiting for a free stage */
#define KREA_DIT_SITE_GEMM_MMA 0x02      /* GEMM MMA warp waiting for operands or an accumulator */
#define KREA_DIT_SITE_GEMM_EPILOGUE 0x04 /* GEMM epilogue waiting for an accumulator */
#define KREA_DIT_SITE_GEMM_TEARDOWN 0x08 /* GEMM draining its own copies before exit */
#define KREA_DIT_SITE_ATTN_LOAD 0x10     /* attention TMA-load warp waiting for a free slot */
#define KREA_DIT_SITE_ATTN_MMA 0x20      /* attention MMA warp waiting for K/V, P or its turn */
#define KREA_DIT_SITE_ATTN_SOFTMAX 0x40  /* attention softmax/epilogue warps waiting for S or O */
#define KREA_DIT_SITE_ATTN_TEARDOWN 0x80 /* attention draining its own copies before exit */

/* Testing aid for the bounded waits above: enqueue on `stream` one CTA per SM that
 * takes 32 tensor-memory columns, waits on an mbarrier that nothing ever arrives at
 * (the same wait routine as the tensor-core kernels, with a limit of limit_ns instead
 * of about one second), gives up, records `site` in the handle's device error word,
 * frees its tensor memory and returns. No copy or MMA is in flight at any point. A
 * following krea_dit_block_device_status returns KREA_DIT_ERR_DEVICE_TIMEOUT with that
 * site; the handle stays usable. site: a nonzero mask of KREA_DIT_SITE_* bits (0xFF);
 * limit_ns: 1000 (1 us) to 1000000000 (1 s); else INVALID_ARG. */
int krea_dit_block_selftest_wait(krea_dit_block_t h, int site, long long limit_ns, krea_dit_stream_t stream);

/* Testing aid: make the next `count` calls of krea_dit_block_forward fail with
 * KREA_DIT_ERR_INJECTED after validation and before any launch. */
int krea_dit_block_inject_fault(krea_dit_block_t h, int count);

/* Kernel names this library launches (for launch accounting): returns the number of
 * names, fills up to cap of them. */
int krea_dit_kernel_names(const char** names, int cap);

#ifdef __cplusplus
}
#endif
#endif /* KREA_DIT_H */
