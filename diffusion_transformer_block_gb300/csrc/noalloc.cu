// Timestep embedding that allocates nothing, for callers that cannot call cudaMalloc.
//
// Some callers must not allocate device memory after start-up: a serving runtime that
// reserves the whole device for its own pool and forbids allocations once warmed up,
// or a latency-critical loop where an allocation could block behind other streams.
// They cannot create a block handle (creation allocates the workspace), so this entry
// point computes the same shared timestep embedding as krea_dit_timestep_embed with
// its scratch in a fixed, file-scope device array instead of the handle's workspace.
//
// The array is KREA_DIT_NOALLOC_SCRATCH_FLOATS floats (1 MiB). With CUDA's lazy module
// loading (the default) a device gets its copy of the array at the first call on that
// device, which looks up the array's address, and holds it until the process exits.
// A caller that reserves all device memory for its own pool must therefore make one call
// on each device at start-up, before the reservation (and before any stream capture);
// later calls allocate nothing. It holds the sinusoid e [B, 256] and the
// hidden layer [B, d] between the two MLP layers, so a call needs B * (256 + d) floats.
// Every call overwrites all of the scratch it uses before reading it, so nothing needs
// clearing between calls; calls that overlap on the GPU share the array and race.
#include <mutex>

#include "internal.h"
#include "krea_dit.h"

namespace {

__device__ __align__(256) float g_temb_scratch[KREA_DIT_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
float* g_scratch_addr[kMaxDevices] = {};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device address of the scratch array on the current device. In host code the
// array's name is a host-side stand-in, not a device address, so the address is
// looked up once per device (with that device current) and cached.
int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KREA_DIT_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return KREA_DIT_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return KREA_DIT_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return KREA_DIT_ERR_NO_DEVICE;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_temb_scratch) != cudaSuccess || !p) return KREA_DIT_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return KREA_DIT_OK;
}

}  // namespace

extern "C" int krea_dit_timestep_embed_noalloc(const float* t, int B, int d_model, const krea_dit_temb_weights* w,
                                               float* mod_shared, krea_dit_stream_t stream) {
  if (!t || !w || !mod_shared || !w->w1 || !w->b1 || !w->w2 || !w->b2) return KREA_DIT_ERR_INVALID_ARG;
  if (B < 0 || d_model <= 0) return KREA_DIT_ERR_INVALID_ARG;
  if (!aligned16(t) || !aligned16(mod_shared) || !aligned16(w->w1) || !aligned16(w->b1) || !aligned16(w->w2) ||
      !aligned16(w->b2))
    return KREA_DIT_ERR_MISALIGNED;
  const long long need = static_cast<long long>(B) * (256 + static_cast<long long>(d_model));
  if (need > KREA_DIT_NOALLOC_SCRATCH_FLOATS) return KREA_DIT_ERR_SCRATCH_TOO_SMALL;
  float* scratch = nullptr;
  const int st_setup = scratch_for_current_device(&scratch);
  if (st_setup != KREA_DIT_OK) return st_setup;
  if (B == 0) return KREA_DIT_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* e = scratch;                                  // [B, 256]
  float* hid = scratch + static_cast<size_t>(B) * 256;  // [B, d]
  cudaError_t r = kd::launch_temb_sinusoid(t, B, e, st);
  if (r == cudaSuccess) r = kd::launch_gemm_simt_f32(e, w->w1, hid, B, d_model, 256, w->b1, 1, st);
  if (r == cudaSuccess) r = kd::launch_gemm_simt_f32(hid, w->w2, mod_shared, B, 6 * d_model, d_model, w->b2, 0, st);
  return r == cudaSuccess ? KREA_DIT_OK : KREA_DIT_ERR_CUDA;
}
