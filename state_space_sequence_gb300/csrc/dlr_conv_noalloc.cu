// dlr_conv_noalloc.cu -- the FFT convolution of dlr_conv for callers that cannot allocate
// device memory.
//
// Who needs it: a program that embeds libdlr inside a host application which owns every byte
// of device memory (a fixed memory plan reserved at start-up, as serving processes and plugin
// hosts often have), or code on a latency-critical path where a cudaMalloc -- which may
// synchronise the whole device -- is not acceptable. Such callers can pass their inputs and
// outputs but have no way to obtain the extra workspace that dlr_conv asks for.
//
// How: the workspace lives in a fixed array in the library's own device memory (below). Every
// GPU that loads the library holds this array until the process exits. Host code cannot use
// the array's name as a device address (in host code it denotes a host-side stand-in), so
// the device address is looked up once per device with cudaGetSymbolAddress, with that device
// current, the first time this entry point runs on it; later calls reuse the cached address.
// The kernels launched are exactly those of dlr_conv.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "dlr.h"

namespace dlr {
// source file number of the bounds-checked build's failing sites
[[maybe_unused]] constexpr int kSiteFile = 5;
size_t conv_workspace_bytes(int64_t H, int64_t L);
cudaError_t launch_dlr_conv_spectrum(const float* K1, const float* K2, int H, int L, void* ws,
                                     cudaStream_t s);
cudaError_t launch_dlr_conv_apply(const float* u, int B, int H, int L, float* y, const void* ws,
                                  cudaStream_t s);
dlr_status status_from_cuda(cudaError_t e);  // api.cu: records the error for dlr_last_cuda_error
}  // namespace dlr

namespace {

// 16 MiB: room for the twiddle tables and the spectra of H channels at length L as long as
// 24 * n + 8 * H * (n + 1) bytes fit (n = next power of two >= L, the twiddle parts rounded up
// to 256 bytes): up to H = 508 channels at L = 4096, up to H = 124 at L = 16384.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

static __device__ __align__(256) unsigned char g_conv_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 128;
std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

// Device address of g_conv_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    p = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      e = cudaGetSymbolAddress(&p, g_conv_scratch);
      if (e != cudaSuccess) return e;
      if (p == nullptr) return cudaErrorInvalidSymbol;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" dlr_status dlr_conv_noalloc(const float* u, const float* K_fwd, const float* K_bwd,
                                       dlr_dir dir, int64_t B, int64_t H, int64_t L, float* y,
                                       dlr_stream_t stream) {
  if (B < 1 || H < 1 || L < 1) return DLR_ERR_INVALID_ARG;
  if (dir != DLR_CAUSAL && dir != DLR_BIDIR) return DLR_ERR_INVALID_ARG;
  if (!u || !y || !K_fwd || !aligned16(u) || !aligned16(y) || !aligned16(K_fwd))
    return DLR_ERR_INVALID_ARG;
  if (dir == DLR_BIDIR && (!K_bwd || !aligned16(K_bwd))) return DLR_ERR_INVALID_ARG;
  if (dir == DLR_CAUSAL && K_bwd) return DLR_ERR_INVALID_ARG;
  const size_t bytes = sizeof(float) * (size_t)B * (size_t)H * (size_t)L;
  {
    uintptr_t a = reinterpret_cast<uintptr_t>(u), b = reinterpret_cast<uintptr_t>(y);
    if (a < b + bytes && b < a + bytes) return DLR_ERR_INVALID_ARG;
  }
  if (L > 16384 || B * H > 2147483647) return DLR_ERR_UNSUPPORTED;
  // The fixed scratch must hold this call's twiddles and spectra.
  if (dlr::conv_workspace_bytes(H, L) > kNoAllocScratchBytes) return DLR_ERR_WORKSPACE;
  void* ws = nullptr;
  cudaError_t e = scratch_address(&ws);
  if (e != cudaSuccess) return dlr::status_from_cuda(e);
  // Nothing in the scratch has to start at zero: the spectrum launch rewrites the whole
  // twiddle table and every spectrum entry that the apply launch then reads.
  cudaStream_t s = (cudaStream_t)stream;
  e = dlr::launch_dlr_conv_spectrum(K_fwd, dir == DLR_BIDIR ? K_bwd : nullptr, (int)H, (int)L,
                                    ws, s);
  if (e == cudaSuccess) e = dlr::launch_dlr_conv_apply(u, (int)B, (int)H, (int)L, y, ws, s);
  return dlr::status_from_cuda(e);
}
