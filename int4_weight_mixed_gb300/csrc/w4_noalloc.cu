// w4_noalloc.cu — w4_gemm_noalloc: the same GEMM as w4_gemm, for callers
// that cannot hand the library a workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// GEMM: a plug-in inside a framework that owns every byte of device memory
// and exposes no allocator to its extensions, or a latency-critical loop that
// must not call cudaMalloc because it can synchronize the whole device.  For
// them the split-K counters, partial sums and (W4A8) bf16 activation copy
// live in a fixed scratch array compiled into this library, instead of a
// caller-provided workspace.  The array exists once on every GPU that loads
// the library and stays resident until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/w4.h"
#include "w4_internal.h"

namespace {

// The scratch area.  In host code `g_scratch` names a host-side stand-in
// (the device array's shadow), not a device address: handing it to a kernel
// would fault, or on systems where the GPU can reach host memory silently
// use the wrong memory.  Host code must use the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_scratch[W4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_mutex;

// Header plus split-K tile counters: the part of the scratch that must be
// zero when a call starts (the library leaves it zero after a normal call,
// but a call that timed out may not).
constexpr size_t kZeroBytes = w4::kWsHeader + w4::kCounterBytes;

}  // namespace

extern "C" w4_status w4_gemm_noalloc(const void* a, int a_type, int64_t M, int64_t K,
                                     const void* b_packed, int wtype, int64_t N,
                                     const void* b_scales, int scale_type, const void* b_zeros,
                                     int64_t group_size, const float* a_token_scales,
                                     const float* ch_scales, void* out, int out_type,
                                     void* stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return W4_ERR_CUDA;
  }
  void* scratch = nullptr;
  {
    // One-time set-up per device, with that device current: look up the
    // device address of the scratch array.
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
      void* p = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || !p) {
        cudaGetLastError();
        return W4_ERR_CUDA;
      }
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }

  // Clear the status word and split-K counters (the rest of the scratch is
  // fully written before it is read).  Clearing our own array is harmless
  // even if the call below then rejects the problem.
  if (M > 0 && N > 0 && K > 0) {
    cudaError_t e = cudaMemsetAsync(scratch, 0, kZeroBytes, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return W4_ERR_CUDA;
  }
  // w4_gemm checks the scratch need of the schedule it picks against the
  // fixed size before it enqueues any kernel, and returns W4_ERR_WORKSPACE
  // (w4_last_error() then names the bytes needed) when it is larger.
  return w4_gemm(a, a_type, M, K, b_packed, wtype, N, b_scales, scale_type, b_zeros, group_size,
                 a_token_scales, ch_scales, out, out_type, scratch, W4_NOALLOC_SCRATCH_BYTES,
                 stream);
}
