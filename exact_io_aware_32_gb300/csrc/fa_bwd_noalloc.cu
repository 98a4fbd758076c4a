// fa_bwd_noalloc: the backward pass for callers that cannot allocate device
// memory. Some callers have no way to obtain a workspace: code running as a
// plug-in inside a host framework that owns every byte of device memory and
// hands out no allocator, or code on a latency-critical path where a
// cudaMalloc (with its implicit synchronisation and unpredictable cost) is not
// allowed. For them this entry point keeps the backward pass's scratch (the
// fp32 row terms D) in a fixed array inside the library. It calls no cudaMalloc, cudaFree or any allocating routine.
//
// The array is a file-scope __device__ variable, so each GPU that loads this
// code holds kFaBwdNoallocMaxScratch bytes of it until the process exits.
// Host code cannot use the array's name as a device address; the device
// address is looked up once per device with cudaGetSymbolAddress, with that
// device current, on the first call made on that device.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa.h"

namespace {

constexpr size_t kFaBwdNoallocMaxScratch = FA_BWD_NOALLOC_MAX_SCRATCH_BYTES;
static_assert(kFaBwdNoallocMaxScratch % 256 == 0, "scratch size must keep 256-byte alignment");

// Shared by every call on a device; holds the previous call's contents.
static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[kFaBwdNoallocMaxScratch];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on the
// first call for that device. Returns FA_OK, FA_ERR_UNSUPPORTED (not an
// sm_103 device: the library holds no code, hence no array, for it, and
// fa_bwd reports the same) or FA_ERR_LAUNCH.
int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();  // leave no error pending for the caller
    return FA_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
    if (major != 10 || minor != 3) return FA_ERR_UNSUPPORTED;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return FA_ERR_LAUNCH;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                              const void* dO, void* dq, void* dk, void* dv, int B, int H, int N, int d, float scale,
                              int causal, void* stream) {
  // fa_bwd checks pointers, shape and alignment before the workspace and
  // touches no device state before those checks: a call without workspace
  // reports any argument error, or FA_ERR_WORKSPACE if the arguments are good.
  int st = fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, nullptr, 0, stream);
  if (st != FA_ERR_WORKSPACE) return st;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0 || need > kFaBwdNoallocMaxScratch) return FA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_on_current_device(&scratch)) != FA_OK) return st;
  // The backward pass writes every scratch value (the row terms D) before it
  // reads it, so the previous call's contents do not matter.
  return fa_bwd(q, k, v, o, lse, dO, dq, dk, dv, B, H, N, d, scale, causal, scratch, kFaBwdNoallocMaxScratch,
                stream);
}
