// fa_bwd_noalloc: the backward for callers that cannot give the library a workspace.
//
// Some callers have no way to obtain device memory for scratch: a plugin whose host framework
// hands it only the input and output buffers, a runtime that pre-plans every byte of device
// memory and forbids cudaMalloc (which also synchronises the device) once it is serving, or code
// whose allocator belongs to someone else. For them this entry point takes its scratch from a
// fixed-size array in the library's own device memory instead of from the caller.
//
// The array is a file-scope __device__ object: every device that loads the library holds
// FA_NOALLOC_SCRATCH_BYTES of it until the process exits. In host code its name is only a host
// stand-in, so its device address is looked up once per device with cudaGetSymbolAddress (with
// that device current, on the first call) and that address is what the kernels receive. Only a
// successful lookup is kept; a failed one is tried again on the next call. The kept address
// belongs to the device's current context: calls after cudaDeviceReset are not supported.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Rows of lse * log2(e) and D for the backward. Nothing here has to start at zero: the
// backward's first kernel writes every entry that its second kernel reads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

struct ScratchSlot {
  void* ptr = nullptr;  // device address of g_noalloc_scratch once looked up
};
ScratchSlot g_slots[kMaxDevices];
std::mutex g_slots_mu;

int scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_slots_mu);
  ScratchSlot& s = g_slots[dev];
  if (s.ptr == nullptr) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      cudaGetLastError();
      return FA_ERR_NO_DEVICE;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return FA_ERR_CUDA;
    }
    s.ptr = ptr;
  }
  *out = s.ptr;
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, float* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal,
                              fa_stream_t stream) {
  // fa_bwd's argument checks first, in its order, so both report the same status for the same
  // bad argument; only then the size limit of the static scratch.
  const int bad = fa::check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, false,
                                     nullptr, nullptr, false);
  if (bad != FA_OK) return bad;
  if (fa_bwd_workspace_bytes(B, H, N, d) > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES))
    return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch, stream);
}
