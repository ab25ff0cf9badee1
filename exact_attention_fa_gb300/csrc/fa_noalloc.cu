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
// that device current, on the first call) and that address is what the kernels receive.
#include <cuda_runtime.h>

#include <mutex>

#include "fa.h"

namespace {

constexpr int kMaxDevices = 64;

// Rows of lse * log2(e) and D for the backward. Nothing here has to start at zero: the
// backward's first kernel writes every entry that its second kernel reads.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

struct ScratchSlot {
  bool looked_up = false;
  int status = FA_OK;
  void* ptr = nullptr;
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
  if (!s.looked_up) {
    s.looked_up = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      cudaGetLastError();
      s.status = FA_ERR_NO_DEVICE;
    } else if (cudaGetSymbolAddress(&s.ptr, g_noalloc_scratch) != cudaSuccess || s.ptr == nullptr) {
      cudaGetLastError();
      s.status = FA_ERR_CUDA;
      s.ptr = nullptr;
    }
  }
  *out = s.ptr;
  return s.status;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dO, const float* lse, float* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, int causal,
                              fa_stream_t stream) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_bytes(B, H, N, d);
  if (need == 0) return FA_ERR_INVALID_ARG;
  if (need > static_cast<size_t>(FA_NOALLOC_SCRATCH_BYTES)) return FA_ERR_SCRATCH_LIMIT;
  void* scratch = nullptr;
  const int st = scratch_on_current_device(&scratch);
  if (st != FA_OK) return st;
  return fa_bwd(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch, stream);
}
