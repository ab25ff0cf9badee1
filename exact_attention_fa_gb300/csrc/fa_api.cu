// C ABI of the exact-attention library: argument validation, per-device state, TMA descriptor
// creation and kernel launches. Declarations and semantics: include/fa.h.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s per barrier wait

// Device error word written by kernels that give up on a barrier (see fa::kErrTimeout).
__device__ unsigned g_error_word;

struct DeviceState {
  bool ready = false;
  int status = FA_OK;
  int num_sms = 0;
  unsigned* err = nullptr;          // device address of g_error_word on this device
};

DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
std::atomic<int> g_exp2_per32{0};  // fa_set_exp2_emulation
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device set-up, once, with that device current: check it is an sm_103 part, look up the
// device address of the error word and the SM count, and opt the kernels in to their shared
// memory (a function attribute of this device's context).
int device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return FA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    st.ready = true;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3) {
      cudaGetLastError();
      st.status = FA_ERR_NO_DEVICE;
    } else if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) !=
                   cudaSuccess ||
               cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err), g_error_word) !=
                   cudaSuccess) {
      cudaGetLastError();
      st.status = FA_ERR_CUDA;
    }
    if (st.status == FA_OK) {
      if (fa::configure_fwd_pair() != cudaSuccess || fa::configure_bwd() != cudaSuccess ||
          fa::configure_decode() != cudaSuccess || fa::configure_fwd_fp32() != cudaSuccess) {
        cudaGetLastError();
        st.status = FA_ERR_CUDA;
      }
    }
    if (st.status == FA_OK && g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q{};
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        st.status = FA_ERR_CUDA;
      } else {
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
      }
    }
    if (st.status != FA_OK) {
      // keep only a successful set-up; a failed one is tried again on the next call
      st.ready = false;
      *out = &st;
      const int failed = st.status;
      st.status = FA_OK;
      return failed;
    }
  }
  *out = &st;
  return st.status;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_common(int B, int H, int N, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * N > (1ll << 31) - 1 || bh > (1ll << 30)) return FA_ERR_TOO_LARGE;
  return FA_OK;
}

// 3-D view [B*H][N][d] of a bf16 tensor, box 64 x rows x 1, 128-byte swizzle, zero fill outside.
bool encode_bf16_map(CUtensorMap* map, const void* base, int BH, int N, int d, int rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * d * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [B*H][N][d] of an fp32 tensor, box 32 x 64 x 1 (128-byte rows), 128-byte swizzle.
bool encode_f32_map(CUtensorMap* map, const void* base, int BH, int N, int d) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 4,
                                 static_cast<cuuint64_t>(N) * d * 4};
  const cuuint32_t box[3] = {32, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view [B*H][N][d] of an 8-bit (e4m3) tensor, box 128 x rows x 1 (128-byte rows), 128-byte
// swizzle, zero fill outside.
bool encode_u8_map(CUtensorMap* map, const void* base, int BH, int N, int d, int rows = 128) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N) * d};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// One thread waits, with the kernels' bounded wait, on a barrier nobody arrives at.
__global__ void selftest_wait_kernel(unsigned* err, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    fa::mbar_init(fa::smem_u32(&bar), 1);
    fa::fence_barrier_init();
  }
  __syncthreads();
  const fa::Ctl ctl{&abort_flag, err, timeout_ns};
  if (threadIdx.x == 0) fa::mbar_wait(fa::smem_u32(&bar), 0, ctl);
}

int fwd_bf16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int N, int d, float scale, int causal, bool sparse, const uint8_t* block_mask,
             fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (sparse && !block_mask) return FA_ERR_INVALID_ARG;
  int st = check_common(B, H, N, scale);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;

  fa::FwdParams p{};
  const int BH = B * H;
  if (!encode_bf16_map(&p.tm_q, q, BH, N, d) || !encode_bf16_map(&p.tm_k, k, BH, N, d) ||
      !encode_bf16_map(&p.tm_v, v, BH, N, d) || !encode_bf16_map(&p.tm_o, o, BH, N, d))
    return FA_ERR_CUDA;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.block_mask = block_mask;
  p.BH = BH;
  p.N = N;
  p.n_tiles = (N + 127) / 128;
  const long long kv_bytes_per_head = 2ll * N * d * 2;
  long long g = (32ll << 20) / kv_bytes_per_head;
  p.heads_per_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_scale = 1.f;
  p.exp2_poly = g_exp2_per32.load(std::memory_order_relaxed) != 0 ? 1 : 0;
  p.err = ds->err;
  p.timeout_ns = kWaitTimeoutNs;
  if (static_cast<long long>(p.n_tiles) * BH > 0x7fffffffll) return FA_ERR_TOO_LARGE;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  // Two 128-row query tiles per CTA, each with its own MMA-issuing warp, K/V streamed once for
  // 256 rows. It beat a one-query-tile kernel with double-buffered scores on every measured shape
  // (TFLOPS, pair / single): d = 128 causal N = 8192 1618 / 1376, dense N = 8192 1692 / 1446,
  // causal N = 4096 1251 / 1125, dense B16 N = 512 593 / 554; d = 64 dense N = 2048 702-728 /
  // ~600; block-sparse d = 64 at 25% density 678 / 632.
  return to_status(fa::launch_fwd_pair(p, d, cs));
}

// The e4m3 forward: the bf16 forward's kernel with 8-bit tiles (d = 128); O stays bf16.
int fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
            int d, float scale, float v_scale, int causal, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int st = check_common(B, H, N, scale);
  if (st != FA_OK) return st;
  if (!isfinite(v_scale)) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  fa::FwdParams p{};
  const int BH = B * H;
  if (!encode_u8_map(&p.tm_q, q, BH, N, d) || !encode_u8_map(&p.tm_k, k, BH, N, d) ||
      !encode_u8_map(&p.tm_v, v, BH, N, d) || !encode_bf16_map(&p.tm_o, o, BH, N, d))
    return FA_ERR_CUDA;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.block_mask = nullptr;
  p.BH = BH;
  p.N = N;
  p.n_tiles = (N + 127) / 128;
  const long long kv_bytes_per_head = 2ll * N * d;
  long long g = (32ll << 20) / kv_bytes_per_head;
  p.heads_per_group = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  p.causal = causal ? 1 : 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.o_scale = v_scale;
  p.err = ds->err;
  p.timeout_ns = kWaitTimeoutNs;
  if (static_cast<long long>(p.n_tiles) * BH > 0x7fffffffll) return FA_ERR_TOO_LARGE;
  return to_status(fa::launch_fwd_fp8(p, reinterpret_cast<cudaStream_t>(stream)));
}

// CTAs for decoding: one per SM (the kernel holds 192 KB of keys and values in flight), never
// more than there are key blocks.
int decode_auto_ctas(int BH, int Nk, int d, const DeviceState& ds) {
  const int kB = fa::decode_tc_block_keys(d);
  const long long blocks = static_cast<long long>(BH) * ((Nk + kB - 1) / kB);
  long long n = ds.num_sms;
  if (n > fa::kDecodeMaxCtas) n = fa::kDecodeMaxCtas;
  return static_cast<int>(n < blocks ? n : blocks);
}

int check_decode(int B, int H, int Nq, int Nk, int d, float scale) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (Nq > fa::kDecodeMaxNq || (d != 64 && d != 128)) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H * (Nk > Nq ? Nk : Nq) > 0x7fffffffll) return FA_ERR_TOO_LARGE;
  return FA_OK;
}

int bwd_bf16(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, float* dq, void* dk, void* dv, int B, int H, int N, int d,
             float scale, int causal, bool sparse, const uint8_t* block_mask, void* workspace,
             fa_stream_t stream) {
  int st = fa::check_bwd_args(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, sparse,
                              block_mask, workspace, true);
  if (st != FA_OK) return st;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  fa::BwdParams p{};
  const int BH = B * H;
  if (!encode_bf16_map(&p.tm_q, q, BH, N, d) || !encode_bf16_map(&p.tm_k, k, BH, N, d) ||
      !encode_bf16_map(&p.tm_v, v, BH, N, d) || !encode_bf16_map(&p.tm_do, dO, BH, N, d) ||
      !encode_f32_map(&p.tm_dq, dq, BH, N, d))
    return FA_ERR_CUDA;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dO = static_cast<const __nv_bfloat16*>(dO);
  p.lse = lse;
  p.dq = dq;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  const size_t rows = static_cast<size_t>(BH) * ((static_cast<size_t>(N) + 127) / 128) * 128;
  p.lse2 = static_cast<float*>(workspace);
  p.Dsum = static_cast<float*>(workspace) + rows;
  p.aug = d == 64 ? static_cast<uint8_t*>(workspace) + rows * 2 * sizeof(float) : nullptr;
  p.ctr = reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) +
                                      rows * fa::bwd_row_workspace_bytes(d));
  p.BH = BH;
  p.N = N;
  p.d = d;
  p.n_tiles = (N + 127) / 128;
  p.causal = causal ? 1 : 0;
  p.block_mask = block_mask;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = ds->err;
  p.timeout_ns = kWaitTimeoutNs;
  return to_status(fa::launch_bwd(p, ds->num_sms, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace

// Argument checks of the backward entry points, in the order every one of them applies them.
int fa::check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dO,
                       const float* lse, const float* dq, const void* dk, const void* dv, int B,
                       int H, int N, int d, float scale, bool sparse, const uint8_t* block_mask,
                       const void* workspace, bool needs_workspace) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv || (needs_workspace && !workspace))
    return FA_ERR_INVALID_ARG;
  if (sparse && !block_mask) return FA_ERR_INVALID_ARG;
  const int st = check_common(B, H, N, scale);
  if (st != FA_OK) return st;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (sparse && (N + 127) / 128 > fa::kBwdMaxMaskTiles) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dO) ||
      !aligned16(lse) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      (needs_workspace && !aligned16(workspace)))
    return FA_ERR_MISALIGNED;
  return FA_OK;
}

extern "C" {

int fa_abi_version(void) { return (2 << 16) | 8; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported head dimension or sequence length";
    case FA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case FA_ERR_CUDA: return "CUDA call failed";
    case FA_ERR_DEVICE_TIMEOUT: return "kernel gave up waiting on an on-chip barrier";
    case FA_ERR_NO_DEVICE: return "no current sm_103 CUDA device";
    case FA_ERR_TOO_LARGE: return "problem too large for the kernels' indexing";
    case FA_ERR_SCRATCH_LIMIT:
      return "problem needs more scratch than fa_bwd_noalloc's static buffer "
             "(FA_NOALLOC_SCRATCH_BYTES) holds";
    default: return "unknown status";
  }
}

int fa_set_exp2_emulation(int per32) {
  if (per32 != 0 && per32 != fa::kExp2EmulationPer32) return FA_ERR_INVALID_ARG;
  g_exp2_per32.store(per32, std::memory_order_relaxed);
  return FA_OK;
}

int fa_get_exp2_emulation(void) { return g_exp2_per32.load(std::memory_order_relaxed); }

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, fa_stream_t stream) {
  return fwd_bf16(q, k, v, o, lse, B, H, N, d, scale, causal, false, nullptr, stream);
}

int fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                       fa_stream_t stream) {
  return fwd_bf16(q, k, v, o, lse, B, H, N, d, scale, causal, true, block_mask, stream);
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, float v_scale, int causal, fa_stream_t stream) {
  return fwd_fp8(q, k, v, o, lse, B, H, N, d, scale, v_scale, causal, stream);
}

namespace {
int fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int H,
             int N, int d, float scale, int causal, bool fa1, fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  int st = check_common(B, H, N, scale);
  if (st != FA_OK) return st;
  if (d < 32 || d > 128 || d % 32 != 0) return FA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_MISALIGNED;
  if (static_cast<long long>(B) * H > 65535) return FA_ERR_TOO_LARGE;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  fa::Fp32FwdParams p{q, k, v, o, lse, B * H, N, d, causal ? 1 : 0,
                      scale * 1.4426950408889634f, fa1 ? 1 : 0};
  return to_status(fa::launch_fwd_fp32(p, ds->num_sms, reinterpret_cast<cudaStream_t>(stream)));
}
}  // namespace

int fa_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  return fwd_fp32(q, k, v, o, lse, B, H, N, d, scale, causal, false, stream);
}

int fa_fwd_fp32_fa1(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                    int H, int N, int d, float scale, int causal, fa_stream_t stream) {
  return fwd_fp32(q, k, v, o, lse, B, H, N, d, scale, causal, true, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 1 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * ((static_cast<size_t>(N) + 127) / 128) * 128;
  // per row lse2 and D (and at d = 64 their operand rows), then the work counters
  return rows * fa::bwd_row_workspace_bytes(d) + fa::bwd_counter_bytes(static_cast<size_t>(B) * H);
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, float* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, fa_stream_t stream) {
  return bwd_bf16(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, false, nullptr,
                  workspace, stream);
}

int fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                       const void* dO, const float* lse, float* dq, void* dk, void* dv, int B,
                       int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                       void* workspace, fa_stream_t stream) {
  return bwd_bf16(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, true, block_mask,
                  workspace, stream);
}

int fa_decode_ctas(int B, int H, int Nq, int Nk, int d) {
  if (check_decode(B, H, Nq, Nk, d, 1.f) != FA_OK) return 0;
  DeviceState* ds = nullptr;
  if (device_state(&ds) != FA_OK) return 0;
  return decode_auto_ctas(B * H, Nk, d, *ds);
}

size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d) {
  if (check_decode(B, H, Nq, Nk, d, 1.f) != FA_OK) return 0;
  const long long BH = static_cast<long long>(B) * H;
  const int kB = fa::decode_tc_block_keys(d);
  long long ctas = BH * ((Nk + kB - 1) / kB);
  if (ctas > fa::kDecodeMaxCtas) ctas = fa::kDecodeMaxCtas;
  return static_cast<size_t>((ctas + BH) * Nq * (d + 1)) * sizeof(float);
}

int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, float scale, int n_ctas, void* workspace,
              fa_stream_t stream) {
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  int st = check_decode(B, H, Nq, Nk, d, scale);
  if (st != FA_OK) return st;
  if (n_ctas < 0 || n_ctas > fa::kDecodeMaxCtas) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return FA_ERR_MISALIGNED;
  DeviceState* ds = nullptr;
  if ((st = device_state(&ds)) != FA_OK) return st;
  const int BH = B * H;
  if (n_ctas == 0) n_ctas = decode_auto_ctas(BH, Nk, d, *ds);
  fa::DecodeParams p{};  // the launcher sets the block count and caps n_ctas at it
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.BH = BH;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_ctas = n_ctas;
  p.ws_o = static_cast<float*>(workspace);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.err = ds->err;
  p.timeout_ns = kWaitTimeoutNs;
  // rows past Nq of the Q tile (16 rows at d = 128, 128 at d = 64) and keys past Nk read as zero
  // through the tensor maps
  if (!encode_bf16_map(&p.tm_q, q, BH, Nq, d, 16) ||
      !encode_bf16_map(&p.tm_k, k, BH, Nk, d) ||
      !encode_bf16_map(&p.tm_v, v, BH, Nk, d))
    return FA_ERR_CUDA;
  return to_status(fa::launch_decode(p, d, reinterpret_cast<cudaStream_t>(stream)));
}

int fa_selftest_wait_timeout(unsigned timeout_us, fa_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 10000000u) return FA_ERR_INVALID_ARG;
  DeviceState* ds = nullptr;
  const int st = device_state(&ds);
  if (st != FA_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      ds->err, static_cast<unsigned long long>(timeout_us) * 1000ull);
  return to_status(cudaGetLastError());
}

int fa_check_device_error(fa_stream_t stream) {
  DeviceState* ds = nullptr;
  int st = device_state(&ds);
  if (st != FA_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  unsigned word = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return FA_ERR_CUDA;
  if (word != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

}  // extern "C"
