// fp32 forward: tiled online softmax on the FMA pipes, for fp32 inputs where a bf16/tf32 tensor-
// core product would miss a 1e-5 accuracy bar.
//
// A CTA owns R consecutive query rows of one (b, h), one warp per row (R = 8; 2 or 4 when a grid
// of 8-row CTAs would leave SMs idle, so that small problems spread over more SMs). Key/value
// blocks of 32 rows are staged in shared memory and shared by the CTA's warps. Lane j scores key j of the
// block (a d-long dot product from shared memory); the warp then applies the online-softmax
// update of "FlashAttention：メモリ効率的なアテンション計算", section "オンライン softmax":
//   m_new = max(m, block max),  alpha = exp(m - m_new),  l = l*alpha + sum p,  o = o*alpha + sum p v
// with each lane owning d/32 output columns, and divides by l once at the end. Exponentials are
// base 2 with log2(e) folded into the scale.
//
// The kFA1 instance keeps the output normalised after every key block instead, the per-block
// update of FlashAttention-1 ("FlashAttention: IOを意識した高速かつメモリ効率の高い厳密なアテンション",
// "手法" steps 1-4): P~ is taken against the block's own max m~, l~ = rowsum P~, and
//   m_new = max(m, m~),  l_new = e^(m - m_new) l + e^(m~ - m_new) l~,
//   o = (l e^(m - m_new) o + e^(m~ - m_new) P~ V_j) / l_new.
// The result is the same up to rounding; the accumulator stays in registers (FA-2's loop order),
// so the per-block read and write of O that FA-1 does through HBM has no counterpart here.
//
// Small problems at d <= 96 (a grid of 8-row CTAs leaves SMs idle and a CTA's whole key range
// fits in shared memory) take fwd_fp32_small_kernel instead, for the FlashAttention-2 form: the CTA
// stages all the keys and values it needs at once (one round trip to L2 instead of one per
// block), each of its two query rows is split over kSplit warps that run the recurrence above on
// their own stretch of keys, and the warps' partial results are combined with the statistics
// merge of the blockwise method: M = max_s m_s, L = sum_s l_s 2^(m_s - M),
// O = sum_s o_s 2^(m_s - M) / L.
#include <cuda_bf16.h>
#include <math.h>

#include <type_traits>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kKeys = 32;  // keys per shared-memory block

template <int D, bool kFA1, int kRows>
__global__ void __launch_bounds__(kRows * 32) fwd_fp32_kernel(const Fp32FwdParams p) {
  constexpr int kThreads = kRows * 32;
  constexpr int C = D / 32;
  __shared__ float ks[kKeys][D + 1];  // +1: lane j reads row j without bank conflicts
  __shared__ __align__(16) float vs[kKeys][D];
  __shared__ float qs[kRows][D];

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row0 = blockIdx.x * kRows;
  const int row = row0 + warp;
  const size_t head = static_cast<size_t>(blockIdx.y) * p.N * D;
  const float* q = p.q + head;
  const float* k = p.k + head;
  const float* v = p.v + head;

#pragma unroll
  for (int i = threadIdx.x; i < kRows * D; i += kThreads) {
    const int r = row0 + i / D;
    qs[i / D][i % D] = r < p.N ? q[static_cast<size_t>(r) * D + i % D] : 0.f;
  }

  float m = -INFINITY, l = 0.f;
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;

  // A key/value block is kKeys x D floats of each; thread t holds float4 number t + u * kThreads
  // of both. The next block's loads are issued before this block's arithmetic, so the latency of
  // global memory overlaps the work instead of adding to it once per block.
  constexpr int kVec = kKeys * D / 4 / kThreads;  // D * 8 / kThreads
  static_assert(kVec * kThreads * 4 == kKeys * D, "a block is a whole number of float4 per thread");
  float4 kr[kVec], vr[kVec];
  auto fetch = [&](int kb) {
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const int e = (threadIdx.x + u * kThreads) * 4;
      const int j = kb + e / D;
      const size_t off = static_cast<size_t>(j) * D + e % D;
      const bool in = j < p.N;
      kr[u] = in ? *reinterpret_cast<const float4*>(k + off) : make_float4(0.f, 0.f, 0.f, 0.f);
      vr[u] = in ? *reinterpret_cast<const float4*>(v + off) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const int e = (threadIdx.x + u * kThreads) * 4;
      const int r = e / D, c = e % D;
      ks[r][c] = kr[u].x;
      ks[r][c + 1] = kr[u].y;
      ks[r][c + 2] = kr[u].z;
      ks[r][c + 3] = kr[u].w;
      *reinterpret_cast<float4*>(&vs[r][c]) = vr[u];
    }
  };

  const int kend = p.causal ? min(p.N, row0 + kRows) : p.N;
  if (kend > 0) fetch(0);
  for (int kb = 0; kb < kend; kb += kKeys) {
    __syncthreads();  // every warp is done with the previous block
    stash();
    __syncthreads();
    if (kb + kKeys < kend) fetch(kb + kKeys);
    if (row >= p.N) continue;

    const int j = kb + lane;
    // the d-long dot product in four independent chains
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < D; c += 4)
#pragma unroll
      for (int u = 0; u < 4; ++u) s4[u] = fmaf(qs[warp][c + u], ks[lane][c + u], s4[u]);
    float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    const bool ok = j < p.N && (!p.causal || j <= row);
    s = ok ? s * p.scale_log2 : -INFINITY;

    float bmax = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(~0u, bmax, off));
    if constexpr (kFA1) {
      if (bmax == -INFINITY) continue;  // no allowed key in this block
      const float pj = ok ? exp2f(s - bmax) : 0.f;  // P~ against the block max m~
      float lt = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) lt += __shfl_xor_sync(~0u, lt, off);
      const float m_new = fmaxf(m, bmax);
      const float c_old = exp2f(m - m_new);  // 0 before the first block (m = -inf)
      const float c_new = exp2f(bmax - m_new);
      const float l_new = c_old * l + c_new * lt;
      float pv[C];
#pragma unroll
      for (int c = 0; c < C; ++c) pv[c] = 0.f;
#pragma unroll 4
      for (int jj = 0; jj < kKeys; ++jj) {
        const float pjj = __shfl_sync(~0u, pj, jj);
#pragma unroll
        for (int c = 0; c < C; ++c) pv[c] = fmaf(pjj, vs[jj][lane + 32 * c], pv[c]);
      }
      const float inv = 1.f / l_new;
      const float keep = l * c_old * inv, add = c_new * inv;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = fmaf(acc[c], keep, pv[c] * add);
      l = l_new;
      m = m_new;
      continue;
    }
    const float m_new = fmaxf(m, bmax);
    if (m_new == -INFINITY) continue;  // no allowed key for this row yet
    const float alpha = exp2f(m - m_new);  // 0 while nothing has been accumulated
    const float pj = ok ? exp2f(s - m_new) : 0.f;
    float psum = pj;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(~0u, psum, off);
    l = l * alpha + psum;
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] *= alpha;
#pragma unroll 4
    for (int jj = 0; jj < kKeys; ++jj) {
      const float pjj = __shfl_sync(~0u, pj, jj);
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] = fmaf(pjj, vs[jj][lane + 32 * c], acc[c]);
    }
    m = m_new;
  }

  if (row < p.N) {
    const float inv = kFA1 ? 1.f : (l > 0.f ? 1.f / l : 0.f);  // FA-1: o is already normalised
    float* o = p.o + head + static_cast<size_t>(row) * D;
#pragma unroll
    for (int c = 0; c < C; ++c) o[lane + 32 * c] = acc[c] * inv;
    if (lane == 0)
      p.lse[static_cast<size_t>(blockIdx.y) * p.N + row] =
          l > 0.f ? (m + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

// ---------------------------------------------------------------------------------------------
constexpr int kSmallRows = 2;   // query rows per CTA
constexpr int kSplit = 8;       // warps per query row, each over its own stretch of keys
constexpr int kSmallThreads = kSmallRows * kSplit * 32;
constexpr int kSmallMaxSmem = 200 * 1024;

// Shared memory of the small kernel for a CTA that stages n keys: K rows padded to D + 4 floats
// (lanes reading rows j as float4 then hit distinct banks), V rows, the query rows, and the
// partial results (m, l, o) of every warp.
__host__ __device__ constexpr size_t small_smem_bytes(int D, int n) {
  return (static_cast<size_t>(n) * (D + 4) + static_cast<size_t>(n) * D + kSmallRows * D +
          kSmallRows * kSplit * (D + 2)) * sizeof(float);
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}

// n_cap: the key rows the shared-memory layout is sized for (>= every CTA's key range).
template <int D>
__global__ void __launch_bounds__(kSmallThreads) fwd_fp32_small_kernel(const Fp32FwdParams p,
                                                                       int n_cap) {
  constexpr int C = D / 32;
  constexpr int kKStride = D + 4;
  extern __shared__ __align__(16) float sm[];
  float* ks = sm;                                // [n_cap][D + 4]
  float* vs = ks + static_cast<size_t>(n_cap) * kKStride;  // [n_cap][D]
  float* qs = vs + static_cast<size_t>(n_cap) * D;         // [kSmallRows][D]
  float* part = qs + kSmallRows * D;             // [kSmallRows][kSplit][D + 2]: o, m, l

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int row0 = blockIdx.x * kSmallRows;
  const int kend = p.causal ? min(p.N, row0 + kSmallRows) : p.N;  // keys this CTA needs
  const size_t head = static_cast<size_t>(blockIdx.y) * p.N * D;
  const float* q = p.q + head;
  const float* k = p.k + head;
  const float* v = p.v + head;

  for (int i = threadIdx.x; i < kend * (D / 4); i += kSmallThreads) {
    const int j = i / (D / 4), c = 4 * (i % (D / 4));
    cp_async16(ks + j * kKStride + c, k + static_cast<size_t>(j) * D + c);
    cp_async16(vs + j * D + c, v + static_cast<size_t>(j) * D + c);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int i = threadIdx.x; i < kSmallRows * D; i += kSmallThreads) {
    const int r = row0 + i / D;
    qs[i] = r < p.N ? q[static_cast<size_t>(r) * D + i % D] : 0.f;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();

  const int r = warp / kSplit, sp = warp % kSplit;
  const int row = row0 + r;
  const int row_end = p.causal ? min(p.N, row + 1) : p.N;  // keys [0, row_end) are allowed
  const int chunk = (kend + kSplit * 32 - 1) / (kSplit * 32) * 32;
  const int k0 = sp * chunk, k1 = min(kend, k0 + chunk);
  float m = -INFINITY, l = 0.f;
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  if (row < p.N) {
    for (int kb = k0; kb < k1; kb += 32) {
      const int j = kb + lane;
      const float* kr = ks + min(j, k1 - 1) * kKStride;  // rows past the stretch: masked below
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < D; c += 4) {
        const float4 kk = *reinterpret_cast<const float4*>(kr + c);
        s4[0] = fmaf(qs[r * D + c], kk.x, s4[0]);
        s4[1] = fmaf(qs[r * D + c + 1], kk.y, s4[1]);
        s4[2] = fmaf(qs[r * D + c + 2], kk.z, s4[2]);
        s4[3] = fmaf(qs[r * D + c + 3], kk.w, s4[3]);
      }
      const bool ok = j < k1 && j < row_end;
      const float sc = ok ? ((s4[0] + s4[1]) + (s4[2] + s4[3])) * p.scale_log2 : -INFINITY;
      float bmax = sc;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(~0u, bmax, off));
      const float m_new = fmaxf(m, bmax);
      if (m_new == -INFINITY) continue;  // no allowed key for this row yet
      const float alpha = exp2f(m - m_new);
      const float pj = ok ? exp2f(sc - m_new) : 0.f;
      float psum = pj;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(~0u, psum, off);
      l = l * alpha + psum;
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c] *= alpha;
      const int nj = min(32, k1 - kb);  // staged rows only
#pragma unroll 4
      for (int jj = 0; jj < nj; ++jj) {
        const float pjj = __shfl_sync(~0u, pj, jj);
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] = fmaf(pjj, vs[(kb + jj) * D + lane + 32 * c], acc[c]);
      }
      m = m_new;
    }
  }
  float* mine = part + (r * kSplit + sp) * (D + 2);
#pragma unroll
  for (int c = 0; c < C; ++c) mine[lane + 32 * c] = acc[c];
  if (lane == 0) {
    mine[D] = m;
    mine[D + 1] = l;
  }
  __syncthreads();
  if (sp != 0 || row >= p.N) return;
  // the statistics merge of the row's kSplit partial results
  const float* pr = part + r * kSplit * (D + 2);
  float M = -INFINITY;
#pragma unroll
  for (int t = 0; t < kSplit; ++t) M = fmaxf(M, pr[t * (D + 2) + D]);
  float L = 0.f, o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;
#pragma unroll
  for (int t = 0; t < kSplit; ++t) {
    const float mt = pr[t * (D + 2) + D];
    const float wt = mt == -INFINITY ? 0.f : exp2f(mt - M);
    L = fmaf(pr[t * (D + 2) + D + 1], wt, L);
#pragma unroll
    for (int c = 0; c < C; ++c) o[c] = fmaf(pr[t * (D + 2) + lane + 32 * c], wt, o[c]);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  float* out = p.o + head + static_cast<size_t>(row) * D;
#pragma unroll
  for (int c = 0; c < C; ++c) out[lane + 32 * c] = o[c] * inv;
  if (lane == 0)
    p.lse[static_cast<size_t>(blockIdx.y) * p.N + row] =
        L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

template <int D, bool F, int R>
cudaError_t launch_rows(const Fp32FwdParams& p, cudaStream_t s) {
  fwd_fp32_kernel<D, F, R><<<dim3((p.N + R - 1) / R, p.BH), R * 32, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D, bool F>
cudaError_t launch_d(const Fp32FwdParams& p, int num_sms, cudaStream_t s) {
  // 8 rows per CTA unless that grid leaves SMs idle; then 2 (4 at d > 64, where a block's
  // prefetch registers per thread would double again)
  constexpr int kSmall = D <= 64 ? 2 : 4;
  const long long ctas8 = static_cast<long long>((p.N + 7) / 8) * p.BH;
  if (ctas8 < num_sms) {
    // (d = 128 would not fit its dot products in the 128 registers a 512-thread CTA allows)
    if constexpr (D <= 96) {
      const size_t smem = small_smem_bytes(D, p.N);
      if (!F && smem <= static_cast<size_t>(kSmallMaxSmem)) {
        const dim3 grid((p.N + kSmallRows - 1) / kSmallRows, p.BH);
        fwd_fp32_small_kernel<D><<<grid, kSmallThreads, smem, s>>>(p, p.N);
        return cudaGetLastError();
      }
    }
    return launch_rows<D, F, kSmall>(p, s);
  }
  return launch_rows<D, F, 8>(p, s);
}

}  // namespace

cudaError_t configure_fwd_fp32() {
  for (auto kern : {fwd_fp32_small_kernel<32>, fwd_fp32_small_kernel<64>, fwd_fp32_small_kernel<96>}) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmallMaxSmem);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_fwd_fp32(const Fp32FwdParams& p, int num_sms, cudaStream_t s) {
  auto go = [&](auto fa1) {
    constexpr bool F = decltype(fa1)::value;
    switch (p.d) {
      case 32: return launch_d<32, F>(p, num_sms, s);
      case 64: return launch_d<64, F>(p, num_sms, s);
      case 96: return launch_d<96, F>(p, num_sms, s);
      case 128: return launch_d<128, F>(p, num_sms, s);
      default: return cudaErrorInvalidValue;
    }
  };
  return p.fa1 ? go(std::true_type{}) : go(std::false_type{});
}

}  // namespace fa
