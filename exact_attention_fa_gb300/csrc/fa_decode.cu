// Decoding attention: a few query rows against a long key/value sequence ("3 · FlashAttention",
// 3.6 "L'attention en décodage" and the Flash-Decoding row of 3.7).
//
// With Nq <= 8 query rows per head the work is a matrix-vector product: every key and value row
// is used Nq times, so the kernel is bound by HBM bandwidth, not by arithmetic, and the tensor
// cores would sit idle (128-row MMA tiles for a handful of rows). GB300 mapping:
//   * Flash-Decoding's split of the keys, balanced for a fixed grid: the key blocks (32 keys at
//     d = 128, 64 at d = 64: 16 KB of K and V either way) of all heads, head after head, are
//     dealt out as G equal contiguous ranges, one per CTA, with G = the CTAs the SMs hold at
//     once (persistent: no tail wave, every SM streams until the end). A range may start or end
//     inside a head and may span several heads;
//   * one warp of the CTA streams its range with 1-D bulk copies (cp.async.bulk) into per-warp
//     shared-memory rings of (K block, V block) pairs (128 KB in flight per CTA), across head
//     boundaries, guarded by full / empty mbarriers;
//   * eight compute warps take the blocks in turn, each with an online softmax state of its own
//     ("3 · FlashAttention", 3.3): lane = key (two keys at d = 64) for the scores q.k (16-byte
//     loads rotated by lane, so no bank conflicts), warp shuffles for the block's max and sum,
//     lane = 4 output columns for O += P V (at d = 64 the two half-warps take alternate keys).
//     No CTA-wide barrier per block: the warps meet only where a head ends inside the range, to
//     merge their states into that (CTA, head) piece;
//   * each piece holds O_c / l_c and its log-sum-exp lse_c; a second kernel merges the pieces of
//     each head with the same statistics merge as the blockwise forward (lse = log Σ exp lse_c,
//     O = Σ exp(lse_c - lse) O_c).
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int kWarps = 8;              // compute warps; warp kWarps streams the blocks in
constexpr int kThreads = 32 * (kWarps + 1);
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DCfg {
  // Each compute warp has a ring of its own (one consumer per stage, so the phase parity of a
  // stage's barrier always refers to the block the warp expects): one 16 KB stage per warp,
  // 128 KB in flight per CTA.
  static constexpr int kStagesPerWarp = 1;
  static constexpr int kStages = kWarps * kStagesPerWarp;
  // keys per block: 16 KB per (K, V) block pair either way, so one key per lane at d = 128 and two
  // at d = 64 (lanes l and l + 32)
  static constexpr int kBK = D == 128 ? 32 : 64;
  static constexpr int kKeysPerLane = kBK / 32;
  static constexpr int kBlockBytes = kBK * D * 2;  // one K or V block, bf16
  static constexpr int kStageBytes = 2 * kBlockBytes;
  static constexpr int kOffQ = kStages * kStageBytes;                // fp32 [kDecodeMaxNq][D]
  static constexpr int kOffO = kOffQ + kDecodeMaxNq * D * 4;         // fp32 [kWarps][Nq][D]
  static constexpr int kOffML = kOffO + kWarps * kDecodeMaxNq * D * 4;  // fp32 [kWarps][Nq][2]
  static constexpr int kOffBar = kOffML + kWarps * kDecodeMaxNq * 8;
  static constexpr int kOffAbort = kOffBar + 16 * kStages;         // full[S], empty[S]
  static constexpr int kSmemBytes = kOffAbort + 16;
  static constexpr int kLanesPerRow = D / 4;   // lanes covering one V row, 4 columns each
  static constexpr int kKeySplit = 32 / kLanesPerRow;  // keys a warp takes at once in O += P V
};

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// CTA of global key block g (blocks of all heads in a row, head-major): blocks are dealt out as
// G contiguous ranges [c*T/G, (c+1)*T/G).
__device__ __forceinline__ int cta_of_block(long long g, long long T, int G) {
  return static_cast<int>(((g + 1) * G - 1) / T);
}

// CTA c streams its range of key blocks. Warp kWarps copies them in order into the rings;
// compute warp w takes the CTA-local blocks i = w (mod kWarps) (lane = key) with an online
// softmax state of its own per head, and at the end of each head's stretch of the range the
// warps' states are merged into the piece (c, head h) at slot c + h: O_piece / l_piece and
// lse_piece (log2 units). Along the ranges (c, h) only ever steps forward, so c + h is unique.
template <int D, int NQ>
__global__ void __launch_bounds__(kThreads, 1) decode_stream_kernel(const __grid_constant__ DecodeParams p) {
  using C = DCfg<D>;
  constexpr int S = C::kStages;
  constexpr int R = C::kStagesPerWarp;
  // CTA-local block i belongs to compute warp i % kWarps, as that warp's k-th block
  // (k = i / kWarps): stage (i % kWarps) * R + k % R, phase k / R of that stage.
  auto stage_of = [&](int i) { return (i % kWarps) * R + (i / kWarps) % R; };
  auto parity_of = [&](int i) { return static_cast<uint32_t>((i / kWarps / R) & 1); };
  constexpr int kKS = C::kKeySplit;
  constexpr int kBK = C::kBK;
  constexpr int kKPL = C::kKeysPerLane;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int Nq = p.Nq;
  const int nb = p.blocks_per_head;
  const long long T = static_cast<long long>(p.BH) * nb;
  const int G = gridDim.x, c = blockIdx.x;
  const long long g0 = c * T / G;
  const int nblk = static_cast<int>((c + 1) * T / G - g0);
  float* qs = reinterpret_cast<float*>(smem + C::kOffQ);
  float* wo = reinterpret_cast<float*>(smem + C::kOffO);
  float* wml = reinterpret_cast<float*>(smem + C::kOffML);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  auto full = [&](int s) { return sbase + C::kOffBar + 8u * s; };
  auto empty = [&](int s) { return sbase + C::kOffBar + 8u * (S + s); };
  auto keys_in = [&](long long g) {
    const int jb = static_cast<int>(g % nb);
    return min(kBK, p.Nk - jb * kBK);
  };

  if (tid == 0) {
    *abort_flag = 0;
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer (whole warp)
    int i = 0;
    bool ok = true;
    for (; i < nblk; ++i) {
      const int s = stage_of(i);
      if (!mbar_wait_warp(empty(s), parity_of(i) ^ 1u, ctl)) { ok = false; break; }
      const long long g = g0 + i;
      const int h = static_cast<int>(g / nb), jb = static_cast<int>(g % nb);
      const uint32_t bytes = static_cast<uint32_t>(keys_in(g)) * D * 2;
      const size_t off = (static_cast<size_t>(h) * p.Nk + static_cast<size_t>(jb) * kBK) * D;
      mbar_arrive_expect_tx(full(s), 2 * bytes);
      tma_bulk_g2s(sbase + s * C::kStageBytes, p.k + off, bytes, full(s));
      tma_bulk_g2s(sbase + s * C::kStageBytes + C::kBlockBytes, p.v + off, bytes, full(s));
    }
    if (!ok) {
      // Give the copies in flight a bounded time to land before the CTA exits.
      Ctl drain = ctl;
      int zero = 0;
      drain.abort_flag = &zero;
      for (int b = max(0, i - S); b < i; ++b) mbar_wait_warp(full(stage_of(b)), parity_of(b), drain);
    }
    return;
  }

  // ------------------------------------------------------------------ compute warps
  constexpr int kChunks = D / 8;  // 16-byte chunks per key row
  const int sub = lane / C::kLanesPerRow, col4 = (lane % C::kLanesPerRow) * 4;
  bool ok = true;
  long long g = g0;
  const long long g_end = g0 + nblk;
  while (g < g_end) {
    const int h = static_cast<int>(g / nb);
    const long long seg_end = min(g_end, static_cast<long long>(h + 1) * nb);
    // q of head h, pre-multiplied by scale * log2(e) so that scores come out in log2 units
    const __nv_bfloat16* qg = p.q + static_cast<size_t>(h) * Nq * D;
    for (int e = tid; e < Nq * D; e += 32 * kWarps) qs[e] = __bfloat162float(qg[e]) * p.scale_log2;
    bar_sync(1, 32 * kWarps);

    float m[NQ], l[NQ], acc[NQ][4];
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      m[j] = -INFINITY;
      l[j] = 0.f;
#pragma unroll
      for (int t = 0; t < 4; ++t) acc[j][t] = 0.f;
    }
    // this warp's blocks of the stretch: CTA-local indices congruent to warp mod kWarps
    const int first = static_cast<int>(g - g0);
    for (int i = first + (warp - first % kWarps + kWarps) % kWarps; ok && g0 + i < seg_end;
         i += kWarps) {
      const long long gb = g0 + i;
      const int s = stage_of(i);
      if (!mbar_wait_warp(full(s), parity_of(i), ctl)) { ok = false; break; }
      const int n = keys_in(gb);
      const __nv_bfloat16* Ks = reinterpret_cast<const __nv_bfloat16*>(smem + s * C::kStageBytes);
      const __nv_bfloat16* Vs = Ks + kBK * D;

      // scores of keys lane + 32 u (16-byte chunks in an order rotated by lane: no bank
      // conflicts), two partial sums per key and query row for short dependency chains
      float sc[NQ][kKPL][2];
#pragma unroll
      for (int j = 0; j < NQ; ++j)
#pragma unroll
        for (int u = 0; u < kKPL; ++u) sc[j][u][0] = sc[j][u][1] = 0.f;
#pragma unroll
      for (int u = 0; u < kKPL; ++u) {
        const int key = lane + 32 * u;
        if (key < n) {
#pragma unroll
          for (int cc = 0; cc < kChunks; ++cc) {
            const int ch = (cc + lane) % kChunks;
            float kf[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4*>(Ks + key * D + ch * 8), kf);
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
              if (j < Nq) {
                const float4 qa = *reinterpret_cast<const float4*>(qs + j * D + ch * 8);
                const float4 qb = *reinterpret_cast<const float4*>(qs + j * D + ch * 8 + 4);
                float a = sc[j][u][cc % 2];
                a = fmaf(qa.x, kf[0], a); a = fmaf(qa.y, kf[1], a);
                a = fmaf(qa.z, kf[2], a); a = fmaf(qa.w, kf[3], a);
                a = fmaf(qb.x, kf[4], a); a = fmaf(qb.y, kf[5], a);
                a = fmaf(qb.z, kf[6], a); a = fmaf(qb.w, kf[7], a);
                sc[j][u][cc % 2] = a;
              }
            }
          }
        }
      }
      // online softmax per query row (the block's scores sit kKPL per lane)
      float pj[NQ][kKPL];
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        if (j < Nq) {
          float sj[kKPL];
          float mx = -INFINITY;
#pragma unroll
          for (int u = 0; u < kKPL; ++u) {
            sj[u] = lane + 32 * u < n ? sc[j][u][0] + sc[j][u][1] : -INFINITY;
            mx = fmaxf(mx, sj[u]);
          }
#pragma unroll
          for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(~0u, mx, o));
          const float m_new = fmaxf(m[j], mx);  // finite: the block has at least one key
          float ps = 0.f;
#pragma unroll
          for (int u = 0; u < kKPL; ++u) {
            pj[j][u] = ex2(sj[u] - m_new);
            ps += pj[j][u];
          }
#pragma unroll
          for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(~0u, ps, o);
          const float alpha = ex2(m[j] - m_new);  // 0 while nothing was accumulated
          l[j] = l[j] * alpha + ps;
          m[j] = m_new;
#pragma unroll
          for (int t = 0; t < 4; ++t) acc[j][t] *= alpha;
        }
      }
      // O += P V: lane owns 4 columns of a V row; at d = 64 the two half-warps take alternate
      // keys (kKS = 2) and are summed at the end. Keys past n contribute p = 0 and v = 0.
      for (int k0 = 0; k0 < n; k0 += 8 * kKS) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int key = k0 + u * kKS + sub;
          uint2 w = make_uint2(0u, 0u);
          if (key < n) w = *reinterpret_cast<const uint2*>(Vs + key * D + col4);
          const float vf[4] = {__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                               __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u)};
#pragma unroll
          for (int j = 0; j < NQ; ++j) {
            if (j < Nq) {
              // key's P sits in lane key % 32, slot key / 32 (the same slot for both
              // half-warps: k0 + u * kKS is even)
              const float pk = __shfl_sync(~0u, pj[j][(k0 + u * kKS) >> 5], key & 31);
#pragma unroll
              for (int t = 0; t < 4; ++t) acc[j][t] = fmaf(pk, vf[t], acc[j][t]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(s));
    }

    // merge the warps' states into the piece (c, h)
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      if (j < Nq) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          float a = acc[j][t];
          if constexpr (kKS == 2) a += __shfl_xor_sync(~0u, a, 16);
          if (sub == 0) wo[(warp * kDecodeMaxNq + j) * D + col4 + t] = a;
        }
        if (lane == 0) {
          wml[(warp * kDecodeMaxNq + j) * 2] = m[j];
          wml[(warp * kDecodeMaxNq + j) * 2 + 1] = l[j];
        }
      }
    }
    if (bar_red_or(1, 32 * kWarps, !ok)) return;
    const size_t slot = static_cast<size_t>(c) + h;
    for (int e = tid; e < Nq * D; e += 32 * kWarps) {
      const int j = e / D, col = e % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wml[(w * kDecodeMaxNq + j) * 2]);
      float L = 0.f, a = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = ex2(wml[(w * kDecodeMaxNq + j) * 2] - M);  // 0 for an idle warp
          L = fmaf(f, wml[(w * kDecodeMaxNq + j) * 2 + 1], L);
          a = fmaf(f, wo[(w * kDecodeMaxNq + j) * D + col], a);
        }
      }
      p.ws_o[(slot * Nq + j) * D + col] = L > 0.f ? a / L : 0.f;
      if (col == 0) p.ws_lse[slot * Nq + j] = L > 0.f ? M + __log2f(L) : -INFINITY;
    }
    bar_sync(1, 32 * kWarps);  // wo, wml and qs are free again
    g = seg_end;
  }
}

// One CTA of D threads per (head, query row): merges the pieces of the CTAs whose block ranges
// cover the head (lse = log2 Σ 2^lse_c, O = Σ 2^(lse_c - lse) O_c). The pieces' weights are
// formed in parallel in shared memory, so the loop over pieces issues independent loads.
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ float wts[kDecodeMaxCtas];
  __shared__ float red[D / 32];
  const int row = blockIdx.x;  // h * Nq + i
  const int h = row / p.Nq, i = row - h * p.Nq;
  const int t = threadIdx.x, lane = t % 32, warp = t / 32;
  const long long T = static_cast<long long>(p.BH) * p.blocks_per_head;
  const int c0 = cta_of_block(static_cast<long long>(h) * p.blocks_per_head, T, p.n_ctas);
  const int c1 = cta_of_block(static_cast<long long>(h + 1) * p.blocks_per_head - 1, T, p.n_ctas);
  const int n = c1 - c0 + 1;  // <= n_ctas <= kDecodeMaxCtas
  auto slot = [&](int k) { return (static_cast<size_t>(c0 + k) + h) * p.Nq + i; };
  auto block_reduce = [&](float v, bool is_max) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float x = __shfl_xor_sync(~0u, v, o);
      v = is_max ? fmaxf(v, x) : v + x;
    }
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < D / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    __syncthreads();
    return r;
  };
  float mx = -INFINITY;
  for (int k = t; k < n; k += D) {
    wts[k] = p.ws_lse[slot(k)];
    mx = fmaxf(mx, wts[k]);
  }
  mx = block_reduce(mx, true);
  const size_t out = static_cast<size_t>(row) * D + t;
  if (mx == -INFINITY) {
    p.o[out] = __float2bfloat16_rn(0.f);
    if (t == 0) p.lse[row] = -INFINITY;
    return;
  }
  float den = 0.f;
  for (int k = t; k < n; k += D) {
    wts[k] = ex2(wts[k] - mx);  // 0 for an empty piece
    den += wts[k];
  }
  den = block_reduce(den, false);  // its barrier also publishes wts
  float a = 0.f;
#pragma unroll 4
  for (int k = 0; k < n; ++k) a = fmaf(wts[k], p.ws_o[slot(k) * D + t], a);
  p.o[out] = __float2bfloat16_rn(a / den);
  if (t == 0) p.lse[row] = (mx + __log2f(den)) * kLn2;
}

template <int D, int NQ>
cudaError_t configure() {
  return cudaFuncSetAttribute(decode_stream_kernel<D, NQ>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<D>::kSmemBytes);
}

template <int D>
cudaError_t configure_d() {
  cudaError_t e = configure<D, 1>();
  if (e == cudaSuccess) e = configure<D, 2>();
  if (e == cudaSuccess) e = configure<D, 4>();
  if (e == cudaSuccess) e = configure<D, 8>();
  return e;
}

// Kernel instances for at most 1, 2, 4 and 8 query rows (registers scale with the bound).
template <int D, int NQ>
cudaError_t launch_nq(const DecodeParams& p, cudaStream_t s) {
  decode_stream_kernel<D, NQ><<<p.n_ctas, kThreads, DCfg<D>::kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch(const DecodeParams& p_in, cudaStream_t s) {
  // the block size is the kernel's: blocks per head, the CTA count (at most one per block) and
  // the pieces' layout in the workspace follow from it
  DecodeParams p = p_in;
  p.blocks_per_head = (p.Nk + DCfg<D>::kBK - 1) / DCfg<D>::kBK;
  const long long blocks = static_cast<long long>(p.BH) * p.blocks_per_head;
  if (p.n_ctas > blocks) p.n_ctas = static_cast<int>(blocks);
  p.ws_lse = p.ws_o + static_cast<size_t>(p.n_ctas + p.BH) * p.Nq * D;
  cudaError_t e = p.Nq <= 1   ? launch_nq<D, 1>(p, s)
                  : p.Nq <= 2 ? launch_nq<D, 2>(p, s)
                  : p.Nq <= 4 ? launch_nq<D, 4>(p, s)
                              : launch_nq<D, 8>(p, s);
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D><<<static_cast<unsigned>(p.BH) * p.Nq, D, 0, s>>>(p);
  return cudaGetLastError();
}

// Resident CTAs per SM of the largest instance (the others use no more registers).
template <int D>
int resident_ctas() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_stream_kernel<D, kDecodeMaxNq>,
                                                    kThreads, DCfg<D>::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n < 1 ? 1 : n;
}

}  // namespace

cudaError_t configure_decode() {
  const cudaError_t e = configure_d<64>();
  return e != cudaSuccess ? e : configure_d<128>();
}

int decode_ctas_per_sm(int d) { return d == 128 ? resident_ctas<128>() : resident_ctas<64>(); }

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t s) {
  if (d == 64) return launch<64>(p, s);
  if (d == 128) return launch<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
