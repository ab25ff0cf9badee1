// Decoding attention: a few query rows against a long key/value sequence ("3 · FlashAttention",
// 3.6 "L'attention en décodage" and the Flash-Decoding row of 3.7).
//
// With Nq <= 8 query rows per head the work is a matrix-vector product: every key and value row
// is used Nq times, so decoding is bound by HBM bandwidth. Two kernels, chosen by measurement
// (fa_api.cu): decode_tc_kernel (further below: the products on the tensor cores, 128-key blocks)
// for d = 128 and for several query rows, and decode_stream_kernel (the CUDA cores) for one query
// row at d = 64, where it keeps up with HBM and the tensor-core kernel's per-block costs do not.
// decode_stream_kernel, GB300 mapping (its template covers more shapes than the one it runs for):
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

// ---------------------------------------------------------------------------------------------
// Decoding with several query rows (2 <= Nq <= kDecodeMaxNq) on the tensor cores. With Nq rows the
// CUDA-core kernel above does 2 Nq d FMAs per key against 4 d bytes of K and V, which at Nq = 8
// runs out of FMA throughput long before HBM runs out of bytes. Here each 128-key block is a small
// forward tile: S = Q K^T and O += P V as tcgen05.mma with Q zero-padded to a 128-row tile by the
// TMA (rows past Nq read as zero), so the tensor core does 128 / Nq times the useful work but
// still needs far less time per block than HBM needs to deliver the block's K and V.
//   * the key blocks of all heads are dealt out as in the kernel above (equal contiguous ranges,
//     one per CTA, head-major), the stretch of one head inside a range being a segment;
//   * warp 1 loads Q of each segment and the (K, V) blocks with TMA into a ring;
//   * warp 2 issues the MMAs: S into one of two TMEM buffers, so that S of the next block is
//     computed while the softmax works on this one, then P V into the segment's O;
//   * warps 0 and 4 are the softmax (both reach TMEM lanes 0-31): thread r of each owns query row
//     r (rows >= Nq carry zeros and are never stored), warp 0 keys 0-63 of a block and warp 4 keys
//     64-127; they exchange the block's row max through shared memory, so both use one reference
//     max, and each keeps its own part of the running sum. Online softmax as in the forward, P as
//     bf16 into TMEM; at the end of a segment O / l and the log-sum-exp are written as the piece
//     (CTA, head), merged per head by decode_merge_kernel.
// TMEM columns: S_0 [0, 128), S_1 [128, 256), P [256, 320), O [320, 320 + D).
template <int D>
struct TcCfg {
  static constexpr int kBK = kDecodeTcBlockKeys;
  static constexpr int kTile = 128 * D * 2;           // Q, a K block or a V block (bf16)
  static constexpr int kBox = 128 * 64 * 2;           // one TMA box: 128 rows x 64 columns
  static constexpr int kStages = D == 128 ? 3 : 6;    // (K, V) pairs in flight: 192 KB
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kTile;
  static constexpr int kOffBar = kOffRing + kStages * 2 * kTile;
  // barriers: full[S], empty[S], q_full, q_empty, s_full[2], s_free[2], p_full, pv_done, o_done,
  // o_free, drain
  static constexpr int kBarFull = 0;
  static constexpr int kBarEmpty = kStages;
  static constexpr int kBarQFull = 2 * kStages;
  static constexpr int kBarQEmpty = kBarQFull + 1;
  static constexpr int kBarSFull = kBarQFull + 2;
  static constexpr int kBarSFree = kBarSFull + 2;
  static constexpr int kBarPFull = kBarSFree + 2;
  static constexpr int kBarPVDone = kBarPFull + 1;
  static constexpr int kBarODone = kBarPVDone + 1;
  static constexpr int kBarOFree = kBarODone + 1;
  static constexpr int kBarDrain = kBarOFree + 1;
  static constexpr int kBarX = kBarDrain + 1;  // [2] the softmax warps' row maxima, per parity
  static constexpr int kBarL = kBarX + 2;      // their running sums at the end of a segment
  static constexpr int kNumBars = kBarL + 1;
  // the two softmax warps' row maxima per block parity and their running sums: [2][2][32] + [2][32]
  static constexpr int kOffX = kOffBar + 8 * kNumBars;
  static constexpr int kOffTmemPtr = kOffX + (2 * 2 * 32 + 2 * 32) * 4;
  static constexpr int kOffAbort = kOffTmemPtr + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KB
  static constexpr uint32_t kColS = 0, kColP = 256, kColO = 320;
};
constexpr int kTcThreads = 160;  // warps: 0 and 4 softmax, 1 TMA, 2 MMA, 3 idle

// The CTA's range [g0, g0 + nblk) of global block indices (head-major) and the segment of head h
// inside it.
struct TcRange {
  long long g0;
  int nblk, nb;
  __device__ __forceinline__ int head(long long g) const { return static_cast<int>(g / nb); }
  // one past the last CTA-local block index of the segment that starts at local index i
  __device__ __forceinline__ int seg_end(int i) const {
    const long long h = (g0 + i) / nb;
    return static_cast<int>(min(g0 + nblk, (h + 1) * nb) - g0);
  }
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ DecodeParams p) {
  using C = TcCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemPtr);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const long long T = static_cast<long long>(p.BH) * p.blocks_per_head;
  const int G = gridDim.x, c = blockIdx.x;
  TcRange rg;
  rg.g0 = c * T / G;
  rg.nblk = static_cast<int>((c + 1) * T / G - rg.g0);
  rg.nb = p.blocks_per_head;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarQFull), 1);
    mbar_init(bar(C::kBarQEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kBarSFull + b), 1);
      mbar_init(bar(C::kBarSFree + b), 64);
    }
    mbar_init(bar(C::kBarPFull), 64);
    mbar_init(bar(C::kBarPVDone), 1);
    mbar_init(bar(C::kBarODone), 1);
    mbar_init(bar(C::kBarOFree), 64);
    mbar_init(bar(C::kBarDrain), 1);
    mbar_init(bar(C::kBarX + 0), 64);
    mbar_init(bar(C::kBarX + 1), 64);
    mbar_init(bar(C::kBarL), 64);
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 1) {
    // ------------------------------------------------------------------- TMA (whole warp)
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    bool ok = true;
    int seg = 0, issued_last = -1;
    for (int i = 0; ok && i < rg.nblk;) {
      const int h = rg.head(rg.g0 + i);
      const int e = rg.seg_end(i);
      if (seg > 0 && !(ok = mbar_wait_warp(bar(C::kBarQEmpty), (seg - 1) & 1, ctl))) break;
      mbar_arrive_expect_tx(bar(C::kBarQFull), C::kTile);
      for (int b = 0; b < D / 64; ++b)
        tma_load_3d(sbase + C::kOffQ + b * C::kBox, &p.tm_q, bar(C::kBarQFull), b * 64, 0, h);
      for (; i < e; ++i) {
        const int st = i % C::kStages, round = i / C::kStages;
        if (!(ok = mbar_wait_warp(bar(C::kBarEmpty + st), (round & 1) ^ 1, ctl))) break;
        const int jb = static_cast<int>((rg.g0 + i) % rg.nb);
        const uint32_t dst = sbase + C::kOffRing + st * 2 * C::kTile;
        mbar_arrive_expect_tx(bar(C::kBarFull + st), 2 * C::kTile);
        for (int b = 0; b < D / 64; ++b) {
          tma_load_3d(dst + b * C::kBox, &p.tm_k, bar(C::kBarFull + st), b * 64, jb * C::kBK, h);
          tma_load_3d(dst + C::kTile + b * C::kBox, &p.tm_v, bar(C::kBarFull + st), b * 64,
                      jb * C::kBK, h);
        }
        issued_last = i;
      }
      ++seg;
    }
    if (!ok) {
      // give the copies in flight a bounded time to land before the CTA exits
      Ctl drain = ctl;
      int zero = 0;
      drain.abort_flag = &zero;
      for (int b = max(0, issued_last - C::kStages + 1); b <= issued_last; ++b)
        mbar_wait_warp(bar(C::kBarFull + b % C::kStages), (b / C::kStages) & 1, drain);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------- MMA (whole warp)
    constexpr uint32_t kIdescS = idesc_bf16(128, C::kBK, 0, 0);  // A = Q, B = K, both K-major
    constexpr uint32_t kIdescPV = idesc_bf16(128, D, 0, 1);      // A = P (TMEM), B = V MN-major
    constexpr uint32_t kHi = sdesc_hi_sw128(1024);
    uint64_t qd[D / 16];
#pragma unroll
    for (int k = 0; k < D / 16; ++k)
      qd[k] = sdesc64(sdesc_lo(sbase + C::kOffQ + (k / 4) * C::kBox + (k % 4) * 32, 16), kHi);
    const uint64_t kd0 = sdesc64(sdesc_lo(sbase + C::kOffRing, 16), kHi);
    const uint64_t vd0 = sdesc64(sdesc_lo(sbase + C::kOffRing + C::kTile, C::kBox), kHi);
    constexpr uint64_t kStageStep = (2 * C::kTile) >> 4;
    bool ok = true;
    int ns = 0;  // S products issued (buffer ns % 2)
    auto issue_s = [&](int i) {  // S of CTA-local block i (its K stage must be full)
      const int b = ns & 1;
      if (ns >= 2) {
        if (!mbar_wait_warp(bar(C::kBarSFree + b), ((ns >> 1) - 1) & 1, ctl)) return false;
        tc_fence_after();
      }
      const int st = i % C::kStages;
      if (!mbar_wait_warp(bar(C::kBarFull + st), (i / C::kStages) & 1, ctl)) return false;
      tc_fence_after();
      if constexpr (D == 128)
        mma_qk_d128(tmem + C::kColS + 128u * b, qd, kd0 + st * kStageStep, kIdescS);
      else
        mma_qk_d64(tmem + C::kColS + 128u * b, qd, kd0 + st * kStageStep, kIdescS);
      mma_commit(bar(C::kBarSFull + b));
      ++ns;
      return true;
    };
    int seg = 0;
    for (int i = 0; ok && i < rg.nblk; ++seg) {
      const int e = rg.seg_end(i);
      if (!(ok = mbar_wait_warp(bar(C::kBarQFull), seg & 1, ctl))) break;
      tc_fence_after();
      if (!(ok = issue_s(i))) break;
      for (int i0 = i; i < e; ++i) {
        if (i + 1 < e) {
          if (!(ok = issue_s(i + 1))) break;
        } else {
          mma_commit(bar(C::kBarQEmpty));  // every S of the segment issued: Q is free after them
        }
        if (!(ok = mbar_wait_warp(bar(C::kBarPFull), i & 1, ctl))) break;
        tc_fence_after();
        if (i == i0 && seg > 0) {  // O still holds the previous segment until the softmax read it
          if (!(ok = mbar_wait_warp(bar(C::kBarOFree), (seg - 1) & 1, ctl))) break;
          tc_fence_after();
        }
        mma_pv_k128(tmem + C::kColO, tmem + C::kColP, vd0 + (i % C::kStages) * kStageStep,
                    kIdescPV, i > i0 ? 1u : 0u);
        mma_commit(bar(C::kBarPVDone));
        mma_commit(bar(C::kBarEmpty + i % C::kStages));
        if (i + 1 == e) mma_commit(bar(C::kBarODone));
      }
    }
    if (!ok) {
      // let the MMAs already issued finish before TMEM is released
      Ctl drain = ctl;
      int zero = 0;
      drain.abort_flag = &zero;
      mma_commit(bar(C::kBarDrain));
      mbar_wait_warp(bar(C::kBarDrain), 0, drain);
    }
  } else if (warp == 0 || warp == 4) {
    // ------------------------------------------------------------------- softmax (thread = row)
    const int hf = warp >> 2;  // half of the block's keys: [64 hf, 64 hf + 64)
    const int r = lane;
    const uint32_t trow = tmem;  // lanes 0-31: the quarter of warps 0 and 4
    float* xm = reinterpret_cast<float*>(smem + C::kOffX);  // [parity][half][row]
    float* xl = xm + 2 * 2 * 32;                              // [half][row]
    const float sl2 = p.scale_log2;
    bool ok = true;
    int seg = 0;
    for (int i = 0; ok && i < rg.nblk; ++seg) {
      const int h = rg.head(rg.g0 + i);
      const int e = rg.seg_end(i);
      float m = -INFINITY, l = 0.f;  // l: this warp's part of the running sum
      for (int i0 = i; i < e; ++i) {
        const int b = i & 1;
        if (!(ok = mbar_wait(bar(C::kBarSFull + b), (i >> 1) & 1, ctl))) break;
        tc_fence_after();
        uint32_t sc[64];
        tmem_ld64(trow + C::kColS + 128u * b + 64u * hf, sc);
        tc_fence_before();
        mbar_arrive(bar(C::kBarSFree + b));
        const int jb = static_cast<int>((rg.g0 + i) % rg.nb);
        const int n = min(C::kBK, p.Nk - jb * C::kBK) - 64 * hf;  // keys of this half
        if (n < 64) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k >= n) sc[k] = __float_as_uint(-INFINITY);
        }
        float mxa[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          mxa[u] = max3(-INFINITY, __uint_as_float(sc[2 * u]), __uint_as_float(sc[2 * u + 1]));
#pragma unroll
        for (int k = 16; k < 64; k += 16)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mxa[u] = max3(mxa[u], __uint_as_float(sc[k + 2 * u]), __uint_as_float(sc[k + 2 * u + 1]));
        const float mh = max3(max3(mxa[0], mxa[1], mxa[2]), max3(mxa[3], mxa[4], mxa[5]),
                              fmaxf(mxa[6], mxa[7])) * sl2;  // -inf for a half with no key
        // the block's row max over both halves: two slots and barriers by block parity (a warp
        // reaches slot b again only after the partner has arrived for the block in between, so
        // after it read the slot), bounded waits, so that a warp that gave up cannot strand the
        // other one
        xm[(b * 2 + hf) * 32 + r] = mh;
        mbar_arrive(bar(C::kBarX + b));
        if (!(ok = mbar_wait(bar(C::kBarX + b), (i >> 1) & 1, ctl))) break;
        const float mx = fmaxf(mh, xm[(b * 2 + (hf ^ 1)) * 32 + r]);
        const float m_new = fmaxf(m, mx);  // finite: a block holds at least one key
        // the exponentials first, into registers: they overlap the previous block's P V, which
        // has to be done only before P is rewritten and O rescaled
        const unsigned long long k2 = f2_pack(sl2, sl2);
        const unsigned long long nm2 = f2_pack(-m_new, -m_new);
        unsigned long long rs[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) rs[u] = f2_pack(0.f, 0.f);
        uint32_t pk[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const unsigned long long x = f2_fma(
              f2_pack(__uint_as_float(sc[2 * u]), __uint_as_float(sc[2 * u + 1])), k2, nm2);
          float x0, x1;
          f2_unpack(x, x0, x1);
          const float p0 = ex2(x0), p1 = ex2(x1);
          rs[u & 3] = f2_add(rs[u & 3], f2_pack(p0, p1));
          pk[u] = pack_bf16(p0, p1);
        }
        if (i > 0) {
          if (!(ok = mbar_wait(bar(C::kBarPVDone), (i - 1) & 1, ctl))) break;
          tc_fence_after();
        }
        if (i > i0 && __any_sync(~0u, m_new > m)) {  // the same decision in both warps
          const float alpha = ex2(m - m_new);
#pragma unroll 1
          for (int cc = hf * (D / 2); cc < (hf + 1) * (D / 2); cc += 32) {
            uint32_t o[32];
            tmem_ld32(trow + C::kColO + cc, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            tmem_st32(trow + C::kColO + cc, o);
          }
          l *= alpha;
        }
        m = m_new;
        tmem_st16(trow + C::kColP + 32u * hf, pk);
        tmem_st16(trow + C::kColP + 32u * hf + 16, pk + 16);
        float rs0, rs1;
        f2_unpack(f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3])), rs0, rs1);
        l += rs0 + rs1;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(C::kBarPFull));
      }
      if (!ok) break;
      // the segment's piece: O / l and its log-sum-exp (log2 units), rows < Nq, each warp half
      // of the columns
      if (!(ok = mbar_wait(bar(C::kBarODone), seg & 1, ctl))) break;
      tc_fence_after();
      xl[hf * 32 + r] = l;
      mbar_arrive(bar(C::kBarL));
      if (!(ok = mbar_wait(bar(C::kBarL), seg & 1, ctl))) break;
      const float lt = xl[r] + xl[32 + r];
      const size_t slot = static_cast<size_t>(c) + h;
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll 1
      for (int cc = hf * (D / 2); cc < (hf + 1) * (D / 2); cc += 32) {
        uint32_t o[32];
        tmem_ld32(trow + C::kColO + cc, o);
        if (r < p.Nq) {
          float4* dst = reinterpret_cast<float4*>(p.ws_o + (slot * p.Nq + r) * D + cc);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(o[4 * k]) * inv, __uint_as_float(o[4 * k + 1]) * inv,
                                 __uint_as_float(o[4 * k + 2]) * inv,
                                 __uint_as_float(o[4 * k + 3]) * inv);
        }
      }
      if (hf == 0 && r < p.Nq) p.ws_lse[slot * p.Nq + r] = lt > 0.f ? m + __log2f(lt) : -INFINITY;
      tc_fence_before();
      mbar_arrive(bar(C::kBarOFree));
    }
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, int NQ>
cudaError_t configure() {
  return cudaFuncSetAttribute(decode_stream_kernel<D, NQ>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<D>::kSmemBytes);
}

// The CUDA-core kernel runs for one query row at d = 64 only (the tensor-core kernel below is
// faster everywhere else): its single instance.
cudaError_t launch_cuda_cores(const DecodeParams& p_in, cudaStream_t s) {
  // the block size is the kernel's: blocks per head, the CTA count (at most one per block) and
  // the pieces' layout in the workspace follow from it
  DecodeParams p = p_in;
  p.blocks_per_head = (p.Nk + DCfg<64>::kBK - 1) / DCfg<64>::kBK;
  const long long blocks = static_cast<long long>(p.BH) * p.blocks_per_head;
  if (p.n_ctas > blocks) p.n_ctas = static_cast<int>(blocks);
  p.ws_lse = p.ws_o + static_cast<size_t>(p.n_ctas + p.BH) * p.Nq * 64;
  decode_stream_kernel<64, 1><<<p.n_ctas, kThreads, DCfg<64>::kSmemBytes, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<64><<<static_cast<unsigned>(p.BH) * p.Nq, 64, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t configure_decode() {
  cudaError_t e = configure<64, 1>();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<64>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<128>::kSmemBytes);
  return e;
}

int decode_ctas_per_sm() {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_stream_kernel<64, 1>, kThreads,
                                                    DCfg<64>::kSmemBytes) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return n < 1 ? 1 : n;
}

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t s) {
  if (d != 64 || p.Nq != 1) return cudaErrorInvalidValue;
  return launch_cuda_cores(p, s);
}

namespace {
template <int D>
cudaError_t launch_tc(const DecodeParams& p_in, cudaStream_t s) {
  DecodeParams p = p_in;
  p.blocks_per_head = (p.Nk + kDecodeTcBlockKeys - 1) / kDecodeTcBlockKeys;
  const long long blocks = static_cast<long long>(p.BH) * p.blocks_per_head;
  if (p.n_ctas > blocks) p.n_ctas = static_cast<int>(blocks);
  p.ws_lse = p.ws_o + static_cast<size_t>(p.n_ctas + p.BH) * p.Nq * D;
  decode_tc_kernel<D><<<p.n_ctas, kTcThreads, TcCfg<D>::kSmemBytes, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D><<<static_cast<unsigned>(p.BH) * p.Nq, D, 0, s>>>(p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_tc(const DecodeParams& p, int d, cudaStream_t s) {
  if (d == 64) return launch_tc<64>(p, s);
  if (d == 128) return launch_tc<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
