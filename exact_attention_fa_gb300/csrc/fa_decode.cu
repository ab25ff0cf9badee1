// Decoding attention: a few query rows against a long key/value sequence ("3 · FlashAttention",
// 3.6 "L'attention en décodage" and the Flash-Decoding row of 3.7).
//
// With Nq <= 8 query rows per head every key and value row is used Nq times: the work is a
// matrix-vector product bound by HBM bandwidth. Flash-Decoding's split of the keys, balanced for a
// fixed grid: the key blocks of all heads, head after head, are dealt out as G equal contiguous
// ranges, one per CTA, with G = the SM count (persistent: no tail wave, every SM streams until the
// end). A range may start or end inside a head and may span several heads. Each CTA turns each
// head's stretch of its range into a piece (O_c / l_c and its log-sum-exp lse_c); a second kernel
// merges the pieces of each head with the same statistics merge as the blockwise forward
// (lse = log sum_c exp lse_c, O = sum_c exp(lse_c - lse) O_c).
//
// The products run on the tensor cores (decode_tc_kernel below). A CUDA-core kernel (lane = key
// for the scores, lane = output columns for P V) did 2 Nq d FMAs per key against 4 d bytes of K
// and V: it reached 6091 GB/s (d = 128) and 6177 (d = 64) with one query row but only 1132 with
// eight; the tensor-core kernel streams 6977 / 6556 GB/s with one row and 7061 / 6508 with eight.
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr float kLn2 = 0.6931471805599453f;

// CTA of global key block g (blocks of all heads in a row, head-major): blocks are dealt out as
// G contiguous ranges [c*T/G, (c+1)*T/G).
__device__ __forceinline__ int cta_of_block(long long g, long long T, int G) {
  return static_cast<int>(((g + 1) * G - 1) / T);
}

// One CTA of D threads per (head, query row): merges the pieces of the CTAs whose block ranges
// cover the head (lse = log2 Σ 2^lse_c, O = Σ 2^(lse_c - lse) O_c). The pieces' weights are
// formed in parallel in shared memory, so the loop over pieces issues independent loads.
// It is launched as a programmatic dependent of the split kernel (the launch overlaps the split
// kernel's tail) and waits here until that grid has completed and its pieces are visible.
template <int D>
__global__ void __launch_bounds__(D) decode_merge_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ float wts[kDecodeMaxCtas];
  __shared__ float red[D / 32];
  asm volatile("griddepcontrol.wait;" ::: "memory");
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
// The decoding kernel. Each key block is a small forward tile: S = Q K^T and O += P V as
// tcgen05.mma with Q zero-padded to a 128-row tile by the TMA (rows past Nq read as zero), so the
// tensor core does 128 / Nq times the useful work but still needs far less time per block than
// HBM needs to deliver the block's K and V.
//   * the stretch of one head inside a CTA's range is a segment;
//   * warp 1 loads Q of each segment and the (K, V) blocks with TMA into a ring;
//   * warp 2 issues the MMAs: S of the next block as soon as the softmax has read this one (two
//     TMEM buffers at d = 128, one of 256 keys at d = 64), then P V into the segment's O;
//   * warps 0 and 4 are the softmax (both reach TMEM lanes 0-31): thread r of each owns query row
//     r (rows >= Nq carry zeros and are never stored), warp 0 the first half of a block's keys and
//     warp 4 the second; they exchange the block's row max through shared memory, so both use one reference
//     max, and each keeps its own part of the running sum. Online softmax as in the forward, P as
//     bf16 into TMEM; at the end of a segment O / l and the log-sum-exp are written as the piece
//     (CTA, head), merged per head by decode_merge_kernel.
// Blocks of 256 keys at d = 64 and 128 at d = 128: 32 KB of K and of V per block either way, so
// that the per-block costs (barrier round trips, MMA issue) weigh the same per byte.
// TMEM columns: d = 128: S_0 [0, 128), S_1 [128, 256), P [256, 320), O [320, 448); d = 64:
// S [0, 256), P [256, 384), O [384, 448).
template <int D>
struct TcCfg {
  static constexpr int kBK = decode_tc_block_keys(D);  // 32 KB of K and of V per block
  static constexpr int kHalfKeys = kBK / 2;            // keys per softmax warp
  static constexpr int kQTile = 128 * D * 2;           // the Q tile (bf16)
  static constexpr int kKV = kBK * D * 2;              // a K or a V block
  static constexpr int kBox = 128 * 64 * 2;            // one TMA box: 128 rows x 64 columns
  static constexpr int kRowBoxes = kBK / 128;          // boxes along the keys of a block
  static constexpr int kColBoxes = D / 64;             // boxes along d
  static constexpr int kStages = 3;                    // (K, V) pairs in flight: 192 KB
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kQTile;
  static constexpr int kOffBar = kOffRing + kStages * 2 * kKV;
  // d = 128: two S buffers of 128 columns; d = 64: one of 256 (S of the next block is still
  // issued as soon as both softmax warps have read this one)
  static constexpr int kSBufs = D == 64 ? 1 : 2;
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
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColP = kSBufs * kBK;    // kBK / 2 columns of bf16 pairs
  static constexpr uint32_t kColO = kColP + kBK / 2;  // D columns; at most 448 in all
  static_assert(kColO + D <= 512, "TMEM columns");
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
  // the merge kernel may be scheduled as soon as every CTA of this grid has started (it waits
  // for this grid's completion before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

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
      mbar_arrive_expect_tx(bar(C::kBarQFull), C::kQTile);
      for (int b = 0; b < C::kColBoxes; ++b)
        tma_load_3d(sbase + C::kOffQ + b * C::kBox, &p.tm_q, bar(C::kBarQFull), b * 64, 0, h);
      for (; i < e; ++i) {
        const int st = i % C::kStages, round = i / C::kStages;
        if (!(ok = mbar_wait_warp(bar(C::kBarEmpty + st), (round & 1) ^ 1, ctl))) break;
        const int jb = static_cast<int>((rg.g0 + i) % rg.nb);
        const uint32_t dst = sbase + C::kOffRing + st * 2 * C::kKV;
        mbar_arrive_expect_tx(bar(C::kBarFull + st), 2 * C::kKV);
        // column box b (64 of d) at b * kBK * 128 bytes, row box rb (128 keys) at rb * 16 KB
        // inside it: the 128-byte-swizzled layout of the whole kBK x D tile
        for (int rb = 0; rb < C::kRowBoxes; ++rb)
          for (int b = 0; b < C::kColBoxes; ++b) {
            const uint32_t off = b * C::kBK * 128 + rb * C::kBox;
            const int row = jb * C::kBK + rb * 128;
            tma_load_3d(dst + off, &p.tm_k, bar(C::kBarFull + st), b * 64, row, h);
            tma_load_3d(dst + C::kKV + off, &p.tm_v, bar(C::kBarFull + st), b * 64, row, h);
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
    const uint64_t vd0 = sdesc64(sdesc_lo(sbase + C::kOffRing + C::kKV, C::kBK * 128), kHi);
    constexpr uint64_t kStageStep = (2 * C::kKV) >> 4;
    bool ok = true;
    int ns = 0;  // S products issued (buffer ns % 2)
    auto issue_s = [&](int i) {  // S of CTA-local block i (its K stage must be full)
      const int b = ns % C::kSBufs;
      if (ns >= C::kSBufs) {
        if (!mbar_wait_warp(bar(C::kBarSFree + b), (ns / C::kSBufs - 1) & 1, ctl)) return false;
        tc_fence_after();
      }
      const int st = i % C::kStages;
      if (!mbar_wait_warp(bar(C::kBarFull + st), (i / C::kStages) & 1, ctl)) return false;
      tc_fence_after();
      if constexpr (D == 128)
        mma_qk_d128(tmem + C::kColS + C::kBK * b, qd, kd0 + st * kStageStep, kIdescS);
      else
        mma_qk_d64(tmem + C::kColS + C::kBK * b, qd, kd0 + st * kStageStep, kIdescS);
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
        // 128 keys per call: P columns 64 apart, V rows 16 KB apart (1024 in 16-byte units)
#pragma unroll
        for (int rb = 0; rb < C::kRowBoxes; ++rb)
          mma_pv_k128(tmem + C::kColO, tmem + C::kColP + 64u * rb,
                      vd0 + (i % C::kStages) * kStageStep + 1024u * rb, kIdescPV,
                      (i > i0 || rb > 0) ? 1u : 0u);
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
        constexpr int kH = C::kHalfKeys;
        const int sb = i % C::kSBufs;
        if (!(ok = mbar_wait(bar(C::kBarSFull + sb), (i / C::kSBufs) & 1, ctl))) break;
        tc_fence_after();
        uint32_t sc[kH];
        if constexpr (kH == 128)
          tmem_ld128(trow + C::kColS + C::kBK * sb + kH * hf, sc);
        else
          tmem_ld64(trow + C::kColS + C::kBK * sb + kH * hf, sc);
        tc_fence_before();
        mbar_arrive(bar(C::kBarSFree + sb));
        const int b = i & 1;  // exchange slot
        const int jb = static_cast<int>((rg.g0 + i) % rg.nb);
        const int n = min(C::kBK, p.Nk - jb * C::kBK) - kH * hf;  // keys of this half
        if (n < kH) {
#pragma unroll
          for (int k = 0; k < kH; ++k)
            if (k >= n) sc[k] = __float_as_uint(-INFINITY);
        }
        float mxa[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          mxa[u] = max3(-INFINITY, __uint_as_float(sc[2 * u]), __uint_as_float(sc[2 * u + 1]));
#pragma unroll
        for (int k = 16; k < kH; k += 16)
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
        uint32_t pk[kH / 2];
#pragma unroll
        for (int u = 0; u < kH / 2; ++u) {
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
#pragma unroll
        for (int u = 0; u < kH / 32; ++u)
          tmem_st16(trow + C::kColP + (kH / 2) * hf + 16u * u, pk + 16 * u);
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

}  // namespace

cudaError_t configure_decode() {
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<64>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<128>::kSmemBytes);
  return e;
}

namespace {
template <int D>
cudaError_t launch_tc(const DecodeParams& p_in, cudaStream_t s) {
  // the block size is the kernel's: blocks per head, the CTA count (at most one per block) and
  // the pieces' layout in the workspace follow from it
  DecodeParams p = p_in;
  p.blocks_per_head = (p.Nk + TcCfg<D>::kBK - 1) / TcCfg<D>::kBK;
  const long long blocks = static_cast<long long>(p.BH) * p.blocks_per_head;
  if (p.n_ctas > blocks) p.n_ctas = static_cast<int>(blocks);
  p.ws_lse = p.ws_o + static_cast<size_t>(p.n_ctas + p.BH) * p.Nq * D;
  decode_tc_kernel<D><<<p.n_ctas, kTcThreads, TcCfg<D>::kSmemBytes, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the merge kernel's launch overlaps the split kernel's tail
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(p.BH) * p.Nq);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
}
}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t s) {
  if (d == 64) return launch_tc<64>(p, s);
  if (d == 128) return launch_tc<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
