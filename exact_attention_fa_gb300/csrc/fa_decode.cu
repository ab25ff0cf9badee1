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
// The products run on the tensor cores (decode_kt_kernel below). A CUDA-core kernel (lane = key
// for the scores, lane = output columns for P V) did 2 Nq d FMAs per key against 4 d bytes of K
// and V: it reached 6091 GB/s (d = 128) and 6177 (d = 64) with one query row but only 1132 with
// eight; the tensor-core kernel streams about 7060 / 6650 GB/s with one row and 7030 / 6570
// with eight.
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

// ---------------------------------------------------------------------------------------------
// The decoding kernel: each key block's two products on the tensor cores, with the keys on the
// TMEM lanes:
//     S^T = K Q^T    (M = 128 keys, N = 16 query columns: Q zero-padded by the TMA)
//     O^T += V^T P^T (M = 128: the d columns of O, N = 16, K = the block's keys; P^T from shared
//                     memory)
// so that thread t of the four softmax warps (warp t / 32 reaches TMEM lanes 32 (t / 32) ...)
// owns key t of each 128-key row box: one exponential per useful query row, spread over all four
// SM sub-partitions. (With the query rows on the lanes instead, every exponential fell on the one
// sub-partition whose warps reach lanes 0-31, one instruction per key whatever Nq; measured on
// the same shapes the transposed form streams 0.7-2% more and calls with few blocks per CTA run 8%
// faster.) The block's max per query is a shuffle reduction in each warp and a bounded exchange
// between the four warps; each thread keeps its own part of the running sums; at the end of a
// segment thread t reads row t of O^T, i.e. column d = t of the piece.
//   * the stretch of one head inside a CTA's range is a segment;
//   * warp 4 loads Q of each segment and the (K, V) blocks with TMA into a ring;
//   * warp 5 issues the MMAs: S^T of the next block as soon as the softmax has read this one (two
//     TMEM buffers), then O^T of this block once P^T is in shared memory;
//   * warps 0-3 are the softmax, conditional rescaling as in the forward.
// A block is 32 KB of K and 32 KB of V at either head dimension (128 keys at d = 128, two row
// boxes of 128 keys at d = 64), so that the per-block costs weigh the same per byte. At d = 64
// the 128-row A operand V^T has only 64 rows: its second 64-row half aliases the first (box
// stride 0), and rows 64-127 of O^T repeat rows 0-63, unread.
// TMEM columns: S^T buffer sb, row box rb at (sb * kRB + rb) * 16; O^T after them (16 columns).
template <int D>
struct KtCfg {
  // a block is kRB row boxes of 128 keys (TMEM lanes of S^T): 32 KB of K and of V either way
  static constexpr int kRB = D == 64 ? 2 : 1;
  static constexpr int kBK = 128 * kRB;            // keys per block
  static_assert(kBK == decode_tc_block_keys(D), "the pieces' layout follows the block size");
  static constexpr int kNP = 16;                   // query columns of S^T, O^T (Nq <= 8)
  static constexpr int kKV = kBK * D * 2;          // a K or a V block: 32 KB
  static constexpr int kBox = 128 * 128;           // a 128-row, 64-column box of it: 16 KB
  static constexpr int kColBoxes = D / 64;         // boxes of row box rb at (rb * kColBoxes + b)
  static constexpr int kSmallBox = kNP * 128;      // a 64-column box of 16 rows: 2 KB
  static constexpr int kSteps = D / 16;            // K-steps of S^T
  static constexpr int kStages = 3;                // 192 KB of K and V in flight
  static constexpr int kOffRing = 0;
  static constexpr int kOffQ = kStages * 2 * kKV;                 // Q: 16 rows, D / 64 boxes
  static constexpr int kOffP = kOffQ + kColBoxes * kSmallBox;      // P^T: 16 rows x kBK keys
  static constexpr int kOffBar = kOffP + 2 * kRB * kSmallBox;
  static constexpr int kBarFull = 0;
  static constexpr int kBarEmpty = kStages;
  static constexpr int kBarQFull = 2 * kStages;
  static constexpr int kBarQEmpty = kBarQFull + 1;
  static constexpr int kBarSFull = kBarQFull + 2;  // [2]
  static constexpr int kBarSFree = kBarSFull + 2;  // [2]
  static constexpr int kBarPFull = kBarSFree + 2;
  static constexpr int kBarPVDone = kBarPFull + 1;
  static constexpr int kBarODone = kBarPVDone + 1;
  static constexpr int kBarOFree = kBarODone + 1;
  static constexpr int kBarDrain = kBarOFree + 1;
  static constexpr int kBarX = kBarDrain + 1;  // [2] the warps' block maxima, per block parity
  static constexpr int kBarL = kBarX + 2;      // their running sums at the end of a segment
  static constexpr int kNumBars = kBarL + 1;
  static constexpr int kOffX = kOffBar + 8 * kNumBars;  // [2][4][8] maxima, then [4][8] sums
  static constexpr int kOffTmemPtr = kOffX + (2 * 4 * 8 + 4 * 8) * 4;
  static constexpr int kOffAbort = kOffTmemPtr + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KB
  // S^T buffer sb, row box rb at kColS + (sb * kRB + rb) * kNP
  static constexpr uint32_t kColS = 0, kColO = 2 * kRB * kNP;
  static constexpr uint32_t kTmemCols = kColO + kNP <= 64 ? 64 : 128;
};
constexpr int kKtThreads = 192;  // warps: 0-3 softmax (thread = key), 4 TMA, 5 MMA

template <int D>
__global__ void __launch_bounds__(kKtThreads, 1) decode_kt_kernel(const __grid_constant__ DecodeParams p) {
  using C = KtCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemPtr);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
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
      mbar_init(bar(C::kBarSFree + b), 128);
      mbar_init(bar(C::kBarX + b), 128);
    }
    mbar_init(bar(C::kBarPFull), 128);
    mbar_init(bar(C::kBarPVDone), 1);
    mbar_init(bar(C::kBarODone), 1);
    mbar_init(bar(C::kBarOFree), 128);
    mbar_init(bar(C::kBarDrain), 1);
    mbar_init(bar(C::kBarL), 128);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
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
      mbar_arrive_expect_tx(bar(C::kBarQFull), C::kColBoxes * C::kSmallBox);
      for (int b = 0; b < C::kColBoxes; ++b)
        tma_load_3d(sbase + C::kOffQ + b * C::kSmallBox, &p.tm_q, bar(C::kBarQFull), b * 64, 0, h);
      for (; i < e; ++i) {
        const int st = i % C::kStages, round = i / C::kStages;
        if (!(ok = mbar_wait_warp(bar(C::kBarEmpty + st), (round & 1) ^ 1, ctl))) break;
        const int jb = static_cast<int>((rg.g0 + i) % rg.nb);
        const uint32_t dst = sbase + C::kOffRing + st * 2 * C::kKV;
        mbar_arrive_expect_tx(bar(C::kBarFull + st), 2 * C::kKV);
        for (int rb = 0; rb < C::kRB; ++rb)
          for (int b = 0; b < C::kColBoxes; ++b) {
            const uint32_t off = (rb * C::kColBoxes + b) * C::kBox;
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
  } else if (warp == 5) {
    // ------------------------------------------------------------------- MMA (whole warp)
    constexpr uint32_t kIdescS = idesc_bf16(128, C::kNP, 0, 0);  // A = K, B = Q: both K-major
    constexpr uint32_t kIdescO = idesc_bf16(128, C::kNP, 1, 0);  // A = V^T MN-major, B = P^T
    constexpr uint32_t kHi = sdesc_hi_sw128(1024);
    constexpr uint64_t kStageStep = (2 * C::kKV) >> 4;
    // per K-step of 16: K rows (32 bytes into the 128-byte swizzled rows, 64-column boxes 16 KB
    // apart), Q and P^T rows (boxes 2 KB apart), V^T (16 key rows = 2 KB further each step).
    // V^T is the 128-row A operand of O^T; at d = 64 its second 64 rows (the MN-major layout's
    // second 64-column box) alias the first (box stride 0): O^T rows 64-127 repeat rows 0-63
    // and are never read.
    uint64_t ka[8], qb[8], pb[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      ka[k] = sdesc64(sdesc_lo(sbase + C::kOffRing + (k / 4) * C::kBox + (k % 4) * 32, 16), kHi);
      qb[k] = sdesc64(sdesc_lo(sbase + C::kOffQ + (k / 4) * C::kSmallBox + (k % 4) * 32, 16), kHi);
      pb[k] = sdesc64(sdesc_lo(sbase + C::kOffP + (k / 4) * C::kSmallBox + (k % 4) * 32, 16), kHi);
    }
    const uint64_t va =
        sdesc64(sdesc_lo(sbase + C::kOffRing + C::kKV, D == 128 ? C::kBox : 0), kHi);
    bool ok = true;
    int ns = 0;  // S^T products issued (buffer ns % 2)
    auto issue_s = [&](int i) {  // S^T of CTA-local block i (its K stage must be full)
      const int b = ns % 2;
      if (ns >= 2) {
        if (!mbar_wait_warp(bar(C::kBarSFree + b), (ns / 2 - 1) & 1, ctl)) return false;
        tc_fence_after();
      }
      const int st = i % C::kStages;
      if (!mbar_wait_warp(bar(C::kBarFull + st), (i / C::kStages) & 1, ctl)) return false;
      tc_fence_after();
#pragma unroll
      for (int rb = 0; rb < C::kRB; ++rb) {
        uint64_t a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
          a[k] = ka[k] + st * kStageStep + ((rb * C::kColBoxes * C::kBox) >> 4);
        const uint32_t dst = tmem + C::kColS + (b * C::kRB + rb) * C::kNP;
        if constexpr (C::kSteps == 8)
          mma_ss_k8(dst, a, qb, kIdescS, 0u);
        else
          mma_ss_k4(dst, a, qb, kIdescS);
      }
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
          mma_commit(bar(C::kBarQEmpty));  // every S^T of the segment issued: Q is free after them
        }
        if (!(ok = mbar_wait_warp(bar(C::kBarPFull), i & 1, ctl))) break;
        tc_fence_after();
        if (i == i0 && seg > 0) {  // O^T still holds the previous segment until the softmax read it
          if (!(ok = mbar_wait_warp(bar(C::kBarOFree), (seg - 1) & 1, ctl))) break;
          tc_fence_after();
        }
#pragma unroll
        for (int rb = 0; rb < C::kRB; ++rb) {
          // keys of row box rb: its V rows, P^T boxes 2 rb and 2 rb + 1
          uint64_t a[8], bp[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            a[k] = va + (i % C::kStages) * kStageStep + ((rb * C::kColBoxes * C::kBox) >> 4) +
                   128u * k;
            bp[k] = pb[k] + ((rb * 2 * C::kSmallBox) >> 4);
          }
          mma_ss_k8(tmem + C::kColO, a, bp, kIdescO, (i > i0 || rb > 0) ? 1u : 0u);
        }
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
  } else {
    // --------------------------------------------------- softmax (warps 0-3, thread = key t)
    const int t = threadIdx.x;  // key t of each block; row t of O^T (column d = t of O)
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float* xm = reinterpret_cast<float*>(smem + C::kOffX);  // [parity][warp][query]
    float* xl = xm + 2 * 4 * 8;                              // [warp][query]
    uint8_t* pt = smem + C::kOffP;
    const float sl2 = p.scale_log2;
    const int nq = p.Nq;
    constexpr float kSlack = 8.f;  // log2 units: P stays <= 256, like the forward
    bool ok = true;
    int seg = 0;
    for (int i = 0; ok && i < rg.nblk; ++seg) {
      const int h = rg.head(rg.g0 + i);
      const int e = rg.seg_end(i);
      float m[8], l[8];  // per query: the reference max (the same in every thread), this
                         // thread's part of the running sum
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        m[q] = -INFINITY;
        l[q] = 0.f;
      }
      for (int i0 = i; i < e; ++i) {
        const int sb = i & 1;
        if (!(ok = mbar_wait(bar(C::kBarSFull + sb), (i >> 1) & 1, ctl))) break;
        tc_fence_after();
        constexpr int R = C::kRB;  // this thread's keys: t + 128 rb
        float x[R][8], wm[8];
        const int jb = static_cast<int>((rg.g0 + i) % rg.nb);
#pragma unroll
        for (int q = 0; q < 8; ++q) wm[q] = -INFINITY;
#pragma unroll
        for (int rb = 0; rb < R; ++rb) {
          uint32_t sv[16];
          tmem_ld16(tl + C::kColS + (sb * R + rb) * C::kNP, sv);
          const bool valid = jb * C::kBK + rb * 128 + t < p.Nk;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            x[rb][q] = (valid && q < nq) ? __uint_as_float(sv[q]) * sl2 : -INFINITY;
            wm[q] = fmaxf(wm[q], x[rb][q]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(C::kBarSFree + sb));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
#pragma unroll
          for (int q = 0; q < 8; ++q) wm[q] = fmaxf(wm[q], __shfl_xor_sync(~0u, wm[q], off));
        // the block max per query over the four warps: slots and barriers by block parity (a
        // warp reaches slot b again only after every warp has arrived for the block in between,
        // so after all of them read it), bounded waits
        const int b = i & 1;
        if (lane == 0)
#pragma unroll
          for (int q = 0; q < 8; ++q) xm[(b * 4 + warp) * 8 + q] = wm[q];
        mbar_arrive(bar(C::kBarX + b));
        if (!(ok = mbar_wait(bar(C::kBarX + b), (i >> 1) & 1, ctl))) break;
        float mb[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
          mb[q] = fmaxf(fmaxf(xm[(b * 4 + 0) * 8 + q], xm[(b * 4 + 1) * 8 + q]),
                        fmaxf(xm[(b * 4 + 2) * 8 + q], xm[(b * 4 + 3) * 8 + q]));
        // conditional rescaling: the reference moves only when a query's block max passes it by
        // more than kSlack (the same decision in every thread: the same inputs)
        bool move = false;
#pragma unroll
        for (int q = 0; q < 8; ++q) move |= q < nq && mb[q] > m[q] + kSlack;
        float alpha[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) alpha[q] = 1.f;
        if (move) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            if (q >= nq) continue;
            const float m_new = fmaxf(m[q], mb[q]);
            alpha[q] = m[q] == -INFINITY ? 0.f : ex2(m[q] - m_new);
            m[q] = m_new;
            l[q] *= alpha[q];
          }
        }
        // the exponentials first: they overlap the previous block's O^T product, which has to
        // be done only before P^T is rewritten and O^T rescaled
        float pv[R][8];
#pragma unroll
        for (int rb = 0; rb < R; ++rb)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            pv[rb][q] = q < nq ? ex2(x[rb][q] - m[q]) : 0.f;  // 0 for keys past Nk (x = -inf)
            l[q] += pv[rb][q];
          }
        if (i > 0) {
          if (!(ok = mbar_wait(bar(C::kBarPVDone), (i - 1) & 1, ctl))) break;
          tc_fence_after();
        }
        if (move && i > i0) {
          uint32_t o[16];
          tmem_ld16(tl + C::kColO, o);
#pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
          tmem_st16(tl + C::kColO, o);
          tmem_st_wait();
        }
        // P^T (row q, key t + 128 rb) as bf16 into the 128-byte-swizzled B tile: 64-key boxes
        // 2 KB apart
#pragma unroll
        for (int rb = 0; rb < R; ++rb) {
          const int kk = t + 128 * rb;
          uint8_t* prow = pt + (kk / 64) * C::kSmallBox + (kk % 8) * 2;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < nq)
              *reinterpret_cast<__nv_bfloat16*>(prow + q * 128 + ((((kk % 64) / 8) ^ q) << 4)) =
                  __float2bfloat16_rn(pv[rb][q]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(C::kBarPFull));
      }
      if (!ok) break;
      // the segment's piece: O / l and its log-sum-exp (log2 units), rows < Nq
      if (!(ok = mbar_wait(bar(C::kBarODone), seg & 1, ctl))) break;
      tc_fence_after();
      float ws[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        ws[q] = l[q];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ws[q] += __shfl_xor_sync(~0u, ws[q], off);
      }
      if (lane == 0)
#pragma unroll
        for (int q = 0; q < 8; ++q) xl[warp * 8 + q] = ws[q];
      mbar_arrive(bar(C::kBarL));
      if (!(ok = mbar_wait(bar(C::kBarL), seg & 1, ctl))) break;
      uint32_t o[16];
      tmem_ld16(tl + C::kColO, o);
      const size_t slot = static_cast<size_t>(c) + h;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (q >= nq) continue;
        const float lt = xl[q] + xl[8 + q] + xl[16 + q] + xl[24 + q];
        if (t < D) p.ws_o[(slot * nq + q) * D + t] = lt > 0.f ? __uint_as_float(o[q]) / lt : 0.f;
        if (t == q) p.ws_lse[slot * nq + q] = lt > 0.f ? m[q] + __log2f(lt) : -INFINITY;
      }
      tc_fence_before();
      mbar_arrive(bar(C::kBarOFree));
    }
  }
  __syncwarp();

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

}  // namespace

cudaError_t configure_decode() {
  cudaError_t e = cudaFuncSetAttribute(decode_kt_kernel<64>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       KtCfg<64>::kSmemBytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(decode_kt_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             KtCfg<128>::kSmemBytes);
  return e;
}

namespace {
template <int D>
cudaError_t launch_tc(const DecodeParams& p_in, cudaStream_t s) {
  // the block size is the kernel's: blocks per head, the CTA count (at most one per block) and
  // the pieces' layout in the workspace follow from it
  DecodeParams p = p_in;
  p.blocks_per_head = (p.Nk + KtCfg<D>::kBK - 1) / KtCfg<D>::kBK;
  const long long blocks = static_cast<long long>(p.BH) * p.blocks_per_head;
  if (p.n_ctas > blocks) p.n_ctas = static_cast<int>(blocks);
  p.ws_lse = p.ws_o + static_cast<size_t>(p.n_ctas + p.BH) * p.Nq * D;
  decode_kt_kernel<D><<<p.n_ctas, kKtThreads, KtCfg<D>::kSmemBytes, s>>>(p);
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
