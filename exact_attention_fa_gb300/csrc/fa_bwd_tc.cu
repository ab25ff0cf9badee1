// Backward by recomputation on the tcgen05 tensor cores.
//
// The forward keeps only O and the row statistic lse; the backward rebuilds S and P tile by tile
// ("3 · FlashAttention", 3.4; "FlashAttention：在线 softmax 与 IO-aware 注意力", section 五) and
// applies softmax calculus:
//     P = exp(scale * Q K^T - lse),  dV = P^T dO,  dP = dO V^T,  D_i = sum_k dO_ik O_ik,
//     dS = P * (dP - D),  dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Kernel 1 (prep): per row, D_i and lse2_i = lse_i * log2(e) into the workspace (padded to whole
// 128-row tiles: +inf / 0 on padding rows so that they contribute nothing); the work counters
// and the dQ rows of the first head group zeroed.
//
// Kernel 2 (main), one CTA per (128-key tile j, head), 16 warps. Heads are taken in groups whose
// inputs fit in L2. At d = 128 the prep kernel zeroes the dQ rows of the first groups, as many as
// about 40 MB of dQ allows; after those, the CTAs of group g zero the rows of group g + 1 when
// they start, and a CTA of group g + 1 adds into dQ only once all of them have. Zeros are thus
// written shortly before they are used, while they are still in L2 (zeroing all of a large dQ up
// front wrote it to DRAM and read most of it back). Work items are then handed out in CTA start
// order through a counter, so the CTAs a CTA waits for have all started before it. At d = 64 the
// prep kernel zeroes all of dQ.
//   * warps 12-15 (d = 128) first zero this CTA's share of the next group's dQ rows;
//   * warp 8 (one elected lane): TMA. K_j and V_j once; then per query tile i, Q_i, dO_i and the 128
//     lse2 / D values of that tile into a ring of stages;
//   * warp 9 (one elected lane): MMAs. S^T = K Q_i^T and dP^T = V dO_i^T (keys on TMEM lanes, queries on
//     columns); dV += P^T dO_i and dK += dS^T Q_i with P^T / dS^T read from TMEM; dQ_i from dS in
//     shared memory (d = 128: dQ_i^T = K^T dS^T, d on lanes; d = 64: dQ_i = dS K, queries on lanes);
//   * warps 0-7 (two warpgroups, one per half of the query columns): thread = key row. Computes
//     P^T = exp2(S^T * scale * log2e - lse2) (causal / tail masked), writes it as bf16 over S^T,
//     then dS^T = P^T * (dP^T - D) as bf16 over dP^T and, transposed by its layout, into the
//     shared-memory operand of the dQ product; at the end stores dV and scale * dK;
//   * warps 12-15: read dQ_i from TMEM and add scale * dQ_i into the fp32 output. d = 128: one
//     thread per column of dQ issues coalesced fp32 reductions from registers; d = 64: the tile is
//     staged in the ring stage and added by TMA bulk reductions. Warps 10-11 only complete the
//     producer / MMA warpgroup, which hands registers to the drain warpgroup.
// TMEM columns: S^T [0,128), dP^T [128,256) (at d = 128 dQ_i^T reuses it after dS^T was consumed),
// dV [256, 256+d), dK [256+d, 256+2d) (d = 64: dQ_i at [384, 448)).
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int BT = 128;  // keys per CTA tile = queries per inner tile
constexpr int kComputeWarps = 8;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kDrainWarp0 = 12;  // warps 12-15; warps 10 and 11 only complete the warpgroup
constexpr int kThreads = 16 * 32;
// Registers per thread after the warpgroups re-balance the 128 each is launched with (per head
// dimension, in BCfg): the producer / MMA warpgroup gives some up; at d = 128 the dQ drain holds a
// whole 128-column row of dQ^T, at d = 64 it only stages 32 columns at a time and the compute
// warpgroups take the difference.

constexpr int kBoxBytes = 128 * 64 * 2;
constexpr int kMaxMaskTiles = kBwdMaxMaskTiles;  // block-sparse: query tiles the bitmask holds

// The query tiles a CTA (key tile j) visits, in order: [first, n_tiles) (first = j when causal),
// and with a tile mask (kMask, a separate kernel instance) only those whose mask entry M[i][j] is
// set. The mask column is turned into a bitmask in shared memory once per CTA, so each role's
// next() is a few integer operations; without a mask it is the identity.
template <bool kMask>
struct QueryPlan {
  const uint32_t* bits;  // shared memory (kMask)
  int first, n_tiles;
  __device__ __forceinline__ int next(int i) const {
    if constexpr (!kMask) return i;
    while (i < n_tiles) {
      const uint32_t w = bits[i >> 5] >> (i & 31);
      if (w) return i + __ffs(w) - 1;
      i = (i | 31) + 1;
    }
    return n_tiles;
  }
  __device__ __forceinline__ int begin() const { return next(first); }
};

template <int D>
struct BCfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kStages = D == 128 ? 2 : 3;
  // d = 64 folds the row statistics into the S^T and dP^T products: one more K-step of 16 whose
  // A operand is a constant tile of ones (columns 0-2) and whose B operand holds -lse2/scale_log2
  // (for S^T) or -D (for dP^T) split into three bf16 parts, so that the products come out as
  // scale_log2^-1 * (S scaled - lse2) and dP - D and the compute warps read no statistics from
  // shared memory. d = 128 has no shared memory left for the operand tiles and reads lse2 / D.
  static constexpr bool kAugStats = D == 64;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffDS = 2 * kTileBytes;           // 128 x 128 bf16, two 64-query boxes
  static constexpr int kOffStage = kOffDS + 2 * kBoxBytes;
  // per stage: Q_i, dO_i, then lse2[128], D[128] (d = 128) or the two 4 KB operand tiles (d = 64)
  static constexpr int kStageQ = 0;
  static constexpr int kStageDO = kTileBytes;
  static constexpr int kStageLse = 2 * kTileBytes;
  static constexpr int kStageD = 2 * kTileBytes + 512;
  static constexpr int kStageQAug = 2 * kTileBytes;
  static constexpr int kStageDOAug = 2 * kTileBytes + 4096;
  static constexpr int kStageBytes = 2 * kTileBytes + (kAugStats ? 8192 : 1024);
  // d = 128 computes dQ_i^T = K^T dS^T (d on TMEM lanes, queries on columns): a warp then holds
  // 32 consecutive d of one query row, so the drain adds it into the fp32 output with coalesced
  // reductions straight from registers. d = 64 computes dQ_i (queries on lanes) and stages it
  // (128-byte-swizzled fp32 boxes of 64 rows x 32 columns, 32 KB) in its own buffer for TMA bulk
  // reductions. Either way the ring stage is free as soon as the MMAs have read Q_i and dO_i.
  static constexpr bool kDQTransposed = D == 128;
  // d = 128: the main kernel zeroes dQ rows itself, one head group ahead, past the groups the
  // prep kernel zeroes; d = 64 (whose dQ rows are half the size) leaves all of it to the prep
  // kernel: measured, the in-kernel form cost the d = 64 kernel 5% and saved it no time.
  static constexpr bool kZeroInKernel = D == 128;
  static constexpr int kOffDQStage = kOffStage + kStages * kStageBytes;
  static constexpr int kDQStageBytes = kDQTransposed ? 0 : 128 * D * 4;
  static constexpr int kOffOnes = kOffDQStage + kDQStageBytes;  // 4 KB constant A tile (d = 64)
  static constexpr int kOffBar = kOffOnes + (kAugStats ? 4096 : 0);
  // d = 128: a stage fills in two halves with barriers of their own, Q_i (+ lse2_i) first, so
  // that S^T of the next query tile waits for half the bytes (measured +3.7%; at d = 64, with
  // three stages, one barrier per stage measured 2% faster).
  static constexpr bool kSplitFull = D == 128;
  static constexpr int kBarKV = 0;
  static constexpr int kBarFull = 1;  // Q_i and lse2_i (or its operand tile); d = 64: the stage
  static constexpr int kBarFullDO = kSplitFull ? 1 + kStages : kBarFull;  // dO_i and D_i
  static constexpr int kBarEmpty = 1 + 2 * kStages;
  static constexpr int kBarS = 1 + 3 * kStages;
  static constexpr int kBarDP = kBarS + 1;
  static constexpr int kBarP = kBarS + 2;
  static constexpr int kBarDS = kBarS + 3;
  static constexpr int kBarDQFull = kBarS + 4;
  static constexpr int kBarDQEmpty = kBarS + 5;
  static constexpr int kBarAcc = kBarS + 6;
  static constexpr int kBarDrain = kBarS + 7;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemPtr = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemPtr + 4;
  static constexpr int kOffTicket = kOffAbort + 4;  // this CTA's work item
  static constexpr int kOffQMask = kOffAbort + 12;  // block-sparse: query tiles to visit (bits)
  static constexpr int kSmemBytes = kOffQMask + kMaxMaskTiles / 8;  // base 1024-aligned (checked)
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  // d = 64 has room for dQ_i in its own columns; at d = 128 it reuses the dP^T columns.
  static constexpr bool kDQAliasesDP = D == 128;
  static constexpr uint32_t kColDQ = kDQAliasesDP ? kColDP : 256 + 2 * D;
  // d = 64 also has room for dS^T (bf16 pairs, 64 columns) outside the dP^T columns, so dP^T of
  // the next query tile can be computed while dK still reads this tile's dS^T. d = 128 packs
  // dS^T over the dP^T columns it was computed from.
  static constexpr bool kSepDS = D == 64;
  static constexpr uint32_t kColDST = kSepDS ? 256 + 3 * D : kColDP;
  static constexpr int kRegsCompute = D == 128 ? 128 : 152;
  static constexpr int kRegsLoadMma = D == 128 ? 104 : 96;
  static constexpr int kRegsDrain = D == 128 ? 144 : 96;
  static_assert(2 * 128 * kRegsCompute + 128 * kRegsLoadMma + 128 * kRegsDrain <= 65536,
                "register split exceeds the launch's 512 x 128 registers");
};

// Work item -> (head, key tile). Heads in L2-sized groups of `group`; inside a group the key
// tiles with the most query tiles to visit (causal: the first ones) come first.
struct BwdItem {
  int bh, j;
  int g, within;  // head group, index of the item within its group
};
__device__ __forceinline__ BwdItem decode_bwd(const BwdParams& p, int group, int item) {
  BwdItem w;
  const int per_group = group * p.n_tiles;
  w.g = item / per_group;
  w.within = item - w.g * per_group;
  const int gsize = min(group, p.BH - w.g * group);
  w.j = w.within / gsize;
  w.bh = w.g * group + w.within % gsize;
  return w;
}

// L2 cache policies: O and dO are read once by the prep kernel (evict first); zeroed dQ rows are
// written to be kept (evict last), so that the main kernel's reductions find them in L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint4 ld_evict_first(const __nv_bfloat16* ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}
__device__ __forceinline__ void st_zero_evict_last(float* ptr, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %1, %1, %1}, %2;" ::"l"(ptr), "f"(0.f),
               "l"(pol)
               : "memory");
}

// The dQ drain warpgroup (warps 12-15), at its start: unless the prep kernel zeroes it (groups
// below zgroups), zero this CTA's share of the dQ rows of head group g + 1 (the group's rows split
// evenly over its CTAs, 16 bytes per store), then count the share done. The counter is raised
// after a barrier of the four warps and a fence, so the stores of all 128 threads are visible at
// gpu scope before it moves.
template <int D>
__device__ void zero_next_group(const BwdParams& p, int group, int zgroups, const BwdItem& w) {
  const int n_groups = (p.BH + group - 1) / group;
  if (w.g + 1 < zgroups || w.g + 1 >= n_groups) return;
  const int t = static_cast<int>(threadIdx.x) - kDrainWarp0 * 32;
  const long long ncta = static_cast<long long>(min(group, p.BH - w.g * group)) * p.n_tiles;
  const int next = min(group, p.BH - (w.g + 1) * group);
  const long long units = static_cast<long long>(next) * p.N * (D / 4);  // float4 units
  const long long u0 = units * w.within / ncta, u1 = units * (w.within + 1) / ncta;
  float* base = p.dq + static_cast<size_t>(w.g + 1) * group * p.N * D;
  const uint64_t pol = l2_policy_evict_last();
  for (long long u = u0 + t; u < u1; u += 128) st_zero_evict_last(base + 4 * u, pol);
  bar_sync(1, 128);
  if (t == 0) {
    __threadfence();
    atomicAdd(p.ctr + 1 + w.g + 1, 1u);
  }
}

// Before any reduction into dQ (right after its own zeroing, while the first dQ_i is still being
// computed), the drain of a CTA of head group g >= zgroups waits until every CTA of group g - 1
// has zeroed its share of group g's rows (the prep kernel zeroes the groups below zgroups). Those
// CTAs took earlier work items, so they have started, and each zeroes before anything else it
// does: the wait ends unless a CTA failed. One thread waits; the caller's barrier of the four
// drain warps orders the others' reductions after it.
__device__ __forceinline__ bool wait_group_zeroed(const BwdParams& p, const Ctl& ctl, int group,
                                                  int zgroups, const BwdItem& w) {
  if (w.g < zgroups || threadIdx.x != kDrainWarp0 * 32) return true;
  if (!wait_counter_geq(p.ctr + 1 + w.g, static_cast<unsigned>(group * p.n_tiles), ctl))
    return false;
  __threadfence();
  return true;
}

// P^T / dS^T as the TMEM operand of dV / dK: the warpgroup owning query columns [64c, 64c+64)
// packs them as bf16 pairs into columns [64c, 64c+32), so K-step k (queries 16k .. 16k+15) reads
// the 8 columns at k < 4 ? 8k : 64 + 8(k - 4) (mma_ts_k128_halves).

template <int D, class Plan>
__device__ void bwd_producer(const BwdParams& p, uint32_t sbase, const Ctl& ctl, int bh, int j,
                             const Plan& plan, int npad) {
  using C = BCfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);
  tma_prefetch_desc(&p.tm_do);
  mbar_arrive_expect_tx(bar(C::kBarKV), 2 * C::kTileBytes);
  for (int b = 0; b < D / 64; ++b) {
    tma_load_3d(sbase + C::kOffK + b * kBoxBytes, &p.tm_k, bar(C::kBarKV), b * 64, j * BT, bh);
    tma_load_3d(sbase + C::kOffV + b * kBoxBytes, &p.tm_v, bar(C::kBarKV), b * 64, j * BT, bh);
  }
  int issued[C::kStages];
#pragma unroll
  for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
  bool ok = true;
  for (int i = plan.begin(), it = 0; i < p.n_tiles; i = plan.next(i + 1), ++it) {
    const int st = it % C::kStages;
    const int round = it / C::kStages;
    if (!mbar_wait_warp(bar(C::kBarEmpty + st), (round & 1) ^ 1, ctl)) { ok = false; break; }
    const uint32_t sb = sbase + C::kOffStage + st * C::kStageBytes;
    constexpr uint32_t kStatBytes = 512;  // one fp32 statistic row (split stages only, d = 128)
    const uint32_t fq = bar(C::kBarFull + st), fd = bar(C::kBarFullDO + st);
    const uint8_t* aug = p.aug + (static_cast<size_t>(bh) * p.n_tiles + i) * 8192;
    const size_t r0 = static_cast<size_t>(bh) * npad + static_cast<size_t>(i) * BT;
    mbar_arrive_expect_tx(fq, C::kSplitFull ? C::kTileBytes + kStatBytes : C::kStageBytes);
    for (int b = 0; b < D / 64; ++b)
      tma_load_3d(sb + C::kStageQ + b * kBoxBytes, &p.tm_q, fq, b * 64, i * BT, bh);
    if constexpr (C::kAugStats)
      tma_bulk_g2s(sb + C::kStageQAug, aug, 8192, fq);  // both operand tiles (one barrier)
    else
      tma_bulk_g2s(sb + C::kStageLse, p.lse2 + r0, 512, fq);
    if constexpr (C::kSplitFull) mbar_arrive_expect_tx(fd, C::kTileBytes + kStatBytes);
    for (int b = 0; b < D / 64; ++b)
      tma_load_3d(sb + C::kStageDO + b * kBoxBytes, &p.tm_do, fd, b * 64, i * BT, bh);
    if constexpr (!C::kAugStats) tma_bulk_g2s(sb + C::kStageD, p.Dsum + r0, 512, fd);
    issued[st] = round;
  }
  if (!ok) {
    Ctl drain = ctl;
    int zero = 0;
    drain.abort_flag = &zero;
    mbar_wait_warp(bar(C::kBarKV), 0, drain);
    for (int s = 0; s < C::kStages; ++s)
      if (issued[s] >= 0) {
        mbar_wait_warp(bar(C::kBarFull + s), issued[s] & 1, drain);
        if (C::kSplitFull) mbar_wait_warp(bar(C::kBarFullDO + s), issued[s] & 1, drain);
      }
  }
}

template <int D, class Plan>
__device__ void bwd_mma(const BwdParams& p, uint32_t sbase, uint32_t tmem, const Ctl& ctl,
                        const Plan& plan) {
  using C = BCfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  constexpr uint32_t kIdescT = idesc_bf16(128, 128, 0, 0);  // S^T, dP^T: both K-major
  constexpr uint32_t kIdescG = idesc_bf16(128, D, 0, 1);    // dV, dK: A in TMEM, B MN-major
  constexpr uint32_t kIdescQ = idesc_bf16(128, D, 1, 1);    // dQ: A = dS MN-major, B = K MN-major
  constexpr uint32_t kIdescQT = idesc_bf16(D, 128, 1, 1);   // dQ^T: A = K MN-major, B = dS MN-major

  bool ok = mbar_wait_poll_warp(bar(C::kBarKV), 0, ctl);
  tc_fence_after();
  // Descriptors precomputed once; each MMA only adds a constant K-step offset (lean issue: the
  // MMA warp shares its SM sub-partition with busy compute warps).
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  constexpr int kSteps = D / 16;
  uint64_t a_k[kSteps], a_v[kSteps];  // K, V as the K-major A operand of S^T / dP^T per K-step
#pragma unroll
  for (int k = 0; k < kSteps; ++k) {
    const uint32_t off = (k / 4) * kBoxBytes + (k % 4) * 32;
    a_k[k] = sdesc64(sdesc_lo(sbase + C::kOffK + off, 16), kHi);
    a_v[k] = sdesc64(sdesc_lo(sbase + C::kOffV + off, 16), kHi);
  }
  const uint64_t k_mn = sdesc64(sdesc_lo(sbase + C::kOffK, kBoxBytes), kHi);    // K, MN-major
  const uint64_t ds_mn = sdesc64(sdesc_lo(sbase + C::kOffDS, kBoxBytes), kHi);  // dS, MN-major
  const uint64_t st_km = sdesc64(sdesc_lo(sbase + C::kOffStage, 16), kHi);       // Q_i / dO_i
  const uint64_t st_mn = sdesc64(sdesc_lo(sbase + C::kOffStage, kBoxBytes), kHi);
  constexpr uint64_t kStageStep = C::kStageBytes >> 4;
  constexpr uint64_t kDOOff = C::kStageDO >> 4;
  const uint32_t tS = tmem + C::kColS, tDP = tmem + C::kColDP, tDQ = tmem + C::kColDQ;
  const uint32_t tDV = tmem + C::kColDV, tDK = tmem + C::kColDK;
  auto qk = [&](uint32_t d_tmem, const uint64_t (&a)[kSteps], uint64_t b) {
    if constexpr (D == 128)
      mma_qk_d128(d_tmem, a, b, kIdescT);
    else
      mma_qk_d64(d_tmem, a, b, kIdescT);
  };
  const uint64_t ones = sdesc_none(sbase + C::kOffOnes, 128, 256);
  auto aug_desc = [&](int it, int which) {  // the statistics tile of query tile `it`
    return sdesc_none(sbase + C::kOffStage + (it % C::kStages) * C::kStageBytes +
                          (which ? C::kStageDOAug : C::kStageQAug), 128, 256);
  };
  auto issue_s = [&](int it) {  // S^T = K Q_i^T (d = 64: minus lse2 / scale_log2)
    qk(tS, a_k, st_km + (it % C::kStages) * kStageStep);
    if constexpr (C::kAugStats) mma_ss(tS, ones, aug_desc(it, 0), kIdescT, 1u);
    mma_commit(bar(C::kBarS));
  };
  // dP^T = V dO_i^T. At d = 64 (dQ and dS^T have TMEM columns of their own) dP^T of the next
  // query tile is issued as soon as the compute warps have read this one, so that they find it
  // ready when they finish P^T; at d = 128 (dQ_i^T reuses the columns) only after dQ_i^T was
  // drained.
  constexpr bool kEarlyDP = !C::kDQAliasesDP;
  auto issue_dp = [&](int it) {  // (d = 64: minus D); false if the wait for dO_i gave up
    // (with one barrier per stage, S^T of this tile has already waited for the whole stage)
    if (C::kSplitFull) {
      if (!mbar_wait_poll_warp(bar(C::kBarFullDO + it % C::kStages), (it / C::kStages) & 1, ctl))
        return false;
      tc_fence_after();
    }
    qk(tDP, a_v, st_km + (it % C::kStages) * kStageStep + kDOOff);
    if constexpr (C::kAugStats) mma_ss(tDP, ones, aug_desc(it, 1), kIdescT, 1u);
    mma_commit(bar(C::kBarDP));
    return true;
  };
  const int ibeg = plan.begin();
  if (ok && ibeg < p.n_tiles) {
    ok = mbar_wait_poll_warp(bar(C::kBarFull + 0), 0, ctl);
    tc_fence_after();
    if (ok) {
      issue_s(0);
      if (kEarlyDP) ok = issue_dp(0);
    }
  }
  const int n_tiles = p.n_tiles;
  for (int i = ibeg, it = 0; ok && i < n_tiles; i = plan.next(i + 1), ++it) {
    const int st = it % C::kStages;
    const uint64_t q_mn = st_mn + st * kStageStep;
    const uint64_t do_mn = q_mn + kDOOff;
    if (!kEarlyDP) {
      if (it > 0) {
        if (!mbar_wait_poll_warp(bar(C::kBarDQEmpty), (it - 1) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
      }
      if (!issue_dp(it)) { ok = false; break; }
    }
    // dV += P^T dO_i
    if (!mbar_wait_poll_warp(bar(C::kBarP), it & 1, ctl)) { ok = false; break; }
    tc_fence_after();
    mma_ts_k128_halves(tDV, tS, do_mn, kIdescG, it > 0 ? 1u : 0u);
    // S^T of the next query tile overwrites P^T: the tensor core runs MMAs in issue order, so
    // the dV product above has read P^T first; the compute warps overlap it with dK, dQ below.
    const bool has_next = plan.next(i + 1) < n_tiles;
    if (has_next) {
      const int nx = it + 1;
      if (!mbar_wait_poll_warp(bar(C::kBarFull + nx % C::kStages), (nx / C::kStages) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      issue_s(nx);
    }
    // dK += dS^T Q_i ; dQ_i = dS K
    if (!mbar_wait_poll_warp(bar(C::kBarDS), it & 1, ctl)) { ok = false; break; }
    tc_fence_after();
    if constexpr (C::kSepDS) {
      // dP^T of the next tile right away (its columns were read before the compute warps
      // signalled dS); dS^T has columns of its own, 8 per K-step in order.
      if (has_next && !issue_dp(it + 1)) { ok = false; break; }
      mma_pv_k128(tDK, tmem + C::kColDST, q_mn, kIdescG, it > 0 ? 1u : 0u);
    } else {
      mma_ts_k128_halves(tDK, tDP, q_mn, kIdescG, it > 0 ? 1u : 0u);
    }
    if (!C::kDQAliasesDP && it > 0) {
      if (!mbar_wait_poll_warp(bar(C::kBarDQEmpty), (it - 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
    }
    if (C::kDQTransposed)
      mma_ss_k128_mn(tDQ, k_mn, ds_mn, kIdescQT);  // dQ_i^T = K^T dS^T
    else
      mma_ss_k128_mn(tDQ, ds_mn, k_mn, kIdescQ);   // dQ_i = dS K
    mma_commit(bar(C::kBarDQFull));
    mma_commit(bar(C::kBarEmpty + st));  // Q_i, dO_i (and its lse2, D rows) are no longer read
    // (d = 64: dP^T of the next tile was issued above; the compute warps wait for this tile's
    // dQ product before they rewrite the dS tile and dS^T.)
  }
  if (ok) {
    mma_commit(bar(C::kBarAcc));
  } else {
    Ctl drain = ctl;
    int zero = 0;
    drain.abort_flag = &zero;
    mma_commit(bar(C::kBarDrain));
    mbar_wait_poll_warp(bar(C::kBarDrain), 0, drain);
  }
}

// P^T for one compute thread's 64 query columns of its key row, in two 32-column chunks: scores
// from TMEM, exp2(S * scale * log2e - lse2) with the row statistics read four at a time from
// shared memory and the arithmetic on packed fp32 pairs; P kept in pv (fp32) for dS and written
// back as packed bf16 over the first 32 of the 64 score columns. kMasked: columns x < lim are 0.
template <bool kMasked, bool kAug>
__device__ __forceinline__ void bwd_p_tile(uint32_t tS, const float4* lse4, unsigned long long k2,
                                           int lim, float (&pv)[64]) {
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    uint32_t s[32];
    tmem_ld32(tS + 32 * ch, s);
    uint32_t pk[16];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int x0 = 32 * ch + 4 * u;
      float a0, a1, a2, a3;
      if constexpr (kAug) {  // the scores already carry -lse2 / scale_log2
        f2_unpack(f2_mul(f2_pack(__uint_as_float(s[4 * u]), __uint_as_float(s[4 * u + 1])), k2),
                  a0, a1);
        f2_unpack(f2_mul(f2_pack(__uint_as_float(s[4 * u + 2]), __uint_as_float(s[4 * u + 3])), k2),
                  a2, a3);
      } else {
        const float4 L = lse4[8 * ch + u];
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * u]), __uint_as_float(s[4 * u + 1])), k2,
                         f2_pack(-L.x, -L.y)), a0, a1);
        f2_unpack(f2_fma(f2_pack(__uint_as_float(s[4 * u + 2]), __uint_as_float(s[4 * u + 3])), k2,
                         f2_pack(-L.z, -L.w)), a2, a3);
      }
      float p0 = ex2(a0), p1 = ex2(a1), p2 = ex2(a2), p3 = ex2(a3);
      if constexpr (kMasked) {
        p0 = x0 < lim ? 0.f : p0;
        p1 = x0 + 1 < lim ? 0.f : p1;
        p2 = x0 + 2 < lim ? 0.f : p2;
        p3 = x0 + 3 < lim ? 0.f : p3;
      }
      pv[x0] = p0;
      pv[x0 + 1] = p1;
      pv[x0 + 2] = p2;
      pv[x0 + 3] = p3;
      pk[2 * u] = pack_bf16(p0, p1);
      pk[2 * u + 1] = pack_bf16(p2, p3);
    }
    tmem_st16(tS + 16 * ch, pk);
  }
}

template <int D, class Plan>
__device__ void bwd_compute(const BwdParams& p, uint32_t sbase, uint8_t* smem, uint32_t tmem,
                            const Ctl& ctl, int bh, int j, const Plan& plan) {
  using C = BCfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int half = warp / 4;  // query columns [64*half, 64*half + 64)
  const int quad = warp % 4;
  const int r = quad * 32 + lane;  // key row within the tile (TMEM lane)
  const int key = j * BT + r;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::kColS + 64 * half;
  const uint32_t tDP = tmem + lane_off + C::kColDP + 64 * half;
  const uint32_t tDST = tmem + lane_off + C::kColDST + (C::kSepDS ? 32 : 64) * half;
  const float sl2 = p.scale_log2;
  uint8_t* ds_row = smem + C::kOffDS + half * kBoxBytes + r * 128;

  bool ok = true;
  int n_done = 0;  // query tiles processed
  for (int i = plan.begin(), it = 0; i < p.n_tiles; i = plan.next(i + 1), ++it) {
    n_done = it + 1;
    const int st = it % C::kStages;
    const float* lse2 = reinterpret_cast<const float*>(smem + C::kOffStage + st * C::kStageBytes +
                                                       C::kStageLse) + 64 * half;
    const float* dsum = reinterpret_cast<const float*>(smem + C::kOffStage + st * C::kStageBytes +
                                                       C::kStageD) + 64 * half;
    if (!mbar_wait(bar(C::kBarFull + st), (it / C::kStages) & 1, ctl)) { ok = false; break; }
    if (!mbar_wait(bar(C::kBarS), it & 1, ctl)) { ok = false; break; }
    tc_fence_after();
    // queries of this thread's columns: q = i*128 + 64*half + x; allowed iff key <= q (causal)
    // and key < N
    int lim;  // number of leading columns x whose P is forced to zero
    if (key >= p.N) lim = 64;
    else if (p.causal && i == j) lim = min(64, max(0, r - 64 * half));
    else lim = 0;

    // P^T = exp2(S^T * scale * log2e - lse2) in two 32-column chunks: row statistics read four at
    // a time, arithmetic on packed fp32 pairs. At d = 64 the mask (diagonal tile, padding keys) is
    // applied only by warps that have masked entries.
    const float4* lse4 = reinterpret_cast<const float4*>(lse2);
    const unsigned long long k2 = f2_pack(sl2, sl2);
    float pv[64];
    if constexpr (D == 64) {
      if (__any_sync(0xffffffffu, lim > 0))
        bwd_p_tile<true, C::kAugStats>(tS, lse4, k2, lim, pv);
      else
        bwd_p_tile<false, C::kAugStats>(tS, lse4, k2, lim, pv);
    } else {
      // a single code path measured faster at d = 128
      bwd_p_tile<true, C::kAugStats>(tS, lse4, k2, lim, pv);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar(C::kBarP));

    if (!mbar_wait(bar(C::kBarDP), it & 1, ctl)) { ok = false; break; }
    if (!C::kAugStats && !mbar_wait(bar(C::kBarFullDO + st), (it / C::kStages) & 1, ctl)) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (C::kSepDS && it > 0) {
      // dP^T of this tile may have been computed before the previous tile's dK / dQ products
      // read the dS tile (shared memory) and dS^T (TMEM): wait for them before rewriting both.
      if (!mbar_wait(bar(C::kBarDQFull), (it - 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
    }
    const float4* d4 = reinterpret_cast<const float4*>(dsum);
#pragma unroll
    for (int ch = 0; ch < 2; ++ch) {
      uint32_t dp[32];
      tmem_ld32(tDP + 32 * ch, dp);
      uint32_t pk[16];
#pragma unroll
      for (int u = 0; u < 8; ++u) {  // dS = P * (dP - D)
        const int x0 = 32 * ch + 4 * u;
        float d0, d1, d2, d3;
        if constexpr (C::kAugStats) {  // the product already carries -D
          f2_unpack(f2_mul(f2_pack(pv[x0], pv[x0 + 1]),
                           f2_pack(__uint_as_float(dp[4 * u]), __uint_as_float(dp[4 * u + 1]))),
                    d0, d1);
          f2_unpack(f2_mul(f2_pack(pv[x0 + 2], pv[x0 + 3]),
                           f2_pack(__uint_as_float(dp[4 * u + 2]), __uint_as_float(dp[4 * u + 3]))),
                    d2, d3);
        } else {
          const float4 Dv = d4[8 * ch + u];
          f2_unpack(f2_mul(f2_pack(pv[x0], pv[x0 + 1]),
                           f2_add(f2_pack(__uint_as_float(dp[4 * u]), __uint_as_float(dp[4 * u + 1])),
                                  f2_pack(-Dv.x, -Dv.y))), d0, d1);
          f2_unpack(f2_mul(f2_pack(pv[x0 + 2], pv[x0 + 3]),
                           f2_add(f2_pack(__uint_as_float(dp[4 * u + 2]), __uint_as_float(dp[4 * u + 3])),
                                  f2_pack(-Dv.z, -Dv.w))), d2, d3);
        }
        pk[2 * u] = pack_bf16(d0, d1);
        pk[2 * u + 1] = pack_bf16(d2, d3);
      }
      tmem_st16(tDST + 16 * ch, pk);
      // dS (queries contiguous per key row) into the 128-byte-swizzled MN-major operand
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int chunk = (4 * ch + u) ^ (r & 7);
        *reinterpret_cast<uint4*>(ds_row + chunk * 16) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      }
    }
    tmem_st_wait();
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(bar(C::kBarDS));
  }
  if (!ok) return;

  // epilogue: dV and scale * dK, this warpgroup's half of the d columns
  if (!mbar_wait(bar(C::kBarAcc), 0, ctl)) return;
  tc_fence_after();
  constexpr int kHalf = D / 2;
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const uint32_t col = (which ? C::kColDK : C::kColDV) + kHalf * half;
    const float mul = which ? p.scale : 1.f;
    __nv_bfloat16* out = (which ? p.dk : p.dv) + (static_cast<size_t>(bh) * p.N + key) * D + kHalf * half;
#pragma unroll 1
    for (int c = 0; c < kHalf; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + col + c, v);
      if (n_done == 0) {  // no query tile visits this key tile: dK = dV = 0 (TMEM never written)
#pragma unroll
        for (int u = 0; u < 32; ++u) v[u] = 0u;
      }
      if (key < p.N) {
        uint4* dst = reinterpret_cast<uint4*>(out + c);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(v[8 * u + 0]) * mul, __uint_as_float(v[8 * u + 1]) * mul);
          w.y = pack_bf16(__uint_as_float(v[8 * u + 2]) * mul, __uint_as_float(v[8 * u + 3]) * mul);
          w.z = pack_bf16(__uint_as_float(v[8 * u + 4]) * mul, __uint_as_float(v[8 * u + 5]) * mul);
          w.w = pack_bf16(__uint_as_float(v[8 * u + 6]) * mul, __uint_as_float(v[8 * u + 7]) * mul);
          dst[u] = w;
        }
      }
    }
  }
}

// dQ_i (TMEM, thread = query row) -> scale -> swizzled fp32 staging tile in shared memory ->
// bulk tensor reduction into the fp32 output (coalesced adds at L2, done by the TMA unit). The
// TMEM columns are handed back as soon as they are read, the staging tile once the TMA has read it.
template <int D, class Plan>
__device__ void bwd_drain(const BwdParams& p, uint32_t sbase, uint8_t* smem, uint32_t tmem,
                          const Ctl& ctl, int bh, const Plan& plan) {
  using C = BCfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quad = warp % 4;
  const int qr = quad * 32 + lane;  // query row within the tile (TMEM lane)
  const bool issuer = warp == kDrainWarp0 && lane == 0;
  const uint32_t tQ = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kColDQ;
  constexpr uint32_t kBox = 64 * 128;       // one TMA box: 64 rows x 128 B
  constexpr uint32_t kColBox = 128 * 128;   // 32 columns of the 128 rows
  for (int i = plan.begin(), it = 0; i < p.n_tiles; i = plan.next(i + 1), ++it) {
    const bool bad = !mbar_wait(bar(C::kBarDQFull), it & 1, ctl);
    if (bar_red_or(1, 128, bad)) return;
    tc_fence_after();
    uint8_t* row = smem + C::kOffDQStage + qr * 128;
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
      uint32_t v[32];
      tmem_ld32(tQ + c, v);
      if (c + 32 == D) {  // every column read: the MMA warp may reuse them
        tc_fence_before();
        mbar_arrive(bar(C::kBarDQEmpty));
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        *reinterpret_cast<float4*>(row + (c / 32) * kColBox + ((u ^ (qr & 7)) << 4)) =
            make_float4(__uint_as_float(v[4 * u]) * p.scale, __uint_as_float(v[4 * u + 1]) * p.scale,
                        __uint_as_float(v[4 * u + 2]) * p.scale,
                        __uint_as_float(v[4 * u + 3]) * p.scale);
    }
    fence_proxy_async_smem();
    bar_sync(1, 128);
    if (issuer) {
      const uint32_t src = sbase + C::kOffDQStage;
      for (int b = 0; b < D / 32; ++b)
        for (int rb = 0; rb < 2; ++rb)
          tma_reduce_add_3d(&p.tm_dq, src + b * kColBox + rb * kBox, 32 * b, i * BT + rb * 64, bh);
      bulk_commit();
      bulk_wait_read_all();  // the staging buffer may be rewritten once every drain thread is past
                             // the barrier at the top of the next iteration
    }
  }
  if (issuer) bulk_wait_all();  // the reductions complete before the kernel ends
}

// The drain paces its reductions: after every FA_RED_PACE_GROUP of them the warp sleeps
// FA_RED_PACE_NS. Issued back to back they fill the SM's memory-instruction queue faster than the
// L2 takes them (~25 B/cycle per SM), and the compute warps' shared / tensor-memory accesses then
// wait behind them (their dS phase was measured 2.9x slower). 150 ns per 16 keeps a warp's 128
// reductions within ~1.2 us, well inside one query-tile iteration; 300 ns was already too slow.
#ifndef FA_RED_PACE_NS
#define FA_RED_PACE_NS 150
#endif
#ifndef FA_RED_PACE_GROUP
#define FA_RED_PACE_GROUP 16
#endif
__device__ __forceinline__ void red_add_f32(float* addr, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(addr), "f"(v) : "memory");
}

// dQ_i^T (TMEM, thread = column d of dQ, 128 query columns) -> scale -> fp32 reductions: for each
// query a warp adds 32 consecutive floats (128 bytes, one coalesced request). The TMEM columns are
// handed back right after the single load, before the reductions are issued.
template <int D, class Plan>
__device__ void bwd_drain_transposed(const BwdParams& p, uint32_t sbase, uint32_t tmem,
                                     const Ctl& ctl, int bh, const Plan& plan) {
  using C = BCfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int quad = warp % 4;
  const int dcol = quad * 32 + lane;  // column of dQ (TMEM lane)
  const uint32_t tQ = tmem + (static_cast<uint32_t>(quad * 32) << 16) + C::kColDQ;
  const float scale = p.scale;
  for (int i = plan.begin(), it = 0; i < p.n_tiles; i = plan.next(i + 1), ++it) {
    const bool bad = !mbar_wait(bar(C::kBarDQFull), it & 1, ctl);
    if (bar_red_or(1, 128, bad)) return;
    tc_fence_after();
    uint32_t v[128];
    tmem_ld64x2(tQ, v);
    tc_fence_before();
    mbar_arrive(bar(C::kBarDQEmpty));
    float* dst = p.dq + (static_cast<size_t>(bh) * p.N + static_cast<size_t>(i) * BT) * D + dcol;
    const int nvalid = min(BT, p.N - i * BT);
    if (nvalid == BT) {
#pragma unroll
      for (int q = 0; q < BT; ++q) {
        red_add_f32(dst + q * D, __uint_as_float(v[q]) * scale);
#if FA_RED_PACE_NS > 0
        if ((q % FA_RED_PACE_GROUP) == FA_RED_PACE_GROUP - 1) __nanosleep(FA_RED_PACE_NS);
#endif
      }
    } else {
#pragma unroll
      for (int q = 0; q < BT; ++q)
        if (q < nvalid) red_add_f32(dst + q * D, __uint_as_float(v[q]) * scale);
    }
  }
}

template <int D, bool kMask>
__global__ void __launch_bounds__(kThreads, 1) bwd_tc_kernel(const __grid_constant__ BwdParams p,
                                                             int group, int zgroups, int npad) {
  using C = BCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemPtr);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  if (sbase & 1023u) {  // swizzled operands need a 1 KB aligned base; report, never misread
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  const int warp = threadIdx.x / 32;
  // the work item: the next one in CTA start order
  // The work item: at d = 128 the next one in CTA start order (the dQ zeroing of later head
  // groups relies on it); at d = 64 the prep kernel zeroes all of dQ and the block index serves.
  int item = static_cast<int>(blockIdx.x);
  if constexpr (C::kZeroInKernel) {
    volatile int* ticket = reinterpret_cast<volatile int*>(smem + C::kOffTicket);
    if (threadIdx.x == 0) *ticket = static_cast<int>(atomicAdd(p.ctr, 1u));
    __syncthreads();
    item = *ticket;
  }
  const BwdItem w = decode_bwd(p, group, item);
  const int bh = w.bh, j = w.j;
  uint32_t* qbits = reinterpret_cast<uint32_t*>(smem + C::kOffQMask);
  const QueryPlan<kMask> plan{qbits, p.causal ? j : 0, p.n_tiles};
  if (kMask) {
    // column j of the tile mask -> bitmask of the query tiles to visit (one load per thread)
    for (int i0 = warp * 32; i0 < p.n_tiles; i0 += kThreads) {
      const int i = i0 + static_cast<int>(threadIdx.x % 32);
      const bool on = i < p.n_tiles && __ldg(p.block_mask + static_cast<size_t>(i) * p.n_tiles + j) != 0;
      const uint32_t w = __ballot_sync(0xffffffffu, on);
      if (threadIdx.x % 32 == 0) qbits[i0 / 32] = w;
    }
  }

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarKV), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      if (C::kSplitFull) mbar_init(bar(C::kBarFullDO + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    mbar_init(bar(C::kBarS), 1);
    mbar_init(bar(C::kBarDP), 1);
    mbar_init(bar(C::kBarP), kComputeWarps * 32);
    mbar_init(bar(C::kBarDS), kComputeWarps * 32);
    mbar_init(bar(C::kBarDQFull), 1);
    mbar_init(bar(C::kBarDQEmpty), 128);
    mbar_init(bar(C::kBarAcc), 1);
    mbar_init(bar(C::kBarDrain), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  if constexpr (C::kAugStats) {
    // the constant A tile of the statistics K-step: 128 rows of [1, 1, 1, 0 ... 0] (16 bf16) in
    // 8-row x 16-byte core matrices (the second core matrix of each row group is all zero)
    if (threadIdx.x < 256) {
      const int c = threadIdx.x;  // 16-byte chunk: row group c / 16, K half (c / 8) % 2, row c % 8
      const uint4 v = ((c / 8) % 2 == 0) ? make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u)
                                         : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + C::kOffOnes + (c / 16) * 256 + ((c / 8) % 2) * 128 +
                                (c % 8) * 16) = v;
      fence_proxy_async_smem();  // read by the tensor core (async proxy)
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < kComputeWarps) {
    if constexpr (C::kRegsCompute > 128) regs_inc<C::kRegsCompute>();
    bwd_compute<D>(p, sbase, smem, tmem, ctl, bh, j, plan);
  } else if (warp < kDrainWarp0) {
    regs_dec<C::kRegsLoadMma>();
    if (warp == kLoadWarp) {
      bwd_producer<D>(p, sbase, ctl, bh, j, plan, npad);  // whole warp: one elected lane issues
    } else if (warp == kMmaWarp) {
      bwd_mma<D>(p, sbase, tmem, ctl, plan);  // whole warp: one elected lane issues
    }
    __syncwarp();
  } else {
    if constexpr (C::kRegsDrain > 128)
      regs_inc<C::kRegsDrain>();
    else
      regs_dec<C::kRegsDrain>();
    if constexpr (C::kZeroInKernel) {
      // zero this CTA's share of the next group's dQ rows, then wait until this group's rows
      // are zero, before the first dQ_i is ready
      zero_next_group<D>(p, group, zgroups, w);
      if (!bar_red_or(1, 128, !wait_group_zeroed(p, ctl, group, zgroups, w)))
        bwd_drain_transposed<D>(p, sbase, tmem, ctl, bh, plan);
    } else {
      bwd_drain<D>(p, sbase, smem, tmem, ctl, bh, plan);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------------------------
// prep: D_i = sum_k dO_ik O_ik, lse2_i = lse_i * log2(e) (padding rows: D = 0, lse2 = +inf),
// the dQ rows of the first zgroups head groups (the main kernel's first zgroups * group heads)
// zeroed, and the main kernel's work counters zeroed. D / 8 threads per row, 8 elements each. The
// rows are walked from the last head to the first: the main kernel starts with the first heads,
// whose zeroed dQ rows (and D, lse2) are then the ones most recently written, still in L2.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __grid_constant__ BwdParams p, int npad,
                                                       int group, int zgroups) {
  constexpr int kTpr = D / 8;
  const long long rows_total = static_cast<long long>(p.BH) * npad;
  const long long total = rows_total * kTpr;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int lane = threadIdx.x % 32;
  const uint64_t pol_first = l2_policy_evict_first(), pol_last = l2_policy_evict_last();
  if (blockIdx.x == 0)
    for (int c = threadIdx.x; c < 1 + (p.BH + group - 1) / group; c += blockDim.x) p.ctr[c] = 0u;
  for (long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; t - lane < total;
       t += stride) {
    const bool valid = t < total;
    const long long row = rows_total - 1 - t / kTpr;
    const int part = static_cast<int>(t % kTpr);
    const int bh = static_cast<int>(row / npad);
    const int q = static_cast<int>(row % npad);
    float acc = 0.f;
    if (valid && q < p.N) {
      const size_t off = (static_cast<size_t>(bh) * p.N + q) * D + part * 8;
      const uint4 a = ld_evict_first(p.dO + off, pol_first);
      const uint4 b = ld_evict_first(p.o + off, pol_first);
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 x = __bfloat1622float2(a2[u]);
        const float2 y = __bfloat1622float2(b2[u]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
      if (bh < zgroups * group) {
        st_zero_evict_last(p.dq + off, pol_last);
        st_zero_evict_last(p.dq + off + 4, pol_last);
      }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(~0u, acc, off);
    if (valid && part == 0) {
      const bool in = q < p.N;
      p.Dsum[row] = in ? acc : 0.f;
      const float l2 = in ? p.lse[static_cast<size_t>(bh) * p.N + q] * 1.4426950408889634f : INFINITY;
      p.lse2[row] = l2;
      if constexpr (D == 64) {
        // the two 32-byte B-operand rows of the statistics K-step: -lse2 / scale_log2 and -D, each
        // as three bf16 parts (hi + lo + lo2 carries ~24 bits) in columns 0-2, zeros elsewhere;
        // row r of tile t sits in 8-row x 16-byte core matrices: (r / 8) * 256 + (r % 8) * 16
        const size_t tile = row / 128;
        const int r = static_cast<int>(row % 128);
        uint8_t* base = p.aug + tile * 8192 + (r / 8) * 256 + (r % 8) * 16;
        const float xs[2] = {-l2 / p.scale_log2, in ? -acc : 0.f};
#pragma unroll
        for (int w = 0; w < 2; ++w) {
          const float x = xs[w];
          const __nv_bfloat16 h = __float2bfloat16_rn(x);
          const bool fin = isfinite(x);
          const float rest = fin ? x - __bfloat162float(h) : 0.f;
          const __nv_bfloat16 lo = __float2bfloat16_rn(rest);
          const __nv_bfloat16 lo2 = __float2bfloat16_rn(fin ? rest - __bfloat162float(lo) : 0.f);
          const uint32_t w0 = static_cast<uint32_t>(__bfloat16_as_ushort(h)) |
                              (static_cast<uint32_t>(__bfloat16_as_ushort(lo)) << 16);
          const uint32_t w1 = static_cast<uint32_t>(__bfloat16_as_ushort(lo2));
          *reinterpret_cast<uint4*>(base + w * 4096) = make_uint4(w0, w1, 0u, 0u);
          *reinterpret_cast<uint4*>(base + w * 4096 + 128) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  }
}

template <int D>
cudaError_t configure_d() {
  for (auto k : {bwd_tc_kernel<D, false>, bwd_tc_kernel<D, true>}) {
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, BCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_d(const BwdParams& p, int num_sms, cudaStream_t s) {
  using C = BCfg<D>;
  const int npad = p.n_tiles * BT;
  const long long head_bytes = 4ll * p.N * D * 2;
  long long g = (32ll << 20) / head_bytes;
  const int group = static_cast<int>(g < 1 ? 1 : (g > p.BH ? p.BH : g));
  // head groups whose dQ rows the prep kernel zeroes: about 40 MB of dQ, which stays in L2 until
  // the main kernel's first groups use it (at least one group)
  const int n_groups = (p.BH + group - 1) / group;
  const long long group_dq_bytes = static_cast<long long>(group) * p.N * D * 4;
  const long long zg = C::kZeroInKernel ? (40ll << 20) / group_dq_bytes : n_groups;
  const int zgroups = static_cast<int>(zg < 1 ? 1 : (zg > n_groups ? n_groups : zg));
  bwd_prep_kernel<D><<<num_sms * 8, 256, 0, s>>>(p, npad, group, zgroups);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.n_tiles) * p.BH;
  if (grid > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  if (p.block_mask)
    bwd_tc_kernel<D, true><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, s>>>(
        p, group, zgroups, npad);
  else
    bwd_tc_kernel<D, false><<<static_cast<unsigned>(grid), kThreads, C::kSmemBytes, s>>>(
        p, group, zgroups, npad);
  return cudaGetLastError();
}

}  // namespace

cudaError_t configure_bwd() {
  const cudaError_t e = configure_d<64>();
  return e != cudaSuccess ? e : configure_d<128>();
}

cudaError_t launch_bwd(const BwdParams& p, int num_sms, cudaStream_t s) {
  if (p.d == 64) return launch_d<64>(p, num_sms, s);
  if (p.d == 128) return launch_d<128>(p, num_sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
