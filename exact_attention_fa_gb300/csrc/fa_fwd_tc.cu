// bf16 forward on the 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// The method is the tiled online-softmax attention of "FlashAttention：メモリ効率的なアテンション計算"
// (sections "オンライン softmax" and "タイル化") in the FlashAttention-2 order of
// "출력을 누적해 메모리 이동을 줄이는 FlashAttention": per query tile, stream the key/value tiles, keep a
// running row max m, running sum l and an unnormalised accumulator O rescaled by exp(m - m_new),
// divide by l once at the end. Neither S nor P ever leaves the SM.
//
// GB300 mapping (one CTA per SM, 6 warps, one 128-row query tile of one (b, h) per CTA; used for
// d = 128 and for block-sparse masks):
//   * warp 5 (one elected lane) streams K_j, V_j with TMA into a ring of 128-byte-swizzled
//     shared-memory stages guarded by full/empty mbarriers, keys two tiles ahead of values; Q is
//     loaded once;
//   * warp 4 (one elected lane) issues every tcgen05.mma. Issue blocks while the tensor pipe is
//     busy, so this warp does nothing else. S = Q K_j^T goes to one of two S buffers in TMEM, so the scores
//     of tile j + 1 are computed while the softmax works on tile j; O += P_j V_j reads P_j from
//     the S buffer it was written into (P aliased over S), after which that buffer takes
//     S_{j+2};
//   * warps 0-3 are the softmax warpgroup: thread r owns query row r (TMEM lane r). Per key tile
//     it loads its 128 scores, applies the scale (log2(e) folded in, exp2 on the SFU) and the
//     causal / tail mask, updates m and l, rescales its O row only when the reference max moves
//     (conditional rescaling), and writes P as bf16 over the S columns. At the end it writes
//     O / l and lse.
//   * causal / block-sparse: key tiles a query tile does not need are never loaded nor multiplied
//     ("3 · FlashAttention", question on the causal mask; "拡張: Block-Sparse FlashAttention").
// TMEM columns: O [0, d), S buffers [128, 256) and [256, 384).
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kThreads = 192;
constexpr int kBoxBytes = 128 * 64 * 2;  // one TMA box: 128 rows x 64 bf16 (128 B rows)
constexpr float kRescaleSlack = 8.f;     // log2 units: P stays <= 256

template <int D>
struct Cfg {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kStages = D == 128 ? 6 : 12;  // K/V ring
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  // barriers: Q, full[S], empty[S], s_full[2], p_full[2], pv_done, o_full, drain
  static constexpr int kBarQ = 0;
  static constexpr int kBarFull = 1;
  static constexpr int kBarEmpty = 1 + kStages;
  static constexpr int kBarS = 1 + 2 * kStages;
  static constexpr int kBarP = kBarS + 2;
  static constexpr int kBarPV = kBarP + 2;
  static constexpr int kBarO = kBarPV + 1;
  static constexpr int kBarDrain = kBarO + 1;
  static constexpr int kNumBars = kBarDrain + 1;
  static constexpr int kOffTmemPtr = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemPtr + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KB
  static constexpr uint32_t kColO = 0;
  __device__ static constexpr uint32_t col_s(int b) { return 128u + 128u * b; }
};

// Key tiles visited by this CTA's query tile, resolved once per role: key tiles [0, last] (last =
// the query tile itself when causal), of which block-sparse query tiles take those their row of
// the tile mask keeps. Kept in registers so that the per-tile bookkeeping stays a few integer compares.
struct TilePlan {
  const uint8_t* mask;  // block-sparse: the query tile's row of the tile mask, else null
  int last, n_tiles;
  // next key tile >= j this query tile needs, or n_tiles
  __device__ __forceinline__ int next(int j) const {
    if (mask == nullptr) return j <= last ? j : n_tiles;
    for (; j <= last; ++j)
      if (__ldg(mask + j) != 0) return j;
    return n_tiles;
  }
};

__device__ __forceinline__ TilePlan make_plan(const FwdParams& p, int qt) {
  TilePlan t;
  t.n_tiles = p.n_tiles;
  t.last = p.causal ? qt : p.n_tiles - 1;
  t.mask = p.block_mask ? p.block_mask + static_cast<size_t>(qt) * p.n_tiles : nullptr;
  return t;
}

// CTA -> (head, query tile). Heads are taken in groups small enough for their K/V to stay in
// L2; inside a group the query tiles with the most key tiles (causal: the last ones) come first.
__device__ __forceinline__ void decode_work(const FwdParams& p, int& bh, int& qt) {
  const int per_group = p.heads_per_group * p.n_tiles;
  const int g = blockIdx.x / per_group;
  const int within = blockIdx.x - g * per_group;
  const int gsize = min(p.heads_per_group, p.BH - g * p.heads_per_group);
  qt = p.n_tiles - 1 - within / gsize;
  bh = g * p.heads_per_group + within % gsize;
}

// Ring order shared by the producer and the MMA warp: K(u0), K(u1), then for each needed tile
// u_i: K(u_{i+2}) (if it exists), V(u_i).

// ---------------------------------------------------------------------------------------------
template <int D>
__device__ void producer(const FwdParams& p, uint32_t sbase, const Ctl& ctl, int bh, int qt) {
  using C = Cfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);

  mbar_arrive_expect_tx(bar(C::kBarQ), C::kTileBytes);
  for (int b = 0; b < D / 64; ++b)
    tma_load_3d(sbase + C::kOffQ + b * kBoxBytes, &p.tm_q, bar(C::kBarQ), b * 64, qt * BM, bh);

  int issued[C::kStages];
#pragma unroll
  for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
  int pos = 0;
  bool ok = true;
  auto load = [&](const void* map, int j) {
    const int s = pos % C::kStages;
    const int round = pos / C::kStages;
    if (!mbar_wait_warp(bar(C::kBarEmpty + s), (round & 1) ^ 1, ctl)) return false;
    mbar_arrive_expect_tx(bar(C::kBarFull + s), C::kTileBytes);
    for (int b = 0; b < D / 64; ++b)
      tma_load_3d(sbase + C::kOffKV + s * C::kTileBytes + b * kBoxBytes, map, bar(C::kBarFull + s),
                  b * 64, j * BN, bh);
    issued[s] = round;
    ++pos;
    return true;
  };
  const TilePlan plan = make_plan(p, qt);
  int j = plan.next(0);
  int j1 = j < p.n_tiles ? plan.next(j + 1) : p.n_tiles;
  if (j < p.n_tiles) ok = load(&p.tm_k, j);
  if (ok && j1 < p.n_tiles) ok = load(&p.tm_k, j1);
  while (ok && j < p.n_tiles) {
    const int j2 = j1 < p.n_tiles ? plan.next(j1 + 1) : p.n_tiles;
    if (j2 < p.n_tiles && !(ok = load(&p.tm_k, j2))) break;
    if (!(ok = load(&p.tm_v, j))) break;
    j = j1;
    j1 = j2;
  }
  if (!ok) {
    // Give the copies already in flight a bounded time to land before the CTA exits.
    Ctl drain = ctl;
    int zero = 0;
    drain.abort_flag = &zero;
    mbar_wait_warp(bar(C::kBarQ), 0, drain);
    for (int s = 0; s < C::kStages; ++s)
      if (issued[s] >= 0) mbar_wait_warp(bar(C::kBarFull + s), issued[s] & 1, drain);
  }
}

// ---------------------------------------------------------------------------------------------
template <int D>
__device__ void mma_issuer(const FwdParams& p, uint32_t sbase, uint32_t tmem, const Ctl& ctl,
                           int qt) {
  using C = Cfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  constexpr uint32_t kIdescQK = idesc_bf16(128, BN, 0, 0);  // A = Q (K-major), B = K (K-major)
  constexpr uint32_t kIdescPV = idesc_bf16(128, D, 0, 1);   // A = P (TMEM), B = V (MN-major)
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  constexpr uint64_t kStageStep = C::kTileBytes >> 4;
  // Descriptors precomputed once: Q for each K-step, the first stage of K (K-major) and V
  // (MN-major); a stage is a constant offset away.
  uint64_t qd[D / 16];
#pragma unroll
  for (int k = 0; k < D / 16; ++k)
    qd[k] = sdesc64(sdesc_lo(sbase + C::kOffQ + (k / 4) * kBoxBytes + (k % 4) * 32, 16), kHi);
  const uint64_t kd0 = sdesc64(sdesc_lo(sbase + C::kOffKV, 16), kHi);
  const uint64_t vd0 = sdesc64(sdesc_lo(sbase + C::kOffKV, kBoxBytes), kHi);
  auto issue_s = [&](int stage, int buf) {
    if constexpr (D == 128)
      mma_qk_d128(tmem + C::col_s(buf), qd, kd0 + stage * kStageStep, kIdescQK);
    else
      mma_qk_d64(tmem + C::col_s(buf), qd, kd0 + stage * kStageStep, kIdescQK);
    mma_commit(bar(C::kBarS + buf));
  };
  auto wait_full = [&](int ps) {
    return mbar_wait_warp(bar(C::kBarFull + ps % C::kStages), (ps / C::kStages) & 1, ctl);
  };
  auto release = [&](int ps) { mma_commit(bar(C::kBarEmpty + ps % C::kStages)); };

  bool ok = mbar_wait_warp(bar(C::kBarQ), 0, ctl);
  const TilePlan plan = make_plan(p, qt);
  int j = plan.next(0);
  int j1 = j < p.n_tiles ? plan.next(j + 1) : p.n_tiles;
  int pos = 0;
  for (int b = 0; b < 2 && ok; ++b) {  // S of the first two tiles
    if ((b ? j1 : j) >= p.n_tiles) break;
    if (!(ok = wait_full(pos))) break;
    tc_fence_after();
    issue_s(pos % C::kStages, b);
    release(pos);
    ++pos;
  }
  uint32_t pph[2] = {0, 0};
  for (int i = 0; ok && j < p.n_tiles; ++i) {
    const int buf = i & 1;
    const int j2 = j1 < p.n_tiles ? plan.next(j1 + 1) : p.n_tiles;
    const int kpos = j2 < p.n_tiles ? pos++ : -1;  // K(u_{i+2})
    const int vpos = pos++;                         // V(u_i)
    // O += P_i V_i once the softmax has written P_i over S buffer `buf`
    if (!mbar_wait_warp(bar(C::kBarP + buf), pph[buf], ctl)) { ok = false; break; }
    pph[buf] ^= 1;
    if (!wait_full(vpos)) { ok = false; break; }
    tc_fence_after();
    mma_pv_k128(tmem + C::kColO, tmem + C::col_s(buf), vd0 + (vpos % C::kStages) * kStageStep,
                kIdescPV, i > 0 ? 1u : 0u);
    mma_commit(bar(C::kBarPV));
    release(vpos);
    // S of the tile after next into the same buffer: the PV above reads P from it first (one
    // thread's MMAs run in issue order).
    if (kpos >= 0) {
      if (!wait_full(kpos)) { ok = false; break; }
      tc_fence_after();
      issue_s(kpos % C::kStages, buf);
      release(kpos);
    }
    j = j1;
    j1 = j2;
  }
  if (ok) {
    mma_commit(bar(C::kBarO));
  } else {
    // Let the MMAs already issued finish before TMEM is released.
    Ctl drain = ctl;
    int zero = 0;
    drain.abort_flag = &zero;
    mma_commit(bar(C::kBarDrain));
    mbar_wait_warp(bar(C::kBarDrain), 0, drain);
  }
}

// ---------------------------------------------------------------------------------------------
template <int D>
__device__ void softmax_wg(const FwdParams& p, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                           const Ctl& ctl, int bh, int qt) {
  using C = Cfg<D>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int r = warp * 32 + lane;
  const int row = qt * BM + r;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tO = tmem + lane_off + C::kColO;
  const float sl2 = p.scale_log2;

  float m = -INFINITY, l = 0.f;
  int i = 0;  // tiles processed
  uint32_t sph[2] = {0, 0};
  bool ok = true;
  const TilePlan plan = make_plan(p, qt);
  for (int j = plan.next(0); j < p.n_tiles; j = plan.next(j + 1), ++i) {
    const int buf = i & 1;
    const uint32_t tS = tmem + lane_off + C::col_s(buf);
    if (!mbar_wait(bar(C::kBarS + buf), sph[buf], ctl)) { ok = false; break; }
    sph[buf] ^= 1;
    tc_fence_after();
    uint32_t s[128];
    tmem_ld128(tS, s);

    const int key0 = j * BN;
    const int lim = (p.causal && j == qt) ? min(p.N, row + 1) : p.N;
    if (key0 + BN > lim) {
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (key0 + c >= lim) s[c] = __float_as_uint(-INFINITY);
    }
    // row max: eight independent chains of 3-input max (short dependency chains)
    float mxa[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mxa[u] = max3(-INFINITY, __uint_as_float(s[2 * u]), __uint_as_float(s[2 * u + 1]));
#pragma unroll
    for (int c = 16; c < 128; c += 16)
#pragma unroll
      for (int u = 0; u < 8; ++u)
        mxa[u] = max3(mxa[u], __uint_as_float(s[c + 2 * u]), __uint_as_float(s[c + 2 * u + 1]));
    const float mx = max3(max3(mxa[0], mxa[1], mxa[2]), max3(mxa[3], mxa[4], mxa[5]),
                          fmaxf(mxa[6], mxa[7])) * sl2;

    // Conditional rescaling (the FA4 idea of "3 · FlashAttention", 3.5): the reference max m
    // only moves when this tile's max exceeds it by more than kRescaleSlack (log2 units), so
    // P <= 2^kRescaleSlack and O, l are rescaled rarely. O = a / l is exact for any reference.
    if (__any_sync(~0u, mx > m + kRescaleSlack)) {
      const float m_new = fmaxf(m, mx);
      const float alpha = ex2(m - m_new);  // 0 when nothing was accumulated (m = -inf)
      if (i > 0) {
        // O must hold all i PV products. S of this tile was issued after PV_{i-2}, so at least
        // i - 1 have completed and the parity of completion i is unambiguous.
        bool good = mbar_wait(bar(C::kBarPV), (i - 1) & 1, ctl);
        if (__any_sync(~0u, !good)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const unsigned long long v = f2_mul(
                f2_pack(__uint_as_float(o[e]), __uint_as_float(o[e + 1])), f2_pack(alpha, alpha));
            float lo, hi;
            f2_unpack(v, lo, hi);
            o[e] = __float_as_uint(lo);
            o[e + 1] = __float_as_uint(hi);
          }
          tmem_st32(tO + c, o);
        }
      }
      l *= alpha;
      m = m_new;
    }
    const float m_use = m == -INFINITY ? 0.f : m;
    const unsigned long long k2 = f2_pack(sl2, sl2);
    const unsigned long long nm2 = f2_pack(-m_use, -m_use);
    unsigned long long rs[4];  // row sum in four independent packed chains
#pragma unroll
    for (int u = 0; u < 4; ++u) rs[u] = f2_pack(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const unsigned long long x = f2_fma(
            f2_pack(__uint_as_float(s[c + 2 * e]), __uint_as_float(s[c + 2 * e + 1])), k2, nm2);
        float x0, x1;
        f2_unpack(x, x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        rs[e & 3] = f2_add(rs[e & 3], f2_pack(p0, p1));
        pk[e] = pack_bf16(p0, p1);
      }
      tmem_st16(tS + c / 2, pk);
    }
    float rs0, rs1;
    f2_unpack(f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3])), rs0, rs1);
    l += rs0 + rs1;
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar(C::kBarP + buf));
  }

  // Every warp of the softmax warpgroup gets here; they agree on failures before the epilogue's
  // named barrier.
  if (bar_red_or(1, 128, !ok)) return;
  const size_t grow = static_cast<size_t>(bh) * p.N + row;
  if (i > 0) {
    const bool bad = !mbar_wait(bar(C::kBarO), 0, ctl);
    if (bar_red_or(1, 128, bad)) return;
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    // O / l as bf16 into this tile's Q buffer (free: every MMA has completed), 128-byte swizzled
    // like the TMA boxes; one thread then stores the tile with the TMA (rows past N are clipped).
    uint8_t* srow = smem + C::kOffQ + r * 128;
#pragma unroll 1
    for (int c = 0; c < D; c += 32) {
      uint32_t o[32];
      tmem_ld32(tO + c, o);
      uint8_t* box = srow + (c / 64) * kBoxBytes;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint4 w;
        w.x = pack_bf16(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
        w.y = pack_bf16(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
        w.z = pack_bf16(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
        w.w = pack_bf16(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
        const int chunk = (c % 64) / 8 + e;
        *reinterpret_cast<uint4*>(box + ((chunk ^ (r & 7)) << 4)) = w;
      }
    }
    fence_proxy_async_smem();
    bar_sync(1, 128);
    if (threadIdx.x == 0) {
      for (int b = 0; b < D / 64; ++b)
        tma_store_3d(&p.tm_o, sbase + C::kOffQ + b * kBoxBytes, b * 64, qt * BM, bh);
      bulk_commit();
      bulk_wait_all();
    }
    if (row < p.N)
      p.lse[grow] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  } else if (row < p.N) {
    uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D);
    for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0, 0, 0, 0);
    p.lse[grow] = -INFINITY;
  }
}

// ---------------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads, 1) fwd_tc_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemPtr);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };

  const int warp = threadIdx.x / 32;
  int bh, qt;
  decode_work(p, bh, qt);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kBarS + b), 1);
      mbar_init(bar(C::kBarP + b), 128);
    }
    mbar_init(bar(C::kBarPV), 1);
    mbar_init(bar(C::kBarO), 1);
    mbar_init(bar(C::kBarDrain), 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoadWarp) {
    producer<D>(p, sbase, ctl, bh, qt);  // whole warp: one elected lane issues
    __syncwarp();
  } else if (warp == kMmaWarp) {
    mma_issuer<D>(p, sbase, tmem, ctl, qt);  // whole warp: one elected lane issues
    __syncwarp();
  } else {
    softmax_wg<D>(p, smem, sbase, tmem, ctl, bh, qt);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
cudaError_t launch(const FwdParams& p, cudaStream_t s) {
  static bool configured = false;
  if (!configured) {
    const cudaError_t e = cudaFuncSetAttribute(
        fwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const unsigned grid = static_cast<unsigned>(p.n_tiles) * static_cast<unsigned>(p.BH);
  fwd_tc_kernel<D><<<grid, kThreads, Cfg<D>::kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdParams& p, int d, int /*num_sms*/, cudaStream_t s) {
  if (d == 64) return launch<64>(p, s);
  if (d == 128) return launch<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
