// bf16 forward on the 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// The method is the tiled online-softmax attention of "FlashAttention：メモリ効率的なアテンション計算"
// (sections "オンライン softmax" and "タイル化") in the FlashAttention-2 order of
// "출력을 누적해 메모리 이동을 줄이는 FlashAttention": per query tile, stream the key/value tiles, keep a
// running row max m, running sum l and an unnormalised accumulator O rescaled by exp(m - m_new),
// divide by l once at the end. Neither S nor P ever leaves the SM.
//
// GB300 mapping (one CTA per SM, 12 warps; every bf16 forward: d = 64 and 128, dense, causal and
// block-sparse):
//   * a CTA owns two 128-row query tiles (t = 0, 1) of one (b, h), so the tensor core works on one
//     tile's QK^T / PV while the other tile's softmax runs on the CUDA cores, and each K/V tile
//     streamed from L2 serves 256 query rows;
//   * warp 8 (one elected lane) streams K_j, V_j with TMA into a ring of 128-byte-swizzled shared-memory
//     stages guarded by full/empty mbarriers, keys one tile ahead of values; Q is loaded once;
//   * warps 9 and 10 (one elected lane each) issue the MMAs of tile 0 and tile 1: S_t = Q_t K_j^T
//     (both operands in shared memory, fp32 result in TMEM) and O_t += P_t V_j (P_t read from
//     TMEM, V_j from shared memory);
//   * warps 0-3 / 4-7 are the softmax warpgroups of tile 0 / 1: thread r owns query row r (TMEM
//     lane r). It loads its 128 scores, applies the scale (log2(e) folded in, exp2 on the SFU),
//     the causal / tail mask, updates m and l, rescales its O row only when the reference max
//     moves (conditional rescaling), writes P as bf16 (e4m3 for e4m3 inputs) into TMEM, and
//     finally normalises O and writes O and lse.
//   * causal / block-sparse: key tiles a query tile does not need are never loaded nor multiplied
//     ("3 · FlashAttention", question on the causal mask; "拡張: Block-Sparse FlashAttention").
// TMEM columns: d = 128: S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512), P_t over S_t
// (e4m3 P: the first 32 columns of S_t); d = 64: S_0, S_1 as above, P_0 [256,320), P_1 [320,384),
// O_0 [384,448), O_1 [448,512).
// The same kernel serves e4m3 inputs at d = 128 ("3 · FlashAttention", 3.5, the FP8 support of
// FlashAttention-3): both products run as tcgen05.mma kind::f8f6f4 on e4m3 operands with fp32
// accumulation; P is rounded to e4m3 for the P V product, l sums the unrounded fp32 P.
#include <cuda_bf16.h>
#include <math.h>

#include "fa_internal.h"
#include "fa_ptx.cuh"

namespace fa {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;    // warps 9 and 10 issue the MMAs of query tiles 0 and 1
constexpr int kThreads = 384;  // warp 11 only completes the producer / MMA warpgroup
// Registers per thread after the warpgroups re-balance the 168 each thread is launched with: the
// softmax warpgroups hold a row of 128 scores plus the row statistics.
constexpr int kRegsSoftmax = 208;
constexpr int kRegsLoadMma = 88;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsLoadMma <= kThreads * 168,
              "register split exceeds the launch's allocation");
constexpr int kBoxBytes = 128 * 64 * 2;  // one TMA box: 128 rows x 64 bf16 (128 B rows)
constexpr float kRescaleSlack = 8.f;     // log2 units: P stays <= 256

// F8: e4m3 Q, K, V (d = 128 only): a tile row is 128 bytes, one TMA box; the products are
// tcgen05.mma kind::f8f6f4 and P goes to TMEM as e4m3. O is still written as bf16, through a
// staging area of its own (the 16 KB e4m3 Q tile is too small for the 32 KB bf16 O tile).
template <int D, bool F8 = false>
struct Cfg {
  static_assert(!F8 || D == 128, "the e4m3 forward is built for d = 128");
  static constexpr int kElemBytes = F8 ? 1 : 2;
  static constexpr int kTileBytes = 128 * D * kElemBytes;
  static constexpr int kBoxCols = 128 / kElemBytes;  // elements per 128-byte TMA box row
  static constexpr int kBoxes = D / kBoxCols;        // TMA boxes per tile
  static constexpr int kStages = F8 ? 8 : (D == 128 ? 4 : 8);  // K/V ring (K, V alternate)
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = 2 * kTileBytes;
  static constexpr int kOTileBytes = 128 * D * 2;  // one bf16 O tile
  static constexpr int kOffOStage = kOffKV + kStages * kTileBytes;  // F8 only
  static constexpr int kOffBar = kOffOStage + (F8 ? 2 * kOTileBytes : 0);
  // barriers: Q, full[S], empty[S], s_full[2], p_full[2], o_full[2], pv_done[2], s_free[2],
  // drain[2]
  static constexpr int kBarQ = 0;
  static constexpr int kBarFull = 1;
  static constexpr int kBarEmpty = 1 + kStages;
  static constexpr int kBarS = 1 + 2 * kStages;
  static constexpr int kBarP = kBarS + 2;
  static constexpr int kBarO = kBarP + 2;
  static constexpr int kBarPV = kBarO + 2;
  static constexpr int kBarSFree = kBarPV + 2;
  static constexpr int kBarDrain = kBarSFree + 2;
  static constexpr int kNumBars = kBarDrain + 2;
  static constexpr int kOffTmemPtr = kOffBar + 8 * kNumBars;
  static constexpr int kOffAbort = kOffTmemPtr + 4;
  static constexpr int kSmemBytes = kOffAbort + 4 + 1024;  // + slack to align the base to 1 KB
  // d = 64: P_t has TMEM columns of its own (S 2 x 128, P 2 x 64, O 2 x 64 = 512 columns). The
  // softmax warps release S_t as soon as they hold its scores in registers, so S_t of the next
  // key tile is computed while they still work on this one, and PV_t reads P_t meanwhile.
  // d = 128 has no room and writes P_t over S_t.
  static constexpr bool kSepP = D == 64;
  __device__ static constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
  __device__ static constexpr uint32_t col_p(int t) { return kSepP ? 256u + 64u * t : col_s(t); }
  __device__ static constexpr uint32_t col_o(int t) {
    return kSepP ? 384u + 64u * t : (t ? 256u + D : 256u);
  }
};

// Key tiles visited by the two query tiles of a CTA, resolved once per role: dense and causal
// query tiles need key tiles [0, last_t] (last_t = -1 past the end of the sequence); block-sparse
// ones additionally look up the tile mask. Kept in registers so that the per-tile bookkeeping of
// the MMA and producer warps stays a few integer compares.
struct TilePlan {
  const uint8_t* mask0;  // block-sparse: mask rows of the two query tiles, else null
  const uint8_t* mask1;
  int last0, last1, n_tiles;
  __device__ __forceinline__ bool active(int t, int j) const {
    const int last = t ? last1 : last0;
    const uint8_t* m = t ? mask1 : mask0;
    return j <= last && (m == nullptr || __ldg(m + j) != 0);
  }
  // next key tile >= j needed by either query tile, or n_tiles
  __device__ __forceinline__ int next(int j) const {
    if (mask0 == nullptr) return j <= max(last0, last1) ? j : n_tiles;
    for (; j < n_tiles; ++j)
      if (active(0, j) || active(1, j)) return j;
    return n_tiles;
  }
};

__device__ __forceinline__ TilePlan make_plan(const FwdParams& p, int qt0, int qt1) {
  TilePlan t;
  t.n_tiles = p.n_tiles;
  const bool sparse = p.block_mask != nullptr;
  auto last = [&](int qt) { return qt * BM >= p.N ? -1 : (p.causal ? qt : p.n_tiles - 1); };
  t.last0 = last(qt0);
  t.last1 = last(qt1);
  t.mask0 = sparse ? p.block_mask + static_cast<size_t>(qt0) * p.n_tiles : nullptr;
  t.mask1 = sparse ? p.block_mask + static_cast<size_t>(qt1) * p.n_tiles : nullptr;
  return t;
}

// CTA -> (head, query-tile pair). Heads are taken in groups small enough for their K/V to stay
// in L2; inside a group the pairs with the most key tiles (causal: the last ones) come first.
__device__ __forceinline__ void decode_work(const FwdParams& p, int& bh, int& pair) {
  const int n_pairs = (p.n_tiles + 1) / 2;
  const int per_group = p.heads_per_group * n_pairs;
  const int g = blockIdx.x / per_group;
  const int within = blockIdx.x - g * per_group;
  const int gsize = min(p.heads_per_group, p.BH - g * p.heads_per_group);
  pair = n_pairs - 1 - within / gsize;
  bh = g * p.heads_per_group + within % gsize;
}

// ---------------------------------------------------------------------------------------------
template <int D, bool F8>
__device__ void producer(const FwdParams& p, uint32_t sbase, const Ctl& ctl, int bh, int qt0,
                         int qt1) {
  using C = Cfg<D, F8>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  tma_prefetch_desc(&p.tm_q);
  tma_prefetch_desc(&p.tm_k);
  tma_prefetch_desc(&p.tm_v);

  mbar_arrive_expect_tx(bar(C::kBarQ), 2 * C::kTileBytes);
  for (int t = 0; t < 2; ++t)
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_3d(sbase + C::kOffQ + t * C::kTileBytes + b * kBoxBytes, &p.tm_q, bar(C::kBarQ),
                  b * C::kBoxCols, (t ? qt1 : qt0) * BM, bh);

  int issued[C::kStages];
#pragma unroll
  for (int s = 0; s < C::kStages; ++s) issued[s] = -1;
  // Ring order: K of the first tile, then per tile K of the next tile ahead of V of this one,
  // so that keys (needed first, by S) run one tile ahead of values (needed last, by PV).
  int pos = 0;
  bool ok = true;
  auto load = [&](const void* map, int j) {
    const int s = pos % C::kStages;
    const int round = pos / C::kStages;
    if (!mbar_wait_warp(bar(C::kBarEmpty + s), (round & 1) ^ 1, ctl)) return false;
    mbar_arrive_expect_tx(bar(C::kBarFull + s), C::kTileBytes);
    for (int b = 0; b < C::kBoxes; ++b)
      tma_load_3d(sbase + C::kOffKV + s * C::kTileBytes + b * kBoxBytes, map, bar(C::kBarFull + s),
                  b * C::kBoxCols, j * BN, bh);
    issued[s] = round;
    ++pos;
    return true;
  };
  const TilePlan plan = make_plan(p, qt0, qt1);
  int j = plan.next(0);
  if (j < p.n_tiles) ok = load(&p.tm_k, j);
  while (ok && j < p.n_tiles) {
    const int jn = plan.next(j + 1);
    if (jn < p.n_tiles && !(ok = load(&p.tm_k, jn))) break;
    if (!(ok = load(&p.tm_v, j))) break;
    j = jn;
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
// MMA issue for query tile t, by warp kMmaWarp + t. At d = 64 one tile's MMAs take about as long
// to issue (about 30-50 cycles per instruction from one thread) as to execute, so each tile has a
// warp of its own: the two issue streams share the tensor pipe and the K/V ring. Both warps walk
// every ring position in the producer's order and release each one (the empty barriers count
// both); a warp waits for a position to be full before releasing it even when its tile skips
// that key tile, so neither can release a stage ahead of the other's use of it.
template <int D, bool F8>
__device__ void mma_issuer(const FwdParams& p, uint32_t sbase, uint32_t tmem, const Ctl& ctl,
                           int qt0, int qt1, int t) {
  using C = Cfg<D, F8>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  // A = Q (K-major), B = K (K-major); PV: A = P (TMEM), B = V (MN-major)
  constexpr uint32_t kIdescQK = F8 ? idesc_e4m3(128, BN, 0, 0) : idesc_bf16(128, BN, 0, 0);
  constexpr uint32_t kIdescPV = F8 ? idesc_e4m3(128, D, 0, 1) : idesc_bf16(128, D, 0, 1);

  // Descriptors precomputed once (Q_t per K-step, first K and V stage); a stage is a constant
  // offset away, so each MMA costs the issuing thread one add. A K-step covers 32 bytes of a
  // 128-byte swizzle row (16 bf16 or 32 e4m3), four steps per TMA box.
  constexpr uint32_t kHi = sdesc_hi_sw128(1024);
  constexpr uint64_t kStageStep = C::kTileBytes >> 4;
  constexpr int kSteps = D * C::kElemBytes / 32;
  uint64_t qd[kSteps];
#pragma unroll
  for (int k = 0; k < kSteps; ++k)
    qd[k] = sdesc64(
        sdesc_lo(sbase + C::kOffQ + t * C::kTileBytes + (k / 4) * kBoxBytes + (k % 4) * 32, 16), kHi);
  const uint64_t kd0 = sdesc64(sdesc_lo(sbase + C::kOffKV, 16), kHi);
  const uint64_t vd0 = sdesc64(sdesc_lo(sbase + C::kOffKV, kBoxBytes), kHi);
  const uint32_t tS = tmem + C::col_s(t);
  auto issue_s = [&](int stage) {
    if constexpr (F8)
      mma_qk_f8_d128(tS, qd, kd0 + stage * kStageStep, kIdescQK);
    else if constexpr (D == 128)
      mma_qk_d128(tS, qd, kd0 + stage * kStageStep, kIdescQK);
    else
      mma_qk_d64(tS, qd, kd0 + stage * kStageStep, kIdescQK);
    mma_commit(bar(C::kBarS + t));
  };
  auto issue_pv = [&](int stage, bool accumulate) {
    if constexpr (F8)
      mma_pv_f8_k128(tmem + C::col_o(t), tmem + C::col_p(t), vd0 + stage * kStageStep, kIdescPV,
                     accumulate ? 1u : 0u);
    else
      mma_pv_k128(tmem + C::col_o(t), tmem + C::col_p(t), vd0 + stage * kStageStep, kIdescPV,
                  accumulate ? 1u : 0u);
  };

  bool ok = mbar_wait_warp(bar(C::kBarQ), 0, ctl);
  tc_fence_after();
  uint32_t pphase = 0, sfphase = 0;
  bool acc = false;
  bool s_pending = false;  // separate P columns: an S_t issued and not yet released
  // Ring positions in the producer's order: K(u0), then per union tile u_i: K(u_{i+1}), V(u_i).
  auto wait_full = [&](int ps) {
    const bool good =
        mbar_wait_warp(bar(C::kBarFull + ps % C::kStages), (ps / C::kStages) & 1, ctl);
    tc_fence_after();
    return good;
  };
  const TilePlan plan = make_plan(p, qt0, qt1);
  int j = plan.next(0);
  int i = 0;  // index of j among the union tiles
  if (ok && j < p.n_tiles) {
    ok = wait_full(0);
    if (ok && plan.active(t, j)) {
      issue_s(0);
      s_pending = true;
    }
    mma_commit(bar(C::kBarEmpty + 0));
  }
  while (ok && j < p.n_tiles) {
    const bool a = plan.active(t, j);
    const int jn = plan.next(j + 1);
    const bool has_next = jn < p.n_tiles;
    const bool n = has_next && plan.active(t, jn);
    const int kpos = 2 * i + 1;                         // K(u_{i+1})
    const int vpos = has_next ? 2 * i + 2 : 2 * i + 1;  // V(u_i)
    const int sv = vpos % C::kStages, skn = kpos % C::kStages;
    if (has_next && !(ok = wait_full(kpos))) break;
    if constexpr (C::kSepP) {
      // S_t of the next tile as soon as the softmax warps hold S_t of this one in registers,
      // then PV_t of this tile once they have written P_t.
      if (n) {
        if (s_pending) {
          if (!(ok = mbar_wait_warp(bar(C::kBarSFree + t), sfphase, ctl))) break;
          sfphase ^= 1;
          tc_fence_after();
        }
        issue_s(skn);
        s_pending = true;
      }
      if (!(ok = wait_full(vpos))) break;
      if (a) {
        if (!(ok = mbar_wait_warp(bar(C::kBarP + t), pphase, ctl))) break;
        pphase ^= 1;
        tc_fence_after();
        issue_pv(sv, acc);
        mma_commit(bar(C::kBarPV + t));
        acc = true;
      }
    } else {
      if (!(ok = wait_full(vpos))) break;
      if (a) {
        if (!(ok = mbar_wait_warp(bar(C::kBarP + t), pphase, ctl))) break;
        pphase ^= 1;
        tc_fence_after();
        issue_pv(sv, acc);
        acc = true;
      }
      // S_t of the next tile overwrites P_t of this one: one thread's MMAs run in issue order,
      // so the PV above has read P_t before this write lands.
      if (n) issue_s(skn);
    }
    if (has_next) mma_commit(bar(C::kBarEmpty + skn));
    mma_commit(bar(C::kBarEmpty + sv));
    ++i;
    j = jn;
  }
  if (ok) {
    mma_commit(bar(C::kBarO + t));
  } else {
    // Let the MMAs already issued finish before TMEM is released.
    Ctl drain = ctl;
    int zero = 0;
    drain.abort_flag = &zero;
    mma_commit(bar(C::kBarDrain + t));
    mbar_wait_warp(bar(C::kBarDrain + t), 0, drain);
  }
}

// ---------------------------------------------------------------------------------------------
// POLY: scores out of every 32 of a row whose exponential is computed on the FMA pipes
// (exp2_poly2) instead of the SFU; 0 in the default instances.
template <int D, bool F8, int POLY>
__device__ void softmax_wg(const FwdParams& p, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                           const Ctl& ctl, int bh, int qt0, int qt1) {
  static_assert(POLY == 0 || (32 % POLY == 0 && POLY % 2 == 0), "POLY: pairs spread evenly");
  using C = Cfg<D, F8>;
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int t = warp / 4;
  const int quad = warp % 4;
  const int r = quad * 32 + lane;
  const int qt = t ? qt1 : qt0;
  const int row = qt * BM + r;
  const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tS = tmem + lane_off + C::col_s(t);
  const uint32_t tP = tmem + lane_off + C::col_p(t);
  const uint32_t tO = tmem + lane_off + C::col_o(t);
  const float sl2 = p.scale_log2;

  float m = -INFINITY, l = 0.f;
  bool any = false;
  int n_done = 0;  // tiles of this query tile processed so far
  uint32_t sphase = 0;
  bool ok = true;
  const TilePlan plan = make_plan(p, qt0, qt1);
  const int last = t ? plan.last1 : plan.last0;
  for (int j = 0; j <= last; ++j) {
    if (!plan.active(t, j)) continue;
    if (!mbar_wait(bar(C::kBarS + t), sphase, ctl)) { ok = false; break; }
    sphase ^= 1;
    tc_fence_after();

    uint32_t s[128];
    tmem_ld128(tS, s);
    if constexpr (C::kSepP) {
      tc_fence_before();
      mbar_arrive(bar(C::kBarSFree + t));
    }

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
    // Separate P columns: S of this tile may have landed before PV of the previous tile
    // completed; O (for a rescale) and the P columns (before they are rewritten) need it first.
    bool pv_ready = !C::kSepP || n_done == 0;
    auto wait_pv = [&]() {
      if (pv_ready) return true;
      pv_ready = true;
      const bool good = mbar_wait(bar(C::kBarPV + t), (n_done - 1) & 1, ctl);
      tc_fence_after();
      return good;
    };
    if (__any_sync(~0u, mx > m + kRescaleSlack)) {
      const float m_new = fmaxf(m, mx);
      const float alpha = ex2(m - m_new);  // 0 when nothing was accumulated (m = -inf)
      if (any) {
        if (!wait_pv()) { ok = false; break; }
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const unsigned long long v = f2_mul(
                f2_pack(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), f2_pack(alpha, alpha));
            float lo, hi;
            f2_unpack(v, lo, hi);
            o[i] = __float_as_uint(lo);
            o[i + 1] = __float_as_uint(hi);
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
    bool fail = false;
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      uint32_t pk[16];
      float q0 = 0.f, q1 = 0.f;  // e4m3: the pair of an even i, packed with the next pair
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const unsigned long long x = f2_fma(
            f2_pack(__uint_as_float(s[c + 2 * i]), __uint_as_float(s[c + 2 * i + 1])), k2, nm2);
        float x0, x1;
        f2_unpack(x, x0, x1);
        float p0, p1;
        if constexpr (POLY > 0) {
          if (i % (32 / POLY) == 0) {  // POLY / 2 pairs of every 16, spread out
            exp2_poly2(x0, x1, p0, p1);
          } else {
            p0 = ex2(x0);
            p1 = ex2(x1);
          }
        } else {
          p0 = ex2(x0);
          p1 = ex2(x1);
        }
        rs[i & 3] = f2_add(rs[i & 3], f2_pack(p0, p1));
        if constexpr (F8) {
          // four e4m3 per TMEM column (keys 4u .. 4u + 3 of this chunk in bytes 0 .. 3)
          if (i & 1) {
            pk[i / 2] = pack_e4m3x4(q0, q1, p0, p1);
          } else {
            q0 = p0;
            q1 = p1;
          }
        } else {
          pk[i] = pack_bf16(p0, p1);
        }
      }
      if (c == 0 && !wait_pv()) fail = true;
      if constexpr (F8)
        tmem_st8(tP + c / 4, pk);
      else
        tmem_st16(tP + c / 2, pk);
    }
    if (fail) { ok = false; break; }
    float rs0, rs1;
    f2_unpack(f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3])), rs0, rs1);
    l += rs0 + rs1;
    any = true;
    ++n_done;
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(bar(C::kBarP + t));
  }

  // Every warp of the softmax warpgroup gets here; they agree on failures before the epilogue's
  // named barrier.
  if (bar_red_or(1 + t, 128, !ok)) return;
  const size_t grow = static_cast<size_t>(bh) * p.N + row;
  if (any) {
    const bool bad = !mbar_wait(bar(C::kBarO + t), 0, ctl);
    if (bar_red_or(1 + t, 128, bad)) return;
    tc_fence_after();
    float inv = l > 0.f ? 1.f / l : 0.f;
    if constexpr (F8) inv *= p.o_scale;
    // O / l as bf16 into this tile's Q buffer (free: every MMA has completed; e4m3: the staging
    // area), 128-byte swizzled like the TMA boxes; one thread then stores the tile with the TMA
    // (rows past N are clipped).
    constexpr int kOStage = F8 ? C::kOffOStage : C::kOffQ;
    constexpr int kOTile = F8 ? C::kOTileBytes : C::kTileBytes;
    uint8_t* srow = smem + kOStage + t * kOTile + r * 128;
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
    bar_sync(1 + t, 128);
    if (threadIdx.x == 128 * t) {
      for (int b = 0; b < D / 64; ++b)
        tma_store_3d(&p.tm_o, sbase + kOStage + t * kOTile + b * kBoxBytes, b * 64, qt * BM, bh);
      bulk_commit();
      bulk_wait_all();
    }
    if (row < p.N)
      p.lse[grow] = l > 0.f ? (m + __log2f(l)) * 0.6931471805599453f : -INFINITY;
  } else if (row < p.N) {
    uint4* dst = reinterpret_cast<uint4*>(p.o + grow * D);
    for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
    p.lse[grow] = -INFINITY;
  }
}

// ---------------------------------------------------------------------------------------------
template <int D, bool F8 = false, int POLY = 0>
__global__ void __launch_bounds__(kThreads, 1) fwd_pair_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D, F8>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffAbort);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffTmemPtr);
  const Ctl ctl{abort_flag, p.err, p.timeout_ns};
  auto bar = [&](int i) { return sbase + C::kOffBar + 8u * i; };

  const int warp = threadIdx.x / 32;
  int bh, pair;
  decode_work(p, bh, pair);
  const int qt0 = 2 * pair, qt1 = 2 * pair + 1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar(C::kBarQ), 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(bar(C::kBarFull + s), 1);
      mbar_init(bar(C::kBarEmpty + s), 2);  // released by both MMA warps
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(C::kBarS + t), 1);
      mbar_init(bar(C::kBarP + t), 128);
      mbar_init(bar(C::kBarPV + t), 1);
      mbar_init(bar(C::kBarO + t), 1);
      mbar_init(bar(C::kBarSFree + t), 128);
    }
    mbar_init(bar(C::kBarDrain + 0), 1);
    mbar_init(bar(C::kBarDrain + 1), 1);
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

  if (warp >= kLoadWarp) {
    regs_dec<kRegsLoadMma>();
    if (warp == kLoadWarp)
      producer<D, F8>(p, sbase, ctl, bh, qt0, qt1);  // whole warp: one elected lane issues
    else if (warp == kMmaWarp || warp == kMmaWarp + 1)
      mma_issuer<D, F8>(p, sbase, tmem, ctl, qt0, qt1, warp - kMmaWarp);  // one elected lane
    __syncwarp();
  } else {
    regs_inc<kRegsSoftmax>();
    softmax_wg<D, F8, POLY>(p, smem, sbase, tmem, ctl, bh, qt0, qt1);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool F8 = false, int POLY = 0>
cudaError_t configure() {
  return cudaFuncSetAttribute(fwd_pair_kernel<D, F8, POLY>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D, F8>::kSmemBytes);
}

template <int D, bool F8 = false, int POLY = 0>
cudaError_t launch(const FwdParams& p, cudaStream_t s) {
  const unsigned grid = static_cast<unsigned>((p.n_tiles + 1) / 2) * static_cast<unsigned>(p.BH);
  fwd_pair_kernel<D, F8, POLY><<<grid, kThreads, Cfg<D, F8>::kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t configure_fwd_pair() {
  cudaError_t e = configure<64>();
  if (e == cudaSuccess) e = configure<128>();
  if (e == cudaSuccess) e = configure<128, true>();
  if (e == cudaSuccess) e = configure<64, false, kExp2EmulationPer32>();
  return e != cudaSuccess ? e : configure<128, false, kExp2EmulationPer32>();
}

cudaError_t launch_fwd_fp8(const FwdParams& p, cudaStream_t s) { return launch<128, true>(p, s); }

cudaError_t launch_fwd_pair(const FwdParams& p, int d, cudaStream_t s) {
  if (p.exp2_poly) {
    if (d == 64) return launch<64, false, kExp2EmulationPer32>(p, s);
    if (d == 128) return launch<128, false, kExp2EmulationPer32>(p, s);
    return cudaErrorInvalidValue;
  }
  if (d == 64) return launch<64>(p, s);
  if (d == 128) return launch<128>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace fa
