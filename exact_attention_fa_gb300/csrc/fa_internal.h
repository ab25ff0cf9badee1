// Internal launch interface between the C ABI (fa_api.cu) and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

// Everything a forward kernel needs. The three tensor maps describe Q, K, V as 3-D tensors
// [B*H][N][d] (bf16, 128-byte swizzle, box 64 x 128 x 1) so that out-of-range rows of a tile
// read as zero.
struct FwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_o;  // the output, same view as tm_q (the epilogue stores O tiles with the TMA)
  __nv_bfloat16* o;
  float* lse;
  const uint8_t* block_mask;  // [n_tiles][n_tiles] tile mask, or null (no tile mask)
  int BH, N;
  int n_tiles;                // ceil(N / 128): query tiles = key tiles = block-mask tiles
  int heads_per_group;        // CTA order: groups of heads whose K/V fit in L2
  int causal;                 // key j > query i masked (combines with a tile mask)
  float scale_log2;           // scale * log2(e)
  float o_scale;              // e4m3 inputs: O is multiplied by this (the scale of V)
  int exp2_poly;              // bf16: 1 = kExp2EmulationPer32 of every 32 exponentials on the FMA pipes
  unsigned* err;
  unsigned long long timeout_ns;
};

struct Fp32FwdParams {
  const float* q;
  const float* k;
  const float* v;
  float* o;
  float* lse;
  int BH, N, d;
  int causal;
  float scale_log2;
  int fa1;  // 1: FlashAttention-1 per-block normalised update
};

// Block-sparse backward: largest tile mask (query tiles) a CTA's shared-memory bitmask holds.
constexpr int kBwdMaxMaskTiles = 2048;

struct BwdParams {
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  CUtensorMap tm_do;
  CUtensorMap tm_dq;  // fp32 [B*H][N][d], box 32 x 64 x 1, 128-byte swizzle (bulk reductions)
  const __nv_bfloat16* o;
  const __nv_bfloat16* dO;
  const float* lse;
  float* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* lse2;   // workspace: lse * log2(e) per row (+inf for rows >= N)
  float* Dsum;   // workspace: D_i = sum_k dO_ik O_ik
  // workspace, d = 64: per 128-row tile two 4 KB bf16 operand tiles (128 rows x 16, K-major,
  // no swizzle) holding -lse2 / scale_log2 and -D, each split into three bf16 parts
  uint8_t* aug;
  // workspace: the main kernel's work counters, zeroed by the prep kernel: [0] hands out work
  // items in CTA start order, [1 + g] counts the CTAs that have zeroed their share of head group
  // g's dQ rows
  unsigned* ctr;
  const uint8_t* block_mask;  // [n_tiles][n_tiles] tile mask (row = query tile), or null
  int BH, N, d;
  int n_tiles;
  int causal;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  unsigned* err;
  unsigned long long timeout_ns;
};

// Decoding: Nq <= kDecodeMaxNq query rows per head against Nk keys. The key blocks of all heads
// (decode_tc_block_keys(d) keys each) are dealt out to n_ctas CTAs in contiguous ranges; piece
// (CTA c, head h) is slot c + h.
constexpr int kDecodeMaxNq = 8;
constexpr int kDecodeMaxCtas = 1024;
// Keys per block: 32 KB of K and of V per block at either head dimension.
constexpr int decode_tc_block_keys(int d) { return d == 64 ? 256 : 128; }
struct DecodeParams {
  // 3-D views [BH][rows][d] of q (rows Nq, box 64 x 16 x 1), k and v (rows Nk, box 64 x 128 x 1),
  // 128-byte swizzle; rows past the extent read as zero
  CUtensorMap tm_q;
  CUtensorMap tm_k;
  CUtensorMap tm_v;
  const __nv_bfloat16* q;  // [BH][Nq][d]
  const __nv_bfloat16* k;  // [BH][Nk][d]
  const __nv_bfloat16* v;
  __nv_bfloat16* o;        // [BH][Nq][d]
  float* lse;              // [BH][Nq]
  float* ws_o;             // [n_ctas + BH][Nq][d] pieces' outputs O_c / l_c
  float* ws_lse;           // [n_ctas + BH][Nq] pieces' lse, log2 units
  int BH, Nq, Nk;
  int blocks_per_head;     // set by the launcher (its block size)
  int n_ctas;              // 1 .. kDecodeMaxCtas; the launcher caps it at the number of blocks
  float scale_log2;
  unsigned* err;
  unsigned long long timeout_ns;
};

// Backward workspace layout: per padded row (B*H*ceil(N/128)*128 rows) lse2 and D, 8 bytes, and
// at d = 64 their two 32-byte operand rows; then the work counters (1 + B*H words), rounded up
// to 16 bytes.
inline size_t bwd_row_workspace_bytes(int d) { return 2 * sizeof(float) + (d == 64 ? 64 : 0); }
inline size_t bwd_counter_bytes(size_t BH) { return ((1 + BH) * sizeof(unsigned) + 15) / 16 * 16; }

// Argument checks shared by the backward entry points (fa_bwd, fa_bwd_blocksparse,
// fa_bwd_noalloc), so that all of them report the same status for the same bad argument: null
// pointers and sizes (FA_ERR_INVALID_ARG), FA_ERR_TOO_LARGE, d or the mask size
// (FA_ERR_UNSUPPORTED), alignment (FA_ERR_MISALIGNED), in that order. The workspace pointer is
// checked only when needs_workspace is set.
int check_bwd_args(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, const float* dq, const void* dk, const void* dv, int B, int H,
                   int N, int d, float scale, bool sparse, const uint8_t* block_mask,
                   const void* workspace, bool needs_workspace);

// Exponentials out of every 32 per row that the bf16 forward computes with a polynomial on the
// FMA pipes when that mode is on (fa_set_exp2_emulation).
constexpr int kExp2EmulationPer32 = 4;

// Launchers; return a cudaError_t (cudaSuccess on success).
cudaError_t launch_fwd_pair(const FwdParams& p, int d, cudaStream_t s);               // 2 tiles/CTA
// The same kernel on e4m3 Q, K, V at d = 128 (tm_q, tm_k, tm_v: 8-bit maps, box 128 x 128 x 1).
cudaError_t launch_fwd_fp8(const FwdParams& p, cudaStream_t s);
cudaError_t launch_fwd_fp32(const Fp32FwdParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_bwd(const BwdParams& p, int num_sms, cudaStream_t s);
// Decoding: the split kernel on the tensor cores (tensor maps in p), then the merge of the pieces.
cudaError_t launch_decode(const DecodeParams& p, int d, cudaStream_t s);
// Opt the kernels that use more than 48 KB of dynamic shared memory in to their size. Function
// attributes belong to a device's context, so these run once per device, with it current.
cudaError_t configure_fwd_pair();
cudaError_t configure_bwd();
cudaError_t configure_decode();
cudaError_t configure_fwd_fp32();

}  // namespace fa
