/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library (libfa_gb300.so).
 *
 * What is computed. For every batch b < B and head h < H, with Q, K, V in R^{N x d}:
 *     S = scale * Q K^T   (S_ij = -inf where masked),
 *     O = softmax(S) V,   lse_i = m_i + ln sum_j exp(S_ij - m_i),  m_i = max_j S_ij
 * -- "3 · FlashAttention" (mkdocs.reaper.mx), 3.1; "FlashAttention：メモリ効率的なアテンション計算"
 * (tech-tldr.com), first formula. The kernels reach it with the online-softmax recurrence of
 * "FlashAttention：メモリ効率的なアテンション計算", section "オンライン softmax" (running max m,
 * running sum l, unnormalised accumulator rescaled by exp(m - m_new), one division by l at the end;
 * FlashAttention-2 order as in "출력을 누적해 메모리 이동을 줄이는 FlashAttention"), so that no N x N
 * matrix is ever written to device memory.
 *
 * Common conventions of every entry point:
 *   - Layout: Q, K, V, O, dO, dQ, dK, dV are dense row-major [B, H, N, d] (d contiguous);
 *     lse is [B, H, N] fp32. The backward workspace is opaque scratch of
 *     fa_bwd_workspace_bytes(...) bytes.
 *   - Pointers are DEVICE pointers owned by the caller, 16-byte aligned; outputs must not alias
 *     inputs. The library allocates no memory on any call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Every call only enqueues work:
 *     it returns after the launches, without synchronising. The current CUDA device must be an
 *     sm_103 GPU and must own the pointers.
 *   - Arguments are validated before anything is enqueued; a non-zero return means nothing
 *     was launched (except FA_ERR_CUDA from a failed launch).
 *   - Kernels never spin forever: every wait on an on-chip barrier gives up after a bounded time
 *     and records FA_ERR_DEVICE_TIMEOUT in a device error word, read by fa_check_device_error.
 *   - The library sets itself up once per device, on the first call with that device current
 *     (kernel attributes, device addresses of its own __device__ objects); a failed set-up is
 *     retried on the next call. Calls after cudaDeviceReset on that device are not supported.
 *   - Masked rows: a query row with no allowed key gets O = 0 and lse = -inf.
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* identical to cudaStream_t */

enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,    /* null pointer, B/H/N < 1, non-finite or non-positive scale      */
  FA_ERR_UNSUPPORTED = 2,    /* head dim d or N not supported by this entry point               */
  FA_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned                                */
  FA_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed (tensor map, launch)       */
  FA_ERR_DEVICE_TIMEOUT = 5, /* a kernel gave up waiting on an on-chip barrier                  */
  FA_ERR_NO_DEVICE = 6,      /* no current CUDA device, or it is not compute capability 10.3   */
  FA_ERR_TOO_LARGE = 7,      /* B*H*N or a grid dimension exceeds what the kernels index        */
  FA_ERR_SCRATCH_LIMIT = 8   /* fa_bwd_noalloc: the problem needs more than its static scratch  */
};

/* Forward, bf16 inputs and output, fp32 accumulation (tensor cores: tcgen05.mma, TMEM).
 * q, k, v : [B,H,N,d] bf16 (read);  o : [B,H,N,d] bf16 (written);  lse : [B,H,N] fp32 (written,
 * natural log of the row's softmax denominator of the scaled scores, the statistic the backward
 * recomputes P from -- "FlashAttention: IOを意識した高速かつメモリ効率の高い厳密なアテンション"
 * (xyznot.com), "主要なアイデア", recomputation from O and (l, m)).
 * d in {64, 128}; any N >= 1 (the last tile is masked). causal != 0 applies the lower-triangular
 * mask key j <= query i and skips whole key tiles above the diagonal ("3 · FlashAttention",
 * question on the causal mask). */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N,
           int d, float scale, int causal, fa_stream_t stream);

/* Forward with fp32 inputs and outputs, computed with fp32 FMAs (no tensor cores), for accuracy
 * at the 1e-5 level. Same semantics as fa_fwd; d a multiple of 32 in [32, 128]. */
int fa_fwd_fp32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                int H, int N, int d, float scale, int causal, fa_stream_t stream);

/* fa_fwd_fp32 in the FlashAttention-1 form ("FlashAttention: IOを意識した高速かつメモリ効率の高い
 * 厳密なアテンション" (xyznot.com), "手法" steps 1-4): after every key block the output row is kept
 * normalised, O <- diag(l_new)^-1 (diag(l) e^(m - m_new) O + e^(m~ - m_new) P~ V_j), with P~ and
 * l~ taken against the block's own max m~. Same arguments, result (to rounding) and errors as
 * fa_fwd_fp32. */
int fa_fwd_fp32_fa1(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                    int H, int N, int d, float scale, int causal, fa_stream_t stream);

/* Block-sparse forward ("FlashAttention: IOを意識した..." (xyznot.com), "拡張: Block-Sparse
 * FlashAttention"): block_mask is a DEVICE uint8 array [T][T] with T = ceil(N/128), row = query
 * tile, column = key tile, shared by all (b, h); a zero entry masks the whole 128 x 128 tile of
 * scores and the kernel never visits it. causal != 0 further applies fa_fwd's causal mask (tiles
 * above the diagonal are skipped whatever the mask says). A row left with no key gets O = 0 and
 * lse = -inf. bf16 like fa_fwd; d in {64, 128}; any N >= 1 (the last tile's keys past N are
 * masked). */
int fa_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                       fa_stream_t stream);

/* Forward with e4m3 (8-bit float: 4 exponent bits, 3 mantissa bits, OCP "e4m3fn") inputs, the
 * FP8 support the FlashAttention-3 row of "3 · FlashAttention" (mkdocs.reaper.mx), 3.5, lists.
 * q, k, v : [B,H,N,d] e4m3 bytes (read);  o : [B,H,N,d] bf16 (written);  lse : [B,H,N] fp32
 * (written), as fa_fwd. Both products run on the tensor cores with e4m3 operands and fp32
 * accumulation: S = scale * Q K^T, and P (the exponentials, at most 2^8 against the running max)
 * is rounded to e4m3 for the product with V, while the row sum l adds the unrounded fp32 values.
 * The result is o = v_scale * softmax(S) V and lse = log-sum-exp of S: for tensors quantised as
 * x = s_x * x8, pass scale * s_q * s_k as `scale` and s_v as `v_scale`. d = 128 only
 * (FA_ERR_UNSUPPORTED otherwise); any N >= 1; causal as fa_fwd. Errors as fa_fwd, plus
 * FA_ERR_INVALID_ARG for a non-finite v_scale. */
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
               int N, int d, float scale, float v_scale, int causal, fa_stream_t stream);

/* The partial software exponential of FlashAttention-4 ("3 · FlashAttention" (mkdocs.reaper.mx),
 * 3.5: some of the softmax's exponentials computed on the FMA units instead of the special
 * function unit). per32 = 4: the bf16 forward (fa_fwd, fa_fwd_blocksparse) computes 4 of every 32
 * exponentials of a row with a degree-3 polynomial (relative error below 7.5e-5, under the bf16
 * rounding of P) on the FMA pipes; per32 = 0 (the default): all on the SFU. The results agree
 * within the bf16 tolerances either way. It is off by default because on GB300 it measures slower
 * (the softmax is limited by its dependency chain and instruction issue, not by the SFU). The
 * setting is process-wide and applies to forward calls enqueued after it; it does not affect
 * fa_fwd_fp8, fa_fwd_fp32 or fa_decode. Returns FA_ERR_INVALID_ARG for other values. */
int fa_set_exp2_emulation(int per32);

/* The current per32 setting of fa_set_exp2_emulation (0 or 4). */
int fa_get_exp2_emulation(void);

/* Bytes of device workspace fa_bwd needs: per row of B*H*ceil(N/128)*128 rows (rows padded to
 * whole 128-row tiles) two fp32 row statistics (8 bytes) and, at d = 64, two 32-byte bf16
 * operand rows made from them (72 bytes in all); then 4 * (1 + B*H) bytes of work counters,
 * rounded up to a multiple of 16. 0 for B, H, N < 1 or d not in {64, 128}. */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/* Backward by recomputation ("3 · FlashAttention", 3.4; "FlashAttention：在线 softmax 与
 * IO-aware 注意力" (quant67.com), section 五): S and P are rebuilt tile by tile from q, k and the
 * saved lse, never stored. Given dO = dL/dO it writes
 *     dq = scale * dS K (fp32, [B,H,N,d]),  dk = scale * dS^T Q (bf16),  dv = P^T dO (bf16),
 * with dS = P * (dP - D), dP = dO V^T, D_i = sum_k dO_ik O_ik.
 * q, k, v, o, dO : bf16 [B,H,N,d] (read; o and lse are the forward's outputs for the same
 * q, k, v, scale, causal);  workspace : fa_bwd_workspace_bytes(...) bytes of scratch, contents
 * undefined on entry and on exit. d in {64, 128}; any N >= 1. */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
           const float* lse, float* dq, void* dk, void* dv, int B, int H, int N, int d,
           float scale, int causal, void* workspace, fa_stream_t stream);

/* Block-sparse backward ("FlashAttention: IOを意識した..." (xyznot.com), "拡張: Block-Sparse
 * FlashAttention": the tile mask skips the same tiles in the backward). Same arguments, results
 * and workspace as fa_bwd, plus block_mask: the DEVICE uint8 [T][T] tile mask (T = ceil(N/128),
 * row = query tile) the forward used, combined with the causal mask when causal != 0. o and lse
 * must come from fa_fwd_blocksparse with the same mask. A key tile that no query tile visits gets
 * dK = dV = 0. T <= 2048 (FA_ERR_UNSUPPORTED above). */
int fa_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o,
                       const void* dO, const float* lse, float* dq, void* dk, void* dv, int B,
                       int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                       void* workspace, fa_stream_t stream);

/* Bytes of device scratch built into the library for fa_bwd_noalloc (per device). */
#define FA_NOALLOC_SCRATCH_BYTES (4u << 20)

/* fa_bwd without a workspace argument, for callers that cannot allocate device memory (a plugin
 * whose host gives it only its input and output buffers, a runtime that forbids cudaMalloc
 * while it serves). The pages have no counterpart of this entry point.
 * Same arguments, results and errors as fa_bwd, minus `workspace`: the scratch comes from a
 * FA_NOALLOC_SCRATCH_BYTES array of device memory that every device holds from the moment the
 * library's module is loaded on it until the process exits. fa_bwd's argument checks run first,
 * in its order (so a bad argument gets the same status from both); then problems whose
 * fa_bwd_workspace_bytes(B, H, N, d) exceeds the array are rejected with FA_ERR_SCRATCH_LIMIT,
 * before anything is enqueued. With B = H = 1, 4 MiB covers N up to 58240 at d = 64 and up to
 * 524160 at d = 128.
 * Allocates nothing: no cudaMalloc/cudaFree or allocating library call. The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture. All calls on a device share the one array and
 * it keeps the last call's contents (none needs clearing); calls whose kernels overlap on the GPU
 * (other streams, other host threads) race on it and must be serialised by the caller. */
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                   const float* lse, float* dq, void* dk, void* dv, int B, int H, int N, int d,
                   float scale, int causal, fa_stream_t stream);

/* Decoding attention ("3 · FlashAttention", 3.6 "L'attention en décodage"; Flash-Decoding in
 * 3.7): Nq (1 .. 8) new query rows per head attend to all Nk keys of that head (no mask):
 *     o = softmax(scale * q K^T) V,   lse = log sum_j exp(scale * q.k_j).
 * q, o : bf16 [B,H,Nq,d];  k, v : bf16 [B,H,Nk,d];  lse : fp32 [B,H,Nq] (all DEVICE pointers,
 * 16-byte aligned, caller-owned; q, k, v read, o and lse written). d in {64, 128}; Nk >= 1.
 * The work is a matrix-vector product bound by HBM bandwidth. The key blocks of all heads (128
 * keys at d = 128, 256 at d = 64) are split into n_ctas equal contiguous ranges streamed by
 * separate CTAs (a range may cut a head and span several), each block's products on the tensor
 * cores with the keys on the accumulator's rows (S^T = K q^T, O^T += V^T P^T, the query rows
 * zero-padded to 16); the pieces of each head are merged with the softmax statistics merge by a
 * second kernel, launched as a programmatic dependent of the first.
 * n_ctas = 0 takes as many CTAs as the device holds at once (fa_decode_ctas); 1 .. 1024 forces
 * the count (capped at the number of key blocks). `workspace`: fa_decode_workspace_bytes(...)
 * bytes of device scratch, contents undefined on entry and on exit. Errors: FA_ERR_INVALID_ARG
 * (null pointer, bad size or scale, n_ctas out of range), FA_ERR_UNSUPPORTED (Nq > 8, d),
 * FA_ERR_MISALIGNED, FA_ERR_TOO_LARGE, FA_ERR_NO_DEVICE, FA_ERR_CUDA; all before any launch. */
int fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int Nq, int Nk, int d, float scale, int n_ctas, void* workspace,
              fa_stream_t stream);

/* The CTA count fa_decode uses for n_ctas = 0 on the current device; 0 for invalid sizes or
 * without a usable device. */
int fa_decode_ctas(int B, int H, int Nq, int Nk, int d);

/* Bytes of workspace fa_decode needs for any n_ctas: (min(B*H*ceil(Nk/K), 1024) + B*H) pieces
 * of Nq rows, K the keys per block (128 at d = 128, 256 at d = 64), each row d + 1 floats (the
 * piece's normalised output and log-sum-exp); 0 for invalid sizes. */
size_t fa_decode_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/* Diagnostic, with no counterpart on the pages: launches one CTA whose thread waits on an
 * on-chip barrier that nothing ever arrives at, bounded by timeout_us (1 .. 10^7 microseconds).
 * The wait gives up, records FA_ERR_DEVICE_TIMEOUT in the device error word and the kernel
 * returns: a stuck pipeline surfaces as a status (via fa_check_device_error), not as a hang,
 * and the CUDA context stays usable. */
int fa_selftest_wait_timeout(unsigned timeout_us, fa_stream_t stream);

/* Synchronises `stream`, then reads and clears the device error word of the current device.
 * Returns FA_OK, FA_ERR_DEVICE_TIMEOUT (a kernel gave up on a barrier; its outputs are invalid),
 * or FA_ERR_CUDA if the synchronisation itself failed. */
int fa_check_device_error(fa_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* fa_status_string(int status);

/* ABI version: (major << 16) | minor. Major 2: fa_fwd_blocksparse takes a causal flag; minor 1:
 * fa_decode; minor 2: fa_bwd_blocksparse; minor 3: fa_fwd_fp32_fa1; minor 4:
 * fa_bwd_workspace_bytes depends on d (8 bytes per row at d = 128); minor 5: fa_fwd_fp8;
 * minor 6: fa_set_exp2_emulation, fa_get_exp2_emulation; minor 7: fa_decode on the tensor cores,
 * fa_decode_workspace_bytes counted with its blocks; minor 8: fa_bwd_workspace_bytes adds the
 * work counters of the backward kernel (4 * (1 + B*H) bytes, rounded up to 16). */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
