/*
 * attn_bwd.h -- C ABI of the GB300 (sm_103a) attention backward pass.
 *
 * The operation (WGSL page "ferrotensor-backend flash_attention_v2_backward.wgsl",
 * header comment and entry points flash_bwd_dq / flash_bwd_dk_dv; the Metal page
 * "rustytorch flash_attention_backward_dq.metal" is its [B,H,S,D] causal-MHA
 * special case):
 *
 *   s_ij    = scale * Q_i . K_j + mask_ij
 *   P_ij    = exp(s_ij - LSE_i)   on visible, non-hard pairs; 0 otherwise
 *   Delta_i = dO_i . O_i
 *   dS_ij   = P_ij * (M_ij * (dO_i . V_j) - Delta_i)
 *   dQ_i    = scale * sum_j dS_ij K_j
 *   dK_j    = scale * sum_i dS_ij Q_i      (summed over the query heads that
 *   dV_j    = sum_i P_ij M_ij dO_i          share the KV head: GQA)
 *
 * Conventions shared by every entry point:
 *  - All pointers are DEVICE pointers unless stated otherwise.  The caller
 *    owns every buffer and the stream; the library allocates nothing and keeps
 *    no state besides one device error word.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream).  The return value reports argument validation and
 *    launch errors only.  A device-side failure (a bounded wait that ran out)
 *    is reported by attn_bwd_check_device_error() after the stream has been
 *    synchronised.
 *  - Outputs are overwritten, not accumulated.
 *  - On any non-OK return nothing has been enqueued, except for
 *    ATTN_ERR_CUDA, which may leave some of the launches enqueued.
 */
#ifndef ATTN_BWD_H_
#define ATTN_BWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID = -1,     /* bad argument (sizes, pointers, probabilities) */
  ATTN_ERR_UNSUPPORTED = -2, /* valid but not implemented (e.g. head_dim 96) */
  ATTN_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed */
  ATTN_ERR_TIMEOUT = -4,     /* a kernel's bounded wait ran out (device error word) */
  ATTN_ERR_WORKSPACE = -5,   /* workspace missing, too small or misaligned */
  ATTN_ERR_SCRATCH_LIMIT = -6 /* problem needs more than the library's fixed scratch array */
} attn_status;

typedef enum {
  ATTN_LAYOUT_BHSD = 0, /* Metal page: Q,O,dO,dQ [B,H,Sq,D]; K,V,dK,dV [B,Hkv,Sk,D] */
  ATTN_LAYOUT_BSHD = 1  /* WGSL page:  Q,O,dO,dQ [B,Sq,H,D]; K,V,dK,dV [B,Sk,Hkv,D] */
} attn_layout;

typedef enum {
  ATTN_F32 = 0, /* fp32 tensors, TF32 tensor-core products, fp32 accumulation */
  ATTN_BF16 = 1 /* bf16 Q,K,V,O,dO,dQ,dK,dV; fp32 LSE, mask, accumulation */
} attn_dtype;

/*
 * Problem statement; mirrors the WGSL page's FlashBwdParams uniform plus the
 * tensor layout and dtype (which that page fixes implicitly).
 *   batch, num_heads (query heads), num_kv_heads (num_heads % num_kv_heads == 0;
 *     query head h uses KV head h / (num_heads / num_kv_heads)),
 *   seq_q, seq_k >= 1, head_dim in {64, 128},
 *   scale: multiplies Q.K before the mask is added,
 *   dropout_prob in [0, 1); seed: 64-bit key of the dropout generator,
 *   causal (0/1), causal_offset >= 0 (query i sits at position i + causal_offset),
 *   window: 0 = off, else a key is visible only if |i + causal_offset - j| < window,
 *   has_mask (0/1) and the mask's element strides (stride_h = 0 broadcasts over heads).
 * Visibility (fab2_visible): qa = i + causal_offset; visible iff
 *   (!causal || j <= qa) && (window == 0 || |qa - j| < window).
 * A pair is hard-masked when mask_ij <= -1e30 (the page's FAB_MASKED sentinel);
 * hard and invisible pairs carry P = 0.
 */
typedef struct {
  int32_t batch;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t seq_q;
  int32_t seq_k;
  int32_t head_dim;
  float scale;
  float dropout_prob;
  uint64_t seed;
  int32_t causal;
  int32_t causal_offset;
  int32_t window;
  int32_t has_mask;
  int64_t mask_stride_b;
  int64_t mask_stride_h;
  int64_t mask_stride_q;
  int64_t mask_stride_k;
  int32_t layout; /* attn_layout */
  int32_t dtype;  /* attn_dtype */
  int32_t deterministic; /* 0/1: dQ reproducible bit for bit (see attn_bwd) */
} attn_bwd_params;

/*
 * Bytes of device workspace attn_bwd needs for `p` (0 only if p is invalid).
 * Holds per-row Delta and LSE*log2(e) and, for bf16, the fp32 dQ accumulator;
 * with p->deterministic also one fp32 dQ slice per key tile,
 * ceil(seq_k / key tile) * batch * num_heads * seq_q * head_dim * 4 bytes.
 */
size_t attn_bwd_workspace_size(const attn_bwd_params* p);

/*
 * The attention backward pass (both WGSL passes, fused the GB300 way).
 *   Q, O, dO: query-side tensors in p->layout, p->dtype.
 *   K, V: key-side tensors in p->layout, p->dtype.
 *   LSE: fp32 [B, H, Sq], natural-log log-sum-exp of each row's scores from the
 *        forward pass; a row with no probability mass may hold any value
 *        (the WGSL page stores 3e38) -- its gradients come out as 0.
 *        NULL: the pass recomputes it first (attn_bwd_lse, written into the
 *        workspace), as the WGSL page's flash_bwd_dq does in its sweep 1.
 *   mask: fp32 additive mask addressed with p->mask_stride_*; NULL iff !has_mask.
 *   dQ (query-side), dK, dV (key-side): outputs, overwritten.  Keys that no
 *        query sees get dK = dV = 0.
 *   workspace: device memory of >= attn_bwd_workspace_size(p) bytes, 256-byte
 *        aligned; its contents on entry do not matter.
 * Every tensor pointer must be 16-byte aligned (TMA).  Tensors are dense in the
 * stated layout.  By default dQ accumulation uses fp32 atomics, so dQ can
 * differ in the last bits from run to run; dK and dV are deterministic.  With
 * p->deterministic every key tile writes its dQ contribution to its own
 * workspace slice and a final kernel sums the slices in key-tile order (the
 * WGSL page's dQ pass is atomic-free for the same reason), so dQ is the same
 * bit for bit on every run, at the cost of that workspace and its traffic.
 * Errors: ATTN_ERR_INVALID (null/misaligned pointer, bad sizes, bad dropout_prob,
 * mask pointer/has_mask mismatch), ATTN_ERR_UNSUPPORTED (head_dim), ATTN_ERR_WORKSPACE,
 * ATTN_ERR_CUDA.
 */
attn_status attn_bwd(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                     const void* O, const void* dO, const float* LSE, const float* mask,
                     void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                     void* stream);

/*
 * attn_bwd as three stages, for callers that want to schedule or time them
 * separately (attn_bwd == prepare, tiles, finish on one stream; same
 * arguments and rules as attn_bwd):
 *  attn_bwd_prepare  per-row Delta_i = dO_i . O_i (the Metal page's
 *                    "D = rowsum(dO * O)") and LSE * log2(e) into the
 *                    workspace and zeroes the fp32 dQ accumulator (fp32:
 *                    dQ itself).
 *  attn_bwd_tiles    the fused tile kernel: recomputes P, forms dS and
 *                    produces dK, dV and the dQ accumulation.
 *  attn_bwd_finish   bf16: converts the fp32 dQ accumulator to dQ; with
 *                    p->deterministic (either dtype): sums the per-key-tile
 *                    dQ slices in key-tile order into dQ.
 */
attn_status attn_bwd_prepare(const attn_bwd_params* p, const void* Q, const void* K,
                             const void* O, const void* dO, const float* LSE, void* dQ,
                             void* workspace, size_t workspace_bytes, void* stream);
/* (attn_bwd_prepare needs a non-NULL LSE; only attn_bwd recomputes it.) */
attn_status attn_bwd_tiles(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                           const void* dO, const float* mask, void* dQ, void* dK, void* dV,
                           void* workspace, size_t workspace_bytes, void* stream);
attn_status attn_bwd_finish(const attn_bwd_params* p, void* dQ, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Row log-sum-exp of the scores (WGSL page "flash_attention_v2_backward.wgsl",
 * flash_bwd_dq, sweep 1), for callers that did not keep the forward's LSE:
 *   LSE_i = log sum_j exp(s_ij)  over the visible keys j with mask_ij > -1e30,
 *   s_ij  = scale * Q_i . K_j + mask_ij,
 * and 3e38 for a row with no such key.  Dropout does not enter (the forward's
 * softmax normaliser is taken before dropout).
 *   Q, K: as for attn_bwd (p->layout, p->dtype); fp32 inputs are multiplied
 *        as TF32, the precision of the backward's own score product.
 *   mask: as for attn_bwd; NULL iff !has_mask.
 *   LSE:  fp32 [B, H, Sq], written (every row).
 * Device pointers, 16-byte aligned; one kernel on `stream`, no workspace.
 * Errors: ATTN_ERR_INVALID, ATTN_ERR_UNSUPPORTED (head_dim), ATTN_ERR_CUDA.
 */
attn_status attn_bwd_lse(const attn_bwd_params* p, const void* Q, const void* K,
                         const float* mask, float* LSE, void* stream);

/*
 * Fused forward pass, producing the backward's inputs on the GPU with the same
 * conventions (the WGSL page's forward is referenced by its backward but not
 * printed; read as the function whose gradients attn_bwd computes):
 *   s_ij  = scale * Q_i . K_j + mask_ij   on visible pairs with mask_ij > -1e30
 *   LSE_i = log sum_j exp(s_ij)           (3e38 for a row with no such pair)
 *   O_i   = sum_j exp(s_ij - LSE_i) M_ij V_j
 * with M the dropout multiplier of attn_bwd (same Philox4x32-10 stream, keep
 * mask identical to attn_dropout_keep_mask), and O_i = 0 for an empty row.
 *   Q, K, V: p->layout, p->dtype; fp32 inputs are multiplied as TF32.
 *   mask: as for attn_bwd.  O: p->layout, p->dtype (written).  LSE: fp32
 *   [B, H, Sq] (written).  workspace: >= attn_fwd_workspace_size(p) bytes,
 *   256-byte aligned (not written: the forward needs no scratch; the
 *   argument is kept so that callers need not change if it ever does).
 * Device pointers, 16-byte aligned.  p->deterministic is ignored (the forward
 * has no atomics).  Errors as for attn_bwd.
 */
size_t attn_fwd_workspace_size(const attn_bwd_params* p);
attn_status attn_fwd(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                     const float* mask, void* O, float* LSE, void* workspace,
                     size_t workspace_bytes, void* stream);

/*
 * Decode (one query per head) backward, pass 1 of the decode page
 * ("rullama attention_backward_dq.wgsl"): probabilities are given and the
 * scores were unscaled, kv = h / (n_heads / n_kv_heads):
 *   d_probs_j  = d_out_h . v_hist[j, kv]
 *   sum_pd     = sum_j probs_hj d_probs_j
 *   d_scores_j = probs_hj (d_probs_j - sum_pd)
 *   d_q_h      = sum_j d_scores_j k_hist[j, kv]
 * Batched over num_seqs independent sequences, all fp32:
 *   k_hist, v_hist [num_seqs, history_len, n_kv_heads, head_dim]
 *   probs, d_scores [num_seqs, n_heads, history_len]
 *   d_out, d_q      [num_seqs, n_heads, head_dim]
 * head_dim is 64, 128 or 256; n_heads % n_kv_heads == 0 and n_heads /
 * n_kv_heads is 1, 2, 4, 8 or 16; history_len >= 1.  Two kernels on `stream`
 * (a V pass, then a K pass that may start while the first finishes); the
 * result does not depend on timing.
 * workspace: >= attn_bwd_decode_workspace_size(p) bytes (256-byte aligned).
 */
typedef struct {
  int32_t num_seqs;
  int32_t n_heads;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t history_len;
} attn_bwd_decode_params;

size_t attn_bwd_decode_workspace_size(const attn_bwd_decode_params* p);

attn_status attn_bwd_decode(const attn_bwd_decode_params* p, const float* k_hist,
                            const float* v_hist, const float* probs, const float* d_out,
                            float* d_scores, float* d_q, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * Decode backward, pass 2: the gradients of the history.  The decode page's
 * pass 1 stages d_scores for a pass 2 that also takes the queries q (that
 * file is not on the pages); read as the gradients of the page's forward
 * (out_h = sum_j probs_hj v_hist[j, kv], unscaled scores q_h . k_hist[j, kv]):
 *   d_k_hist[j, kv] = sum_{h of kv} d_scores_hj q_h
 *   d_v_hist[j, kv] = sum_{h of kv} probs_hj d_out_h
 *   q, d_out           [num_seqs, n_heads, head_dim]
 *   probs, d_scores    [num_seqs, n_heads, history_len]   (d_scores from attn_bwd_decode)
 *   d_k_hist, d_v_hist [num_seqs, history_len, n_kv_heads, head_dim]  (written, every element)
 * Same parameter rules as attn_bwd_decode; device pointers, 16-byte aligned;
 * no workspace; one kernel on `stream`.  Errors: ATTN_ERR_INVALID /
 * ATTN_ERR_UNSUPPORTED for the parameters or pointers, ATTN_ERR_CUDA if the
 * launch fails.
 */
attn_status attn_bwd_decode_kv(const attn_bwd_decode_params* p, const float* q,
                               const float* probs, const float* d_out, const float* d_scores,
                               float* d_k_hist, float* d_v_hist, void* stream);

/*
 * attn_bwd_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point.  Some callers cannot give the
 * library a workspace: code that runs where no allocator is available or
 * allowed -- a plugin interface that only passes input and output tensors, a
 * process whose device memory is planned up front and may not grow, a
 * real-time path where cudaMalloc's implicit synchronisation and failure modes
 * are not acceptable.  This variant takes the same inputs and outputs as
 * attn_bwd_decode but no workspace; it calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Scratch: the partial sums go to one fixed array of
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES (8 MiB) of device memory inside the
 * library; every GPU that loads the library keeps that array until the
 * process exits.  The array must hold the partial sums of at least one
 * history split, about num_seqs * n_heads * (head_dim + 8) floats plus one
 * counter per (sequence, KV head) pair (e.g. 64 sequences x 8 heads x
 * head_dim 256: 0.5 MiB); larger problems are rejected with
 * ATTN_ERR_SCRATCH_LIMIT.  When the usual number of splits does not fit,
 * fewer are used, so results can differ from attn_bwd_decode in the last bits.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current, and again after the device's context
 * has been replaced, e.g. by cudaDeviceReset): make that first call before
 * capturing the stream into a CUDA graph.  All calls share the one array and nothing in
 * it is cleared between calls (each call rewrites every value it reads), so
 * calls that can overlap on the GPU -- on different streams or from different
 * host threads -- race; the caller must order them.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (8u << 20)
attn_status attn_bwd_decode_noalloc(const attn_bwd_decode_params* p, const float* k_hist,
                                    const float* v_hist, const float* probs, const float* d_out,
                                    float* d_scores, float* d_q, void* stream);

/*
 * Writes the dropout keep mask of slice (b, h) as bytes keep[i * seq_k + j]
 * (1 = kept, 0 = dropped), into a device buffer of seq_q * seq_k bytes.  Uses
 * the same device generator as attn_bwd: Philox4x32-10 (Salmon et al., SC'11)
 * with key (seed lo, seed hi), counter (i >> 2, j, b * num_heads + h, 0),
 * word i & 3, kept iff word >= min(floor(p * 2^32), 2^32 - 1).
 */
attn_status attn_dropout_keep_mask(const attn_bwd_params* p, int32_t b, int32_t h,
                                   uint8_t* keep, void* stream);

/*
 * Host-side tile planner (no GPU needed): the half-open range
 * [*q_begin, *q_end) of queries that can see any key in [k0, k1] under the
 * causal / causal_offset / window rules (the dK/dV pass's query range).
 */
attn_status attn_bwd_query_range(const attn_bwd_params* p, int32_t k0, int32_t k1,
                                 int32_t* q_begin, int32_t* q_end);

/*
 * Synchronises nothing: reads (and, if clear_it, resets) the device error
 * word with a blocking copy on the current device.  Returns ATTN_OK or
 * ATTN_ERR_TIMEOUT.  Call after synchronising the streams that ran kernels.
 * The word is a __device__ variable of the library; its address is looked up
 * per device and again whenever the device's context has changed (after
 * cudaDeviceReset the word starts at 0 in the new context).
 */
attn_status attn_bwd_check_device_error(int32_t clear_it);

/*
 * Tensor-core self test: C[M, N] = A[M, K] * B[N, K]^T computed by one CTA
 * with tcgen05.mma from operands staged in 128-byte-swizzled shared memory.
 *   dtype: ATTN_F32 (TF32) or ATTN_BF16; A and B are fp32 or bf16 row-major
 *   host layouts [M][K] / [N][K]; a_mn / b_mn = 1 stage the operand in
 *   MN-major form (rows along K) instead of K-major; a TF32 MN-major operand
 *   uses the 128-byte swizzle of 32-byte atoms, the layout the tile kernels
 *   read Q, dO, K and V in.
 *   a_tmem = 1 takes A from tensor memory instead (row m in the lane of
 *   accumulator row m, K along 32-bit columns, two bf16 per column).
 *   M in {64, 128}, N in {32, 64, 128, 256} (N <= 256), K a multiple of the
 *   tile width (32 fp32 / 64 bf16) and <= 128.
 *   tmem_dump (optional, fp32 [128][N]): raw accumulator contents, lane-major.
 */
attn_status attn_selftest_mma(int32_t dtype, int32_t M, int32_t N, int32_t K, int32_t a_mn,
                              int32_t b_mn, int32_t a_tmem, const void* A, const void* B,
                              float* C, float* tmem_dump, void* stream);

/*
 * Failure-path self test: enqueues one tiny kernel whose single wait can never
 * be satisfied (an mbarrier nothing arrives on).  The bounded wait every
 * kernel of the library uses gives up after about a second and raises the
 * device error word; after synchronising, attn_bwd_check_device_error reports
 * ATTN_ERR_TIMEOUT (and clears the word if asked), and the context stays
 * usable.  No trap, no fault, no hang.
 */
attn_status attn_selftest_wait_timeout(void* stream);

/* Human-readable name of a status code (static string). */
const char* attn_status_string(attn_status s);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H_ */
