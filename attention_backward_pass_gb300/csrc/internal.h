// Internal declarations shared by the host dispatcher and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "attn_bwd.h"

namespace attnbwd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBlockN = 128;   // keys per CTA of the dK/dV kernel (MMA M = 128)
constexpr int kRowPad = 128;   // per-row workspace arrays are padded to this many rows

// Everything a tile kernel needs besides tensor maps (plain values, by value).
struct TileArgs {
  int B, H, Hkv, Sq, Sk, D;
  int group;          // H / Hkv
  int sq_pad;         // per-(b,h) row stride of the Delta / LSE2 workspace arrays
  int layout;         // 0 BHSD, 1 BSHD
  float scale;        // multiplies Q.K
  float scale_log2e;  // scale * log2(e)
  int causal;
  long long causal_offset;
  long long window;
  int has_mask;
  long long msb, msh, msq, msk;
  const float* mask;
  int dropout;            // 0 / 1
  uint32_t drop_threshold;  // keep iff philox word >= threshold
  float drop_inv_keep;      // 1 / (1 - p)
  uint32_t seed_lo, seed_hi;
  const float* lse2;   // [B*H][sq_pad]  -LSE * log2(e), -inf in padding rows
  const float* delta;  // [B*H][sq_pad]  rowsum(dO * O), 0 in padding rows
  float* dq_acc;       // fp32 dQ accumulator, same layout as dQ (dQ itself for fp32);
                       // deterministic: the per-key-tile slices [n_kv_tiles*B][H][Sq][D]
  int det;             // 1: store dQ slices instead of adding into dq_acc
  void* dK;
  void* dV;
  const void* V;       // V itself (configurations that load it into tensor memory directly)
  int n_kv_tiles;
  int pdl;             // launched as a programmatic dependent of the prepare kernel
  unsigned int* err;
};

// Element offset of row (b, h, i) of a [B,H,S,D] or [B,S,H,D] tensor.
__host__ __device__ __forceinline__ long long row_offset(int layout, int b, int h, int i, int H,
                                                        int S, int D) {
  return layout == 0 ? ((long long)(b * (long long)H + h) * S + i) * D
                     : (((long long)b * S + i) * H + h) * D;
}

// Queries [q_begin, q_end) that can see at least one key of [k0, k1] under the
// causal / causal_offset / window rules (WGSL page, flash_bwd_dk_dv query
// range, restated): causal needs q + off >= k0; the window needs
// q + off < k1 + window and, without causal, q + off > k0 - window.
__host__ __device__ __forceinline__ void query_range(int Sq, int causal, long long off,
                                                     long long window, long long k0,
                                                     long long k1, int* qb, int* qe) {
  long long b = 0, e = Sq;
  if (causal) b = k0 - off > 0 ? k0 - off : 0;
  if (window > 0) {
    long long hi = k1 + window - off;
    if (hi < e) e = hi;
    if (!causal) {
      long long lo = k0 - window - off + 1;
      if (lo > b) b = lo;
    }
  }
  if (e < 0) e = 0;
  if (b > e) b = e;
  *qb = (int)b;
  *qe = (int)e;
}

unsigned int* device_error_word();
// Driver context current on this thread (opaque handle; nullptr if none).
void* current_context();

attn_status selftest_wait_launch(cudaStream_t stream);
attn_status selftest_mma_launch(int dtype, int M, int N, int K, int a_mn, int b_mn, int a_tmem,
                                const void* A, const void* B, float* C, float* dump,
                                cudaStream_t stream);

// Delta / LSE2 rows and zeroing of the dQ accumulator.
cudaError_t launch_prep(const attn_bwd_params& p, const void* O, const void* dO, const float* LSE,
                        float* delta, float* lse2, int sq_pad, float* dq_acc,
                        cudaStream_t stream);
cudaError_t launch_dq_convert(const attn_bwd_params& p, const float* dq_acc, void* dQ,
                              cudaStream_t stream);
// Deterministic dQ: dQ = sum over key tiles kt (ascending) of slice kt, over
// the query tiles the dK/dV CTA of kt visited (block sizes bn x bm).
cudaError_t launch_dq_reduce(const attn_bwd_params& p, const float* slices, void* dQ, int bn,
                             int bm, cudaStream_t stream);

struct TileMaps {
  CUtensorMap q, k, v, dout;  // natural [.., S, .., D] tensors
  CUtensorMap qt, kt, dot;    // fp32: Q, K, dO again, 32-byte-atom swizzle (MN-major reads)
  CUtensorMap dq;             // fp32 dQ accumulator (reduce-add target)
  CUtensorMap dk, dv;         // outputs, the key tiles' layout (TMA stores)
};
// after_prepare: programmatic dependent launch behind the prepare kernel
cudaError_t launch_dkdv(const attn_bwd_params& p, const TileMaps& maps, const TileArgs& a,
                        cudaStream_t stream, bool after_prepare);
int dkdv_block_m(int dtype, int head_dim);
int dkdv_block_n(int dtype, int head_dim);
int dkdv_dq_box_d(int dtype, int head_dim);  // head-dim columns per dQ reduce box


uint32_t dropout_threshold(float prob);
cudaError_t launch_dropout_mask(const attn_bwd_params& p, int b, int h, uint8_t* keep,
                                cudaStream_t stream);

cudaError_t launch_decode(const attn_bwd_decode_params& p, const float* k_hist,
                          const float* v_hist, const float* probs, const float* d_out,
                          float* d_scores, float* d_q, float* partials, int n_split,
                          cudaStream_t stream);
int decode_num_splits(const attn_bwd_decode_params& p);
cudaError_t launch_decode_kv(const attn_bwd_decode_params& p, const float* q, const float* probs,
                             const float* d_out, const float* d_scores, float* d_k, float* d_v,
                             cudaStream_t stream);
CUresult make_f32_map(CUtensorMap* m, const void* base, int rank, const long long* dims,
                      const int* box, bool swizzle128);
size_t decode_partials_floats(const attn_bwd_decode_params& p, int n_split);

// Row log-sum-exp (the WGSL page's sweep 1) on the tensor cores.
struct LseArgs {
  int B, H, group, Sq, Sk, sq_pad;
  float scale_log2e;  // scale * log2(e)
  int causal;
  long long causal_offset, window;
  int has_mask, mask_vec;  // mask_vec: rows are contiguous and 16-byte aligned
  long long msb, msh, msq, msk;
  const float* mask;
  int out_mode;  // 0: LSE [B*H][Sq] (3e38 for empty rows); 1: -LSE*log2(e) [B*H][sq_pad], -inf
  float* out;
  unsigned int* err;
};
// Fused forward (O and LSE) on the tensor cores.
struct FwdArgs {
  int B, H, group, Sq, Sk, layout;
  float scale_log2e;  // scale * log2(e)
  int causal;
  long long causal_offset, window;
  int has_mask, mask_vec;  // mask_vec: rows are contiguous and 16-byte aligned
  long long msb, msh, msq, msk;
  const float* mask;
  int dropout;              // 0 / 1
  uint32_t drop_threshold;  // keep iff philox word >= threshold
  float drop_inv_keep;      // 1 / (1 - p)
  uint32_t seed_lo, seed_hi;
  void* O;     // [B,H,Sq,D] or [B,Sq,H,D], the problem's dtype
  float* LSE;  // [B*H][Sq]
  unsigned int* err;
};
// tq: Q, boxes of 128 rows; tk: K and tv: V, boxes of fwd_block_n rows (fp32
// V in the 128-byte swizzle of 32-byte atoms, read MN-major).
int fwd_block_n(int dtype, int head_dim);
cudaError_t launch_fwd(const attn_bwd_params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdArgs& a, cudaStream_t stream);

constexpr float kHardMask = -1.0e30f;     // a mask value at or below this hides the pair
constexpr float kEmptyRowLse = 3.0e38f;   // LSE of a row with no probability mass
// tq: Q in the problem's layout, boxes of 128 rows; tk: K, boxes of
// lse_block_n(dtype, head_dim) rows.
int lse_block_n(int dtype, int head_dim);
cudaError_t launch_lse(const attn_bwd_params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const LseArgs& a, cudaStream_t stream);

}  // namespace attnbwd
