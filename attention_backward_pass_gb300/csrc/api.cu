// Host side of the C ABI: argument validation, workspace carving, TMA
// descriptor encoding and kernel launches.  Every entry point only enqueues
// work on the caller's stream; nothing here allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "attn_bwd.h"
#include "internal.h"

namespace attnbwd {

namespace {

__device__ unsigned int g_error_word_storage = 0u;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned int* g_err_ptr[kMaxDevices] = {nullptr};
void* g_err_ctx[kMaxDevices] = {nullptr};  // context the cached address belongs to

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int round_up(int x, int m) { return (x + m - 1) / m * m; }

attn_status validate(const attn_bwd_params* p) {
  if (!p) return ATTN_ERR_INVALID;
  if (p->batch < 1 || p->num_heads < 1 || p->num_kv_heads < 1 || p->seq_q < 1 || p->seq_k < 1)
    return ATTN_ERR_INVALID;
  if (p->num_heads % p->num_kv_heads != 0) return ATTN_ERR_INVALID;
  if (p->head_dim != 64 && p->head_dim != 128) return ATTN_ERR_UNSUPPORTED;
  if (p->dtype != ATTN_F32 && p->dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  if (p->layout != ATTN_LAYOUT_BHSD && p->layout != ATTN_LAYOUT_BSHD) return ATTN_ERR_INVALID;
  if (!(p->dropout_prob >= 0.f && p->dropout_prob < 1.f)) return ATTN_ERR_INVALID;
  if (!std::isfinite(p->scale)) return ATTN_ERR_INVALID;
  if (p->causal != 0 && p->causal != 1) return ATTN_ERR_INVALID;
  if (p->causal_offset < 0 || p->window < 0) return ATTN_ERR_INVALID;
  if (p->has_mask != 0 && p->has_mask != 1) return ATTN_ERR_INVALID;
  if (p->deterministic != 0 && p->deterministic != 1) return ATTN_ERR_INVALID;
  // row and element counts must fit the kernels' index arithmetic
  const long long rows_q = (long long)p->batch * p->num_heads * p->seq_q;
  const long long rows_k = (long long)p->batch * p->num_kv_heads * p->seq_k;
  if (rows_q * p->head_dim >= (1LL << 40) || rows_k * p->head_dim >= (1LL << 40))
    return ATTN_ERR_INVALID;
  if ((long long)p->seq_q + p->causal_offset >= (1LL << 31)) return ATTN_ERR_INVALID;
  if ((long long)p->batch * p->num_heads >= (1LL << 31) / 1024) return ATTN_ERR_INVALID;
  const long long kv_tiles = (p->seq_k + 63) / 64;  // smallest key tile
  if (kv_tiles * p->batch * p->num_kv_heads >= (1LL << 31)) return ATTN_ERR_INVALID;
  if (p->deterministic && kv_tiles * rows_q * p->head_dim >= (1LL << 40)) return ATTN_ERR_INVALID;
  return ATTN_OK;
}

// Workspace carve-up (each region 256-byte aligned):
//   delta, lse2   [B*H][sq_pad] fp32
//   dq_acc        fp32 dQ accumulator (bf16 only; fp32 accumulates in dQ)
//   dqp           deterministic dQ: one fp32 slice per key tile,
//                 [n_kv_tiles * B][H][Sq][D]
struct WsLayout {
  size_t delta, lse2, dq_acc, dqp, total;
  int sq_pad, sk_pad;
};

WsLayout ws_layout(const attn_bwd_params& p) {
  WsLayout w;
  w.sq_pad = round_up(p.seq_q, kRowPad);
  w.sk_pad = round_up(p.seq_k, kRowPad);
  const size_t rows = (size_t)p.batch * p.num_heads * w.sq_pad;
  const bool bf = p.dtype == ATTN_BF16;
  w.delta = 0;
  w.lse2 = align256(rows * 4);
  w.dq_acc = w.lse2 + align256(rows * 4);
  const size_t dq = bf ? align256((size_t)p.batch * p.num_heads * p.seq_q * p.head_dim * 4) : 0;
  w.dqp = w.dq_acc + dq;
  size_t dqp = 0;
  if (p.deterministic) {
    const size_t n_kt = (size_t)((p.seq_k + dkdv_block_n(p.dtype, p.head_dim) - 1) /
                                 dkdv_block_n(p.dtype, p.head_dim));
    dqp = align256(n_kt * p.batch * p.num_heads * p.seq_q * p.head_dim * 4);
  }
  w.total = w.dqp + dqp;
  return w;
}

// fp32 dQ accumulator in the problem's layout, unswizzled boxes of
// box_d x box_rows: the TMA reduce-add target of the tile kernel.
CUresult make_map_dq(CUtensorMap* m, void* base, int D, int S, int H, int B, int layout,
                     int box_d, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3];
  if (layout == ATTN_LAYOUT_BHSD) {
    strides[0] = (cuuint64_t)D * 4;
    strides[1] = (cuuint64_t)S * D * 4;
    strides[2] = (cuuint64_t)H * S * D * 4;
  } else {
    strides[0] = (cuuint64_t)H * D * 4;
    strides[1] = (cuuint64_t)D * 4;
    strides[2] = (cuuint64_t)S * H * D * 4;
  }
  cuuint32_t box[4] = {(cuuint32_t)box_d, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, base, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Natural [.., S, .., D] tensor as a whole-tile operand map.  The D columns
// are split into W-element column blocks (W = 128 bytes of elements) that
// form a dimension of their own, after the rows: dims {W, S, D / W, H, B}.
// One box {W, box_rows, D / W} then lands in shared memory as
// [D / W][box_rows][W], the column-block layout of the operand tiles, in a
// single copy (one copy per tile instead of one per column block: measured
// ~10 % faster for the fp32 D = 128 tile kernel, which issues several tile
// copies per query tile).  128-byte swizzle (K-major operand tiles); atom32
// (fp32 only): the 128-byte swizzle of 32-byte atoms, the layout of a TF32
// operand read MN-major.  fp32 tensors are fetched as TF32.
CUresult make_map(CUtensorMap* m, const void* base, int dtype, int D, int S, int H, int B,
                  int layout, int box_rows, bool atom32 = false) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return CUDA_ERROR_NOT_INITIALIZED;
  const int e = dtype == ATTN_BF16 ? 2 : 4;
  const int W = 128 / e;
  cuuint64_t dims[5] = {(cuuint64_t)W, (cuuint64_t)S, (cuuint64_t)(D / W), (cuuint64_t)H,
                        (cuuint64_t)B};
  cuuint64_t strides[4];  // bytes, dims 1..4
  if (layout == ATTN_LAYOUT_BHSD) {
    strides[0] = (cuuint64_t)D * e;
    strides[1] = 128;
    strides[2] = (cuuint64_t)S * D * e;
    strides[3] = (cuuint64_t)H * S * D * e;
  } else {
    strides[0] = (cuuint64_t)H * D * e;
    strides[1] = 128;
    strides[2] = (cuuint64_t)D * e;
    strides[3] = (cuuint64_t)S * H * D * e;
  }
  cuuint32_t box[5] = {(cuuint32_t)W, (cuuint32_t)box_rows, (cuuint32_t)(D / W), 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, dtype == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_TFLOAT32,
             5, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             atom32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

// Dense fp32 tensor of `rank` dimensions (dims[0] innermost and contiguous,
// each further dimension packed after the previous; base and dims[0] * 4
// 16-byte aligned), copied in boxes of box[] elements, plain or with the
// 128-byte swizzle.  Elements outside the tensor read as zero and are not
// written.
CUresult make_f32_map(CUtensorMap* m, const void* base, int rank, const long long* dims,
                      const int* box, bool swizzle128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  unsigned long long stride = 4;
  for (int i = 0; i < rank; ++i) {
    d[i] = (cuuint64_t)dims[i];
    bx[i] = (cuuint32_t)box[i];
    es[i] = 1;
    stride *= (unsigned long long)dims[i];
    if (i + 1 < rank) st[i] = (cuuint64_t)stride;
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, (cuuint32_t)rank, const_cast<void*>(base), d, st,
             bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Handle of the driver context current on this thread (nullptr if none or
// if the driver entry point is unavailable).  The device addresses of the
// library's __device__ variables belong to that context: after
// cudaDeviceReset the runtime creates a new primary context, in which they
// are loaded again at other addresses.
void* current_context() {
  using CtxGetCurrentFn = CUresult (*)(CUcontext*);
  static CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return reinterpret_cast<void*>(ctx);
}

unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev] || g_err_ctx[dev] != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_error_word_storage) != cudaSuccess) return nullptr;
    g_err_ptr[dev] = reinterpret_cast<unsigned int*>(ptr);
    g_err_ctx[dev] = current_context();  // the lookup created it if there was none
  }
  return g_err_ptr[dev];
}

}  // namespace attnbwd

using namespace attnbwd;

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device wait timed out";
    case ATTN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case ATTN_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed no-allocation scratch array";
  }
  return "unknown status";
}

size_t attn_bwd_workspace_size(const attn_bwd_params* p) {
  if (validate(p) != ATTN_OK) return 0;
  return ws_layout(*p).total;
}

namespace {

struct Plan {
  WsLayout wl;
  float *delta, *lse2, *dq_acc, *dqp;
};

attn_status make_plan(const attn_bwd_params* p, void* dQ, void* workspace, size_t workspace_bytes,
                      Plan* pl) {
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!dQ || !aligned16(dQ)) return ATTN_ERR_INVALID;
  pl->wl = ws_layout(*p);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
      workspace_bytes < pl->wl.total)
    return ATTN_ERR_WORKSPACE;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  pl->delta = reinterpret_cast<float*>(ws + pl->wl.delta);
  pl->lse2 = reinterpret_cast<float*>(ws + pl->wl.lse2);
  pl->dq_acc = p->dtype == ATTN_BF16 ? reinterpret_cast<float*>(ws + pl->wl.dq_acc)
                                     : reinterpret_cast<float*>(dQ);
  pl->dqp = reinterpret_cast<float*>(ws + pl->wl.dqp);
  return ATTN_OK;
}

bool all_aligned(std::initializer_list<const void*> ptrs) {
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return false;
  return true;
}

}  // namespace

namespace {

// Row log-sum-exp on the tensor cores, written either as LSE [B,H,Sq]
// (out_mode 0) or as -LSE*log2(e) into the workspace rows the tile kernel
// reads (out_mode 1, sq_pad rows per (b, h)).
attn_status run_lse(const attn_bwd_params* p, const void* Q, const void* K, const float* mask,
                    float* out, int out_mode, int sq_pad, cudaStream_t stream) {
  unsigned int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;
  CUtensorMap tq, tk;
  if (make_map(&tq, Q, p->dtype, p->head_dim, p->seq_q, p->num_heads, p->batch, p->layout,
               128) != CUDA_SUCCESS ||
      make_map(&tk, K, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch, p->layout,
               lse_block_n(p->dtype, p->head_dim)) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  LseArgs a;
  memset(&a, 0, sizeof(a));
  a.B = p->batch;
  a.H = p->num_heads;
  a.group = p->num_heads / p->num_kv_heads;
  a.Sq = p->seq_q;
  a.Sk = p->seq_k;
  a.sq_pad = sq_pad;
  a.scale_log2e = p->scale * kLog2e;
  a.causal = p->causal;
  a.causal_offset = p->causal_offset;
  a.window = p->window;
  a.has_mask = p->has_mask;
  a.msb = p->mask_stride_b;
  a.msh = p->mask_stride_h;
  a.msq = p->mask_stride_q;
  a.msk = p->mask_stride_k;
  a.mask = mask;
  a.mask_vec = p->has_mask && aligned16(mask) && a.msk == 1 && a.msq % 4 == 0 &&
               a.msh % 4 == 0 && a.msb % 4 == 0;
  a.out_mode = out_mode;
  a.out = out;
  a.err = err;
  return launch_lse(*p, tq, tk, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// attn_bwd_prepare without the LSE check: LSE == NULL leaves the workspace's
// -LSE*log2(e) rows as run_lse wrote them.
attn_status prepare_impl(const attn_bwd_params* p, const void* Q, const void* K, const void* O,
                         const void* dO, const float* LSE, void* dQ, void* workspace,
                         size_t workspace_bytes, void* stream_v) {
  Plan pl;
  attn_status st = make_plan(p, dQ, workspace, workspace_bytes, &pl);
  if (st != ATTN_OK) return st;
  if (!all_aligned({Q, K, O, dO})) return ATTN_ERR_INVALID;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  const cudaError_t e =
      launch_prep(*p, O, dO, LSE, pl.delta, pl.lse2, pl.wl.sq_pad, pl.dq_acc, stream);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

attn_status attn_bwd_prepare(const attn_bwd_params* p, const void* Q, const void* K,
                             const void* O, const void* dO, const float* LSE, void* dQ,
                             void* workspace, size_t workspace_bytes, void* stream_v) {
  const attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!LSE || !aligned16(LSE)) return ATTN_ERR_INVALID;
  return prepare_impl(p, Q, K, O, dO, LSE, dQ, workspace, workspace_bytes, stream_v);
}

attn_status attn_bwd_lse(const attn_bwd_params* p, const void* Q, const void* K,
                         const float* mask, float* LSE, void* stream) {
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!all_aligned({Q, K, LSE})) return ATTN_ERR_INVALID;
  if ((p->has_mask != 0) != (mask != nullptr)) return ATTN_ERR_INVALID;
  return run_lse(p, Q, K, mask, LSE, 0, 0, reinterpret_cast<cudaStream_t>(stream));
}

namespace {

// The tile stage.  after_prepare: launched right after this library's own
// prepare kernel on the same stream, so it may start while that kernel
// finishes (programmatic dependent launch; everything that reads the
// prepare's outputs waits for it first).  A direct attn_bwd_tiles call
// follows whatever the caller ran last and launches normally.
attn_status tiles_impl(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                       const void* dO, const float* mask, void* dQ, void* dK, void* dV,
                       void* workspace, size_t workspace_bytes, void* stream_v,
                       bool after_prepare) {
  Plan pl;
  attn_status st = make_plan(p, dQ, workspace, workspace_bytes, &pl);
  if (st != ATTN_OK) return st;
  if (!all_aligned({Q, K, V, dO, dK, dV})) return ATTN_ERR_INVALID;
  if ((p->has_mask != 0) != (mask != nullptr)) return ATTN_ERR_INVALID;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  unsigned int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;

  TileMaps maps;
  memset(&maps, 0, sizeof(maps));
  const int bm = dkdv_block_m(p->dtype, p->head_dim);
  const int bn = dkdv_block_n(p->dtype, p->head_dim);
  // fp32: the MN-major copies of Q, dO and K (GEMM3/4/5) come from the same
  // tensors, fetched with the 128-byte swizzle of 32-byte atoms
  if (p->dtype != ATTN_BF16 &&
      (make_map(&maps.qt, Q, p->dtype, p->head_dim, p->seq_q, p->num_heads, p->batch, p->layout,
                bm, true) != CUDA_SUCCESS ||
       make_map(&maps.dot, dO, p->dtype, p->head_dim, p->seq_q, p->num_heads, p->batch,
                p->layout, bm, true) != CUDA_SUCCESS ||
       make_map(&maps.kt, K, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch,
                p->layout, bn, true) != CUDA_SUCCESS))
    return ATTN_ERR_CUDA;
  if (make_map(&maps.q, Q, p->dtype, p->head_dim, p->seq_q, p->num_heads, p->batch, p->layout,
               bm) != CUDA_SUCCESS ||
      make_map(&maps.dout, dO, p->dtype, p->head_dim, p->seq_q, p->num_heads, p->batch,
               p->layout, bm) != CUDA_SUCCESS ||
      make_map(&maps.k, K, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch, p->layout,
               bn) != CUDA_SUCCESS ||
      make_map(&maps.v, V, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch, p->layout,
               bn) != CUDA_SUCCESS ||
      make_map(&maps.dk, dK, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch,
               p->layout, bn) != CUDA_SUCCESS ||
      make_map(&maps.dv, dV, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch,
               p->layout, bn) != CUDA_SUCCESS ||
      (p->deterministic
           ? make_map_dq(&maps.dq, pl.dqp, p->head_dim, p->seq_q, p->num_heads,
                         p->batch * ((p->seq_k + bn - 1) / bn), ATTN_LAYOUT_BHSD,
                         dkdv_dq_box_d(p->dtype, p->head_dim), bm)
           : make_map_dq(&maps.dq, pl.dq_acc, p->head_dim, p->seq_q, p->num_heads, p->batch,
                         p->layout, dkdv_dq_box_d(p->dtype, p->head_dim), bm)) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;

  TileArgs a;
  memset(&a, 0, sizeof(a));
  a.B = p->batch;
  a.H = p->num_heads;
  a.Hkv = p->num_kv_heads;
  a.Sq = p->seq_q;
  a.Sk = p->seq_k;
  a.D = p->head_dim;
  a.group = p->num_heads / p->num_kv_heads;
  a.sq_pad = pl.wl.sq_pad;
  a.layout = p->layout;
  a.scale = p->scale;
  a.scale_log2e = p->scale * kLog2e;
  a.causal = p->causal;
  a.causal_offset = p->causal_offset;
  a.window = p->window;
  a.has_mask = p->has_mask;
  a.msb = p->mask_stride_b;
  a.msh = p->mask_stride_h;
  a.msq = p->mask_stride_q;
  a.msk = p->mask_stride_k;
  a.mask = mask;
  a.dropout = p->dropout_prob > 0.f ? 1 : 0;
  a.drop_threshold = dropout_threshold(p->dropout_prob);
  a.drop_inv_keep = (float)(1.0 / (1.0 - (double)p->dropout_prob));
  a.seed_lo = (uint32_t)(p->seed & 0xFFFFFFFFu);
  a.seed_hi = (uint32_t)(p->seed >> 32);
  a.lse2 = pl.lse2;
  a.delta = pl.delta;
  a.dq_acc = p->deterministic ? pl.dqp : pl.dq_acc;
  a.det = p->deterministic;
  a.dK = dK;
  a.dV = dV;
  a.V = V;
  a.n_kv_tiles = (p->seq_k + bn - 1) / bn;
  a.err = err;
  if (launch_dkdv(*p, maps, a, stream, after_prepare) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace

attn_status attn_bwd_tiles(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                           const void* dO, const float* mask, void* dQ, void* dK, void* dV,
                           void* workspace, size_t workspace_bytes, void* stream_v) {
  return tiles_impl(p, Q, K, V, dO, mask, dQ, dK, dV, workspace, workspace_bytes, stream_v, false);
}

attn_status attn_bwd_finish(const attn_bwd_params* p, void* dQ, void* workspace,
                            size_t workspace_bytes, void* stream_v) {
  Plan pl;
  attn_status st = make_plan(p, dQ, workspace, workspace_bytes, &pl);
  if (st != ATTN_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  if (p->deterministic) {
    if (launch_dq_reduce(*p, pl.dqp, dQ, dkdv_block_n(p->dtype, p->head_dim),
                         dkdv_block_m(p->dtype, p->head_dim), stream) != cudaSuccess)
      return ATTN_ERR_CUDA;
  } else if (p->dtype == ATTN_BF16 &&
             launch_dq_convert(*p, pl.dq_acc, dQ, stream) != cudaSuccess) {
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

attn_status attn_bwd(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                     const void* O, const void* dO, const float* LSE, const float* mask,
                     void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes,
                     void* stream) {
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!all_aligned({Q, K, V, O, dO, dQ, dK, dV})) return ATTN_ERR_INVALID;
  if (LSE && !aligned16(LSE)) return ATTN_ERR_INVALID;
  if ((p->has_mask != 0) != (mask != nullptr)) return ATTN_ERR_INVALID;
  if (!LSE) {
    // no saved LSE: recompute it into the workspace rows the tiles read
    Plan pl;
    st = make_plan(p, dQ, workspace, workspace_bytes, &pl);
    if (st != ATTN_OK) return st;
    st = run_lse(p, Q, K, mask, pl.lse2, 1, pl.wl.sq_pad, reinterpret_cast<cudaStream_t>(stream));
    if (st != ATTN_OK) return st;
  }
  st = prepare_impl(p, Q, K, O, dO, LSE, dQ, workspace, workspace_bytes, stream);
  if (st != ATTN_OK) return st;
  st = tiles_impl(p, Q, K, V, dO, mask, dQ, dK, dV, workspace, workspace_bytes, stream, true);
  if (st != ATTN_OK) return st;
  return attn_bwd_finish(p, dQ, workspace, workspace_bytes, stream);
}

size_t attn_fwd_workspace_size(const attn_bwd_params* p) {
  if (validate(p) != ATTN_OK) return 0;
  return 256;  // not used: the forward needs no scratch
}

attn_status attn_fwd(const attn_bwd_params* p, const void* Q, const void* K, const void* V,
                     const float* mask, void* O, float* LSE, void* workspace,
                     size_t workspace_bytes, void* stream_v) {
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!all_aligned({Q, K, V, O, LSE})) return ATTN_ERR_INVALID;
  if ((p->has_mask != 0) != (mask != nullptr)) return ATTN_ERR_INVALID;
  const size_t need = attn_fwd_workspace_size(p);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return ATTN_ERR_WORKSPACE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  unsigned int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;
  const int bn = fwd_block_n(p->dtype, p->head_dim);
  CUtensorMap tq, tk, tv;
  if (make_map(&tq, Q, p->dtype, p->head_dim, p->seq_q, p->num_heads, p->batch, p->layout,
               128) != CUDA_SUCCESS ||
      make_map(&tk, K, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch, p->layout,
               bn) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  // V is read MN-major by O += P . V (fp32: in the 32-byte-atom swizzle)
  if (make_map(&tv, V, p->dtype, p->head_dim, p->seq_k, p->num_kv_heads, p->batch, p->layout, bn,
               p->dtype != ATTN_BF16) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  FwdArgs a;
  memset(&a, 0, sizeof(a));
  a.B = p->batch;
  a.H = p->num_heads;
  a.group = p->num_heads / p->num_kv_heads;
  a.Sq = p->seq_q;
  a.Sk = p->seq_k;
  a.layout = p->layout;
  a.scale_log2e = p->scale * kLog2e;
  a.causal = p->causal;
  a.causal_offset = p->causal_offset;
  a.window = p->window;
  a.has_mask = p->has_mask;
  a.msb = p->mask_stride_b;
  a.msh = p->mask_stride_h;
  a.msq = p->mask_stride_q;
  a.msk = p->mask_stride_k;
  a.mask = mask;
  a.mask_vec = p->has_mask && aligned16(mask) && a.msk == 1 && a.msq % 4 == 0 &&
               a.msh % 4 == 0 && a.msb % 4 == 0;
  a.dropout = p->dropout_prob > 0.f ? 1 : 0;
  a.drop_threshold = dropout_threshold(p->dropout_prob);
  a.drop_inv_keep = (float)(1.0 / (1.0 - (double)p->dropout_prob));
  a.seed_lo = (uint32_t)(p->seed & 0xFFFFFFFFu);
  a.seed_hi = (uint32_t)(p->seed >> 32);
  a.O = O;
  a.LSE = LSE;
  a.err = err;
  return launch_fwd(*p, tq, tk, tv, a, stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status validate_decode(const attn_bwd_decode_params* p) {
  if (!p) return ATTN_ERR_INVALID;
  if (p->num_seqs < 1 || p->n_heads < 1 || p->n_kv_heads < 1 || p->history_len < 1)
    return ATTN_ERR_INVALID;
  if (p->n_heads % p->n_kv_heads != 0) return ATTN_ERR_INVALID;
  const int G = p->n_heads / p->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return ATTN_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return ATTN_ERR_UNSUPPORTED;
  if ((long long)p->num_seqs * p->n_heads >= 65536LL * 65535LL) return ATTN_ERR_INVALID;
  if ((long long)p->num_seqs * p->n_kv_heads > 65535 || p->n_heads > 65535 ||
      p->num_seqs > 65535)
    return ATTN_ERR_INVALID;
  return ATTN_OK;
}

attn_status attn_bwd_decode_kv(const attn_bwd_decode_params* p, const float* q,
                               const float* probs, const float* d_out, const float* d_scores,
                               float* d_k_hist, float* d_v_hist, void* stream) {
  attn_status st = validate_decode(p);
  if (st != ATTN_OK) return st;
  const void* ptrs[] = {q, probs, d_out, d_scores, d_k_hist, d_v_hist};
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return ATTN_ERR_INVALID;
  if (launch_decode_kv(*p, q, probs, d_out, d_scores, d_k_hist, d_v_hist,
                       reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

size_t attn_bwd_decode_workspace_size(const attn_bwd_decode_params* p) {
  if (validate_decode(p) != ATTN_OK) return 0;
  return align256(decode_partials_floats(*p, decode_num_splits(*p)) * 4);
}

attn_status attn_bwd_decode(const attn_bwd_decode_params* p, const float* k_hist,
                            const float* v_hist, const float* probs, const float* d_out,
                            float* d_scores, float* d_q, void* workspace,
                            size_t workspace_bytes, void* stream) {
  attn_status st = validate_decode(p);
  if (st != ATTN_OK) return st;
  const void* ptrs[] = {k_hist, v_hist, probs, d_out, d_scores, d_q};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return ATTN_ERR_INVALID;
  const int n_split = decode_num_splits(*p);
  const size_t need = align256(decode_partials_floats(*p, n_split) * 4);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < need)
    return ATTN_ERR_WORKSPACE;
  if (launch_decode(*p, k_hist, v_hist, probs, d_out, d_scores, d_q,
                    reinterpret_cast<float*>(workspace), n_split,
                    reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status attn_dropout_keep_mask(const attn_bwd_params* p, int32_t b, int32_t h, uint8_t* keep,
                                   void* stream) {
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!keep || b < 0 || b >= p->batch || h < 0 || h >= p->num_heads) return ATTN_ERR_INVALID;
  if (launch_dropout_mask(*p, b, h, keep, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status attn_bwd_query_range(const attn_bwd_params* p, int32_t k0, int32_t k1,
                                 int32_t* q_begin, int32_t* q_end) {
  attn_status st = validate(p);
  if (st != ATTN_OK) return st;
  if (!q_begin || !q_end || k0 < 0 || k1 < k0 || k1 >= p->seq_k) return ATTN_ERR_INVALID;
  int b = 0, e = 0;
  query_range(p->seq_q, p->causal, p->causal_offset, p->window, k0, k1, &b, &e);
  *q_begin = b;
  *q_end = e;
  return ATTN_OK;
}

attn_status attn_bwd_check_device_error(int32_t clear_it) {
  unsigned int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (clear_it && v != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  return v == 0 ? ATTN_OK : ATTN_ERR_TIMEOUT;
}

attn_status attn_selftest_wait_timeout(void* stream) {
  return selftest_wait_launch(reinterpret_cast<cudaStream_t>(stream));
}

attn_status attn_selftest_mma(int32_t dtype, int32_t M, int32_t N, int32_t K, int32_t a_mn,
                              int32_t b_mn, int32_t a_tmem, const void* A, const void* B,
                              float* C, float* tmem_dump, void* stream) {
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_INVALID;
  return selftest_mma_launch(dtype, M, N, K, a_mn, b_mn, a_tmem, A, B, C, tmem_dump,
                             reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
