// Memory-bound helper kernels of the backward pass.
//
//  prep_kernel      Delta_i = dO_i . O_i (the Metal page's "D = rowsum(dO * O)",
//                   the WGSL page's delta4 sum), NL_i = -LSE_i * log2(e) for
//                   the tile kernel's exp2 (P = exp2(s * scale * log2e + NL)),
//                   padding rows (Delta 0, NL -inf so P = 0), and zeroing of
//                   the fp32 dQ accumulator row.  One
//                   group of D*esize/16 threads per row, 16-byte loads,
//                   shuffle reduction inside the group.
//  dq_convert       fp32 dQ accumulator -> bf16 dQ (round to nearest even).
//  dropout_mask     the keep mask of one (b, h) slice, for bit-exact tests.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace attnbwd {

namespace {

template <bool BF16, int D>
__global__ void __launch_bounds__(256) prep_kernel(const void* __restrict__ O,
                                                   const void* __restrict__ dO,
                                                   const float* __restrict__ LSE,
                                                   float* __restrict__ delta,
                                                   float* __restrict__ lse2,
                                                   float* __restrict__ dq_acc, int B, int H,
                                                   int Sq, int sq_pad, int layout) {
  constexpr int E = BF16 ? 2 : 4;
  constexpr int G = D * E / 16;  // threads per row
  constexpr int ROWS = 256 / G;
  // the tile kernel behind this one may start its CTAs once every block has
  // started (it waits for this kernel before it reads anything written here)
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int sub = threadIdx.x % G;
  const long long r = (long long)blockIdx.x * ROWS + threadIdx.x / G;
  const long long nrows = (long long)B * H * sq_pad;
  // nrows is a multiple of kRowPad (>= ROWS), so every launched row exists and
  // no lane leaves before the group shuffle below
  if (r >= nrows) return;
  const int i = (int)(r % sq_pad);
  const int bh = (int)(r / sq_pad);
  const int b = bh / H, h = bh % H;
  float acc = 0.f;
  long long off = 0;
  if (i < Sq) {
    off = row_offset(layout, b, h, i, H, Sq, D);
    if constexpr (BF16) {
      const uint4 o = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(O) + off)[sub];
      const uint4 g = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(dO) + off)[sub];
      const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[k]));
        const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[k]));
        acc = fmaf(of.x, gf.x, acc);
        acc = fmaf(of.y, gf.y, acc);
      }
    } else {
      const float4 o = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(O) + off)[sub];
      const float4 g = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(dO) + off)[sub];
      acc = fmaf(o.x, g.x, acc);
      acc = fmaf(o.y, g.y, acc);
      acc = fmaf(o.z, g.z, acc);
      acc = fmaf(o.w, g.w, acc);
    }
    // zero this row of the dQ accumulator (D fp32 = D/4 float4 over G threads)
    float4* zq = reinterpret_cast<float4*>(dq_acc + off);
#pragma unroll
    for (int c = sub; c < D / 4; c += G) zq[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = G / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m, G);
  if (sub == 0) {
    const long long w = (long long)bh * sq_pad + i;
    if (i < Sq) {
      delta[w] = acc;
      if (LSE) lse2[w] = -LSE[(long long)bh * Sq + i] * kLog2e;
    } else {
      delta[w] = 0.f;
      if (LSE) lse2[w] = __int_as_float(0xff800000);  // -inf: P = exp2(x - inf) = 0
    }
  }
}

template <bool BF16, int D>
cudaError_t prep_impl(const attn_bwd_params& p, const void* O, const void* dO, const float* LSE,
                      float* delta, float* lse2, int sq_pad, float* dq_acc, cudaStream_t stream) {
  constexpr int G = D * (BF16 ? 2 : 4) / 16;
  constexpr int ROWS = 256 / G;
  const long long nrows = (long long)p.batch * p.num_heads * sq_pad;
  const long long blocks = (nrows + ROWS - 1) / ROWS;
  prep_kernel<BF16, D><<<(unsigned)blocks, 256, 0, stream>>>(
      O, dO, LSE, delta, lse2, dq_acc, p.batch, p.num_heads, p.seq_q, sq_pad, p.layout);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ src,
                                                         uint2* __restrict__ dst, long long n4) {
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n4;
       k += (long long)gridDim.x * blockDim.x) {
    const float4 v = src[k];
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    dst[k] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}

__global__ void __launch_bounds__(256) dropout_mask_kernel(uint8_t* __restrict__ keep, int Sq,
                                                           int Sk, uint32_t bh, uint32_t seed_lo,
                                                           uint32_t seed_hi, uint32_t threshold) {
  const long long n = (long long)Sq * Sk;
  for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n;
       k += (long long)gridDim.x * blockDim.x) {
    const uint32_t i = (uint32_t)(k / Sk), j = (uint32_t)(k % Sk);
    const Philox4 r = philox4x32_10(i >> 2, j, bh, 0u, seed_lo, seed_hi);
    keep[k] = r.w[i & 3] >= threshold ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_prep(const attn_bwd_params& p, const void* O, const void* dO, const float* LSE,
                        float* delta, float* lse2, int sq_pad, float* dq_acc,
                        cudaStream_t stream) {
  const bool bf = p.dtype == ATTN_BF16;
  if (p.head_dim == 64)
    return bf ? prep_impl<true, 64>(p, O, dO, LSE, delta, lse2, sq_pad, dq_acc, stream)
              : prep_impl<false, 64>(p, O, dO, LSE, delta, lse2, sq_pad, dq_acc, stream);
  return bf ? prep_impl<true, 128>(p, O, dO, LSE, delta, lse2, sq_pad, dq_acc, stream)
            : prep_impl<false, 128>(p, O, dO, LSE, delta, lse2, sq_pad, dq_acc, stream);
}

namespace {

// Deterministic dQ: one group of G = D/4 threads per dQ row (b, h, q), one
// float4 each; the row is the sum, in ascending key-tile order, of the slices
// of the key tiles whose dK/dV CTA visited the row's query tile (the same
// query ranges as the tile kernel's, so unvisited slices, which hold no data,
// are never read).  Per round of G key tiles every thread of the group tests
// one tile, a ballot hands the group the visited set, and the group then
// loads up to four slices before adding them, in order.
template <bool BF16, int D>
__global__ void __launch_bounds__(256) dq_reduce_kernel(const float* __restrict__ slices,
                                                        void* __restrict__ dQ, int B, int H,
                                                        int Sq, int Sk, int layout, int causal,
                                                        long long off, long long window, int bn,
                                                        int bm, int n_kt) {
  constexpr int G = D / 4;           // threads per row (16 or 32)
  constexpr int ROWS = 256 / G;      // rows per block
  const long long row = (long long)blockIdx.x * ROWS + threadIdx.x / G;
  const int sub = threadIdx.x % G;
  const int lane = threadIdx.x & 31;
  const long long nrows = (long long)B * H * Sq;
  const bool row_ok = row < nrows;  // every lane stays for the ballots
  const long long rr = row_ok ? row : 0;
  const int q = (int)(rr % Sq);
  const int bh = (int)(rr / Sq);
  const int b = bh / H, h = bh % H;
  const float4* base = reinterpret_cast<const float4*>(slices) + sub;
  const long long kt_stride = (long long)B * H * Sq * (D / 4);  // float4 per slice
  const long long row4 = (((long long)b * H + h) * Sq + q) * (D / 4);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](const float4& v) {
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  };
  for (int kt0 = 0; kt0 < n_kt; kt0 += G) {
    const int kt = kt0 + sub;
    bool vis = false;
    if (row_ok && kt < n_kt) {
      const long long k0 = (long long)kt * bn;
      const long long k1 = (k0 + bn < Sk ? k0 + bn : Sk) - 1;
      int qb = 0, qe = 0;
      query_range(Sq, causal, off, window, k0, k1, &qb, &qe);
      if (qe > qb) {
        const int q_first = (qb / bm) * bm;
        const int tiles = (qe - q_first + bm - 1) / bm;
        vis = q >= q_first && q < q_first + tiles * bm;
      }
    }
    unsigned bits = __ballot_sync(0xffffffffu, vis);
    if constexpr (G < 32) bits = (bits >> (lane & ~(G - 1))) & ((1u << G) - 1u);
    while (bits) {
      int j[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        j[u] = bits ? __ffs(bits) - 1 : -1;
        bits &= bits ? bits - 1 : 0u;
      }
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j[u] >= 0) v[u] = base[(long long)(kt0 + j[u]) * kt_stride + row4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j[u] >= 0) add(v[u]);
    }
  }
  if (!row_ok) return;
  const long long o = row_offset(layout, b, h, q, H, Sq, D) + 4 * sub;
  if constexpr (BF16) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(dQ) + o) =
        make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  } else {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(dQ) + o) = acc;
  }
}

template <bool BF16, int D>
cudaError_t dq_reduce_impl(const attn_bwd_params& p, const float* slices, void* dQ, int bn,
                           int bm, cudaStream_t stream) {
  constexpr int ROWS = 256 / (D / 4);
  const long long nrows = (long long)p.batch * p.num_heads * p.seq_q;
  const long long blocks = (nrows + ROWS - 1) / ROWS;
  const int n_kt = (p.seq_k + bn - 1) / bn;
  dq_reduce_kernel<BF16, D><<<(unsigned)blocks, 256, 0, stream>>>(
      slices, dQ, p.batch, p.num_heads, p.seq_q, p.seq_k, p.layout, p.causal, p.causal_offset,
      p.window, bn, bm, n_kt);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dq_reduce(const attn_bwd_params& p, const float* slices, void* dQ, int bn,
                             int bm, cudaStream_t stream) {
  const bool bf = p.dtype == ATTN_BF16;
  if (p.head_dim == 64)
    return bf ? dq_reduce_impl<true, 64>(p, slices, dQ, bn, bm, stream)
              : dq_reduce_impl<false, 64>(p, slices, dQ, bn, bm, stream);
  return bf ? dq_reduce_impl<true, 128>(p, slices, dQ, bn, bm, stream)
            : dq_reduce_impl<false, 128>(p, slices, dQ, bn, bm, stream);
}

cudaError_t launch_dq_convert(const attn_bwd_params& p, const float* dq_acc, void* dQ,
                              cudaStream_t stream) {
  const long long n4 = (long long)p.batch * p.num_heads * p.seq_q * p.head_dim / 4;
  long long blocks = (n4 + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  dq_convert_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      reinterpret_cast<const float4*>(dq_acc), reinterpret_cast<uint2*>(dQ), n4);
  return cudaGetLastError();
}

// keep iff word >= T, T = min(floor(p * 2^32), 2^32 - 1), computed in fp64
uint32_t dropout_threshold(float prob) {
  if (!(prob > 0.f)) return 0u;
  double t = (double)prob * 4294967296.0;
  if (t >= 4294967295.0) return 0xFFFFFFFFu;
  return (uint32_t)t;
}

cudaError_t launch_dropout_mask(const attn_bwd_params& p, int b, int h, uint8_t* keep,
                                cudaStream_t stream) {
  const long long n = (long long)p.seq_q * p.seq_k;
  long long blocks = (n + 255) / 256;
  if (blocks > 152 * 32) blocks = 152 * 32;
  if (blocks < 1) blocks = 1;
  dropout_mask_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      keep, p.seq_q, p.seq_k, (uint32_t)(b * p.num_heads + h), (uint32_t)(p.seed & 0xFFFFFFFFu),
      (uint32_t)(p.seed >> 32), dropout_threshold(p.dropout_prob));
  return cudaGetLastError();
}

}  // namespace attnbwd
