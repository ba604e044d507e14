// Log-sum-exp of every query row's scores, for callers of the backward pass
// that did not keep the forward's LSE (the WGSL page's flash_bwd_dq, sweep 1:
// a running maximum m and sum l over the visible, non-hard keys of the row,
// lse = m + log l, and 3e38 for a row with no probability mass).
//
// Persistent: one CTA per SM walks work items (a tile of 128 query rows of
// one (batch, query head)), largest first.  The scores come from the tensor
// cores, S [128 queries, BN keys] = Q . K^T per key tile, so TMEM lane r holds
// query row r and every reduction thread owns one row and a share of the
// key columns: maximum and sum stay in registers, and the four partial sums of
// a row are merged through shared memory once per item.  The pipeline runs on
// across items: Q tiles are double-buffered, K tiles stream through a ring,
// scores through NSB TMEM buffers.
//
// Warp roles (640 threads):
//   warp 0      TMA producer: Q tile per item, K tiles through the ring
//   warp 1      MMA issuer (one elected lane)
//   warp 2      TMEM allocator
//   warp 3      idle
//   warps 4-19  reduction: warp w reads TMEM sub-partition w % 4 (its 32
//               query rows); without a mask two groups of 8 warps take
//               alternate key tiles, half of the columns each, with a mask
//               every warp takes a quarter of every tile's columns
// Scores are kept in the log2 domain, x = s * scale * log2(e) + mask * log2(e),
// so every exponential is one ex2; the row result is LSE = ln 2 * (m + log2 l).
// fp32 inputs are fetched as TF32 (the operand type of the products), exactly
// as the backward's score product reads them.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace attnbwd {

namespace {

constexpr int kLseThreads = 640;
constexpr int kLseRedThreads = 512;
constexpr int kLseSmsFallback = 152;
constexpr float kLn2 = 0.6931471805599453f;

template <bool BF16, int D>
struct LseLayout {
  static constexpr int BM = 128;  // query rows per item (MMA M, TMEM lanes)
  static constexpr int E = BF16 ? 2 : 4;
  // keys per tile (MMA N): 64 for fp32 D = 128, whose Q tiles are 64 KB each
  static constexpr int BN = (!BF16 && D == 128) ? 64 : 128;
  static constexpr int W = 128 / E;      // elements per 128-byte segment
  static constexpr int KSTEP = 32 / E;   // K elements per MMA instruction
  static constexpr int Q_BYTES = BM * D * E;
  static constexpr int K_BYTES = BN * D * E;
  static constexpr int NQ = 2;           // Q buffers
  static constexpr int NK = (200 * 1024 - NQ * Q_BYTES) / K_BYTES >= 4 ? 4 : 2;  // K stages
  static constexpr int NSB = 512 / BN >= 4 ? 4 : 512 / BN;  // score buffers in TMEM
  static constexpr int QC = BN / 4;      // key columns per reduction thread (with a mask)
  static constexpr int QC2 = BN / 2;     // key columns per reduction thread (without)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
  static constexpr int OFF_RED = OFF_K + NK * K_BYTES;  // [4][BM] partial (m, l)
  static constexpr int OFF_BAR = OFF_RED + 4 * BM * 8;
  static constexpr int NUM_BARS = 2 * NQ + 2 * NK + 2 * NSB + 1;
  static constexpr int OFF_TMEMPTR = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
  // at least 120 KB, so that a second CTA never shares the SM's tensor memory
  static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr int T_ALLOC = NSB * BN <= 256 ? 256 : 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(NSB * BN <= 512 && NK >= 2, "buffers");
  static_assert(D % W == 0 && QC % 16 == 0, "whole column blocks and TMEM loads");
  static_assert(NSB % 2 == 0, "the two reduction groups take alternate buffers");
};

// Bounded wait that ignores the error word: used only on the unwinding path to
// let copies or products already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait_any(uint64_t* bar, uint32_t parity) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles / 4) return;
  }
}

// Warp-uniform bounded wait: true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait_all(uint64_t* bar, uint32_t parity, unsigned int* err) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, err));
}

__device__ __forceinline__ float lse_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// packed fp32x2 arithmetic (sm_100+)
__device__ __forceinline__ uint64_t lse_pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void lse_up2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t lse_fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t lse_add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Sum of ex2(lo / hi half of fma(v, c, d)) over QC values, two at a time, in
// two packed accumulators.
template <int QC>
__device__ __forceinline__ float sum_ex2(const float (&v)[QC], uint64_t c2, uint64_t d2) {
  uint64_t acc0 = 0, acc1 = 0;  // the bit pattern of (0.f, 0.f)
#pragma unroll
  for (int e = 0; e < QC; e += 4) {
    float a0, a1, b0, b1;
    lse_up2(lse_fma2(lse_pk2(v[e], v[e + 1]), c2, d2), a0, a1);
    lse_up2(lse_fma2(lse_pk2(v[e + 2], v[e + 3]), c2, d2), b0, b1);
    acc0 = lse_add2(acc0, lse_pk2(lse_ex2(a0), lse_ex2(a1)));
    acc1 = lse_add2(acc1, lse_pk2(lse_ex2(b0), lse_ex2(b1)));
  }
  float s0, s1, s2, s3;
  lse_up2(acc0, s0, s1);
  lse_up2(acc1, s2, s3);
  return (s0 + s1) + (s2 + s3);
}

// Maximum (or, for a negative scale, minimum) of QC values as a tree.
template <int QC, bool MAX>
__device__ __forceinline__ float tree_ext(const float (&v)[QC]) {
  float t8[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x = v[e];
#pragma unroll
    for (int f = e + 8; f < QC; f += 8) x = MAX ? fmaxf(x, v[f]) : fminf(x, v[f]);
    t8[e] = x;
  }
#pragma unroll
  for (int w = 4; w > 0; w >>= 1)
#pragma unroll
    for (int e = 0; e < w; ++e) t8[e] = MAX ? fmaxf(t8[e], t8[e + w]) : fminf(t8[e], t8[e + w]);
  return t8[0];
}

// One thread's share of a tile: N consecutive keys from kb of one row, whose
// visible keys are [lo, hi).  Updates the running maximum m and sum l (log2
// domain).  A share with no visible key is skipped; one that is wholly visible
// and unmasked needs only the scores (max of s * c is c * max s, or c * min s
// for a negative scale); otherwise every key is tested.
template <int N, bool MASK, typename MV>
__device__ __forceinline__ void lse_share(const uint32_t (&sv)[N], const MV (&mv)[N], int kb,
                                          int lo, int hi, float c, uint64_t c2, uint64_t one2,
                                          float& m, float& l) {
  if (kb >= hi || kb + N <= lo) return;
  if (!MASK && kb >= lo && kb + N <= hi) {
    float sf[N];
#pragma unroll
    for (int e = 0; e < N; ++e) sf[e] = __uint_as_float(sv[e]);
    const float mx = c >= 0.f ? tree_ext<N, true>(sf) * c : tree_ext<N, false>(sf) * c;
    const float mn = fmaxf(m, mx);
    const float sum = sum_ex2<N>(sf, c2, lse_pk2(-mn, -mn));
    l = fmaf(l, lse_ex2(m - mn), sum);
    m = mn;
  } else {
    float x[N];
#pragma unroll
    for (int e = 0; e < N; ++e) {
      bool vis = (unsigned)(kb + e - lo) < (unsigned)(hi - lo);
      float add = 0.f;
      if constexpr (MASK) {
        vis = vis && mv[e] > kHardMask;
        add = mv[e] * kLog2e;
      }
      x[e] = vis ? fmaf(__uint_as_float(sv[e]), c, add) : -INFINITY;
    }
    const float mn = fmaxf(m, tree_ext<N, true>(x));
    if (mn != -INFINITY) {
      const float sum = sum_ex2<N>(x, one2, lse_pk2(-mn, -mn));
      l = fmaf(l, lse_ex2(m - mn), sum);
      m = mn;
    }
  }
}

__device__ __forceinline__ void red_sync() {
  asm volatile("bar.sync 1, 512;" ::: "memory");
}

// Keys [k_start, k_end) that a row of [q0, q1] can see (WGSL page,
// fab2_key_range restated): causal stops at the last row's position, the
// window starts past the first row's position minus the window and, without
// causal, ends before the last row's position plus the window.  k_start is
// rounded down to a multiple of 16 so that mask rows can be read as float4.
__device__ __forceinline__ void lse_key_range(const LseArgs& a, int q0, int q1, int* ks,
                                              int* ke) {
  const long long qa_min = (long long)q0 + a.causal_offset;
  const long long qa_max = (long long)q1 + a.causal_offset;
  long long lo = 0, hi = a.Sk;
  if (a.causal && qa_max + 1 < hi) hi = qa_max + 1;
  if (a.window > 0) {
    if (qa_min - a.window + 1 > lo) lo = qa_min - a.window + 1;
    if (!a.causal && qa_max + a.window < hi) hi = qa_max + a.window;
  }
  if (hi < lo) hi = lo;
  lo &= ~15LL;
  *ks = (int)lo;
  *ke = (int)hi;
}

// Work item i (0 .. n_qt * B * H - 1): the largest query tiles first (with
// causal they see the most keys), then (batch, head).
struct LseItem {
  int q0, bh, b, h, k_start, T;
};

template <int BM, int BN>
__device__ __forceinline__ LseItem lse_item(const LseArgs& a, int n_qt, int i) {
  LseItem it;
  const int BH = a.B * a.H;
  const int qt = n_qt - 1 - i / BH;
  it.bh = i % BH;
  it.b = it.bh / a.H;
  it.h = it.bh % a.H;
  it.q0 = qt * BM;
  const int q1 = min(it.q0 + BM, a.Sq) - 1;
  int ke;
  lse_key_range(a, it.q0, q1, &it.k_start, &ke);
  it.T = ke > it.k_start ? (ke - it.k_start + BN - 1) / BN : 0;
  return it;
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kLseThreads, 1)
    lse_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const LseArgs a) {
  using L = LseLayout<BF16, D>;
  constexpr int BM = L::BM, BN = L::BN, NK = L::NK, NSB = L::NSB, NQ = L::NQ,
                QC = L::QC, QC2 = L::QC2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;               // [NQ] Q tile landed
  uint64_t* q_empty = q_full + NQ;       // [NQ] products done with the Q buffer
  uint64_t* k_full = q_empty + NQ;       // [NK] K tile landed
  uint64_t* k_empty = k_full + NK;       // [NK] products done with the K stage
  uint64_t* s_full = k_empty + NK;       // [NSB] scores of a tile in buffer b
  uint64_t* s_free = s_full + NSB;       // [NSB] reduction warps have read buffer b
  uint64_t* final_bar = s_free + NSB;    // every product issued is done
  float2* red = reinterpret_cast<float2*>(smem + L::OFF_RED);
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEMPTR);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_qt = (a.Sq + BM - 1) / BM;
  const int n_items = n_qt * a.B * a.H;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int s = 0; s < NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&s_full[s], 1);
      // every reduction thread reads every tile with a mask; half of them
      // (the group of the tile's parity) without
      mbar_init(&s_free[s], a.has_mask ? kLseRedThreads : kLseRedThreads / 2);
    }
    mbar_init(final_bar, 1);
    fence_barrier_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_ptr, L::T_ALLOC);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_ptr;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (elect_one_sync()) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      int g = 0, nz = 0;  // K tiles issued, non-empty items begun
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const LseItem it = lse_item<BM, BN>(a, n_qt, i);
        if (it.T == 0) continue;
        const int qb = nz % NQ;
        if (nz >= NQ && !mbar_wait(&q_empty[qb], ((nz / NQ) - 1) & 1, a.err)) break;
        mbar_expect_tx(&q_full[qb], L::Q_BYTES);
        tma_load_5d(smem + L::OFF_Q + qb * L::Q_BYTES, &tm_q, &q_full[qb], 0, it.q0, 0, it.h,
                    it.b);
        ++nz;
        const int kvh = it.h / a.group;
        for (int t = 0; t < it.T; ++t, ++g) {
          const int s = g % NK;
          if (g >= NK && !mbar_wait(&k_empty[s], ((g / NK) - 1) & 1, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&k_full[s], L::K_BYTES);
          tma_load_5d(smem + L::OFF_K + s * L::K_BYTES, &tm_k, &k_full[s], 0, it.k_start + t * BN,
                      0, kvh, it.b);
        }
      }
      // let every copy still in flight land before the CTA can exit
      for (int j = (nz > NQ ? nz - NQ : 0); j < nz; ++j) drain_wait_any(&q_full[j % NQ], (j / NQ) & 1);
      for (int j = (g > NK ? g - NK : 0); j < g; ++j) drain_wait_any(&k_full[j % NK], (j / NK) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      constexpr uint32_t idesc = make_idesc(BF16, BM, BN, false, false);
      // K-major 128-byte-swizzled tiles: LBO unused, SBO = 8 rows x 128 B
      const uint64_t dQ0 = sw128_desc(smem_u32(smem + L::OFF_Q), 16, 1024);
      const uint64_t dK0 = sw128_desc(smem_u32(smem + L::OFF_K), 16, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) -> uint64_t { return d + (uint64_t)(bytes >> 4); };
      int g = 0, nz = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const LseItem it = lse_item<BM, BN>(a, n_qt, i);
        if (it.T == 0) continue;
        const int qb = nz % NQ;
        if (!mbar_wait(&q_full[qb], (nz / NQ) & 1, a.err)) break;
        const uint64_t dQ = adv(dQ0, qb * L::Q_BYTES);
        for (int t = 0; t < it.T; ++t, ++g) {
          const int s = g % NK, sb = g % NSB;
          if (!mbar_wait(&k_full[s], (g / NK) & 1, a.err) ||
              (g >= NSB && !mbar_wait(&s_free[sb], ((g / NSB) - 1) & 1, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dK = adv(dK0, s * L::K_BYTES);
#pragma unroll
          for (int ks = 0; ks < D / L::KSTEP; ++ks) {
            const uint32_t kb = ks * 32;
            const uint32_t qa = (kb / 128) * BM * 128 + (kb % 128);
            const uint32_t ka = (kb / 128) * BN * 128 + (kb % 128);
            mma_ss<BF16>(tmem + sb * BN, adv(dQ, qa), adv(dK, ka), idesc, ks > 0);
          }
          mma_commit(&s_full[sb]);
          mma_commit(&k_empty[s]);
        }
        mma_commit(&q_empty[qb]);
        ++nz;
      }
      mma_commit(final_bar);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ reduction
    // Without a mask the 16 warps form two groups that take alternate key
    // tiles (group = tile parity), each thread covering half of a tile's
    // columns, so one group's TMEM loads overlap the other group's arithmetic.
    // With a mask every warp reads every tile, a quarter of its columns, and
    // the quarter's mask values are requested before the wait for the scores.
    const int sp = warp & 3, w4 = warp - 4;
    const int r = sp * 32 + lane;  // query row of the item (TMEM lane)
    const bool split = !a.has_mask;
    const int grp = split ? (w4 >> 3) : 0;
    const int part = split ? ((w4 >> 2) & 1) : (w4 >> 2);  // column share of the tile
    const int ncol = split ? QC2 : QC;
    const uint32_t t_row = tmem + ((uint32_t)(sp * 32) << 16) + part * ncol;
    const float c = a.scale_log2e;
    const uint64_t c2 = lse_pk2(c, c), one2 = lse_pk2(1.f, 1.f);
    int g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
      const LseItem it = lse_item<BM, BN>(a, n_qt, i);
      const int q = it.q0 + r;
      const bool q_ok = q < a.Sq;
      // this row's visible keys [lo, hi) (fab2_visible restated): causal
      // stops at qa, the window keeps |qa - k| < window, keys end at Sk
      int lo = 0, hi = 0;
      if (q_ok) {
        const long long qa = (long long)q + a.causal_offset;
        long long l0 = 0, h0 = a.Sk;
        if (a.causal && qa + 1 < h0) h0 = qa + 1;
        if (a.window > 0) {
          if (qa - a.window + 1 > l0) l0 = qa - a.window + 1;
          if (!a.causal && qa + a.window < h0) h0 = qa + a.window;
        }
        if (h0 < l0) h0 = l0;
        lo = (int)l0;
        hi = (int)h0;
      }
      float m = -INFINITY, l = 0.f;
      if (split) {
        for (int t = 0; ok && t < it.T; ++t, ++g) {
          if ((g & 1) != grp) continue;
          const int sb = g % NSB;
          const int kb = it.k_start + t * BN + part * QC2;  // first key of this share
          if (!warp_wait_all(&s_full[sb], (g / NSB) & 1, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sv[QC2];
          __syncwarp();
#pragma unroll
          for (int c0 = 0; c0 < QC2; c0 += 16) {
            uint32_t rr[16];
            tmem_ld16(t_row + sb * BN + c0, rr);
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[c0 + e] = rr[e];
          }
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&s_free[sb]);
          lse_share<QC2, false>(sv, sv, kb, lo, hi, c, c2, one2, m, l);
        }
      } else {
        const float* mrow = q_ok ? a.mask + (long long)it.b * a.msb + (long long)it.h * a.msh +
                                       (long long)q * a.msq
                                 : nullptr;
        for (int t = 0; ok && t < it.T; ++t, ++g) {
          const int sb = g % NSB;
          const int kb = it.k_start + t * BN + part * QC;  // first key of this share
          // the share's mask values, requested before the wait for the scores
          float mv[QC];
#pragma unroll
          for (int e = 0; e < QC; ++e) mv[e] = 0.f;
          if (mrow && kb < hi && kb + QC > lo) {
            if (a.mask_vec) {
#pragma unroll
              for (int e = 0; e < QC; e += 4) {
                if (kb + e + 4 <= a.Sk) {
                  const float4 v4 = __ldg(reinterpret_cast<const float4*>(mrow + kb + e));
                  mv[e] = v4.x;
                  mv[e + 1] = v4.y;
                  mv[e + 2] = v4.z;
                  mv[e + 3] = v4.w;
                } else {
#pragma unroll
                  for (int u = 0; u < 4; ++u)
                    if (kb + e + u < a.Sk) mv[e + u] = __ldg(mrow + kb + e + u);
                }
              }
            } else {
#pragma unroll
              for (int e = 0; e < QC; ++e)
                if (kb + e < a.Sk) mv[e] = __ldg(mrow + (long long)(kb + e) * a.msk);
            }
          }
          if (!warp_wait_all(&s_full[sb], (g / NSB) & 1, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint32_t sv[QC];
          __syncwarp();
#pragma unroll
          for (int c0 = 0; c0 < QC; c0 += 16) {
            uint32_t rr[16];
            tmem_ld16(t_row + sb * BN + c0, rr);
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[c0 + e] = rr[e];
          }
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&s_free[sb]);
          lse_share<QC, true>(sv, mv, kb, lo, hi, c, c2, one2, m, l);
        }
      }
      // merge the four partial (m, l) of each row; every reduction thread
      // arrives at both barriers, also after a failed wait
      const int q4 = split ? grp * 2 + part : part;
      red[q4 * BM + r] = make_float2(m, l);
      red_sync();
      if (q4 == 0) {
        float2 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = red[u * BM + r];
        const float mm = fmaxf(fmaxf(v[0].x, v[1].x), fmaxf(v[2].x, v[3].x));
        float ll = 0.f;
        if (mm != -INFINITY) {
#pragma unroll
          for (int u = 0; u < 4; ++u) ll += v[u].y * lse_ex2(v[u].x - mm);
        }
        const bool empty = !(ll > 0.f);
        const float lse2 = mm + log2f(ll);  // LSE * log2(e)
        if (a.out_mode == 0) {
          if (q_ok) a.out[(long long)it.bh * a.Sq + q] = empty ? kEmptyRowLse : lse2 * kLn2;
        } else {
          a.out[(long long)it.bh * a.sq_pad + q] = (empty || !q_ok) ? -INFINITY : -lse2;
        }
      }
      red_sync();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    // products still in flight (only on the unwinding path) must finish first
    drain_wait_any(final_bar, 0);
    tc_fence_after();
    tmem_dealloc(tmem, L::T_ALLOC);
  }
}

template <bool BF16, int D>
cudaError_t lse_impl(const CUtensorMap& tq, const CUtensorMap& tk, const LseArgs& a,
                     cudaStream_t stream) {
  using L = LseLayout<BF16, D>;
  auto kern = lse_kernel<BF16, D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = (long long)((a.Sq + L::BM - 1) / L::BM) * a.B * a.H;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = kLseSmsFallback;
  const int grid = (int)(items < sms ? items : sms);
  kern<<<grid, kLseThreads, L::SMEM_BYTES, stream>>>(tq, tk, a);
  return cudaGetLastError();
}

}  // namespace

int lse_block_n(int dtype, int head_dim) {
  if (dtype == ATTN_BF16) return head_dim == 64 ? LseLayout<true, 64>::BN : LseLayout<true, 128>::BN;
  return head_dim == 64 ? LseLayout<false, 64>::BN : LseLayout<false, 128>::BN;
}

cudaError_t launch_lse(const attn_bwd_params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const LseArgs& a, cudaStream_t stream) {
  const bool bf = p.dtype == ATTN_BF16;
  if (p.head_dim == 64)
    return bf ? lse_impl<true, 64>(tq, tk, a, stream) : lse_impl<false, 64>(tq, tk, a, stream);
  return bf ? lse_impl<true, 128>(tq, tk, a, stream) : lse_impl<false, 128>(tq, tk, a, stream);
}

}  // namespace attnbwd
