// Fused attention forward for sm_103a: O and LSE with the backward pass's
// conventions (visibility, additive mask with the -1e30 hard sentinel,
// Philox dropout on P, 3e38 for a row without probability mass), so that the
// backward's inputs can be produced on the GPU.
//
//   s_ij  = scale * Q_i . K_j + mask_ij           (visible, non-hard pairs)
//   LSE_i = log sum_j exp(s_ij)                    (3e38 if there is no pair)
//   O_i   = sum_j exp(s_ij - LSE_i) M_ij V_j       (M: dropout multiplier)
//
// Persistent: one CTA per SM walks work items (128 query rows of one
// (batch, query head)), largest first, like the LSE sweep.  Per key tile the
// tensor cores form S = Q . K^T in TMEM (lane = query row); 16 softmax warps
// (four per TMEM sub-partition, a quarter of the key columns each) take the
// row maximum through shared memory, write P o M in place over S as the
// TMEM A operand, and the tensor cores add P . V into the O accumulator in
// TMEM.  The running maximum is raised lazily: O and the running sums are
// rescaled only when a tile's maximum exceeds the current one by more than
// 2^8 (P <= 256 otherwise, far inside fp32 / bf16 range).  At the end of an
// item the four partial sums of a row are merged, O is divided by the sum and
// stored, and LSE = ln 2 * (m + log2 l).
//
// Warp roles (640 threads):
//   warp 0      TMA producer: Q per item, K and V tiles through two rings
//   warp 1      MMA issuer (one elected lane)
//   warp 2      TMEM allocator
//   warp 3      idle
//   warps 4-19  softmax / correction / epilogue
// Operands: Q and K K-major (128-byte swizzle) for S; for O += P . V the A
// operand is P in TMEM and the B operand is the natural [keys][D] tile of V
// read MN-major: 128-byte swizzle for bf16; for fp32 the 128-byte swizzle of
// 32-byte atoms, the layout TF32 operands read MN-major take.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace attnbwd {

namespace {

constexpr int kFwdThreads = 640;
constexpr int kFwdSoftThreads = 512;
constexpr int kFwdSmsFallback = 152;
constexpr float kFwdLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;  // lazy rescale threshold (log2 domain)

template <bool BF16, int D>
struct FwdLayout {
  static constexpr int BM = 128;  // query rows per item (MMA M, TMEM lanes)
  static constexpr int E = BF16 ? 2 : 4;
  static constexpr int BN = (!BF16 && D == 128) ? 64 : 128;  // keys per tile
  static constexpr int W = 128 / E;     // elements per 128-byte segment
  static constexpr int KSTEP = 32 / E;  // K elements per MMA instruction
  static constexpr int Q_BYTES = BM * D * E;
  static constexpr int K_BYTES = BN * D * E;
  static constexpr int V_BYTES = BN * D * E;  // [D / W column blocks][BN][W]
  static constexpr int NQ = (!BF16 && D == 128) ? 1 : 2;
  static constexpr int NK = 2, NV = 2, NSB = 2;
  static constexpr int QC = BN / 4;  // key columns per softmax thread
  static constexpr int OC = D / 4;   // O columns per softmax thread
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQ * Q_BYTES;
  static constexpr int OFF_V = OFF_K + NK * K_BYTES;
  static constexpr int OFF_RMAX = OFF_V + NV * V_BYTES;  // [2][4][BM] partial maxima
  static constexpr int OFF_RSUM = OFF_RMAX + 2 * 4 * BM * 4;  // [4][BM] partial sums
  static constexpr int OFF_BAR = OFF_RSUM + 4 * BM * 4;
  static constexpr int NUM_BARS = 2 * NQ + 2 * NK + 2 * NV + 3 * NSB + 2;
  static constexpr int OFF_TMEMPTR = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_TMEMPTR + 16 + 1024;
  // at least 120 KB, so that a second CTA never shares the SM's tensor memory
  static constexpr int SMEM_BYTES = SMEM_USED > 120 * 1024 ? SMEM_USED : 120 * 1024;
  static constexpr int T_S = 0;                 // NSB score buffers of BN columns
  static constexpr int T_O = NSB * BN;          // O accumulator, D columns
  static constexpr int T_ALLOC = T_O + D <= 256 ? 256 : 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(T_O + D <= 512, "tensor memory budget");
  static_assert(QC % 16 == 0 && OC % 16 == 0 && D % W == 0 && BN % W == 0, "tile shapes");
};

__device__ __forceinline__ void fwd_drain(uint64_t* bar, uint32_t parity) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles / 4) return;
  }
}

__device__ __forceinline__ bool fwd_warp_wait(uint64_t* bar, uint32_t parity, unsigned int* err) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, err));
}

__device__ __forceinline__ float fwd_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The four softmax warps of TMEM sub-partition sp (one per quarter of the key
// columns) hold the four shares of the same 32 rows: named barrier 2 + sp
// over their 128 threads.
__device__ __forceinline__ void sp_sync(int sp) {
  asm volatile("bar.sync %0, 128;" ::"r"(2 + sp) : "memory");
}

// packed fp32x2 arithmetic (sm_100+)
__device__ __forceinline__ uint64_t fpk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void fup2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t ff2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t ff2add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t fwd_pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Keys [k_start, k_end) that a row of [q0, q1] can see; k_start rounded down
// to a multiple of 16 so that mask rows can be read as float4 (the same range
// rule as the LSE sweep); an empty range stays empty (no tile is loaded).
__device__ __forceinline__ void fwd_key_range(const FwdArgs& a, int q0, int q1, int* ks,
                                              int* ke) {
  const long long qa_min = (long long)q0 + a.causal_offset;
  const long long qa_max = (long long)q1 + a.causal_offset;
  long long lo = 0, hi = a.Sk;
  if (a.causal && qa_max + 1 < hi) hi = qa_max + 1;
  if (a.window > 0) {
    if (qa_min - a.window + 1 > lo) lo = qa_min - a.window + 1;
    if (!a.causal && qa_max + a.window < hi) hi = qa_max + a.window;
  }
  if (hi <= lo) {
    *ks = 0;
    *ke = 0;
    return;
  }
  lo &= ~15LL;
  *ks = (int)lo;
  *ke = (int)hi;
}

struct FwdItem {
  int q0, bh, b, h, k_start, T;
};

template <int BM, int BN>
__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int n_qt, int i) {
  FwdItem it;
  const int BH = a.B * a.H;
  const int qt = n_qt - 1 - i / BH;
  it.bh = i % BH;
  it.b = it.bh / a.H;
  it.h = it.bh % a.H;
  it.q0 = qt * BM;
  const int q1 = min(it.q0 + BM, a.Sq) - 1;
  int ke;
  fwd_key_range(a, it.q0, q1, &it.k_start, &ke);
  it.T = ke > it.k_start ? (ke - it.k_start + BN - 1) / BN : 0;
  return it;
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const FwdArgs a) {
  using L = FwdLayout<BF16, D>;
  constexpr int BM = L::BM, BN = L::BN, NK = L::NK, NV = L::NV, NSB = L::NSB, NQ = L::NQ,
                QC = L::QC, OC = L::OC;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;             // [NQ] Q tile landed
  uint64_t* q_empty = q_full + NQ;     // [NQ] products done with the Q buffer
  uint64_t* k_full = q_empty + NQ;     // [NK]
  uint64_t* k_empty = k_full + NK;     // [NK]
  uint64_t* v_full = k_empty + NK;     // [NV]
  uint64_t* v_empty = v_full + NV;     // [NV]
  uint64_t* s_full = v_empty + NV;     // [NSB] S of a tile in buffer b
  uint64_t* p_full = s_full + NSB;     // [NSB] P o M written over buffer b (softmax)
  uint64_t* pv_done = p_full + NSB;    // [NSB] O += P . V of buffer b done
  uint64_t* o_free = pv_done + NSB;    // O read out by the softmax warps (per item)
  uint64_t* final_bar = o_free + 1;    // every product issued is done
  float* rmax = reinterpret_cast<float*>(smem + L::OFF_RMAX);
  float* rsum = reinterpret_cast<float*>(smem + L::OFF_RSUM);
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
    for (int s = 0; s < NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], kFwdSoftThreads);
      mbar_init(&pv_done[s], 1);
    }
    mbar_init(o_free, kFwdSoftThreads);
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
      tma_prefetch_desc(&tm_v);
      int gk = 0, gv = 0, nz = 0;  // K tiles, V tiles, non-empty items issued
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const FwdItem it = fwd_item<BM, BN>(a, n_qt, i);
        if (it.T == 0) continue;
        const int qb = nz % NQ;
        if (nz >= NQ && !mbar_wait(&q_empty[qb], ((nz / NQ) - 1) & 1, a.err)) break;
        mbar_expect_tx(&q_full[qb], L::Q_BYTES);
        tma_load_5d(smem + L::OFF_Q + qb * L::Q_BYTES, &tm_q, &q_full[qb], 0, it.q0, 0, it.h,
                    it.b);
        ++nz;
        const int kvh = it.h / a.group;
        for (int t = 0; t < it.T; ++t) {
          const int k0 = it.k_start + t * BN;
          const int sk = gk % NK;
          if (gk >= NK && !mbar_wait(&k_empty[sk], ((gk / NK) - 1) & 1, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&k_full[sk], L::K_BYTES);
          tma_load_5d(smem + L::OFF_K + sk * L::K_BYTES, &tm_k, &k_full[sk], 0, k0, 0, kvh, it.b);
          ++gk;
          const int sv = gv % NV;
          if (gv >= NV && !mbar_wait(&v_empty[sv], ((gv / NV) - 1) & 1, a.err)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&v_full[sv], L::V_BYTES);
          // natural V [D / W column blocks][BN keys][W]
          tma_load_5d(smem + L::OFF_V + sv * L::V_BYTES, &tm_v, &v_full[sv], 0, k0, 0, kvh, it.b);
          ++gv;
        }
      }
      for (int j = (nz > NQ ? nz - NQ : 0); j < nz; ++j) fwd_drain(&q_full[j % NQ], (j / NQ) & 1);
      for (int j = (gk > NK ? gk - NK : 0); j < gk; ++j) fwd_drain(&k_full[j % NK], (j / NK) & 1);
      for (int j = (gv > NV ? gv - NV : 0); j < gv; ++j) fwd_drain(&v_full[j % NV], (j / NV) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one_sync()) {
      constexpr uint32_t id_s = make_idesc(BF16, BM, BN, false, false);
      // O += P . V: A = P in TMEM; B = V read MN-major
      constexpr uint32_t id_o = make_idesc(BF16, BM, D, false, true);
      const uint64_t dQ0 = sw128_desc(smem_u32(smem + L::OFF_Q), 16, 1024);
      const uint64_t dK0 = sw128_desc(smem_u32(smem + L::OFF_K), 16, 1024);
      const uint64_t dV0 = BF16 ? sw128_desc(smem_u32(smem + L::OFF_V), BN * 128, 1024)
                                : mn32_desc(smem_u32(smem + L::OFF_V), BN * 128);
      auto adv = [](uint64_t d, uint32_t bytes) -> uint64_t { return d + (uint64_t)(bytes >> 4); };
      int g = 0, gs = 0, nz = 0;  // tiles whose P . V was issued, S issued, items
      bool ok = true;
      // S of global tile gs (of the current item) into buffer gs % NSB, once
      // the P . V that last read that buffer is done
      auto issue_s = [&](uint64_t dQ) -> bool {
        const int sk = gs % NK, sb = gs % NSB;
        if (!mbar_wait(&k_full[sk], (gs / NK) & 1, a.err)) return false;
        if (gs >= NSB && !mbar_wait(&pv_done[sb], ((gs / NSB) - 1) & 1, a.err)) return false;
        tc_fence_after();
        const uint64_t dK = adv(dK0, sk * L::K_BYTES);
#pragma unroll
        for (int ks = 0; ks < D / L::KSTEP; ++ks) {
          const uint32_t kb = ks * 32;
          const uint32_t qa = (kb / 128) * BM * 128 + (kb % 128);
          const uint32_t ka = (kb / 128) * BN * 128 + (kb % 128);
          mma_ss<BF16>(tmem + L::T_S + sb * BN, adv(dQ, qa), adv(dK, ka), id_s, ks > 0);
        }
        mma_commit(&s_full[sb]);
        mma_commit(&k_empty[sk]);
        ++gs;
        return true;
      };
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const FwdItem it = fwd_item<BM, BN>(a, n_qt, i);
        if (it.T == 0) continue;
        const int qb = nz % NQ;
        if (!mbar_wait(&q_full[qb], (nz / NQ) & 1, a.err)) break;
        const uint64_t dQ = adv(dQ0, qb * L::Q_BYTES);
        ok = issue_s(dQ) && (it.T < 2 || issue_s(dQ));
        for (int t = 0; ok && t < it.T; ++t, ++g) {
          const int sb = g % NSB, sv = g % NV;
          if (!mbar_wait(&p_full[sb], (g / NSB) & 1, a.err) ||
              !mbar_wait(&v_full[sv], (g / NV) & 1, a.err) ||
              (t == 0 && nz > 0 && !mbar_wait(o_free, (nz - 1) & 1, a.err))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dV = adv(dV0, sv * L::V_BYTES);
#pragma unroll
          for (int ks = 0; ks < BN / L::KSTEP; ++ks) {
            // 8 TMEM columns hold one K step of P (8 tf32, or 16 bf16 in pairs)
            const uint32_t va = ks * L::KSTEP * 128;  // K step = KSTEP rows
            mma_ts<BF16>(tmem + L::T_O, tmem + L::T_S + sb * BN + ks * 8, adv(dV, va), id_o,
                         (t > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(&pv_done[sb]);
          mma_commit(&v_empty[sv]);
          if (t + 2 < it.T && !issue_s(dQ)) {
            ok = false;
            ++g;
            break;
          }
        }
        mma_commit(&q_empty[qb]);
        ++nz;
      }
      mma_commit(final_bar);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int sp = warp & 3, part = (warp - 4) >> 2;
    const int r = sp * 32 + lane;  // query row of the item (TMEM lane)
    const uint32_t lane_base = (uint32_t)(sp * 32) << 16;
    const float c = a.scale_log2e;
    int g = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
      const FwdItem it = fwd_item<BM, BN>(a, n_qt, i);
      const int q = it.q0 + r;
      const bool q_ok = q < a.Sq;
      // this row's visible keys [lo, hi)
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
      const float* mrow = a.has_mask && q_ok ? a.mask + (long long)it.b * a.msb +
                                                   (long long)it.h * a.msh + (long long)q * a.msq
                                             : nullptr;
      const uint32_t bh32 = (uint32_t)it.bh;
      float m = -INFINITY, l = 0.f;
      for (int t = 0; t < it.T; ++t, ++g) {
        const int sb = g % NSB;
        const int kb = it.k_start + t * BN + part * QC;  // first key of this share
        float mv[QC];
#pragma unroll
        for (int e = 0; e < QC; ++e) mv[e] = 0.f;
        if (mrow && kb < hi && kb + QC > lo) {
          if (a.mask_vec) {
            // contiguous, 16-byte aligned mask rows (kb is a multiple of 16)
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
        uint32_t sv[QC];
#pragma unroll
        for (int e = 0; e < QC; ++e) sv[e] = 0u;
        if (ok) ok = fwd_warp_wait(&s_full[sb], (g / NSB) & 1, a.err);
        if (ok) {
          tc_fence_after();
          __syncwarp();
#pragma unroll
          for (int c0 = 0; c0 < QC; c0 += 16) {
            uint32_t rr[16];
            tmem_ld16(tmem + lane_base + L::T_S + sb * BN + part * QC + c0, rr);
#pragma unroll
            for (int e = 0; e < 16; ++e) sv[c0 + e] = rr[e];
          }
          tmem_ld_wait();
        }
        float x[QC];
        float pm = -INFINITY;
        // a share without mask or dropout that lies wholly inside the row's
        // visible keys needs no per-key test: two scores per packed multiply
        const bool plain = !mrow && !a.dropout && kb >= lo && kb + QC <= hi;
        if (plain) {
          const uint64_t c2 = fpk2(c, c);
#pragma unroll
          for (int e = 0; e < QC; e += 2)
            fup2(ff2mul(fpk2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2), x[e],
                 x[e + 1]);
#pragma unroll
          for (int e = 0; e < QC; ++e) pm = fmaxf(pm, x[e]);
        } else {
#pragma unroll
          for (int e = 0; e < QC; ++e) {
            const bool vis = (unsigned)(kb + e - lo) < (unsigned)(hi - lo) && mv[e] > kHardMask;
            x[e] = vis ? fmaf(__uint_as_float(sv[e]), c, mv[e] * kLog2e) : -INFINITY;
            pm = fmaxf(pm, x[e]);
          }
        }
        // the row's maximum over the tile: the four shares meet in shared
        // memory (double-buffered by tile parity); every softmax thread of the
        // sub-partition reaches this barrier on every tile, also after a
        // failed wait
        rmax[((g & 1) * 4 + part) * BM + r] = pm;
        sp_sync(sp);
        float mt = rmax[((g & 1) * 4 + 0) * BM + r];
#pragma unroll
        for (int u = 1; u < 4; ++u) mt = fmaxf(mt, rmax[((g & 1) * 4 + u) * BM + r]);
        // lazy rescale: raise m only when the tile's maximum exceeds it by
        // more than 2^8 (the same decision in all four threads of a row).
        // The decision is per row, i.e. per lane, so the rescale of O below
        // (warp-collective TMEM accesses and a warp-wide wait) runs for the
        // whole warp whenever any lane needs it, with factor 1 in the others.
        float f = 1.f;
        if (mt != -INFINITY) {
          if (m == -INFINITY) {
            m = mt;  // no mass so far: O and l are zero
          } else if (mt > m + kRescaleLog2) {
            f = fwd_ex2(m - mt);
            l *= f;
            m = mt;
          }
        }
        if (t > 0 && ok && __any_sync(0xffffffffu, f != 1.f)) {
          // O *= f on this thread's D/4 columns, after the previous P . V
          const int gp = g - 1;
          ok = fwd_warp_wait(&pv_done[gp % NSB], (gp / NSB) & 1, a.err);
          if (ok) {
            tc_fence_after();
            __syncwarp();
#pragma unroll
            for (int c0 = 0; c0 < OC; c0 += 16) {
              uint32_t ov[16];
              tmem_ld16(tmem + lane_base + L::T_O + part * OC + c0, ov);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
              tmem_st16(tmem + lane_base + L::T_O + part * OC + c0, ov);
            }
            tmem_st_wait();
          }
        }
        // dropout keep bits of the share (bit e: key kb + e) from Philox4x32-10
        // with counter (q >> 2, key, b * H + h, 0), word q & 3.  The four rows
        // of one q >> 2 are lanes 4m .. 4m + 3 of the warp (the item starts at a
        // multiple of 128 rows), so each call serves all four: for keys
        // 4j .. 4j + 3 lane 4m + i computes key 4j + i, and a 4 x 4 transpose by
        // XOR shuffles hands every lane its own word of the four keys
        uint32_t keep = 0xFFFFFFFFu;
        if (a.dropout) {
          keep = 0u;
          const int li = lane & 3;
#pragma unroll 1
          for (int j = 0; j < QC; j += 4) {
            const Philox4 rnd = philox4x32_10((uint32_t)q >> 2, (uint32_t)(kb + j + li), bh32,
                                              0u, a.seed_lo, a.seed_hi);
            // word w of this lane's key belongs to query (q & ~3) + w = lane (lane & ~3) | w
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int w = li ^ m;  // the word the partner lane needs
              const uint32_t send = w == 0 ? rnd.w[0] : w == 1 ? rnd.w[1] : w == 2 ? rnd.w[2] : rnd.w[3];
              // from partner li ^ m: its key j + (li ^ m), our word li
              const uint32_t word = m == 0 ? send : __shfl_xor_sync(0xffffffffu, send, m);
              keep |= (word >= a.drop_threshold ? 1u : 0u) << (j + (li ^ m));
            }
          }
        }
        const float mul = a.dropout ? a.drop_inv_keep : 1.f;
        // P = exp2(x - m) (0 where x = -inf), its row sum without dropout,
        // and P o M written over this share's S columns
        uint32_t pw[QC];
        float ls = 0.f;
        if (m == -INFINITY) {  // nothing visible in the row so far
#pragma unroll
          for (int e = 0; e < QC; ++e) pw[e] = 0u;
        } else if (!a.dropout) {
          // x - m two at a time (exp2(-inf) = 0 for hidden keys), partial sums in pairs
          const uint64_t nm2 = fpk2(-m, -m);
          uint64_t ls2 = fpk2(0.f, 0.f);
#pragma unroll
          for (int e = 0; e < QC; e += 2) {
            float d0, d1;
            fup2(ff2add(fpk2(x[e], x[e + 1]), nm2), d0, d1);
            const float p0 = fwd_ex2(d0), p1 = fwd_ex2(d1);
            ls2 = ff2add(ls2, fpk2(p0, p1));
            pw[e] = __float_as_uint(p0);
            pw[e + 1] = __float_as_uint(p1);
          }
          float l0, l1;
          fup2(ls2, l0, l1);
          ls = l0 + l1;
        } else {
#pragma unroll
          for (int e = 0; e < QC; ++e) {
            const float pe = fwd_ex2(x[e] - m);
            ls += pe;
            pw[e] = __float_as_uint(((keep >> e) & 1u) ? pe * mul : 0.f);
          }
        }
        l += ls;
        if (ok) {
          __syncwarp();
          if constexpr (BF16) {
            // two keys per column, the lower key in the low half
            uint32_t pk[QC / 2];
#pragma unroll
            for (int e = 0; e < QC / 2; ++e)
              pk[e] = fwd_pack_bf16(__uint_as_float(pw[2 * e]), __uint_as_float(pw[2 * e + 1]));
#pragma unroll
            for (int c0 = 0; c0 < QC / 2; c0 += 16) {
              uint32_t st[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) st[e] = pk[c0 + e];
              tmem_st16(tmem + lane_base + L::T_S + sb * BN + part * (QC / 2) + c0, st);
            }
          } else {
#pragma unroll
            for (int c0 = 0; c0 < QC; c0 += 16) {
              uint32_t st[16];
#pragma unroll
              // TF32, rounded to nearest: half a TF32 unit added to the bits
              // (the tensor cores ignore the low 13 bits)
              for (int e = 0; e < 16; ++e) st[e] = pw[c0 + e] + 0x1000u;
              tmem_st16(tmem + lane_base + L::T_S + sb * BN + part * QC + c0, st);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_full[sb]);
        }
      }
      // ---- item epilogue: merge the partial sums, read O, divide, store
      rsum[part * BM + r] = l;
      sp_sync(sp);
      float ll = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) ll += rsum[u * BM + r];
      const bool empty = !(ll > 0.f);
      const float inv = empty ? 0.f : 1.f / ll;
      const long long off =
          row_offset(a.layout, it.b, it.h, q_ok ? q : 0, a.H, a.Sq, D) + part * OC;
      // 16 columns of O at a time: divided by the row sum and stored
      auto store16 = [&](int c0, const float (&o)[16]) {
        if (!q_ok) return;
        if constexpr (BF16) {
          uint4* dst =
              reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.O) + off + c0);
#pragma unroll
          for (int e = 0; e < 16; e += 8)
            dst[e / 8] = make_uint4(fwd_pack_bf16(o[e], o[e + 1]), fwd_pack_bf16(o[e + 2], o[e + 3]),
                                    fwd_pack_bf16(o[e + 4], o[e + 5]),
                                    fwd_pack_bf16(o[e + 6], o[e + 7]));
        } else {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.O) + off + c0);
#pragma unroll
          for (int e = 0; e < 16; e += 4) dst[e / 4] = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
        }
      };
      bool have_o = false;
      if (it.T > 0 && ok) {
        ok = fwd_warp_wait(&pv_done[(g - 1) % NSB], ((g - 1) / NSB) & 1, a.err);
        have_o = ok;
      }
      if (have_o) {
        tc_fence_after();
        __syncwarp();
#pragma unroll
        for (int c0 = 0; c0 < OC; c0 += 16) {
          uint32_t ov[16];
          tmem_ld16(tmem + lane_base + L::T_O + part * OC + c0, ov);
          tmem_ld_wait();
          float o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __uint_as_float(ov[e]) * inv;
          store16(c0, o);
        }
        tc_fence_before();
        mbar_arrive(o_free);
      } else {
        float z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < OC; c0 += 16) store16(c0, z);
      }
      if (q_ok && part == 0)
        a.LSE[(long long)it.bh * a.Sq + q] = empty ? kEmptyRowLse : (m + log2f(ll)) * kFwdLn2;
      sp_sync(sp);  // rsum is reused by the next item
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    fwd_drain(final_bar, 0);
    tc_fence_after();
    tmem_dealloc(tmem, L::T_ALLOC);
  }
}

template <bool BF16, int D>
cudaError_t fwd_impl(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<BF16, D>;
  auto kern = fwd_kernel<BF16, D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const long long items = (long long)((a.Sq + L::BM - 1) / L::BM) * a.B * a.H;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = kFwdSmsFallback;
  const int grid = (int)(items < sms ? items : sms);
  kern<<<grid, kFwdThreads, L::SMEM_BYTES, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

int fwd_block_n(int dtype, int head_dim) {
  if (dtype == ATTN_BF16) return head_dim == 64 ? FwdLayout<true, 64>::BN : FwdLayout<true, 128>::BN;
  return head_dim == 64 ? FwdLayout<false, 64>::BN : FwdLayout<false, 128>::BN;
}

cudaError_t launch_fwd(const attn_bwd_params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdArgs& a, cudaStream_t stream) {
  const bool bf = p.dtype == ATTN_BF16;
  if (p.head_dim == 64)
    return bf ? fwd_impl<true, 64>(tq, tk, tv, a, stream) : fwd_impl<false, 64>(tq, tk, tv, a, stream);
  return bf ? fwd_impl<true, 128>(tq, tk, tv, a, stream) : fwd_impl<false, 128>(tq, tk, tv, a, stream);
}

}  // namespace attnbwd
