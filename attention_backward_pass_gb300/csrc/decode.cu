// Decode (one query per head) attention backward, memory-bound.
//
// The decode page ("rullama attention_backward_dq.wgsl") runs one workgroup
// per query head and sweeps the K/V history three times (d_probs, d_scores,
// then d_q with a strided, uncoalesced k_hist walk).  Here each history
// tensor is read from HBM exactly once for all the G query heads that share
// a KV head, in two passes split at sum_pd_h = sum_j probs_hj dp_hj:
//   decode_dp (reads V):  dp_hj = d_out_h . v_j; parks probs_hj dp_hj in
//                         d_scores; per-CTA partial sums of sum_pd_h
//   decode_dq (reads K):  d_scores_hj = probs_hj dp_hj - probs_hj sum_pd_h
//                         (final values), d_q_h = sum_j d_scores_hj k_j
// The split costs one extra read of the parked values (G floats per key,
// next to the 2 D floats of K and V).  A single pass would need two d_q
// accumulators instead (sum_j probs dp k_j and sum_j probs k_j, combined
// once sum_pd is known): 2 G D multiply-adds per key in place of G D.
//
// Both kernels run one CTA per SM.  The (sequence, KV head) x chunk space
// (chunks of CH keys) is split evenly over the CTAs, identically in both
// passes, so a CTA's range covers one or a few (sequence, KV head) pairs
// ("segments").  A producer warp streams each chunk's K or V rows (one 4-D
// tensor copy) through a ring of NS shared-memory stages, and -- when the
// history length is a multiple of 4 -- the chunk's [G][CH] slices of probs /
// d_scores with one 3-D tensor copy each; the compute warps meet it on
// mbarriers.
//   decode_dp compute warps: lane-split over d (D/32 per lane, d_out held in
//     registers); key groups of warps take interleaved keys of every chunk.
//     Each lane keeps its heads' d_out in an order permuted by its lane bits
//     so that the warp reduction of the G per-key sums is a chain of plain
//     shuffle-adds (no selects); one lane per head ends with the head's dp.
//     probs*dp goes to a staging array of the stage, which the producer
//     writes back with one tensor store when it recycles the stage.
//   decode_dq: two warps form the chunk's G x CH d_scores (coalesced stores,
//     a copy in a small shared ring) ahead of 16 accumulating warps (8 when a
//     KV head serves 16 query heads; four
//     d per thread, KG2 key groups) that add d_q.  The partial d_q of a
//     segment is summed over the key groups in shared memory and written to
//     the workspace; the last CTA of a pair to finish (a counter in the
//     workspace, zeroed by decode_dp) sums the partials in CTA order and
//     writes d_q, so the result does not depend on timing.  decode_dq is a
//     programmatic dependent of decode_dp: its producer streams the first K
//     chunks while decode_dp finishes, and everything that reads decode_dp's
//     outputs waits for it first (griddepcontrol.wait).
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace attnbwd {

namespace {

constexpr int kDecChunk = 64;                 // keys per chunk
constexpr int kDecSmsFallback = 152;

struct DecArgs {
  const float* k;
  const float* v;
  const float* probs;
  const float* d_out;
  float* d_scores;
  float* d_q;
  float* part1;          // decode_dp: partial sum_pd   [grid][max_seg][SLOT1]
  float* part2;          // decode_dq: partial d_q      [grid][max_seg][SLOT2]
  unsigned int* count;   // per (sequence, KV head) pair: decode_dq CTAs done
  int n_heads, n_kv, D, hist;
  int grid;              // CTAs of either kernel
  int cpp;               // chunks per (sequence, KV head) pair
  int n_pairs;
  long long n_chunks;
  int max_seg;           // partial slots per CTA
  int side_tma;          // [G][CH] slices of probs / d_scores move by tensor copies
  unsigned int* err;
};

__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// N consecutive floats (N = 2 or a multiple of 4) from a 4N-byte aligned address.
template <int N>
__device__ __forceinline__ void load_vec(float (&dst)[N], const float* src) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int k = 0; k < N; k += 4) {
      const float4 t = *reinterpret_cast<const float4*>(src + k);
      dst[k] = t.x, dst[k + 1] = t.y, dst[k + 2] = t.z, dst[k + 3] = t.w;
    }
  } else {
    static_assert(N == 2, "load_vec width");
    const float2 t = *reinterpret_cast<const float2*>(src);
    dst[0] = t.x, dst[1] = t.y;
  }
}

// bar.red.or over the `threads` threads of named barrier `id`.
__device__ __forceinline__ bool named_bar_or(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Sum G per-lane values over the warp so that the lanes of head g =
// lane >> (5 - log2 G) all end up holding head g's total: halving exchange
// rounds (each lane keeps the half of the heads its lane bit selects) followed
// by plain butterfly rounds on the single remaining value.
template <int G>
__device__ __forceinline__ float warp_reduce_scatter(float (&x)[G], int lane) {
  int n = G;
  int off = 16;
#pragma unroll
  for (int round = 0; (1 << round) < G; ++round) {
    const int half = n >> 1;
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < G / 2; ++k) {
      if (k < half) {
        const float send = upper ? x[k] : x[k + half];
        const float keep = upper ? x[k + half] : x[k];
        x[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
    n = half;
    off >>= 1;
  }
  float r = x[0];
  for (; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

// Chunk range [f0, f1) of CTA i; the CTA that owns chunk f.  32-bit
// arithmetic whenever the products fit (a 64-bit division is a long software
// sequence on the GPU, and these run inside the kernels' segment changes).
__host__ __device__ __forceinline__ long long dec_begin(long long i, long long n, int grid) {
  if (n * grid < (1LL << 32)) return (long long)((uint32_t)(i * n) / (uint32_t)grid);
  return i * n / grid;
}
__host__ __device__ __forceinline__ int dec_cta_of(long long f, long long n, int grid) {
  if ((f + 1) * grid + n < (1LL << 32))
    return (int)(((uint32_t)((f + 1) * grid) + (uint32_t)n - 1u) / (uint32_t)n) - 1;
  return (int)(((f + 1) * grid + n - 1) / n - 1);
}

// The (sequence, KV head) pair of CTA i's first chunk (cpp chunks per pair).
__device__ __forceinline__ int dec_pair0(int i, long long n, int grid, int cpp) {
  const long long f = dec_begin(i, n, grid);
  return n < (1LL << 31) ? (int)((uint32_t)f / (uint32_t)cpp) : (int)(f / cpp);
}

constexpr int kDecDefer = 8;  // d_q segments whose completion the accumulators defer

constexpr int kDecSmemMax = 227 * 1024;  // dynamic + static shared memory of one CTA

__host__ __device__ constexpr int dec_clamp(int x, int lo, int hi) { return x < lo ? lo : x > hi ? hi : x; }
__host__ __device__ constexpr int dec_round(int x, int m) { return (x + m - 1) / m * m; }

template <int D, int G>
struct DecCfg {
  static constexpr int CH = kDecChunk;                    // keys per chunk
  static constexpr int SIDE = G * CH;                     // floats of one [G][CH] side array
  static constexpr int ROWS_BYTES = CH * D * 4;           // the chunk's K or V rows
  static constexpr int STAGE = dec_round(ROWS_BYTES + 2 * SIDE * 4, 128);
  // decode_dp: stage = [V rows [CH][D] | probs [G][CH] | probs*dp [G][CH]]
  static constexpr int DPL = D / 32;                          // d per lane
  static constexpr int HPW = G * DPL <= 64 ? G : 64 / DPL;    // heads per warp
  static constexpr int LOG_HPW = HPW == 1 ? 0 : HPW == 2 ? 1 : HPW == 4 ? 2 : HPW == 8 ? 3 : 4;
  static constexpr int NHG = G / HPW;                         // head groups
  static constexpr int P1W = 8;                               // compute warps
  static constexpr int KG = P1W / NHG;                        // key groups
  static constexpr int NS1 = dec_clamp((kDecSmemMax - 2048) / STAGE, 2, 12);
  static constexpr int SMEM1 = NS1 * STAGE + 128;             // + alignment slack
  static constexpr int SLOT1 = KG * G;                        // sum_pd[KG][G]
  // decode_dq: stage = [K rows [CH][D] | parked probs*dp | probs]
  static constexpr int P2W = G <= 8 ? 16 : 8;             // accumulating warps
  static constexpr int P2T = 32 * P2W;
  static constexpr int DPT = 4;                           // d per accumulating thread
  static constexpr int KG2 = P2T * DPT / D;               // key groups
  static constexpr int NB = 4;                            // d_scores buffers
  static constexpr int DSW = 2;                           // d_scores warps
  static constexpr int DSB_BYTES = NB * CH * G * 4 + G * D * 4;  // d_scores ring, d_q reduction
  static constexpr int NS2 = dec_clamp((kDecSmemMax - 2048 - DSB_BYTES) / STAGE, 2, 12);
  static constexpr int SMEM2 = NS2 * STAGE + 128;
  static constexpr int SLOT2 = G * D;                     // d_q[G][D]
  static_assert(HPW * DPL <= 64 && G % HPW == 0 && KG >= 1 && CH % KG == 0 && D % 64 == 0 &&
                    D <= 256, "decode_dp split");
  static_assert(KG2 >= 1 && CH % KG2 == 0 && CH % 32 == 0, "decode_dq split");
  static_assert(SMEM1 + 1024 <= kDecSmemMax && SMEM2 + DSB_BYTES + 1024 <= kDecSmemMax,
                "decode shared memory");
};

// DPL = D / 32 values of a row for this lane: 16-byte pieces at 4 lane + 128 q
// (q < DPL / 4), or 8 bytes at 2 lane when DPL = 2, so that a warp's loads
// cover contiguous 512- / 256-byte runs.
template <int DPL>
__device__ __forceinline__ void load_lane(float (&dst)[DPL], const float* row, int lane) {
  if constexpr (DPL % 4 == 0) {
#pragma unroll
    for (int q = 0; q < DPL / 4; ++q) {
      const float4 t = *reinterpret_cast<const float4*>(row + q * 128 + 4 * lane);
      dst[4 * q] = t.x, dst[4 * q + 1] = t.y, dst[4 * q + 2] = t.z, dst[4 * q + 3] = t.w;
    }
  } else {
    static_assert(DPL == 2, "load_lane width");
    const float2 t = *reinterpret_cast<const float2*>(row + 2 * lane);
    dst[0] = t.x, dst[1] = t.y;
  }
}

// Head held in slot 0 after warp_reduce_perm by lane `lane`: its top log2(HPW)
// lane bits, bit-reversed.
template <int LOG>
__device__ __forceinline__ int perm_head(int lane) {
  int m = 0;
#pragma unroll
  for (int r = 0; r < LOG; ++r) m |= ((lane >> (4 - r)) & 1) << (LOG - 1 - r);
  return m;
}

// Warp sums of HPW per-lane values whose slot i holds head i ^ perm_head(lane):
// halving rounds (each lane adds the partner's upper half into its lower half,
// which with that slot order is always the same head), then butterflies.
// Every lane returns the total of head perm_head(lane).
template <int HPW>
__device__ __forceinline__ float warp_reduce_perm(float (&x)[HPW]) {
  int off = 16;
#pragma unroll
  for (int n = HPW; n > 1; n >>= 1, off >>= 1) {
#pragma unroll
    for (int k = 0; k < n / 2; ++k) x[k] += __shfl_xor_sync(0xffffffffu, x[k + n / 2], off);
  }
  float r = x[0];
#pragma unroll
  for (; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
  return r;
}

// --------------------------------------------------------------- decode_dp
// tm_v: V as {D, n_kv, hist, seqs}, boxes {D, 1, CH, 1}.
// tm_p, tm_s: probs / d_scores as {hist, n_heads, seqs}, boxes {CH, G, 1}.
template <int D, int G>
__global__ void __launch_bounds__(32 * (1 + DecCfg<D, G>::P1W), 1)
    decode_dp_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_p,
                     const __grid_constant__ CUtensorMap tm_s, const DecArgs a) {
  using C = DecCfg<D, G>;
  constexpr int CH = C::CH, NS = C::NS1, DPL = C::DPL, HPW = C::HPW, KG = C::KG, P1W = C::P1W;
  extern __shared__ uint8_t smem_raw[];
  // [NS][V rows [CH][D] | probs [G][CH] | probs * dp [G][CH]], 128-byte aligned
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ __align__(8) uint64_t full[NS], empty[NS];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long f0 = dec_begin(blockIdx.x, a.n_chunks, a.grid);
  const long long f1 = dec_begin(blockIdx.x + 1, a.n_chunks, a.grid);
  const int nch = (int)(f1 - f0);
  const int pair0 = (int)(f0 / a.cpp), lc0 = (int)(f0 % a.cpp);

  if (blockIdx.x == 0)  // decode_dq's per-pair completion counters
    for (int i = threadIdx.x; i < a.n_pairs; i += blockDim.x) a.count[i] = 0u;
  // decode_dq may start its CTAs (and stream K) as SMs free up; it waits for
  // this grid before it reads anything written here
  if (threadIdx.x == 0) griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], P1W);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // write the probs*dp staging array of chunk c (pair pp, chunk lc) back to d_scores
      auto park = [&](int c, int pp, int lc) {
        tma_store_3d(&tm_s, smem + (c % NS) * C::STAGE + C::ROWS_BYTES + C::SIDE * 4, lc * CH,
                     (pp % a.n_kv) * G, pp / a.n_kv);  // keys >= hist are clipped
        bulk_commit();
      };
      bool ok = true;
      int issued = 0;
      int pair = pair0, lc = lc0;     // chunk c
      int ppair = pair0, plc = lc0;   // chunk c - NS (next to write back)
      for (int c = 0; c < nch; ++c) {
        const int s = c % NS;
        if (c >= NS) {
          if (!mbar_wait(&empty[s], ((c / NS) - 1) & 1, a.err)) {
            ok = false;
            break;
          }
          if (a.side_tma) {
            park(c - NS, ppair, plc);
            bulk_wait_read();  // the staging array is rewritten after this chunk lands
          }
          if (++plc == a.cpp) plc = 0, ++ppair;
        }
        const int seq = pair / a.n_kv, kv = pair % a.n_kv, j0 = lc * CH;
        uint8_t* st = smem + s * C::STAGE;
        mbar_expect_tx(&full[s], C::ROWS_BYTES + (a.side_tma ? C::SIDE * 4u : 0u));
        tma_load_4d(st, &tm_v, &full[s], 0, kv, j0, seq);
        if (a.side_tma) tma_load_3d(st + C::ROWS_BYTES, &tm_p, &full[s], j0, kv * G, seq);
        issued = c + 1;
        if (++lc == a.cpp) lc = 0, ++pair;
      }
      // the last chunks: wait for their consumers, write their staging arrays back
      for (int c = issued > NS ? issued - NS : 0; ok && c < issued; ++c) {
        if (!mbar_wait(&empty[c % NS], (c / NS) & 1, a.err)) {
          ok = false;
          break;
        }
        if (a.side_tma) park(c, ppair, plc);
        if (++plc == a.cpp) plc = 0, ++ppair;
      }
      if (!ok) {  // copies still in flight land before the CTA exits
        for (int c = issued > NS ? issued - NS : 0; c < issued; ++c) {
          const long long t0 = clock64();
          while (!mbar_try_wait(&full[c % NS], (c / NS) & 1) &&
                 clock64() - t0 < kWaitLimitCycles / 4) {
          }
        }
      }
      bulk_wait_all();
    }
    __syncwarp();
    return;
  }

  // -------------------------------------------------------------- compute
  // Warp (kgp, hg) takes keys kgp, kgp + KG, .. of every chunk for the HPW
  // heads of head group hg.  Lane-split over d (DPL per lane), d_out in
  // registers with slot i holding head i ^ perm_head(lane), so that
  // warp_reduce_perm needs no selects; lane `lane` ends with head g_own.
  const int pw = warp - 1, kgp = pw % KG, hg = pw / KG;
  const int g_own = perm_head<C::LOG_HPW>(lane);
  const bool owner = (lane & ((32 >> C::LOG_HPW) - 1)) == 0;  // one lane per head writes
  float* slots = a.part1 + (size_t)blockIdx.x * a.max_seg * C::SLOT1;
  float dout[HPW][DPL];
  float sumpd = 0.f;
  int cur_pair = -1, seg = -1;
  int pair = pair0, lc = lc0, seq = pair0 / a.n_kv, kv = pair0 % a.n_kv;
  bool ok = true;
  for (int c = 0; c < nch; ++c) {
    const int j0 = lc * CH, rows = min(CH, a.hist - j0);
    const int h_own = kv * G + hg * HPW + g_own;  // query head of this lane's sums
    if (pair != cur_pair) {
      if (seg >= 0 && owner) slots[(size_t)seg * C::SLOT1 + kgp * G + hg * HPW + g_own] = sumpd;
      sumpd = 0.f;
      cur_pair = pair;
      seg = pair - pair0;
#pragma unroll
      for (int i = 0; i < HPW; ++i)
        load_lane<DPL>(dout[i],
                       a.d_out + ((size_t)seq * a.n_heads + kv * G + hg * HPW + (i ^ g_own)) * D, lane);
    }
    const int s = c % NS;
    ok = mbar_wait(&full[s], (c / NS) & 1, a.err);
    ok = !__any_sync(0xffffffffu, !ok);
    if (!ok) break;
    uint8_t* st = smem + s * C::STAGE;
    const float* vs = reinterpret_cast<const float*>(st);
    const float* ps = reinterpret_cast<const float*>(st + C::ROWS_BYTES) + (hg * HPW + g_own) * CH;
    float* ws = reinterpret_cast<float*>(st + C::ROWS_BYTES + C::SIDE * 4) + (hg * HPW + g_own) * CH;
    const size_t grow = ((size_t)seq * a.n_heads + h_own) * a.hist + j0;
    // dp of key jj for this warp's heads (every lane; no branch, so that the
    // keys of a chunk interleave)
    auto key_dot = [&](int jj) {
      float vv[DPL];
      load_lane<DPL>(vv, vs + jj * D, lane);
      // packed products over consecutive d (even and odd partial sums)
      float part[HPW];
#pragma unroll
      for (int i = 0; i < HPW; ++i) {
        uint64_t acc = 0;
#pragma unroll
        for (int k = 0; k < DPL; k += 2)
          acc = f2fma(pk2(dout[i][k], dout[i][k + 1]), pk2(vv[k], vv[k + 1]), acc);
        float lo, hi;
        up2(acc, lo, hi);
        part[i] = lo + hi;
      }
      return warp_reduce_perm<HPW>(part);
    };
    // the owner lanes form probs * dp
    auto own = [&](int jj, float dp) {
      const float pj = a.side_tma ? ps[jj] : __ldg(a.probs + grow + jj);
      const float w = pj * dp;
      sumpd += w;
      if (a.side_tma)
        ws[jj] = w;
      else
        a.d_scores[grow + jj] = w;
    };
    if (rows == CH) {  // full chunk
      float dps[CH / KG];
#pragma unroll
      for (int i = 0; i < CH / KG; ++i) dps[i] = key_dot(kgp + KG * i);
      if (owner) {
#pragma unroll
        for (int i = 0; i < CH / KG; ++i) own(kgp + KG * i, dps[i]);
      }
    } else {
      for (int i = 0; i < CH / KG; ++i) {
        if (kgp + KG * i < rows) {  // warp-uniform
          const float dp = key_dot(kgp + KG * i);
          if (owner) own(kgp + KG * i, dp);
        }
      }
    }
    if (a.side_tma) fence_proxy_async_smem();  // the staging array is read by a tensor store
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (++lc == a.cpp) {
      lc = 0, ++pair;
      if (++kv == a.n_kv) kv = 0, ++seq;
    }
  }
  if (ok && seg >= 0 && owner) slots[(size_t)seg * C::SLOT1 + kgp * G + hg * HPW + g_own] = sumpd;
}

// --------------------------------------------------------------- decode_dq
// tm_k: K as {D, n_kv, hist, seqs}, boxes {D, 1, CH, 1}.
// Warps: 0 producer; 1 .. P2W accumulate d_q (P2T threads, DPT d each, KG2
// key groups); the last DSW warps form each chunk's d_scores (each warp every
// DSW-th head) into a ring of NB shared buffers, ahead of the accumulating
// warps.
template <int D, int G>
__global__ void __launch_bounds__(32 * (1 + DecCfg<D, G>::P2W + DecCfg<D, G>::DSW), 1)
    decode_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_p,
                     const __grid_constant__ CUtensorMap tm_s, const DecArgs a) {
  using C = DecCfg<D, G>;
  constexpr int CH = C::CH, NS = C::NS2, NB = C::NB, P2T = C::P2T, P2W = C::P2W, KG2 = C::KG2;
  constexpr int DPT = C::DPT, DSW = C::DSW;
  constexpr int NACC = G == 1 ? DPT / 2 : DPT * (G / 2);  // packed accumulators
  extern __shared__ uint8_t smem_raw[];
  // [NS][K rows [CH][D] | parked probs * dp [G][CH] | probs [G][CH]], 128-byte aligned
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ __align__(16) float dsb[NB][CH][G];  // chunks' d_scores, key-major
  __shared__ __align__(16) float red[G * D];      // the CTA's d_q partial of a segment
  __shared__ int dpair_s[kDecDefer], dlast_s[kDecDefer];  // deferred segment completions
  __shared__ __align__(8) uint64_t full[NS], empty[NS], ds_full[NB], ds_empty[NB];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long f0 = dec_begin(blockIdx.x, a.n_chunks, a.grid);
  const long long f1 = dec_begin(blockIdx.x + 1, a.n_chunks, a.grid);
  const int nch = (int)(f1 - f0);
  const int pair0 = (int)(f0 / a.cpp), lc0 = (int)(f0 % a.cpp);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], P2W + DSW);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&ds_full[b], 32 * DSW);
      mbar_init(&ds_empty[b], P2W);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int issued = 0;
      int pair = pair0, lc = lc0;  // chunk c
      // The first NS chunks' K rows and probs are requested before the d_p
      // pass has finished; their parked probs*dp slices (written by it) only
      // after griddep_wait.
      int pre_seq[NS], pre_kv[NS], pre_j0[NS];
      const int pre = nch < NS ? nch : NS;
      for (int c = 0; c < nch; ++c) {
        const int s = c % NS;
        if (c >= NS && !mbar_wait(&empty[s], ((c / NS) - 1) & 1, a.err)) break;
        const int seq = pair / a.n_kv, kv = pair % a.n_kv;
        const int j0 = lc * CH;
        if (++lc == a.cpp) lc = 0, ++pair;
        uint8_t* st = smem + s * C::STAGE;
        mbar_expect_tx(&full[s], C::ROWS_BYTES + (a.side_tma ? 2u * C::SIDE * 4u : 0u));
        tma_load_4d(st, &tm_k, &full[s], 0, kv, j0, seq);
        if (a.side_tma) {
          tma_load_3d(st + C::ROWS_BYTES + C::SIDE * 4, &tm_p, &full[s], j0, kv * G, seq);
          if (c < pre) {
            pre_seq[c] = seq, pre_kv[c] = kv, pre_j0[c] = j0;
          } else {
            tma_load_3d(st + C::ROWS_BYTES, &tm_s, &full[s], j0, kv * G, seq);
          }
        }
        issued = c + 1;
        if (c + 1 == pre) {
          griddep_wait();
          if (a.side_tma)
            for (int i = 0; i < pre; ++i)
              tma_load_3d(smem + i * C::STAGE + C::ROWS_BYTES, &tm_s, &full[i], pre_j0[i],
                          pre_kv[i] * G, pre_seq[i]);
        }
      }
      if (issued < pre) griddep_wait();  // (left early on an error)
      // copies still in flight land before the CTA exits
      for (int c = issued > NS ? issued - NS : 0; c < issued; ++c) {
        const long long t0 = clock64();
        while (!mbar_try_wait(&full[c % NS], (c / NS) & 1) && clock64() - t0 < kWaitLimitCycles / 4) {
        }
      }
    }
    __syncwarp();
    return;
  }

  if (warp > P2W) {
    // ------------------------------------------------------ d_scores warps
    // lane j = keys j, j + 32, .. of the chunk: d_scores = probs*dp - probs * sum_pd for
    // heads dw, dw + DSW, ..., stored to global memory and to dsb
    const int dw = warp - 1 - P2W;
    griddep_wait();  // sum_pd partials and parked values come from decode_dp
    float sp[G];  // sum_pd of the current pair, every head
    int cur = -1;
    int pair = pair0, lc = lc0, seq = pair0 / a.n_kv, kv = pair0 % a.n_kv;
    for (int c = 0; c < nch; ++c) {
      const int j0 = lc * CH, rows = min(CH, a.hist - j0);
      if (pair != cur) {
        // sum_pd of the pair from decode_dp's partials: the lanes load the
        // (CTA, key group, head) terms side by side, lane l only terms of
        // head l % G, then lanes of equal l % G are summed
        cur = pair;
        const long long fa = (long long)pair * a.cpp;
        const int ia = dec_cta_of(fa, a.n_chunks, a.grid);
        const int ib = dec_cta_of(fa + a.cpp - 1, a.n_chunks, a.grid);
        const int nt = (ib - ia + 1) * C::SLOT1;
        float v = 0.f;
#pragma unroll 4
        for (int t = lane; t < nt; t += 32) {
          const int i = ia + t / C::SLOT1;
          const int sg = pair - (int)(dec_begin(i, a.n_chunks, a.grid) / a.cpp);
          v += a.part1[((size_t)i * a.max_seg + sg) * C::SLOT1 + t % C::SLOT1];
        }
#pragma unroll
        for (int off = 16; off >= G; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
#pragma unroll
        for (int g = 0; g < G; ++g) sp[g] = __shfl_sync(0xffffffffu, v, g);
      }
      const int s = c % NS, b = c % NB;
      bool ok = mbar_wait(&full[s], (c / NS) & 1, a.err) &&
                (c < NB || mbar_wait(&ds_empty[b], ((c / NB) - 1) & 1, a.err));
      if (__any_sync(0xffffffffu, !ok)) break;
      const float* wsd = reinterpret_cast<const float*>(smem + s * C::STAGE + C::ROWS_BYTES);
      const float* psd = wsd + C::SIDE;
#pragma unroll
      for (int r = 0; r < CH / 32; ++r) {
        const int jl = lane + 32 * r;  // key of the chunk
        const bool in = jl < rows;
        const size_t gi0 = ((size_t)seq * a.n_heads + kv * G) * a.hist + j0 + jl;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (g % DSW != dw) continue;
          float w, pv;
          if (a.side_tma) {
            w = wsd[g * CH + jl];
            pv = psd[g * CH + jl];
          } else {
            w = in ? a.d_scores[gi0 + (size_t)g * a.hist] : 0.f;
            pv = in ? __ldg(a.probs + gi0 + (size_t)g * a.hist) : 0.f;
          }
          const float ds = fmaf(-pv, sp[g], w);
          if (in) a.d_scores[gi0 + (size_t)g * a.hist] = ds;
          dsb[b][jl][g] = ds;
        }
      }
      mbar_arrive(&ds_full[b]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++lc == a.cpp) {
        lc = 0, ++pair;
        if (++kv == a.n_kv) kv = 0, ++seq;
      }
    }
    return;
  }

  // -------------------------------------------------------- accumulators
  // Thread t2 (key group kg, index tk within it) owns DPT head-dim elements:
  // dd(i) = 4 tk + i for i < 4 and, when DPT = 8, D / 2 + 4 tk + i - 4 (two
  // 16-byte pieces, so a warp's loads cover contiguous runs), for the keys kg,
  // kg + KG2, ... of every chunk.  For even G the packed accumulators pair
  // consecutive heads: acc[i (G/2) + hp] = (d_q[2hp][dd(i)], d_q[2hp+1][dd(i)]);
  // for G = 1, acc[i] = (d_q[0][dd(2i)], d_q[0][dd(2i+1)]).
  griddep_wait();  // the pair counters are zeroed by decode_dp
  const int t2 = threadIdx.x - 32;
  const int kg = t2 / (D / DPT), tk = t2 % (D / DPT);
  auto dd = [&](int i) { return i < 4 ? 4 * tk + i : D / 2 + 4 * tk + i - 4; };
  float* slots = a.part2 + (size_t)blockIdx.x * a.max_seg * C::SLOT2;
  uint64_t acc[NACC];
#pragma unroll
  for (int i = 0; i < NACC; ++i) acc[i] = 0;
  int cur_pair = -1, seg = -1;
  bool ok = true;

  // Completion of the deferred segments: make this CTA's partials visible,
  // count this CTA in for each of their pairs, and let the last CTA of a pair
  // sum the partials in CTA order and write d_q.  Deferred to the end of the
  // chunk loop (or until kDecDefer are pending) because every global round
  // trip costs microseconds under the streaming load.
  int ndef = 0;
  auto complete = [&]() {
    __threadfence();
    named_bar_sync(1, P2T);
    if (t2 == 0) {
      for (int k = 0; k < ndef; ++k) {
        const long long fa = (long long)dpair_s[k] * a.cpp;
        const int ia = dec_cta_of(fa, a.n_chunks, a.grid);
        const int ib = dec_cta_of(fa + a.cpp - 1, a.n_chunks, a.grid);
        dlast_s[k] = ia == ib || atomicAdd(&a.count[dpair_s[k]], 1u) == (unsigned)(ib - ia);
      }
    }
    named_bar_sync(1, P2T);
    for (int k = 0; k < ndef; ++k) {
      if (!dlast_s[k]) continue;
      __threadfence();
      const int p = dpair_s[k];
      const long long fa = (long long)p * a.cpp;
      const int ia = dec_cta_of(fa, a.n_chunks, a.grid);
      const int ib = dec_cta_of(fa + a.cpp - 1, a.n_chunks, a.grid);
      const int seq = p / a.n_kv, kv = p % a.n_kv;
      constexpr int NO = (G * D + P2T - 1) / P2T;  // outputs per thread
      float t[NO];
#pragma unroll
      for (int q = 0; q < NO; ++q) t[q] = 0.f;
      for (int i = ia; i <= ib; ++i) {
        const int sg = p - dec_pair0(i, a.n_chunks, a.grid, a.cpp);
        const float* p2 = a.part2 + ((size_t)i * a.max_seg + sg) * C::SLOT2;
#pragma unroll
        for (int q = 0; q < NO; ++q)
          if (t2 + q * P2T < G * D) t[q] += __ldcg(p2 + t2 + q * P2T);
      }
#pragma unroll
      for (int q = 0; q < NO; ++q)
        if (t2 + q * P2T < G * D) a.d_q[((size_t)seq * a.n_heads + kv * G) * D + t2 + q * P2T] = t[q];
    }
    named_bar_sync(1, P2T);  // dpair_s / dlast_s may be reused
    ndef = 0;
  };

  // segment `seg` (pair cur_pair) is complete in this CTA: sum the key
  // groups in shared memory (in key-group order) and store the CTA's partial;
  // its completion is deferred
  auto finish = [&]() {
    float x[G][DPT];
    if constexpr (G == 1) {
#pragma unroll
      for (int i = 0; i < DPT / 2; ++i) up2(acc[i], x[0][2 * i], x[0][2 * i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < DPT; ++i)
#pragma unroll
        for (int hp = 0; hp < G / 2; ++hp) up2(acc[i * (G / 2) + hp], x[2 * hp][i], x[2 * hp + 1][i]);
    }
    for (int r = 0; r < KG2; ++r) {
      if (kg == r) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int q = 0; q < DPT / 4; ++q) {
            float4* dst = reinterpret_cast<float4*>(red + g * D + dd(4 * q));
            float4 v = make_float4(x[g][4 * q], x[g][4 * q + 1], x[g][4 * q + 2], x[g][4 * q + 3]);
            if (r > 0) {
              const float4 o = *dst;
              v.x += o.x, v.y += o.y, v.z += o.z, v.w += o.w;
            }
            *dst = v;
          }
      }
      named_bar_sync(1, P2T);
    }
    float* sl = slots + (size_t)seg * C::SLOT2;
    for (int o = 4 * t2; o < G * D; o += 4 * P2T)
      *reinterpret_cast<float4*>(sl + o) = *reinterpret_cast<const float4*>(red + o);
    if (t2 == 0) dpair_s[ndef] = cur_pair;
    ++ndef;
    named_bar_sync(1, P2T);  // red read out; dpair_s written
    if (ndef == kDecDefer) complete();
  };

  int pair = pair0, lc = lc0;
  for (int c = 0; c < nch; ++c) {
    const int rows = min(CH, a.hist - lc * CH);
    if (pair != cur_pair) {
      if (seg >= 0) finish();
      cur_pair = pair;
      seg = pair - pair0;
#pragma unroll
      for (int i = 0; i < NACC; ++i) acc[i] = 0;
    }
    const int s = c % NS, b = c % NB;
    ok = mbar_wait(&full[s], (c / NS) & 1, a.err) && mbar_wait(&ds_full[b], (c / NB) & 1, a.err);
    if (named_bar_or(1, P2T, !ok)) {  // every accumulating thread leaves together
      ok = false;
      break;
    }
    const float* ks = reinterpret_cast<const float*>(smem + s * C::STAGE);
    auto key_dq = [&](int jj) {
      float kk[DPT];
#pragma unroll
      for (int q = 0; q < DPT / 4; ++q) {
        const float4 t = *reinterpret_cast<const float4*>(ks + jj * D + dd(4 * q));
        kk[4 * q] = t.x, kk[4 * q + 1] = t.y, kk[4 * q + 2] = t.z, kk[4 * q + 3] = t.w;
      }
      if constexpr (G == 1) {
        const float dv = dsb[b][jj][0];
        const uint64_t d2 = pk2(dv, dv);
#pragma unroll
        for (int i = 0; i < DPT / 2; ++i) acc[i] = f2fma(d2, pk2(kk[2 * i], kk[2 * i + 1]), acc[i]);
      } else {
        uint64_t w2[G / 2];
        if constexpr (G == 2) {
          w2[0] = *reinterpret_cast<const uint64_t*>(&dsb[b][jj][0]);
        } else {
#pragma unroll
          for (int hp = 0; hp < G / 2; hp += 2) {
            const ulonglong2 t = *reinterpret_cast<const ulonglong2*>(&dsb[b][jj][2 * hp]);
            w2[hp] = t.x, w2[hp + 1] = t.y;
          }
        }
#pragma unroll
        for (int i = 0; i < DPT; ++i) {
          const uint64_t kd = pk2(kk[i], kk[i]);
#pragma unroll
          for (int hp = 0; hp < G / 2; ++hp)
            acc[i * (G / 2) + hp] = f2fma(w2[hp], kd, acc[i * (G / 2) + hp]);
        }
      }
    };
    if (rows == CH) {
#pragma unroll
      for (int i = 0; i < CH / KG2; ++i) key_dq(kg + KG2 * i);
    } else {
      for (int jj = kg; jj < rows; jj += KG2) key_dq(jj);
    }
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[s]);
      mbar_arrive(&ds_empty[b]);
    }
    if (++lc == a.cpp) lc = 0, ++pair;
  }
  if (ok && seg >= 0) {
    finish();
    complete();
  }
}

template <int D, int G>
cudaError_t decode_impl(const DecArgs& a, cudaStream_t stream) {
  using C = DecCfg<D, G>;
  const long long seqs = a.n_pairs / a.n_kv;
  CUtensorMap tm_v, tm_k, tm_p, tm_s;
  memset(&tm_p, 0, sizeof(tm_p));
  memset(&tm_s, 0, sizeof(tm_s));
  {
    const long long dims[4] = {D, a.n_kv, a.hist, seqs};
    const int box[4] = {D, 1, C::CH, 1};
    if (make_f32_map(&tm_v, a.v, 4, dims, box, false) != CUDA_SUCCESS ||
        make_f32_map(&tm_k, a.k, 4, dims, box, false) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (a.side_tma) {
    const long long dims[3] = {a.hist, a.n_heads, seqs};
    const int box[3] = {C::CH, G, 1};
    if (make_f32_map(&tm_p, a.probs, 3, dims, box, false) != CUDA_SUCCESS ||
        make_f32_map(&tm_s, a.d_scores, 3, dims, box, false) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto k1 = decode_dp_kernel<D, G>;
  auto k2 = decode_dq_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM1);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM2);
  if (e != cudaSuccess) return e;
  k1<<<a.grid, 32 * (1 + C::P1W), C::SMEM1, stream>>>(tm_v, tm_p, tm_s, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // decode_dq may begin while decode_dp finishes (programmatic dependent
  // launch); it synchronises with griddep_wait before using dp's outputs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(32 * (1 + C::P2W + C::DSW));
  cfg.dynamicSmemBytes = C::SMEM2;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k2, tm_k, tm_p, tm_s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int D, int G>
void decode_slots(int& s1, int& s2) {
  s1 = DecCfg<D, G>::SLOT1;
  s2 = DecCfg<D, G>::SLOT2;
}

// Slot sizes of the two kernels for a supported (D, G); false otherwise.
template <int D>
bool dec_slots_by_group(int G, int& s1, int& s2) {
  switch (G) {
    case 1: decode_slots<D, 1>(s1, s2); return true;
    case 2: decode_slots<D, 2>(s1, s2); return true;
    case 4: decode_slots<D, 4>(s1, s2); return true;
    case 8: decode_slots<D, 8>(s1, s2); return true;
    case 16: decode_slots<D, 16>(s1, s2); return true;
    default: return false;
  }
}
bool dec_slots(int D, int G, int& s1, int& s2) {
  switch (D) {
    case 64: return dec_slots_by_group<64>(G, s1, s2);
    case 128: return dec_slots_by_group<128>(G, s1, s2);
    case 256: return dec_slots_by_group<256>(G, s1, s2);
    default: return false;
  }
}

template <int D>
cudaError_t decode_by_group(const DecArgs& a, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return decode_impl<D, 1>(a, stream);
    case 2: return decode_impl<D, 2>(a, stream);
    case 4: return decode_impl<D, 4>(a, stream);
    case 8: return decode_impl<D, 8>(a, stream);
    case 16: return decode_impl<D, 16>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

long long dec_chunks(const attn_bwd_decode_params& p) {
  const long long cpp = (p.history_len + kDecChunk - 1) / kDecChunk;
  return (long long)p.num_seqs * p.n_kv_heads * cpp;
}

// Partial slots one CTA needs: the most (sequence, KV head) pairs a range of
// ceil(n / grid) chunks can touch.
int dec_max_seg(const attn_bwd_decode_params& p, int grid) {
  const long long cpp = (p.history_len + kDecChunk - 1) / kDecChunk;
  const long long n = dec_chunks(p);
  const long long per = (n + grid - 1) / grid;
  return (int)((per + cpp - 1) / cpp + 1);
}

}  // namespace

// Number of CTAs of either decode kernel: one per SM of the current device
// (152 when no device can be queried), at most one per chunk.
int decode_num_splits(const attn_bwd_decode_params& p) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0) {
    cudaGetLastError();  // clear the error of a host without a device
    sms = kDecSmsFallback;
  }
  const long long n = dec_chunks(p);
  return (int)(n < sms ? n : sms);
}

// Workspace floats: both kernels' partial slots, then one counter per pair.
size_t decode_partials_floats(const attn_bwd_decode_params& p, int n_split) {
  int s1 = 0, s2 = 0;
  if (!dec_slots(p.head_dim, p.n_heads / p.n_kv_heads, s1, s2)) return 0;
  const size_t per_cta = (size_t)dec_max_seg(p, n_split) * (s1 + s2);
  return (size_t)n_split * per_cta + (size_t)p.num_seqs * p.n_kv_heads;
}

cudaError_t launch_decode(const attn_bwd_decode_params& p, const float* k_hist,
                          const float* v_hist, const float* probs, const float* d_out,
                          float* d_scores, float* d_q, float* partials, int n_split,
                          cudaStream_t stream) {
  const int G = p.n_heads / p.n_kv_heads;
  int s1 = 0, s2 = 0;
  if (!dec_slots(p.head_dim, G, s1, s2)) return cudaErrorInvalidValue;
  DecArgs a;
  a.k = k_hist;
  a.v = v_hist;
  a.probs = probs;
  a.d_out = d_out;
  a.d_scores = d_scores;
  a.d_q = d_q;
  a.n_heads = p.n_heads;
  a.n_kv = p.n_kv_heads;
  a.D = p.head_dim;
  a.hist = p.history_len;
  a.cpp = (p.history_len + kDecChunk - 1) / kDecChunk;
  a.n_pairs = p.num_seqs * p.n_kv_heads;
  a.n_chunks = dec_chunks(p);
  a.grid = n_split;
  a.max_seg = dec_max_seg(p, n_split);
  a.part1 = partials;
  a.part2 = partials + (size_t)n_split * a.max_seg * s1;
  a.count = reinterpret_cast<unsigned int*>(a.part2 + (size_t)n_split * a.max_seg * s2);
  // the [.., hist] tensor maps need a 16-byte row stride (every pointer is
  // 16-byte aligned, checked by the API)
  a.side_tma = p.history_len % 4 == 0;
  a.err = device_error_word();
  if (!a.err) return cudaErrorUnknown;
  if (a.grid < 1 || a.grid > a.n_chunks) return cudaErrorInvalidValue;
  switch (p.head_dim) {
    case 64: return decode_by_group<64>(a, G, stream);
    case 128: return decode_by_group<128>(a, G, stream);
    case 256: return decode_by_group<256>(a, G, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attnbwd


// ------------------------------------------------------------------------
// Decode backward, pass 2: the history's gradients
//   d_k_hist[j, kv] = sum_h d_scores_hj q_h,  d_v_hist[j, kv] = sum_h probs_hj d_out_h
// over the G query heads h of KV head kv (the decode page's pass 2 consumes
// pass 1's d_scores and takes q; these are the gradients of its forward).
// Bound by the two history-sized writes.  One CTA per (pair, chunk of 64
// keys): its threads stage the chunk's d_scores / probs slices [key][head] in
// shared memory with coalesced loads, hold q and d_out of the group for their
// DPT head-dim elements in registers, and write each key row with contiguous
// vector stores.
// ------------------------------------------------------------------------
namespace attnbwd {
namespace {

constexpr int kKvChunk = 64;
constexpr int kKvThreads = 256;

struct KvArgs {
  const float* q;
  const float* probs;
  const float* d_out;
  const float* d_scores;
  float* d_k;
  float* d_v;
  int n_heads, n_kv, hist, cpp;
};

template <int D, int G>
__global__ void __launch_bounds__(kKvThreads) decode_kv_kernel(const KvArgs a) {
  constexpr int CH = kKvChunk;
  constexpr int DPT = G <= 8 ? 4 : 2;  // head-dim elements per thread
  constexpr int TPK = D / DPT;         // threads per key row
  constexpr int KGRP = kKvThreads / TPK;
  static_assert(TPK <= kKvThreads && CH % KGRP == 0, "decode_kv split");
  __shared__ __align__(16) float ds_s[CH][G];
  __shared__ __align__(16) float pr_s[CH][G];
  const int pair = (int)(blockIdx.x / (unsigned)a.cpp), lc = (int)(blockIdx.x % (unsigned)a.cpp);
  const int seq = pair / a.n_kv, kv = pair % a.n_kv;
  const int j0 = lc * CH, rows = min(CH, a.hist - j0);
  const int t = threadIdx.x, kg = t / TPK, d = DPT * (t % TPK);
  const size_t hrow = (size_t)seq * a.n_heads + kv * G;  // first query head of the group
  for (int i = t; i < G * CH; i += kKvThreads) {
    const int g = i / CH, jj = i % CH;
    float ds = 0.f, pv = 0.f;
    if (jj < rows) {
      const size_t gi = (hrow + g) * a.hist + j0 + jj;
      ds = __ldg(a.d_scores + gi);
      pv = __ldg(a.probs + gi);
    }
    ds_s[jj][g] = ds;
    pr_s[jj][g] = pv;
  }
  // packed (d, d+1) pairs of q and d_out for every head of the group
  uint64_t q2[G][DPT / 2], o2[G][DPT / 2];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float* qr = a.q + (hrow + g) * D + d;
    const float* orow = a.d_out + (hrow + g) * D + d;
    if constexpr (DPT == 4) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(qr));
      const float4 y = __ldg(reinterpret_cast<const float4*>(orow));
      q2[g][0] = pk2(x.x, x.y), q2[g][1] = pk2(x.z, x.w);
      o2[g][0] = pk2(y.x, y.y), o2[g][1] = pk2(y.z, y.w);
    } else {
      const float2 x = __ldg(reinterpret_cast<const float2*>(qr));
      const float2 y = __ldg(reinterpret_cast<const float2*>(orow));
      q2[g][0] = pk2(x.x, x.y);
      o2[g][0] = pk2(y.x, y.y);
    }
  }
  __syncthreads();
  for (int jj = kg; jj < rows; jj += KGRP) {
    uint64_t dk[DPT / 2], dv[DPT / 2];
#pragma unroll
    for (int i = 0; i < DPT / 2; ++i) dk[i] = dv[i] = 0;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float ds = ds_s[jj][g], pv = pr_s[jj][g];
      const uint64_t ds2 = pk2(ds, ds), pv2 = pk2(pv, pv);
#pragma unroll
      for (int i = 0; i < DPT / 2; ++i) {
        dk[i] = f2fma(ds2, q2[g][i], dk[i]);
        dv[i] = f2fma(pv2, o2[g][i], dv[i]);
      }
    }
    const size_t row = (((size_t)seq * a.hist + j0 + jj) * a.n_kv + kv) * D + d;
    if constexpr (DPT == 4) {
      float x0, x1, x2, x3;
      up2(dk[0], x0, x1);
      up2(dk[1], x2, x3);
      *reinterpret_cast<float4*>(a.d_k + row) = make_float4(x0, x1, x2, x3);
      up2(dv[0], x0, x1);
      up2(dv[1], x2, x3);
      *reinterpret_cast<float4*>(a.d_v + row) = make_float4(x0, x1, x2, x3);
    } else {
      float x0, x1;
      up2(dk[0], x0, x1);
      *reinterpret_cast<float2*>(a.d_k + row) = make_float2(x0, x1);
      up2(dv[0], x0, x1);
      *reinterpret_cast<float2*>(a.d_v + row) = make_float2(x0, x1);
    }
  }
}

template <int D>
cudaError_t kv_by_group(const KvArgs& a, int G, unsigned grid, cudaStream_t stream) {
  switch (G) {
    case 1: decode_kv_kernel<D, 1><<<grid, kKvThreads, 0, stream>>>(a); break;
    case 2: decode_kv_kernel<D, 2><<<grid, kKvThreads, 0, stream>>>(a); break;
    case 4: decode_kv_kernel<D, 4><<<grid, kKvThreads, 0, stream>>>(a); break;
    case 8: decode_kv_kernel<D, 8><<<grid, kKvThreads, 0, stream>>>(a); break;
    case 16: decode_kv_kernel<D, 16><<<grid, kKvThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_kv(const attn_bwd_decode_params& p, const float* q, const float* probs,
                             const float* d_out, const float* d_scores, float* d_k, float* d_v,
                             cudaStream_t stream) {
  KvArgs a;
  a.q = q;
  a.probs = probs;
  a.d_out = d_out;
  a.d_scores = d_scores;
  a.d_k = d_k;
  a.d_v = d_v;
  a.n_heads = p.n_heads;
  a.n_kv = p.n_kv_heads;
  a.hist = p.history_len;
  a.cpp = (p.history_len + kKvChunk - 1) / kKvChunk;
  const long long n = (long long)p.num_seqs * p.n_kv_heads * a.cpp;
  if (n < 1 || n > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int G = p.n_heads / p.n_kv_heads;
  switch (p.head_dim) {
    case 64: return kv_by_group<64>(a, G, (unsigned)n, stream);
    case 128: return kv_by_group<128>(a, G, (unsigned)n, stream);
    case 256: return kv_by_group<256>(a, G, (unsigned)n, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace attnbwd

// ------------------------------------------------------------------------
// Decode backward without a caller-supplied workspace.
//
// The per-split partial sums live in a fixed device array compiled into the
// library instead of caller memory.  Every GPU that loads the library holds
// this array until the process exits.  Its device address is looked up once
// per device (on the first call made with that device current).
// ------------------------------------------------------------------------
#include <mutex>

namespace attnbwd {
namespace {

constexpr size_t kNoAllocScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
float* g_noalloc_ptr[kNoAllocMaxDevices] = {nullptr};
void* g_noalloc_ctx[kNoAllocMaxDevices] = {nullptr};  // context of the cached address

// Device address of the scratch array for the current device (nullptr on
// error).  Looked up on the first call with the device current, and again
// whenever the device's context has changed since (after cudaDeviceReset
// the array lives at another address in the new context).
float* noalloc_scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
    float* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return nullptr;
    g_noalloc_ptr[dev] = ptr;
    g_noalloc_ctx[dev] = current_context();  // the lookup created it if there was none
  }
  return g_noalloc_ptr[dev];
}

}  // namespace
}  // namespace attnbwd

extern "C" attn_status attn_bwd_decode_noalloc(const attn_bwd_decode_params* p,
                                               const float* k_hist, const float* v_hist,
                                               const float* probs, const float* d_out,
                                               float* d_scores, float* d_q, void* stream) {
  using namespace attnbwd;
  // argument checks of attn_bwd_decode (0 means the problem is invalid)
  if (attn_bwd_decode_workspace_size(p) == 0) return ATTN_ERR_INVALID;
  const void* ptrs[] = {k_hist, v_hist, probs, d_out, d_scores, d_q};
  for (const void* q : ptrs)
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15u)) return ATTN_ERR_INVALID;
  // as many history splits as the fixed array can hold, at most the usual number
  int n_split = decode_num_splits(*p);
  while (n_split > 1 && decode_partials_floats(*p, n_split) * sizeof(float) > kNoAllocScratchBytes)
    --n_split;
  if (decode_partials_floats(*p, n_split) * sizeof(float) > kNoAllocScratchBytes)
    return ATTN_ERR_SCRATCH_LIMIT;
  float* scratch = noalloc_scratch_for_current_device();
  if (!scratch) return ATTN_ERR_CUDA;
  // every split's slot is fully rewritten by the kernel: nothing to clear
  if (launch_decode(*p, k_hist, v_hist, probs, d_out, d_scores, d_q, scratch, n_split,
                    reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}
