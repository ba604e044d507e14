// Fused attention backward tile kernel for sm_103a (tcgen05 + TMA + TMEM).
//
// One CTA owns a tile of BN keys of one (batch, KV head) and walks the query
// tiles of every query head that shares that KV head (the GQA group loop of
// the WGSL page's flash_bwd_dk_dv), so dK and dV accumulate in tensor memory
// without atomics.  Per query tile of BM rows it issues the five dense
// products of the backward pass on the tensor cores:
//   GEMM1  S^T  [BN,BM] = K . Q^T              (scores, unscaled)
//   GEMM2  dP^T [BN,BM] = V . dO^T
//   GEMM3  dV   [BN,D] += (P o M)^T . dO
//   GEMM4  dK   [BN,D] += dS'^T . Q            (dS' = scale * dS)
//   GEMM5  dQ^T [D,BM]  = K^T . dS'^T          (or dQ [BM,D] = dS' . K)
// and adds dQ into an fp32 accumulator with global atomics (instead of the
// WGSL page's separate atomic-free dQ pass, which would recompute GEMM1/2).
//
// Operand staging.  Shared-memory tiles are 128-byte swizzled row tiles,
// [column block][row][128 bytes] with the 16-byte chunk index XOR (row & 7):
// exactly what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B.
//  * bf16: one copy of each tile serves as a K-major operand (rows = M/N) and
//    as an MN-major operand (rows = K).
//  * fp32 (TF32 products): a TF32 operand read MN-major must be laid out in
//    the 128-byte swizzle of 32-byte atoms ([MN / 32][K rows][128 bytes],
//    32-byte chunk index XOR (row & 3)), which differs from the K-major
//    tiles' swizzle.  So the contractions over queries (GEMM3/4) and keys
//    (GEMM5) read second copies of the Q, dO and K tiles that TMA loads from
//    the same tensors with that swizzle (the "MN-major copies"), and the
//    softmax warps write dS' in [query][key] orientation.  The natural tiles
//    (GEMM1/2) and the MN-major copies (GEMM3/4) travel in separate rings, so
//    a natural stage is released as soon as GEMM1/2 are done with it.
//
// Pipeline.  GEMM1/2 of tile t + NSB are issued as soon as score buffer
// t % NSB is free (NSB = 1 or 2 score buffers), then GEMM3-5 of tile t once
// its P / dS' are written; the softmax warps compute tile t while the tensor
// cores finish earlier tiles and start later ones.  With separate P / dS'
// columns a score buffer is free once the softmax warps have read it, and
// they wait for GEMM3-5 of tile t - PB (PB = 1 or 2 P / dS' buffers) before
// overwriting P / dS'.  In place (fp32, D = 64) a score buffer is free only
// after GEMM3/4 have read the P / dS' written over it: GEMM3/4 (t), GEMM5 (t),
// then GEMM1/2 (t + 2) once GEMM3/4 (t) are complete.  The tensor cores read operands from shared memory at
// up to 128 bytes per clock; while they do, other shared-memory traffic
// (including mbarrier operations) is served slowly, so the fp32 softmax reads
// per-query LSE / Delta once per tile in 16x256b fragments.
//
// Warp roles (512 threads):
//   warp 0       TMA producer: resident key tiles, natural Q / dO ring
//   warp 1       MMA issuer (one elected lane)
//   warp 2       TMEM allocator
//   warp 3       TMA producer of the MN-major Q / dO copies (fp32)
//   warps 4-11   softmax: warp w serves TMEM sub-partition w % 4 (its key
//                rows) and half (w - 4) / 4 of the query columns; turns S^T
//                and dP^T into P o M and dS', stores them as MMA operands, and
//                at the end stages dK and dV in shared memory for two TMA
//                stores
//   warps 12-15  dQ: drain the GEMM5 accumulator into global memory
// Accumulators with M = 64 rows live in lanes 0-15 of each 32-lane TMEM
// sub-partition (row r -> lane (r / 16) * 32 + r % 16); M = 128 rows map
// one-to-one.  Every tcgen05.ld is executed by whole warps.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"

namespace attnbwd {

namespace {

template <bool BF16, int D>
struct Cfg;
// MNCOPY (fp32): GEMM3/4 read a second copy of the tile's Q / dO and GEMM5 a
// second copy of K, fetched in the 128-byte swizzle of 32-byte atoms and
// read MN-major; the softmax writes dS' as [query][key] for GEMM5.  Without
// it (bf16) one copy of each tile serves both majors and dS' is [key][query].
// INPL: P and dS' overwrite S^T and dP^T in tensor memory (no separate P /
// dS' columns), and the shared-memory dS' tile of query tile t is written over
// tile t's own natural Q / dO stage (GEMM1/2 are done with it by then), which
// is released to the producer only after GEMM5; VTM: V lives in tensor memory
// as GEMM2's A operand, so GEMM2 reads only the dO tile from shared memory.
//
// The fp32 D = 128 configuration adds four options (all false elsewhere):
// SPLITQ: Q and dO travel in rings of their own (NAT Q slots, NDO dO slots);
//   a dO slot is released as soon as GEMM2 has read it, a Q slot holds the
//   tile's dS' after GEMM1 and is released after GEMM5.
// VGL: V goes from global memory straight into tensor memory (softmax warps,
//   rounded to TF32), without a shared-memory staging copy.
// DQA: the dQ^T accumulator of tile t lives in the P columns of score buffer
//   t % NSB: GEMM5 (t) is issued once GEMM3/4 (t) are complete, and GEMM1/2
//   (t + NSB) wait until the dQ warps have drained it.
// DQSLOT: the dQ warps stage dQ of tile t in tile t's own Q slot (which held
//   its dS' until GEMM5) and add it with one TMA reduce-add; the slot goes
//   back to the producer once the copy engine has read it.
// FRAG: the unmasked fp32 softmax uses 16x256b fragments (BM = 64 only).
template <>
struct Cfg<false, 64> {  // fp32, D = 64
  static constexpr int BN = 128, BM = 64, NAT = 3, TR = 1, NSB = 2, PB = 1, NDO = 3;
  static constexpr bool MNCOPY = true, DQT = true, INPL = true, VTM = true;
  static constexpr bool SPLITQ = false, VGL = false, DQA = false, DQSLOT = false, FRAG = true;
};
template <>
struct Cfg<false, 128> {  // fp32, D = 128
  static constexpr int BN = 128, BM = 32, NAT = 3, TR = 1, NSB = 2, PB = 1, NDO = 1;
  static constexpr bool MNCOPY = true, DQT = true, INPL = true, VTM = true;
  static constexpr bool SPLITQ = true, VGL = true, DQA = true, DQSLOT = true, FRAG = false;
};
template <>
struct Cfg<true, 64> {  // bf16, D = 64
  static constexpr int BN = 128, BM = 128, NAT = 3, TR = 0, NSB = 1, PB = 1, NDO = 3;
  static constexpr bool MNCOPY = false, DQT = false, INPL = false, VTM = false;
  static constexpr bool SPLITQ = false, VGL = false, DQA = false, DQSLOT = false, FRAG = false;
};
template <>
struct Cfg<true, 128> {  // bf16, D = 128
  static constexpr int BN = 128, BM = 64, NAT = 3, TR = 0, NSB = 1, PB = 1, NDO = 3;
  static constexpr bool MNCOPY = false, DQT = true, INPL = false, VTM = false;
  static constexpr bool SPLITQ = false, VGL = false, DQA = false, DQSLOT = false, FRAG = false;
};

// the dQ^T accumulator [M5 lanes][N5 columns] fits in the BM P columns
constexpr bool L_N5_FITS(int n5, int bm) { return n5 <= bm; }

template <bool BF16, int D>
struct Layout {
  using C = Cfg<BF16, D>;
  static constexpr int BM = C::BM, BN = C::BN, NAT = C::NAT, TR = C::TR, NSB = C::NSB,
                       PB = C::PB;
  static constexpr bool MNCOPY = C::MNCOPY, DQT = C::DQT, INPL = C::INPL, VTM = C::VTM;
  static constexpr bool SPLITQ = C::SPLITQ, VGL = C::VGL, DQA = C::DQA, DQSLOT = C::DQSLOT,
                        FRAG = C::FRAG;
  static constexpr int NDO = SPLITQ ? C::NDO : NAT;  // dO slots (= NAT unless SPLITQ)
  static constexpr int E = BF16 ? 2 : 4;  // element bytes
  static constexpr int W = 128 / E;       // elements per 128-byte segment
  static constexpr int KSTEP = 32 / E;    // K elements per MMA instruction
  static constexpr int K_BYTES = BN * D * E;
  static constexpr int Q_BYTES = BM * D * E;
  static constexpr int P_BYTES = BN * BM * E;
  // shared memory map (offsets from a 1024-aligned base)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + K_BYTES;  // must follow K (padded GEMM5 reads it)
  static constexpr int OFF_KT = OFF_V + (VTM ? 0 : K_BYTES);
  // natural ring [NAT]: separate Q and dO rings, or (INPL) stages of
  // [Q tile][dO tile] that later hold the tile's dS' [BM rows][BN keys], or
  // (SPLITQ) NAT Q slots (later dS') and NDO dO slots
  static constexpr int OFF_Q = OFF_KT + (MNCOPY ? K_BYTES : 0);
  static constexpr bool JOINT = INPL && !SPLITQ;  // [Q | dO] stages
  static constexpr int NAT_STRIDE = JOINT ? 2 * Q_BYTES : Q_BYTES;
  static constexpr int OFF_DO = OFF_Q + (JOINT ? Q_BYTES : NAT * Q_BYTES);
  static constexpr int OFF_QT =
      SPLITQ ? OFF_DO + NDO * Q_BYTES : OFF_Q + 2 * NAT * Q_BYTES;  // MN-major copy ring [TR]
  static constexpr int OFF_DOT = OFF_QT + TR * Q_BYTES;
  // bf16: dS'^T [BN rows][BM] (GEMM4 A, GEMM5 operand); fp32: PB x dS' [BM rows][BN]
  static constexpr int OFF_DS = OFF_DOT + TR * Q_BYTES;
  static constexpr int OFF_DSN = OFF_DS + (MNCOPY ? 0 : P_BYTES);
  static constexpr int ROW_ST = 4;  // stages of the LSE2 / Delta ring
  static constexpr int OFF_LSE = OFF_DSN + (MNCOPY && !INPL ? PB * P_BYTES : 0);
  // VTM: V lands in the (not yet used) MN-major copy ring and is moved into
  // tensor memory before the first MN-major copies are fetched
  static constexpr int OFF_VLOAD = VTM ? OFF_QT : OFF_V;
  // dK / dV staged for their TMA stores once every product is complete: dK
  // over the K tile, dV over K's MN-major copy (fp32) or the V tile (bf16)
  static constexpr int OFF_DKST = OFF_K;
  static constexpr int OFF_DVST = MNCOPY ? OFF_KT : OFF_V;
  static constexpr int OFF_DELTA = OFF_LSE + ROW_ST * BM * 4;
  // dQ staging tile [BM][STG_D] fp32 (query-major), STG_D head-dim columns per
  // pass (DQSLOT: all D in one pass, in the tile's Q slot, no region of its own)
  static constexpr int STG_D = DQT ? (DQSLOT ? D : (D > 64 ? 64 : D)) : 0;
  static constexpr int OFF_STG = OFF_DELTA + ROW_ST * BM * 4;
  // (fp32, D=64) dropout keep bits of two query tiles, [2][BN keys][BM / 16]
  // x 16 bits, drawn by the dQ warps one tile ahead of the softmax warps; the
  // other configurations draw them in the softmax warps
  static constexpr bool DBITS = !BF16 && D == 64;
  static constexpr int NCH = BM / 16;
  static constexpr int OFF_BITS = OFF_STG + (DQSLOT ? 0 : BM * STG_D * 4);
  static constexpr int OFF_BAR = OFF_BITS + (DBITS ? 2 * BN * NCH * 2 : 0);
  static constexpr int NUM_BARS = 2 * NAT + 2 * TR + 2 * ROW_ST + 4 * NSB + 2 + PB + 9 +
                                  2 * NDO + 2 * NSB;
  static constexpr int OFF_TMEMPTR = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_TMEMPTR + 16 + 1024;  // + alignment slack
  // bytes landing per stage and for the resident key tiles
  static constexpr int NAT_TX = SPLITQ ? Q_BYTES : 2 * Q_BYTES;
  static constexpr int TR_TX = 2 * Q_BYTES;
  static constexpr int ROW_TX = 2 * BM * 4;
  static constexpr int KV_TX = ((MNCOPY ? 3 : 2) - (VGL ? 1 : 0)) * K_BYTES;
  // GEMM5 shape: dQ^T [D (padded to 128 if not MNCOPY), BM] or dQ [BM, D]
  static constexpr int M5 = DQT ? (MNCOPY ? D : 128) : BM;
  static constexpr int N5 = DQT ? BM : D;
  // tensor memory columns: NSB x (S^T, dP^T), PB x P^T (fp32: one column per
  // element; bf16: two per column), fp32: PB x dS'^T, then dV, dK, dQ
  static constexpr int PCOLS = BF16 ? BM / 2 : BM;
  static constexpr int T_P = 2 * BM * NSB;
  static constexpr int T_DS = T_P + (INPL ? 0 : PB * PCOLS);
  static constexpr int T_DV = T_DS + (MNCOPY && !INPL ? PB * BM : 0), T_DK = T_DV + D,
                       T_DQ = T_DK + D;
  static constexpr int T_V = T_DQ + (DQA ? 0 : N5);
  static constexpr int T_USED = T_V + (VTM ? D : 0);
  static constexpr int T_ALLOC = T_USED <= 256 ? 256 : 512;
  // softmax split: two warps per TMEM sub-partition, each on half the columns
  static constexpr int COLS = BM / 2;
  static_assert(T_USED <= 512 && TR_TX > 0, "tensor memory budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(COLS % 16 == 0, "softmax column chunks");
  static_assert(!MNCOPY || (D % W == 0 && BM % KSTEP == 0 && TR >= 1), "MN-major copies");
  static_assert(MNCOPY || NAT >= 2, "stages are released only after GEMM3/4");
  static_assert(PB == 1 || PB == 2, "P / dS buffers");
  static_assert(BN == 64 || BN == 128, "key tile");
  static_assert(!INPL || (MNCOPY && !BF16 && NAT_STRIDE >= P_BYTES && NAT >= 3),
                "in-place P / dS' is the fp32 layout; dS' fits a natural stage");
  static_assert(!VTM || (INPL && BN == 128 && (VGL || (2 * TR * Q_BYTES >= K_BYTES && D / W == 2))),
                "V staging through the MN-major copy ring, one column block per softmax half");
  static_assert(!SPLITQ || (INPL && NDO >= 1), "split rings hold dS' in the Q slot");
  static_assert(!DQA || (INPL && NSB == 2 && MNCOPY && BF16 == false && L_N5_FITS(N5, BM)),
                "dQ^T aliases the P columns of its score buffer");
  static_assert(!DQSLOT || (SPLITQ && INPL && DQT && MNCOPY && M5 == D && N5 == BM &&
                              BM * D * 4 == Q_BYTES),
                "dQ [BM][D] fp32 staged in the tile's Q slot");
  static_assert(!FRAG || (INPL && BM == 64 && D == 64), "16x256b softmax fragments");
  static_assert(M5 == 64 || M5 == 128, "GEMM5 rows");
};

constexpr int kThreads = 512;
constexpr int kSoftmaxThreads = 256;
constexpr int kDqThreads = 128;

__device__ __forceinline__ uint32_t sw_off(int blk, int rows, int row, int pos_bytes) {
  return (uint32_t)(blk * rows * 128 + row * 128 + ((((pos_bytes >> 4) ^ (row & 7))) << 4) +
                    (pos_bytes & 15));
}

// Accumulator row held by TMEM lane `lane128` (0..127) for an M-row product;
// -1 for lanes that hold no row (M = 64 uses 16 lanes per sub-partition).
template <int M>
__device__ __forceinline__ int acc_row(int lane128) {
  if constexpr (M == 128) {
    return lane128;
  } else {
    return (lane128 & 31) < 16 ? (lane128 >> 5) * 16 + (lane128 & 15) : -1;
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Round to TF32 (nearest, ties away from zero in magnitude) by adding half
// a TF32 unit to the bit pattern; the tensor cores ignore the low 13 bits.
// Same result as cvt.rna.tf32.f32 for every finite value, on the ALU pipe.
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x) + 0x1000u; }

// packed fp32x2 arithmetic (sm_100+)
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
__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Bounded wait that ignores the error word: used only on the unwinding path to
// let copies or products already in flight land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitLimitCycles / 4) return;
  }
}

// Warp-uniform bounded wait: true only if every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, unsigned int* err) {
  return !__any_sync(0xffffffffu, !mbar_wait(bar, parity, err));
}

// Named barrier 1 over the 128 dQ threads, combined with a vote: true only if
// every participating thread passed `ok`.  All 128 threads always arrive, so
// the group cannot split even when a wait gave up.
__device__ __forceinline__ bool dq_group_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 128, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void dq_group_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Named barrier 2 over the 256 softmax threads with the same vote.
__device__ __forceinline__ bool softmax_group_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 2, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)ok)
      : "memory");
  return r != 0;
}


struct TileWork {
  int b, kvh, k0, q_begin, q_end, q_first, tiles_per_head, total;
};

template <int BN, int BM>
__device__ __forceinline__ TileWork tile_work(const TileArgs& a) {
  TileWork w;
  const int bh = blockIdx.x % (a.B * a.Hkv);
  const int kt = blockIdx.x / (a.B * a.Hkv);
  w.b = bh / a.Hkv;
  w.kvh = bh % a.Hkv;
  w.k0 = kt * BN;
  const long long k1 = (long long)min(w.k0 + BN, a.Sk) - 1;
  query_range(a.Sq, a.causal, a.causal_offset, a.window, w.k0, k1, &w.q_begin, &w.q_end);
  w.q_first = (w.q_begin / BM) * BM;
  w.tiles_per_head = w.q_end > w.q_begin ? (w.q_end - w.q_first + BM - 1) / BM : 0;
  w.total = w.tiles_per_head * a.group;
  return w;
}

// True when every (query, key) pair of the tile is in range and visible and
// no mask or dropout applies, so P needs no per-pair test.
__device__ __forceinline__ bool tile_is_plain(const TileArgs& a, int q0, int BM, int k0, int BN) {
  if (a.has_mask || a.dropout) return false;
  if (q0 + BM > a.Sq || k0 + BN > a.Sk) return false;
  const long long qa_min = (long long)q0 + a.causal_offset, qa_max = qa_min + BM - 1;
  const long long k_min = k0, k_max = (long long)k0 + BN - 1;
  if (a.causal && k_max > qa_min) return false;
  if (a.window > 0) {
    const long long far = max(qa_max - k_min, k_max - qa_min);
    if (far >= a.window) return false;
  }
  return true;
}

// fp32 in-place softmax step in 16x256b fragments, for tiles without an
// additive mask or dropout.  A softmax warp covers the 32 key rows of its TMEM
// sub-partition and a 32-column share of the query tile; thread t owns key
// rows t/4 + 8k (k < 4) and query columns 8x + 2(t%4) + e (x < 4, e < 2), so
// it needs -LSE*log2e and Delta of only 8 queries, loaded once per tile (the
// per-column broadcast loads of a one-key-per-thread layout queue behind the
// tensor cores' shared-memory operand reads).  Writes P (TF32) over S^T and
// dS' over dP^T, and dS' into the swizzled [query rows][keys] tile.
//   t_s, t_dp   tensor-memory address of the share (sub-partition lane base,
//               first column of the share)
//   sNL, sDelta the share's first query in the LSE2 / Delta rows
//   q0, k0      first query of the share, first key of the sub-partition
//   dsn         this thread's base address in the dS' tile (see the caller)
//   xo2         swizzle term of key group k and column parity e, [2k + e]
__device__ __forceinline__ void softmax_frag(const TileArgs& a, uint32_t t_s, uint32_t t_dp,
                                             const float* sNL, const float* sDelta, bool plain,
                                             int q0, int k0, bool (&key_ok)[4], uint32_t dsn,
                                             const uint32_t (&xo2)[8]) {
  const int lane = threadIdx.x & 31, tq = lane & 3, tr = lane >> 2;
  uint64_t nl2[4], dl2[4];
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    nl2[x] = *reinterpret_cast<const uint64_t*>(sNL + 8 * x + 2 * tq);
    dl2[x] = *reinterpret_cast<const uint64_t*>(sDelta + 8 * x + 2 * tq);
  }
  const uint64_t c2 = pk2(a.scale_log2e, a.scale_log2e);
  const uint64_t sc2 = pk2(a.scale, a.scale);
#pragma unroll
  for (int lb = 0; lb < 2; ++lb) {  // lanes 0-15, then 16-31 of the sub-partition
    uint32_t sv[16], dv[16];
    __syncwarp();  // tcgen05.ld / st are warp-collective
    tmem_ld_16x256b_x4(t_s + ((uint32_t)(16 * lb) << 16), sv);
    tmem_ld_16x256b_x4(t_dp + ((uint32_t)(16 * lb) << 16), dv);
    tmem_ld_wait();
#pragma unroll
    for (int x = 0; x < 4; ++x) {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int i = 4 * x + 2 * r;
        const uint64_t xx = f2fma(pk2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2,
                                  nl2[x]);
        float x0, x1;
        up2(xx, x0, x1);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const uint64_t d = f2mul(
            f2mul(pk2(p0, p1), sc2),
            f2sub(pk2(__uint_as_float(dv[i]), __uint_as_float(dv[i + 1])), dl2[x]));
        float d0, d1;
        up2(d, d0, d1);
        sv[i] = __float_as_uint(p0);
        sv[i + 1] = __float_as_uint(p1);
        dv[i] = __float_as_uint(d0);
        dv[i + 1] = __float_as_uint(d1);
      }
    }
    if (!plain) {
      // tiles that straddle the causal diagonal, the window edge or the
      // sequence ends: zero the pairs the visibility rule excludes
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int kk = 2 * lb + ((i >> 1) & 1);  // key group of register i
        const int kj = k0 + tr + 8 * kk;
        const int q = q0 + 8 * (i >> 2) + 2 * tq + (i & 1);
        const int qa = q + (int)a.causal_offset;
        bool vis = (q < a.Sq) && key_ok[kk];
        if (a.causal) vis = vis && (kj <= qa);
        if (a.window > 0) vis = vis && (abs(qa - kj) < (int)a.window);
        sv[i] = vis ? sv[i] : 0u;
        dv[i] = vis ? dv[i] : 0u;
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      sv[i] = to_tf32(__uint_as_float(sv[i]));
      dv[i] = to_tf32(__uint_as_float(dv[i]));
    }
    __syncwarp();
    tmem_st_16x256b_x4(t_s + ((uint32_t)(16 * lb) << 16), sv);
    tmem_st_16x256b_x4(t_dp + ((uint32_t)(16 * lb) << 16), dv);
    // dS' tile: query row 8x + 2(t%4) + e of the share, key group 2 lb + r
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int x = i >> 2, r = (i >> 1) & 1, e = i & 1;
      st_shared_b32(dsn + (8 * x + e) * 128 + xo2[2 * (2 * lb + r) + e], dv[i]);
    }
  }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_qt,
                const __grid_constant__ CUtensorMap tm_kt,
                const __grid_constant__ CUtensorMap tm_dot,
                const __grid_constant__ CUtensorMap tm_dq,
                const __grid_constant__ CUtensorMap tm_dk,
                const __grid_constant__ CUtensorMap tm_dv, const TileArgs a) {
  using L = Layout<BF16, D>;
  constexpr int BM = L::BM, NAT = L::NAT, TR = L::TR, NSB = L::NSB, PB = L::PB, BN = L::BN,
                W = L::W, E = L::E;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* nat_full = bars;                 // [NAT] natural tiles landed (TMA tx)
  uint64_t* nat_empty = nat_full + NAT;      // [NAT] natural stage free (MMA commit)
  uint64_t* tr_full = nat_empty + NAT;       // [TR] MN-major Q / dO copies landed
  uint64_t* tr_empty = tr_full + TR;         // [TR] MN-major copy stage free (MMA commit)
  uint64_t* row_full = tr_empty + TR;        // [ROW_ST] LSE2 / Delta of a tile landed
  uint64_t* row_empty = row_full + L::ROW_ST;  // [ROW_ST] softmax warps done with them
  uint64_t* s_full = row_empty + L::ROW_ST;  // [NSB] GEMM1/2 done into score buffer b
  uint64_t* s_free = s_full + NSB;           // [NSB] softmax warps have read buffer b
  uint64_t* p_full = s_free + NSB;           // [2] P / dS' of a tile written (by parity)
  uint64_t* mma5_par = p_full + 2;           // [PB] GEMM3/4/5 of a tile done (by t % PB)
  uint64_t* kv_full = mma5_par + PB;         // resident key tiles landed
  uint64_t* mma5_done = kv_full + 1;         // GEMM3/4/5 done (every tile, dQ warps)
  uint64_t* dq_free = kv_full + 2;           // dQ accumulator drained
  uint64_t* acc_done = kv_full + 3;          // all products done
  uint64_t* final_bar = kv_full + 4;         // unwinding: products in flight done
  uint64_t* v_ready = kv_full + 5;           // (VTM) V copied into tensor memory
  uint64_t* pfree = kv_full + 6;             // [NSB] (INPL) GEMM3/4 done with buffer b
  uint64_t* bits_full = pfree + NSB;         // [2] dropout keep bits of a tile drawn (by parity)
  uint64_t* do_full = bits_full + 2;         // [NDO] (SPLITQ) dO tile landed
  uint64_t* do_empty = do_full + L::NDO;     // [NDO] (SPLITQ) GEMM2 done with the dO slot
  uint64_t* dq_free_b = do_empty + L::NDO;   // [NSB] (DQA) GEMM3 has read P of buffer b
  uint64_t* dq_drained = dq_free_b + NSB;    // [NSB] (DQA) dQ^T of buffer b drained
  uint16_t* bits_s = reinterpret_cast<uint16_t*>(smem + L::OFF_BITS);
  uint32_t* tmem_ptr = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEMPTR);
  constexpr int RST = L::ROW_ST;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const TileWork w = tile_work<BN, BM>(a);
  const int T = w.total;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NAT; ++s) {
      mbar_init(&nat_full[s], 1);
      mbar_init(&nat_empty[s], 1);
    }
    for (int s = 0; s < TR; ++s) {
      mbar_init(&tr_full[s], 1);
      mbar_init(&tr_empty[s], 1);
    }
    for (int s = 0; s < L::ROW_ST; ++s) {
      mbar_init(&row_full[s], 1);
      mbar_init(&row_empty[s], kSoftmaxThreads);
    }
    for (int s = 0; s < NSB; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&s_free[s], kSoftmaxThreads);
    }
    mbar_init(&p_full[0], kSoftmaxThreads);
    mbar_init(&p_full[1], kSoftmaxThreads);
    for (int s = 0; s < PB; ++s) mbar_init(&mma5_par[s], 1);
    mbar_init(kv_full, 1);
    mbar_init(mma5_done, 1);
    mbar_init(dq_free, kDqThreads);
    mbar_init(acc_done, 1);
    mbar_init(final_bar, 1);
    mbar_init(v_ready, kSoftmaxThreads);
    for (int s = 0; s < NSB; ++s) mbar_init(&pfree[s], 1);
    mbar_init(&bits_full[0], kDqThreads);
    mbar_init(&bits_full[1], kDqThreads);
    for (int s = 0; s < L::NDO; ++s) {
      mbar_init(&do_full[s], 1);
      mbar_init(&do_empty[s], 1);
    }
    for (int s = 0; s < NSB; ++s) mbar_init(&dq_free_b[s], 1);
    for (int s = 0; s < NSB; ++s) mbar_init(&dq_drained[s], kDqThreads);
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
    if (elect_one_sync() && T > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_do);
      mbar_expect_tx(kv_full, L::KV_TX);
      // whole tiles [D / W column blocks][BN keys][W], one copy each
      tma_load_5d(smem + L::OFF_K, &tm_k, kv_full, 0, w.k0, 0, w.kvh, w.b);
      if constexpr (!L::VGL)
        tma_load_5d(smem + L::OFF_VLOAD, &tm_v, kv_full, 0, w.k0, 0, w.kvh, w.b);
      if constexpr (L::MNCOPY)  // MN-major copy of K for GEMM5
        tma_load_5d(smem + L::OFF_KT, &tm_kt, kv_full, 0, w.k0, 0, w.kvh, w.b);
      int nat_issued = 0, row_issued = 0, do_issued = 0;
      for (int t = 0; t < T; ++t) {
        const int g = t / w.tiles_per_head;
        const int h = w.kvh * a.group + g;
        const int bh = w.b * a.H + h;
        const int q0 = w.q_first + (t % w.tiles_per_head) * BM;
        const long long row = (long long)bh * a.sq_pad + q0;
        // natural Q / dO tiles (and, for bf16, LSE2 / Delta)
        const int s = t % NAT;
        if (t >= NAT && !mbar_wait(&nat_empty[s], ((t / NAT) - 1) & 1, a.err)) break;
        mbar_expect_tx(&nat_full[s], L::NAT_TX);
        tma_load_5d(smem + L::OFF_Q + s * L::NAT_STRIDE, &tm_q, &nat_full[s], 0, q0, 0, h, w.b);
        if constexpr (!L::SPLITQ)
          tma_load_5d(smem + L::OFF_DO + s * L::NAT_STRIDE, &tm_do, &nat_full[s], 0, q0, 0, h,
                      w.b);
        nat_issued = t + 1;
        if constexpr (L::SPLITQ) {
          // dO slot of its own, released by GEMM2
          const int so = t % L::NDO;
          if (t >= L::NDO && !mbar_wait(&do_empty[so], ((t / L::NDO) - 1) & 1, a.err)) break;
          mbar_expect_tx(&do_full[so], L::Q_BYTES);
          tma_load_5d(smem + L::OFF_DO + so * L::Q_BYTES, &tm_do, &do_full[so], 0, q0, 0, h, w.b);
          do_issued = t + 1;
        }
        // LSE2 / Delta rows of the tile: a ring of their own, released by the
        // softmax warps as soon as they finish the tile
        const int rr = t % RST;
        if (t == 0 && a.pdl) griddep_wait();  // the rows are written by the prepare kernel
        if (t >= RST && !mbar_wait(&row_empty[rr], ((t / RST) - 1) & 1, a.err)) break;
        mbar_expect_tx(&row_full[rr], L::ROW_TX);
        bulk_load(smem + L::OFF_LSE + rr * BM * 4, a.lse2 + row, BM * 4, &row_full[rr]);
        bulk_load(smem + L::OFF_DELTA + rr * BM * 4, a.delta + row, BM * 4, &row_full[rr]);
        row_issued = t + 1;
      }
      // let every copy still in flight land before the CTA can exit
      drain_wait(kv_full, 0);
      for (int t = (nat_issued > NAT ? nat_issued - NAT : 0); t < nat_issued; ++t)
        drain_wait(&nat_full[t % NAT], (t / NAT) & 1);
      for (int t = (do_issued > L::NDO ? do_issued - L::NDO : 0); t < do_issued; ++t)
        drain_wait(&do_full[t % L::NDO], (t / L::NDO) & 1);
      for (int t = (row_issued > RST ? row_issued - RST : 0); t < row_issued; ++t)
        drain_wait(&row_full[t % RST], (t / RST) & 1);
    }
    __syncwarp();  // reconverge before the block-wide barrier at the end
  } else if (warp == 3) {
    // ------------------------------------------------- MN-major copy producer
    // (fp32) the tile's Q and dO again, [D / W blocks][BM rows][W columns] in
    // the 32-byte-atom swizzle, in a ring of its own so it never holds up the
    // natural tiles that GEMM1/2 wait for
    if constexpr (L::MNCOPY) {
      if (elect_one_sync() && T > 0) {
        tma_prefetch_desc(&tm_qt);
        tma_prefetch_desc(&tm_dot);
        int tr_issued = 0;
        // VTM: the first MN-major copies overwrite the staged V, so they wait
        // until the softmax warps have moved it into tensor memory
        const bool v_ok = !L::VTM || L::VGL || mbar_wait(v_ready, 0, a.err);
        for (int t = 0; v_ok && t < T; ++t) {
          const int g = t / w.tiles_per_head;
          const int h = w.kvh * a.group + g;
          const int q0 = w.q_first + (t % w.tiles_per_head) * BM;
          const int r = t % TR;
          if (t >= TR && !mbar_wait(&tr_empty[r], ((t / TR) - 1) & 1, a.err)) break;
          mbar_expect_tx(&tr_full[r], L::TR_TX);
          tma_load_5d(smem + L::OFF_QT + r * L::Q_BYTES, &tm_qt, &tr_full[r], 0, q0, 0, h, w.b);
          tma_load_5d(smem + L::OFF_DOT + r * L::Q_BYTES, &tm_dot, &tr_full[r], 0, q0, 0, h, w.b);
          tr_issued = t + 1;
        }
        for (int t = (tr_issued > TR ? tr_issued - TR : 0); t < tr_issued; ++t)
          drain_wait(&tr_full[t % TR], (t / TR) & 1);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Shared-memory descriptors are built once; every product then only adds
    // a constant byte offset (>> 4) to the 14-bit start-address field.  Shared
    // addresses stay below 256 KB, so the add never carries out of the field.
    if (elect_one_sync() && T > 0) {
      constexpr uint32_t id_s = make_idesc(BF16, BN, BM, false, false);
      // GEMM3/4 read dO / Q MN-major; GEMM5 reads K MN-major (and, bf16, dS')
      constexpr uint32_t id_acc = make_idesc(BF16, BN, D, false, true);
      constexpr uint32_t id_dq = make_idesc(BF16, L::M5, L::N5, true, !L::MNCOPY);
      // K-major tiles: LBO unused, SBO = 8 rows x 128 B
      const uint64_t dK = sw128_desc(smem_u32(smem + L::OFF_K), 16, 1024);
      const uint64_t dV = sw128_desc(smem_u32(smem + L::OFF_V), 16, 1024);
      const uint64_t dS = sw128_desc(smem_u32(smem + L::OFF_DS), 16, 1024);
      // fp32 dS' [BM rows][BN keys]: its own region, or (INPL) natural stage 0
      const uint64_t dSN =
          sw128_desc(smem_u32(smem + (L::INPL ? L::OFF_Q : L::OFF_DSN)), 16, 1024);
      const uint64_t dQ0 = sw128_desc(smem_u32(smem + L::OFF_Q), 16, 1024);
      const uint64_t dDO0 = sw128_desc(smem_u32(smem + L::OFF_DO), 16, 1024);
      // (fp32) MN-major copies in the 32-byte-atom swizzle: K [D / W][BN][W],
      // Q and dO [D / W][BM][W]
      const uint64_t aKT = mn32_desc(smem_u32(smem + L::OFF_KT), BN * 128);
      const uint64_t aQT0 = mn32_desc(smem_u32(smem + L::OFF_QT), BM * 128);
      const uint64_t aDOT0 = mn32_desc(smem_u32(smem + L::OFF_DOT), BM * 128);
      // MN-major views (bf16): LBO = bytes between 128-byte column blocks
      const uint64_t mQ0 = sw128_desc(smem_u32(smem + L::OFF_Q), BM * 128, 1024);
      const uint64_t mDO0 = sw128_desc(smem_u32(smem + L::OFF_DO), BM * 128, 1024);
      const uint64_t mK = sw128_desc(smem_u32(smem + L::OFF_K), BN * 128, 1024);
      const uint64_t mS = sw128_desc(smem_u32(smem + L::OFF_DS), BN * 128, 1024);
      auto adv = [](uint64_t d, uint32_t bytes) -> uint64_t { return d + (uint64_t)(bytes >> 4); };
      bool ok = mbar_wait(kv_full, 0, a.err);
      auto issue_front = [&](int t) -> bool {  // GEMM1, GEMM2 of tile t
        const int s = t % NAT, b = t % NSB, so = t % L::NDO;
        if (!mbar_wait(&nat_full[s], (t / NAT) & 1, a.err)) return false;
        if (L::SPLITQ && !mbar_wait(&do_full[so], (t / L::NDO) & 1, a.err)) return false;
        // buffer b is free once the softmax warps have read its scores, or
        // (in place) once GEMM3/4 have read the P / dS' written over them,
        // and (DQA) once the dQ warps have drained the dQ^T held there
        if (t >= NSB &&
            !mbar_wait(L::INPL ? &pfree[b] : &s_free[b], ((t / NSB) - 1) & 1, a.err))
          return false;
        if (L::DQA && t >= NSB && !mbar_wait(&dq_drained[b], ((t / NSB) - 1) & 1, a.err))
          return false;
        tc_fence_after();
        const uint64_t dQ = adv(dQ0, s * L::NAT_STRIDE);
        const uint64_t dDO = adv(dDO0, L::SPLITQ ? so * L::Q_BYTES : s * L::NAT_STRIDE);
        const uint32_t t_s = tmem + b * 2 * BM, t_dp = t_s + BM;
#pragma unroll
        for (int ks = 0; ks < D / L::KSTEP; ++ks) {
          const uint32_t kb = ks * 32;
          const uint32_t ka = (kb / 128) * BN * 128 + (kb % 128);
          const uint32_t qa = (kb / 128) * BM * 128 + (kb % 128);
          mma_ss<BF16>(t_s, adv(dK, ka), adv(dQ, qa), id_s, ks > 0);
          if constexpr (L::VTM) {  // V [BN lanes][D columns] in tensor memory
            mma_ts<BF16>(t_dp, tmem + L::T_V + ks * 8, adv(dDO, qa), id_s, ks > 0);
          } else {
            mma_ss<BF16>(t_dp, adv(dV, ka), adv(dDO, qa), id_s, ks > 0);
          }
        }
        mma_commit(&s_full[b]);
        // natural tiles done with (INPL: the stage then holds dS' until GEMM5)
        if constexpr (L::MNCOPY && !L::INPL) mma_commit(&nat_empty[s]);
        if constexpr (L::SPLITQ) mma_commit(&do_empty[so]);
        return true;
      };
      auto issue_back34 = [&](int t) -> bool {  // GEMM3, GEMM4 of tile t
        if (!mbar_wait(&p_full[t & 1], (t >> 1) & 1, a.err)) return false;
        const int s = t % NAT, r = L::MNCOPY ? t % TR : 0, pb = t % PB, b = t % NSB;
        // P^T and (fp32) dS'^T: A operands of GEMM3/4 in tensor memory
        const uint32_t t_p = L::INPL ? tmem + b * 2 * BM : tmem + L::T_P + pb * L::PCOLS;
        const uint32_t t_ds = L::INPL ? t_p + BM : tmem + L::T_DS + pb * BM;
        if constexpr (L::MNCOPY) {
          if (!mbar_wait(&tr_full[r], (t / TR) & 1, a.err)) return false;
        }
        tc_fence_after();
        uint64_t bdo0, bq0;
        if constexpr (L::MNCOPY) {  // MN-major copies of the tile's dO / Q
          bdo0 = adv(aDOT0, r * L::Q_BYTES);
          bq0 = adv(aQT0, r * L::Q_BYTES);
        } else {  // natural tiles [BM rows][D] read MN-major
          bdo0 = adv(mDO0, s * L::NAT_STRIDE);
          bq0 = adv(mQ0, s * L::NAT_STRIDE);
        }
        if constexpr (L::DQA) {
          // GEMM3 (reads P) first, then GEMM4: GEMM5, which overwrites the P
          // columns, only waits for GEMM3
#pragma unroll
          for (int ks = 0; ks < BM / L::KSTEP; ++ks) {
            const uint32_t ba = ks * L::KSTEP * 128;  // K step = KSTEP rows
            mma_ts<BF16>(tmem + L::T_DV, t_p + ks * 8, adv(bdo0, ba), id_acc, (t > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(&dq_free_b[b]);  // (DQA) P of buffer b read
#pragma unroll
          for (int ks = 0; ks < BM / L::KSTEP; ++ks) {
            const uint32_t ba = ks * L::KSTEP * 128;
            mma_ts<BF16>(tmem + L::T_DK, t_ds + ks * 8, adv(bq0, ba), id_acc, (t > 0 || ks > 0) ? 1u : 0u);
          }
        } else {
#pragma unroll
        for (int ks = 0; ks < BM / L::KSTEP; ++ks) {
          const uint32_t kb = ks * 32;
          const uint32_t pa = (kb / 128) * BN * 128 + (kb % 128);
          const uint32_t ba = ks * L::KSTEP * 128;  // MN-major: K step = KSTEP rows
          const uint32_t acc = (t > 0 || ks > 0) ? 1u : 0u;
          // 8 TMEM columns hold one K step (8 tf32, or 16 bf16 packed in pairs)
          mma_ts<BF16>(tmem + L::T_DV, t_p + ks * 8, adv(bdo0, ba), id_acc, acc);
          if constexpr (L::MNCOPY) {
            mma_ts<BF16>(tmem + L::T_DK, t_ds + ks * 8, adv(bq0, ba), id_acc, acc);
          } else {
            mma_ss<BF16>(tmem + L::T_DK, adv(dS, pa), adv(bq0, ba), id_acc, acc);
          }
        }
        }
        if constexpr (L::INPL) mma_commit(&pfree[b]);  // score buffer b reusable
        if constexpr (L::MNCOPY) mma_commit(&tr_empty[r]);  // GEMM5 does not read them
        return true;
      };
      auto issue_g5 = [&](int t) -> bool {  // GEMM5 of tile t
        const int s = t % NAT, pb = t % PB, b = t % NSB;
        if constexpr (L::DQA) {
          // GEMM5 writes dQ^T over the P columns of buffer b: GEMM3/4 (t),
          // which read them, must be complete.  The dQ warps must also have
          // taken tile t - 1's accumulator (already true when GEMM1/2 (t + 1)
          // were issued), so that mma5_done never runs two phases ahead of them
          if (!mbar_wait(&dq_free_b[b], (t / NSB) & 1, a.err)) return false;  // GEMM3 (t) done
          if (t > 0 && !mbar_wait(&dq_drained[(t - 1) % NSB], ((t - 1) / NSB) & 1, a.err))
            return false;
        } else {
          if (t > 0 && !mbar_wait(dq_free, (t - 1) & 1, a.err)) return false;
        }
        tc_fence_after();
        const uint32_t t_dq = L::DQA ? tmem + (uint32_t)(b * 2 * BM) : tmem + L::T_DQ;
#pragma unroll
        for (int ks = 0; ks < BN / L::KSTEP; ++ks) {
          if constexpr (L::MNCOPY) {  // dQ^T = K^T . dS'^T: K MN-major, dS' K-major
            const uint32_t kb = ks * 32;
            const uint32_t ka = ks * L::KSTEP * 128;
            const uint32_t na = (L::INPL ? s * L::NAT_STRIDE : pb * L::P_BYTES) +
                                (kb / 128) * BM * 128 + (kb % 128);
            mma_ss<BF16>(t_dq, adv(aKT, ka), adv(dSN, na), id_dq, ks > 0);
          } else if constexpr (L::DQT) {
            const uint32_t ra = ks * L::KSTEP * 128;
            mma_ss<BF16>(t_dq, adv(mK, ra), adv(mS, ra), id_dq, ks > 0);
          } else {
            const uint32_t ra = ks * L::KSTEP * 128;
            mma_ss<BF16>(t_dq, adv(mS, ra), adv(mK, ra), id_dq, ks > 0);
          }
        }
        mma_commit(mma5_done);
        mma_commit(&mma5_par[pb]);
        // (DQSLOT: the dQ warps release the slot after staging dQ in it)
        if constexpr ((!L::MNCOPY || L::INPL) && !L::DQSLOT) mma_commit(&nat_empty[s]);
        return true;
      };
      // GEMM1/2 run NSB tiles ahead of GEMM3-5: front(t + NSB) only needs the
      // softmax warps to have read tile t's scores (s_free), which happens
      // before they finish tile t (p_full), so the tensor cores compute the
      // next scores while the softmax warps are still busy.  In place, score
      // buffer t % NSB cycles through GEMM1/2 (t), the softmax warps and
      // GEMM3/4 (t) before GEMM1/2 (t + NSB) may rewrite it; GEMM5 (t) runs
      // while the issuer waits for GEMM3/4 (t) to complete.
      if constexpr (L::VTM) {
        ok = ok && mbar_wait(v_ready, 0, a.err);
        tc_fence_after();
      }
      // DQA: GEMM1/2 run one tile ahead (a buffer is busy until its dQ^T is
      // drained): front (t + 1) is issued before waiting for the softmax of
      // tile t, so the softmax of t + 1 overlaps GEMM3/4 (t) and GEMM5 (t);
      // front (t + 1) itself waits for the dQ warps to take dQ^T (t - 1)
      constexpr int NPRE = L::DQA ? 1 : NSB;
      for (int t = 0; ok && t < NPRE && t < T; ++t)
        if (!issue_front(t)) ok = false;
      for (int t = 0; ok && t < T; ++t) {
        if constexpr (L::DQA) {
          ok = (t + 1 >= T || issue_front(t + 1)) && issue_back34(t) && issue_g5(t);
        } else if constexpr (L::INPL) {
          ok = issue_back34(t) && issue_g5(t) && (t + NSB >= T || issue_front(t + NSB));
        } else {
          ok = (t + NSB >= T || issue_front(t + NSB)) && issue_back34(t) && issue_g5(t);
        }
      }
      if (ok) mma_commit(acc_done);
      mma_commit(final_bar);
    }
    __syncwarp();  // reconverge before the block-wide barrier at the end
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ softmax warps
    const int quad = warp & 3, half = (warp - 4) >> 2;
    const int j = acc_row<BN>(quad * 32 + lane);  // key row of this lane, or -1
    const int kj = w.k0 + (j >= 0 ? j : 0);
    const bool key_ok = j >= 0 && kj < a.Sk;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    uint8_t* sdS = smem + L::OFF_DS;
    const int cbeg = half * L::COLS;
    // fp32: this lane's column j of the swizzled dS' tile [BM rows][BN keys]:
    // row r lives at base + r * 128 + xo[r & 7]
    const int jj = j >= 0 ? j : 0;
    const uint32_t dsn_lane = (jj / W) * BM * 128 + ((jj % W) * 4 & 15);
    uint32_t xo[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) xo[k] = (uint32_t)(((((jj % W) * 4) >> 4) ^ k) << 4);
    // fp32 in-place tiles without mask / dropout use 16x256b fragments (see
    // softmax_frag): this thread's key rows, its offset in the dS' tile and the
    // swizzle term of each (key group, column parity)
    const int tq = lane & 3, tr = lane >> 2;
    bool key_ok4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) key_ok4[k] = w.k0 + quad * 32 + tr + 8 * k < a.Sk;
    const uint32_t dsn_frag = quad * BM * 128 + (cbeg + 2 * tq) * 128 + (tr % 4) * 4;
    uint32_t xo2[8];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int e = 0; e < 2; ++e) xo2[2 * k + e] = (uint32_t)((((tr / 4 + 2 * k) ^ (2 * tq + e))) << 4);
    bool ok = true;
    if constexpr (L::VTM && L::VGL) {
      if (T > 0) {
        // V into tensor memory (GEMM2's A operand) straight from global
        // memory: this lane's key row, this warp's half of the head dimension,
        // rounded to TF32 like the tiles TMA delivers; keys past the end of
        // the sequence are zero
        constexpr int DH = D / 2;
        const float* vrow = reinterpret_cast<const float*>(a.V) +
                            row_offset(a.layout, w.b, w.kvh, key_ok ? kj : 0, a.Hkv, a.Sk, D) +
                            half * DH;
#pragma unroll 1
        for (int c0 = 0; c0 < DH; c0 += 16) {
          uint32_t rv[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 v4 = key_ok ? __ldg(reinterpret_cast<const float4*>(vrow + c0) + c)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
            rv[4 * c] = to_tf32(v4.x);
            rv[4 * c + 1] = to_tf32(v4.y);
            rv[4 * c + 2] = to_tf32(v4.z);
            rv[4 * c + 3] = to_tf32(v4.w);
          }
          __syncwarp();  // tcgen05.st is warp-collective
          tmem_st16(tmem + lane_base + L::T_V + half * DH + c0, rv);
        }
        tmem_st_wait();
        // releases tensor memory's V to the MMA issuer
        tc_fence_before();
        mbar_arrive(v_ready);
      }
    } else if constexpr (L::VTM) {
      if (T > 0) {
        // V into tensor memory (GEMM2's A operand): this lane's key row, this
        // warp's column block of the swizzled tile, 32 fp32 = 32 columns
        ok = warp_wait(kv_full, 0, a.err);
        if (ok) {
          const uint8_t* vrow = smem + L::OFF_VLOAD + half * BN * 128 + jj * 128;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t rv[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int chunk = h2 * 4 + c;
              const uint4 v4 =
                  *reinterpret_cast<const uint4*>(vrow + ((chunk ^ (jj & 7)) << 4));
              rv[4 * c] = v4.x;
              rv[4 * c + 1] = v4.y;
              rv[4 * c + 2] = v4.z;
              rv[4 * c + 3] = v4.w;
            }
            tmem_st16(tmem + lane_base + L::T_V + half * W + h2 * 16, rv);
          }
          tmem_st_wait();
        }
        // releases the staged V to the MN-major copy producer and tensor
        // memory's V to the MMA issuer
        tc_fence_before();
        mbar_arrive(v_ready);
      }
    }
    for (int t = 0; ok && t < T; ++t) {
      const int b = t % NSB, rs = t % RST, pb = t % PB;
      const int g = t / w.tiles_per_head;
      const int h = w.kvh * a.group + g;
      const int q0 = w.q_first + (t % w.tiles_per_head) * BM;
      // the tile's -LSE*log2(e) / Delta rows land well ahead of its scores:
      // wait for them first and (one 16-column chunk per thread) take this
      // half's values into registers while GEMM1/2 still run, so the
      // arithmetic after s_full reads no shared memory for them
      if (!warp_wait(&row_full[rs], (t / RST) & 1, a.err)) {
        ok = false;
        break;
      }
      const float* sLSE = reinterpret_cast<const float*>(smem + L::OFF_LSE + rs * BM * 4);
      const float* sDelta = reinterpret_cast<const float*>(smem + L::OFF_DELTA + rs * BM * 4);
      constexpr bool PRE = L::COLS == 16;  // fp32, D = 128
      uint64_t nlr[PRE ? 8 : 1], dlr[PRE ? 8 : 1];
      if constexpr (PRE) {
        const uint64_t* n2 = reinterpret_cast<const uint64_t*>(sLSE + cbeg);
        const uint64_t* d2 = reinterpret_cast<const uint64_t*>(sDelta + cbeg);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          nlr[i] = n2[i];
          dlr[i] = d2[i];
        }
      }
      if (!warp_wait(&s_full[b], (t / NSB) & 1, a.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const bool plain = tile_is_plain(a, q0, BM, w.k0, BN);
      const uint32_t t_s = tmem + lane_base + b * 2 * BM, t_dp = t_s + BM;
      const uint32_t t_p = L::INPL ? t_s : tmem + lane_base + L::T_P + pb * L::PCOLS;
      const uint32_t t_ds = L::INPL ? t_dp : tmem + lane_base + L::T_DS + pb * BM;
      // fp32 dS' tile of this query tile: its own buffer, or (INPL) the
      // tile's natural stage, which GEMM1/2 finished reading before s_full
      const uint32_t dsn_base = smem_u32(
          smem + (L::INPL ? L::OFF_Q + (t % NAT) * L::NAT_STRIDE : L::OFF_DSN + pb * L::P_BYTES));
      const uint32_t dsn_tile = dsn_lane + dsn_base;
      // dropout: this tile's keep bits, drawn by the dQ warps
      if (L::DBITS && a.dropout && !warp_wait(&bits_full[t & 1], (t >> 1) & 1, a.err)) {
        ok = false;
        break;
      }
      const uint16_t* kbits = bits_s + ((t & 1) * BN + jj) * L::NCH;
      if (L::FRAG && !a.has_mask && !a.dropout) {
        softmax_frag(a, t_s + cbeg, t_dp + cbeg, sLSE + cbeg, sDelta + cbeg, plain, q0 + cbeg,
                     w.k0 + quad * 32, key_ok4, dsn_base + dsn_frag, xo2);
      } else {
#pragma unroll 1
        for (int c0 = cbeg; c0 < cbeg + L::COLS; c0 += 16) {
          uint32_t rs16[16], rd16[16];
          __syncwarp();  // tcgen05.ld / st are warp-collective; the math below diverges on j
          tmem_ld16(t_s + c0, rs16);
          tmem_ld16(t_dp + c0, rd16);
          tmem_ld_wait();
          if (!L::INPL && c0 + 16 == cbeg + L::COLS) {  // last read of the score buffer
            tc_fence_before();
            mbar_arrive(&s_free[b]);
          }
          float pm[16], ds[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pm[c] = ds[c] = 0.f;
          if (j >= 0) {
            if (!a.has_mask && !a.dropout) {
              // two queries at a time with packed fp32x2 arithmetic
              const uint64_t* nl2 = PRE ? nlr : reinterpret_cast<const uint64_t*>(sLSE + c0);
              const uint64_t* dl2 = PRE ? dlr : reinterpret_cast<const uint64_t*>(sDelta + c0);
              const uint64_t c2 = pk2(a.scale_log2e, a.scale_log2e);
              const uint64_t sc2 = pk2(a.scale, a.scale);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint64_t x = f2fma(pk2(__uint_as_float(rs16[2 * i]),
                                             __uint_as_float(rs16[2 * i + 1])),
                                         c2, nl2[i]);
                float x0, x1;
                up2(x, x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                const uint64_t d = f2mul(f2mul(pk2(p0, p1), sc2),
                                         f2sub(pk2(__uint_as_float(rd16[2 * i]),
                                                   __uint_as_float(rd16[2 * i + 1])),
                                               dl2[i]));
                pm[2 * i] = p0;
                pm[2 * i + 1] = p1;
                up2(d, ds[2 * i], ds[2 * i + 1]);
              }
              if (!plain) {
                // tiles that straddle the causal diagonal, the window edge or the
                // sequence ends: zero the pairs the visibility rule excludes
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                  const int q = q0 + c0 + c;
                  const int qa = q + (int)a.causal_offset;
                  bool vis = (q < a.Sq) && key_ok;
                  if (a.causal) vis = vis && (kj <= qa);
                  if (a.window > 0) vis = vis && (abs(qa - kj) < (int)a.window);
                  pm[c] = vis ? pm[c] : 0.f;
                  ds[c] = vis ? ds[c] : 0.f;
                }
              }
            } else {
              // additive mask and / or dropout: per-pair exponent addend
              // (-inf for invisible or hard-masked pairs) and multiplier, then
              // the same packed arithmetic as above.  The chunk's dropout keep
              // mask (16 bits, one per query) was drawn by the dQ warps (fp32,
              // D=64) or is drawn here first (four Philox calls, one per four
              // consecutive queries of this key), and its 16 mask values are
              // loaded together from in-range addresses, so the loads overlap.
              uint32_t keep_bits = 0xffffu;
              if constexpr (L::DBITS) {
                if (a.dropout) keep_bits = kbits[c0 / 16];
              } else if (a.dropout) {
                keep_bits = 0u;
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                  const Philox4 r = philox4x32_10((uint32_t)(q0 + c0 + 4 * g4) >> 2, (uint32_t)kj,
                                                  (uint32_t)(w.b * a.H + h), 0u, a.seed_lo,
                                                  a.seed_hi);
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    keep_bits |= (r.w[e] >= a.drop_threshold ? 1u : 0u) << (4 * g4 + e);
                }
              }
              float mv[16];
              if (a.has_mask) {
                const float* mr = a.mask + w.b * a.msb + h * a.msh +
                                  (long long)(kj < a.Sk ? kj : a.Sk - 1) * a.msk;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                  const int q = q0 + c0 + c < a.Sq ? q0 + c0 + c : a.Sq - 1;
                  mv[c] = __ldg(mr + (long long)q * a.msq);
                }
              }
              float add[16], mul[16];
#pragma unroll
              for (int c = 0; c < 16; ++c) {
                const int q = q0 + c0 + c;
                const int qa = q + (int)a.causal_offset;
                bool vis = (q < a.Sq) && key_ok;
                if (a.causal) vis = vis && (kj <= qa);
                if (a.window > 0) vis = vis && (abs(qa - kj) < (int)a.window);
                float ad = sLSE[c0 + c];
                if (a.has_mask) {
                  vis = vis && mv[c] > -1.0e30f;
                  ad = fmaf(mv[c], kLog2e, ad);
                }
                add[c] = vis ? ad : __int_as_float(0xff800000);
                mul[c] = ((keep_bits >> c) & 1u) ? (a.dropout ? a.drop_inv_keep : 1.f) : 0.f;
              }
              const uint64_t* dl2 = reinterpret_cast<const uint64_t*>(sDelta + c0);
              const uint64_t c2 = pk2(a.scale_log2e, a.scale_log2e);
              const uint64_t sc2 = pk2(a.scale, a.scale);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const uint64_t x = f2fma(pk2(__uint_as_float(rs16[2 * i]),
                                             __uint_as_float(rs16[2 * i + 1])),
                                         c2, pk2(add[2 * i], add[2 * i + 1]));
                float x0, x1;
                up2(x, x0, x1);
                const uint64_t p2 = pk2(ex2_approx(x0), ex2_approx(x1));
                const uint64_t m2 = pk2(mul[2 * i], mul[2 * i + 1]);
                const uint64_t dp2 = f2mul(pk2(__uint_as_float(rd16[2 * i]),
                                               __uint_as_float(rd16[2 * i + 1])),
                                           m2);
                const uint64_t d = f2mul(f2mul(p2, sc2), f2sub(dp2, dl2[i]));
                up2(f2mul(p2, m2), pm[2 * i], pm[2 * i + 1]);
                up2(d, ds[2 * i], ds[2 * i + 1]);
              }
            }
          }
          // GEMM3-5 of tile t - PB must be done with this tile's P / dS' buffers
          // (in place: only the shared-memory dS' tile, waited for below)
          if (!L::INPL && c0 == cbeg && t >= PB &&
              !warp_wait(&mma5_par[pb], ((t / PB) - 1) & 1, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          __syncwarp();
          // P^T (and, for fp32, dS'^T) into tensor memory: the A operands of
          // GEMM3 / GEMM4.  Whole warps: tcgen05.st is warp-collective.
          if constexpr (BF16) {
            uint32_t pk[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) pk[c] = pack_bf16(pm[2 * c], pm[2 * c + 1]);
            tmem_st8(t_p + c0 / 2, pk);
          } else {
            uint32_t pr[16], dr[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              pr[c] = to_tf32(pm[c]);
              dr[c] = to_tf32(ds[c]);
            }
            tmem_st16(t_p + c0, pr);
            tmem_st16(t_ds + c0, dr);
            if (j >= 0) {
              // dS' as [BM rows (queries)][BN keys] for GEMM5's K-major operand
              const uint32_t rowbase = dsn_tile + c0 * 128;
#pragma unroll
              for (int c = 0; c < 16; ++c) st_shared_b32(rowbase + c * 128 + xo[c & 7], dr[c]);
            }
          }
          if constexpr (BF16) {
            if (j >= 0) {
              // dS'^T [BN rows][BM]: GEMM4's A and GEMM5's operand
              const int blk = c0 / W;
              const int pos = (c0 % W) * E;
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t off = sw_off(blk, BN, j, pos + h2 * 16);
                st_shared_v4(smem_u32(sdS + off), pack_bf16(ds[h2 * 8 + 0], ds[h2 * 8 + 1]),
                             pack_bf16(ds[h2 * 8 + 2], ds[h2 * 8 + 3]),
                             pack_bf16(ds[h2 * 8 + 4], ds[h2 * 8 + 5]),
                             pack_bf16(ds[h2 * 8 + 6], ds[h2 * 8 + 7]));
              }
            }
          }
        }
      }
      if (!ok) break;
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&p_full[t & 1]);
      mbar_arrive(&row_empty[rs]);
    }
    // --------------------------------------------------------- dK / dV epilogue
    // Each lane's key row of dK and dV goes into shared memory (regions idle
    // once every product is complete) in the 128-byte swizzle of the key-tile
    // maps, and one thread stores both tiles with two TMA copies; rows past
    // the end of the sequence fall outside the maps and are not written.
    // Every softmax thread reaches the vote, so the group cannot split.
    bool have = ok && T > 0;
    if (have) {
      have = warp_wait(acc_done, 0, a.err);
      tc_fence_after();
    }
    const bool stage = have || T == 0;
    if (stage) {
      uint8_t* sdk = smem + L::OFF_DKST;
      uint8_t* sdv = smem + L::OFF_DVST;
      constexpr int DH = D / 2;  // this warp's half of the head dimension
#pragma unroll 1
      for (int c0 = half * DH; c0 < (half + 1) * DH; c0 += 16) {
        uint32_t rv[16], rk[16];
        __syncwarp();  // tcgen05.ld is warp-collective
        if (have) {
          tmem_ld16(tmem + lane_base + L::T_DV + c0, rv);
          tmem_ld16(tmem + lane_base + L::T_DK + c0, rk);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) rv[c] = rk[c] = 0u;
        }
        if (j >= 0) {
          const int blk = c0 / W;
          const int pos = (c0 % W) * E;
          if constexpr (BF16) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int c = h2 * 8;
              const uint32_t off = sw_off(blk, BN, j, pos + h2 * 16);
              st_shared_v4(smem_u32(sdv + off),
                           pack_bf16(__uint_as_float(rv[c]), __uint_as_float(rv[c + 1])),
                           pack_bf16(__uint_as_float(rv[c + 2]), __uint_as_float(rv[c + 3])),
                           pack_bf16(__uint_as_float(rv[c + 4]), __uint_as_float(rv[c + 5])),
                           pack_bf16(__uint_as_float(rv[c + 6]), __uint_as_float(rv[c + 7])));
              st_shared_v4(smem_u32(sdk + off),
                           pack_bf16(__uint_as_float(rk[c]), __uint_as_float(rk[c + 1])),
                           pack_bf16(__uint_as_float(rk[c + 2]), __uint_as_float(rk[c + 3])),
                           pack_bf16(__uint_as_float(rk[c + 4]), __uint_as_float(rk[c + 5])),
                           pack_bf16(__uint_as_float(rk[c + 6]), __uint_as_float(rk[c + 7])));
            }
          } else {
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) {
              const uint32_t off = sw_off(blk, BN, j, pos + h4 * 16);
              st_shared_v4(smem_u32(sdv + off), rv[h4 * 4], rv[h4 * 4 + 1], rv[h4 * 4 + 2],
                           rv[h4 * 4 + 3]);
              st_shared_v4(smem_u32(sdk + off), rk[h4 * 4], rk[h4 * 4 + 1], rk[h4 * 4 + 2],
                           rk[h4 * 4 + 3]);
            }
          }
        }
      }
      fence_proxy_async_smem();
    }
    if (softmax_group_all(stage) && threadIdx.x == 128) {
      tma_store_5d(&tm_dk, smem + L::OFF_DKST, 0, w.k0, 0, w.kvh, w.b);
      tma_store_5d(&tm_dv, smem + L::OFF_DVST, 0, w.k0, 0, w.kvh, w.b);
      bulk_commit();
      bulk_wait_all();  // both stores complete before the CTA can exit
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------ dQ warps
    // Per tile: read the GEMM5 accumulator out of TMEM, release it, and add
    // it into the fp32 dQ accumulator in global memory.  The transposed
    // accumulator (dQ^T: lanes = head dim, columns = queries) is staged through
    // shared memory as [query][d] (fp32, D = 128: in the tile's own Q slot)
    // and added by TMA reduce-adds; a row-per-lane dQ (bf16, D = 64) goes out
    // as 16-byte vector atomics along each dQ row.
    const int quad = warp & 3;
    const int tid = threadIdx.x - 384;  // 0..127
    const int r = acc_row<L::M5>(quad * 32 + lane);  // accumulator row, or -1
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    float* stg = reinterpret_cast<float*>(smem + L::OFF_STG);
    const long long rstride = a.layout == 0 ? D : (long long)a.H * D;
    // dropout keep bits of tile tt into buffer tt & 1: for key row jr and
    // 16-query chunk ci, bit 4 g4 + e keeps query q0 + 16 ci + 4 g4 + e (one
    // Philox4x32-10 call per four consecutive queries of a key)
    auto draw_bits = [&](int tt) {
      const int h2 = w.kvh * a.group + tt / w.tiles_per_head;
      const int q02 = w.q_first + (tt % w.tiles_per_head) * BM;
      const uint32_t bh2 = (uint32_t)(w.b * a.H + h2);
      uint16_t* dst = bits_s + (tt & 1) * BN * L::NCH;
      for (int jr = tid; jr < BN; jr += kDqThreads) {
#pragma unroll 1
        for (int ci = 0; ci < L::NCH; ++ci) {
          uint32_t kb = 0u;
#pragma unroll
          for (int g4 = 0; g4 < 4; ++g4) {
            const Philox4 r = philox4x32_10((uint32_t)(q02 + 16 * ci + 4 * g4) >> 2,
                                            (uint32_t)(w.k0 + jr), bh2, 0u, a.seed_lo, a.seed_hi);
#pragma unroll
            for (int e = 0; e < 4; ++e) kb |= (r.w[e] >= a.drop_threshold ? 1u : 0u) << (4 * g4 + e);
          }
          dst[jr * L::NCH + ci] = (uint16_t)kb;
        }
      }
      mbar_arrive(&bits_full[tt & 1]);
    };
    // tile t + 1's buffer was last read by the softmax of tile t - 1, which
    // finished before GEMM5 of t - 1 (waited for in the previous iteration)
    if constexpr (L::DBITS) {
      if (a.dropout && T > 0) draw_bits(0);
    }
    for (int t = 0; t < T; ++t) {
      if constexpr (L::DBITS) {
        if (a.dropout && t + 1 < T) draw_bits(t + 1);
      }
      const int g = t / w.tiles_per_head;
      const int h = w.kvh * a.group + g;
      const int q0 = w.q_first + (t % w.tiles_per_head) * BM;
      // (staged dQ) every dQ thread is also done writing tile t - 1's stage
      if (!dq_group_all(mbar_wait(mma5_done, t & 1, a.err))) break;
      if (t == 0 && a.pdl) griddep_wait();  // the accumulator is zeroed by the prepare kernel
      tc_fence_after();
      __syncwarp();  // tcgen05.ld is warp-collective; the staging below diverges on r
      // (DQA) the accumulator of tile t sits in the P columns of its buffer
      const uint32_t t_dq =
          L::DQA ? (uint32_t)((t % NSB) * 2 * BM) : (uint32_t)L::T_DQ;
      float v[L::N5];
#pragma unroll
      for (int c0 = 0; c0 < L::N5; c0 += 16) {
        uint32_t rr[16];
        tmem_ld16(tmem + lane_base + t_dq + c0, rr);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c0 + c] = __uint_as_float(rr[c]);
      }
      tc_fence_before();
      mbar_arrive(L::DQA ? &dq_drained[t % NSB] : dq_free);
      const int nq = min(BM, a.Sq - q0);
      // deterministic: this key tile's own dQ slice, [kt * B + b][h][q][d]
      const int kt = w.k0 / BN;
      float* gbase = a.det ? a.dq_acc + row_offset(0, kt * a.B + w.b, h, q0, a.H, a.Sq, D)
                           : a.dq_acc + row_offset(a.layout, w.b, h, q0, a.H, a.Sq, D);
      if constexpr (L::DQSLOT) {
        // stage [BM queries][D] fp32 in the tile's Q slot (GEMM5, the last
        // reader of its dS', is complete: mma5_done), then one TMA
        // reduce-add (deterministic mode: a store into this key tile's
        // slice); rows past Sq fall outside the tensor map and are skipped
        const int s = t % NAT;
        float* slot = reinterpret_cast<float*>(smem + L::OFF_Q + s * L::NAT_STRIDE);
#pragma unroll
        for (int c = 0; c < BM; ++c) slot[c * D + r] = v[c];
        fence_proxy_async_smem();
        dq_group_sync();
        if (tid == 0) {
          if (a.det)
            tma_store_4d(&tm_dq, slot, 0, q0, h, kt * a.B + w.b);
          else
            tma_reduce_add_4d(&tm_dq, slot, 0, q0, h, w.b);
          bulk_commit();
          bulk_wait_read();  // the copy engine has read the slot: back to the producer
          mbar_arrive(&nat_empty[s]);
        }
        (void)gbase;
        (void)nq;
      } else if constexpr (L::DQT) {
        // stage [BM queries][STG d] and hand the tile to the TMA engine as one
        // reduce-add (rows past Sq fall outside the tensor map and are skipped)
        constexpr int STG = L::STG_D;
#pragma unroll 1
        for (int d0 = 0; d0 < D; d0 += STG) {
          if (tid == 0) bulk_wait_read();  // previous reduce has read the stage
          dq_group_sync();
          if (r >= d0 && r < d0 + STG) {
#pragma unroll
            for (int c = 0; c < BM; ++c) stg[c * STG + (r - d0)] = v[c];
          }
          fence_proxy_async_smem();
          dq_group_sync();
          if (tid == 0) {
            if (a.det)
              tma_store_4d(&tm_dq, stg, d0, q0, h, kt * a.B + w.b);
            else
              tma_reduce_add_4d(&tm_dq, stg, d0, q0, h, w.b);
            bulk_commit();
          }
        }
        (void)gbase;
        (void)nq;
      } else {
        // dQ: row r = query of the tile, columns = d (already contiguous)
        if (r >= 0 && r < nq) {
          float4* dst = reinterpret_cast<float4*>(gbase + r * (a.det ? D : rstride));
          if (a.det) {
#pragma unroll
            for (int c = 0; c < D / 4; ++c)
              dst[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
          } else {
#pragma unroll
            for (int c = 0; c < D / 4; ++c)
              atomicAdd(dst + c, make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]));
          }
        }
      }
    }
    if (tid == 0) bulk_wait_all();  // reductions complete before the CTA exits
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    // products still in flight (only on the unwinding path) must finish first
    if (T > 0) drain_wait(final_bar, 0);
    tc_fence_after();
    tmem_dealloc(tmem, L::T_ALLOC);
  }
}

template <bool BF16, int D>
cudaError_t launch_impl(const TileMaps& m, const TileArgs& a0, cudaStream_t stream, bool pdl) {
  TileArgs a = a0;
  a.pdl = pdl ? 1 : 0;
  using L = Layout<BF16, D>;
  auto kern = dkdv_kernel<BF16, D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = a.n_kv_tiles * a.B * a.Hkv;
  if (!pdl) {
    kern<<<grid, kThreads, L::SMEM_BYTES, stream>>>(m.q, m.k, m.v, m.dout, m.qt, m.kt, m.dot,
                                                    m.dq, m.dk, m.dv, a);
    return cudaGetLastError();
  }
  // may start while the prepare kernel finishes: key tiles, query tiles and
  // GEMM1/2 need nothing it writes; the LSE / Delta rows and the dQ
  // accumulator are touched only after griddep_wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, m.q, m.k, m.v, m.dout, m.qt, m.kt, m.dot, m.dq, m.dk, m.dv,
                         a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int dkdv_block_m(int dtype, int head_dim) {
  if (dtype == ATTN_BF16) return head_dim == 64 ? Cfg<true, 64>::BM : Cfg<true, 128>::BM;
  return head_dim == 64 ? Cfg<false, 64>::BM : Cfg<false, 128>::BM;
}

int dkdv_dq_box_d(int dtype, int head_dim) {
  int d;
  if (dtype == ATTN_BF16)
    d = head_dim == 64 ? Layout<true, 64>::STG_D : Layout<true, 128>::STG_D;
  else
    d = head_dim == 64 ? Layout<false, 64>::STG_D : Layout<false, 128>::STG_D;
  return d > 0 ? d : 64;  // configurations without a staged dQ still get a valid map
}

int dkdv_block_n(int dtype, int head_dim) {
  if (dtype == ATTN_BF16) return head_dim == 64 ? Cfg<true, 64>::BN : Cfg<true, 128>::BN;
  return head_dim == 64 ? Cfg<false, 64>::BN : Cfg<false, 128>::BN;
}

cudaError_t launch_dkdv(const attn_bwd_params& p, const TileMaps& maps, const TileArgs& a,
                        cudaStream_t stream, bool after_prepare) {
  if (p.dtype == ATTN_BF16) {
    return p.head_dim == 64 ? launch_impl<true, 64>(maps, a, stream, after_prepare)
                            : launch_impl<true, 128>(maps, a, stream, after_prepare);
  }
  // (fp32, D = 128 launches normally: as a dependent its first wave competed
  // with the prepare kernel's tail and the step was 0.7 % slower)
  return p.head_dim == 64 ? launch_impl<false, 64>(maps, a, stream, after_prepare)
                          : launch_impl<false, 128>(maps, a, stream, false);
}

}  // namespace attnbwd
