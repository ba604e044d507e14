// Decode (one query per head) attention backward, memory-bound.
//
// The decode page ("rullama attention_backward_dq.wgsl") runs one workgroup
// per query head and sweeps the K/V history three times (d_probs, d_scores,
// then d_q with a strided, uncoalesced k_hist walk).  Here the history of a
// (sequence, KV head) is read from HBM exactly once for all the query heads
// that share it, using
//   d_q_h = sum_j probs_hj (dp_hj - sum_pd_h) k_j
//         = sum_j probs_hj dp_hj k_j  -  sum_pd_h * sum_j probs_hj k_j,
// so one pass over the history can accumulate both sums together with
// sum_pd_h = sum_j probs_hj dp_hj, and a small finalize kernel combines them.
//
// decode_main: grid (splits, seqs * n_kv).  Each CTA streams its share of the
//   history in chunks of CH keys, double-buffered in shared memory with bulk
//   async copies.  Phase 1 (warp per key): dp_hj = d_out_h . v_j for all G
//   heads, lane-split over d and reduced with a transposing butterfly; dp is
//   parked in d_scores.  Phase 2 (thread per d): accumulate
//   A_h[d] += probs_hj dp_hj k_j[d] and B_h[d] += probs_hj k_j[d].
//   Per-CTA partials (sum_pd, A, B) go to the workspace.
// decode_finalize: grid (n_heads, seqs).  Sums the partials, writes
//   d_q = A - sum_pd B, and rewrites d_scores = probs (dp - sum_pd).
#include <cuda_runtime.h>

#include "internal.h"
#include "ptx.cuh"

namespace attnbwd {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecChunk = 16;     // keys per pipeline stage
constexpr int kDecStages = 3;     // 3 stages x (K + V) x 16 rows x 1 KB = 96 KB at D = 256
constexpr int kDecCtasPerSm = 2;
constexpr int kDecSlots = 152 * kDecCtasPerSm;

struct DecArgs {
  const float* k;
  const float* v;
  const float* probs;
  const float* d_out;
  float* d_scores;
  float* d_q;
  float* partials;
  int n_heads, n_kv, D, hist, n_split, keys_per_split;
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

template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, (G * D / 32 <= 64) ? kDecCtasPerSm : 1)
    decode_main_kernel(const DecArgs a) {
  constexpr int DPL = D / 32;               // d values per lane in phase 1
  constexpr int NKG = kDecThreads / D;      // key groups in phase 2
  constexpr int LOG_G = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : G == 8 ? 3 : 4;
  constexpr int ROW_BYTES = D * 4;
  constexpr int STAGE_BYTES = 2 * kDecChunk * ROW_BYTES;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  float* stage_base = reinterpret_cast<float*>(smem_raw);  // [stages][K|V][CH][D]
  // key-major so that one vector load returns consecutive heads of a key
  __shared__ __align__(16) float w1_s[kDecChunk][G];     // probs * dp
  __shared__ __align__(16) float pr_s[2][kDecChunk][G];  // probs (chunk parity)
  __shared__ float red_s[NKG > 1 ? NKG : 1][2 * G][NKG > 1 ? D : 1];  // only used if NKG > 1
  __shared__ float sumpd_s[kDecThreads / 32][G];
  __shared__ __align__(8) uint64_t full[kDecStages];

  const int split = blockIdx.x;
  const int pair = blockIdx.y;  // seq * n_kv + kv
  const int seq = pair / a.n_kv, kv = pair % a.n_kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j_begin = split * a.keys_per_split;
  const int j_end = min(a.hist, j_begin + a.keys_per_split);
  const int nchunks = j_end > j_begin ? (j_end - j_begin + kDecChunk - 1) / kDecChunk : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  int issued = 0;            // chunks requested so far (tracked by warp 0)
  auto issue = [&](int c) {  // warp 0: bring chunk c into stage c % kDecStages
    const int s = c % kDecStages;
    issued = c + 1;
    const int j0 = j_begin + c * kDecChunk;
    const int rows = min(kDecChunk, j_end - j0);
    float* ks = stage_base + (size_t)s * (STAGE_BYTES / 4);
    float* vs = ks + kDecChunk * D;
    if (lane == 0) mbar_expect_tx(&full[s], 2u * rows * ROW_BYTES);
    __syncwarp();
    if (a.n_kv == 1) {
      // the chunk's rows are contiguous: one copy per tensor
      if (lane == 0) {
        const size_t row = (size_t)seq * a.hist + j0;
        bulk_load(ks, a.k + row * D, rows * ROW_BYTES, &full[s]);
        bulk_load(vs, a.v + row * D, rows * ROW_BYTES, &full[s]);
      }
    } else if (lane < rows) {
      const size_t row = ((size_t)seq * a.hist + j0 + lane) * a.n_kv + kv;
      bulk_load(ks + lane * D, a.k + row * D, ROW_BYTES, &full[s]);
      bulk_load(vs + lane * D, a.v + row * D, ROW_BYTES, &full[s]);
    }
  };
  if (warp == 0) {
    for (int c = 0; c < kDecStages - 1 && c < nchunks; ++c) issue(c);
  }

  // d_out of the G heads, lane-split over d (phase 1 operand, kept in registers)
  float dout[G][DPL];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float* src = a.d_out + ((size_t)seq * a.n_heads + kv * G + g) * D + lane * DPL;
#pragma unroll
    for (int k = 0; k < DPL; ++k) dout[g][k] = src[k];
  }
  float sumpd_part = 0.f;  // valid in the lanes that own a head after the reduction
  float accA[G], accB[G];
#pragma unroll
  for (int g = 0; g < G; ++g) accA[g] = accB[g] = 0.f;
  uint64_t accA2[G / 2 > 0 ? G / 2 : 1], accB2[G / 2 > 0 ? G / 2 : 1];
#pragma unroll
  for (int i = 0; i < (G / 2 > 0 ? G / 2 : 1); ++i) accA2[i] = accB2[i] = 0;
  const int d2 = threadIdx.x % D, kg = threadIdx.x / D;
  bool ok = true;
  // probabilities of a chunk, G x kDecChunk values, staged one chunk ahead so
  // phase 1 never waits on a global load
  auto load_probs = [&](int c) {
    if (threadIdx.x < G * kDecChunk && c < nchunks) {
      const int g = threadIdx.x / kDecChunk, jj = threadIdx.x % kDecChunk;
      const int j = j_begin + c * kDecChunk + jj;
      pr_s[c & 1][jj][g] =
          j < j_end ? a.probs[((size_t)seq * a.n_heads + kv * G + g) * a.hist + j] : 0.f;
    }
  };
  load_probs(0);
  __syncthreads();

  for (int c = 0; c < nchunks; ++c) {
    const int s = c % kDecStages;
    const int j0 = j_begin + c * kDecChunk;
    const int rows = min(kDecChunk, j_end - j0);
    // keep kDecStages - 1 chunks in flight: the stage refilled here was
    // released by the __syncthreads that ended chunk c - 1
    if (warp == 0 && c + kDecStages - 1 < nchunks) issue(c + kDecStages - 1);
    load_probs(c + 1);  // visible after this chunk's closing __syncthreads
    ok = mbar_wait(&full[s], (c / kDecStages) & 1, a.err);
    const float* ks = stage_base + (size_t)s * (STAGE_BYTES / 4);
    const float* vs = ks + kDecChunk * D;
    // phase 1: dp for the G heads, one key per warp at a time (unrolled so the
    // shuffle chains of a warp's keys interleave)
#pragma unroll
    for (int jj = warp; jj < kDecChunk; jj += kDecThreads / 32) {
      float part[G];
      if (jj < rows) {
        float vv[DPL];
#pragma unroll
        for (int k = 0; k < DPL; k += 4) {
          const float4 t = *reinterpret_cast<const float4*>(vs + jj * D + lane * DPL + k);
          vv[k] = t.x;
          if (k + 1 < DPL) vv[k + 1] = t.y;
          if (k + 2 < DPL) vv[k + 2] = t.z;
          if (k + 3 < DPL) vv[k + 3] = t.w;
        }
        if constexpr (G % 2 == 0) {
          // two heads per packed fma
#pragma unroll
          for (int g = 0; g < G; g += 2) {
            uint64_t acc = 0;
#pragma unroll
            for (int k = 0; k < DPL; ++k)
              acc = f2fma(pk2(dout[g][k], dout[g + 1][k]), pk2(vv[k], vv[k]), acc);
            up2(acc, part[g], part[g + 1]);
          }
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < DPL; ++k) acc = fmaf(dout[g][k], vv[k], acc);
            part[g] = acc;
          }
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) part[g] = 0.f;
      }
      const float dp = warp_reduce_scatter<G>(part, lane);
      const int g = lane >> (5 - LOG_G);
      if ((lane & ((32 >> LOG_G) - 1)) == 0) {
        float w1 = 0.f;
        if (jj < rows) {
          const size_t idx = ((size_t)seq * a.n_heads + kv * G + g) * a.hist + j0 + jj;
          w1 = pr_s[c & 1][jj][g] * dp;
          a.d_scores[idx] = dp;  // parked; finalize turns it into d_scores
          sumpd_part += w1;
        }
        w1_s[jj][g] = w1;
      }
    }
    // block-uniform exit if any thread's wait gave up (error path only)
    if (__syncthreads_or(!ok)) {
      ok = false;
      break;
    }
    // phase 2: A += (probs dp) k, B += probs k, thread per d; heads in pairs
    // with packed fma, weights of a key read as vectors (keys past `rows`
    // carry zero weights)
    for (int jj = kg; jj < rows; jj += NKG) {
      const float kval = ks[jj * D + d2];
      if constexpr (G % 2 == 0) {
        const uint64_t k2 = pk2(kval, kval);
        const uint64_t* w2 = reinterpret_cast<const uint64_t*>(&w1_s[jj][0]);
        const uint64_t* p2 = reinterpret_cast<const uint64_t*>(&pr_s[c & 1][jj][0]);
#pragma unroll
        for (int i = 0; i < G / 2; ++i) {
          accA2[i] = f2fma(w2[i], k2, accA2[i]);
          accB2[i] = f2fma(p2[i], k2, accB2[i]);
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          accA[g] = fmaf(w1_s[jj][g], kval, accA[g]);
          accB[g] = fmaf(pr_s[c & 1][jj][g], kval, accB[g]);
        }
      }
    }
    __syncthreads();  // stage s and w1_s / pr_s are free again
  }

  if constexpr (G % 2 == 0) {
#pragma unroll
    for (int i = 0; i < G / 2; ++i) {
      up2(accA2[i], accA[2 * i], accA[2 * i + 1]);
      up2(accB2[i], accB[2 * i], accB[2 * i + 1]);
    }
  }
  // per-warp sum_pd partials -> smem
  {
    const int g = lane >> (5 - LOG_G);
    if ((lane & ((32 >> LOG_G) - 1)) == 0) sumpd_s[warp][g] = sumpd_part;
  }
  if (NKG > 1) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      red_s[kg][g][d2] = accA[g];
      red_s[kg][G + g][d2] = accB[g];
    }
  }
  __syncthreads();
  float* out = a.partials + ((size_t)pair * a.n_split + split) * G * (1 + 2 * D);
  if (threadIdx.x < G) {
    float t = 0.f;
    for (int w = 0; w < kDecThreads / 32; ++w) t += sumpd_s[w][threadIdx.x];
    out[threadIdx.x * (1 + 2 * D)] = ok ? t : 0.f;
  }
  if (kg == 0) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float sa = accA[g], sb = accB[g];
      for (int q = 1; q < NKG; ++q) {
        sa += red_s[q][g][d2];
        sb += red_s[q][G + g][d2];
      }
      out[g * (1 + 2 * D) + 1 + d2] = sa;
      out[g * (1 + 2 * D) + 1 + D + d2] = sb;
    }
  }
  // copies still in flight (only when a wait gave up) must land before exit
  if (!ok && threadIdx.x == 0) {
    for (int c = issued > kDecStages ? issued - kDecStages : 0; c < issued; ++c) {
      long long t0 = clock64();
      while (!mbar_try_wait(&full[c % kDecStages], (c / kDecStages) & 1) &&
             clock64() - t0 < kWaitLimitCycles / 4) {
      }
    }
  }
}

__global__ void __launch_bounds__(256) decode_finalize_kernel(const DecArgs a, int G) {
  const int h = blockIdx.x, seq = blockIdx.y;
  const int kv = h / G, g = h % G;
  const int pair = seq * a.n_kv + kv;
  const int D = a.D;
  const float* base = a.partials + (size_t)pair * a.n_split * G * (1 + 2 * D);
  __shared__ float sumpd_sh;
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int s = 0; s < a.n_split; ++s) t += base[((size_t)s * G + g) * (1 + 2 * D)];
    sumpd_sh = t;
  }
  __syncthreads();
  const float sumpd = sumpd_sh;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float A = 0.f, Bs = 0.f;
    for (int s = 0; s < a.n_split; ++s) {
      const float* pp = base + ((size_t)s * G + g) * (1 + 2 * D);
      A += pp[1 + d];
      Bs += pp[1 + D + d];
    }
    a.d_q[((size_t)seq * a.n_heads + h) * D + d] = A - sumpd * Bs;
  }
  const size_t row = ((size_t)seq * a.n_heads + h) * a.hist;
  for (int j = threadIdx.x; j < a.hist; j += blockDim.x) {
    const float dp = a.d_scores[row + j];
    a.d_scores[row + j] = a.probs[row + j] * (dp - sumpd);
  }
}

template <int D, int G>
cudaError_t main_impl(const DecArgs& a, dim3 grid, cudaStream_t stream) {
  const int smem = kDecStages * 2 * kDecChunk * D * 4;
  auto kern = decode_main_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDecThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int D>
cudaError_t main_by_group(const DecArgs& a, int G, dim3 grid, cudaStream_t stream) {
  switch (G) {
    case 1: return main_impl<D, 1>(a, grid, stream);
    case 2: return main_impl<D, 2>(a, grid, stream);
    case 4: return main_impl<D, 4>(a, grid, stream);
    case 8: return main_impl<D, 8>(a, grid, stream);
    case 16: return main_impl<D, 16>(a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int decode_num_splits(const attn_bwd_decode_params& p) {
  const long long pairs = (long long)p.num_seqs * p.n_kv_heads;
  long long s = kDecSlots / (pairs > 0 ? pairs : 1);
  const long long max_s = (p.history_len + kDecChunk - 1) / kDecChunk;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  return (int)s;
}

size_t decode_partials_floats(const attn_bwd_decode_params& p, int n_split) {
  const int G = p.n_heads / p.n_kv_heads;
  return (size_t)p.num_seqs * p.n_kv_heads * n_split * G * (1 + 2 * (size_t)p.head_dim);
}

cudaError_t launch_decode(const attn_bwd_decode_params& p, const float* k_hist,
                          const float* v_hist, const float* probs, const float* d_out,
                          float* d_scores, float* d_q, float* partials, int n_split,
                          cudaStream_t stream) {
  DecArgs a;
  a.k = k_hist;
  a.v = v_hist;
  a.probs = probs;
  a.d_out = d_out;
  a.d_scores = d_scores;
  a.d_q = d_q;
  a.partials = partials;
  a.n_heads = p.n_heads;
  a.n_kv = p.n_kv_heads;
  a.D = p.head_dim;
  a.hist = p.history_len;
  a.n_split = n_split;
  const int per = (p.history_len + n_split - 1) / n_split;
  a.keys_per_split = (per + kDecChunk - 1) / kDecChunk * kDecChunk;
  a.err = device_error_word();
  if (!a.err) return cudaErrorUnknown;
  const int G = p.n_heads / p.n_kv_heads;
  dim3 grid(n_split, p.num_seqs * p.n_kv_heads);
  cudaError_t e;
  switch (p.head_dim) {
    case 64: e = main_by_group<64>(a, G, grid, stream); break;
    case 128: e = main_by_group<128>(a, G, grid, stream); break;
    case 256: e = main_by_group<256>(a, G, grid, stream); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  decode_finalize_kernel<<<dim3(p.n_heads, p.num_seqs), 256, 0, stream>>>(a, G);
  return cudaGetLastError();
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

// Device address of the scratch array for the current device (nullptr on error).
float* noalloc_scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    float* ptr = nullptr;
    if (cudaGetSymbolAddress((void**)&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return nullptr;
    g_noalloc_ptr[dev] = ptr;
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
