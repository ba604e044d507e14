// Tensor-core self test: one CTA computes C = A * B^T with tcgen05.mma from
// operands staged in 128-byte-swizzled shared memory, in K-major or MN-major
// form (TF32 MN-major: the 128-byte swizzle of 32-byte atoms), and reads the
// accumulator back from tensor memory.  This is the
// building block every tile kernel of the library relies on (same descriptor
// and swizzle helpers), checked in isolation against a CPU product.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_bwd.h"
#include "internal.h"
#include "ptx.cuh"

namespace attnbwd {

namespace {

constexpr int kMaxDim = 256;

// Byte offset of element `pos` (0..W-1) of row `row` in column block `blk`
// of a 128-byte-swizzled tile with `rows` rows per block.
__device__ __forceinline__ uint32_t sw128_offset(int blk, int rows, int row, int pos_bytes) {
  const int chunk = (pos_bytes >> 4) ^ (row & 7);
  return (uint32_t)(blk * rows * 128 + row * 128 + chunk * 16 + (pos_bytes & 15));
}

// The same for the 128-byte swizzle of 32-byte atoms (TF32 MN-major
// operands): the 32-byte chunk index is XORed with (row & 3).
__device__ __forceinline__ uint32_t sw128a32_offset(int blk, int rows, int row, int pos_bytes) {
  const int chunk = (pos_bytes >> 5) ^ (row & 3);
  return (uint32_t)(blk * rows * 128 + row * 128 + chunk * 32 + (pos_bytes & 31));
}

template <bool BF16>
__global__ void __launch_bounds__(128) selftest_mma_kernel(int M, int N, int K, int a_mn, int b_mn, int a_tmem,
                                                           const void* __restrict__ A,
                                                           const void* __restrict__ B,
                                                           float* __restrict__ C,
                                                           float* __restrict__ dump,
                                                           unsigned int* err) {
  using T = typename std::conditional<BF16, __nv_bfloat16, float>::type;
  constexpr int E = sizeof(T);
  constexpr int W = 128 / E;  // elements per 128-byte row segment
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;                                  // up to 128 x 128 fp32 = 64 KB
  uint8_t* sB = smem + 65536;                          // up to 256 x 128 fp32 = 128 KB
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;

  const T* gA = reinterpret_cast<const T*>(A);
  const T* gB = reinterpret_cast<const T*>(B);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;

  // Stage A [M][K] and B [N][K].  K-major: blocks along K, rows = M (or N).
  // MN-major: blocks along M (or N), rows = K.
  for (int idx = tid; idx < M * K; idx += blockDim.x) {
    const int m = idx / K, k = idx % K;
    uint32_t off = a_mn ? (BF16 ? sw128_offset(m / W, K, k, (m % W) * E)
                                : sw128a32_offset(m / W, K, k, (m % W) * E))
                        : sw128_offset(k / W, M, m, (k % W) * E);
    *reinterpret_cast<T*>(sA + off) = gA[idx];
  }
  for (int idx = tid; idx < N * K; idx += blockDim.x) {
    const int n = idx / K, k = idx % K;
    uint32_t off = b_mn ? (BF16 ? sw128_offset(n / W, K, k, (n % W) * E)
                                : sw128a32_offset(n / W, K, k, (n % W) * E))
                        : sw128_offset(k / W, N, n, (k % W) * E);
    *reinterpret_cast<T*>(sB + off) = gB[idx];
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  uint32_t ncols = 32;
  while ((int)ncols < N) ncols <<= 1;
  if (a_tmem) ncols = 512;  // A at column 256
  if (warp == 0) {
    tmem_alloc(&tmem_base, ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (a_tmem) {
    // A [M][K] into TMEM: row m in the lane that holds accumulator row m,
    // K along 32-bit columns (two bf16 per column)
    const int lane128 = warp * 32 + (tid & 31);
    int row = -1;
    if (M == 128) row = lane128;
    else if ((lane128 & 31) < 16) row = (lane128 >> 5) * 16 + (lane128 & 15);
    const int kcols = BF16 ? K / 2 : K;
    for (int c0 = 0; c0 < kcols; c0 += 16) {
      uint32_t r[16];
      for (int c = 0; c < 16; ++c) {
        uint32_t v = 0;
        if (row >= 0 && row < M) {
          if constexpr (BF16) {
            const uint16_t lo = *reinterpret_cast<const uint16_t*>(&gA[row * K + 2 * (c0 + c)]);
            const uint16_t hi = *reinterpret_cast<const uint16_t*>(&gA[row * K + 2 * (c0 + c) + 1]);
            v = (uint32_t)lo | ((uint32_t)hi << 16);
          } else {
            v = __float_as_uint(*reinterpret_cast<const float*>(&gA[row * K + c0 + c]));
          }
        }
        r[c] = v;
      }
      tmem_st16(tmem + ((uint32_t)(warp * 32) << 16) + 256 + c0, r);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  if (warp == 1 && elect_one_sync()) {
    const uint32_t idesc = make_idesc(BF16, M, N, a_mn != 0, b_mn != 0);
    const uint32_t a0 = smem_u32(sA), b0 = smem_u32(sB);
    constexpr int KSTEP = 32 / E;  // elements of K per instruction (32 bytes)
    for (int ks = 0; ks < K / KSTEP; ++ks) {
      uint64_t ad = 0, bd;
      // MN-major: a K step is KSTEP rows; LBO = bytes between MN blocks
      if (a_mn) {
        ad = BF16 ? sw128_desc(a0 + ks * KSTEP * 128, (uint32_t)K * 128u, 1024u)
                  : mn32_desc(a0 + ks * KSTEP * 128, (uint32_t)K * 128u);
      } else {
        const int kb = ks * 32;
        ad = sw128_desc(a0 + (kb / 128) * M * 128 + (kb % 128), 16u, 1024u);
      }
      if (b_mn) {
        bd = BF16 ? sw128_desc(b0 + ks * KSTEP * 128, (uint32_t)K * 128u, 1024u)
                  : mn32_desc(b0 + ks * KSTEP * 128, (uint32_t)K * 128u);
      } else {
        const int kb = ks * 32;
        bd = sw128_desc(b0 + (kb / 128) * N * 128 + (kb % 128), 16u, 1024u);
      }
      if (a_tmem) {
        // KSTEP elements of K = 8 columns (fp32) or 8 columns of bf16 pairs
        mma_ts<BF16>(tmem, tmem + 256 + ks * 8, bd, idesc, ks > 0 ? 1u : 0u);
      } else {
        mma_ss<BF16>(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
      }
    }
    mma_commit(&bar);
  }
  __syncwarp();
  const bool ok = mbar_wait(&bar, 0, err);
  tc_fence_after();

  // Every warp reads its 32-lane sub-partition: lane = warp*32 + (tid & 31).
  const int lane = warp * 32 + (tid & 31);
  if (ok) {
    for (int c0 = 0; c0 < N; c0 += 16) {
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, r);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j) {
        const float v = __uint_as_float(r[j]);
        if (dump) dump[lane * N + c0 + j] = v;
        int row = -1;
        if (M == 128) {
          row = lane;
        } else if ((lane & 31) < 16) {  // M = 64: 16 lanes per sub-partition
          row = (lane >> 5) * 16 + (lane & 15);
        }
        if (row >= 0 && row < M) C[row * N + c0 + j] = v;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

// Failure-path hook: one thread waits on an mbarrier that nothing ever
// arrives on.  The library's bounded wait gives up after about a second, raises
// the device error word and returns, so the kernel ends normally.
__global__ void __launch_bounds__(32) selftest_wait_kernel(unsigned int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, err);
  __syncwarp();
}

}  // namespace

attn_status selftest_wait_launch(cudaStream_t stream) {
  unsigned int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, stream>>>(err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status selftest_mma_launch(int dtype, int M, int N, int K, int a_mn, int b_mn, int a_tmem,
                                const void* A, const void* B, float* C, float* dump,
                                cudaStream_t stream) {
  const int W = dtype == ATTN_BF16 ? 64 : 32;
  if (!(M == 64 || M == 128)) return ATTN_ERR_INVALID;
  if (N < 16 || N > kMaxDim || N % 16 != 0) return ATTN_ERR_INVALID;
  if (K < W || K > 128 || K % W != 0) return ATTN_ERR_INVALID;
  if ((a_mn && M % W) || (b_mn && N % W)) return ATTN_ERR_INVALID;
  if (!A || !B || !C) return ATTN_ERR_INVALID;
  if (a_tmem && (a_mn || N > 256)) return ATTN_ERR_INVALID;
  unsigned int* err = device_error_word();
  if (!err) return ATTN_ERR_CUDA;
  const size_t smem = 1024 + 65536 + 131072;
  cudaError_t e;
  if (dtype == ATTN_BF16) {
    e = cudaFuncSetAttribute(selftest_mma_kernel<true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
      selftest_mma_kernel<true><<<1, 128, smem, stream>>>(M, N, K, a_mn, b_mn, a_tmem, A, B, C,
                                                          dump, err);
      e = cudaGetLastError();
    }
  } else {
    e = cudaFuncSetAttribute(selftest_mma_kernel<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
      selftest_mma_kernel<false><<<1, 128, smem, stream>>>(M, N, K, a_mn, b_mn, a_tmem, A, B, C,
                                                           dump, err);
      e = cudaGetLastError();
    }
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attnbwd
