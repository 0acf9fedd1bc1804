// Diagnostic entry points (include/attn_diag.h): single-tile tcgen05 MMAs in
// each operand form the backward kernel uses, so that descriptor or layout
// mistakes show up in isolation, and a bounded-wait self-test for the
// device timeout path.  They use the same helpers as the production kernels.
#include "../../include/attn_bwd.h"
#include "../../include/attn_diag.h"
#include "common.cuh"

namespace attn {
namespace {

constexpr uint32_t kChunk = 128 * 128;

// mode 0: C[128x128] = A[128xD] B[128xD]^T            (A, B K-major via TMA)
// mode 1: C[128xD]   = A[128x128] B[128xD]             (A from TMEM, B MN-major via TMA)
// mode 2: C[128xD]   = At[128x128]^T B[128xD]          (At written to smem with the
//                                                       manual 128-byte swizzle, MN-major A)
template <typename T, int D>
__global__ void __launch_bounds__(128, 1)
    diag_mma_kernel(int mode, const __grid_constant__ CUtensorMap tA,
                    const __grid_constant__ CUtensorMap tB, const T* a_rows, float* c,
                    unsigned int* status, unsigned long long timeout_ns) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {
    if (threadIdx.x == 0) atomicCAS(status, 0u, 0xD1A00001u);
    return;
  }
  const uint32_t sA = sb, sB = sb + 2 * kChunk;
  const uint32_t bar_tma = sb + 4 * kChunk, bar_mma = bar_tma + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 4 * kChunk + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 4 * kChunk + 20);
  const WaitCtl ctl{abort_flag, status, timeout_ns};
  const uint32_t warp = warp_id(), lane = lane_id();
  constexpr int kBf = Pack<T>::kIsBf16;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(bar_tma, 1);
    mbar_init(bar_mma, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const int r = threadIdx.x;  // row / TMEM lane
  const uint32_t tl = tmem + ((warp * 32) << 16);

  if (threadIdx.x == 0) {
    uint32_t bytes = (D / 64) * kChunk;
    if (mode == 0) bytes += (D / 64) * kChunk;
    mbar_expect_tx(bar_tma, bytes);
    for (int cc = 0; cc < D / 64; ++cc) {
      if (mode == 0) tma_load_4d(sA + cc * kChunk, &tA, bar_tma, cc * 64, 0, 0, 0);
      tma_load_4d(sB + cc * kChunk, &tB, bar_tma, cc * 64, 0, 0, 0);
    }
  }
  if (mode == 1) {  // A row r -> TMEM lane r, packed pairs in columns [0, 64)
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t pk[16];
      for (int e = 0; e < 16; ++e) {
        const T* src = a_rows + r * 128 + cc * 32 + 2 * e;
        pk[e] = Pack<T>::two(static_cast<float>(src[0]), static_cast<float>(src[1]));
      }
      tmem_st16(tl + cc * 16, pk);
    }
    tmem_wait_st();
  }
  if (mode == 2) {  // At row r (128 elements) -> swizzled MN-major smem, as dS^T in the kernel
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t pk[16];
      for (int e = 0; e < 16; ++e) {
        const T* src = a_rows + r * 128 + cc * 32 + 2 * e;
        pk[e] = Pack<T>::two(static_cast<float>(src[0]), static_cast<float>(src[1]));
      }
      const uint32_t row_base = (cc >> 1) * kChunk + r * 128;
      for (int q = 0; q < 4; ++q) {
        const uint32_t unit = ((cc & 1) * 4 + q) ^ (r & 7);
        *reinterpret_cast<uint4*>(smem + row_base + unit * 16) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (threadIdx.x == 0) {
    if (wait1(bar_tma, 0, ctl, 0xD1A00002u)) {
      tc_fence_after();
      if (mode == 0) {
        constexpr uint32_t id = idesc_f16(kBf, 0, 0, 128, 128);
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + 0, sdesc_sw128(sA + koff, 16, 1024), sdesc_sw128(sB + koff, 16, 1024), id,
                 kk > 0);
        }
      } else if (mode == 1) {
        constexpr uint32_t id = idesc_f16(kBf, 0, 1, 128, D);
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tmem + 128, tmem + kk * 8, sdesc_sw128(sB + kk * 2048, kChunk, 1024), id, kk > 0);
      } else {
        constexpr uint32_t id = idesc_f16(kBf, 1, 1, 128, D);
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tmem + 256, sdesc_sw128(sA + kk * 2048, kChunk, 1024),
                 sdesc_sw128(sB + kk * 2048, kChunk, 1024), id, kk > 0);
      }
    }
    tc_commit(bar_mma);
  }
  if (wait_warp(bar_mma, 0, ctl, 0xD1A00003u)) {
    tc_fence_after();
    const int ncols = (mode == 0) ? 128 : D;
    const uint32_t col0 = (mode == 0) ? 0 : (mode == 1 ? 128 : 256);
    for (int cc = 0; cc < ncols / 32; ++cc) {
      uint32_t v[32];
      tmem_ld32(tl + col0 + cc * 32, v);
      tmem_wait_ld();
      for (int e = 0; e < 32; ++e) c[r * ncols + cc * 32 + e] = __uint_as_float(v[e]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 512);
}

// Spins on a flag that nothing sets; must give up after timeout_ns and
// record the site in the status word.
__global__ void diag_wait_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const WaitCtl ctl{&abort_flag, status, timeout_ns};
  wait_warp(smem_u32(&bar), 0, ctl, 0xD1A0000Fu);  // phase 0 never completes
  __syncthreads();
}

__global__ void diag_tanh_kernel(const float* x, float* y, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    y[i] = tanh_exp(x[i]);
}

template <typename T, int D>
int diag_mma_t(int mode, const void* a, const void* b, float* c, cudaStream_t stream,
               unsigned int* status, unsigned long long timeout_ns) {
  const int dtype = Pack<T>::kIsBf16 ? ATTN_BF16 : ATTN_FP16;
  CUtensorMap tA, tB;
  TensorArg ta{a, 0, D, D};
  TensorArg tb{b, 0, D, D};
  if (mode == 0 && !encode_tmap_bshd(&tA, ta, dtype, 128, 1, 1, D, 128)) return ATTN_ERR_CUDA;
  if (!encode_tmap_bshd(&tB, tb, dtype, 128, 1, 1, D, 128)) return ATTN_ERR_CUDA;
  if (mode != 0) tA = tB;
  const int smem = 4 * kChunk + 64;
  cudaFuncSetAttribute(diag_mma_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  diag_mma_kernel<T, D><<<1, 128, smem, stream>>>(mode, tA, tB, static_cast<const T*>(a), c,
                                                  status, timeout_ns);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

int attn_diag_mma(int mode, int dtype, int head_dim, const void* a, const void* b, float* c,
                  attn_stream_t stream) {
  if (mode < 0 || mode > 2) return ATTN_ERR_ARG;
  if (head_dim != 64 && head_dim != 128) return ATTN_ERR_SHAPE;
  if (a == nullptr || b == nullptr || c == nullptr) return ATTN_ERR_NULL;
  unsigned int* st = status_word();
  if (st == nullptr) return ATTN_ERR_CUDA;
  const unsigned long long to = 2000000000ull;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == ATTN_BF16)
    return head_dim == 64 ? diag_mma_t<__nv_bfloat16, 64>(mode, a, b, c, s, st, to)
                          : diag_mma_t<__nv_bfloat16, 128>(mode, a, b, c, s, st, to);
  if (dtype == ATTN_FP16)
    return head_dim == 64 ? diag_mma_t<__half, 64>(mode, a, b, c, s, st, to)
                          : diag_mma_t<__half, 128>(mode, a, b, c, s, st, to);
  return ATTN_ERR_DTYPE;
}

int attn_diag_tanh(const float* x, float* y, int n, attn_stream_t stream) {
  if (x == nullptr || y == nullptr) return ATTN_ERR_NULL;
  if (n <= 0) return ATTN_ERR_ARG;
  diag_tanh_kernel<<<64, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(x, y, n);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_diag_wait_timeout(int64_t timeout_ns, attn_stream_t stream) {
  if (timeout_ns <= 0 || timeout_ns > 2000000000LL) return ATTN_ERR_ARG;
  unsigned int* st = status_word();
  if (st == nullptr) return ATTN_ERR_CUDA;
  diag_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      st, static_cast<unsigned long long>(timeout_ns));
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"
