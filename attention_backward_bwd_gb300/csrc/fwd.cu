// Attention forward (supporting kernel): produces O and the natural-log LSE
// that the backward consumes.  Not on the timed path.
//
// Online-softmax forward as in TileLang test_tilelang_kernel_mha_bwd.py,
// flashattn_fwd: scores in base 2 (scale * log2 e folded in), running row max
// and sum, causal loop stopped at the diagonal tile with an elementwise mask
// there.  Differences from that page: LSE is returned in natural log (the
// FlashAttention convention the backward API takes), causal uses bottom-right
// alignment (key j allowed iff j <= i + Sk - Sq), GQA and varlen are handled,
// and rows with no allowed key give O = 0, LSE = +inf.
//
// Design: 4 warps per CTA, 64 query rows (16 per warp), 64-key tiles,
// mma.sync m16n8k16 with fp32 accumulation, cp.async double-buffered K/V.
#include <atomic>

#include "common.cuh"

namespace attn {

namespace {

constexpr int kBM = 64, kBN = 64, kFwdThreads = 128;

template <typename T>
struct MmaOp;
template <>
struct MmaOp<__nv_bfloat16> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};
template <>
struct MmaOp<__half> {
  static __device__ __forceinline__ void run(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(ok ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Copy rows [row0, row0 + 64) of a (rows x D) head slice into smem (row stride LD),
// zero-filling rows at or beyond `valid_rows`.
template <typename T, int D, int LD>
__device__ __forceinline__ void load_tile(T* dst, const T* src, int64_t row_stride, int row0,
                                          int valid_rows, int valid_cols) {
  constexpr int kChunks = kBN * D / 8;
  for (int c = threadIdx.x; c < kChunks; c += kFwdThreads) {
    const int r = c / (D / 8);
    const int col = (c % (D / 8)) * 8;
    const int gr = row0 + r;
    // rows past the sequence and columns past a padded head dimension read as 0
    const bool ok = gr < valid_rows && col < valid_cols;
    const T* g = ok ? src + static_cast<int64_t>(gr) * row_stride + col : src;  // no read if !ok
    cp_async16(smem_u32(dst + r * LD + col), g, ok);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kFwdThreads) fwd_kernel(FwdParams p) {
  constexpr int LD = D + 8;  // padded row stride (elements) keeps ldmatrix conflict-free
  extern __shared__ __align__(128) unsigned char smem_raw[];
  T* sQ = reinterpret_cast<T*>(smem_raw);
  T* sK = sQ + kBM * LD;       // [2][kBN][LD]
  T* sV = sK + 2 * kBN * LD;   // [2][kBN][LD]
  if (p.input_bad != nullptr && *p.input_bad) return;

  const int b = blockIdx.z, h = blockIdx.y;
  const SeqInfo si = seq_info(p.seq, b);
  const int m0 = blockIdx.x * kBM;
  if (m0 >= si.sq) return;
  const bool varlen = p.seq.cu_q != nullptr;
  const int hk = h / (p.h_q / p.h_k);
  const T* qg = static_cast<const T*>(p.q.ptr) + (varlen ? 0 : b * p.q.sb) +
                static_cast<int64_t>(si.q_start) * p.q.ss + static_cast<int64_t>(h) * p.q.sh;
  const T* kg = static_cast<const T*>(p.k.ptr) + (varlen ? 0 : b * p.k.sb) +
                static_cast<int64_t>(si.k_start) * p.k.ss + static_cast<int64_t>(hk) * p.k.sh;
  const T* vg = static_cast<const T*>(p.v.ptr) + (varlen ? 0 : b * p.v.sb) +
                static_cast<int64_t>(si.k_start) * p.v.ss + static_cast<int64_t>(hk) * p.v.sh;
  T* og = const_cast<T*>(static_cast<const T*>(p.o.ptr)) + (varlen ? 0 : b * p.o.sb) +
          static_cast<int64_t>(si.q_start) * p.o.ss + static_cast<int64_t>(h) * p.o.sh;

  const int off = si.sk - si.sq;  // bottom-right alignment of causal / window masks
  // key tiles holding a key that some query of this tile sees
  const int n_start = window_first_key(m0, si.sq, si.sk, p.win_left) / kBN;
  int n_end = ceil_div(si.sk, kBN);
  if (p.win_right >= 0) {
    const int last_key = m0 + kBM - 1 + off + p.win_right;
    n_end = min(n_end, last_key < 0 ? 0 : last_key / kBN + 1);
  }

  load_tile<T, D, LD>(sQ, qg, p.q.ss, m0, si.sq, p.head_dim);
  cp_async_commit();
  if (n_end > n_start) {
    load_tile<T, D, LD>(sK, kg, p.k.ss, n_start * kBN, si.sk, p.head_dim);
    load_tile<T, D, LD>(sV, vg, p.v.ss, n_start * kBN, si.sk, p.head_dim);
  }
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  uint32_t qf[D / 16][4];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t a = smem_u32(sQ + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
    ldsm_x4(a, qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lpart[2] = {0.f, 0.f};
  const int row_lo = m0 + warp * 16 + g;

  for (int n = n_start; n < n_end; ++n) {
    const int buf = (n - n_start) & 1;
    if (n + 1 < n_end) {
      load_tile<T, D, LD>(sK + (buf ^ 1) * kBN * LD, kg, p.k.ss, (n + 1) * kBN, si.sk,
                          p.head_dim);
      load_tile<T, D, LD>(sV + (buf ^ 1) * kBN * LD, vg, p.v.ss, (n + 1) * kBN, si.sk,
                          p.head_dim);
    }
    cp_async_commit();
    const T* cK = sK + buf * kBN * LD;
    const T* cV = sV + buf * kBN * LD;

    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t r0, r1, r2, r3;
        const int key = np * 16 + (lane >> 4) * 8 + (lane & 7);
        const int col = kk * 16 + ((lane >> 3) & 1) * 8;
        ldsm_x4(smem_u32(cK + key * LD + col), r0, r1, r2, r3);
        MmaOp<T>::run(s[2 * np], qf[kk], r0, r1);
        MmaOp<T>::run(s[2 * np + 1], qf[kk], r2, r3);
      }
    }

    const bool need_mask = (n * kBN + kBN > si.sk) ||
                           (p.win_right >= 0 && n * kBN + kBN - 1 > m0 + off + p.win_right) ||
                           (p.win_left >= 0 && n * kBN < m0 + kBM - 1 + off - p.win_left);
    float tmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        // logit in log2 units; with a cap c: c tanh(S scale / c) log2 e
        float x = p.softcap > 0.f ? tanh_exp(s[nt][e] * p.cap_in) * p.cap_out
                                  : s[nt][e] * p.scale_log2;
        if (need_mask) {
          const int key = n * kBN + nt * 8 + 2 * t + (e & 1);
          const int row = row_lo + (e >> 1) * 8;
          const bool ok = key < si.sk && (p.win_right < 0 || key <= row + off + p.win_right) &&
                          (p.win_left < 0 || key >= row + off - p.win_left);
          x = ok ? x : -INFINITY;
        }
        s[nt][e] = x;
        tmax[e >> 1] = fmaxf(tmax[e >> 1], x);
      }
    }
    float alpha[2], muse[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 1));
      tmax[r] = fmaxf(tmax[r], __shfl_xor_sync(0xffffffffu, tmax[r], 2));
      const float mnew = fmaxf(mrow[r], tmax[r]);
      muse[r] = (mnew == -INFINITY) ? 0.f : mnew;
      alpha[r] = ex2(mrow[r] - muse[r]);
      mrow[r] = mnew;
      lpart[r] *= alpha[r];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = ex2(s[nt][e] - muse[e >> 1]);
        s[nt][e] = pv;
        lpart[e >> 1] += pv;
      }
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      o[dn][0] *= alpha[0];
      o[dn][1] *= alpha[0];
      o[dn][2] *= alpha[1];
      o[dn][3] *= alpha[1];
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t a[4];
      a[0] = Pack<T>::two(s[2 * kk][0], s[2 * kk][1]);
      a[1] = Pack<T>::two(s[2 * kk][2], s[2 * kk][3]);
      a[2] = Pack<T>::two(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = Pack<T>::two(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t r0, r1, r2, r3;
        const int key = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int col = dp * 16 + (lane >> 4) * 8;
        ldsm_x4_t(smem_u32(cV + key * LD + col), r0, r1, r2, r3);
        MmaOp<T>::run(o[2 * dp], a, r0, r1);
        MmaOp<T>::run(o[2 * dp + 1], a, r2, r3);
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }

  float inv[2], lse[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = lpart[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    inv[r] = l > 0.f ? 1.f / l : 0.f;
    // natural log: (m + log2 l) * ln 2
    lse[r] = l > 0.f ? (mrow[r] + __log2f(l)) * 0.6931471805599453f : INFINITY;
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int row = row_lo + r * 8;
    if (row < si.sq) {
      T* orow = og + static_cast<int64_t>(row) * p.o.ss;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        const uint32_t v = Pack<T>::two(o[dn][2 * r] * inv[r], o[dn][2 * r + 1] * inv[r]);
        if (dn * 8 < p.head_dim)  // a padded head dimension stops early
          *reinterpret_cast<uint32_t*>(orow + dn * 8 + 2 * t) = v;
      }
      if (t == 0) {
        const int64_t li = varlen ? static_cast<int64_t>(h) * p.seq.seqlen_q + si.q_start + row
                                  : (static_cast<int64_t>(b) * p.h_q + h) * p.seq.seqlen_q + row;
        p.lse[li] = lse[r];
      }
    }
  }
}

template <typename T, int D>
cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t stream) {
  constexpr int LD = D + 8;
  const size_t smem = static_cast<size_t>(5) * kBM * LD * sizeof(T);
  // Kernel attributes are per device: set them once on each.
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  dim3 grid(ceil_div(p.max_seqlen_q, kBM), p.h_q, p.seq.batch);
  fwd_kernel<T, D><<<grid, kFwdThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int dtype, cudaStream_t stream) {
  if (dtype == 1) {
    return pad_head_dim(p.head_dim) == 64 ? launch_fwd_t<__nv_bfloat16, 64>(p, stream)
                                          : launch_fwd_t<__nv_bfloat16, 128>(p, stream);
  }
  return pad_head_dim(p.head_dim) == 64 ? launch_fwd_t<__half, 64>(p, stream)
                                        : launch_fwd_t<__half, 128>(p, stream);
}

}  // namespace attn
