// Backward preprocess and postprocess kernels (memory-bound streaming).
//
// Preprocess (TileLang test_tilelang_kernel_mha_bwd.py, flashattn_bwd_preprocess;
// flash-attention hopper/flash_bwd_launch_template.h, run_flash_bwd's
// preprocess launch with Clear_dQaccum):
//   Delta[h, row] = sum_d O[b, i, h, d] * dO[b, i, h, d]   (fp32)
//   LSE2[h, row]  = LSE[b, h, i] * log2(e)                 (base-2 copy)
//   dQaccum = 0, dq semaphores = 0.
// Postprocess (mslk flash_bwd_postprocess.py, FlashAttentionBackwardPostprocess;
// flash_bwd_launch_template.h, FlashAttnBwdPostprocessConvertdQ):
//   dQ[b, i, h, :] = scale * dQaccum[h, row, :]  cast to fp16/bf16.
//
// Both walk rows in [token][head] order so that each group of D/8 threads
// reads or writes one contiguous 16-byte-per-thread head row.
#include <atomic>

#include "common.cuh"

namespace attn {

namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Address of query-side row i of sequence b, head h (padded: batch slab b; varlen: packed row).
template <typename T>
__device__ __forceinline__ const T* row_ptr(const TensorArg& t, bool varlen, const SeqInfo& si,
                                            int b, int i, int h) {
  const T* base = static_cast<const T*>(t.ptr);
  const int64_t bo = varlen ? 0 : static_cast<int64_t>(b) * t.sb;
  return base + bo + static_cast<int64_t>(si.q_start + i) * t.ss + static_cast<int64_t>(h) * t.sh;
}

// Workspace row -> (sequence, row within it).  Returns false for padding rows.
__device__ __forceinline__ bool ws_row_to_seq(const SeqParams& s, int64_t row, int& b, int& i,
                                              SeqInfo& si) {
  if (s.cu_q == nullptr) {
    const int sr = round_up(s.seqlen_q, kTileRows);
    b = static_cast<int>(row / sr);
    i = static_cast<int>(row - static_cast<int64_t>(b) * sr);
    if (b >= s.batch) return false;
    si = seq_info(s, b);
    return i < si.sq;
  }
  // ws_row0(b) = kTileRows * (cu_q[b] / kTileRows + b) is increasing in b.
  int lo = 0, hi = s.batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    const int64_t r0 = static_cast<int64_t>(kTileRows) * (s.cu_q[mid] / kTileRows + mid);
    if (r0 <= row) lo = mid; else hi = mid - 1;
  }
  b = lo;
  si = seq_info(s, b);
  const int64_t ii = row - si.ws_row0;
  if (ii < 0 || ii >= si.sq) return false;
  i = static_cast<int>(ii);
  return true;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 8) preprocess_kernel(BwdParams p) {
  if (p.input_bad != nullptr && *p.input_bad) return;
  constexpr int kGroup = D / 8;  // threads per head row, 16 B each
  const int64_t n_groups = p.ws_rows * p.h_q;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  const int c = threadIdx.x % kGroup;

  // Phase 1: Delta and LSE2 for every workspace row (0 for padding rows), and the
  // row's fp32 dQ accumulator cleared (those stores and the O/dO loads are in flight together).
  // Iterate per warp so every lane reaches the shuffles below.
  constexpr int kGroupsPerWarp = 32 / kGroup;
  const int64_t warp_g = gtid / 32;
  const int64_t n_warps = nthreads / 32;
  for (int64_t base = warp_g * kGroupsPerWarp; base < n_groups; base += n_warps * kGroupsPerWarp) {
    const int64_t g = base + (threadIdx.x & 31) / kGroup;
    const bool in_range = g < n_groups;
    const int64_t row = in_range ? g / p.h_q : 0;
    const int h = in_range ? static_cast<int>(g - row * p.h_q) : 0;
    int b = 0, i = 0;
    SeqInfo si;
    const bool valid = in_range && ws_row_to_seq(p.seq, row, b, i, si);
    if (in_range) {
      float4* z = reinterpret_cast<float4*>(
          p.dqacc + (static_cast<int64_t>(h) * p.ws_rows + row) * D + c * 8);
      z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc = 0.f;
    if (valid && c * 8 < p.head_dim) {  // a padded head dimension has fewer columns
      const uint4 ov = *reinterpret_cast<const uint4*>(row_ptr<T>(p.o, p.seq.cu_q != nullptr, si, b, i, h) + c * 8);
      const uint4 dv = *reinterpret_cast<const uint4*>(row_ptr<T>(p.dout, p.seq.cu_q != nullptr, si, b, i, h) + c * 8);
      const uint32_t* o32 = reinterpret_cast<const uint32_t*>(&ov);
      const uint32_t* d32 = reinterpret_cast<const uint32_t*>(&dv);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 a = Pack<T>::unpack(o32[e]);
        const float2 d = Pack<T>::unpack(d32[e]);
        acc = fmaf(a.x, d.x, acc);
        acc = fmaf(a.y, d.y, acc);
      }
    }
#pragma unroll
    for (int off = kGroup / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (c == 0 && in_range) {
      float l2 = 0.f;
      if (valid) {
        const int64_t li = (p.seq.cu_q == nullptr)
                               ? (static_cast<int64_t>(b) * p.h_q + h) * p.seq.seqlen_q + i
                               : static_cast<int64_t>(h) * p.seq.seqlen_q + si.q_start + i;
        l2 = p.lse[li] * kLog2e;
      }
      const int64_t wi = static_cast<int64_t>(h) * p.ws_rows + row;
      p.delta[wi] = valid ? acc : 0.f;
      p.lse2[wi] = l2;
    }
  }

  // Phase 2: clear the deterministic-mode semaphores and the work counters after them.
  const int64_t ns = p.ws_rows / kTileRows * p.h_q * 4 + kSchedCounters;
  for (int64_t e = gtid; e < ns; e += nthreads) p.sem[e] = 0;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) postprocess_kernel(BwdParams p) {
  if (p.input_bad != nullptr && *p.input_bad) return;
  constexpr int kGroup = D / 8;
  const int64_t tokens = (p.seq.cu_q == nullptr)
                             ? static_cast<int64_t>(p.seq.batch) * p.seq.seqlen_q
                             : static_cast<int64_t>(p.seq.seqlen_q);
  const int64_t n_groups = tokens * p.h_q;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  const int c = threadIdx.x % kGroup;
  for (int64_t g = gtid / kGroup; g < n_groups; g += nthreads / kGroup) {
    const int64_t tok = g / p.h_q;
    const int h = static_cast<int>(g - tok * p.h_q);
    int b, i;
    if (p.seq.cu_q == nullptr) {
      b = static_cast<int>(tok / p.seq.seqlen_q);
      i = static_cast<int>(tok - static_cast<int64_t>(b) * p.seq.seqlen_q);
    } else {
      b = seq_of_row(p.seq.cu_q, p.seq.batch, static_cast<int>(tok));
      i = static_cast<int>(tok) - p.seq.cu_q[b];
    }
    const SeqInfo si = seq_info(p.seq, b);
    if (i >= si.sq) continue;  // past a used length: left as it was
    const float* src = p.dqacc + ((static_cast<int64_t>(h) * p.ws_rows + si.ws_row0 + i) * D + c * 8);
    const float4 a = reinterpret_cast<const float4*>(src)[0];
    const float4 d = reinterpret_cast<const float4*>(src)[1];
    uint4 out;
    out.x = Pack<T>::two(a.x * p.scale, a.y * p.scale);
    out.y = Pack<T>::two(a.z * p.scale, a.w * p.scale);
    out.z = Pack<T>::two(d.x * p.scale, d.y * p.scale);
    out.w = Pack<T>::two(d.z * p.scale, d.w * p.scale);
    T* dst = const_cast<T*>(row_ptr<T>(p.dq, p.seq.cu_q != nullptr, si, b, i, h)) + c * 8;
    if (c * 8 < p.head_dim) *reinterpret_cast<uint4*>(dst) = out;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    zero_rows_kernel(TensorArg t, int nseq, int rows_per_seq, const int* cu, int total_rows,
                     int heads, int head_dim) {
  constexpr int kGroup = D / 8;
  const int64_t rows = (cu == nullptr) ? static_cast<int64_t>(nseq) * rows_per_seq : total_rows;
  const int64_t n_groups = rows * heads;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kThreads;
  const int c = threadIdx.x % kGroup;
  for (int64_t g = gtid / kGroup; g < n_groups; g += nthreads / kGroup) {
    const int64_t r = g / heads;
    const int h = static_cast<int>(g - r * heads);
    int64_t off;
    if (cu == nullptr) {
      const int64_t b = r / rows_per_seq;
      off = b * t.sb + (r - b * rows_per_seq) * t.ss + static_cast<int64_t>(h) * t.sh;
    } else {
      off = r * t.ss + static_cast<int64_t>(h) * t.sh;
    }
    T* dst = const_cast<T*>(static_cast<const T*>(t.ptr)) + off + c * 8;
    if (c * 8 < head_dim) *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// Checks the used-length arrays: 0 <= used[b] <= the rows of sequence b.
__global__ void validate_used_kernel(SeqParams s, unsigned int* bad) {
  for (int b = threadIdx.x; b < s.batch; b += blockDim.x) {
    unsigned int code = 0;
    const int cap_q = s.cu_q != nullptr ? s.cu_q[b + 1] - s.cu_q[b] : s.seqlen_q;
    const int cap_k = s.cu_k != nullptr ? s.cu_k[b + 1] - s.cu_k[b] : s.seqlen_k;
    if (s.used_q != nullptr && (s.used_q[b] < 0 || s.used_q[b] > cap_q)) code = 0xB0000005u;
    if (s.used_k != nullptr && (s.used_k[b] < 0 || s.used_k[b] > cap_k)) code = 0xB0000006u;
    if (code) atomicCAS(bad, 0u, code);
  }
}

// Checks that cu_seqlens describe a valid packing: start at 0, nondecreasing,
// end at the total row count, no sequence longer than max_seqlen.  Any
// violation sets *bad, and every later kernel of the call returns at once.
__global__ void validate_cu_kernel(const int* cu_q, const int* cu_k, int batch, int total_q,
                                   int total_k, int max_q, int max_k, unsigned int* bad) {
  for (int b = threadIdx.x; b <= batch; b += blockDim.x) {
    unsigned int code = 0;
    const int q1 = cu_q[b], k1 = cu_k[b];
    if (b == 0 && (q1 != 0 || k1 != 0)) code = 0xB0000001u;
    if (b == batch && (q1 != total_q || k1 != total_k)) code = 0xB0000002u;
    if (b > 0) {
      const int lq = q1 - cu_q[b - 1], lk = k1 - cu_k[b - 1];
      if (lq < 0 || lk < 0) code = 0xB0000003u;
      if (lq > max_q || lk > max_k) code = 0xB0000004u;
    }
    if (code) atomicCAS(bad, 0u, code);
  }
}

// Blocks per SM of one kernel, looked up once per device (the first launch on a
// device must not happen inside a stream capture).
struct Occupancy {
  static constexpr int kMaxDevices = 64;
  std::atomic<int> per_sm[kMaxDevices];
};

// Grid-stride launches: one full wave (as many blocks as fit on every SM at once), so
// no block starts late and runs in a half-empty second wave.
template <typename K>
inline int grid_for(int64_t work_threads, K kernel, Occupancy& occ) {
  int dev = 0;
  int per_sm = 0;
  const bool dev_ok =
      cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < Occupancy::kMaxDevices;
  if (dev_ok) per_sm = occ.per_sm[dev].load(std::memory_order_relaxed);
  if (per_sm < 1) {
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel,
                                                                        kThreads, 0);
    if (e != cudaSuccess || per_sm < 1)
      per_sm = 1;
    else if (dev_ok)
      occ.per_sm[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t want = (work_threads + kThreads - 1) / kThreads;
  const int64_t cap = static_cast<int64_t>(num_sms()) * per_sm;
  return static_cast<int>(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

template <typename T>
static cudaError_t launch_pre_t(const BwdParams& p, cudaStream_t stream) {
  const int64_t work = p.ws_rows * p.h_q * (pad_head_dim(p.head_dim) / 8);
  static Occupancy occ64, occ128, occ256;
  if (pad_head_dim(p.head_dim) == 64)
    preprocess_kernel<T, 64>
        <<<grid_for(work, preprocess_kernel<T, 64>, occ64), kThreads, 0, stream>>>(p);
  else if (pad_head_dim(p.head_dim) == 128)
    preprocess_kernel<T, 128>
        <<<grid_for(work, preprocess_kernel<T, 128>, occ128), kThreads, 0, stream>>>(p);
  else
    preprocess_kernel<T, 256>
        <<<grid_for(work, preprocess_kernel<T, 256>, occ256), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const BwdParams& p, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_pre_t<__nv_bfloat16>(p, stream) : launch_pre_t<__half>(p, stream);
}

template <typename T>
static cudaError_t launch_post_t(const BwdParams& p, cudaStream_t stream) {
  const int64_t tokens = (p.seq.cu_q == nullptr)
                             ? static_cast<int64_t>(p.seq.batch) * p.seq.seqlen_q
                             : static_cast<int64_t>(p.seq.seqlen_q);
  const int64_t work = tokens * p.h_q * (pad_head_dim(p.head_dim) / 8);
  if (work == 0) return cudaSuccess;
  static Occupancy occ64, occ128, occ256;
  if (pad_head_dim(p.head_dim) == 64)
    postprocess_kernel<T, 64>
        <<<grid_for(work, postprocess_kernel<T, 64>, occ64), kThreads, 0, stream>>>(p);
  else if (pad_head_dim(p.head_dim) == 128)
    postprocess_kernel<T, 128>
        <<<grid_for(work, postprocess_kernel<T, 128>, occ128), kThreads, 0, stream>>>(p);
  else
    postprocess_kernel<T, 256>
        <<<grid_for(work, postprocess_kernel<T, 256>, occ256), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_postprocess(const BwdParams& p, int dtype, cudaStream_t stream) {
  return dtype == 1 ? launch_post_t<__nv_bfloat16>(p, stream) : launch_post_t<__half>(p, stream);
}

template <typename T>
static cudaError_t launch_zero_t(const TensorArg& t, int nseq, int rows_per_seq, const int* cu,
                                 int total_rows, int heads, int head_dim, cudaStream_t stream) {
  const int64_t rows = (cu == nullptr) ? static_cast<int64_t>(nseq) * rows_per_seq : total_rows;
  const int64_t work = rows * heads * (pad_head_dim(head_dim) / 8);
  if (work == 0) return cudaSuccess;
  static Occupancy occ64, occ128, occ256;
  if (pad_head_dim(head_dim) == 64)
    zero_rows_kernel<T, 64><<<grid_for(work, zero_rows_kernel<T, 64>, occ64), kThreads, 0,
                              stream>>>(t, nseq, rows_per_seq, cu, total_rows, heads, head_dim);
  else if (pad_head_dim(head_dim) == 128)
    zero_rows_kernel<T, 128><<<grid_for(work, zero_rows_kernel<T, 128>, occ128), kThreads, 0,
                               stream>>>(t, nseq, rows_per_seq, cu, total_rows, heads, head_dim);
  else
    zero_rows_kernel<T, 256><<<grid_for(work, zero_rows_kernel<T, 256>, occ256), kThreads, 0,
                               stream>>>(t, nseq, rows_per_seq, cu, total_rows, heads, head_dim);
  return cudaGetLastError();
}

cudaError_t launch_validate_cu(const int* cu_q, const int* cu_k, int batch, int total_q,
                               int total_k, int max_q, int max_k, unsigned int* bad,
                               cudaStream_t stream) {
  validate_cu_kernel<<<1, 256, 0, stream>>>(cu_q, cu_k, batch, total_q, total_k, max_q, max_k, bad);
  return cudaGetLastError();
}

cudaError_t launch_validate_used(const SeqParams& s, unsigned int* bad, cudaStream_t stream) {
  validate_used_kernel<<<1, 256, 0, stream>>>(s, bad);
  return cudaGetLastError();
}

cudaError_t launch_zero_rows(const TensorArg& t, int dtype, int nseq, int rows_per_seq,
                             const int* cu, int total_rows, int heads, int head_dim,
                             cudaStream_t stream) {
  return dtype == 1 ? launch_zero_t<__nv_bfloat16>(t, nseq, rows_per_seq, cu, total_rows, heads,
                                                   head_dim, stream)
                    : launch_zero_t<__half>(t, nseq, rows_per_seq, cu, total_rows, heads, head_dim,
                                            stream);
}

}  // namespace attn
