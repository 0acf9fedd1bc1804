// Attention forward for sm_103a: produces O and the natural-log LSE that the
// backward consumes.  tcgen05 MMAs with TMEM accumulators, TMA tile loads,
// warp-specialised, persistent over work units.
//
// Algorithm (TileLang test_tilelang_kernel_mha_bwd.py, flashattn_fwd): online
// softmax over key tiles in base 2 (scale * log2 e folded into the exponent),
// the causal / window range of key tiles only, with an element mask on the
// tiles a mask cuts.  Differences from that page: LSE is returned in natural
// log (the FlashAttention convention the backward API takes), masks are
// bottom-right aligned (key j allowed for query i iff j <= i + Sk - Sq, plus a
// left window side), GQA, varlen, used lengths and a logit cap are handled, and
// rows with no allowed key give O = 0, LSE = +inf.
//
// One work unit = (query tile m of BM = 128 rows, query head h, sequence b).
// For each key tile n of BN = 128 keys in the unit's range:
//   S = Q K_n^T                     (TMEM fp32, one of three S buffers)
//   P = exp2(S * scale * log2 e - m_ref)     (bf16/fp16, written over S)
//   O += P V_n                      (TMEM fp32; A = P from TMEM, B = V in smem)
// The reference maximum m_ref of a row only moves when the row's running
// maximum exceeds it by more than 2^8 (then O and the row sum are rescaled);
// otherwise P is at most 2^8 and O, the row sum and the LSE stay consistent
// with the stale reference, so the result is the same softmax.
//
// Warp roles (256 threads): warp 0 TMA producer (Q and K), warp 3 V producer,
// warp 1 issues S = Q K^T, warp 2 allocates TMEM and issues O += P V (one
// thread each), warps 4-7 softmax and epilogue (thread = query row = TMEM
// lane).  S runs up to two tiles ahead of the softmax (three S buffers), so
// the tensor pipe computes S of the next tile while the softmax warps work on
// the current one.  (At D = 192 and 256 the same roles work on the chunk rings.)
//
// TMEM columns (512 allocated): S buffers [0,128), [128,256), [256,384);
// O [384, 384 + D).  Shared memory: 2 Q stages, 3 K stages, 2 V stages.
// Head dimensions above 128 run on D = 192 tiles up to 192, D = 256 tiles above
// (extra columns zero): O takes TMEM [256,256+D) next to two S buffers, the
// unit's Q tile (48 or 64 KiB) stays in shared memory, and K and V stream
// through rings of 64-column chunks (six for K; three or four, one tile, for V),
// filled by the two producer threads in their consumers' order.
#include <atomic>

#include "common.cuh"

namespace attn {

namespace {

constexpr int FBM = 128;  // query tile
constexpr int FBN = 128;  // key tile
constexpr int kFThreads = 256;
constexpr int kQSt = 2, kKSt = 3, kVSt = 2;
constexpr uint32_t kFChunk = 128 * 128;  // one 64-column (128-byte) slice of a 128-row tile
constexpr uint32_t kFTmemCols = 512;
constexpr uint32_t TF_S = 0;
// D = 192 and 256: K and V stream through rings of 64-column chunks (K: four
// resp. six slots, measured best of 4 and 6 at each width; V: one tile, three
// resp. four slots, so a tile's chunk pairs never wrap)
constexpr int kFKRingMax = 6, kFVRingMax = 4;

// Per head-dimension layout: three S buffers and O at column 384 up to D = 128;
// two S buffers and O at column 256 for the D = 192 and 256 tiles.
template <int D>
struct FCfg {
  static constexpr bool kWide = D > 128;
  static constexpr int kSBufs = kWide ? 2 : 3;
  static constexpr uint32_t kO = kWide ? 256 : 384;
  static constexpr int kVRing = D == 192 ? 3 : 4;
  static constexpr int kKRing = D == 192 ? 4 : 6;
};
constexpr float kRescaleLog2 = 8.f;  // P stays below 2^8 between rescales

enum FBar : uint32_t {
  F_QFULL = 0,
  F_QEMPTY = F_QFULL + kQSt,
  F_KFULL = F_QEMPTY + kQSt,    // K and V stages are released by SFULL / PVDONE
  F_VFULL = F_KFULL + kKSt,
  F_SFULL = F_VFULL + kVSt,     // per S buffer (up to 3): S computed
  F_PREADY = F_SFULL + 3,       // per S buffer: P written over it (4 softmax warps)
  F_PVDONE = F_PREADY + 3,      // per S buffer: O += P V has read it
  F_OFULL = F_PVDONE + 3,       // the unit's last O += P V done
  F_FINAL,
  F_FINAL2,                     // the O += P V issuer's own drain before TMEM is released
  F_RFULL,                      // D > 128: K ring slots, then V ring slots (released by SFULL / PVDONE)
  F_COUNT = F_RFULL + kFKRingMax + kFVRingMax
};

template <int D>
struct FSmem {
  // 64-column chunks of a tile row (D = 96: two, the second zero-filled past D)
  static constexpr uint32_t kTile = ((D + 63) / 64) * kFChunk;
  static constexpr uint32_t kQ = 0;
  // up to D = 128: Q, K and V tile stages; above: one Q tile, the K and V chunk rings
  static constexpr uint32_t kK = kQ + (FCfg<D>::kWide ? 1 : kQSt) * kTile;
  static constexpr uint32_t kV = kK + (FCfg<D>::kWide ? FCfg<D>::kKRing * kFChunk : kKSt * kTile);
  static constexpr uint32_t kBar =
      kV + (FCfg<D>::kWide ? FCfg<D>::kVRing * kFChunk : kVSt * kTile);
  static constexpr uint32_t kTmemSlot = kBar + F_COUNT * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kTotal = kAbort + 4;
};
static_assert(FSmem<128>::kTotal <= 232448, "shared memory budget");
static_assert(FSmem<256>::kTotal <= 232448, "shared memory budget (D = 256)");
static_assert(FSmem<192>::kTotal <= 232448, "shared memory budget (D = 192)");
static_assert(FSmem<96>::kTotal == FSmem<128>::kTotal, "D = 96 uses the D = 128 layout");

struct FUnit {
  int m, h, b;
  SeqInfo si;
  bool active;         // the query tile holds rows of the sequence
  int n_start, n_end;  // key tiles [n_start, n_end) seen by some query of the tile
};

// Unit u -> (query tile m, sequence b, head h): query tiles from the last to the
// first (causal units are longest first), heads fastest so that CTAs running at
// the same time share the K/V tiles of a group in L2.  Query-tile major over all
// sequences, or with kSeqMajor (packed batches without a logit cap, a kernel
// instance of its own) sequence major: with many packed sequences, query-tile
// major spreads the running CTAs over every (sequence, head) and each streams
// its own K/V from DRAM (16 sequences of up to 8192 x 16 heads: 7.35 GB read per
// launch, 60 % of the DRAM peak).
template <bool kSeqMajor>
__device__ __forceinline__ FUnit fwd_unit(const FwdParams& p, int u, int n_mt) {
  FUnit r;
  int mr;
  if constexpr (kSeqMajor) {
    const int per_b = n_mt * p.h_q;
    r.b = u / per_b;
    const int rem = u - r.b * per_b;
    mr = rem / p.h_q;
    r.h = rem - mr * p.h_q;
  } else {
    const int per_m = p.seq.batch * p.h_q;
    mr = u / per_m;
    const int rem = u - mr * per_m;
    r.b = rem / p.h_q;
    r.h = rem - r.b * p.h_q;
  }
  r.m = n_mt - 1 - mr;
  r.si = seq_info(p.seq, r.b);
  const int m0 = r.m * FBM;
  r.active = m0 < r.si.sq;
  r.n_start = r.n_end = 0;
  if (!r.active) return r;
  const int off = r.si.sk - r.si.sq;
  r.n_start = window_first_key(m0, r.si.sq, r.si.sk, p.win_left) / FBN;
  int n_end = ceil_div(r.si.sk, FBN);
  if (p.win_right >= 0) {
    const int last_key = min(m0 + FBM, r.si.sq) - 1 + off + p.win_right;
    n_end = min(n_end, last_key < 0 ? 0 : last_key / FBN + 1);
  }
  r.n_end = max(n_end, r.n_start);
  return r;
}

template <typename T, int D, bool kCap, bool kSeqMajor>
__global__ void __launch_bounds__(kFThreads, 1)
    fwd_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using L = FSmem<D>;
  constexpr bool kWide = FCfg<D>::kWide;
  constexpr int kSBufs = FCfg<D>::kSBufs;
  constexpr uint32_t TF_O = FCfg<D>::kO;
  constexpr int kFVRing = FCfg<D>::kVRing;
  constexpr int kFKRing = FCfg<D>::kKRing;
  constexpr int kDC = (D + 63) / 64;  // 64-column chunks of a tile row
  extern __shared__ __align__(1024) unsigned char smem[];
  if (p.input_bad != nullptr && *p.input_bad) return;
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, 0xA2100000u);
    return;
  }
  auto bar = [&](uint32_t i) -> uint32_t { return sb + L::kBar + i * 8; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const int G = p.h_q / p.h_k;
  const bool varlen = p.seq.cu_q != nullptr;
  const int n_mt = ceil_div(p.max_seqlen_q, FBM);
  const int num_units = n_mt * p.seq.batch * p.h_q;
  constexpr int kIsBf16 = Pack<T>::kIsBf16;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kQSt; ++s) {
      mbar_init(bar(F_QFULL + s), 1);
      mbar_init(bar(F_QEMPTY + s), 1);
    }
    for (int s = 0; s < kKSt; ++s) mbar_init(bar(F_KFULL + s), 1);
    for (int s = 0; s < kVSt; ++s) mbar_init(bar(F_VFULL + s), 1);
    for (int s = 0; s < kSBufs; ++s) {
      mbar_init(bar(F_SFULL + s), 1);
      mbar_init(bar(F_PREADY + s), 4);
      mbar_init(bar(F_PVDONE + s), 1);
    }
    mbar_init(bar(F_OFULL), 1);
    mbar_init(bar(F_FINAL), 1);
    mbar_init(bar(F_FINAL2), 1);
    for (int r = 0; r < kFKRingMax + kFVRingMax; ++r) mbar_init(bar(F_RFULL + r), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(sb + L::kTmemSlot, kFTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    // D > 128: warps 0 and 3 fill the K and V chunk rings.  Up to D = 128:
    // warp 0 loads Q and K, warp 3 loads V, so that a K load never waits behind
    // the release of a V stage (which comes one tile later, after O += P V).
    if (lane == 0 && kWide) {
      const bool loads_v = warp == 3;
      prefetch_tmap(loads_v ? &tmV : &tmQ);
      if (!loads_v) prefetch_tmap(&tmK);
      uint32_t qc = 0, q = 0;  // Q tiles and chunks (K or V) whose loads were issued
      const int ring = loads_v ? kFVRing : kFKRing;
      const uint32_t base = loads_v ? L::kV : L::kK;
      const uint32_t fbar = loads_v ? F_RFULL + kFKRingMax : F_RFULL;
      bool stop = false;
      for (int u = blockIdx.x; u < num_units && !stop; u += gridDim.x) {
        const FUnit un = fwd_unit<kSeqMajor>(p, u, n_mt);
        if (!un.active || un.n_end == un.n_start) continue;
        const int bq = varlen ? 0 : un.b;
        const int hk = un.h / G;
        if (!loads_v) {
          if (qc > 0 && !wait1(bar(F_QEMPTY), (qc - 1) & 1, ctl, 0xA2000001u)) break;
          mbar_expect_tx(bar(F_QFULL), L::kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sb + L::kQ + c * kFChunk, &tmQ, bar(F_QFULL), c * 64,
                        un.si.q_start + un.m * FBM, un.h, bq);
          ++qc;
        }
        for (int n = un.n_start; n < un.n_end && !stop; ++n) {
          const int krow = un.si.k_start + n * FBN;
          for (int c = 0; c < D / 64; ++c, ++q) {
            const uint32_t r = q % ring;
            if (q >= static_cast<uint32_t>(ring)) {
              // the slot's previous chunk belonged to tile tp: free once S (K) or
              // O += P V (V) of that tile is done.  Neither barrier can have moved
              // on by a further phase: that would need chunks not yet loaded.
              const uint32_t tp = (q - ring) / (D / 64);
              const uint32_t rel = loads_v ? F_PVDONE : F_SFULL;
              if (!wait1(bar(rel + tp % kSBufs), (tp / kSBufs) & 1, ctl, 0xA2000002u)) {
                stop = true;
                break;
              }
            }
            mbar_expect_tx(bar(fbar + r), kFChunk);
            tma_load_4d(sb + base + r * kFChunk, loads_v ? &tmV : &tmK, bar(fbar + r), c * 64,
                        krow, hk, bq);
          }
        }
        if (*abort_flag) break;
      }
      // Before exit, wait (bounded, ignoring the abort flag) for the copies that may
      // still be in flight: the last Q tile and the last issue into each ring slot.
      if (qc > 0) wait1(bar(F_QFULL), (qc - 1) & 1, ctl, 0xA2000004u, false);
      for (uint32_t i = q > static_cast<uint32_t>(ring) ? q - ring : 0; i < q; ++i)
        wait1(bar(fbar + i % ring), (i / ring) & 1, ctl, 0xA2000005u, false);
    } else if (lane == 0 && !kWide) {
      const bool loads_v = warp == 3;
      prefetch_tmap(loads_v ? &tmV : &tmQ);
      if (!loads_v) prefetch_tmap(&tmK);
      uint32_t qc = 0, kc = 0, vc = 0;  // Q, K and V tiles whose loads were issued
      bool stop = false;
      for (int u = blockIdx.x; u < num_units && !stop; u += gridDim.x) {
        const FUnit un = fwd_unit<kSeqMajor>(p, u, n_mt);
        if (!un.active || un.n_end == un.n_start) continue;
        const int bq = varlen ? 0 : un.b;
        const int hk = un.h / G;
        if (!loads_v) {
          const uint32_t s = qc % kQSt, use = qc / kQSt;
          if (use > 0 && !wait1(bar(F_QEMPTY + s), (use - 1) & 1, ctl, 0xA2000001u)) break;
          mbar_expect_tx(bar(F_QFULL + s), L::kTile);
#pragma unroll
          for (int c = 0; c < kDC; ++c)
            tma_load_4d(sb + L::kQ + s * L::kTile + c * kFChunk, &tmQ, bar(F_QFULL + s), c * 64,
                        un.si.q_start + un.m * FBM, un.h, bq);
          ++qc;
        }
        for (int n = un.n_start; n < un.n_end; ++n) {
          const int krow = un.si.k_start + n * FBN;
          if (loads_v) {
            // V stage vc % kVSt last held V of tile vc - kVSt: free once that tile's
            // O += P V is done (the MMA thread's PVDONE of its S buffer; K/V tile and
            // S tile counters coincide).  That barrier cannot have moved on by a
            // further phase: that would need the V this thread has not loaded yet.
            const uint32_t vs = vc % kVSt;
            if (vc >= static_cast<uint32_t>(kVSt)) {
              const uint32_t pt = vc - kVSt;
              if (!wait1(bar(F_PVDONE + pt % kSBufs), (pt / kSBufs) & 1, ctl, 0xA2000003u)) {
                stop = true;
                break;
              }
            }
            mbar_expect_tx(bar(F_VFULL + vs), L::kTile);
#pragma unroll
            for (int c = 0; c < kDC; ++c)
              tma_load_4d(sb + L::kV + vs * L::kTile + c * kFChunk, &tmV, bar(F_VFULL + vs),
                          c * 64, krow, hk, bq);
            ++vc;
            continue;
          }
          // K stage kc % kKSt (= S buffer kc % kSBufs) last held K of tile kc - kKSt:
          // free once that tile's S is done (its SFULL), which cannot have moved on
          // by a further phase before this K is loaded.
          static_assert(kKSt == 3 && FCfg<128>::kSBufs == 3, "K stages follow the S buffers");
          const uint32_t ks = kc % kKSt;
          if (kc >= static_cast<uint32_t>(kKSt) &&
              !wait1(bar(F_SFULL + ks), ((kc - kKSt) / kKSt) & 1, ctl, 0xA2000002u)) {
            stop = true;
            break;
          }
          mbar_expect_tx(bar(F_KFULL + ks), L::kTile);
#pragma unroll
          for (int c = 0; c < kDC; ++c)
            tma_load_4d(sb + L::kK + ks * L::kTile + c * kFChunk, &tmK, bar(F_KFULL + ks), c * 64,
                        krow, hk, bq);
          ++kc;
        }
        if (*abort_flag) break;
      }
      // Before exit, wait (bounded, ignoring the abort flag) until every copy this
      // thread issued has landed, so no TMA write targets a finished CTA.  Only the
      // last issue into each stage can be outstanding: an earlier one was consumed
      // (its stage released) before the stage was refilled.
      for (uint32_t i = qc > kQSt ? qc - kQSt : 0; i < qc; ++i)
        wait1(bar(F_QFULL + i % kQSt), (i / kQSt) & 1, ctl, 0xA2000004u, false);
      for (uint32_t i = kc > kKSt ? kc - kKSt : 0; i < kc; ++i)
        wait1(bar(F_KFULL + i % kKSt), (i / kKSt) & 1, ctl, 0xA2000005u, false);
      for (uint32_t i = vc > kVSt ? vc - kVSt : 0; i < vc; ++i)
        wait1(bar(F_VFULL + i % kVSt), (i / kVSt) & 1, ctl, 0xA2000006u, false);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && kWide) {
      // D > 128: S = Q K^T from the unit's Q tile and the K ring
      constexpr uint32_t kIdS = idesc_f16(kIsBf16, 0, 0, FBM, FBN);  // Q, K both K-major
      uint32_t qc = 0, it = 0, q = 0;  // Q tiles, S tiles, K ring chunks consumed
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const FUnit un = fwd_unit<kSeqMajor>(p, u, n_mt);
        if (!un.active || un.n_end == un.n_start) continue;
        const int nt = un.n_end - un.n_start;
        if (!wait1(bar(F_QFULL), qc & 1, ctl, 0xA2000013u)) goto mma_exit_w;
        for (int j = 0; j < nt; ++j) {
          const uint32_t t = it + j, buf = t % kSBufs;
          // S buffer `buf` last held tile t - 2, whose O += P V must have read its P
          if (t >= kSBufs &&
              !wait1(bar(F_PVDONE + buf), ((t - kSBufs) / kSBufs) & 1, ctl, 0xA2000014u))
            goto mma_exit_w;
          for (int c = 0; c < D / 64; ++c, ++q) {
            if (!wait1(bar(F_RFULL + q % kFKRing), (q / kFKRing) & 1, ctl, 0xA2000016u))
              goto mma_exit_w;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + TF_S + buf * 128, sdesc_sw128(sb + L::kQ + c * kFChunk + kk * 32, 16, 1024),
                     sdesc_sw128(sb + L::kK + (q % kFKRing) * kFChunk + kk * 32, 16, 1024), kIdS,
                     (c > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(F_SFULL + buf));  // also frees the tile's K ring slots
          if (j == nt - 1) tc_commit(bar(F_QEMPTY));
        }
        it += nt;
        ++qc;
      }
    mma_exit_w:
      // make sure no MMA is still running before TMEM is released
      tc_commit(bar(F_FINAL));
      wait1(bar(F_FINAL), 0, ctl, 0xA200001Fu, false);
    } else if (lane == 0 && !kWide) {
      // Up to D = 128 this thread issues the S = Q K^T products and warp 2 the
      // O += P V products: each tcgen05.mma blocks its issuing thread for about
      // its own execution time, so with one issuer every wait and commit between
      // the two kinds of product left the tensor pipe idle.  The barriers order
      // what the two threads share: S of tile t waits for O += P V of tile t - 3
      // (the S buffer's previous P), O += P V of tile t for P of tile t.
      constexpr uint32_t kIdS = idesc_f16(kIsBf16, 0, 0, FBM, FBN);  // Q, K both K-major
      uint32_t qc = 0, it = 0;  // Q tiles, S tiles
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const FUnit un = fwd_unit<kSeqMajor>(p, u, n_mt);
        if (!un.active || un.n_end == un.n_start) continue;
        const int nt = un.n_end - un.n_start;
        const uint32_t qs = qc % kQSt;
        if (!wait1(bar(F_QFULL + qs), (qc / kQSt) & 1, ctl, 0xA2000013u)) goto s_exit;
        const uint32_t sQ = sb + L::kQ + qs * L::kTile;
        for (int j = 0; j < nt; ++j) {
          const uint32_t t = it + j;
          const uint32_t buf = t % kSBufs, ks = t % kKSt;  // K/V and S tile counters coincide
          // S buffer `buf` last held tile t - 3, whose O += P V must have read its P
          if (t >= kSBufs &&
              !wait1(bar(F_PVDONE + buf), ((t - kSBufs) / kSBufs) & 1, ctl, 0xA2000014u))
            goto s_exit;
          if (!wait1(bar(F_KFULL + ks), (t / kKSt) & 1, ctl, 0xA2000015u)) goto s_exit;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kFChunk + (kk & 3) * 32;
            mma_ss(tmem + TF_S + buf * 128, sdesc_sw128(sQ + koff, 16, 1024),
                   sdesc_sw128(sb + L::kK + ks * L::kTile + koff, 16, 1024), kIdS, kk > 0);
          }
          tc_commit(bar(F_SFULL + buf));  // also frees K stage ks for the producer
          if (j == nt - 1) tc_commit(bar(F_QEMPTY + qs));
        }
        it += nt;
        ++qc;
      }
    s_exit:
      // make sure no MMA is still running before TMEM is released
      tc_commit(bar(F_FINAL));
      wait1(bar(F_FINAL), 0, ctl, 0xA200001Fu, false);
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ---------------------------------------------------- O += P V issuer
      // (D = 192 and 256: O in N = 128 parts over V chunk pairs from the V ring,
      // the odd last chunk at D = 192 as an N = 64 part)
      constexpr uint32_t kIdPV =
          idesc_f16(kIsBf16, 0, 1, FBM, kWide ? 128 : D);  // P from TMEM, V MN-major
      constexpr uint32_t kIdPV64 = idesc_f16(kIsBf16, 0, 1, FBM, 64);
      uint32_t it = 0, q = 0;  // P tiles; D > 128: V ring chunks consumed
      for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
        const FUnit un = fwd_unit<kSeqMajor>(p, u, n_mt);
        if (!un.active || un.n_end == un.n_start) continue;
        const int nt = un.n_end - un.n_start;
        for (int j = 0; j < nt; ++j) {
          const uint32_t t = it + j;
          const uint32_t buf = t % kSBufs, vs = t % kVSt;
          if (!wait1(bar(F_PREADY + buf), (t / kSBufs) & 1, ctl, 0xA2000011u)) goto pv_exit;
          if (kWide) {
#pragma unroll 1
            for (int pr = 0; pr < (D / 64 + 1) / 2; ++pr) {
              const bool pair = 2 * pr + 1 < D / 64;
              const uint32_t r0 = kFKRingMax + q % kFVRing;
              if (!wait1(bar(F_RFULL + r0), (q / kFVRing) & 1, ctl, 0xA2000012u) ||
                  (pair &&
                   !wait1(bar(F_RFULL + r0 + 1), ((q + 1) / kFVRing) & 1, ctl, 0xA2000012u)))
                goto pv_exit;
              tc_fence_after();
              const uint32_t sV = sb + L::kV + (q % kFVRing) * kFChunk;
#pragma unroll
              for (int kk = 0; kk < FBN / 16; ++kk)
                mma_ts(tmem + TF_O + 128 * pr, tmem + TF_S + buf * 128 + kk * 8,
                       sdesc_sw128(sV + kk * 2048, kFChunk, 1024), pair ? kIdPV : kIdPV64,
                       (j > 0 || kk > 0) ? 1u : 0u);
              q += pair ? 2 : 1;
            }
          } else {
            if (!wait1(bar(F_VFULL + vs), (t / kVSt) & 1, ctl, 0xA2000012u)) goto pv_exit;
            tc_fence_after();
            const uint32_t sV = sb + L::kV + vs * L::kTile;
#pragma unroll
            for (int kk = 0; kk < FBN / 16; ++kk)
              mma_ts(tmem + TF_O, tmem + TF_S + buf * 128 + kk * 8,
                     sdesc_sw128(sV + kk * 2048, kFChunk, 1024), kIdPV,
                     (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(F_PVDONE + buf));  // also frees the tile's V stage / V ring slots
        }
        tc_commit(bar(F_OFULL));
        it += nt;
      }
    pv_exit:
      tc_commit(bar(F_FINAL2));
      wait1(bar(F_FINAL2), 0, ctl, 0xA200002Fu, false);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------- softmax / epilogue
    const uint32_t quad = warp & 3;
    const int row = static_cast<int>(quad * 32 + lane);  // query row within the tile
    const uint32_t tl = tmem + ((quad * 32) << 16);     // this warp's TMEM lanes
    // logits in log2 units: x * mul with x the raw score (kCap: already in log2 units).
    // A nonpositive scale is multiplied in first, so the running maximum is taken
    // over the final logits either way.
    const bool pre_scale = !kCap && !(p.scale_log2 > 0.f);
    const float mul = (kCap || pre_scale) ? 1.f : p.scale_log2;
    uint32_t it = 0, uc = 0;
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      const FUnit un = fwd_unit<kSeqMajor>(p, u, n_mt);
      if (!un.active) continue;
      const int m0 = un.m * FBM;
      const int qi = m0 + row;  // query index within the sequence
      const bool row_ok = qi < un.si.sq;
      const int off = un.si.sk - un.si.sq;
      const int nt = un.n_end - un.n_start;
      float m_ref = -INFINITY, lsum = 0.f;
      for (int j = 0; j < nt; ++j, ++it) {
        const int n = un.n_start + j;
        const uint32_t buf = it % kSBufs;
        const uint32_t sbase = TF_S + buf * 128;
        const int k0 = n * FBN;
        const bool need_mask =
            (k0 + FBN > un.si.sk) ||
            (p.win_right >= 0 && k0 + FBN - 1 > m0 + off + p.win_right) ||
            (p.win_left >= 0 && k0 < m0 + FBM - 1 + off - p.win_left);
        // allowed keys of this row, in tile column coordinates: lo <= c < hi
        int lo = 0, hi = min(FBN, un.si.sk - k0);
        if (p.win_right >= 0) hi = min(hi, qi + off + p.win_right - k0 + 1);
        if (p.win_left >= 0) lo = max(0, qi + off - p.win_left - k0);
        if (!wait_warp(bar(F_SFULL + buf), (it / kSBufs) & 1, ctl, 0xA2000021u)) goto done;
        tc_fence_after();
        float x[FBN];
        {
          uint32_t sv[FBN];
#pragma unroll
          for (int c = 0; c < FBN / 32; ++c) tmem_ld32p(tl + sbase + 32 * c, sv + 32 * c);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < FBN; ++c) x[c] = __uint_as_float(sv[c]);
        }
        if (kCap) {
#pragma unroll
          for (int c = 0; c < FBN; ++c) x[c] = tanh_exp(x[c] * p.cap_in) * p.cap_out;
        } else if (pre_scale) {
#pragma unroll
          for (int c = 0; c < FBN; ++c) x[c] *= p.scale_log2;
        }
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < FBN; ++c) x[c] = (c >= lo && c < hi) ? x[c] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = x[e];
#pragma unroll
        for (int c = 8; c < FBN; ++c) mx[c & 7] = fmaxf(mx[c & 7], x[c]);
        const float tmax =
            fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                  fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * mul;
        // move the reference only when the maximum rose by more than 2^8
        const bool grow = tmax > m_ref + kRescaleLog2;  // false for tmax = -inf
        const bool had_ref = m_ref != -INFINITY;
        const float alpha = grow ? (had_ref ? ex2(m_ref - tmax) : 0.f) : 1.f;
        if (grow) m_ref = tmax;
        lsum *= alpha;
        // O holds earlier tiles' P V under the old reference: rescale it (rare)
        const bool rescale = grow && had_ref && j > 0;
        if (__any_sync(0xffffffffu, rescale)) {
          const uint32_t pt = it - 1;  // the previous tile's O += P V must have landed
          if (!wait_warp(bar(F_PVDONE + pt % kSBufs), (pt / kSBufs) & 1, ctl, 0xA2000022u))
            goto done;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tl + TF_O + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16(tl + TF_O + 32 * c, *reinterpret_cast<uint32_t(*)[16]>(o));
            tmem_st16(tl + TF_O + 32 * c + 16, *reinterpret_cast<uint32_t(*)[16]>(o + 16));
          }
          tmem_wait_st();
        }
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c16 = 0; c16 < FBN / 32; ++c16) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float p0 = ex2(fmaf(x[32 * c16 + 2 * e], mul, -m_use));
            const float p1 = ex2(fmaf(x[32 * c16 + 2 * e + 1], mul, -m_use));
            ls[e & 3] += p0 + p1;
            pk[e] = Pack<T>::two(p0, p1);
          }
          tmem_st16(tl + sbase + 16 * c16, pk);
        }
        lsum += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(F_PREADY + buf));
      }
      // ---- epilogue: O / l and the LSE of this row
      {
        T* orow = static_cast<T*>(const_cast<void*>(p.o.ptr)) + (varlen ? 0 : un.b * p.o.sb) +
                  static_cast<int64_t>(un.si.q_start + qi) * p.o.ss +
                  static_cast<int64_t>(un.h) * p.o.sh;
        const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
        if (nt > 0) {
          if (!wait_warp(bar(F_OFULL), uc & 1, ctl, 0xA2000023u)) goto done;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tl + TF_O + 32 * c, o);
            tmem_wait_ld();
            if (row_ok) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 v;
                v.x = Pack<T>::two(__uint_as_float(o[8 * q + 0]) * inv,
                                   __uint_as_float(o[8 * q + 1]) * inv);
                v.y = Pack<T>::two(__uint_as_float(o[8 * q + 2]) * inv,
                                   __uint_as_float(o[8 * q + 3]) * inv);
                v.z = Pack<T>::two(__uint_as_float(o[8 * q + 4]) * inv,
                                   __uint_as_float(o[8 * q + 5]) * inv);
                v.w = Pack<T>::two(__uint_as_float(o[8 * q + 6]) * inv,
                                   __uint_as_float(o[8 * q + 7]) * inv);
                if (32 * c + 8 * q < p.head_dim)  // a padded head dimension stops early
                  reinterpret_cast<uint4*>(orow + 32 * c)[q] = v;
              }
            }
          }
          tc_fence_before();
          ++uc;
        } else if (row_ok) {  // no key tile at all: O = 0
#pragma unroll
          for (int c = 0; c < D / 8; ++c)
            if (8 * c < p.head_dim) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
        }
        if (row_ok) {
          const int64_t li =
              varlen ? static_cast<int64_t>(un.h) * p.seq.seqlen_q + un.si.q_start + qi
                      : (static_cast<int64_t>(un.b) * p.h_q + un.h) * p.seq.seqlen_q + qi;
          // natural log: (m_ref + log2 l) * ln 2; a row without an allowed key: +inf
          p.lse[li] = lsum > 0.f ? (m_ref + __log2f(lsum)) * 0.6931471805599453f : INFINITY;
        }
      }
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kFTmemCols);
}

template <typename T, int D, bool kCap, bool kSeqMajor>
cudaError_t launch_fwd_t(const FwdParams& p, int dtype, cudaStream_t stream) {
  const bool varlen = p.seq.cu_q != nullptr;
  const int nb = varlen ? 1 : p.seq.batch;
  CUtensorMap tq, tk, tv;
  // the maps span the logical head dimension: columns up to D read as zero
  const int d = p.head_dim;
  if (!encode_tmap_bshd(&tq, p.q, dtype, p.seq.seqlen_q, p.h_q, nb, d, FBM) ||
      !encode_tmap_bshd(&tk, p.k, dtype, p.seq.seqlen_k, p.h_k, nb, d, FBN) ||
      !encode_tmap_bshd(&tv, p.v, dtype, p.seq.seqlen_k, p.h_k, nb, d, FBN))
    return cudaErrorInvalidValue;
  // Every CTA allocates all 512 TMEM columns, so two CTAs on one SM would
  // serialise in the allocator: the launch reserves enough shared memory (the
  // D = 128 layout's) to keep one CTA per SM at any head dimension.
  constexpr uint32_t smem =
      FSmem<D>::kTotal > FSmem<128>::kTotal ? FSmem<D>::kTotal : FSmem<128>::kTotal;
  // Kernel attributes are per device: set them once on each.
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    const cudaError_t e = cudaFuncSetAttribute(fwd_kernel<T, D, kCap, kSeqMajor>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int units = ceil_div(p.max_seqlen_q, FBM) * p.seq.batch * p.h_q;
  if (units <= 0) return cudaSuccess;
  const int grid = units < num_sms() ? units : num_sms();
  fwd_kernel<T, D, kCap, kSeqMajor><<<grid, kFThreads, smem, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

template <bool kCap, bool kSeqMajor>
cudaError_t launch_fwd_cap(const FwdParams& p, int dtype, cudaStream_t stream) {
  // tiles of 64, 96, 128, 192 or 256 head-dim columns (the columns past D zero)
  const int dp = p.head_dim <= 64    ? 64
                 : p.head_dim <= 96  ? 96
                 : p.head_dim <= 128 ? 128
                 : p.head_dim <= 192 ? 192
                                     : 256;
  if (dtype == 1)
    return dp == 64    ? launch_fwd_t<__nv_bfloat16, 64, kCap, kSeqMajor>(p, dtype, stream)
           : dp == 96  ? launch_fwd_t<__nv_bfloat16, 96, kCap, kSeqMajor>(p, dtype, stream)
           : dp == 128 ? launch_fwd_t<__nv_bfloat16, 128, kCap, kSeqMajor>(p, dtype, stream)
           : dp == 192 ? launch_fwd_t<__nv_bfloat16, 192, kCap, kSeqMajor>(p, dtype, stream)
                       : launch_fwd_t<__nv_bfloat16, 256, kCap, kSeqMajor>(p, dtype, stream);
  return dp == 64    ? launch_fwd_t<__half, 64, kCap, kSeqMajor>(p, dtype, stream)
         : dp == 96  ? launch_fwd_t<__half, 96, kCap, kSeqMajor>(p, dtype, stream)
         : dp == 128 ? launch_fwd_t<__half, 128, kCap, kSeqMajor>(p, dtype, stream)
         : dp == 192 ? launch_fwd_t<__half, 192, kCap, kSeqMajor>(p, dtype, stream)
                     : launch_fwd_t<__half, 256, kCap, kSeqMajor>(p, dtype, stream);
}

}  // namespace

cudaError_t launch_fwd(const FwdParams& p, int dtype, cudaStream_t stream) {
  if (p.softcap > 0.f) return launch_fwd_cap<true, false>(p, dtype, stream);
  // packed sequences: the sequence-major unit order (see fwd_unit)
  return p.seq.cu_q != nullptr ? launch_fwd_cap<false, true>(p, dtype, stream)
                               : launch_fwd_cap<false, false>(p, dtype, stream);
}

}  // namespace attn
