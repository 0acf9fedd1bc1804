// Main attention-backward kernel for sm_103a: tcgen05 MMAs with TMEM
// accumulators, TMA tile loads, warp-specialised, persistent over work units.
//
// Algorithm (TileLang test_tilelang_kernel_mha_bwd.py, flashattn_bwd): KV
// stationary.  One work unit = (KV tile n of BN=128 keys, kv head g, sequence
// b).  K_n and V_n are loaded once; for each of the G query heads of the
// group and each query tile m of BM=128 rows that sees key tile n (all of them,
// or the causal / local-window range, bottom-right aligned):
//   S^T  = K_n Q_m^T                        (TMEM, fp32)
//   P^T  = exp2(S^T * scale * log2 e - LSE2[query]), masked  (bf16/fp16, TMEM)
//          (with a logit cap c: exp2(c tanh(S^T scale / c) log2 e - LSE2))
//   dP^T = V_n dO_m^T                       (TMEM, fp32)
//   dV  += P^T dO_m                         (TMEM accumulator, A operand from TMEM)
//   dS^T = P^T * (dP^T - Delta[query])      (smem, bf16/fp16; times 1 - tanh^2 with a cap)
//   dK  += dS^T Q_m                         (TMEM accumulator, A operand from smem)
//   dQ_m = dS K_n -> reduced into the fp32 dQaccum in global memory
// dK (times scale) and dV are written once per unit; dK/dV of a GQA group are
// summed in TMEM over the group's query heads (the group sum of
// flash-attention csrc/flash_attn_ck/mha_bwd.cpp, done without extra memory).
// dQaccum is reduced with TMA tensor reduce-adds (fp32), or, in deterministic
// mode, in ascending KV-tile order behind per-(head, query tile, 32-row quarter)
// semaphores (the dq_semaphore of flash-attention
// hopper/flash_bwd_launch_template.h).
// D is 64, 96 or 128 here (96: the D = 128 shared-memory layout, whose second
// 64-column chunk the TMA loads zero-fill past column 96, with 6 instead of 8
// head-dim steps for S^T and dP^T and N = 96 products for dV, dK and dQ);
// other head dims (multiples of 8) run zero-padded to the next of those.
// Template switches: kCap (logit cap), kLeft (a left window side); the default
// instantiation has neither.
//
// Warp roles (768 threads = 6 warpgroups): warp 0 TMA producer, warp 1 MMA
// issuer (one thread), warp 2 TMEM allocator, warps 4-19 softmax / dS / dK-dV
// epilogue (four warps per TMEM lane quadrant: thread = key row, warp group g =
// (warp - 4) / 4 takes query columns [32 g, 32 g + 32)), warps 20-23 dQ drain
// (thread = query row).  A compile-time switch keeps the 8-softmax-warp form
// (512 threads, 64 columns per warp).
//
// TMEM columns (512 allocated, 128 lanes):
//   [  0,128) S^T fp32; each column group keeps its packed P^T in the first half
//             of the S^T columns it has read itself
//   [128,256) dP^T fp32, then dQ in [128,128+D)
//   [256,256+D) dK, [384,384+D) dV; at D = 64 a second pair at [320,384) and
//   [448,512) for every other unit
// dS^T goes to a swizzled shared-memory tile read by both the dQ and dK MMAs.
// The tensor pipe runs dP, dV, then the next tile's S (as soon as dV and the
// dS phase have read P^T), then dQ and dK; dP of the next tile waits for the dQ
// drain to have read dQ out of TMEM.  At D = 64 the K/V tiles and dK/dV are
// double-buffered across units, so the next unit's K/V load during this one
// and the last tile of a unit issues the next unit's first S like any other.
// Every mbarrier wait is bounded (see WaitCtl): on timeout the kernel records
// the site in the status word and unwinds.
#include <atomic>

#include "bwd_units.cuh"
#include "common.cuh"

namespace attn {

namespace {

constexpr int BM = 128;  // query tile
constexpr int BN = 128;  // key tile
#ifndef ATTN_SOFTMAX_WARPS
#define ATTN_SOFTMAX_WARPS 16
#endif
constexpr int kSoftmaxWarps = ATTN_SOFTMAX_WARPS;  // 8 or 16: 2 or 4 column groups per lane quadrant
constexpr int kGroups = kSoftmaxWarps / 4;         // query-column groups of the softmax warps
constexpr int kCols = 128 / kGroups;               // query columns per softmax warp
constexpr int kThreads = 32 * (4 + kSoftmaxWarps + 4);
static_assert(kSoftmaxWarps == 8 || kSoftmaxWarps == 16, "softmax warps");
// Per-thread registers of the warpgroups after the split done at kernel entry:
// warpgroup 0 (producer, MMA issuer, allocator), the softmax warpgroups (which
// keep their launch count) and the dQ drain warpgroup.  An increase that the
// launch allocation cannot cover would wait forever, so the host checks the
// kernel's launch register count against kRegLaunch before every launch.
constexpr uint32_t kRegLaunch = kSoftmaxWarps == 8 ? 128 : 80;
constexpr uint32_t kRegWg0 = kSoftmaxWarps == 8 ? 80 : 64;
constexpr uint32_t kRegDrain = kSoftmaxWarps == 8 ? 176 : 96;
static_assert(kRegWg0 * 128 + kRegLaunch * 32 * kSoftmaxWarps + kRegDrain * 128 ==
                  kRegLaunch * kThreads,
              "register split must use exactly the launch allocation");
constexpr int kStages = 2;
constexpr uint32_t kChunk = 128 * 128;  // one 64-column (128-byte) slice of a 128-row tile
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TM_S = 0, TM_P = 0, TM_DP = 128;  // P^T: + 64 per query half
constexpr uint32_t TM_DQ = 128, TM_DK = 256, TM_DV = 384;

enum Bar : uint32_t {
  B_FULLQ = 0,
  B_FULLDO = B_FULLQ + kStages,
  B_EMPTY = B_FULLDO + kStages,    // Q stage (+ LSE2) free: dK done (committed after the
                                   // softmax's DSREADY, so LSE2 has been read too)
  B_EMPTYDO = B_EMPTY + kStages,   // dO stage (+ Delta) free: dV done and the dQ drain, which
                                   // stages its reduce-adds there, done with it (the drain
                                   // starts after dQ, i.e. after the softmax read Delta)
  B_KVFULL = B_EMPTYDO + kStages,
  B_KVEMPTY,
  B_SFULL,
  B_DPFULL,
  B_PREADY,
  B_PVDONE,                        // dV done: P^T in TMEM no longer read by the tensor pipe
  B_PREAD,                         // the dS phase has read P^T from TMEM
  B_DSREADY,
  B_DQFULL,
  B_DQFREE,
  B_DKDONE,
  B_DKDVFULL,
  B_DKDVFREE,
  B_UNITFULL,                      // 2 slots: next work unit published by the producer
  B_UNITEMPTY = B_UNITFULL + 2,    // 2 slots: every consumer role has read it
  B_FINAL = B_UNITEMPTY + 2,
  B_FULLQ2,                        // 2 slots: second head-dim chunk of the Q tile (D = 128)
  B_KVFULL1 = B_FULLQ2 + kStages,  // second K/V slot and dK/dV buffer (D = 64)
  B_KVEMPTY1,
  B_DKDVFULL1,
  B_DKDVFREE1,
  B_COUNT
};

template <int D>
struct Smem {
  static constexpr uint32_t kTile = ((D + 63) / 64) * kChunk;  // 64-column chunks (D = 96: 2)
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kK + kTile;
  static constexpr uint32_t kQ = kV + kTile;
  static constexpr uint32_t kDO = kQ + kStages * kTile;
  static constexpr uint32_t kDS = kDO + kStages * kTile;  // dS^T [BN keys][BM queries], 2 chunks
  static constexpr uint32_t kLSE = kDS + 2 * kChunk;
  static constexpr uint32_t kDelta = kLSE + kStages * BM * 4;
  static constexpr uint32_t kBar = kDelta + kStages * BM * 4;
  static constexpr uint32_t kRing = kBar + B_COUNT * 8;  // 2 x int32 unit ring
  static constexpr uint32_t kTmemSlot = kRing + 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  // D = 64: a second K/V slot, so that the next unit's K/V load while this unit
  // runs (its dK/dV accumulate in a second TMEM range meanwhile)
  static constexpr uint32_t kKVSlots = D == 64 ? 2 : 1;
  static constexpr uint32_t kK1 = (kAbort + 4 + 1023) / 1024 * 1024;
  static constexpr uint32_t kV1 = kK1 + kTile;
  // D = 64: the dQ drain warps also write dK/dV, staged here as 32-row boxes
  static constexpr uint32_t kEpi = kV1 + kTile;
  static constexpr uint32_t kTotal = kKVSlots == 2 ? kEpi + 2 * 128 * D * 2 : kAbort + 4;
};
static_assert(Smem<128>::kTotal <= 232448, "shared memory budget");
static_assert(Smem<64>::kTotal <= 232448, "shared memory budget");
static_assert(Smem<96>::kTotal == Smem<128>::kTotal, "D = 96 uses the D = 128 layout");

template <typename T, int D, bool kCap, bool kLeft>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ,
                    const __grid_constant__ CUtensorMap tmDK,
                    const __grid_constant__ CUtensorMap tmDV) {
  using L = Smem<D>;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (p.input_bad != nullptr && *p.input_bad) return;
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, 0xA1100000u);
    return;
  }
  auto bar = [&](uint32_t i) -> uint32_t { return sb + L::kBar + i * 8; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const int G = p.h_q / p.h_k;
  const bool varlen = p.seq.cu_q != nullptr;
  const int n_tiles = ceil_div(p.max_seqlen_k, BN);
  const int num_units = n_tiles * p.seq.batch * p.h_k;
  constexpr int kIsBf16 = Pack<T>::kIsBf16;
  constexpr int kDC = (D + 63) / 64;  // 64-column chunks of a tile row (the last one zero-filled
                                      // past D by the TMA loads at D = 96)
  constexpr bool kSplitQ = kDC == 2;
  // Who writes a unit's dK/dV: the softmax warps, or the dQ drain warps once the
  // unit's last tile is drained (so the softmax warps go straight on to the next
  // unit): with two K/V slots (D = 64), and in the left-window instantiation
  // without a logit cap (its units are short: +0.8 %; the default and the
  // logit-cap instantiations measured 0 and -3 % that way)
  constexpr bool kDrainEpi = L::kKVSlots == 2 || (kLeft && !kCap);
  // the left side of a local window; without one (the usual case) a constant,
  // so the unmasked and causal schedules carry none of its arithmetic
  const int wleft = kLeft ? p.win_left : -1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_FULLQ + s), 1);
      mbar_init(bar(B_FULLQ2 + s), 1);
      mbar_init(bar(B_FULLDO + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);       // MMA commit
      mbar_init(bar(B_EMPTYDO + s), 1 + 4);  // MMA commit + the 4 dQ drain warps
    }
    mbar_init(bar(B_KVFULL), 1);
    mbar_init(bar(B_KVEMPTY), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_DPFULL), 1);
    mbar_init(bar(B_PREADY), kSoftmaxWarps);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_PREAD), kSoftmaxWarps);
    mbar_init(bar(B_DSREADY), kSoftmaxWarps);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQFREE), 4);
    mbar_init(bar(B_DKDONE), 1);
    mbar_init(bar(B_DKDVFULL), 1);
    // the dK/dV epilogue: the softmax warps, or the 4 dQ drain warps
    mbar_init(bar(B_DKDVFREE), kDrainEpi ? 4 : kSoftmaxWarps);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_UNITFULL + k), 1);
      mbar_init(bar(B_UNITEMPTY + k), 1 + kSoftmaxWarps + 4);  // MMA + softmax + drain warps
    }
    mbar_init(bar(B_FINAL), 1);
    if (L::kKVSlots == 2) {
      mbar_init(bar(B_KVFULL1), 1);
      mbar_init(bar(B_KVEMPTY1), 1);
      mbar_init(bar(B_DKDVFULL1), 1);
      mbar_init(bar(B_DKDVFREE1), 4);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(sb + L::kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
  // Register split.  With 8 softmax warps (512 threads, 128 registers each at
  // launch) warpgroup 0 (producer, MMA issuer, allocator) gives 48 up and the dQ
  // drain warpgroup takes them to hold a whole dQ row per thread:
  // 80 * 128 + 128 * 256 + 176 * 128 = 512 * 128.  With 16 (768 threads, 80 at
  // launch) warpgroup 0 gives 16 to the drain: 64 * 128 + 80 * 512 + 96 * 128 =
  // 768 * 80 (measured best of the splits that fit).
  constexpr bool kDrainWholeRow = kSoftmaxWarps == 8;  // else two 64-column passes
  volatile int* ring = reinterpret_cast<volatile int*>(smem + L::kRing);
  // Work units come from a persistent scheduler: the first unit of CTA c is c,
  // later ones are taken by the producer from a global counter in
  // unit order of get_unit (longest first) and published through a 2-slot ring
  // that every role reads.  A published index >= num_units means "done".
  // Consumer side (single thread when `warp_wide` is false):
  auto take_unit = [&](uint32_t k, bool warp_wide, int& u) -> bool {
    const uint32_t slot = k & 1;
    const bool ok = warp_wide ? wait_warp(bar(B_UNITFULL + slot), (k >> 1) & 1, ctl, 0xA0000041u)
                              : wait1(bar(B_UNITFULL + slot), (k >> 1) & 1, ctl, 0xA0000042u);
    if (!ok) return false;
    u = ring[slot];
    if (!warp_wide || lane_id() == 0) mbar_arrive(bar(B_UNITEMPTY + slot));
    return true;
  };
  if (warp < 4) {
    setmaxnreg_dec<kRegWg0>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      prefetch_tmap(&tmDO);
      prefetch_tmap(&tmDQ);
      // K/V tiles are read by this CTA only, once per unit: evicted first from L2,
      // which leaves room for the Q/dO tiles and dQ accumulator lines other CTAs
      // share (+0.3 to +0.7 % on every workload measured)
      const uint64_t kv_pol = l2_policy_evict_first();
      uint32_t it = 0, uc = 0;  // iterations and units whose loads were issued
      bool do_pending_skipped = false;  // last iteration issued Q but not dO
      int u = blockIdx.x;
      for (uint32_t k = 0;; ++k) {
        // publish unit k (slot k & 1 was read by every role for unit k - 2)
        if (k >= 2 && !wait1(bar(B_UNITEMPTY + (k & 1)), ((k >> 1) - 1) & 1, ctl, 0xA0000043u))
          break;
        ring[k & 1] = u;
        mbar_arrive(bar(B_UNITFULL + (k & 1)));
        if (u >= num_units) break;
        // fetch the next unit now; the atomic's latency overlaps this unit's loads
        const int u_next = static_cast<int>(gridDim.x) + atomicAdd(p.sched, 1);
        const Unit un = get_unit(p, u, G, wleft);
        u = u_next;
        if (un.n_iters == 0) continue;
        // unit uc takes K/V slot uc % kKVSlots, freed by the unit kKVSlots before it
        const uint32_t kvs = uc % L::kKVSlots, kvuse = uc / L::kKVSlots;
        if (kvuse > 0 &&
            !wait1(bar(kvs ? B_KVEMPTY1 : B_KVEMPTY), (kvuse - 1) & 1, ctl, 0xA0000001u))
          break;
        ++uc;
        {
          const int krow = un.si.k_start + un.n * BN;
          const int bk = varlen ? 0 : un.b;
          const uint32_t kvfull = bar(kvs ? B_KVFULL1 : B_KVFULL);
          const uint32_t sK = sb + (kvs ? L::kK1 : L::kK), sV = sb + (kvs ? L::kV1 : L::kV);
          mbar_expect_tx(kvfull, 2 * L::kTile);
#pragma unroll
          for (int c = 0; c < kDC; ++c) {
            tma_load_4d_hint(sK + c * kChunk, &tmK, kvfull, c * 64, krow, un.g, bk, kv_pol);
            tma_load_4d_hint(sV + c * kChunk, &tmV, kvfull, c * 64, krow, un.g, bk, kv_pol);
          }
        }
        for (int j = 0; j < un.n_iters; ++j, ++it) {
          const uint32_t s = it % kStages;
          const uint32_t use = it / kStages;
          int h, m;
          iter_hm(un, j, G, h, m);
          const int qrow = un.si.q_start + m * BM;
          const int bq = varlen ? 0 : un.b;
          const int64_t ws = static_cast<int64_t>(h) * p.ws_rows + un.si.ws_row0 + m * BM;
          // Q (+ LSE2) first: its stage is released after dK, the dO stage only
          // once the dQ drain of that iteration has read its staged rows
          if (use > 0 && !wait1(bar(B_EMPTY + s), (use - 1) & 1, ctl, 0xA0000002u)) break;
          // With D = 128 the two 64-column chunks of Q complete separate barriers:
          // the first half of S^T needs only the first (and the softmax only LSE2).
          if (kSplitQ) {
            mbar_expect_tx(bar(B_FULLQ + s), kChunk + BM * 4);
            tma_load_4d(sb + L::kQ + s * L::kTile, &tmQ, bar(B_FULLQ + s), 0, qrow, h, bq);
            bulk_load(sb + L::kLSE + s * BM * 4, p.lse2 + ws, BM * 4, bar(B_FULLQ + s));
            mbar_expect_tx(bar(B_FULLQ2 + s), kChunk);
            tma_load_4d(sb + L::kQ + s * L::kTile + kChunk, &tmQ, bar(B_FULLQ2 + s), 64, qrow, h,
                        bq);
          } else {
            mbar_expect_tx(bar(B_FULLQ + s), L::kTile + BM * 4);
#pragma unroll
            for (int c = 0; c < kDC; ++c)
              tma_load_4d(sb + L::kQ + s * L::kTile + c * kChunk, &tmQ, bar(B_FULLQ + s), c * 64,
                          qrow, h, bq);
            bulk_load(sb + L::kLSE + s * BM * 4, p.lse2 + ws, BM * 4, bar(B_FULLQ + s));
          }
          if (use > 0 && !wait1(bar(B_EMPTYDO + s), (use - 1) & 1, ctl, 0xA0000006u)) {
            ++it;  // the Q copies of this iteration are in flight
            do_pending_skipped = true;
            break;
          }
          mbar_expect_tx(bar(B_FULLDO + s), L::kTile + BM * 4);
#pragma unroll
          for (int c = 0; c < kDC; ++c)
            tma_load_4d(sb + L::kDO + s * L::kTile + c * kChunk, &tmDO, bar(B_FULLDO + s), c * 64,
                        qrow, h, bq);
          bulk_load(sb + L::kDelta + s * BM * 4, p.delta + ws, BM * 4, bar(B_FULLDO + s));
        }
        if (*abort_flag) break;
      }
      // Before exit, wait (bounded, ignoring the abort flag) until every copy this
      // thread issued has landed, so no TMA write targets a finished CTA.
      for (uint32_t d = 1; d <= L::kKVSlots && d <= uc; ++d) {  // the last K/V loads of each slot
        const uint32_t v = uc - d;
        wait1(bar(v % L::kKVSlots ? B_KVFULL1 : B_KVFULL), (v / L::kKVSlots) & 1, ctl, 0xA0000003u,
              false);
      }
      for (uint32_t s = 0; s < kStages && s < it; ++s) {
        const uint32_t last = (it - 1 - s) / kStages;  // uses of stage (it-1-s) % kStages
        const uint32_t st = (it - 1 - s) % kStages;
        wait1(bar(B_FULLQ + st), last & 1, ctl, 0xA0000004u, false);
        if (kSplitQ) wait1(bar(B_FULLQ2 + st), last & 1, ctl, 0xA0000007u, false);
        if (!(s == 0 && do_pending_skipped))
          wait1(bar(B_FULLDO + st), last & 1, ctl, 0xA0000005u, false);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per query tile: dP^T, dV, then the next tile's S^T as soon as dV and the
    // dS phase have read P^T (so S^T runs while the softmax warps compute dS),
    // then dQ and dK once dS^T is in shared memory.  The first S^T of a unit
    // waits for its K/V tiles.
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_f16(kIsBf16, 0, 0, BN, BM);
      constexpr uint32_t kIdKV = idesc_f16(kIsBf16, 0, 1, BN, D);
      constexpr uint32_t kIdDQ = idesc_f16(kIsBf16, 1, 1, BM, D);
      // Shared-memory descriptors.  At D = 128 a descriptor is a per-CTA base plus
      // (address offset >> 4): the start-address field holds the address >> 4 in
      // its low 14 bits, so for addresses below 256 KiB the sum equals the
      // descriptor built from the address, in fewer instructions of this one
      // issuing thread (measured +2.2 to +2.9 % at D = 128; the D = 64
      // instantiations, 4 % slower that way, build each from its address).
      constexpr bool kBaseDesc = D != 64;
      const uint64_t dKM = sdesc_sw128(sb, 16, 1024);      // K-major (LBO unused)
      const uint64_t dMN = sdesc_sw128(sb, kChunk, 1024);  // MN-major
      auto dk_at = [&](uint32_t a) -> uint64_t {
        return kBaseDesc ? dKM + ((a - sb) >> 4) : sdesc_sw128(a, 16, 1024);
      };
      auto dm_at = [&](uint32_t a) -> uint64_t {
        return kBaseDesc ? dMN + ((a - sb) >> 4) : sdesc_sw128(a, kChunk, 1024);
      };
      // S^T = K Q^T   (M = keys, N = queries, K = head dim; both K-major)
      auto issue_s = [&](uint32_t sK, uint32_t sQ, uint32_t st, uint32_t ph) -> bool {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if (kSplitQ && kk == 4) {  // the second head-dim chunk of Q lands separately
            if (!wait1(bar(B_FULLQ2 + st), ph, ctl, 0xA000001Bu)) return false;
            tc_fence_after();
          }
          const uint32_t koff = (kk >> 2) * kChunk + (kk & 3) * 32;
          mma_ss(tmem + TM_S, dk_at(sK + koff), dk_at(sQ + koff),
                 kIdS, kk > 0);
        }
        tc_commit(bar(B_SFULL));
        return true;
      };
      // S^T of iteration `it` overwrites the packed P^T of iteration it - 1:
      // dV must have completed and the dS phase must have read it
      auto wait_p_consumed = [&](uint32_t prev) -> bool {
        return wait1(bar(B_PVDONE), prev & 1, ctl, 0xA0000014u) &&
               wait1(bar(B_PREAD), prev & 1, ctl, 0xA0000019u);
      };
      uint32_t it = 0, uc = 0;
      // With two K/V slots the last tile of a unit also issues the next unit's
      // first S^T (its K is already in the other slot): that unit is then taken
      // early (pk) and its S^T not issued again (s_pre).
      int u_pk = 0;
      bool pk = false, s_pre = false;
      for (uint32_t k = 0;; ++k) {
        int u;
        if (pk) {
          u = u_pk;
          pk = false;
        } else if (!take_unit(k, false, u)) {
          goto mma_exit;
        }
        if (u >= num_units) break;
        const Unit un = get_unit(p, u, G, wleft);
        if (un.n_iters == 0) continue;
        const uint32_t kvs = uc % L::kKVSlots;
        const uint32_t sK = sb + (kvs ? L::kK1 : L::kK), sV = sb + (kvs ? L::kV1 : L::kV);
        const uint32_t tDK = tmem + TM_DK + kvs * 64, tDV = tmem + TM_DV + kvs * 64;
        if (!s_pre) {
          if (!wait1(bar(kvs ? B_KVFULL1 : B_KVFULL), (uc / L::kKVSlots) & 1, ctl, 0xA0000011u))
            goto mma_exit;
          const uint32_t s = it % kStages;
          if (!wait1(bar(B_FULLQ + s), (it / kStages) & 1, ctl, 0xA0000013u)) goto mma_exit;
          if (it > 0 && !wait_p_consumed(it - 1)) goto mma_exit;
          tc_fence_after();
          if (!issue_s(sK, sb + L::kQ + s * L::kTile, s, (it / kStages) & 1)) goto mma_exit;
        }
        s_pre = false;
        for (int j = 0; j < un.n_iters; ++j, ++it) {
          const uint32_t s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          const uint32_t sQ = sb + L::kQ + s * L::kTile;
          const uint32_t sDO = sb + L::kDO + s * L::kTile;
          if (!wait1(bar(B_FULLDO + s), ph, ctl, 0xA0000015u)) goto mma_exit;
          // dP^T overwrites the previous dQ, which must have been drained
          if (it > 0 && !wait1(bar(B_DQFREE), (it - 1) & 1, ctl, 0xA0000016u)) goto mma_exit;
          tc_fence_after();
          // dP^T = V dO^T
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kChunk + (kk & 3) * 32;
            mma_ss(tmem + TM_DP, dk_at(sV + koff), dk_at(sDO + koff),
                   kIdS, kk > 0);
          }
          tc_commit(bar(B_DPFULL));
          // dV += P^T dO   (A = P^T from TMEM, B = dO MN-major, K = queries)
          if (!wait1(bar(B_PREADY), it & 1, ctl, 0xA0000017u)) goto mma_exit;
          // the previous unit's epilogue must have read dK/dV before they restart
          if (j == 0 && uc >= L::kKVSlots &&
              !wait1(bar(kvs ? B_DKDVFREE1 : B_DKDVFREE), ((uc / L::kKVSlots) - 1) & 1, ctl,
                     0xA0000012u))
            goto mma_exit;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_ts(tDV, tmem + TM_P + (16 * kk / kCols) * kCols + (16 * kk % kCols) / 2,
                   dm_at(sDO + kk * 2048),
                   kIdKV, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(B_PVDONE));
          tc_commit(bar(B_EMPTYDO + s));
          // the next tile's S^T, within this unit (same K tile); the Q tile usually
          // lands last, so its wait comes last
          if (j + 1 < un.n_iters) {
            const uint32_t s1 = (it + 1) % kStages;
            if (!wait_p_consumed(it)) goto mma_exit;
            if (!wait1(bar(B_FULLQ + s1), ((it + 1) / kStages) & 1, ctl, 0xA000001Au))
              goto mma_exit;
            tc_fence_after();
            if (!issue_s(sK, sb + L::kQ + s1 * L::kTile, s1, ((it + 1) / kStages) & 1))
              goto mma_exit;
          } else if constexpr (L::kKVSlots == 2) {
            // the next unit's first S^T, from the other K/V slot
            if (!take_unit(k + 1, false, u_pk)) goto mma_exit;
            pk = true;
            if (u_pk < num_units && get_unit(p, u_pk, G, wleft).n_iters > 0) {
              const uint32_t kvs2 = (uc + 1) % 2;
              const uint32_t s1 = (it + 1) % kStages;
              if (!wait1(bar(kvs2 ? B_KVFULL1 : B_KVFULL), ((uc + 1) / 2) & 1, ctl, 0xA000001Cu))
                goto mma_exit;
              if (!wait_p_consumed(it)) goto mma_exit;
              if (!wait1(bar(B_FULLQ + s1), ((it + 1) / kStages) & 1, ctl, 0xA000001Du))
                goto mma_exit;
              tc_fence_after();
              if (!issue_s(sb + (kvs2 ? L::kK1 : L::kK), sb + L::kQ + s1 * L::kTile, s1,
                           ((it + 1) / kStages) & 1))
                goto mma_exit;
              s_pre = true;
            }
          }
          if (!wait1(bar(B_DSREADY), it & 1, ctl, 0xA0000018u)) goto mma_exit;
          tc_fence_after();
          // dQ = dS K   (A = dS MN-major from the dS^T tile, B = K MN-major, N = D)
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ss(tmem + TM_DQ, dm_at(sb + L::kDS + kk * 2048), dm_at(sK + kk * 2048), kIdDQ,
                   kk > 0);
          tc_commit(bar(B_DQFULL));
          // dK += dS^T Q   (A = dS^T K-major from the dS^T tile, B = Q MN-major)
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kChunk + (kk & 3) * 32;
            mma_ss(tDK, dk_at(sb + L::kDS + koff), dm_at(sQ + kk * 2048), kIdKV,
                   (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(bar(B_DKDONE));
          tc_commit(bar(B_EMPTY + s));
        }
        tc_commit(bar(kvs ? B_DKDVFULL1 : B_DKDVFULL));
        tc_commit(bar(kvs ? B_KVEMPTY1 : B_KVEMPTY));
        ++uc;
      }
    mma_exit:
      // make sure no MMA is still running before TMEM is released
      tc_commit(bar(B_FINAL));
      wait1(bar(B_FINAL), 0, ctl, 0xA000001Fu, false);
    }
  }
  } else if (warp < 4 + kSoftmaxWarps) {
    // ------------------------------------------------- softmax / dS / epilogue
    // Thread = key row jl (TMEM lane).  Column group `grp` of the softmax warps
    // owns query columns [c0, c0 + kCols): their S^T and dP^T values, and keeps
    // their packed P^T in TMEM columns [c0, c0 + kCols / 2), inside the S^T
    // columns the warp itself has read, so the groups never wait for each other.
    const uint32_t quad = warp & 3;
    const int grp = static_cast<int>(warp - 4) >> 2;
    const int c0 = kCols * grp;
    const int jl = static_cast<int>(quad * 32 + lane);  // key row within the tile
    const uint32_t tl = tmem + ((quad * 32) << 16);    // this warp's TMEM lanes
    const float sl2 = p.scale_log2;
    // epilogue share: the first half of the groups writes dK, the second dV,
    // each group a contiguous block of eCols head-dim columns
    constexpr int kEGroups = kGroups / 2;
    constexpr int eCols = D / kEGroups;
    const bool writes_dk = grp < kEGroups;
    const int e0 = (grp % kEGroups) * eCols;
    uint32_t it = 0, uc = 0;
    for (uint32_t k = 0;; ++k) {
      int u;
      if (!take_unit(k, true, u)) goto done;
      if (u >= num_units) break;
      const Unit un = get_unit(p, u, G, wleft);
      if (!un.has_keys) continue;
      const int key = un.n * BN + jl;
      const bool key_ok = key < un.si.sk;
      const TensorArg& outp = writes_dk ? p.dk : p.dv;
      T* out_row = static_cast<T*>(const_cast<void*>(outp.ptr)) + (varlen ? 0 : un.b * outp.sb) +
                   static_cast<int64_t>(un.si.k_start + key) * outp.ss +
                   static_cast<int64_t>(un.g) * outp.sh + e0;
      if (un.n_iters == 0) {  // keys but no queries: dK = dV = 0
        if (key_ok) {
#pragma unroll
          for (int c = 0; c < eCols / 8; ++c)
            if (e0 + 8 * c < p.head_dim)  // a padded head dimension stops early
              reinterpret_cast<uint4*>(out_row)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int off = un.si.sk - un.si.sq;
      for (int j = 0; j < un.n_iters; ++j, ++it) {
        const uint32_t s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        int h_unused, m;
        iter_hm(un, j, G, h_unused, m);
        const int q0 = m * BM;
        const bool need_mask =
            (q0 + BM > un.si.sq) || (un.n * BN + BN > un.si.sk) ||
            (p.win_right >= 0 && un.n * BN + BN - 1 > q0 + off + p.win_right) ||
            (wleft >= 0 && un.n * BN < q0 + BM - 1 + off - wleft);
        const float* lse2 = reinterpret_cast<const float*>(smem + L::kLSE + s * BM * 4) + c0;
        const float* dlt = reinterpret_cast<const float*>(smem + L::kDelta + s * BM * 4) + c0;
        // valid queries of this key row, in this group's column coordinates: lo <= c < hi
        int lo = 0, hi = key_ok ? min(kCols, un.si.sq - q0 - c0) : 0;
        if (p.win_right >= 0) lo = max(0, key - off - p.win_right - q0 - c0);
        if (wleft >= 0) hi = min(hi, key - off + wleft - q0 - c0 + 1);
        if (!wait_warp(bar(B_FULLQ + s), ph, ctl, 0xA0000021u)) goto done;
        if (!wait_warp(bar(B_SFULL), it & 1, ctl, 0xA0000022u)) goto done;
        tc_fence_after();
        {
          uint32_t sv[kCols];
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) tmem_ld32p(tl + TM_S + c0 + 32 * c, sv + 32 * c);
          tmem_wait_ld();
          // P^T = exp2(S^T * scale * log2 e - LSE2[query]), masked.  With a logit
          // cap the logit is c tanh(S^T scale / c), and the cap's derivative
          // 1 - tanh^2 goes (packed) into the half of this group's S^T columns
          // that P^T does not use, for the dS phase.
          uint32_t pk[kCols / 2];
#pragma unroll
          for (int e4 = 0; e4 < kCols / 4; ++e4) {
            const float4 l = reinterpret_cast<const float4*>(lse2)[e4];
            const uint32_t* v = sv + e4 * 4;
            float x0, x1, x2, x3;
            if constexpr (kCap) {
              const float t0 = tanh_exp(__uint_as_float(v[0]) * p.cap_in);
              const float t1 = tanh_exp(__uint_as_float(v[1]) * p.cap_in);
              const float t2 = tanh_exp(__uint_as_float(v[2]) * p.cap_in);
              const float t3 = tanh_exp(__uint_as_float(v[3]) * p.cap_in);
              x0 = ex2(fmaf(t0, p.cap_out, -l.x));
              x1 = ex2(fmaf(t1, p.cap_out, -l.y));
              x2 = ex2(fmaf(t2, p.cap_out, -l.z));
              x3 = ex2(fmaf(t3, p.cap_out, -l.w));
              // sv is no longer needed: its first half holds the packed derivative
              sv[e4 * 2] = Pack<T>::two(fmaf(-t0, t0, 1.f), fmaf(-t1, t1, 1.f));
              sv[e4 * 2 + 1] = Pack<T>::two(fmaf(-t2, t2, 1.f), fmaf(-t3, t3, 1.f));
            } else {
              x0 = ex2(fmaf(__uint_as_float(v[0]), sl2, -l.x));
              x1 = ex2(fmaf(__uint_as_float(v[1]), sl2, -l.y));
              x2 = ex2(fmaf(__uint_as_float(v[2]), sl2, -l.z));
              x3 = ex2(fmaf(__uint_as_float(v[3]), sl2, -l.w));
            }
            if (need_mask) {
              const int c = e4 * 4;
              x0 = (c + 0 >= lo && c + 0 < hi) ? x0 : 0.f;
              x1 = (c + 1 >= lo && c + 1 < hi) ? x1 : 0.f;
              x2 = (c + 2 >= lo && c + 2 < hi) ? x2 : 0.f;
              x3 = (c + 3 >= lo && c + 3 < hi) ? x3 : 0.f;
            }
            pk[e4 * 2] = Pack<T>::two(x0, x1);
            pk[e4 * 2 + 1] = Pack<T>::two(x2, x3);
          }
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c)
            tmem_st16(tl + TM_P + c0 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(pk + 16 * c));
          if constexpr (kCap) {
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c)
              tmem_st16(tl + TM_S + c0 + kCols / 2 + 16 * c,
                        *reinterpret_cast<uint32_t(*)[16]>(sv + 16 * c));
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PREADY));

        if (!wait_warp(bar(B_FULLDO + s), ph, ctl, 0xA0000023u)) goto done;
        // the dS^T tile was last read by the previous tile's dQ and dK MMAs (checked
        // here, while dP^T is usually still running)
        if (it > 0 && !wait_warp(bar(B_DKDONE), (it - 1) & 1, ctl, 0xA0000026u)) goto done;
        if (!wait_warp(bar(B_DPFULL), it & 1, ctl, 0xA0000024u)) goto done;
        tc_fence_after();
        {
          // dS^T = P^T (dP^T - Delta[query]) for this group's queries, in
          // sub-chunks of 32, to the smem dS^T tile, whose chunk c holds queries
          // [64 c, +64): row jl is 128 bytes and its 16-byte unit u is stored
          // at u ^ (jl % 8) (128-byte swizzle).
          uint32_t dpv[kCols], pv[kCols / 2];
          uint32_t cv[kCap ? kCols / 2 : 1];  // packed cap derivative (logit cap only)
#pragma unroll
          for (int c = 0; c < kCols / 32; ++c) tmem_ld32p(tl + TM_DP + c0 + 32 * c, dpv + 32 * c);
          if (kCols == 64) {
            tmem_ld32p(tl + TM_P + c0, pv);
          } else {
            tmem_ld16(tl + TM_P + c0, *reinterpret_cast<uint32_t(*)[16]>(pv));
          }
          if constexpr (kCap) {
#pragma unroll
            for (int c = 0; c < kCols / 32; ++c)
              tmem_ld16(tl + TM_S + c0 + kCols / 2 + 16 * c,
                        *reinterpret_cast<uint32_t(*)[16]>(cv + 16 * c));
          }
          tmem_wait_ld();
          // P^T has been read: the next tile's S^T may overwrite it
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_PREAD));
#pragma unroll
          for (int sub = 0; sub < kCols / 32; ++sub) {
            const int qc = c0 + 32 * sub;  // first query column of this sub-chunk
            const uint32_t row_base = L::kDS + (qc / 64) * kChunk + jl * 128;
            uint32_t pk[16];
#pragma unroll
            for (int e4 = 0; e4 < 8; ++e4) {
              const float4 dl = reinterpret_cast<const float4*>(dlt)[sub * 8 + e4];
              float2 p01 = Pack<T>::unpack(pv[sub * 16 + e4 * 2]);
              float2 p23 = Pack<T>::unpack(pv[sub * 16 + e4 * 2 + 1]);
              if constexpr (kCap) {  // dS of the uncapped logit: times 1 - tanh^2
                const float2 c01 = Pack<T>::unpack(cv[sub * 16 + e4 * 2]);
                const float2 c23 = Pack<T>::unpack(cv[sub * 16 + e4 * 2 + 1]);
                p01.x *= c01.x;
                p01.y *= c01.y;
                p23.x *= c23.x;
                p23.y *= c23.y;
              }
              const uint32_t* v = dpv + sub * 32 + e4 * 4;
              pk[e4 * 2] = Pack<T>::two(p01.x * (__uint_as_float(v[0]) - dl.x),
                                        p01.y * (__uint_as_float(v[1]) - dl.y));
              pk[e4 * 2 + 1] = Pack<T>::two(p23.x * (__uint_as_float(v[2]) - dl.z),
                                            p23.y * (__uint_as_float(v[3]) - dl.w));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint32_t unit = (((qc % 64) / 8) + q) ^ (jl & 7);
              *reinterpret_cast<uint4*>(smem + row_base + unit * 16) =
                  make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DSREADY));
      }
      // ---- epilogue: this group's columns of dK = scale * acc or dV = acc (or
      // the dQ drain warps write dK/dV instead)
      if constexpr (!kDrainEpi) {
        if (!wait_warp(bar(B_DKDVFULL), uc & 1, ctl, 0xA0000025u)) goto done;
        tc_fence_after();
        {
          const uint32_t src = (writes_dk ? TM_DK : TM_DV) + e0;
          const float mul = writes_dk ? p.scale : 1.0f;
          constexpr int kEStep = eCols % 32 == 0 ? 32 : 16;  // TMEM columns per load
#pragma unroll 1
          for (int c = 0; c < eCols / kEStep; ++c) {
            uint32_t a[kEStep];
            if constexpr (kEStep == 32) {
              tmem_ld32(tl + src + c * 32, a);
            } else {
              tmem_ld16(tl + src + c * 16, a);
            }
            tmem_wait_ld();
            if (key_ok) {
#pragma unroll
              for (int q = 0; q < kEStep / 8; ++q) {
                uint4 o;
                o.x = Pack<T>::two(__uint_as_float(a[8 * q + 0]) * mul, __uint_as_float(a[8 * q + 1]) * mul);
                o.y = Pack<T>::two(__uint_as_float(a[8 * q + 2]) * mul, __uint_as_float(a[8 * q + 3]) * mul);
                o.z = Pack<T>::two(__uint_as_float(a[8 * q + 4]) * mul, __uint_as_float(a[8 * q + 5]) * mul);
                o.w = Pack<T>::two(__uint_as_float(a[8 * q + 6]) * mul, __uint_as_float(a[8 * q + 7]) * mul);
                if (e0 + c * kEStep + 8 * q < p.head_dim)  // a padded head dimension stops early
                  reinterpret_cast<uint4*>(out_row + c * kEStep)[q] = o;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DKDVFREE));
      }
      ++uc;
    }
  } else {
    setmaxnreg_inc<kRegDrain>();
    // ------------------------------------------------------------ dQ drain
    // Thread = query row (TMEM lane); warp q owns rows [32q, 32q+32) of the tile.
    // The rows go out in two passes, staged in the iteration's dO stage (free
    // once the dV MMA, issued before dQ, has read it) as 32x32 fp32 boxes with
    // the 128-byte swizzle, each box added to dQaccum by a TMA reduce (whole
    // 128-byte lines at L2).  The stage goes back to the producer (EMPTYDO)
    // once the reduces have read it.  Rows past the sequence end hold exact
    // zeros (their dS is 0) and stay inside the sequence's padded workspace
    // rows, so they need no mask.
    // In deterministic mode a warp waits until the key tiles before n that see
    // this query tile (0..n-1, or from the first one inside a left window) have
    // completed their adds to the warp's 32 rows (one arrival each on the
    // semaphore of those rows) and releases once its own adds have completed.
    // With two K/V slots (D = 64) these warps also write each unit's dK and dV
    // once its last tile is drained (the epilogue below), so that the softmax
    // warps go straight on to the next unit.
    const uint32_t quad = warp & 3;
    const uint32_t tl = tmem + ((quad * 32) << 16);
    // Per warp and pass: up to kBoxes boxes of 32 rows x 32 fp32 columns (4 KB
    // each); the 4 warps' staging fills the dO stage exactly (kTile bytes).  At
    // D = 96 the second pass has one box.
    constexpr int kBoxes = static_cast<int>(L::kTile / (4 * 4096));
    constexpr int kPassCols = 32 * kBoxes;
    constexpr int kPasses = (D + kPassCols - 1) / kPassCols;
    static_assert(4 * kBoxes * 4096 == L::kTile, "dQ staging must fit the dO stage");
    constexpr int kLastBoxes = D / 32 - (kPasses - 1) * kBoxes;  // kBoxes unless D = 96
    uint32_t it = 0, uc = 0;
    for (uint32_t k = 0;; ++k) {
      int u;
      if (!take_unit(k, true, u)) goto done;
      if (u >= num_units) break;
      const Unit un = get_unit(p, u, G, wleft);
      if (un.n_iters == 0) continue;
      for (int j = 0; j < un.n_iters; ++j, ++it) {
        int h, m;
        iter_hm(un, j, G, h, m);
        const int row0 = static_cast<int>(static_cast<int64_t>(h) * p.ws_rows + un.si.ws_row0 +
                                          m * BM + quad * 32);
        // one semaphore per (head, query tile, drain warp): the 32 rows of warp
        // `quad` take their adds in key-tile order, independently of the others
        int* sem = p.sem + (static_cast<int64_t>(h) * (p.ws_rows / kTileRows) +
                            un.si.ws_row0 / kTileRows + m) * 4 + quad;
        const uint32_t s = it % kStages;
        const uint32_t stage_off = L::kDO + s * L::kTile + quad * (kBoxes * 4096);
        if (!wait_warp(bar(B_DQFULL), it & 1, ctl, 0xA0000031u)) goto done;
        tc_fence_after();
        // With registers for it, the whole row first (the next tile's dP^T reuses
        // these TMEM columns); otherwise one pass at a time.
        constexpr int kHeld = kDrainWholeRow ? D : kPassCols;
        uint32_t a[kHeld];
        // columns read before the first pass: the whole row, or the first pass's
        constexpr int kFirstCols =
            kDrainWholeRow ? D : (kPasses == 1 ? 32 * kLastBoxes : kPassCols);
#pragma unroll
        for (int c = 0; c < kFirstCols / 32; ++c) tmem_ld32p(tl + TM_DQ + c * 32, a + c * 32);
        tmem_wait_ld();
        if (kDrainWholeRow) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_DQFREE));
        }
        if (p.deterministic) {
          int stop = 0;
          if (lane == 0) {
            // key tiles before this one that see query tile m (all of them
            // unless a left window starts the range later)
            const int want = un.n - window_first_key(m * BM, un.si.sq, un.si.sk, wleft) / BN;
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t spin = 0;; ++spin) {
              if (ld_acquire(sem) >= want) break;
              if ((spin & 15) == 15) {
                if (*abort_flag) { stop = 1; break; }
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                  raise_abort(ctl, 0xA0000033u);
                  stop = 1;
                  break;
                }
              }
            }
            fence_proxy_async_global();
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) goto done;
        }
#pragma unroll
        for (int pass = 0; pass < kPasses; ++pass) {
          if (!kDrainWholeRow && pass > 0) {
#pragma unroll
            for (int c = 0; c < (pass == kPasses - 1 ? kLastBoxes : kBoxes); ++c)
              tmem_ld32p(tl + TM_DQ + pass * kPassCols + c * 32, a + c * 32);
            tmem_wait_ld();
            if (pass == kPasses - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar(B_DQFREE));
            }
          }
          if (pass > 0) {
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int bx = 0; bx < (pass == kPasses - 1 ? kLastBoxes : kBoxes); ++bx) {
            const uint32_t box = stage_off + bx * 4096;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint32_t* v = a + (kDrainWholeRow ? pass * kPassCols : 0) + bx * 32 + q * 4;
              *reinterpret_cast<uint4*>(smem + box + lane * 128 + ((q ^ (lane & 7)) * 16)) =
                  make_uint4(v[0], v[1], v[2], v[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int bx = 0; bx < (pass == kPasses - 1 ? kLastBoxes : kBoxes); ++bx)
              tma_reduce_add_2d(&tmDQ, sb + stage_off + bx * 4096, pass * kPassCols + bx * 32,
                                row0);
            bulk_commit();
          }
        }
        if (lane == 0) {
          if (p.deterministic) {
            bulk_wait_all();
            fence_proxy_async_global();
            __threadfence();
            red_release_add(sem, 1);
          } else {
            bulk_wait_read_all();
          }
        }
        __syncwarp();
        // with one K/V slot and the drain-side epilogue, the unit's last dO stage
        // stages dK/dV and goes back to the producer after the epilogue
        if (lane == 0 && (L::kKVSlots == 2 || !kDrainEpi || j + 1 < un.n_iters))
          mbar_arrive(bar(B_EMPTYDO + s));
      }
      if constexpr (L::kKVSlots == 1 && kDrainEpi) {
        // ---- epilogue: rows [32 quad, +32) of dK = scale * acc and dV = acc.  A key
        // tile wholly inside the sequence is staged in this warp's quarter of the
        // unit's last dO stage as 32-row x 64-column boxes (128-byte rows, 128-byte
        // swizzle) and leaves through TMA tile stores (whole lines, and no per-row
        // stores in the load/store pipe every warp's barrier operations use); a
        // ragged tile stores per row and stops at the sequence end.
        const uint32_t s = (it - 1) % kStages;
        const uint32_t stage_off = L::kDO + s * L::kTile + quad * (L::kTile / 4);
        const int key = un.n * BN + static_cast<int>(quad) * 32 + static_cast<int>(lane);
        const bool tile_store = un.n * BN + BN <= un.si.sk;
        if (!wait_warp(bar(B_DKDVFULL), uc & 1, ctl, 0xA0000035u)) goto done;
        tc_fence_after();
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          const TensorArg& outp = t == 0 ? p.dk : p.dv;
          const float mul = t == 0 ? p.scale : 1.0f;
          if (t == 1 && tile_store) {  // the dK stores must have read the staging
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t a[32];
            tmem_ld32(tl + (t == 0 ? TM_DK : TM_DV) + c * 32, a);
            tmem_wait_ld();
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = Pack<T>::two(__uint_as_float(a[2 * i]) * mul,
                                  __uint_as_float(a[2 * i + 1]) * mul);
            if (tile_store) {
              // columns [32 c, 32 c + 32): 16-byte units 4 (c & 1) .. + 3 of box c / 2
              const uint32_t row = stage_off + (c >> 1) * 4096 + lane * 128;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(smem + row + ((((c & 1) * 4 + q) ^ (lane & 7)) << 4)) =
                    make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            } else if (key < un.si.sk) {
              T* out_row = static_cast<T*>(const_cast<void*>(outp.ptr)) +
                           (varlen ? 0 : un.b * outp.sb) +
                           static_cast<int64_t>(un.si.k_start + key) * outp.ss +
                           static_cast<int64_t>(un.g) * outp.sh + c * 32;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (c * 32 + 8 * q < p.head_dim)  // a padded head dimension stops early
                  reinterpret_cast<uint4*>(out_row)[q] =
                      make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
          }
          if (t == 1) {  // dK and dV have left TMEM: the next unit may restart them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_DKDVFREE));
          }
          if (tile_store) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
              for (int bx = 0; bx < D / 64; ++bx)
                if (bx * 64 < p.head_dim)  // a padded head dimension stops early
                  tma_store_4d(t == 0 ? &tmDK : &tmDV, sb + stage_off + bx * 4096, bx * 64,
                               un.si.k_start + un.n * BN + static_cast<int>(quad) * 32, un.g,
                               varlen ? 0 : un.b);
              bulk_commit();
            }
          }
        }
        // the stores have read the staging: the stage goes back to the producer
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_EMPTYDO + s));
        ++uc;
      }
      if constexpr (L::kKVSlots == 2) {
        // ---- epilogue: rows [32 quad, +32) of dK = scale * acc and dV = acc from
        // the unit's TMEM buffer.  A key tile wholly inside the sequence is staged
        // as two 32-row x 64-column boxes (128-byte rows, 128-byte swizzle) and
        // leaves through TMA tile stores (whole lines, and no per-row stores in
        // the load/store pipe every warp's barrier operations use); a ragged tile
        // stores per row and stops at the sequence end.
        const uint32_t kvs = uc % 2;
        const uint32_t stg = L::kEpi + quad * 8192;  // dK box, then dV box
        const int key = un.n * BN + static_cast<int>(quad) * 32 + static_cast<int>(lane);
        const bool tile_store = un.n * BN + BN <= un.si.sk;
        if (!wait_warp(bar(kvs ? B_DKDVFULL1 : B_DKDVFULL), (uc / 2) & 1, ctl, 0xA0000035u))
          goto done;
        tc_fence_after();
        if (lane == 0) bulk_wait_read_all();  // the previous unit's stores have read the staging
        __syncwarp();
#pragma unroll 1
        for (int t = 0; t < 2; ++t) {
          const TensorArg& outp = t == 0 ? p.dk : p.dv;
          const float mul = t == 0 ? p.scale : 1.0f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t a[32];
            tmem_ld32(tl + (t == 0 ? TM_DK : TM_DV) + kvs * 64 + c * 32, a);
            tmem_wait_ld();
            uint32_t o[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = Pack<T>::two(__uint_as_float(a[2 * i]) * mul,
                                  __uint_as_float(a[2 * i + 1]) * mul);
            if (tile_store) {
              // columns [32 c, 32 c + 32): 16-byte units 4 c .. 4 c + 3 of the row
              const uint32_t row = stg + t * 4096 + lane * 128;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(smem + row + (((c * 4 + q) ^ (lane & 7)) << 4)) =
                    make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            } else if (key < un.si.sk) {
              T* out_row = static_cast<T*>(const_cast<void*>(outp.ptr)) +
                           (varlen ? 0 : un.b * outp.sb) +
                           static_cast<int64_t>(un.si.k_start + key) * outp.ss +
                           static_cast<int64_t>(un.g) * outp.sh + c * 32;
#pragma unroll
              for (int q = 0; q < 4; ++q)
                if (c * 32 + 8 * q < p.head_dim)  // a padded head dimension stops early
                  reinterpret_cast<uint4*>(out_row)[q] =
                      make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
            }
          }
        }
        // dK and dV have left TMEM: the unit two ahead may restart this buffer
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kvs ? B_DKDVFREE1 : B_DKDVFREE));
        if (tile_store) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int row0 = un.si.k_start + un.n * BN + static_cast<int>(quad) * 32;
            tma_store_4d(&tmDK, sb + stg, 0, row0, un.g, varlen ? 0 : un.b);
            tma_store_4d(&tmDV, sb + stg + 4096, 0, row0, un.g, varlen ? 0 : un.b);
            bulk_commit();
          }
        }
        ++uc;
      }
    }
    if (lane == 0) bulk_wait_all();
  }

done:
  if constexpr (kDrainEpi) {
    if (lane == 0) bulk_wait_all();  // no store may still read this CTA's shared memory
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

template <typename T, int D, bool kCap, bool kLeft>
cudaError_t launch_t(const BwdParams& p_in, int dtype, cudaStream_t stream) {
  const bool varlen = p_in.seq.cu_q != nullptr;
  // unit order (see get_unit): sequence major for packed batches and, at D = 128,
  // for padded MHA outside deterministic mode; key-tile major otherwise
  BwdParams p = p_in;
  p.unit_seq_major = varlen || (D == 128 && p.h_q == p.h_k && !p.deterministic);
  p.unit_per = p.unit_seq_major ? ceil_div(p.max_seqlen_k, BN) * p.h_k : p.seq.batch * p.h_k;
  const int nb = varlen ? 1 : p.seq.batch;
  CUtensorMap tq, tk, tv, tdo;
  // the maps span the logical head dimension: columns up to D read as zero
  const int d = p.head_dim;
  if (!encode_tmap_bshd(&tq, p.q, dtype, p.seq.seqlen_q, p.h_q, nb, d, BM) ||
      !encode_tmap_bshd(&tk, p.k, dtype, p.seq.seqlen_k, p.h_k, nb, d, BN) ||
      !encode_tmap_bshd(&tv, p.v, dtype, p.seq.seqlen_k, p.h_k, nb, d, BN) ||
      !encode_tmap_bshd(&tdo, p.dout, dtype, p.seq.seqlen_q, p.h_q, nb, d, BM))
    return cudaErrorInvalidValue;
  CUtensorMap tdq;
  // the accumulator rows are pad_head_dim wide (128 for the D = 96 kernel)
  if (!encode_tmap_f32_2d(&tdq, p.dqacc, p.ws_rows * p.h_q, pad_head_dim(p.head_dim)))
    return cudaErrorInvalidValue;
  CUtensorMap tdk, tdv;  // dK/dV tile stores (D = 64), 32-row boxes
  if (!encode_tmap_bshd(&tdk, p.dk, dtype, p.seq.seqlen_k, p.h_k, nb, d, 32) ||
      !encode_tmap_bshd(&tdv, p.dv, dtype, p.seq.seqlen_k, p.h_k, nb, d, 32))
    return cudaErrorInvalidValue;
  constexpr uint32_t smem = Smem<D>::kTotal;
  // Kernel attributes are per device: set (and check) them once on each.
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bwd_main_kernel<T, D, kCap, kLeft>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // The warpgroup register split assumes exactly kRegLaunch registers per
    // thread at launch; anything else could leave a register increase waiting.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, bwd_main_kernel<T, D, kCap, kLeft>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kRegLaunch)) return cudaErrorInvalidConfiguration;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int n_tiles = ceil_div(p.max_seqlen_k, BN);
  const int units = n_tiles * p.seq.batch * p.h_k;
  if (units <= 0) return cudaSuccess;
  const int grid = units < num_sms() ? units : num_sms();
  bwd_main_kernel<T, D, kCap, kLeft><<<grid, kThreads, smem, stream>>>(p, tq, tk, tv, tdo, tdq,
                                                                        tdk, tdv);
  return cudaGetLastError();
}

template <bool kCap, bool kLeft>
cudaError_t launch_cap(const BwdParams& p, int dtype, cudaStream_t stream) {
  const bool d64 = pad_head_dim(p.head_dim) == 64;
  // head dims in (64, 96] have a native D = 96 kernel without a cap or a left
  // window side; with either they run zero-padded on the D = 128 one
  if constexpr (!kCap && !kLeft) {
    if (p.head_dim > 64 && p.head_dim <= 96)
      return dtype == 1 ? launch_t<__nv_bfloat16, 96, false, false>(p, dtype, stream)
                        : launch_t<__half, 96, false, false>(p, dtype, stream);
  }
  if (dtype == 1) {
    return d64 ? launch_t<__nv_bfloat16, 64, kCap, kLeft>(p, dtype, stream)
               : launch_t<__nv_bfloat16, 128, kCap, kLeft>(p, dtype, stream);
  }
  return d64 ? launch_t<__half, 64, kCap, kLeft>(p, dtype, stream)
             : launch_t<__half, 128, kCap, kLeft>(p, dtype, stream);
}

}  // namespace

cudaError_t launch_bwd_main(const BwdParams& p, int dtype, cudaStream_t stream) {
  // the logit cap and a left window side are separate instantiations: the
  // default kernel keeps the code of the unmasked / causal schedule
  const bool cap = p.softcap > 0.f, left = p.win_left >= 0;
  if (cap) return left ? launch_cap<true, true>(p, dtype, stream)
                       : launch_cap<true, false>(p, dtype, stream);
  return left ? launch_cap<false, true>(p, dtype, stream)
              : launch_cap<false, false>(p, dtype, stream);
}

}  // namespace attn
