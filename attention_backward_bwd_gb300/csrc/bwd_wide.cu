// Attention backward for head dimensions above 128 (sm_103a): tcgen05 MMAs
// with TMEM accumulators, TMA loads, warp-specialised, persistent.  A tile row
// is kNC chunks of 64 head-dim columns: four (256 wide) for D in (192, 256],
// three (192 wide) for D in (128, 192]; the columns past D are zero (TMA
// out-of-bounds fill, masked stores).
//
// Same mathematics and work units as the D <= 128 kernel (TileLang
// test_tilelang_kernel_mha_bwd.py, flashattn_bwd; KV stationary, one unit =
// key tile n of 128 keys x key/value head g x sequence b).  At D = 256 the dK
// and dV accumulators of 128 keys fill all 512 TMEM columns, and K, V, Q and
// dO tiles of 128 rows need 256 KiB of shared memory, so the work of a unit is
// done in two passes (two launches) over its query tiles:
//   pass dV:    S^T = K Q^T, P^T = exp2(S^T scale log2 e - LSE2), dV += P^T dO
//   pass dK/dQ: S^T, P^T, dP^T = V dO^T, dS^T = P^T (dP^T - Delta),
//               dK += dS^T Q (times scale at the end), dQ = dS K -> dQaccum
// (S^T is computed in both passes: 6/5 of the minimal tensor work).  K stays
// in shared memory for the whole unit; the other operands stream through a
// ring of 64-column chunks (128 rows x 128 bytes, 128-byte swizzle), loaded in
// exactly the order the MMA thread consumes them:
//   pass dV, per query tile j: Q_j's kNC chunks (S^T_j), then dO_{j-1}'s kNC
//     chunks (dV_{j-1}), since S^T of the next tile is issued before dV of this
//     one so that it runs while the softmax warps compute P;
//   pass dK/dQ, per query tile: Q chunks (S^T), V and dO chunk pairs (dP^T),
//     Q chunks again (dK).
// dQ is drained in kNC 64-column passes through a 32 KiB staging buffer with
// TMA reduce-adds (in deterministic mode ordered by the per-(head, query tile,
// 32-row quarter) semaphore, as in the D <= 128 kernel).
//
// Warp roles (768 threads): warp 0 TMA producer, warp 1 MMA issuer, warp 2
// TMEM allocator, warps 4-19 softmax / dS / epilogue (thread = key row; warp
// group g = (warp - 4) / 4 takes query columns [32 g, 32 g + 32)), warps 20-23
// dQ drain (pass dK/dQ only; thread = query row).
//
// TMEM columns (512): pass dV: S^T buffers [0,128) and [128,256), dV
// [256,512).  Pass dK/dQ: S^T [0,128), dP^T [128,256), then dQ [0,64 kNC) once
// the dS phase has read both; dK [256,512).  dV and dK are accumulated as
// N = 128 products over chunk pairs (and an N = 64 product for an odd last
// chunk).
#include <atomic>

#include "bwd_units.cuh"
#include "common.cuh"

namespace attn {

namespace {

constexpr int WD = 256;                 // accumulator width (head dimension padded to 256)
constexpr uint32_t kWChunk = 128 * 128; // bytes of one chunk
constexpr int kWSoftWarps = 16;
constexpr int kWCols = 32;              // query columns per softmax warp
constexpr int kWThreads = 32 * (4 + kWSoftWarps + 4);
constexpr uint32_t kWRegLaunch = 80, kWRegWg0 = 64, kWRegDrain = 96;
static_assert(kWRegWg0 * 128 + kWRegLaunch * 32 * kWSoftWarps + kWRegDrain * 128 ==
                  kWRegLaunch * kWThreads,
              "register split must use exactly the launch allocation");
constexpr uint32_t kWTmemCols = 512;

enum WPass : int { kPassDV = 0, kPassDKDQ = 1 };

enum WBar : uint32_t {
  W_RFULL = 0,                 // ring slots (6)
  W_REMPTY = W_RFULL + 6,
  W_KFULL = W_REMPTY + 6,      // the unit's K tile
  W_KEMPTY,
  W_STFULL,                    // 2 stages of LSE2 (+ Delta)
  W_STEMPTY = W_STFULL + 2,
  W_SFULL = W_STEMPTY + 2,     // 2 (pass dV: per S buffer)
  W_PREADY = W_SFULL + 2,      // 2
  W_PVDONE = W_PREADY + 2,     // 2 (pass dV: dV read the buffer's P^T)
  W_DPFULL = W_PVDONE + 2,
  W_DSREADY,
  W_DQFULL,
  W_DQFREE0,                   // drain read dQ columns [0,128)
  W_DQFREE1,                   // drain read dQ columns [128,64 kNC)
  W_DKDONE,                    // dK (and dQ) MMAs of a tile done: dS^T tile free
  W_ACCFULL,                   // the unit's dV (pass dV) / dK (pass dK/dQ) complete
  W_ACCFREE,                   // the epilogue read it
  W_UNITFULL,                  // 2 slots
  W_UNITEMPTY = W_UNITFULL + 2,
  W_FINAL = W_UNITEMPTY + 2,
  W_COUNT
};

// kNC: 64-column chunks per tile row (4 at D in (192, 256], 3 at D in (128, 192]).
template <int kPass, int kNC>
struct WSmem {
  // ring slots.  The chunks of a tile arrive in groups of kNC (Q, dO, or
  // V/dO interleaved); an N = 128 product reads a pair of chunks starting at
  // an even offset of its group as one operand, so both must sit in adjacent
  // slots: the ring is even (four chunks) or a multiple of three (three).
  // Six slots in both passes (pass dV measured 0.7 to 0.8 % faster with six
  // than with ten at D = 256 or nine at D = 192).
  static constexpr int kRing = 6;
  static_assert(kRing % (kNC == 4 ? 2 : 3) == 0, "chunk pairs must not wrap the ring");
  static_assert(kRing == W_REMPTY - W_RFULL, "one full and one empty barrier per ring slot");
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kDS = kK + kNC * kWChunk;                         // pass dK/dQ
  static constexpr uint32_t kStage = kDS + (kPass == kPassDKDQ ? 2 * kWChunk : 0);
  static constexpr uint32_t kR = kStage + (kPass == kPassDKDQ ? 2 * kWChunk : 0);
  static constexpr uint32_t kLSE = kR + kRing * kWChunk;                      // 2 x 128 fp32
  static constexpr uint32_t kDelta = kLSE + 2 * 128 * 4;                      // 2 x 128 fp32
  static constexpr uint32_t kBar = kDelta + (kPass == kPassDKDQ ? 2 * 128 * 4 : 0);
  static constexpr uint32_t kUnitRing = kBar + W_COUNT * 8;
  static constexpr uint32_t kTmemSlot = kUnitRing + 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kTotal = kAbort + 4;
};
static_assert(WSmem<kPassDV, 4>::kTotal <= 232448, "shared memory budget (pass dV)");
static_assert(WSmem<kPassDKDQ, 4>::kTotal <= 232448, "shared memory budget (pass dK/dQ)");
static_assert(WSmem<kPassDV, 3>::kTotal <= 232448, "shared memory budget (pass dV, D <= 192)");
static_assert(WSmem<kPassDKDQ, 3>::kTotal <= 232448, "shared memory budget (pass dK/dQ, D <= 192)");

template <typename T, int kPass, bool kCap, int kNC>
__global__ void __launch_bounds__(kWThreads, 1)
    bwd_wide_kernel(const BwdParams p, const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmDQ) {
  using L = WSmem<kPass, kNC>;
  constexpr int R = L::kRing;
  constexpr bool kKQ = kPass == kPassDKDQ;
  extern __shared__ __align__(1024) unsigned char smem[];
  if (p.input_bad != nullptr && *p.input_bad) return;
  const uint32_t sb = smem_u32(smem);
  if (sb & 1023u) {  // 128-byte swizzled tiles need a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.status, 0u, 0xA3100000u);
    return;
  }
  auto bar = [&](uint32_t i) -> uint32_t { return sb + L::kBar + i * 8; };
  auto slot = [&](uint32_t q) -> uint32_t { return sb + L::kR + (q % R) * kWChunk; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const int G = p.h_q / p.h_k;
  const bool varlen = p.seq.cu_q != nullptr;
  const int n_tiles = ceil_div(p.max_seqlen_k, kTileRows);
  const int num_units = n_tiles * p.seq.batch * p.h_k;
  int* const sched = p.sched + kPass;  // each pass has its own work counter
  constexpr int kIsBf16 = Pack<T>::kIsBf16;
  constexpr int kNumConsumers = 1 + kWSoftWarps + (kKQ ? 4 : 0);

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int r = 0; r < R; ++r) {
      mbar_init(bar(W_RFULL + r), 1);
      mbar_init(bar(W_REMPTY + r), 1);
    }
    mbar_init(bar(W_KFULL), 1);
    mbar_init(bar(W_KEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(W_STFULL + s), 1);
      mbar_init(bar(W_STEMPTY + s), kWSoftWarps);
      mbar_init(bar(W_SFULL + s), 1);
      mbar_init(bar(W_PREADY + s), kWSoftWarps);
      mbar_init(bar(W_PVDONE + s), 1);
    }
    mbar_init(bar(W_DPFULL), 1);
    mbar_init(bar(W_DSREADY), kWSoftWarps);
    mbar_init(bar(W_DQFULL), 1);
    mbar_init(bar(W_DQFREE0), 4);
    mbar_init(bar(W_DQFREE1), 4);
    mbar_init(bar(W_DKDONE), 1);
    mbar_init(bar(W_ACCFULL), 1);
    mbar_init(bar(W_ACCFREE), kWSoftWarps);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(W_UNITFULL + k), 1);
      mbar_init(bar(W_UNITEMPTY + k), kNumConsumers);
    }
    mbar_init(bar(W_FINAL), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_proxy_async_smem();
  }
  if (warp == 2) {
    tmem_alloc(sb + L::kTmemSlot, kWTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);
  volatile int* uring = reinterpret_cast<volatile int*>(smem + L::kUnitRing);
  // Work units come from a persistent scheduler (first unit of CTA c is c, later
  // ones from the pass's global counter, longest first), published by the
  // producer through a 2-slot ring that every consumer role reads.
  auto take_unit = [&](uint32_t k, bool warp_wide, int& u) -> bool {
    const uint32_t s = k & 1;
    const bool ok = warp_wide ? wait_warp(bar(W_UNITFULL + s), (k >> 1) & 1, ctl, 0xA3000041u)
                              : wait1(bar(W_UNITFULL + s), (k >> 1) & 1, ctl, 0xA3000042u);
    if (!ok) return false;
    u = uring[s];
    if (!warp_wide || lane_id() == 0) mbar_arrive(bar(W_UNITEMPTY + s));
    return true;
  };

  if (warp < 4) {
    setmaxnreg_dec<kWRegWg0>();
    if (warp == 0) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmDO);
        uint32_t q = 0, uc = 0, st = 0;  // ring chunks, units with K loaded, stat stages
        bool stop = false;
        // one 64-column chunk into the next ring slot
        auto ring_load = [&](const CUtensorMap* map, int col, int row, int head, int bb) -> bool {
          const uint32_t r = q % R, use = q / R;
          if (use > 0 && !wait1(bar(W_REMPTY + r), (use - 1) & 1, ctl, 0xA3000001u)) return false;
          mbar_expect_tx(bar(W_RFULL + r), kWChunk);
          tma_load_4d(slot(q), map, bar(W_RFULL + r), col, row, head, bb);
          ++q;
          return true;
        };
        int u = blockIdx.x;
        for (uint32_t k = 0; !stop; ++k) {
          if (k >= 2 && !wait1(bar(W_UNITEMPTY + (k & 1)), ((k >> 1) - 1) & 1, ctl, 0xA3000043u))
            break;
          uring[k & 1] = u;
          mbar_arrive(bar(W_UNITFULL + (k & 1)));
          if (u >= num_units) break;
          const int u_next = static_cast<int>(gridDim.x) + atomicAdd(sched, 1);
          const Unit un = get_unit(p, u, G, p.win_left);
          u = u_next;
          if (un.n_iters == 0) continue;
          const int bk = varlen ? 0 : un.b;
          if (uc > 0 && !wait1(bar(W_KEMPTY), (uc - 1) & 1, ctl, 0xA3000002u)) break;
          ++uc;
          mbar_expect_tx(bar(W_KFULL), kNC * kWChunk);
          const int krow = un.si.k_start + un.n * kTileRows;
#pragma unroll
          for (int c = 0; c < kNC; ++c)
            tma_load_4d(sb + L::kK + c * kWChunk, &tmK, bar(W_KFULL), c * 64, krow, un.g, bk);
          // the stat stage (LSE2, and Delta in pass dK/dQ) of iteration j
          auto stat_load = [&](int j) -> bool {
            int h, m;
            iter_hm(un, j, G, h, m);
            const int64_t ws = static_cast<int64_t>(h) * p.ws_rows + un.si.ws_row0 + m * kTileRows;
            const uint32_t s = st & 1, use = st >> 1;
            if (use > 0 && !wait1(bar(W_STEMPTY + s), (use - 1) & 1, ctl, 0xA3000003u)) return false;
            mbar_expect_tx(bar(W_STFULL + s), kKQ ? 1024 : 512);
            bulk_load(sb + L::kLSE + s * 512, p.lse2 + ws, 512, bar(W_STFULL + s));
            if (kKQ) bulk_load(sb + L::kDelta + s * 512, p.delta + ws, 512, bar(W_STFULL + s));
            ++st;
            return true;
          };
          auto tile_rows = [&](int j, int& row, int& h) {
            int m;
            iter_hm(un, j, G, h, m);
            row = un.si.q_start + m * kTileRows;
          };
          const int bq = varlen ? 0 : un.b;
          for (int j = 0; j < un.n_iters && !stop; ++j) {
            int row, h;
            tile_rows(j, row, h);
            if (!stat_load(j)) { stop = true; break; }
            if (kKQ) {
              // S^T: Q chunks; dP^T: V and dO chunk pairs; dK: Q chunks again
              for (int c = 0; c < kNC && !stop; ++c) stop = !ring_load(&tmQ, c * 64, row, h, bq);
              for (int c = 0; c < kNC && !stop; ++c) {
                stop = !ring_load(&tmV, c * 64, krow, un.g, bk);
                if (!stop) stop = !ring_load(&tmDO, c * 64, row, h, bq);
              }
              for (int c = 0; c < kNC && !stop; ++c) stop = !ring_load(&tmQ, c * 64, row, h, bq);
            } else {
              // S^T_j: Q_j chunks; then dV_{j-1}: dO_{j-1} chunks
              for (int c = 0; c < kNC && !stop; ++c) stop = !ring_load(&tmQ, c * 64, row, h, bq);
              if (j > 0) {
                int row1, h1;
                tile_rows(j - 1, row1, h1);
                for (int c = 0; c < kNC && !stop; ++c)
                  stop = !ring_load(&tmDO, c * 64, row1, h1, bq);
              }
            }
          }
          if (!kKQ && !stop) {  // dV of the unit's last tile
            int row1, h1;
            tile_rows(un.n_iters - 1, row1, h1);
            for (int c = 0; c < kNC && !stop; ++c) stop = !ring_load(&tmDO, c * 64, row1, h1, bq);
          }
          if (*abort_flag) break;
        }
        // Before exit, wait (bounded, ignoring the abort flag) until every copy this
        // thread issued has landed: only the last issue into each slot, the last K
        // tile and the last two stat stages can still be in flight.
        for (uint32_t i = q > static_cast<uint32_t>(R) ? q - R : 0; i < q; ++i)
          wait1(bar(W_RFULL + i % R), (i / R) & 1, ctl, 0xA3000004u, false);
        if (uc > 0) wait1(bar(W_KFULL), (uc - 1) & 1, ctl, 0xA3000005u, false);
        for (uint32_t i = st > 2 ? st - 2 : 0; i < st; ++i)
          wait1(bar(W_STFULL + (i & 1)), (i >> 1) & 1, ctl, 0xA3000006u, false);
      }
    } else if (warp == 1) {
      // ----------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t kIdS = idesc_f16(kIsBf16, 0, 0, 128, 128);     // K, Q K-major
        constexpr uint32_t kIdN128 = idesc_f16(kIsBf16, 0, 1, 128, 128);  // B MN-major, N = 128
        constexpr uint32_t kIdN64 = idesc_f16(kIsBf16, 0, 1, 128, 64);    // B MN-major, N = 64
        constexpr uint32_t kIdDQ = idesc_f16(kIsBf16, 1, 1, 128, 64 * kNC);  // dS, K MN-major
        uint32_t q = 0, it = 0, uc = 0;
        auto ring_wait = [&](uint32_t qq) -> bool {
          return wait1(bar(W_RFULL + qq % R), (qq / R) & 1, ctl, 0xA3000011u);
        };
        // S^T = K Q^T into TMEM column `dst` from the ring's next kNC Q chunks
        auto issue_s = [&](uint32_t dst) -> bool {
          for (int c = 0; c < kNC; ++c, ++q) {
            if (!ring_wait(q)) return false;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(tmem + dst, sdesc_sw128(sb + L::kK + c * kWChunk + kk * 32, 16, 1024),
                     sdesc_sw128(slot(q) + kk * 32, 16, 1024), kIdS, (c > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar(W_REMPTY + q % R));
          }
          return true;
        };
        for (uint32_t k = 0;; ++k) {
          int u;
          if (!take_unit(k, false, u)) goto mma_exit;
          if (u >= num_units) break;
          const Unit un = get_unit(p, u, G, p.win_left);
          if (un.n_iters == 0) continue;
          if (!wait1(bar(W_KFULL), uc & 1, ctl, 0xA3000012u)) goto mma_exit;
          tc_fence_after();
          if (!kKQ) {
            // ---- pass dV: S^T_j, then dV_{j-1} (P^T of tile j-1 from TMEM, dO chunk pairs)
            auto issue_dv = [&](uint32_t t, bool first) -> bool {
              const uint32_t buf = t & 1;
              if (!wait1(bar(W_PREADY + buf), (t >> 1) & 1, ctl, 0xA3000013u)) return false;
              // the previous unit's epilogue must have read dV before it restarts
              if (first && uc > 0 && !wait1(bar(W_ACCFREE), (uc - 1) & 1, ctl, 0xA3000014u))
                return false;
              // chunk pairs as N = 128 products, an odd last chunk as N = 64
              for (int pr = 0; pr < (kNC + 1) / 2; ++pr) {
                const uint32_t q0 = q + 2 * pr;
                const bool pair = 2 * pr + 1 < kNC;
                if (!ring_wait(q0) || (pair && !ring_wait(q0 + 1))) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                  mma_ts(tmem + 256 + 128 * pr, tmem + buf * 128 + (16 * kk / kWCols) * kWCols +
                                                    (16 * kk % kWCols) / 2,
                         sdesc_sw128(slot(q0) + kk * 2048, kWChunk, 1024), pair ? kIdN128 : kIdN64,
                         (!first || kk > 0) ? 1u : 0u);
                tc_commit(bar(W_REMPTY + q0 % R));
                if (pair) tc_commit(bar(W_REMPTY + (q0 + 1) % R));
              }
              q += kNC;
              tc_commit(bar(W_PVDONE + buf));
              return true;
            };
            for (int j = 0; j < un.n_iters; ++j) {
              const uint32_t t = it + j, buf = t & 1;
              // S buffer `buf` last held tile t - 2, whose dV must have read its P^T
              if (t >= 2 && !wait1(bar(W_PVDONE + buf), ((t - 2) >> 1) & 1, ctl, 0xA3000015u))
                goto mma_exit;
              if (!issue_s(buf * 128)) goto mma_exit;
              tc_commit(bar(W_SFULL + buf));
              if (j == un.n_iters - 1) tc_commit(bar(W_KEMPTY));
              if (j > 0 && !issue_dv(t - 1, j == 1)) goto mma_exit;
            }
            if (!issue_dv(it + un.n_iters - 1, un.n_iters == 1)) goto mma_exit;
            tc_commit(bar(W_ACCFULL));
          } else {
            // ---- pass dK/dQ
            for (int j = 0; j < un.n_iters; ++j) {
              const uint32_t t = it + j;
              // S^T overwrites dQ columns [0,128) of the previous tile
              if (t > 0 && !wait1(bar(W_DQFREE0), (t - 1) & 1, ctl, 0xA3000016u)) goto mma_exit;
              if (!issue_s(0)) goto mma_exit;
              tc_commit(bar(W_SFULL));
              // dP^T = V dO^T over chunk pairs (V chunk, dO chunk); overwrites dQ [128,64 kNC)
              if (t > 0 && !wait1(bar(W_DQFREE1), (t - 1) & 1, ctl, 0xA3000017u)) goto mma_exit;
              for (int c = 0; c < kNC; ++c, q += 2) {
                if (!ring_wait(q) || !ring_wait(q + 1)) goto mma_exit;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_ss(tmem + 128, sdesc_sw128(slot(q) + kk * 32, 16, 1024),
                         sdesc_sw128(slot(q + 1) + kk * 32, 16, 1024), kIdS,
                         (c > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(W_REMPTY + q % R));
                tc_commit(bar(W_REMPTY + (q + 1) % R));
              }
              tc_commit(bar(W_DPFULL));
              if (!wait1(bar(W_DSREADY), t & 1, ctl, 0xA3000018u)) goto mma_exit;
              tc_fence_after();
              // dQ = dS K   (A = dS MN-major from the dS^T tile, B = K MN-major, N = 64 kNC)
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                mma_ss(tmem + 0, sdesc_sw128(sb + L::kDS + kk * 2048, kWChunk, 1024),
                       sdesc_sw128(sb + L::kK + kk * 2048, kWChunk, 1024), kIdDQ, kk > 0);
              tc_commit(bar(W_DQFULL));
              if (j == un.n_iters - 1) tc_commit(bar(W_KEMPTY));
              // dK += dS^T Q   (A = dS^T K-major, B = Q chunk pairs MN-major)
              if (j == 0 && uc > 0 && !wait1(bar(W_ACCFREE), (uc - 1) & 1, ctl, 0xA3000019u))
                goto mma_exit;
              for (int pr = 0; pr < (kNC + 1) / 2; ++pr) {
                const uint32_t q0 = q + 2 * pr;
                const bool pair = 2 * pr + 1 < kNC;  // an odd last chunk: N = 64
                if (!ring_wait(q0) || (pair && !ring_wait(q0 + 1))) goto mma_exit;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  const uint32_t koff = (kk >> 2) * kWChunk + (kk & 3) * 32;
                  mma_ss(tmem + 256 + 128 * pr, sdesc_sw128(sb + L::kDS + koff, 16, 1024),
                         sdesc_sw128(slot(q0) + kk * 2048, kWChunk, 1024),
                         pair ? kIdN128 : kIdN64, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(W_REMPTY + q0 % R));
                if (pair) tc_commit(bar(W_REMPTY + (q0 + 1) % R));
              }
              q += kNC;
              tc_commit(bar(W_DKDONE));
            }
            tc_commit(bar(W_ACCFULL));
          }
          it += un.n_iters;
          ++uc;
        }
      mma_exit:
        // make sure no MMA is still running before TMEM is released
        tc_commit(bar(W_FINAL));
        wait1(bar(W_FINAL), 0, ctl, 0xA300001Fu, false);
      }
    }
  } else if (warp < 4 + kWSoftWarps) {
    // ------------------------------------------------- softmax / dS / epilogue
    const uint32_t quad = warp & 3;
    const int grp = static_cast<int>(warp - 4) >> 2;
    const int c0 = kWCols * grp;
    const int jl = static_cast<int>(quad * 32 + lane);  // key row within the tile
    const uint32_t tl = tmem + ((quad * 32) << 16);
    const float sl2 = p.scale_log2;
    constexpr int eCols = WD / 4;  // epilogue: each column group writes 64 head-dim columns
    const int e0 = grp * eCols;
    uint32_t it = 0, uc = 0;
    for (uint32_t k = 0;; ++k) {
      int u;
      if (!take_unit(k, true, u)) goto done;
      if (u >= num_units) break;
      const Unit un = get_unit(p, u, G, p.win_left);
      if (!un.has_keys) continue;
      const int key = un.n * kTileRows + jl;
      const bool key_ok = key < un.si.sk;
      const TensorArg& outp = kKQ ? p.dk : p.dv;
      T* out_row = static_cast<T*>(const_cast<void*>(outp.ptr)) + (varlen ? 0 : un.b * outp.sb) +
                   static_cast<int64_t>(un.si.k_start + key) * outp.ss +
                   static_cast<int64_t>(un.g) * outp.sh + e0;
      if (un.n_iters == 0) {  // keys but no queries: the pass's gradient is 0
        if (key_ok) {
#pragma unroll
          for (int c = 0; c < eCols / 8; ++c)
            if (e0 + 8 * c < p.head_dim) reinterpret_cast<uint4*>(out_row)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int off = un.si.sk - un.si.sq;
      for (int j = 0; j < un.n_iters; ++j, ++it) {
        int h_unused, m;
        iter_hm(un, j, G, h_unused, m);
        const int q0 = m * kTileRows;
        const uint32_t ss = it & 1;  // stat stage; in pass dV also the S buffer
        const uint32_t sbuf = kKQ ? 0 : ss * 128;
        const bool need_mask =
            (q0 + kTileRows > un.si.sq) || (un.n * kTileRows + kTileRows > un.si.sk) ||
            (p.win_right >= 0 && un.n * kTileRows + kTileRows - 1 > q0 + off + p.win_right) ||
            (p.win_left >= 0 && un.n * kTileRows < q0 + kTileRows - 1 + off - p.win_left);
        const float* lse2 = reinterpret_cast<const float*>(smem + L::kLSE + ss * 512) + c0;
        const float* dlt = reinterpret_cast<const float*>(smem + L::kDelta + ss * 512) + c0;
        int lo = 0, hi = key_ok ? min(kWCols, un.si.sq - q0 - c0) : 0;
        if (p.win_right >= 0) lo = max(0, key - off - p.win_right - q0 - c0);
        if (p.win_left >= 0) hi = min(hi, key - off + p.win_left - q0 - c0 + 1);
        if (!wait_warp(bar(W_STFULL + ss), (it >> 1) & 1, ctl, 0xA3000021u)) goto done;
        if (!wait_warp(bar(W_SFULL + (kKQ ? 0 : ss)), kKQ ? (it & 1) : ((it >> 1) & 1), ctl,
                       0xA3000022u))
          goto done;
        tc_fence_after();
        {
          uint32_t sv[kWCols];
          tmem_ld32p(tl + sbuf + c0, sv);
          tmem_wait_ld();
          uint32_t pk[kWCols / 2];
#pragma unroll
          for (int e4 = 0; e4 < kWCols / 4; ++e4) {
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
              // the first half of sv holds the packed derivative 1 - tanh^2 for the dS phase
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
          tmem_st16(tl + sbuf + c0, *reinterpret_cast<uint32_t(*)[16]>(pk));
          if (kCap && kKQ) tmem_st16(tl + c0 + kWCols / 2, *reinterpret_cast<uint32_t(*)[16]>(sv));
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(W_PREADY + (kKQ ? 0 : ss)));
          if (!kKQ) mbar_arrive(bar(W_STEMPTY + ss));  // pass dV reads no Delta
        }
        if (kKQ) {
          // the dS^T tile was last read by the previous tile's dQ and dK MMAs
          if (it > 0 && !wait_warp(bar(W_DKDONE), (it - 1) & 1, ctl, 0xA3000023u)) goto done;
          if (!wait_warp(bar(W_DPFULL), it & 1, ctl, 0xA3000024u)) goto done;
          tc_fence_after();
          uint32_t dpv[kWCols], pv[kWCols / 2];
          uint32_t cv[kCap ? kWCols / 2 : 1];
          tmem_ld32p(tl + 128 + c0, dpv);
          tmem_ld16(tl + c0, *reinterpret_cast<uint32_t(*)[16]>(pv));
          if constexpr (kCap) tmem_ld16(tl + c0 + kWCols / 2, *reinterpret_cast<uint32_t(*)[16]>(cv));
          tmem_wait_ld();
          // dS^T = P^T (dP^T - Delta[query]) for this group's 32 queries -> the
          // swizzled dS^T tile (chunk c holds queries [64 c, +64); row jl is 128
          // bytes and its 16-byte unit u is stored at u ^ (jl % 8))
          const uint32_t row_base = L::kDS + (c0 / 64) * kWChunk + jl * 128;
          uint32_t pk[16];
#pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            const float4 dl = reinterpret_cast<const float4*>(dlt)[e4];
            float2 p01 = Pack<T>::unpack(pv[e4 * 2]);
            float2 p23 = Pack<T>::unpack(pv[e4 * 2 + 1]);
            if constexpr (kCap) {
              const float2 c01 = Pack<T>::unpack(cv[e4 * 2]);
              const float2 c23 = Pack<T>::unpack(cv[e4 * 2 + 1]);
              p01.x *= c01.x;
              p01.y *= c01.y;
              p23.x *= c23.x;
              p23.y *= c23.y;
            }
            const uint32_t* v = dpv + e4 * 4;
            pk[e4 * 2] = Pack<T>::two(p01.x * (__uint_as_float(v[0]) - dl.x),
                                      p01.y * (__uint_as_float(v[1]) - dl.y));
            pk[e4 * 2 + 1] = Pack<T>::two(p23.x * (__uint_as_float(v[2]) - dl.z),
                                          p23.y * (__uint_as_float(v[3]) - dl.w));
          }
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const uint32_t unit = (((c0 % 64) / 8) + qq) ^ (jl & 7);
            *reinterpret_cast<uint4*>(smem + row_base + unit * 16) =
                make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar(W_DSREADY));
            mbar_arrive(bar(W_STEMPTY + ss));
          }
        }
      }
      // ---- epilogue: this group's 64 columns of dK = scale * acc (pass dK/dQ) or dV = acc
      // (with three chunks the fourth group has none)
      if (!wait_warp(bar(W_ACCFULL), uc & 1, ctl, 0xA3000025u)) goto done;
      tc_fence_after();
      if (e0 < 64 * kNC) {
        const float mul = kKQ ? p.scale : 1.0f;
#pragma unroll 1
        for (int c = 0; c < eCols / 32; ++c) {
          uint32_t a[32];
          tmem_ld32(tl + 256 + e0 + c * 32, a);
          tmem_wait_ld();
          if (key_ok) {
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
              uint4 o;
              o.x = Pack<T>::two(__uint_as_float(a[8 * qq + 0]) * mul, __uint_as_float(a[8 * qq + 1]) * mul);
              o.y = Pack<T>::two(__uint_as_float(a[8 * qq + 2]) * mul, __uint_as_float(a[8 * qq + 3]) * mul);
              o.z = Pack<T>::two(__uint_as_float(a[8 * qq + 4]) * mul, __uint_as_float(a[8 * qq + 5]) * mul);
              o.w = Pack<T>::two(__uint_as_float(a[8 * qq + 6]) * mul, __uint_as_float(a[8 * qq + 7]) * mul);
              if (e0 + c * 32 + 8 * qq < p.head_dim)  // a padded head dimension stops early
                reinterpret_cast<uint4*>(out_row + c * 32)[qq] = o;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(W_ACCFREE));
      ++uc;
    }
  } else if (kKQ) {
    setmaxnreg_inc<kWRegDrain>();
    // ------------------------------------------------------------ dQ drain
    // Thread = query row (TMEM lane); warp q owns rows [32 q, 32 q + 32).  kNC
    // passes of 64 columns, each staged as two 32x32 fp32 boxes per warp (the
    // 128-byte swizzle) in the staging buffer and added to dQaccum by TMA
    // reduces; after the first two passes the S^T columns are free again, after
    // the last one the dP^T columns.
    const uint32_t quad = warp & 3;
    const uint32_t tl = tmem + ((quad * 32) << 16);
    const uint32_t stage_off = L::kStage + quad * 8192;
    uint32_t it = 0;
    for (uint32_t k = 0;; ++k) {
      int u;
      if (!take_unit(k, true, u)) goto done;
      if (u >= num_units) break;
      const Unit un = get_unit(p, u, G, p.win_left);
      if (un.n_iters == 0) continue;
      for (int j = 0; j < un.n_iters; ++j, ++it) {
        int h, m;
        iter_hm(un, j, G, h, m);
        const int row0 = static_cast<int>(static_cast<int64_t>(h) * p.ws_rows + un.si.ws_row0 +
                                          m * kTileRows + quad * 32);
        // one semaphore per (head, query tile, drain warp), as in the D <= 128 kernel
        int* sem = p.sem + (static_cast<int64_t>(h) * (p.ws_rows / kTileRows) +
                            un.si.ws_row0 / kTileRows + m) * 4 + quad;
        if (!wait_warp(bar(W_DQFULL), it & 1, ctl, 0xA3000031u)) goto done;
        tc_fence_after();
        uint32_t a[64];
        tmem_ld32p(tl + 0, a);
        tmem_ld32p(tl + 32, a + 32);
        tmem_wait_ld();
        if (p.deterministic) {
          int stop = 0;
          if (lane == 0) {
            // key tiles before this one that see query tile m
            const int want =
                un.n - window_first_key(m * kTileRows, un.si.sq, un.si.sk, p.win_left) / kTileRows;
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t spin = 0;; ++spin) {
              if (ld_acquire(sem) >= want) break;
              if ((spin & 15) == 15) {
                if (*abort_flag) { stop = 1; break; }
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                  raise_abort(ctl, 0xA3000033u);
                  stop = 1;
                  break;
                }
              }
            }
            fence_proxy_async_global();
          }
          if (__shfl_sync(0xffffffffu, stop, 0)) goto done;
        }
#pragma unroll 1
        for (int pass = 0; pass < kNC; ++pass) {
          if (pass > 0) {
            tmem_ld32p(tl + pass * 64, a);
            tmem_ld32p(tl + pass * 64 + 32, a + 32);
            tmem_wait_ld();
          }
          if (pass == 1 || pass == kNC - 1) {  // columns [0,128) resp. [128,64 kNC) read
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(pass == 1 ? W_DQFREE0 : W_DQFREE1));
          }
          // the staging buffer's previous reduces must have read it
          if (lane == 0) bulk_wait_read_all();
          __syncwarp();
#pragma unroll
          for (int bx = 0; bx < 2; ++bx) {
            const uint32_t box = stage_off + bx * 4096;
#pragma unroll
            for (int qq = 0; qq < 8; ++qq) {
              const uint32_t* v = a + bx * 32 + qq * 4;
              *reinterpret_cast<uint4*>(smem + box + lane * 128 + ((qq ^ (lane & 7)) * 16)) =
                  make_uint4(v[0], v[1], v[2], v[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
#pragma unroll
            for (int bx = 0; bx < 2; ++bx)
              tma_reduce_add_2d(&tmDQ, sb + stage_off + bx * 4096, pass * 64 + bx * 32, row0);
            bulk_commit();
          }
        }
        if (lane == 0 && p.deterministic) {
          bulk_wait_all();
          fence_proxy_async_global();
          __threadfence();
          red_release_add(sem, 1);
        }
        __syncwarp();
      }
    }
    if (lane == 0) bulk_wait_all();
  }

done:
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kWTmemCols);
}

template <typename T, int kPass, bool kCap, int kNC>
cudaError_t launch_wide_t(const BwdParams& p, int dtype, cudaStream_t stream,
                          const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq) {
  constexpr uint32_t smem = WSmem<kPass, kNC>::kTotal;
  constexpr int kMaxDevices = 64;
  static std::atomic<bool> attr_done[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(bwd_wide_kernel<T, kPass, kCap, kNC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // the warpgroup register split assumes exactly kWRegLaunch registers at launch
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, bwd_wide_kernel<T, kPass, kCap, kNC>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != static_cast<int>(kWRegLaunch)) return cudaErrorInvalidConfiguration;
    attr_done[dev].store(true, std::memory_order_release);
  }
  const int units = ceil_div(p.max_seqlen_k, kTileRows) * p.seq.batch * p.h_k;
  if (units <= 0) return cudaSuccess;
  const int grid = units < num_sms() ? units : num_sms();
  bwd_wide_kernel<T, kPass, kCap, kNC><<<grid, kWThreads, smem, stream>>>(p, tq, tk, tv, tdo, tdq);
  return cudaGetLastError();
}

template <typename T, bool kCap, int kNC>
cudaError_t launch_wide_passes(const BwdParams& p_in, int dtype, cudaStream_t stream) {
  const bool varlen = p_in.seq.cu_q != nullptr;
  // unit order (see get_unit): sequence major for packed batches only
  BwdParams p = p_in;
  p.unit_seq_major = varlen;
  p.unit_per = varlen ? ceil_div(p.max_seqlen_k, kTileRows) * p.h_k : p.seq.batch * p.h_k;
  const int nb = varlen ? 1 : p.seq.batch;
  const int d = p.head_dim;
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!encode_tmap_bshd(&tq, p.q, dtype, p.seq.seqlen_q, p.h_q, nb, d, kTileRows) ||
      !encode_tmap_bshd(&tk, p.k, dtype, p.seq.seqlen_k, p.h_k, nb, d, kTileRows) ||
      !encode_tmap_bshd(&tv, p.v, dtype, p.seq.seqlen_k, p.h_k, nb, d, kTileRows) ||
      !encode_tmap_bshd(&tdo, p.dout, dtype, p.seq.seqlen_q, p.h_q, nb, d, kTileRows))
    return cudaErrorInvalidValue;
  if (!encode_tmap_f32_2d(&tdq, p.dqacc, p.ws_rows * p.h_q, WD)) return cudaErrorInvalidValue;
  cudaError_t e = launch_wide_t<T, kPassDKDQ, kCap, kNC>(p, dtype, stream, tq, tk, tv, tdo, tdq);
  if (e != cudaSuccess) return e;
  return launch_wide_t<T, kPassDV, kCap, kNC>(p, dtype, stream, tq, tk, tv, tdo, tdq);
}

// three 64-column chunks per row up to D = 192, four above
template <typename T, bool kCap>
cudaError_t launch_wide_width(const BwdParams& p, int dtype, cudaStream_t stream) {
  return p.head_dim <= 192 ? launch_wide_passes<T, kCap, 3>(p, dtype, stream)
                           : launch_wide_passes<T, kCap, 4>(p, dtype, stream);
}

}  // namespace

cudaError_t launch_bwd_wide(const BwdParams& p, int dtype, cudaStream_t stream) {
  const bool cap = p.softcap > 0.f;
  if (dtype == 1)
    return cap ? launch_wide_width<__nv_bfloat16, true>(p, dtype, stream)
               : launch_wide_width<__nv_bfloat16, false>(p, dtype, stream);
  return cap ? launch_wide_width<__half, true>(p, dtype, stream)
             : launch_wide_width<__half, false>(p, dtype, stream);
}

}  // namespace attn
