// Persistent band + global attention kernel (forward) for sm_103a.
//
// Each CTA owns one SM and walks its share of the work list.  A work item
// (see WorkItem) carries two 128-row query tiles, "slots" 0 and 1, that run
// side by side over one shared stream of 128-key blocks:
//   * band pair (kind 0): two neighbouring query tiles of one residue class
//     of a head.  The stream holds only the key blocks their windows touch
//     (the block-sparse realisation of the sliding window: "Block-Sparse
//     Attention Longformer", §2-3), each tile using the contiguous run it
//     needs, then the gathered global keys as extra blocks (the union of
//     Longformer explained §2's patterns under one softmax, §4).  Window
//     edges and sequence ends are masked inside the boundary blocks; globals
//     already inside a row's window are masked in the gathered block.  Rows
//     of global tokens are computed but not stored.
//   * global rows (kind 1): the gathered global queries of a head against
//     one chunk of all L keys (Longformer explained §2, global attention),
//     the two slots taking alternate blocks; each slot writes un-normalised
//     partials (O, m, l) that the combine kernel merges.
//
// Roles (384 threads = three warpgroups, one CTA per SM):
//   warps 0..3  softmax + epilogue of slot 0 (thread = query row = TMEM lane)
//   warps 4..7  softmax + epilogue of slot 1
//   warp 8      TMA producer: Q tiles of both slots, then the K/V blocks into
//               a ring of shared-memory stages
//   warp 9      TMEM owner; MMA issuer of slot 0 (tcgen05.mma): S_0 = Q_0 K^T
//               into TMEM, then O_0 += P_0 V with P_0 read from TMEM
//   warp 10     MMA issuer of slot 1
//   warp 11     idle
// While one slot's softmax warps exponentiate, the tensor core works on the
// other slot, and each SM sub-partition holds one softmax warp of each slot.
// The launch gives every thread kRegsLaunch registers; the third warpgroup
// hands most of its share to the two softmax warpgroups (setmaxnreg), which
// hold a whole 128-score row each.
//
// TMEM (512 columns): S_0, S_1 (128 fp32 columns each), P_0, P_1 (bf16 pairs,
// 64 columns each; for D = 128 they alias the first half of S_X, written
// only after S_X has been read, and the MMA warp issues S_X(next) after
// PV_X(prev), so the in-order tensor pipe never overwrites a live P), O_0,
// O_1 (D columns each).
//
// Softmax is the online form with fp32 running max m (log2 units) and sum l
// per row.  O is only rescaled when the max grows by more than 2^8: any
// common reference point gives the same O / l, and this keeps the rescale (a
// TMEM round trip) off the common path.  Warps find, per 16-key chunk of a
// block, whether all of their 32 rows see the chunk fully, not at all, or in
// part: only chunks not every row sees are masked, and a block no row of the
// warp sees is skipped (P = 0).
//
// Every mbarrier wait is bounded in time; on expiry the kernel records
// kStatusTimeout in the device status word, all roles leave their loops,
// outstanding TMA and MMA work is drained with bounded waits and TMEM is
// freed before the CTA exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <type_traits>

#include "lf_common.cuh"
#include "lf_ptx.cuh"

#ifndef LF_SLOT_OFFSET
#define LF_SLOT_OFFSET 1   // start slot 1 half a block after slot 0 (D = 64)
#endif
#ifndef LF_REGS_SM64
#define LF_REGS_SM64 216   // register split, softmax / other warpgroups (D = 64)
#define LF_REGS_OT64 72
#endif
#ifndef LF_REGS_SM128
#define LF_REGS_SM128 216  // (D = 128)
#define LF_REGS_OT128 72
#endif

namespace lf {

template <int D>
struct KCfg {
  static constexpr int NH = D / 64;                 // 128-byte swizzle atoms along D
  static constexpr uint32_t HALF = 128u * 128u;     // one [128 rows][64] bf16 atom column
  static constexpr uint32_t QB = NH * HALF;         // Q tile bytes
  static constexpr uint32_t KVB = NH * HALF;        // K (or V) block bytes
  static constexpr int NQ = (D == 64) ? 2 : 1;      // Q buffers per slot
  static constexpr int NST = (D == 64) ? 4 : 2;     // K/V stages
  static constexpr bool P_ALIAS = (D != 64);        // P_X lives in S_X's columns
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128;
  static constexpr uint32_t TM_P0 = P_ALIAS ? 0 : 256, TM_P1 = P_ALIAS ? 128 : 320;
  static constexpr uint32_t TM_O0 = P_ALIAS ? 256 : 384, TM_O1 = P_ALIAS ? 384 : 448;
  // barrier index map
  static constexpr int B_QF = 0;                    // [X * NQ + b] Q buffer full
  static constexpr int B_QE = B_QF + 2 * NQ;        // [X * NQ + b] Q buffer free
  static constexpr int B_KF = B_QE + 2 * NQ;        // [stage] K/V full
  static constexpr int B_KE = B_KF + NST;           // [stage] K/V free
  static constexpr int B_SF = B_KE + NST;           // [X] S_X written
  static constexpr int B_SR = B_SF + 2;             // [X] S_X read (free)
  static constexpr int B_PF = B_SR + 2;             // [X] P_X written
  static constexpr int B_PV = B_PF + 2;             // [X] O_X += P_X V done
  static constexpr int B_OE = B_PV + 2;             // [X] O_X read by the epilogue
  static constexpr int B_DR = B_OE + 2;             // [X] drain
  static constexpr int NBAR = B_DR + 2;
  static constexpr uint32_t TILE_BYTES = 2u * NQ * QB + 2u * NST * KVB;
  static constexpr uint32_t SMEM_BYTES = TILE_BYTES + NBAR * 8 + 64 + 1024;
  static constexpr int THREADS = 384;
  // per-thread registers of the softmax warpgroups / the third warpgroup
  static constexpr uint32_t REGS_SOFTMAX = (D == 64) ? LF_REGS_SM64 : LF_REGS_SM128;
  static constexpr uint32_t REGS_OTHER = (D == 64) ? LF_REGS_OT64 : LF_REGS_OT128;
};

// Register split (per thread): at launch, after the hand-over.  The launch
// pool is THREADS * kRegsLaunch; the split must not exceed it (the host
// checks the kernel's launch register count against kRegsLaunch).
constexpr uint32_t kRegsLaunch = 168;
static_assert(8 * KCfg<64>::REGS_SOFTMAX + 4 * KCfg<64>::REGS_OTHER <= 12 * kRegsLaunch,
              "register split (D = 64)");
static_assert(8 * KCfg<128>::REGS_SOFTMAX + 4 * KCfg<128>::REGS_OTHER <= 12 * kRegsLaunch,
              "register split (D = 128)");

struct Waiter {
  volatile int* abort;
  unsigned* status;
  uint32_t iters;   // try_wait attempts before giving up (host-computed from the timeout)
};

// Bounded wait for an mbarrier phase.  Each try_wait suspends the thread for
// at most kWaitSliceNs, so `iters` attempts bound the wait at about the
// host-set timeout.  On expiry (or when another role has given up, if
// honour_abort) it records the timeout and returns false.  Kept small: it is
// inlined at every wait site.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Waiter& w,
                                          bool honour_abort) {
  if (mbar_try_wait(bar, parity)) return true;   // already complete: no suspend hint
  for (uint32_t it = 0; it < w.iters; ++it) {
    if (mbar_try_wait_hint(bar, parity, kWaitSliceNs)) return true;
    if (honour_abort && (it & 255u) == 255u && *w.abort) return false;
  }
  *w.abort = 1;
  atomicOr(w.status, kStatusTimeout);
  return false;
}

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const Waiter& w) {
  return wait_slow(bar, parity, w, true);
}

// Wait for the asynchronous copies / products a role has in flight before
// its CTA exits after an abort.  Bounded by a fixed 2 s, independent of the
// host-set timeout: in-flight TMA and tensor-core work always completes, and
// a short host timeout must not let the CTA leave before it does.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  constexpr uint32_t kDrainIters = 2000000000u / kWaitSliceNs;
  for (uint32_t it = 0; it < kDrainIters; ++it)
    if (mbar_try_wait_hint(bar, parity, kWaitSliceNs)) return;
}

// Self-test of the bounded wait: one thread waits, with the attention
// kernel's own wait code, on an mbarrier that nothing arrives at; the wait
// runs out after wait_iters slices and records kStatusTimeout.  No copy or
// tensor-core work is in flight, so the kernel then simply returns.
__global__ void lf_selftest_wait_kernel(unsigned* status, uint32_t wait_iters) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const Waiter w{&abort_flag, status, wait_iters};
    (void)bwait(smem_u32(&bar), 0, w);
  }
}

// O_X += P_X V of one block, issued once its P is written (and, for the first
// block of an item, once the epilogue has read O_X of the previous item).
// Out of line: the issuer calls it from several places.
template <int D>
__device__ __noinline__ bool issue_pv_block(uint32_t b0, int X, uint32_t sV, uint32_t to,
                                            uint32_t tp, uint32_t id_pv, int stage, int kext,
                                            bool first, uint32_t item, uint32_t kP,
                                            const Waiter& W) {
  using C = KCfg<D>;
  auto BAR = [&](int idx) -> uint32_t { return b0 + 8u * idx; };
  if (first && item > 0 && !bwait(BAR(C::B_OE + X), (item - 1) & 1, W)) return false;
  if (!bwait(BAR(C::B_PF + X), kP & 1, W)) return false;
  tc_fence_after();
  const uint32_t vb = sV + stage * C::KVB;
  for (int kk = 0; kk < kext / 16; ++kk)
    mma_ts(to, tp + kk * 8, sdesc_sw128(vb + kk * 2048u, C::HALF, 1024), id_pv,
           (!first || kk > 0) ? 1u : 0u);
  mma_commit(BAR(C::B_PV + X));
  mma_commit(BAR(C::B_KE + stage));
  return true;
}

// BIAS: the relative-position-bias variant (p.rel_bias): each window key
// j = i + d*t of a non-global row gains rel_bias[h][t + w] on its scaled
// score.  XB: band items carry extra key blocks per tile slot (random /
// strided block patterns, p.xitem / p.xlist).  Separate instantiations, so
// the kernel without them is unchanged.
template <int D, bool BIAS = false, bool XB = false>
__global__ void __launch_bounds__(384, 1) lf_attn_main_kernel(const __grid_constant__ MainParams p) {
  using C = KCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);                 // [X][NQ] Q tiles
  const uint32_t sK = sQ + 2 * C::NQ * C::QB;         // [NST] K blocks
  const uint32_t sV = sK + C::NST * C::KVB;           // [NST] V blocks
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILE_BYTES);
  const uint32_t b0 = smem_u32(bars);
  auto BAR = [&](int idx) -> uint32_t { return b0 + 8u * idx; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::TILE_BYTES + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int q = 0; q < 2 * C::NQ; ++q) {
      mbar_init(BAR(C::B_QF + q), 1);
      mbar_init(BAR(C::B_QE + q), 1);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 2);   // one arrival per slot
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(BAR(C::B_SF + x), 1);
      mbar_init(BAR(C::B_SR + x), 128);
      mbar_init(BAR(C::B_PF + x), 128);
      mbar_init(BAR(C::B_PV + x), 1);
      mbar_init(BAR(C::B_OE + x), 128);
    }
    mbar_init(BAR(C::B_DR), 1);
    mbar_init(BAR(C::B_DR + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8 && lane == 0) {
    for (int s = 0; s < kMaxDilSlots; ++s) {
      if (p.dil[s] > 0) {
        tma_prefetch_desc(&p.tmQ[s]);
        tma_prefetch_desc(&p.tmK[s]);
        tma_prefetch_desc(&p.tmV[s]);
      }
    }
    if (p.n_g > 0) {
      tma_prefetch_desc(&p.tmKg);
      tma_prefetch_desc(&p.tmVg);
      tma_prefetch_desc(&p.tmQg);
      tma_prefetch_desc(&p.tmKp);
      tma_prefetch_desc(&p.tmVp);
    }
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  Waiter W{abort_flag, p.status, p.wait_iters};
  const int it_begin = p.cta_begin[blockIdx.x], it_end = p.cta_begin[blockIdx.x + 1];

  if (warp >= 8) {
    regs_dec<C::REGS_OTHER>();
    if (warp == 8 && lane == 0) {
    // ------------------------------------------------------------ producer
    {
      uint32_t nb = 0;                 // K/V blocks armed
      uint32_t qn[2] = {0u, 0u};       // Q loads armed per slot
      bool ok = true;
      for (int it = it_begin; it < it_end && ok; ++it) {
        const WorkItem wi = p.items[it];
        int xo = 0, nxt = 0;
        if (XB && wi.kind == 0) {
          const int4 xi = p.xitem[it];
          xo = xi.x;
          nxt = xi.y + xi.z;
        }
#pragma unroll
        for (int X = 0; X < 2; ++X) {
          if (!ok || blk_count(wi, X) == 0) continue;
          const int qb = qn[X] % C::NQ;
          const uint32_t qu = qn[X] / C::NQ;
          const int bi = X * C::NQ + qb;
          if (qu > 0 && !bwait(BAR(C::B_QE + bi), (qu - 1) & 1, W)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(C::B_QF + bi), C::QB);
          const uint32_t qdst = sQ + bi * C::QB;
#pragma unroll
          for (int hh = 0; hh < C::NH; ++hh) {
            if (wi.kind == 0)
              tma_load_4d(qdst + hh * C::HALF, &p.tmQ[wi.slot], BAR(C::B_QF + bi), 64 * hh, wi.r,
                          wi.t0 + kBM * X, wi.bh);
            else
              tma_load_3d(qdst + hh * C::HALF, &p.tmQg, BAR(C::B_QF + bi), 64 * hh, wi.r * kBM,
                          wi.bh);
          }
          ++qn[X];
        }
        if (!ok) break;
        const int nbt = wi.nkb + wi.ngb + nxt;
        for (int j = 0; j < nbt; ++j) {
          const int st = nb % C::NST;
          const uint32_t su = nb / C::NST;
          if (su > 0 && !bwait(BAR(C::B_KE + st), (su - 1) & 1, W)) { ok = false; break; }
          const uint32_t kd = sK + st * C::KVB, vd = sV + st * C::KVB;
          const bool gblk = XB ? (j >= wi.nkb && j < wi.nkb + wi.ngb) : j >= wi.nkb;
          if (!gblk) {
            // band block, or an extra block (band-type, from the list)
            const int kpos = (XB && j >= wi.nkb) ? p.xlist[xo + j - wi.nkb - wi.ngb].kpos0
                                                 : wi.kb0 + kBN * j;
            mbar_arrive_expect_tx(BAR(C::B_KF + st), 2u * C::KVB);
#pragma unroll
            for (int hh = 0; hh < C::NH; ++hh) {
              if (wi.kind == 0) {
                tma_load_4d(kd + hh * C::HALF, &p.tmK[wi.slot], BAR(C::B_KF + st), 64 * hh, wi.r,
                            kpos, wi.bh);
                tma_load_4d(vd + hh * C::HALF, &p.tmV[wi.slot], BAR(C::B_KF + st), 64 * hh, wi.r,
                            kpos, wi.bh);
              } else {
                tma_load_3d(kd + hh * C::HALF, &p.tmKp, BAR(C::B_KF + st), 64 * hh, kpos, wi.bh);
                tma_load_3d(vd + hh * C::HALF, &p.tmVp, BAR(C::B_KF + st), 64 * hh, kpos, wi.bh);
              }
            }
          } else {
            const int gb = j - wi.nkb;
            mbar_arrive_expect_tx(BAR(C::B_KF + st), 2u * C::NH * p.NGB * 128u);
#pragma unroll
            for (int hh = 0; hh < C::NH; ++hh) {
              tma_load_3d(kd + hh * C::HALF, &p.tmKg, BAR(C::B_KF + st), 64 * hh, gb * p.NGB, wi.bh);
              tma_load_3d(vd + hh * C::HALF, &p.tmVg, BAR(C::B_KF + st), 64 * hh, gb * p.NGB, wi.bh);
            }
          }
          ++nb;
        }
      }
      if (!ok) {
        // drain: the last load armed on every buffer completes before the CTA exits
        for (uint32_t n = (nb > (uint32_t)C::NST ? nb - C::NST : 0u); n < nb; ++n)
          drain_wait(BAR(C::B_KF + n % C::NST), (n / C::NST) & 1);
        for (int X = 0; X < 2; ++X)
          for (uint32_t t = (qn[X] > (uint32_t)C::NQ ? qn[X] - C::NQ : 0u); t < qn[X]; ++t)
            drain_wait(BAR(C::B_QF + X * C::NQ + t % C::NQ), (t / C::NQ) & 1);
      }
    }
    } else if ((warp == 9 || warp == 10) && lane == 0) {
    // ------------------------------------------------------- MMA issuers
    // One thread per slot (warp 9: slot 0, warp 10: slot 1) walks the CTA's
    // block stream in order: S_X(b) = Q_X K_b^T for each block the slot
    // uses and O_X += P_X V_b after its softmax wrote P_X.  Two issuing
    // threads keep the tensor core fed (issuing one tcgen05.mma costs its
    // thread tens of cycles, more than a 128x64x16 product takes).
    // K/V stage b is released by one arrival per slot: the slot's PV commit
    // if it uses the block, else a plain arrival once the block is loaded.
    {
      const int X = warp - 9;
      const uint32_t id_s = idesc_bf16(128, 128, false);
      const uint32_t id_g = idesc_bf16(128, p.NGB, false);
      const uint32_t id_pv = idesc_bf16(128, D, true);
      const uint32_t ds = tmem + (X ? C::TM_S1 : C::TM_S0);
      const uint32_t to = tmem + (X ? C::TM_O1 : C::TM_O0);
      const uint32_t tp = tmem + (X ? C::TM_P1 : C::TM_P0);
      uint32_t nb = 0, kS = 0, kP = 0, qn = 0, items = 0;
      bool pend = false, p_first = false;
      int p_stage = 0, p_kext = 0;
      uint32_t p_nb = 0, p_item = 0;
      bool ok = true;
      // Slot 1 starts half a block after slot 0 (its first S waits until slot
      // 0 has read its first S), so that the two softmax warps sharing each
      // SM sub-partition work out of phase: one exponentiates while the
      // other loads and reduces.
      if (LF_SLOT_OFFSET && !C::P_ALIAS && X == 1 && it_begin < it_end &&
          blk_count(p.items[it_begin], 0) > 0 && !bwait(BAR(C::B_SR + 0), 0, W))
        ok = false;
      // O_X += P_X V of the pending block, once its P is written
      auto issue_pv = [&]() -> bool {
        const bool r = issue_pv_block<D>(b0, X, sV, to, tp, id_pv, p_stage, p_kext, p_first,
                                         p_item, kP, W);
        ++kP;
        pend = false;
        return r;
      };
      for (int it = it_begin; it < it_end && ok; ++it) {
        const WorkItem wi = p.items[it];
        int nx0 = 0, nx1 = 0;
        if (XB && wi.kind == 0) {
          const int4 xi = p.xitem[it];
          nx0 = xi.y;
          nx1 = xi.z;
        }
        const SlotBlocks sb(wi, X, nx0, nx1);
        const int nbt = wi.nkb + wi.ngb + nx0 + nx1;
        const int cnt = sb.count();
        const bool present = sb.jlo <= sb.jhi;
        int seen = 0;
        for (int j = 0; j < nbt; ++j, ++nb) {
          const int st = nb % C::NST;
          // block nb reuses the stage of block nb - NST, which the producer
          // refills only after that block's PVs
          if (pend && p_nb + C::NST <= nb && !issue_pv()) { ok = false; break; }
          const bool use =
              XB ? sb.uses(j)
                 : (wi.kind == 0 ? present && (j >= wi.nkb || (j >= sb.jlo && j <= sb.jhi))
                                 : (j < wi.nkb && (j & 1) == X));
          if (!use) {
            if (!bwait(BAR(C::B_KF + st), (nb / C::NST) & 1, W)) { ok = false; break; }
            mbar_arrive(BAR(C::B_KE + st));
            continue;
          }
          if (C::P_ALIAS && pend && !issue_pv()) { ok = false; break; }
          const int bi = X * C::NQ + qn % C::NQ;
          if (seen == 0 && !bwait(BAR(C::B_QF + bi), (qn / C::NQ) & 1, W)) { ok = false; break; }
          if (!bwait(BAR(C::B_KF + st), (nb / C::NST) & 1, W)) { ok = false; break; }
          if (!C::P_ALIAS && kS > 0 && !bwait(BAR(C::B_SR + X), (kS - 1) & 1, W)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const bool gblk = XB ? (j >= wi.nkb && j < wi.nkb + wi.ngb) : j >= wi.nkb;
          const uint32_t qa = sQ + bi * C::QB, ka = sK + st * C::KVB;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::HALF + (k & 3) * 32u;
            mma_ss(ds, sdesc_sw128(qa + off, 16, 1024), sdesc_sw128(ka + off, 16, 1024),
                   gblk ? id_g : id_s, k > 0 ? 1u : 0u);
          }
          mma_commit(BAR(C::B_SF + X));
          const bool last = seen == cnt - 1;
          if (last) {
            mma_commit(BAR(C::B_QE + bi));
            ++qn;
          }
          if (!C::P_ALIAS && pend && !issue_pv()) { ok = false; break; }
          if (seen == 0) ++items;
          pend = true;
          p_stage = st;
          p_kext = gblk ? p.NGB : kBN;
          p_first = seen == 0;
          p_item = items - 1;
          p_nb = nb;
          ++seen;
          ++kS;
          // the slot's last block of the item: its PV goes at once, so that
          // the epilogue does not wait for the next item's loads
          if (last && !issue_pv()) { ok = false; break; }
        }
      }
      if (ok && pend && !issue_pv()) ok = false;
      if (!ok) {
        mma_commit(BAR(C::B_DR + X));
        drain_wait(BAR(C::B_DR + X), 0);
      }
    }
    }
    // teardown (this warpgroup): all TMEM traffic of the CTA is done after the barrier
    __syncwarp();
    tc_fence_before();
    cta_bar_sync();
    if (warp == 9) {
      tc_fence_after();
      tmem_dealloc(tmem, 512);
    }
  } else {
    regs_inc<C::REGS_SOFTMAX>();
    // -------------------------------------------------- softmax + epilogue
    const int X = warp >> 2;
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t tS = tl + (X ? C::TM_S1 : C::TM_S0);
    const uint32_t tP = tl + (X ? C::TM_P1 : C::TM_P0);
    const uint32_t tO = tl + (X ? C::TM_O1 : C::TM_O0);
    const float sl2 = p.sl2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const unsigned FULL = 0xffffffffu;
    uint32_t k = 0;   // blocks processed by this slot
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const WorkItem wi = p.items[it];
      const bool band = wi.kind == 0;
      int nx0 = 0, nx1 = 0;
      if (XB && band) {
        const int4 xi = p.xitem[it];
        nx0 = xi.y;
        nx1 = xi.z;
      }
      const SlotBlocks sb(wi, X, nx0, nx1);
      if (sb.count() == 0) {
        if (!band) {
          // the slot had no block of this chunk: an empty partial
          const int gi = wi.r * kBM + row;
          if (gi < p.n_g) {
            const size_t pidx = (static_cast<size_t>(wi.bh) * p.NGQ + gi) * p.n_chunks +
                                (2 * wi.slot + X);
            float4* dst = reinterpret_cast<float4*>(p.part_o + pidx * D);
#pragma unroll
            for (int c = 0; c < D; c += 4) dst[c >> 2] = make_float4(0.f, 0.f, 0.f, 0.f);
            p.part_ml[pidx * 2 + 0] = NEG_INF;
            p.part_ml[pidx * 2 + 1] = 0.f;
          }
        }
        continue;
      }
      int d = 1, i = 0, wlo = 0, whi = p.L - 1, gi = 0;
      // windows of the warp's first row and of its last valid row (every
      // row of a global-row item sees all L keys)
      int wf_lo = 0, wf_hi = p.L - 1, wl_lo = 0, wl_hi = p.L - 1;
      bool rowvalid;
      if (band) {
        d = p.dil[wi.slot];
        const int Lr = residue_len(p.L, d, wi.r);
        const int tf = wi.t0 + kBM * X + q4 * 32;
        const int t = tf + lane;
        i = wi.r + d * t;
        rowvalid = t < Lr;
        band_window(t, p.w, Lr, wlo, whi);
        band_window(tf, p.w, Lr, wf_lo, wf_hi);
        band_window(min(tf + 31, Lr - 1), p.w, Lr, wl_lo, wl_hi);
      } else {
        gi = wi.r * kBM + row;
        rowvalid = gi < p.n_g;
      }
      const bool active = __any_sync(FULL, rowvalid);
      // globals inside the row's window: G[ga .. gz) (band items only); for
      // dilated heads only those on the row's residue class are in band(i).
      // Whether the row itself is a global token (its output then comes from
      // the global-row items).  Independent loads from the prefix-count
      // table, issued here and first needed blocks later.
      int ga = 0, gz = 0;
      bool row_glob = false;
      if (band && p.n_g > 0) {
        const int a = min(max(i - d * p.w, 0), p.L), b = min(max(i + d * p.w + 1, 0), p.L);
        const int ic = min(i, p.L - 1);
        ga = __ldg(p.gcnt + a);
        gz = __ldg(p.gcnt + b);
        row_glob = __ldg(p.gcnt + ic + 1) != __ldg(p.gcnt + ic);
      }
      float m_ref = NEG_INF, l = 0.f;
      bool firstblk = true;
      for (int j = sb.first(); j >= 0; j = sb.next(j), ++k) {
        ok = bwait(BAR(C::B_SF + X), k & 1, W);
        if (!__all_sync(FULL, ok)) { ok = false; break; }
        tc_fence_after();
        if (!active) {
          // no row of this warp is a real query: keep the barrier phases only
          tc_fence_before();
          if (!C::P_ALIAS) mbar_arrive(BAR(C::B_SR + X));
          if (k > 0) {
            ok = bwait(BAR(C::B_PV + X), (k - 1) & 1, W);
            if (!__all_sync(FULL, ok)) { ok = false; break; }
          }
          mbar_arrive(BAR(C::B_PF + X));
          continue;
        }
        // Which 16-key chunks of the block the warp's rows see: by some row
        // (vis) / by every row (full).  v0..v3 hold this row's visible
        // columns; they are only read for chunks seen in part.
        uint32_t v0 = ~0u, v1 = ~0u, v2 = ~0u, v3 = ~0u;
        uint32_t vis = 0xFFu, full = 0xFFu;
        // Gathered blocks of many globals (or at D = 128, where P aliases
        // S and the previous product has completed by now) take the chunked
        // path below.  At D = 64 a narrow gathered block keeps the full-row
        // path: its exponentials cover the wait for the previous product,
        // which the short chunked path would expose.
        const bool gathered = (XB ? (j >= wi.nkb && j < wi.nkb + wi.ngb) : j >= wi.nkb) &&
                              (C::P_ALIAS || p.NGB >= 64);
        if (j < wi.nkb) {
          // band block / key chunk: the rows' windows [wlo, whi] grow with
          // the row, so the warp's union is [wlo(first), whi(last)] and its
          // intersection [wlo(last), whi(first)]: the chunk classes follow
          // from warp-uniform scalars
          const int kpos0 = wi.kb0 + kBN * j;
          vis = chunk_overlap_bits(wf_lo - kpos0, wl_hi - kpos0);
          full = chunk_inside_bits(wl_lo - kpos0, wf_hi - kpos0);
          if (vis != full) {
            const int clo = wlo - kpos0, chi1 = whi - kpos0 + 1;
            v0 = range_bits(clo, chi1, 0);
            v1 = range_bits(clo, chi1, 32);
            v2 = range_bits(clo, chi1, 64);
            v3 = range_bits(clo, chi1, 96);
          }
        } else {
          if (XB && j >= wi.nkb + wi.ngb) {
            // extra block: its keys inside [0, Lr), minus the row's window
            // (the band blocks hold those) and the global positions (the
            // gathered blocks hold those)
            const XBlock& xb = p.xlist[p.xitem[it].x + j - wi.nkb - wi.ngb];
            const uint4 gm = *reinterpret_cast<const uint4*>(xb.gm);
            const int kpos0 = xb.kpos0;
            const int nv = residue_len(p.L, d, wi.r) - kpos0;
            const int clo = wlo - kpos0, chi1 = whi - kpos0 + 1;
            v0 = range_bits(0, nv, 0) & ~range_bits(clo, chi1, 0) & ~gm.x;
            v1 = range_bits(0, nv, 32) & ~range_bits(clo, chi1, 32) & ~gm.y;
            v2 = range_bits(0, nv, 64) & ~range_bits(clo, chi1, 64) & ~gm.z;
            v3 = range_bits(0, nv, 96) & ~range_bits(clo, chi1, 96) & ~gm.w;
          } else {
            // gathered globals G[gbase + c]: not the padding, and not a global
            // already in the row's window (columns [c_lo, c_hi) hold
            // G[ga .. gz); for dilated heads only those on the row's residue
            // class are in band(i): the off bits mark the others)
            const int gbase = (j - wi.nkb) * p.NGB;
            const int c_lo = ga - gbase, c_hi = gz - gbase, nvalid = p.n_g - gbase;
            uint32_t off0 = 0, off1 = 0, off2 = 0, off3 = 0;
            if (d > 1) {
              const int cb = c_lo > 0 ? c_lo : 0, ce = c_hi < p.NGB ? c_hi : p.NGB;
#pragma unroll 1
              for (int c = cb; c < ce; ++c) {
                const int diff = __ldg(p.gidx + gbase + c) - i;
                if (diff % d != 0) {
                  const uint32_t bit = 1u << (c & 31);
                  const int wsel = c >> 5;
                  off0 |= wsel == 0 ? bit : 0u;
                  off1 |= wsel == 1 ? bit : 0u;
                  off2 |= wsel == 2 ? bit : 0u;
                  off3 |= wsel == 3 ? bit : 0u;
                }
              }
            }
            v0 = range_bits(0, nvalid, 0) & ~(range_bits(c_lo, c_hi, 0) & ~off0);
            v1 = range_bits(0, nvalid, 32) & ~(range_bits(c_lo, c_hi, 32) & ~off1);
            v2 = range_bits(0, nvalid, 64) & ~(range_bits(c_lo, c_hi, 64) & ~off2);
            v3 = range_bits(0, nvalid, 96) & ~(range_bits(c_lo, c_hi, 96) & ~off3);
          }
          if (!gathered) {
            const uint32_t o0 = __reduce_or_sync(FULL, v0), o1 = __reduce_or_sync(FULL, v1);
            const uint32_t o2 = __reduce_or_sync(FULL, v2), o3 = __reduce_or_sync(FULL, v3);
            const uint32_t a0 = __reduce_and_sync(FULL, v0), a1 = __reduce_and_sync(FULL, v1);
            const uint32_t a2 = __reduce_and_sync(FULL, v2), a3 = __reduce_and_sync(FULL, v3);
            const uint32_t ow[4] = {o0, o1, o2, o3}, aw[4] = {a0, a1, a2, a3};
            vis = 0;
            full = 0;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
              const uint32_t oh = (ow[ch >> 1] >> (16 * (ch & 1))) & 0xffffu;
              const uint32_t ah = (aw[ch >> 1] >> (16 * (ch & 1))) & 0xffffu;
              vis |= (oh != 0u ? 1u : 0u) << ch;
              full |= (ah == 0xffffu ? 1u : 0u) << ch;
            }
          }
        }
        // P_X (and O_X) are free once the previous O += P V of this slot has
        // completed; that is awaited just before the first write (for
        // D = 128, S_X(k) was issued after PV_X(k-1), so it already has)
        bool pfree = C::P_ALIAS || k == 0;
        auto await_pfree = [&]() -> bool {
          if (pfree) return true;
          const bool w_ok = bwait(BAR(C::B_PV + X), (k - 1) & 1, W);
          pfree = true;
          if (!__all_sync(FULL, w_ok)) return false;
          tc_fence_after();
          return true;
        };

        // Moves the row's reference m_ref to the block's row max mxs (log2
        // units) where that is more than 2^8 above it: any common reference
        // gives the same O / l, and O and l are rescaled by 2^(m_old - m_new).
        auto rebase = [&](float mxs) -> bool {
          const bool need = mxs > m_ref + 8.0f;
          const float alpha = need ? (m_ref == NEG_INF ? 0.f : ex2_approx(m_ref - mxs)) : 1.f;
          if (__any_sync(FULL, need && m_ref != NEG_INF) && !firstblk) {
            if (!await_pfree()) return false;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t r[32];
              tmem_ld32(tO + c0, r);
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(tO + c0, r);
            }
            tmem_st_wait();
          }
          l *= alpha;
          if (need) m_ref = mxs;
          return true;
        };

        if (gathered) {
          // Gathered global keys: the product wrote only the block's first
          // NGB columns, so the row is handled in 16-column chunks of them:
          // the row max first, then P (columns past NGB are never read by
          // O += P V, whose K extent is NGB).
          const int nch = p.NGB >> 4;
          float mx = NEG_INF;
#pragma unroll 1
          for (int c = 0; c < nch; ++c) {
            uint32_t r[16];
            tmem_ld16(tS + 16 * c, r);
            const uint32_t vw = (c < 2 ? v0 : (c < 4 ? v1 : (c < 6 ? v2 : v3))) >> (16 * (c & 1));
#pragma unroll
            for (int e = 0; e < 16; e += 2)
              mx = fmax3(mx, ((vw >> e) & 1u) ? __uint_as_float(r[e]) : NEG_INF,
                         ((vw >> (e + 1)) & 1u) ? __uint_as_float(r[e + 1]) : NEG_INF);
          }
          if (!rebase(mx * sl2)) { ok = false; break; }
          const float mu = (m_ref == NEG_INF) ? 0.f : m_ref;
          const float2 nmu = make_float2(-mu, -mu), sl2v = make_float2(sl2, sl2);
          float2 acc[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[e] = make_float2(0.f, 0.f);
          if (!await_pfree()) { ok = false; break; }
#pragma unroll 1
          for (int c = 0; c < nch; ++c) {
            uint32_t r[16];
            tmem_ld16(tS + 16 * c, r);
            const uint32_t vw = (c < 2 ? v0 : (c < 4 ? v1 : (c < 6 ? v2 : v3))) >> (16 * (c & 1));
            uint32_t pk8[8];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const float2 sv = make_float2(((vw >> e) & 1u) ? __uint_as_float(r[e]) : NEG_INF,
                                            ((vw >> (e + 1)) & 1u) ? __uint_as_float(r[e + 1]) : NEG_INF);
              const float2 x = fma2(sv, sl2v, nmu);
              const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
              acc[(e >> 1) & 3] = add2(acc[(e >> 1) & 3], pv);
              pk8[e >> 1] = pack_bf16x2(pv.x, pv.y);
            }
            tmem_st8(tP + 8 * c, pk8);
          }
          if (!C::P_ALIAS) {
            tc_fence_before();
            mbar_arrive(BAR(C::B_SR + X));
          }
          l += ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
               ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
        } else if (vis == 0u) {
          // no row of the warp sees a key of this block: P = 0
          if (!C::P_ALIAS) {
            tc_fence_before();
            mbar_arrive(BAR(C::B_SR + X));
          }
          if (!await_pfree()) { ok = false; break; }
          uint32_t z[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) z[e] = 0u;
          tmem_st32(tP, z);
          tmem_st32(tP + 32, z);
        } else {
          // ---- the whole 128-score row in one TMEM load; S_X is then free
          // for the next block's product (D = 64)
          float s[128];
          {
            uint32_t r[128];
            tmem_ld128(tS, r);
#pragma unroll
            for (int e = 0; e < 128; ++e) s[e] = __uint_as_float(r[e]);
          }
          if (!C::P_ALIAS) {
            tc_fence_before();
            mbar_arrive(BAR(C::B_SR + X));
          }
          if (BIAS && band && j < wi.nkb) {
            // rel_bias / scale added to the raw score, so that everything
            // after (max, rescale, exponentials) sees scale*q.k + rel_bias.
            // The row's 128 values start at I = kBiasPad + w + kpos0 - t in
            // the zero-padded table (t the row's residue index; the columns
            // outside the window read padding or neighbours and are masked
            // below).  Copy I % 4 of the table is shifted so that this start
            // is 16-byte aligned: 16-byte loads.
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int I = kBiasPad + p.w + wi.kb0 + kBN * j + 64 * hf - (wi.t0 + kBM * X + row);
              const int sft = I & 3;
              const float4* tp = reinterpret_cast<const float4*>(
                  p.rel_bias + static_cast<size_t>((wi.bh % p.H) * 4 + sft) * bias_row_len(p.w) +
                  (I - sft));
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const float4 bv = __ldg(tp + e);
                float* sv = s + 64 * hf + 4 * e;
                const float2 lo = add2(make_float2(sv[0], sv[1]), make_float2(bv.x, bv.y));
                const float2 hi = add2(make_float2(sv[2], sv[3]), make_float2(bv.z, bv.w));
                sv[0] = lo.x;
                sv[1] = lo.y;
                sv[2] = hi.x;
                sv[3] = hi.y;
              }
            }
          }
          // mask every chunk that not all rows see: unseen ones whole, the
          // others by the row's own bits (one straight-line path: branching
          // around unseen chunks measured slower)
          if (full != 0xFFu) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              if (!(full & (1u << c))) {
                const uint32_t vw = (vis & (1u << c)) ? (c < 2 ? v0 : (c < 4 ? v1 : (c < 6 ? v2 : v3))) : 0u;
#pragma unroll
                for (int e = 0; e < 16; ++e)
                  s[16 * c + e] = ((vw >> (16 * (c & 1) + e)) & 1u) ? s[16 * c + e] : NEG_INF;
              }
            }
          }
          const float2 sl2v = make_float2(sl2, sl2);
          // Moves the row's reference m_ref to this block's row max where
          // that is more than 2^8 above it (any common reference gives the
          // same O / l; O and l are rescaled by 2^(m_old - m_new))
          auto move_reference = [&]() -> bool {
            float m4[4] = {NEG_INF, NEG_INF, NEG_INF, NEG_INF};
#pragma unroll
            for (int e = 0; e < 128; e += 2)
              m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], s[e], s[e + 1]);
            return rebase(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2);
          };
          // a row without a reference yet (its first visible keys) takes
          // this block's max
          if (__any_sync(FULL, m_ref == NEG_INF) && !move_reference()) { ok = false; break; }
          // P = 2^(s*sl2 - m_ref), speculatively without this block's max:
          // each half's bf16 pairs and row sum (masked keys give 0).  Half 0
          // goes to TMEM while half 1 is computed.
          uint32_t pk0[32], pk1[32];
          float lb;
          {
            const float mu = (m_ref == NEG_INF) ? 0.f : m_ref;
            const float2 nmu = make_float2(-mu, -mu);
            float2 acc[4];
            exp2_half<0>(s, sl2v, nmu, pk0, acc);
            if (!await_pfree()) { ok = false; break; }
            tmem_st32(tP, pk0);
            exp2_half<64>(s, sl2v, nmu, pk1, acc);
            lb = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                 ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
          }
          // Rare: a score far above the reference (the block's sum exceeds
          // 2^16).  The reference moves to the block's max and the block's
          // P is recomputed.
          if (__any_sync(FULL, !(lb <= 65536.0f))) {
            if (!move_reference()) { ok = false; break; }
            const float mu = (m_ref == NEG_INF) ? 0.f : m_ref;
            const float2 nmu = make_float2(-mu, -mu);
            float2 acc[4];
            exp2_half<0>(s, sl2v, nmu, pk0, acc);
            tmem_st32(tP, pk0);
            exp2_half<64>(s, sl2v, nmu, pk1, acc);
            lb = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                 ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y));
          }
          tmem_st32(tP + 32, pk1);
          l += lb;
        }
        firstblk = false;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_PF + X));
      }
      if (!ok) break;

      // ---- epilogue: O_X of the item is final once its last PV completed
      ok = bwait(BAR(C::B_PV + X), (k - 1) & 1, W);
      if (!__all_sync(FULL, ok)) { ok = false; break; }
      tc_fence_after();
      if (!active) {
        tc_fence_before();
        mbar_arrive(BAR(C::B_OE + X));
        continue;
      }
      // O is read 32 columns at a time and written straight out
      if (band) {
        const bool store = rowvalid && !row_glob;
        const float inv = l > 0.f ? 1.0f / l : 0.f;
        // the row's log-sum-exp, for a backward pass: l sums 2^(s log2e - m_ref)
        if (store && p.lse != nullptr)
          p.lse[static_cast<size_t>(wi.bh) * p.L + i] = (m_ref + __log2f(l)) * 0.69314718f;
        const size_t base = (static_cast<size_t>(wi.bh) * p.L + i) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c0, r);
          if (store) {
            if (p.out_f32) {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base + c0);
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                dst[c >> 2] = make_float4(__uint_as_float(r[c]) * inv, __uint_as_float(r[c + 1]) * inv,
                                          __uint_as_float(r[c + 2]) * inv,
                                          __uint_as_float(r[c + 3]) * inv);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + base + c0);
#pragma unroll
              for (int c = 0; c < 32; c += 8)
                dst[c >> 3] = make_uint4(
                    pack_bf16x2(__uint_as_float(r[c]) * inv, __uint_as_float(r[c + 1]) * inv),
                    pack_bf16x2(__uint_as_float(r[c + 2]) * inv, __uint_as_float(r[c + 3]) * inv),
                    pack_bf16x2(__uint_as_float(r[c + 4]) * inv, __uint_as_float(r[c + 5]) * inv),
                    pack_bf16x2(__uint_as_float(r[c + 6]) * inv, __uint_as_float(r[c + 7]) * inv));
            }
          }
        }
      } else {
        const size_t pidx = (static_cast<size_t>(wi.bh) * p.NGQ + gi) * p.n_chunks +
                            (2 * wi.slot + X);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c0, r);
          if (rowvalid) {
            float4* dst = reinterpret_cast<float4*>(p.part_o + pidx * D + c0);
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              dst[c >> 2] = make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                        __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
          }
        }
        if (rowvalid) {
          p.part_ml[pidx * 2 + 0] = m_ref;
          p.part_ml[pidx * 2 + 1] = l;
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(C::B_OE + X));
    }
    // teardown (this warpgroup)
    __syncwarp();
    tc_fence_before();
    cta_bar_sync();
  }
}

}  // namespace lf
