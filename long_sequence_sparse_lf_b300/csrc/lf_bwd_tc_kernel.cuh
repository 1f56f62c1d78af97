// Backward of the sparse attention on the 5th-generation tensor core
// (tcgen05 / TMEM / TMA) for sm_103a: dq, dk, dv of sum(out * dout).
//
// With s_ij = scale q_i.k_j over the key set K(i) (band(i) ∪ G, or every key
// for a global row i), p_ij = exp(s_ij - lse_i) (lse from the forward) and
// out_i = sum_j p_ij v_j, the chain rule gives per attended pair (i, j):
//   dv_j += p_ij dout_i,   dp_ij = dout_i . v_j,
//   ds_ij = p_ij (dp_ij - delta_i),   delta_i = dout_i . out_i,
//   dq_i += scale ds_ij k_j,   dk_j += scale ds_ij q_i.
// (The pages give only the forward; this is the derivative of its plain
// definition: "Longformer explained" §2, §4.)
//
// The attended pairs (i, j) split into three classes ("Longformer explained"
// §2: sliding and dilated windows, global attention):
//   band        i not global, j in band(i);
//   global rows i global, every j;
//   global keys j global, i not global, j not in band(i).
// A band tile (kind 0) owns 128 keys of one residue class of one head and
// walks the query blocks of its keys' windows, then the gathered global
// query rows (which see every key): the band and global-row classes.  A
// global-key tile (kind 1) owns up to 128 gathered global keys of a head and
// walks a chunk of the head's query rows in natural order, keeping the
// pairs outside the key's window.
//
// band(i) is symmetric in residue space (t_j - t_i in [-w, w] within one
// residue class), so a band tile keeps K and V in shared memory and walks the
// query blocks its keys' windows reach (64 queries at D = 64, where two
// CTAs share an SM; 128 at D = 128).  Per query block, with keys on the
// TMEM lanes:
//   S^T  = K Q^T            (M = 128 keys, N = block queries, K = D)
//   dP^T = V dO^T
//   P^T  = 2^(S^T scale log2e - lse log2e), masked    (softmax warps, fp32)
//   dS^T = P^T (dP^T - delta)
//   dV  += P^T dO           (A = P^T from TMEM, as bf16; B = dO)
//   dK  += dS^T Q           (A = dS^T from TMEM)
//   dQ^T = K^T dS^T         (A = K^T: the K tile read M-major; B = dS^T,
//                            written to shared memory by the softmax warps)
// dV and dK accumulate in TMEM over the tile's query blocks; a band tile
// stores them (every key has exactly one band tile), a global-key tile,
// launched afterwards, adds its keys' with atomics.  dQ^T of each block is
// read out of TMEM and added to dq with atomics (several key tiles reach
// each query).
//
// P^T (bf16) is written over the first half of S^T's columns after the
// whole block of S^T has been read, dS^T over the first half of dP^T's
// (adjacent to S^T).  dQ^T lands in the columns from S^T's second half on:
// S^T's second half has been read, and the tensor pipe runs this thread's
// products in order, so the dV and dK products have read P^T and dS^T
// before dQ^T overwrites dS^T.  At D = 64 the M = 128 product K^T dS^T
// reads the V tile as the missing 64 rows of K^T: those rows land in TMEM
// lanes 64..127, which nothing reads (the columns' earlier contents, P^T and
// dS^T of keys 64..127, have been consumed by then).
//
// dQ^T is read out of TMEM into staging rows [query][D] fp32 in shared
// memory and added to dq by one tiled bulk reduce-add per 64 columns (through
// the fp32 residue view of dq), or per row for gathered global rows.
//
// Query rows without pairs of a block's class (global tokens in the band
// and global-key blocks, padding rows) carry -lse log2e = -inf in the
// block's statistics, so their P is 0.
//
// Roles (192 threads): warps 0-3, thread = key = TMEM lane: P, dS, the dQ
// read-out and the final dK, dV; warp 4: TMA producer; warp 5: TMEM owner
// and MMA issuer.  Every wait is bounded as in the forward kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "lf_attn_kernel.cuh"

namespace lf {

constexpr int kBtcKeys = 128;   // keys per tile (TMEM lanes)
// Global tokens up to which the prep kernel does the global-key pairs (on the
// CUDA cores, fp32), and the rows a warp takes at a time there
constexpr int kBwdPrepGlobals = 4;
constexpr int kBtcQPad = 128;   // padding of each residue class of the statistics

// A unit of the backward kernel.
//   kind 0 (band tile): keys t0 .. t0+127 of residue class r of head bh
//     (dilation slot `slot`); its query blocks are those of the keys'
//     windows, then the blocks of gathered global query rows.
//   kind 1 (global-key tile): gathered global keys t0 .. t0+127 of head bh
//     (dilation slot `slot`) against the nqb query blocks from row q0 on.
struct BtcTile {
  int bh, kind, r, t0, slot, q0, nqb, pad_;
};

struct BwdTcParams {
  CUtensorMap tmK[kMaxDilSlots];   // 4-D residue views {D, d, L/d, B*H}, box {64, 1, 128, 1}
  CUtensorMap tmV[kMaxDilSlots];
  CUtensorMap tmQ[kMaxDilSlots];   // box {64, 1, QB, 1}
  CUtensorMap tmO[kMaxDilSlots];   // dout
  CUtensorMap tmQn, tmOn;          // undilated views of q and dout (box {64, 1, QB, 1})
  CUtensorMap tmQg, tmOg;          // gathered global rows {D, NGQ, B*H}, box {64, QB, 1}
  CUtensorMap tmKg, tmVg;          // gathered global rows, box {64, 128, 1}
  CUtensorMap tmDQ[kMaxDilSlots];  // fp32 residue views of dq, box {64, 1, QB, 1}, no swizzle
  CUtensorMap tmDQn;               // the undilated fp32 view of dq
  int dil[kMaxDilSlots];
  const BtcTile* tiles;
  // per query row (-lse log2e, -delta, 0, 0), or (-inf, 0, 0, 0) where the
  // row has no pairs of the block's class; 16 bytes an entry, so that a
  // bulk copy from any entry starts 16-byte aligned
  const float4* stats;             // per (bh, r, t), residue order
  long long stats_bh;              // entries per bh
  const float4* stats_g;           // [B*H][NGQ]: the gathered global rows
  const float4* stats_n;           // [B*H][L + 128]: natural order
  const int32_t* gidx;             // [n_g] sorted global positions
  int n_g, NGQ;
  float* dq;                       // [B*H, L, D] fp32, accumulated (zeroed or set first)
  // global-key pairs done by the prep kernel (few global tokens): their dk,
  // dv sums [B*H][n_g][D], which the band tiles add to the global keys' rows;
  // null when global-key tiles run instead
  const float* dkg;
  const float* dvg;
  const uint8_t* is_glob;          // [L]
  const int32_t* gcnt;             // [L + 1] global positions below x
  float* dk;                       // [B*H, L, D] fp32, stored
  float* dv;
  int L, w;
  float scale, sl2;                // scale, scale * log2(e)
  unsigned* status;
  uint32_t wait_iters;
};

// Entries of one residue class of the statistics (Lr + a block of padding,
// so that a block starting anywhere in the class stays inside it).
__host__ __device__ __forceinline__ int btc_class_len(int L, int d) { return L / d + kBtcQPad; }

// Bits lo .. hi (clipped to 0 .. 31) set, or none when the range misses them.
__device__ __forceinline__ uint32_t range_bits32(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 31);
  if (lo > hi) return 0u;
  return (0xffffffffu >> (31 - hi)) & (0xffffffffu << lo);
}

template <int D>
struct BtcCfg {
  static constexpr int QB = (D == 64) ? 64 : 128;         // queries per block
  static constexpr int CTAS = (D == 64) ? 2 : 1;          // CTAs per SM
  static constexpr int NH = D / 64;
  static constexpr uint32_t HALF = 128u * 128u;           // [128 rows][64] bf16, SW128
  static constexpr uint32_t QHALF = QB * 128u;            // [QB rows][64] bf16
  static constexpr uint32_t TILE = NH * HALF;             // a [128 x D] bf16 tile
  static constexpr uint32_t QTILE = NH * QHALF;           // a [QB x D] bf16 tile
  static constexpr int NQB = (D == 64) ? 2 : 1;           // Q / dO / stats buffers
  static constexpr uint32_t OFF_K = 0, OFF_V = TILE, OFF_Q = 2 * TILE;
  static constexpr uint32_t OFF_O = OFF_Q + NQB * QTILE;
  // dS^T [128 keys][QB queries] bf16
  static constexpr uint32_t OFF_DS = OFF_O + NQB * QTILE;
  static constexpr uint32_t DS_TILE = (QB / 64) * HALF;
  // the dQ staging rows [QB queries][D] fp32: a buffer of their own at
  // D = 64 (the reduce-add's reads of it then overlap the next block), over
  // the dS^T buffer (grown to fit) at D = 128, where shared memory is short
  static constexpr bool STG_OWN = (D == 64);
  static constexpr uint32_t STG_BYTES = QB * D * 4u;
  static constexpr uint32_t OFF_STG = STG_OWN ? OFF_DS + DS_TILE : OFF_DS;
  static constexpr uint32_t OFF_ST =   // stats [NQB][QB] float4
      STG_OWN ? OFF_STG + STG_BYTES : OFF_DS + (DS_TILE > STG_BYTES ? DS_TILE : STG_BYTES);
  static constexpr uint32_t OFF_BAR = OFF_ST + NQB * QB * 16;
  // barriers
  // B_ST: the dQ read-out threads' staging writes (D arrivals per block)
  static constexpr int B_KV = 0, B_QF = 1, B_QE = B_QF + NQB, B_SP = B_QE + NQB, B_PD = B_SP + 1,
                       B_DQ = B_PD + 1, B_DF = B_DQ + 1, B_DR = B_DF + 1, B_ST = B_DR + 1,
                       NBAR = B_ST + 1;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns
  static constexpr uint32_t TM_S = 0, TM_DP = QB, TM_DV = 2 * QB, TM_DK = 2 * QB + D;
  static constexpr uint32_t TM_DQ = QB / 2;               // dQ^T: QB columns from here
  static constexpr uint32_t TM_COLS = (D == 64) ? 256 : 512;
  static constexpr int THREADS = 192;
  // the dQ read-out: D threads, one staging row (query) each
  static_assert(QB <= D, "one read-out thread per staging row");
  static_assert(QB % 64 == 0, "the read-out loads 64 query columns at a time");
  static_assert(SMEM_BYTES * CTAS <= 228u * 1024u && SMEM_BYTES <= 227u * 1024u,
                "shared memory of the CTAs of one SM");
};

template <int D>
__global__ void __launch_bounds__(192, BtcCfg<D>::CTAS)
    lf_bwd_band_tc_kernel(const __grid_constant__ BwdTcParams p) {
  using C = BtcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t b0 = sb + C::OFF_BAR;
  auto BAR = [&](int idx) -> uint32_t { return b0 + 8u * idx; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const float4* stats_s = reinterpret_cast<const float4*>(smem + C::OFF_ST);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BtcTile tile = p.tiles[blockIdx.x];
  const int bh = tile.bh, r = tile.r, t0 = tile.t0, slot = tile.slot;
  const bool gkeys = tile.kind == 1;
  const int d = p.dil[slot];
  const int Lr = residue_len(p.L, d, r);
  // band tile: the query blocks of the keys' windows [t0 - w, t0 + 127 + w]
  // (clipped), then the gathered global rows; global-key tile: nqb blocks
  // from q0 on
  const int qs0 = gkeys ? tile.q0 : max(t0 - p.w, 0);
  const int nqb_band =
      gkeys ? tile.nqb : (min(t0 + kBtcKeys - 1 + p.w, Lr - 1) - qs0) / C::QB + 1;
  const int nqb = nqb_band + (gkeys ? 0 : (p.n_g + C::QB - 1) / C::QB);

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_KV), 1);
    for (int b = 0; b < C::NQB; ++b) {
      mbar_init(BAR(C::B_QF + b), 1);
      mbar_init(BAR(C::B_QE + b), 1);
    }
    mbar_init(BAR(C::B_SP), 1);
    mbar_init(BAR(C::B_PD), 128);
    mbar_init(BAR(C::B_DQ), 1);
    mbar_init(BAR(C::B_DF), 128);
    mbar_init(BAR(C::B_DR), 1);
    mbar_init(BAR(C::B_ST), D);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  Waiter W{abort_flag, p.status, p.wait_iters};

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t armed = 0;
      bool ok = true;
      mbar_arrive_expect_tx(BAR(C::B_KV), 2u * C::TILE);
#pragma unroll
      for (int hh = 0; hh < C::NH; ++hh) {
        if (gkeys) {
          tma_load_3d(sb + C::OFF_K + hh * C::HALF, &p.tmKg, BAR(C::B_KV), 64 * hh, t0, bh);
          tma_load_3d(sb + C::OFF_V + hh * C::HALF, &p.tmVg, BAR(C::B_KV), 64 * hh, t0, bh);
        } else {
          tma_load_4d(sb + C::OFF_K + hh * C::HALF, &p.tmK[slot], BAR(C::B_KV), 64 * hh, r, t0, bh);
          tma_load_4d(sb + C::OFF_V + hh * C::HALF, &p.tmV[slot], BAR(C::B_KV), 64 * hh, r, t0, bh);
        }
      }
      const float4* st_src = p.stats + static_cast<long long>(bh) * p.stats_bh +
                             static_cast<long long>(r) * btc_class_len(p.L, d);
      const float4* stg_src = p.stats_g + static_cast<long long>(bh) * p.NGQ;
      const float4* stn_src = p.stats_n + static_cast<long long>(bh) * (p.L + kBtcQPad);
      for (int j = 0; j < nqb && ok; ++j) {
        const int b = j % C::NQB;
        const uint32_t u = j / C::NQB;
        if (u > 0 && !bwait(BAR(C::B_QE + b), (u - 1) & 1, W)) { ok = false; break; }
        const int qs = qs0 + C::QB * j;
        const int gq = (j - nqb_band) * C::QB;   // first gathered row of a global-row block
        mbar_arrive_expect_tx(BAR(C::B_QF + b), 2u * C::QTILE + C::QB * 16u);
        const uint32_t qd = sb + C::OFF_Q + b * C::QTILE, od = sb + C::OFF_O + b * C::QTILE;
#pragma unroll
        for (int hh = 0; hh < C::NH; ++hh) {
          if (gkeys) {
            tma_load_4d(qd + hh * C::QHALF, &p.tmQn, BAR(C::B_QF + b), 64 * hh, 0, qs, bh);
            tma_load_4d(od + hh * C::QHALF, &p.tmOn, BAR(C::B_QF + b), 64 * hh, 0, qs, bh);
          } else if (j < nqb_band) {
            tma_load_4d(qd + hh * C::QHALF, &p.tmQ[slot], BAR(C::B_QF + b), 64 * hh, r, qs, bh);
            tma_load_4d(od + hh * C::QHALF, &p.tmO[slot], BAR(C::B_QF + b), 64 * hh, r, qs, bh);
          } else {
            tma_load_3d(qd + hh * C::QHALF, &p.tmQg, BAR(C::B_QF + b), 64 * hh, gq, bh);
            tma_load_3d(od + hh * C::QHALF, &p.tmOg, BAR(C::B_QF + b), 64 * hh, gq, bh);
          }
        }
        const float4* src = gkeys ? stn_src + qs : (j < nqb_band ? st_src + qs : stg_src + gq);
        bulk_load(sb + C::OFF_ST + b * C::QB * 16, src, C::QB * 16u, BAR(C::B_QF + b));
        ++armed;
      }
      // drain: every armed load completes before the CTA exits
      drain_wait(BAR(C::B_KV), 0);
      for (uint32_t n = (armed > (uint32_t)C::NQB ? armed - C::NQB : 0u); n < armed; ++n)
        drain_wait(BAR(C::B_QF + n % C::NQB), (n / C::NQB) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_ab(128, C::QB, false, false);
      const uint32_t id_g = idesc_bf16_ab(128, D, false, true);     // dV, dK
      const uint32_t id_q = idesc_bf16_ab(128, C::QB, true, true);  // dQ^T
      const uint32_t tS = tmem + C::TM_S, tP = tmem + C::TM_DP;
      const uint32_t tV = tmem + C::TM_DV, tK = tmem + C::TM_DK;
      // K^T as an M-major A operand: 64-row groups of M (= D) lie C::HALF
      // apart; at D = 64 the second group is the V tile (rows never read)
      const uint32_t lbo_kt = (D == 128) ? C::HALF : (C::OFF_V - C::OFF_K);
      bool ok = bwait(BAR(C::B_KV), 0, W);
      for (int j = 0; j < nqb && ok; ++j) {
        const int b = j % C::NQB;
        const uint32_t u = j / C::NQB;
        if (!bwait(BAR(C::B_QF + b), u & 1, W)) { ok = false; break; }
        // S^T and dP^T (and the previous block's dQ^T) columns are free once
        // the previous block's dQ^T has been read out
        if (j > 0 && !bwait(BAR(C::B_DF), (j - 1) & 1, W)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qa = sb + C::OFF_Q + b * C::QTILE, oa = sb + C::OFF_O + b * C::QTILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32u;
          mma_ss(tS, sdesc_sw128(sb + C::OFF_K + (kk >> 2) * C::HALF + off, 16, 1024),
                 sdesc_sw128(qa + (kk >> 2) * C::QHALF + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32u;
          mma_ss(tP, sdesc_sw128(sb + C::OFF_V + (kk >> 2) * C::HALF + off, 16, 1024),
                 sdesc_sw128(oa + (kk >> 2) * C::QHALF + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR(C::B_SP));
        if (!bwait(BAR(C::B_PD), j & 1, W)) { ok = false; break; }
        tc_fence_after();
        // dV += P^T dO, dK += dS^T Q  (K = QB queries in steps of 16)
#pragma unroll
        for (int kk = 0; kk < C::QB / 16; ++kk)
          mma_ts(tV, tS + kk * 8, sdesc_sw128(oa + kk * 2048u, C::QHALF, 1024), id_g,
                 (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < C::QB / 16; ++kk)
          mma_ts(tK, tP + kk * 8, sdesc_sw128(qa + kk * 2048u, C::QHALF, 1024), id_g,
                 (j > 0 || kk > 0) ? 1u : 0u);
        // dQ^T = K^T dS^T into the QB columns from S^T's second half on
        // (K = 128 keys in 8 steps)
#pragma unroll
        for (int kk = 0; kk < kBtcKeys / 16; ++kk)
          mma_ss(tmem + C::TM_DQ, sdesc_sw128(sb + C::OFF_K + kk * 2048u, lbo_kt, 1024),
                 sdesc_sw128(sb + C::OFF_DS + kk * 2048u, C::HALF, 1024), id_q, kk > 0 ? 1u : 0u);
        mma_commit(BAR(C::B_DQ));
        mma_commit(BAR(C::B_QE + b));
      }
      if (!ok) {
        mma_commit(BAR(C::B_DR));
        drain_wait(BAR(C::B_DR), 0);
      }
    }
  } else {
    // -------------------------------------------- P, dS, dQ read-out, dK, dV
    const unsigned FULL = 0xffffffffu;
    const int row = warp * 32 + lane;   // key row = TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int tk = t0 + row;
    // the key row's position, and whether it exists
    const bool kvalid = gkeys ? tk < p.n_g : tk < Lr;
    const int kpos = gkeys ? (kvalid ? __ldg(p.gidx + tk) : 0) : r + d * tk;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float2 sl2v = make_float2(p.sl2, p.sl2);
    uint8_t* ds_s = smem + C::OFF_DS;
    bool ok = true;
    for (int j = 0; j < nqb && ok; ++j) {
      const int b = j % C::NQB;
      const uint32_t u = j / C::NQB;
      const int qs = qs0 + C::QB * j;
      const bool gblock = !gkeys && j >= nqb_band;   // gathered global query rows
      const int gq = (j - nqb_band) * C::QB;
      ok = bwait(BAR(C::B_QF + b), u & 1, W) && bwait(BAR(C::B_SP), j & 1, W);
      if (!__all_sync(FULL, ok)) { ok = false; break; }
      tc_fence_after();
      const float4* st = stats_s + b * C::QB;
      // the block's query rows that have band gradients (not a global token,
      // inside the class): bit c of qv[c >> 5].  Kept in registers: the
      // statistics buffer is refilled once this block's products are done,
      // before its dQ has been read out.
      uint32_t qv[C::QB / 32];
#pragma unroll
      for (int x = 0; x < C::QB / 32; ++x)
        qv[x] = __ballot_sync(FULL, st[32 * x + lane].x != NEG_INF &&
                                        (gblock || gkeys || qs + 32 * x + lane < Lr));
      // the columns [clo, chi] of this key's pairs in a band block (the
      // window t_q in [tk - w, tk + w]) or a global-row block (every row);
      // in a global-key block, the columns of the key's window [elo, ehi]
      // (positions on its residue class) are the ones left out
      int clo = 1, chi = 0;
      if (kvalid && !gkeys) {
        clo = gblock ? 0 : tk - p.w - qs;
        chi = gblock ? C::QB - 1 : tk + p.w - qs;
      }
      const int elo = kpos - d * p.w - qs, ehi = kpos + d * p.w - qs;
#pragma unroll 1
      for (int c4 = 0; c4 < C::QB / 32; ++c4) {
        uint32_t sr[32], pr[32];
        tmem_ld32_issue(tl + C::TM_S + 32 * c4, sr);
        tmem_ld32_issue(tl + C::TM_DP + 32 * c4, pr);
        tmem_ld_wait();
        // bit e: column 32 c4 + e holds one of this key's pairs
        uint32_t inm;
        if (!gkeys) {
          inm = range_bits32(clo - 32 * c4, chi - 32 * c4);
        } else if (!kvalid) {
          inm = 0u;
        } else if (d == 1) {
          inm = ~range_bits32(elo - 32 * c4, ehi - 32 * c4);
        } else {
          // the window's columns on the key's residue class: elo, elo + d, ..
          uint32_t ex = 0u;
          const int lo = max(elo, 32 * c4), hi = min(ehi, 32 * c4 + 31);
          for (int c = lo + ((elo - lo) % d + d) % d; c <= hi; c += d) ex |= 1u << (c - 32 * c4);
          inm = ~ex;
        }
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          // columns e, e + 1: (-lse log2e, -delta) of each
          const float2 s0 = *reinterpret_cast<const float2*>(st + 32 * c4 + e);
          const float2 s1 = *reinterpret_cast<const float2*>(st + 32 * c4 + e + 1);
          float2 x = fma2(make_float2(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])), sl2v,
                          make_float2(s0.x, s1.x));
          x.x = ((inm >> e) & 1u) ? x.x : NEG_INF;
          x.y = ((inm >> (e + 1)) & 1u) ? x.y : NEG_INF;
          const float2 pv = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          const float2 dv2 = mul2(
              pv, add2(make_float2(__uint_as_float(pr[e]), __uint_as_float(pr[e + 1])),
                       make_float2(s0.y, s1.y)));
          pp[e >> 1] = pack_bf16x2(pv.x, pv.y);
          dd[e >> 1] = pack_bf16x2(dv2.x, dv2.y);
        }
        // P^T over S^T's first half, dS^T over dP^T's (both already read)
        tmem_st16(tl + C::TM_S + 16 * c4, pp);
        tmem_st16(tl + C::TM_DP + 16 * c4, dd);
        // dS^T into shared memory, [key][query] with the 128-byte swizzle:
        // queries 64a .. 64a+63 form atom a; 16-byte chunk c of row `row`
        // sits at chunk c ^ (row & 7) of its 128-byte line
        const int a = c4 >> 1;
        uint8_t* line = ds_s + a * C::HALF + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const int chunk = (c4 & 1) * 4 + cc;
          *reinterpret_cast<uint4*>(line + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(dd[4 * cc], dd[4 * cc + 1], dd[4 * cc + 2], dd[4 * cc + 3]);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      // the previous block's reduce-add has read its staging rows before
      // this block's dQ^T overwrites them (the read-out follows this arrival
      // through the products)
      if (C::STG_OWN && threadIdx.x == 0) bulk_wait_read_all();
      tc_fence_before();
      mbar_arrive(BAR(C::B_PD));
      // ---- dQ of the block: dQ^T lanes are D's rows (warps with 32 * warp < D)
      ok = bwait(BAR(C::B_DQ), j & 1, W);
      if (!__all_sync(FULL, ok)) { ok = false; break; }
      tc_fence_after();
      if (warp * 32 < D) {
        // dQ^T (lane = element `row` of D, column = query) into the staging
        // rows (at D = 128 over the dS^T buffer, whose last reader, the dQ^T
        // product, has completed): NH halves [QB queries][64] fp32, half hh
        // holding elements 64 hh .. 64 hh + 63
        float* stg = reinterpret_cast<float*>(smem + C::OFF_STG);
        float* my = stg + (row >> 6) * (C::QB * 64) + (row & 63);
#pragma unroll 1
        for (int c2 = 0; c2 < C::QB / 32; c2 += 2) {
          uint32_t qa[32], qb[32];
          tmem_ld32_issue(tl + C::TM_DQ + 32 * c2, qa);
          tmem_ld32_issue(tl + C::TM_DQ + 32 * c2 + 32, qb);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            my[(32 * c2 + e) * 64] = p.scale * __uint_as_float(qa[e]);
            my[(32 * c2 + 32 + e) * 64] = p.scale * __uint_as_float(qb[e]);
          }
        }
        fence_proxy_async_smem();
        // every read-out thread arrives once per block; a thread that issues
        // reduce-adds waits (bounded) for all the staging writes
        mbar_arrive(BAR(C::B_ST));
        const uint32_t stg_a = smem_u32(stg);
        if (!gblock) {
          // the block's query rows are one box of the residue (or natural)
          // view of dq; rows without pairs of the block's class hold zeros,
          // rows past the end are skipped
          if (row == 0 && bwait(BAR(C::B_ST), j & 1, W)) {
#pragma unroll
            for (int hh = 0; hh < C::NH; ++hh)
              tma_reduce_add_4d(stg_a + hh * (C::QB * 64 * 4), gkeys ? &p.tmDQn : &p.tmDQ[slot],
                                64 * hh, gkeys ? 0 : r, qs, bh);
            bulk_commit_group();
          }
        } else if (bwait(BAR(C::B_ST), j & 1, W) && ((qv[row >> 5] >> (row & 31)) & 1u)) {
          // gathered global rows: one reduce-add per 64 elements of the row
          const int i = __ldg(p.gidx + gq + row);
#pragma unroll
          for (int hh = 0; hh < C::NH; ++hh)
            bulk_reduce_add_f32(p.dq + (static_cast<size_t>(bh) * p.L + i) * D + 64 * hh,
                                stg_a + (hh * (C::QB * 64) + row * 64) * 4, 256u);
          bulk_commit_group();
        }
        // before the staging rows are written again: at D = 128 the next
        // block's dS^T (so here); at D = 64 the next read-out (thread 0
        // waits before the next block's products); the gathered rows' adds
        // wait here
        if (!C::STG_OWN || gblock) bulk_wait_read_all();
      }
      tc_fence_before();
      mbar_arrive(BAR(C::B_DF));
    }
    bulk_wait_all();
    // ---- the tile's dV and dK rows: a band tile stores them (every key has
    // one band tile), a global-key tile adds to them; the warp's TMEM loads
    // stay converged, the stores are per row
    if (ok) {
      const size_t base = (static_cast<size_t>(bh) * p.L + kpos) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t vr[32], kr[32];
        tmem_ld32(tl + C::TM_DV + c0, vr);
        tmem_ld32(tl + C::TM_DK + c0, kr);
        if (kvalid && !gkeys) {
          if (p.dkg != nullptr && p.is_glob[kpos]) {
            // a global key: add its global-key pairs' sums (prep kernel)
            const size_t gb = (static_cast<size_t>(bh) * p.n_g + p.gcnt[kpos]) * D + c0;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              vr[e] = __float_as_uint(__uint_as_float(vr[e]) + p.dvg[gb + e]);
              kr[e] = __float_as_uint(__uint_as_float(kr[e]) + p.dkg[gb + e] / p.scale);
            }
          }
          float4* dvp = reinterpret_cast<float4*>(p.dv + base + c0);
          float4* dkp = reinterpret_cast<float4*>(p.dk + base + c0);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            dvp[e >> 2] = make_float4(__uint_as_float(vr[e]), __uint_as_float(vr[e + 1]),
                                      __uint_as_float(vr[e + 2]), __uint_as_float(vr[e + 3]));
            dkp[e >> 2] = make_float4(p.scale * __uint_as_float(kr[e]),
                                      p.scale * __uint_as_float(kr[e + 1]),
                                      p.scale * __uint_as_float(kr[e + 2]),
                                      p.scale * __uint_as_float(kr[e + 3]));
          }
        } else if (kvalid) {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            atomicAdd(p.dv + base + c0 + e, __uint_as_float(vr[e]));
            atomicAdd(p.dk + base + c0 + e, p.scale * __uint_as_float(kr[e]));
          }
        }
      }
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TM_COLS);
  }
}

// Inputs of the backward kernel, in one pass over the rows:
//   stats   [bh][r][t]: residue order, each class padded by kBtcQPad
//           entries; row r + d t's (-lse log2e, -delta), (-inf, 0) for a
//           global token and for the padding (band blocks);
//   stats_n [bh][i]: natural order, (-inf, 0) for global tokens and for the
//           kBtcQPad entries past L (global-key blocks);
//   stats_g [bh][g]: gathered global row g < n_g, (-inf, 0) past n_g
//           (global-row blocks);
//   qg, og, kg, vg [bh][g][:]: rows gidx[g] of q, dout, k, v, zero past n_g;
// with delta_i = dout_i . out_i (bf16 rows, fp32 sum).  A row is read by
// D / 8 threads, 16 bytes each.  The first nb0 blocks take the rows, the next
// nb1 the gathered global rows, the rest the padding entries.
//
// GK (at most kBwdPrepGlobals global tokens): the global-key pairs (j in G,
// i not global, j not in band(i)) are done here too, in fp32 on the CUDA
// cores, instead of by global-key tiles:
//   s = q_i.k_j, p = 2^(s scale log2e - lse_i log2e), ds = p (dout_i.v_j - delta_i)
//   dq_i  = scale sum_j ds k_j          (written: dq's initial value, so dq
//                                         needs no zeroing; the band tiles add)
//   dkg_j += scale ds q_i, dvg_j += p dout_i   (fp32 [B*H][n_g][D], zeroed
//                                         first; the band tiles add them to the
//                                         global keys' dk, dv rows)
// A block then takes a contiguous range of rows (`rows_per_block`, at most L,
// so at most two heads), its warps runs of 2 steps of 32 / (D / 8)
// consecutive rows whose loads they issue together (two steps keep the
// registers low enough for three blocks per SM with one global token: the
// pass is bound by latency, not bandwidth).  A row group keeps
// partial dkg, dvg sums in registers and adds them to the block's two head
// slots in shared memory when its head changes; the block adds its slots to
// dkg, dvg at the end.  GKN: the register arrays' size in global keys
// (n_g <= GKN), 0 for the plain pass.
template <int D, int GKN = 0>
__global__ void __launch_bounds__(256, GKN == 1 ? 3 : 2) lf_bwd_tc_prep_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                      const uint4* __restrict__ v, const uint4* __restrict__ out,
                                      const uint4* __restrict__ dout,
                                      const float* __restrict__ lse,
                                      const uint8_t* __restrict__ is_glob,
                                      const int32_t* __restrict__ head_dil,
                                      const int32_t* __restrict__ gidx, int n_g, int NGQ, int H,
                                      int L, long long stats_bh, long long BH,
                                      float4* __restrict__ stats, float4* __restrict__ stats_n,
                                      float4* __restrict__ stats_g, uint4* __restrict__ qg,
                                      uint4* __restrict__ og, uint4* __restrict__ kg,
                                      uint4* __restrict__ vg, int nb0, int nb1,
                                      float* __restrict__ dq = nullptr,
                                      float* __restrict__ dkg = nullptr,
                                      float* __restrict__ dvg = nullptr, int w = 0,
                                      float scale = 0.f, int rows_per_block = 0) {
  constexpr int G = D / 8;   // threads per row (a divisor of 32)
  const float INF = __int_as_float(0x7f800000);
  const float LOG2E = 1.4426950408889634f;
  const int lane = threadIdx.x & 31, sub = lane % G;
  const int part = blockIdx.x < nb0 ? 0 : blockIdx.x < nb0 + nb1 ? 1 : 2;
  const int pb = blockIdx.x - (part == 0 ? 0 : part == 1 ? nb0 : nb0 + nb1);
  const int pnb = part == 0 ? nb0 : part == 1 ? nb1 : (int)gridDim.x - nb0 - nb1;
  const long long warp0 = (pb * (long long)blockDim.x + threadIdx.x) / 32;
  const long long wstride = (long long)pnb * blockDim.x / 32;
  // delta of row `row` (all lanes of the warp take part; invalid rows give 0)
  auto delta_of = [&](bool ok, long long row) -> float {
    float s = 0.f;
    if (ok) {
      const uint4 a = out[row * G + sub], b = dout[row * G + sub];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[e]));
        const float2 y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[e]));
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
      }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
  };
  constexpr bool GK = GKN > 0;
  if (part == 0 && !GK) {
    // B*H*L < 2^31 (the entry point checks it): 32-bit row arithmetic
    const int rows = (int)(BH * L);
    for (long long w0 = warp0; w0 * (32 / G) < rows; w0 += wstride) {
      const int row = (int)(w0 * (32 / G)) + lane / G;
      const bool ok = row < rows;
      const float dl = delta_of(ok, row);
      if (ok && sub == 0) {
        const int bh = row / L;
        const int i = row - bh * L;
        const int d = head_dil[bh % H];
        const int r = i % d, t = i / d;
        const float4 o = is_glob[i] ? make_float4(-INF, 0.f, 0.f, 0.f)
                                    : make_float4(-lse[row] * LOG2E, -dl, 0.f, 0.f);
        stats[(long long)bh * stats_bh + (long long)r * btc_class_len(L, d) + t] = o;
        stats_n[(long long)bh * (L + kBtcQPad) + i] = o;
      }
    }
  } else if (part == 0) {
    constexpr int NGM = GK ? GKN : 1;
    constexpr int RPI = 32 / G;                      // rows per warp step
    constexpr int NS = 2;                            // steps per run
    constexpr int RUN = NS * RPI;
    const int rows = (int)(BH * L);
    const float sl2 = scale * LOG2E;
    // this lane's 8 elements (of D) of each global key row, per head: loaded
    // when the group's head changes
    float kj[NGM][8], vj[NGM][8], dkp[NGM][8], dvp[NGM][8];
    int cur_bh = -1;
    // the block's rows and its head slots [2][NGM][2][D]
    const int r_begin = pb * rows_per_block;
    const int r_end = min(rows, r_begin + rows_per_block);
    const int bh_first = r_begin / L;
    __shared__ float acc_s[2 * NGM * 2 * D];
    for (int x = threadIdx.x; x < 2 * NGM * 2 * D; x += blockDim.x) acc_s[x] = 0.f;
    __syncthreads();
    auto flush = [&]() {
      if (cur_bh < 0) return;
      float* slot = acc_s + (cur_bh - bh_first) * (NGM * 2 * D);
#pragma unroll
      for (int j = 0; j < NGM; ++j) {
        if (j >= n_g) break;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          atomicAdd(slot + (j * 2 + 0) * D + 8 * sub + e, dkp[j][e]);
          atomicAdd(slot + (j * 2 + 1) * D + 8 * sub + e, dvp[j][e]);
        }
      }
    };
    auto unpack8 = [](const uint4 u, float (&f)[8]) {
      const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        f[2 * e] = __uint_as_float(w4[e] << 16);
        f[2 * e + 1] = __uint_as_float(w4[e] & 0xffff0000u);
      }
    };
    const int wib = threadIdx.x / 32, nwb = blockDim.x / 32;
    for (int run0 = r_begin + wib * RUN; run0 < r_end; run0 += nwb * RUN) {
      // the run's loads first, all in flight together
      uint4 ou[NS], du[NS], qu[NS];
      float lsv[NS];
#pragma unroll
      for (int st = 0; st < NS; ++st) {
        const int row = run0 + st * RPI + lane / G;
        const bool ok = row < r_end;
        ou[st] = ok ? out[(size_t)row * G + sub] : make_uint4(0, 0, 0, 0);
        du[st] = ok ? dout[(size_t)row * G + sub] : make_uint4(0, 0, 0, 0);
        qu[st] = ok ? q[(size_t)row * G + sub] : make_uint4(0, 0, 0, 0);
        lsv[st] = ok ? lse[row] : 0.f;
      }
      // the group's first row of the run: head and position (then stepped,
      // RPI <= L rows at a time)
      int bh = (run0 + lane / G) / L, i = run0 + lane / G - bh * L;
      int d = head_dil[min(bh, (int)BH - 1) % H];
#pragma unroll
      for (int st = 0; st < NS; ++st) {
        const int row = run0 + st * RPI + lane / G;
        const bool ok = row < r_end;
        const int rr = ok ? row : 0;
        if (st > 0) {
          i += RPI;
          if (i >= L) {
            i -= L;
            ++bh;
            d = head_dil[min(bh, (int)BH - 1) % H];
          }
        }
        // all lanes take part in the group reductions below
        float of[8], df[8], qf[8];
        unpack8(ou[st], of);
        unpack8(du[st], df);
        unpack8(qu[st], qf);
        float dl = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) dl = fmaf(of[e], df[e], dl);
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
        if (ok && bh != cur_bh) {
          flush();
          cur_bh = bh;
#pragma unroll
          for (int j = 0; j < NGM; ++j) {
            const size_t gr = (static_cast<size_t>(bh) * L + (j < n_g ? gidx[j] : 0)) * G + sub;
            float t8[8];
            unpack8(j < n_g ? k[gr] : make_uint4(0, 0, 0, 0), t8);
#pragma unroll
            for (int e = 0; e < 8; ++e) kj[j][e] = t8[e];
            unpack8(j < n_g ? v[gr] : make_uint4(0, 0, 0, 0), t8);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              vj[j][e] = t8[e];
              dkp[j][e] = 0.f;
              dvp[j][e] = 0.f;
            }
          }
        }
        const bool glob = ok && is_glob[i];
        const float nl = ok ? -lsv[st] * LOG2E : 0.f;
        float dqa[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) dqa[e] = 0.f;
#pragma unroll
        for (int j = 0; j < NGM; ++j) {
          if (j >= n_g) break;
          float sd = 0.f, pd = 0.f;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            sd = fmaf(qf[e], kj[j][e], sd);
            pd = fmaf(df[e], vj[j][e], pd);
          }
#pragma unroll
          for (int o = G / 2; o > 0; o >>= 1) {
            sd += __shfl_xor_sync(0xffffffffu, sd, o);
            pd += __shfl_xor_sync(0xffffffffu, pd, o);
          }
          const int diff = gidx[j] - i;
          const bool in_band = (diff <= d * w && diff >= -d * w && (d == 1 || diff % d == 0));
          if (ok && !glob && !in_band) {
            const float pp = ex2_approx(fmaf(sd, sl2, nl));
            const float ds = pp * (pd - dl);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              dqa[e] = fmaf(scale * ds, kj[j][e], dqa[e]);
              dkp[j][e] = fmaf(scale * ds, qf[e], dkp[j][e]);
              dvp[j][e] = fmaf(pp, df[e], dvp[j][e]);
            }
          }
        }
        if (ok) {
          float4* dqr = reinterpret_cast<float4*>(dq + (size_t)rr * D + 8 * sub);
          dqr[0] = make_float4(dqa[0], dqa[1], dqa[2], dqa[3]);
          dqr[1] = make_float4(dqa[4], dqa[5], dqa[6], dqa[7]);
          if (sub == 0) {
            const int t = d == 1 ? i : i / d, r = i - t * d;
            const float4 o = glob ? make_float4(-INF, 0.f, 0.f, 0.f) : make_float4(nl, -dl, 0.f, 0.f);
            stats[(long long)bh * stats_bh + (long long)r * btc_class_len(L, d) + t] = o;
            stats_n[(long long)bh * (L + kBtcQPad) + i] = o;
          }
        }
      }
    }
    flush();
    __syncthreads();
    // the block's head slots to dkg, dvg
    for (int x = threadIdx.x; x < 2 * NGM * 2 * D; x += blockDim.x) {
      const int sl = x / (NGM * 2 * D), rem = x - sl * (NGM * 2 * D);
      const int j = rem / (2 * D), kv = (rem / D) & 1, e = rem % D;
      const int bh = bh_first + sl;
      if (j < n_g && bh < BH && bh * L < r_end) {
        float* dst = (kv == 0 ? dkg : dvg) + (static_cast<size_t>(bh) * n_g + j) * D + e;
        atomicAdd(dst, acc_s[x]);
      }
    }
  } else if (part == 1) {
    const long long grows = BH * NGQ;
    for (long long w0 = warp0; w0 * (32 / G) < grows; w0 += wstride) {
      const long long gr = w0 * (32 / G) + lane / G;
      const bool in = gr < grows;
      const long long bh = in ? gr / NGQ : 0;
      const int g = in ? (int)(gr - bh * NGQ) : 0;
      const bool ok = in && g < n_g;
      const long long row = ok ? bh * L + gidx[g] : 0;
      const float dl = delta_of(ok, row);
      if (in) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        const long long dst = gr * G + sub;
        qg[dst] = ok ? q[row * G + sub] : z;
        og[dst] = ok ? dout[row * G + sub] : z;
        kg[dst] = ok ? k[row * G + sub] : z;
        vg[dst] = ok ? v[row * G + sub] : z;
        if (sub == 0)
          stats_g[gr] = ok ? make_float4(-lse[row] * LOG2E, -dl, 0.f, 0.f)
                           : make_float4(-INF, 0.f, 0.f, 0.f);
      }
    }
  } else {
    // per bh: d classes of kBtcQPad entries past each class's end, and
    // kBtcQPad entries past L in natural order
    const float4 pad = make_float4(-INF, 0.f, 0.f, 0.f);
    for (long long x = pb * (long long)blockDim.x + threadIdx.x; x < BH * 2 * kBtcQPad;
         x += (long long)pnb * blockDim.x) {
      const long long bh = x / (2 * kBtcQPad);
      const int e = (int)(x - bh * 2 * kBtcQPad);
      if (e >= kBtcQPad) {
        stats_n[bh * (L + kBtcQPad) + L + (e - kBtcQPad)] = pad;
      } else {
        const int d = head_dil[bh % H];
        const int cl = btc_class_len(L, d);
        for (int r = 0; r < d; ++r) stats[bh * stats_bh + (long long)r * cl + (cl - kBtcQPad) + e] = pad;
      }
    }
  }
}

}  // namespace lf
