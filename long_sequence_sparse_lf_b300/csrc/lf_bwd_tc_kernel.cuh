// Backward of the sparse attention, band pairs, on the 5th-generation tensor
// core (tcgen05 / TMEM / TMA) for sm_103a.
//
// The pairs (i, j) with i not a global token and j in band(i) ("Longformer
// explained" §2: the sliding and dilated windows) are the bulk of the
// backward.  band(i) is symmetric in residue space (t_j - t_i in [-w, w]
// within one residue class), so one CTA owns a tile of 128 keys of one
// residue class of one head, keeps K and V in shared memory, and walks the
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
// dV and dK accumulate in TMEM over the tile's query blocks and are stored
// once (every key has exactly one band tile, so plain stores; the global
// classes add to them afterwards).  dQ^T of each block is read out of TMEM
// and added to dq with atomics (several key tiles reach each query).
//
// P^T (bf16) is written over the first half of S^T's columns after the
// whole block of S^T has been read, dS^T over the first half of dP^T's
// (adjacent to S^T).  dQ^T lands in the columns from S^T's second half on:
// S^T's second half has been read, and the tensor pipe runs this thread's
// products in order, so the dV and dK products have read P^T and dS^T
// before dQ^T overwrites dS^T.  At D = 64 the M = 128 product K^T dS^T
// reads a zero tile as the missing 64 rows of K^T.
//
// Query rows that are global tokens (their gradients come from the
// global-row class) and padding rows past the residue class's end carry
// lse = +inf in the per-block statistics, so their P is 0.
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
constexpr int kBtcQPad = 128;   // padding of each residue class of the statistics

struct BwdTcParams {
  CUtensorMap tmK[kMaxDilSlots];   // 4-D residue views {D, d, L/d, B*H}, box {64, 1, 128, 1}
  CUtensorMap tmV[kMaxDilSlots];
  CUtensorMap tmQ[kMaxDilSlots];
  CUtensorMap tmO[kMaxDilSlots];   // dout
  int dil[kMaxDilSlots];
  const int4* tiles;               // (bh, residue r, first key t0, dilation slot)
  const float4* stats;             // per (bh, r, t): (lse log2e or +inf, delta, 0, 0)
  long long stats_bh;              // entries per bh
  float* dq;                       // [B*H, L, D] fp32, accumulated (zeroed first)
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
  static constexpr uint32_t OFF_DS = OFF_O + NQB * QTILE; // dS^T [128 keys][QB queries] bf16
  static constexpr uint32_t OFF_Z = OFF_DS + (QB / 64) * HALF;   // zero tile (D = 64)
  static constexpr uint32_t OFF_ST = OFF_Z + (D == 64 ? HALF : 0);   // stats [NQB][QB] float4
  static constexpr uint32_t OFF_BAR = OFF_ST + NQB * QB * 16;
  // barriers
  static constexpr int B_KV = 0, B_QF = 1, B_QE = B_QF + NQB, B_SP = B_QE + NQB, B_PD = B_SP + 1,
                       B_DQ = B_PD + 1, B_DF = B_DQ + 1, B_DR = B_DF + 1, NBAR = B_DR + 1;
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;
  // TMEM columns
  static constexpr uint32_t TM_S = 0, TM_DP = QB, TM_DV = 2 * QB, TM_DK = 2 * QB + D;
  static constexpr uint32_t TM_DQ = QB / 2;               // dQ^T: QB columns from here
  static constexpr uint32_t TM_COLS = (D == 64) ? 256 : 512;
  static constexpr int THREADS = 192;
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
  const int4 tile = p.tiles[blockIdx.x];
  const int bh = tile.x, r = tile.y, t0 = tile.z, slot = tile.w;
  const int d = p.dil[slot];
  const int Lr = residue_len(p.L, d, r);
  // the query blocks: the keys' windows [t0 - w, t0 + 127 + w], clipped
  const int qs0 = max(t0 - p.w, 0);
  const int qend = min(t0 + kBtcKeys - 1 + p.w, Lr - 1);
  const int nqb = (qend - qs0) / C::QB + 1;

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
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  if (D == 64 && warp < 4) {
    // the zero rows standing in for K^T's rows 64..127 in the M = 128 dQ product
    uint4* z = reinterpret_cast<uint4*>(smem + C::OFF_Z);
    for (int x = threadIdx.x; x < (int)(C::HALF / 16); x += 128) z[x] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
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
        tma_load_4d(sb + C::OFF_K + hh * C::HALF, &p.tmK[slot], BAR(C::B_KV), 64 * hh, r, t0, bh);
        tma_load_4d(sb + C::OFF_V + hh * C::HALF, &p.tmV[slot], BAR(C::B_KV), 64 * hh, r, t0, bh);
      }
      const float4* st_src = p.stats + static_cast<long long>(bh) * p.stats_bh +
                             static_cast<long long>(r) * btc_class_len(p.L, d);
      for (int j = 0; j < nqb && ok; ++j) {
        const int b = j % C::NQB;
        const uint32_t u = j / C::NQB;
        if (u > 0 && !bwait(BAR(C::B_QE + b), (u - 1) & 1, W)) { ok = false; break; }
        const int qs = qs0 + C::QB * j;
        mbar_arrive_expect_tx(BAR(C::B_QF + b), 2u * C::QTILE + C::QB * 16u);
#pragma unroll
        for (int hh = 0; hh < C::NH; ++hh) {
          tma_load_4d(sb + C::OFF_Q + b * C::QTILE + hh * C::QHALF, &p.tmQ[slot],
                      BAR(C::B_QF + b), 64 * hh, r, qs, bh);
          tma_load_4d(sb + C::OFF_O + b * C::QTILE + hh * C::QHALF, &p.tmO[slot],
                      BAR(C::B_QF + b), 64 * hh, r, qs, bh);
        }
        bulk_load(sb + C::OFF_ST + b * C::QB * 16, st_src + qs, C::QB * 16u, BAR(C::B_QF + b));
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
      // apart; at D = 64 the second group is the zero tile
      const uint32_t lbo_kt = (D == 128) ? C::HALF : (C::OFF_Z - C::OFF_K);
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
    const bool kvalid = tk < Lr;
    const float NEG_INF = -__int_as_float(0x7f800000);
    uint8_t* ds_s = smem + C::OFF_DS;
    bool ok = true;
    for (int j = 0; j < nqb && ok; ++j) {
      const int b = j % C::NQB;
      const uint32_t u = j / C::NQB;
      const int qs = qs0 + C::QB * j;
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
        qv[x] = __ballot_sync(FULL, st[32 * x + lane].x != __int_as_float(0x7f800000) &&
                                        qs + 32 * x + lane < Lr);
      // this key's queries: t_q in [tk - w, tk + w], as block columns
      const int clo = kvalid ? tk - p.w - qs : 1, chi = kvalid ? tk + p.w - qs : 0;
#pragma unroll 1
      for (int c4 = 0; c4 < C::QB / 32; ++c4) {
        uint32_t sr[32], pr[32];
        tmem_ld32(tl + C::TM_S + 32 * c4, sr);
        tmem_ld32(tl + C::TM_DP + 32 * c4, pr);
        uint32_t pp[16], dd[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pv[2], dv2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int col = 32 * c4 + e + h;
            const float4 sv = st[col];
            const bool in = col >= clo && col <= chi;
            const float x = in ? fmaf(__uint_as_float(sr[e + h]), p.sl2, -sv.x) : NEG_INF;
            pv[h] = ex2_approx(x);
            dv2[h] = pv[h] * (__uint_as_float(pr[e + h]) - sv.y);
          }
          pp[e >> 1] = pack_bf16x2(pv[0], pv[1]);
          dd[e >> 1] = pack_bf16x2(dv2[0], dv2[1]);
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
      tc_fence_before();
      mbar_arrive(BAR(C::B_PD));
      // ---- dQ of the block: dQ^T lanes are D's rows (warps with 32 * warp < D)
      ok = bwait(BAR(C::B_DQ), j & 1, W);
      if (!__all_sync(FULL, ok)) { ok = false; break; }
      tc_fence_after();
      if (warp * 32 < D) {
        const int dcol = row;   // lane = row of dQ^T = element of D
#pragma unroll 1
        for (int c2 = 0; c2 < C::QB / 32; ++c2) {
          uint32_t qr[32];
          tmem_ld32(tl + C::TM_DQ + 32 * c2, qr);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int col = 32 * c2 + e;
            // global query rows and padding rows: no contribution (and no
            // valid position)
            if ((qv[col >> 5] >> (col & 31)) & 1u) {
              const size_t i = static_cast<size_t>(r) + static_cast<size_t>(d) * (qs + col);
              atomicAdd(p.dq + (static_cast<size_t>(bh) * p.L + i) * D + dcol,
                        p.scale * __uint_as_float(qr[e]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(C::B_DF));
    }
    // ---- the tile's dV and dK rows (every key has one band tile: stored);
    // the warp's TMEM loads stay converged, the stores are per row
    if (ok) {
      const size_t base = (static_cast<size_t>(bh) * p.L + r + static_cast<size_t>(d) * tk) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t vr[32], kr[32];
        tmem_ld32(tl + C::TM_DV + c0, vr);
        tmem_ld32(tl + C::TM_DK + c0, kr);
        if (kvalid) {
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

// Per (bh, residue class, t) statistics of the band kernel's query rows:
// (lse log2e, delta) of row i = r + d t, or lse = +inf for a global token
// or a padding entry past the class's end (their band gradients are 0).
__global__ void lf_bwd_tc_stats_kernel(const float* __restrict__ lse,
                                       const float* __restrict__ delta,
                                       const uint8_t* __restrict__ is_glob,
                                       const int32_t* __restrict__ head_dil, int H, int L,
                                       long long stats_bh, long long total, float4* __restrict__ stats) {
  const float INF = __int_as_float(0x7f800000);
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const long long bh = x / stats_bh;
    const int e = (int)(x - bh * stats_bh);
    const int d = head_dil[bh % H];
    const int cl = btc_class_len(L, d);
    float4 o = make_float4(INF, 0.f, 0.f, 0.f);
    if (e < d * cl) {
      const int r = e / cl, t = e - r * cl;
      if (t < residue_len(L, d, r)) {
        const int i = r + d * t;
        if (!is_glob[i]) o = make_float4(lse[bh * L + i] * 1.4426950408889634f, delta[bh * L + i], 0.f, 0.f);
      }
    }
    stats[x] = o;
  }
}

}  // namespace lf
