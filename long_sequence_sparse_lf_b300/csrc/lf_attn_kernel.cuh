// Persistent band + global attention kernel (forward) for sm_103a.
//
// What one CTA does, per work item (see WorkItem):
//   * band tile (kind 0): 128 consecutive queries of one residue class of a
//     head (all of a head when d = 1).  It visits only the key blocks the
//     tile's windows touch (block-sparse realisation of the sliding window:
//     "Block-Sparse Attention Longformer", §2-3), masks the window edges and
//     the sequence ends inside the boundary blocks, then folds in the
//     gathered global keys as extra blocks, masking globals already in the
//     row's window (the union of Longformer explained §2's patterns under one
//     softmax, §4).  Rows of global tokens are computed but not stored.
//   * global-row tile (kind 1): up to 128 gathered global queries of a head
//     against one chunk of all L keys (Longformer explained §2, global
//     attention); writes un-normalised partials (O, m, l) that a combine
//     kernel merges.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: Q tile, then K/V blocks into a ring of stages
//   warp 1      TMEM owner and single-thread MMA issuer (tcgen05.mma):
//               S = Q K^T into TMEM, then O += P V with P read from TMEM
//   warps 2..5  softmax + epilogue; thread = query row = TMEM lane
//
// Softmax is the online form with fp32 running max m (in log2 units) and sum
// l per row.  O is only rescaled when the max grows by more than 2^8, since
// any common reference point gives the same O/l; this keeps the rescale (a
// TMEM round trip) off the common path.
//
// Every mbarrier wait is bounded in time; on expiry the kernel records
// kStatusTimeout in the device status word, all roles leave their loops,
// outstanding TMA and MMA work is drained with bounded waits and TMEM is
// freed before the CTA exits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "lf_common.cuh"
#include "lf_ptx.cuh"

namespace lf {

template <int D>
struct KCfg {
  static constexpr int NH = D / 64;                 // 128-byte swizzle atoms along D
  static constexpr uint32_t HALF = 128u * 128u;     // one [128 rows][64] bf16 atom column
  static constexpr uint32_t QB = NH * HALF;         // Q tile bytes
  static constexpr uint32_t KVB = NH * HALF;        // K (or V) block bytes
  static constexpr int NQ = 2;                      // Q tile buffers
  static constexpr int NST = (D == 64) ? 4 : 2;     // K/V stages
  // TMEM columns (512 allocated): two S buffers, two P buffers, O.
  static constexpr uint32_t TM_S0 = 0, TM_S1 = 128, TM_P0 = 256, TM_P1 = 320, TM_O = 384;
  static constexpr int NBAR = 2 * NQ + 2 * NST + 2 + 2 + 2 + 2 + 1 + 1;
  static constexpr uint32_t TILE_BYTES = NQ * QB + 2u * NST * KVB;
  static constexpr uint32_t SMEM_BYTES = TILE_BYTES + NBAR * 8 + 64 + 1024;
};

struct Waiter {
  volatile int* abort;
  unsigned* status;
  unsigned long long timeout_ns;
};

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const Waiter& w,
                                       bool honour_abort) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (honour_abort && *w.abort) return false;
      if (globaltimer_ns() - t0 > w.timeout_ns || it > (1u << 28)) {
        *w.abort = 1;
        atomicOr(w.status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, const Waiter& w) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, w, true);
}

template <int D>
__global__ void __launch_bounds__(192, 1) lf_attn_main_kernel(const __grid_constant__ MainParams p) {
  using C = KCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK = sQ + C::NQ * C::QB;
  const uint32_t sV = sK + C::NST * C::KVB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILE_BYTES);
  const uint32_t b0 = smem_u32(bars);
  auto BAR = [&](int idx) -> uint32_t { return b0 + 8u * idx; };
  // barrier index map
  const int iQF = 0, iQE = C::NQ, iKF = 2 * C::NQ, iKE = 2 * C::NQ + C::NST;
  const int iSF = 2 * C::NQ + 2 * C::NST, iSR = iSF + 2, iPF = iSR + 2, iPV = iPF + 2;
  const int iOF = iPV + 2, iDR = iOF + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::TILE_BYTES + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int q = 0; q < C::NQ; ++q) {
      mbar_init(BAR(iQF + q), 1);
      mbar_init(BAR(iQE + q), 1);
    }
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(BAR(iKF + s), 1);
      mbar_init(BAR(iKE + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(iSF + b), 1);
      mbar_init(BAR(iSR + b), 128);
      mbar_init(BAR(iPF + b), 128);
      mbar_init(BAR(iPV + b), 1);
    }
    mbar_init(BAR(iOF), 128);
    mbar_init(BAR(iDR), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
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
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  Waiter W{abort_flag, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t nb = 0;   // K/V loads armed
      uint32_t nq = 0;   // Q loads armed
      bool ok = true;
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
        const WorkItem wi = p.items[it];
        const int qb = nq % C::NQ;
        const uint32_t qu = nq / C::NQ;
        if (qu > 0 && !bwait(BAR(iQE + qb), (qu - 1) & 1, W)) { ok = false; break; }
        mbar_arrive_expect_tx(BAR(iQF + qb), C::QB);
        const uint32_t qdst = sQ + qb * C::QB;
#pragma unroll
        for (int hh = 0; hh < C::NH; ++hh) {
          if (wi.kind == 0)
            tma_load_4d(qdst + hh * C::HALF, &p.tmQ[wi.slot], BAR(iQF + qb), 64 * hh, wi.r, wi.t0,
                        wi.bh);
          else
            tma_load_3d(qdst + hh * C::HALF, &p.tmQg, BAR(iQF + qb), 64 * hh, wi.r * kBM, wi.bh);
        }
        ++nq;
        const int nbt = wi.nkb + wi.ngb;
        for (int j = 0; j < nbt; ++j) {
          const int st = nb % C::NST;
          const uint32_t su = nb / C::NST;
          if (su > 0 && !bwait(BAR(iKE + st), (su - 1) & 1, W)) { ok = false; break; }
          const uint32_t kd = sK + st * C::KVB, vd = sV + st * C::KVB;
          if (j < wi.nkb) {
            const int kpos = wi.kb0 + kBN * j;
            mbar_arrive_expect_tx(BAR(iKF + st), 2u * C::KVB);
#pragma unroll
            for (int hh = 0; hh < C::NH; ++hh) {
              if (wi.kind == 0) {
                tma_load_4d(kd + hh * C::HALF, &p.tmK[wi.slot], BAR(iKF + st), 64 * hh, wi.r, kpos,
                            wi.bh);
                tma_load_4d(vd + hh * C::HALF, &p.tmV[wi.slot], BAR(iKF + st), 64 * hh, wi.r, kpos,
                            wi.bh);
              } else {
                tma_load_3d(kd + hh * C::HALF, &p.tmKp, BAR(iKF + st), 64 * hh, kpos, wi.bh);
                tma_load_3d(vd + hh * C::HALF, &p.tmVp, BAR(iKF + st), 64 * hh, kpos, wi.bh);
              }
            }
          } else {
            const int gb = j - wi.nkb;
            mbar_arrive_expect_tx(BAR(iKF + st), 2u * C::NH * p.NGB * 128u);
#pragma unroll
            for (int hh = 0; hh < C::NH; ++hh) {
              tma_load_3d(kd + hh * C::HALF, &p.tmKg, BAR(iKF + st), 64 * hh, gb * p.NGB, wi.bh);
              tma_load_3d(vd + hh * C::HALF, &p.tmVg, BAR(iKF + st), 64 * hh, gb * p.NGB, wi.bh);
            }
          }
          ++nb;
        }
      }
      if (!ok) {
        // drain: the last load armed on every stage completes before the CTA exits
        for (uint32_t n = (nb > (uint32_t)C::NST ? nb - C::NST : 0u); n < nb; ++n)
          wait_slow(BAR(iKF + n % C::NST), (n / C::NST) & 1, W, false);
        for (uint32_t t = (nq > (uint32_t)C::NQ ? nq - C::NQ : 0u); t < nq; ++t)
          wait_slow(BAR(iQF + t % C::NQ), (t / C::NQ) & 1, W, false);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16(128, 128, false);
      const uint32_t id_g = idesc_bf16(128, p.NGB, false);
      const uint32_t id_pv = idesc_bf16(128, D, true);
      uint32_t nb = 0, nt = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++nt) {
        const WorkItem wi = p.items[it];
        const int qb = nt % C::NQ;
        if (!bwait(BAR(iQF + qb), (nt / C::NQ) & 1, W)) { ok = false; break; }
        tc_fence_after();
        const int nbt = wi.nkb + wi.ngb;
        auto issue_pv = [&](uint32_t n, int jj) -> bool {
          const int st = n % C::NST;
          const int sb = n & 1;
          if (jj == 0 && nt > 0 && !bwait(BAR(iOF), (nt - 1) & 1, W)) return false;
          if (!bwait(BAR(iPF + sb), (n >> 1) & 1, W)) return false;
          tc_fence_after();
          const int kext = (jj >= wi.nkb) ? p.NGB : kBN;
          const uint32_t pt = tmem + (sb ? C::TM_P1 : C::TM_P0);
          for (int kk = 0; kk < kext / 16; ++kk) {
            const uint64_t bdesc = sdesc_sw128(sV + st * C::KVB + kk * 2048u, C::HALF, 1024);
            mma_ts(tmem + C::TM_O, pt + kk * 8, bdesc, id_pv, (jj > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(BAR(iKE + st));
          mma_commit(BAR(iPV + sb));
          return true;
        };
        for (int j = 0; j < nbt; ++j) {
          const uint32_t n = nb + j;
          const int st = n % C::NST;
          const int sb = n & 1;
          if (!bwait(BAR(iKF + st), (n / C::NST) & 1, W)) { ok = false; break; }
          if (n >= 2 && !bwait(BAR(iSR + sb), ((n >> 1) - 1) & 1, W)) { ok = false; break; }
          tc_fence_after();
          const bool gblk = j >= wi.nkb;
          const uint32_t ds = tmem + (sb ? C::TM_S1 : C::TM_S0);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::HALF + (k & 3) * 32u;
            const uint64_t ad = sdesc_sw128(sQ + qb * C::QB + off, 16, 1024);
            const uint64_t bd = sdesc_sw128(sK + st * C::KVB + off, 16, 1024);
            mma_ss(ds, ad, bd, gblk ? id_g : id_s, k > 0 ? 1u : 0u);
          }
          mma_commit(BAR(iSF + sb));
          if (j == nbt - 1) mma_commit(BAR(iQE + qb));
          if (j > 0 && !issue_pv(n - 1, j - 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(nb + nbt - 1, nbt - 1)) { ok = false; break; }
        nb += nbt;
      }
      if (!ok) {
        mma_commit(BAR(iDR));
        wait_slow(BAR(iDR), 0, W, false);
      }
    }
  } else {
    // -------------------------------------------------- softmax + epilogue
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const float sl2 = p.sl2;
    const float NEG_INF = -__int_as_float(0x7f800000);
    uint32_t nb = 0, nt = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++nt) {
      const WorkItem wi = p.items[it];
      const bool band = wi.kind == 0;
      const int nbt = wi.nkb + wi.ngb;
      int d = 1, Lr = p.L, t = 0, i = 0, wlo = 0, whi = 0;
      if (band) {
        d = p.dil[wi.slot];
        Lr = residue_len(p.L, d, wi.r);
        t = wi.t0 + row;
        i = wi.r + d * t;
        band_window(t, p.w, Lr, wlo, whi);
      }
      float m_ref = NEG_INF, l = 0.f;
      for (int j = 0; j < nbt; ++j) {
        const uint32_t n = nb + j;
        const int sb = n & 1;
        ok = bwait(BAR(iSF + sb), (n >> 1) & 1, W);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        tc_fence_after();
        const bool gblk = j >= wi.nkb;
        const int nch = gblk ? (p.NGB >> 4) : 8;   // 16-column chunks in this block
        float s[128];
        const uint32_t sadr = tl + (sb ? C::TM_S1 : C::TM_S0);
        if (!gblk) {
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t r[32];
            tmem_ld32(sadr + c4 * 32, r);
#pragma unroll
            for (int e = 0; e < 32; ++e) s[c4 * 32 + e] = __uint_as_float(r[e]);
          }
        } else {
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            if (ch < nch) {
              uint32_t r[16];
              tmem_ld16(sadr + ch * 16, r);
#pragma unroll
              for (int e = 0; e < 16; ++e) s[ch * 16 + e] = __uint_as_float(r[e]);
            } else {
#pragma unroll
              for (int e = 0; e < 16; ++e) s[ch * 16 + e] = NEG_INF;
            }
          }
        }
        tc_fence_before();
        mbar_arrive(BAR(iSR + sb));

        // ---- masks
        if (!gblk) {
          const int kpos0 = wi.kb0 + kBN * j;
          int clo, chi;
          if (band) {
            clo = wlo - kpos0;
            chi = whi - kpos0;
          } else {
            clo = -kpos0;
            chi = p.L - 1 - kpos0;
          }
          if (clo > 0 || chi < kBN - 1) {
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = (c >= clo && c <= chi) ? s[c] : NEG_INF;
          }
        } else {
          const int gb = j - wi.nkb;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            if (ch < nch) {
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int gi = gb * p.NGB + ch * 16 + e;
                bool valid = gi < p.n_g;
                if (valid) valid = !in_band_abs(i, __ldg(p.gidx + gi), d, p.w);
                s[ch * 16 + e] = valid ? s[ch * 16 + e] : NEG_INF;
              }
            }
          }
        }

        // ---- running max (log2 units), rare rescale of O
        float mx = NEG_INF;
#pragma unroll
        for (int c = 0; c < 128; ++c) mx = fmaxf(mx, s[c]);
        const float mxs = mx * sl2;
        if (j == 0) {
          m_ref = mxs;
        } else {
          // per-row decision; the TMEM round trip below is warp-collective
          const bool need = mxs > m_ref + 8.0f;
          const float alpha = need ? (m_ref == NEG_INF ? 0.f : ex2_approx(m_ref - mxs)) : 1.f;
          if (__any_sync(0xffffffffu, need && m_ref != NEG_INF)) {
            const uint32_t np = n - 1;
            ok = bwait(BAR(iPV + (np & 1)), (np >> 1) & 1, W);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t r[32];
              tmem_ld32(tl + C::TM_O + c0, r);
#pragma unroll
              for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
              tmem_st32(tl + C::TM_O + c0, r);
            }
            tmem_st_wait();
          }
          l *= alpha;
          if (need) m_ref = mxs;
        }
        const float mu = (m_ref == NEG_INF) ? 0.f : m_ref;

        // ---- P = exp2(s*sl2 - m), row sum, pack to bf16 pairs
        uint32_t pk[64];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          if (ch < nch) {
#pragma unroll
            for (int c = ch * 16; c < ch * 16 + 16; c += 2) {
              const float p0 = ex2_approx(fmaf(s[c], sl2, -mu));
              const float p1 = ex2_approx(fmaf(s[c + 1], sl2, -mu));
              l += p0 + p1;
              pk[c >> 1] = pack_bf16x2(p0, p1);
            }
          } else {
#pragma unroll
            for (int c = ch * 16; c < ch * 16 + 16; c += 2) pk[c >> 1] = 0u;
          }
        }
        // P buffer sb was last read by PV(n-2)
        if (n >= 2) {
          ok = bwait(BAR(iPV + sb), ((n >> 1) - 1) & 1, W);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc_fence_after();
        }
        const uint32_t padr = tl + (sb ? C::TM_P1 : C::TM_P0);
        if (!gblk) {
          uint32_t a[32], b[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) { a[e] = pk[e]; b[e] = pk[32 + e]; }
          tmem_st32(padr, a);
          tmem_st32(padr + 32, b);
        } else {
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            if (2 * ch < nch) {   // 16 packed columns hold 32 keys (unused ones are 0)
              uint32_t a[16];
#pragma unroll
              for (int e = 0; e < 16; ++e) a[e] = pk[ch * 16 + e];
              tmem_st16(padr + ch * 16, a);
            }
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(iPF + sb));
      }
      if (!ok) break;

      // ---- epilogue
      const uint32_t nl = nb + nbt - 1;
      ok = bwait(BAR(iPV + (nl & 1)), (nl >> 1) & 1, W);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc_fence_after();
      float o[D];
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tl + C::TM_O + c0, r);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[c0 + e] = __uint_as_float(r[e]);
      }
      tc_fence_before();
      mbar_arrive(BAR(iOF));

      if (band) {
        const bool store = (t < Lr) && (p.is_glob[i] == 0);
        if (store) {
          const float inv = l > 0.f ? 1.0f / l : 0.f;
          const size_t base = (static_cast<size_t>(wi.bh) * p.L + i) * D;
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + base);
#pragma unroll
            for (int c = 0; c < D; c += 4)
              dst[c >> 2] = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + base);
#pragma unroll
            for (int c = 0; c < D; c += 8)
              dst[c >> 3] = make_uint4(pack_bf16x2(o[c] * inv, o[c + 1] * inv),
                                       pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv),
                                       pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv),
                                       pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv));
          }
        }
      } else {
        const int gi = wi.r * kBM + row;
        if (gi < p.n_g) {
          const size_t pidx =
              (static_cast<size_t>(wi.bh) * p.NGQ + gi) * p.n_chunks + wi.slot;
          float4* dst = reinterpret_cast<float4*>(p.part_o + pidx * D);
#pragma unroll
          for (int c = 0; c < D; c += 4) dst[c >> 2] = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
          p.part_ml[pidx * 2 + 0] = m_ref;
          p.part_ml[pidx * 2 + 1] = l;
        }
      }
      nb += nbt;
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace lf
