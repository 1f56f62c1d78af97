// Dense products of the Longformer layer forward ("基于Block-Sparse
// Attention的Longformer" (block-sparse Longformer), §6 "Longformer的整体架构":
// the q, k, v linear maps and the feed-forward map) on the 5th-generation
// tensor core (tcgen05 / TMEM / TMA) for sm_103a, with the steps that follow
// each product fused into its epilogue.
//
//   C[M, N] = A[M, K] B[N, K]^T      A: activations (token rows), B: weights
//                                    as nn.Linear stores them; bf16 inputs,
//                                    fp32 accumulation in TMEM
//
// EPI 0 (q, k, v): q, k, v = bf16(C + b), written straight into three
//   [B, H, L, D] tensors (column n: part n / hidden, head (n % hidden) / D).
// EPI 1 (feed-forward): y = bf16(LN(x1 + C + b)), LN over the hidden axis
//   (biased variance, gamma and beta).  A row's hidden columns are split over
//   a cluster of CTAs (NT columns each, the TMEM width of one CTA).  Each CTA
//   takes its columns' mean and centred sum of squares M2 (per 32-column
//   chunk, merged chunk by chunk with the pairwise update of Chan, Golub and
//   LeVeque); the CTAs exchange (mean, M2) through distributed shared memory
//   once and merge them the same way.
//
// A CTA owns one 128 x NT output tile: 128 rows on the TMEM lanes, NT fp32
// columns.  Roles (192 threads): warps 0-3 the epilogue (thread = row = TMEM
// lane), warp 4 the TMA producer (A and B k-blocks of 64 into a ring of
// STAGES stages, 128-byte swizzle), warp 5 the TMEM owner and MMA issuer (one
// thread: four 128 x NT x 16 products per k-block).  Every mbarrier wait is
// bounded as in the attention kernel; on expiry the kernel records the status
// bit, drains what it has in flight, still takes part in the cluster's
// barriers and frees TMEM.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "lf_attn_kernel.cuh"

namespace lf {

constexpr int kGemmBM = 128;          // rows per tile (TMEM lanes)
constexpr int kGemmBK = 64;           // K per stage: one 128-byte swizzle atom of bf16
constexpr int kGemmMaxCluster = 8;    // CTAs sharing a row in the LayerNorm epilogue

// NT: columns per tile; MH: 128-row halves per tile (MH = 2: two M = 128
// accumulators side by side in TMEM, sharing each B k-block); ST: pipeline
// stages (0: the default for the shape).  Three CTAs fit an SM when their
// shared memory allows (the feed-forward map's two-stage build).
template <int NT, int MH = 1, int ST = 0>
struct GemmCfg {
  static_assert(NT == 64 || NT == 128 || NT == 256, "tile width");
  static_assert(MH == 1 || MH == 2, "tile height");
  static constexpr int BM = kGemmBM * MH;              // rows per tile
  static constexpr int STAGES =
      ST > 0 ? ST : ((MH == 2) ? 3 : ((NT == 256) ? 4 : (NT == 128 ? 3 : 4)));
  static constexpr uint32_t A_BYTES = BM * 128;        // BM rows x 64 bf16
  static constexpr uint32_t B_BYTES = NT * 128;        // NT rows x 64 bf16
  static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
  static constexpr uint32_t OFF_RED = STAGES * STAGE;  // [2][kGemmMaxCluster][128] fp32
  static constexpr uint32_t OFF_VEC = OFF_RED + 2 * kGemmMaxCluster * kGemmBM * 4;  // [3][NT] fp32
  static constexpr uint32_t OFF_BAR = OFF_VEC + 3 * NT * 4;
  // B_VEC: the tile's bias (gamma, beta) columns in shared memory; B_STG: the
  // staging rows; 128 arrivals each, one per epilogue thread
  static constexpr int B_FULL = 0, B_EMPTY = STAGES, B_ACC = 2 * STAGES, B_DR = B_ACC + 1,
                       B_VEC = B_DR + 1, B_STG = B_VEC + 1, NBAR = B_STG + 1;
  // the output staging rows ([128][NT] bf16) fit in the consumed stages
  static_assert(BM * NT * 2 <= STAGES * STAGE, "staging rows");
  static constexpr uint32_t SMEM_BYTES = OFF_BAR + NBAR * 8 + 16 + 1024;
  static constexpr int CTAS =
      (3 * (SMEM_BYTES + 1024) <= 228u * 1024u) ? 3 : ((2 * SMEM_BYTES <= 228u * 1024u) ? 2 : 1);
  static constexpr uint32_t TM_COLS = NT * MH;         // a power of two >= 32
  static constexpr int THREADS = 192;
  static_assert(SMEM_BYTES <= 227u * 1024u, "shared memory of one CTA");
};

struct GemmParams {
  CUtensorMap tmA;        // A [M, K] bf16: dims {K, M}, box {64, 128}, SW128
  CUtensorMap tmB;        // B [N, K] bf16: dims {K, N}, box {64, NT}, SW128
  // outputs, box {64, 128(, 1)}, SW128: EPI 0 q, k, v as {D, L, B*H};
  // EPI 1 y as {hidden, M} (tmO[0])
  CUtensorMap tmO[3];
  int M, K, hidden;
  const float* bias;      // [N]
  // EPI 0
  uint16_t* qkv;          // three consecutive [B, H, L, D] bf16 tensors
  int B, H, L, D;
  // EPI 1
  const uint16_t* resid;  // x1 [M, hidden] bf16
  const float* ln;        // gamma [hidden] then beta [hidden]
  uint16_t* out;          // [M, hidden] bf16
  float eps;
  unsigned* status;
  uint32_t wait_iters;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Tiled bulk stores shared -> global (rows or columns outside the tensor
// are skipped; coordinates non-negative, the innermost a multiple of 16
// bytes), tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* m, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::
                   "l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::
          "l"(reinterpret_cast<uint64_t>(m)), "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return n;
}
// Every thread of every CTA of the cluster arrives, then waits: shared-memory
// writes before it (local or remote) are visible to all of them after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Stores v at the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

template <int NT, int EPI, int MH = 1, int ST = 0>
__global__ void __launch_bounds__(192, GemmCfg<NT, MH, ST>::CTAS)
    lf_gemm_tc_kernel(const __grid_constant__ GemmParams p) {
  using C = GemmCfg<NT, MH, ST>;
  static_assert(EPI == 0 || MH == 1, "the LayerNorm epilogue takes 128-row tiles");
  constexpr int BM = C::BM;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  const uint32_t b0 = sb + C::OFF_BAR;
  auto BAR = [&](int idx) -> uint32_t { return b0 + 8u * idx; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + C::NBAR * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* vec = reinterpret_cast<float*>(smem + C::OFF_VEC);   // bias | gamma | beta

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * NT;
  // EPI 0: row tiles per batch element (tile = 128 positions l0.. of one b,
  // so that its rows are one box of the [B, H, L, D] outputs); EPI 1: rows
  // m0.. of [M, hidden]
  const int tiles_b = (p.L + BM - 1) / BM;
  const int b_t = (EPI == 0) ? static_cast<int>(blockIdx.y) / tiles_b : 0;
  const int l0 = (EPI == 0) ? (static_cast<int>(blockIdx.y) - b_t * tiles_b) * BM : 0;
  const int m0 = (EPI == 0) ? b_t * p.L + l0 : static_cast<int>(blockIdx.y) * BM;
  // rows of the tile that are outputs
  const int rows_out = (EPI == 0) ? min(BM, p.L - l0) : min(BM, p.M - m0);
  const int KB = p.K / kGemmBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(BAR(C::B_FULL + s), 1);
      mbar_init(BAR(C::B_EMPTY + s), 1);
    }
    mbar_init(BAR(C::B_ACC), 1);
    mbar_init(BAR(C::B_DR), 1);
    mbar_init(BAR(C::B_VEC), 128);
    mbar_init(BAR(C::B_STG), 128);
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

  bool ok = true;
  // EPI 1: this row's mean and M2 over this CTA's columns, then over the row
  float mean = 0.f, m2 = 0.f;
  const int row = warp * 32 + lane;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);
  const int m = m0 + row;
  const bool valid = row < rows_out;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t armed = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % C::STAGES;
        const uint32_t u = kb / C::STAGES;
        if (u > 0 && !bwait(BAR(C::B_EMPTY + s), (u - 1) & 1, W)) break;
        const uint32_t st = sb + s * C::STAGE;
        mbar_arrive_expect_tx(BAR(C::B_FULL + s), C::STAGE);
        tma_load_2d(st, &p.tmA, BAR(C::B_FULL + s), kGemmBK * kb, m0);
        tma_load_2d(st + C::A_BYTES, &p.tmB, BAR(C::B_FULL + s), kGemmBK * kb, n0);
        ++armed;
      }
      // every armed load completes before the CTA exits
      for (uint32_t n = (armed > (uint32_t)C::STAGES ? armed - C::STAGES : 0u); n < armed; ++n)
        drain_wait(BAR(C::B_FULL + n % C::STAGES), (n / C::STAGES) & 1);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_ab(kGemmBM, NT, false, false);
      bool iok = true;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % C::STAGES;
        const uint32_t u = kb / C::STAGES;
        if (!bwait(BAR(C::B_FULL + s), u & 1, W)) { iok = false; break; }
        tc_fence_after();
        const uint32_t st = sb + s * C::STAGE;
#pragma unroll
        for (int kk = 0; kk < kGemmBK / 16; ++kk)
#pragma unroll
          for (int h = 0; h < MH; ++h)
            mma_ss(tmem + h * NT, sdesc_sw128(st + h * (kGemmBM * 128) + kk * 32u, 16, 1024),
                   sdesc_sw128(st + C::A_BYTES + kk * 32u, 16, 1024), idesc,
                   (kb > 0 || kk > 0) ? 1u : 0u);
        mma_commit(BAR(C::B_EMPTY + s));
      }
      if (iok) {
        mma_commit(BAR(C::B_ACC));
      } else {
        mma_commit(BAR(C::B_DR));
        drain_wait(BAR(C::B_DR), 0);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // while the products run: the tile's bias (and gamma, beta) columns into
    // shared memory, and (EPI 1) the first columns of this row of x1 into
    // registers
    for (int c = threadIdx.x; c < NT; c += 128) {
      vec[c] = __ldg(p.bias + n0 + c);
      if (EPI == 1) {
        vec[NT + c] = __ldg(p.ln + n0 + c);
        vec[2 * NT + c] = __ldg(p.ln + p.hidden + n0 + c);
      }
    }
    mbar_arrive(BAR(C::B_VEC));
    // prefetched uint4 of the row of x1 (fewer with three CTAs per SM, for
    // their register budget)
    constexpr int XPF = (EPI == 1) ? (C::CTAS >= 3 ? 4 : (NT <= 128 ? NT / 8 : 16)) : 1;
    uint4 xpf[XPF];
    const uint16_t* xr = p.resid + static_cast<size_t>(valid ? m : 0) * p.hidden + n0;
    if (EPI == 1) {
#pragma unroll
      for (int q = 0; q < XPF; ++q)
        xpf[q] = valid ? *reinterpret_cast<const uint4*>(xr + 8 * q) : make_uint4(0, 0, 0, 0);
    }
    ok = bwait(BAR(C::B_VEC), 0, W) && bwait(BAR(C::B_ACC), 0, W);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (EPI == 0) {
      // bf16(C + b) into staging boxes in the (consumed) stage buffers: one
      // [128 rows][64 columns] bf16 box per 64 columns, 16-byte chunk c of
      // row r at chunk c ^ (r & 7) (the tensor maps' 128-byte swizzle)
      uint8_t* stg = smem;
#pragma unroll 1
      for (int hc = 0; hc < (ok ? MH * NT : 0); hc += 32) {
        const int h = hc / NT, c0 = hc - h * NT;   // row half, column
        uint32_t r[32];
        tmem_ld32(tl + hc, r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 bv = *reinterpret_cast<const float4*>(vec + c0 + e);
          pk[e / 2] = pack_bf16x2(__uint_as_float(r[e]) + bv.x, __uint_as_float(r[e + 1]) + bv.y);
          pk[e / 2 + 1] =
              pack_bf16x2(__uint_as_float(r[e + 2]) + bv.z, __uint_as_float(r[e + 3]) + bv.w);
        }
        const int rh = row + kGemmBM * h;
        uint8_t* rowp = stg + (c0 / 64) * (BM * 128) + rh * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int chunk = (c0 & 63) / 8 + q;
          *reinterpret_cast<uint4*>(rowp + ((chunk ^ (rh & 7)) << 4)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      fence_proxy_async_smem();
      // every epilogue thread arrives (also after a failed wait), so the
      // bounded wait below completes unless a wait ran out
      mbar_arrive(BAR(C::B_STG));
      const bool staged = bwait(BAR(C::B_STG), 0, W) && ok;
      if (threadIdx.x == 0 && staged) {
        // box (64 hh_col, l0, b H + head) of q, k or v per 64 columns; rows
        // past L are skipped
#pragma unroll 1
        for (int cb = 0; cb < NT / 64; ++cb) {
          const int n = n0 + 64 * cb;
          const int part = n / p.hidden, hc = n - part * p.hidden;
          const int hh = hc / p.D, dcol = hc - hh * p.D;
          tma_store_3d(&p.tmO[part], smem_u32(stg) + cb * (BM * 128), dcol, l0,
                       b_t * p.H + hh);
        }
        bulk_commit_group();
        bulk_wait_all();
      }
    } else {
      // pass 1: y = (x1 + C) + b, kept in TMEM over the accumulator; the
      // row's partial sum over this CTA's columns
      if (ok) {
#pragma unroll 1
        for (int c0 = 0; c0 < NT; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tl + c0, r);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int qi = c0 / 8 + q;
            uint4 xv;
            if (qi < XPF) {
              xv = xpf[0];
#pragma unroll
              for (int t = 1; t < XPF; ++t)
                if (t == qi) xv = xpf[t];
            } else {
              xv = valid ? *reinterpret_cast<const uint4*>(xr + 8 * qi) : make_uint4(0, 0, 0, 0);
            }
            const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
            const float4 b_lo = *reinterpret_cast<const float4*>(vec + c0 + 8 * q);
            const float4 b_hi = *reinterpret_cast<const float4*>(vec + c0 + 8 * q + 4);
            const float bb[8] = {b_lo.x, b_lo.y, b_lo.z, b_lo.w, b_hi.x, b_hi.y, b_hi.z, b_hi.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float xe = __uint_as_float((e & 1) ? (xw[e >> 1] & 0xffff0000u)
                                                       : (xw[e >> 1] << 16));
              r[8 * q + e] = __float_as_uint((xe + __uint_as_float(r[8 * q + e])) + bb[e]);
            }
          }
          tmem_st32(tl + c0, r);
          // the chunk's mean and M2, merged into the running pair (c0 columns
          // so far)
          float cs = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) cs += __uint_as_float(r[e]);
          const float cm = cs * (1.0f / 32.0f);
          float cq = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float dv = __uint_as_float(r[e]) - cm;
            cq = fmaf(dv, dv, cq);
          }
          const float dm = cm - mean, wn = 32.0f / static_cast<float>(c0 + 32);
          mean = fmaf(dm, wn, mean);
          m2 += cq + dm * dm * static_cast<float>(c0) * wn;
        }
        tmem_st_wait();
      }
    }
  }

  if (EPI == 1) {
    // ---- the row's (mean, M2) over the cluster's CTAs: one exchange, then
    // the pairwise merge of equal-sized parts (NT columns each)
    const uint32_t rank = cluster_rank(), ncta = cluster_size();
    __syncwarp();
    if (warp < 4) {
      const uint32_t a0 = smem_u32(red + (0 * kGemmMaxCluster + rank) * kGemmBM + row);
      const uint32_t a1 = smem_u32(red + (1 * kGemmMaxCluster + rank) * kGemmBM + row);
      for (uint32_t c = 0; c < ncta; ++c) {
        st_cluster_f32(a0, c, mean);
        st_cluster_f32(a1, c, m2);
      }
    }
    cluster_sync_all();
    if (warp < 4) {
      float s = 0.f;
      for (uint32_t c = 0; c < ncta; ++c) s += red[(0 * kGemmMaxCluster + c) * kGemmBM + row];
      const float mu = s / static_cast<float>(ncta);
      float q = 0.f;
      for (uint32_t c = 0; c < ncta; ++c) {
        const float dm = red[(0 * kGemmMaxCluster + c) * kGemmBM + row] - mu;
        q += red[(1 * kGemmMaxCluster + c) * kGemmBM + row] + static_cast<float>(NT) * dm * dm;
      }
      mean = mu;
      m2 = q;
    }
    // pass 3: the normalised row into staging boxes [128 rows][64 columns]
    // bf16 (the 128-byte swizzle, as for EPI 0), then one bulk store per 64
    // columns (rows past M are skipped)
    uint8_t* stg = smem;
    if (warp < 4 && ok) {
      const float rstd = rsqrtf(m2 * (1.0f / p.hidden) + p.eps);
#pragma unroll 1
      for (int c0 = 0; c0 < NT; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(tl + c0, r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 g = *reinterpret_cast<const float4*>(vec + NT + c0 + e);
          const float4 bt = *reinterpret_cast<const float4*>(vec + 2 * NT + c0 + e);
          pk[e / 2] = pack_bf16x2((__uint_as_float(r[e]) - mean) * rstd * g.x + bt.x,
                                  (__uint_as_float(r[e + 1]) - mean) * rstd * g.y + bt.y);
          pk[e / 2 + 1] = pack_bf16x2((__uint_as_float(r[e + 2]) - mean) * rstd * g.z + bt.z,
                                      (__uint_as_float(r[e + 3]) - mean) * rstd * g.w + bt.w);
        }
        uint8_t* rowp = stg + (c0 / 64) * (kGemmBM * 128) + row * 128;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const int chunk = (c0 & 63) / 8 + q4;
          *reinterpret_cast<uint4*>(rowp + ((chunk ^ (row & 7)) << 4)) =
              make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
        }
      }
    }
    if (warp < 4) {
      fence_proxy_async_smem();
      mbar_arrive(BAR(C::B_STG));
      const bool staged = bwait(BAR(C::B_STG), 0, W) && ok;
      if (threadIdx.x == 0 && staged) {
#pragma unroll 1
        for (int cb = 0; cb < NT / 64; ++cb)
          tma_store_2d(&p.tmO[0], smem_u32(stg) + cb * (kGemmBM * 128), n0 + 64 * cb, m0);
        bulk_commit_group();
        bulk_wait_all();
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

}  // namespace lf
