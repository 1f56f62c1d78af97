// Backward of the Longformer sparse attention: dq, dk, dv of sum(out * dout).
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
// The attended pairs split into three classes:
//   band        i not global, j in band(i): the tcgen05 kernel of
//               lf_bwd_tc_kernel.cuh;
//   global keys j global, i not global, j not in band(i): per 64 gathered
//               global keys, over every query block (this file);
//   global rows i global, every j: per 64 gathered global rows, over every
//               key block (this file).
// The two global classes split their streamed side into chunks of kBwdChunk
// blocks, one CTA each, so that a few global tokens still fill the GPU.
// Each block pair computes S = Q K^T and dP = dO V^T with WMMA (bf16 in, fp32
// accumulation) into shared memory, forms P and dS (bf16) element by element
// with the class's mask, then dV += P^T dO, dK += dS^T Q and dQ += dS K.  The
// CTA's fixed rows (keys, or global rows) sum in WMMA accumulator fragments,
// each warp holding its share of the tiles for the CTA's whole life, and are
// added to the fp32 gradients (zeroed first) once, with atomics; the streamed
// rows' sums are added with atomics after every block pair.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <mma.h>
#include <type_traits>

namespace lf {

constexpr int kBwdB = 64;        // rows of a query block and of a key block
constexpr int kBwdThreads = 256; // eight warps
constexpr int kBwdChunk = 8;     // streamed blocks per CTA of the global kernels

struct BwdParams {
  const __nv_bfloat16* q;        // [B*H, L, D]
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const __nv_bfloat16* dout;
  const float* lse;              // [B*H, L]
  const float* delta;            // [B*H, L]
  float* dq;                     // [B*H, L, D], accumulated
  float* dk;
  float* dv;
  const int32_t* gidx;           // [n_g] sorted global positions
  const uint8_t* is_glob;        // [L]
  const int32_t* head_dil;       // [H]
  int H, L, w, n_g;
  float scale;
};

// delta[bh, i] = dout_i . out_i (bf16 rows, fp32 sum); one warp per row.
template <int D>
__global__ void lf_bwd_delta_kernel(const __nv_bfloat16* __restrict__ out,
                                    const __nv_bfloat16* __restrict__ dout,
                                    float* __restrict__ delta, long long rows) {
  const long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float s = 0.f;
#pragma unroll
  for (int e = lane; e < D; e += 32)
    s += __bfloat162float(out[r * D + e]) * __bfloat162float(dout[r * D + e]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) delta[r] = s;
}

// Row strides of the shared-memory tiles, padded by 16 bytes so that the
// column-wise fragment loads of a tile (P^T, dS^T) do not fall on one bank.
template <int D>
struct BwdLd {
  static constexpr int X = D + 8;       // bf16 [64 x D] tiles (q, k, v, dout)
  static constexpr int SQ = kBwdB + 4;  // fp32 [64 x 64] (S, dP)
  static constexpr int PQ = kBwdB + 8;  // bf16 [64 x 64] (P, dS)
  static constexpr int A = D + 4;       // fp32 [64 x D] (products, sums)
};

template <int D>
struct BwdSmem {
  using LD = BwdLd<D>;
  __nv_bfloat16 q[kBwdB * LD::X], k[kBwdB * LD::X], v[kBwdB * LD::X], dout[kBwdB * LD::X];
  float s[kBwdB * LD::SQ];
  float dp[kBwdB * LD::SQ];
  __nv_bfloat16 p[kBwdB * LD::PQ], ds[kBwdB * LD::PQ];
  float acc[kBwdB * LD::A];      // product tile before it is added to global memory
  float lse[kBwdB], delta[kBwdB];
  int qpos[kBwdB], kpos[kBwdB];  // positions of the block's rows (-1: none)
  int qglob[kBwdB];              // the query row is a global token
};

// rows[c] (positions, -1 = none) of X [B*H, L, D] into shared memory (zeros
// for missing rows); 16 bytes per thread and step
template <int D>
__device__ __forceinline__ void bwd_load_rows(__nv_bfloat16* dst, const __nv_bfloat16* src,
                                              size_t bh, int L, const int* rows) {
  constexpr int PCS = D / 8;
  for (int x = threadIdx.x; x < kBwdB * PCS; x += blockDim.x) {
    const int c = x / PCS, pc = x - c * PCS;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (rows[c] >= 0)
      val = reinterpret_cast<const uint4*>(src + (bh * L + rows[c]) * D)[pc];
    reinterpret_cast<uint4*>(dst + c * BwdLd<D>::X)[pc] = val;
  }
}

// C[64 x N] (= A[64 x K] B, or C += A B with ACCUM) in shared memory, fp32; A row-major (lda), B
// row-major [K x N] (b_rowmajor, ldb) or B = X^T for X row-major [N x K]
// (ldb = K); a_colmajor reads A as the transpose of a row-major [K x 64].
template <int N, int K, bool A_COL, bool B_ROW, bool ACCUM = false>
__device__ __forceinline__ void bwd_gemm(float* C, int ldc, const __nv_bfloat16* A, int lda,
                                         const __nv_bfloat16* B, int ldb) {
  using namespace nvcuda;
  const int warp = threadIdx.x >> 5;
  constexpr int TN = N / 16;
  for (int t = warp; t < 4 * TN; t += kBwdThreads / 32) {
    const int mi = t / TN, ni = t - mi * TN;
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> c;
    if (ACCUM)   // C += A B (C already holds the running sum)
      wmma::load_matrix_sync(c, C + (size_t)mi * 16 * ldc + ni * 16, ldc, wmma::mem_row_major);
    else
      wmma::fill_fragment(c, 0.f);
#pragma unroll
    for (int kk = 0; kk < K / 16; ++kk) {
      using ALay = typename std::conditional<A_COL, wmma::col_major, wmma::row_major>::type;
      using BLay = typename std::conditional<B_ROW, wmma::row_major, wmma::col_major>::type;
      wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, ALay> a;
      wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, BLay> b;
      const __nv_bfloat16* ap = A_COL ? A + (size_t)kk * 16 * lda + mi * 16
                                      : A + (size_t)mi * 16 * lda + kk * 16;
      const __nv_bfloat16* bp = B_ROW ? B + (size_t)kk * 16 * ldb + ni * 16
                                      : B + (size_t)ni * 16 * ldb + kk * 16;
      wmma::load_matrix_sync(a, ap, lda);
      wmma::load_matrix_sync(b, bp, ldb);
      wmma::mma_sync(c, a, b, c);
    }
    wmma::store_matrix_sync(C + (size_t)mi * 16 * ldc + ni * 16, c, ldc, wmma::mem_row_major);
  }
}

// A [64 x N] fp32 sum held in registers: warp w keeps the accumulator
// fragments of tiles w, w + 8, ... of the 4 x N/16 grid of 16 x 16 tiles.
// mma() adds A B with bwd_gemm's operand conventions; store() writes the sum
// to shared memory (row stride ldc).
template <int N>
struct BwdFragAcc {
  static constexpr int TN = N / 16;
  static constexpr int NF = 4 * TN / (kBwdThreads / 32);
  static_assert(NF * (kBwdThreads / 32) == 4 * TN, "tiles must split evenly over the warps");
  nvcuda::wmma::fragment<nvcuda::wmma::accumulator, 16, 16, 16, float> f[NF];

  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int m = 0; m < NF; ++m) nvcuda::wmma::fill_fragment(f[m], 0.f);
  }
  template <int K, bool A_COL, bool B_ROW>
  __device__ __forceinline__ void mma(const __nv_bfloat16* A, int lda, const __nv_bfloat16* B,
                                      int ldb) {
    using namespace nvcuda;
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < NF; ++m) {
      const int t = warp + m * (kBwdThreads / 32);
      const int mi = t / TN, ni = t - mi * TN;
#pragma unroll
      for (int kk = 0; kk < K / 16; ++kk) {
        using ALay = typename std::conditional<A_COL, wmma::col_major, wmma::row_major>::type;
        using BLay = typename std::conditional<B_ROW, wmma::row_major, wmma::col_major>::type;
        wmma::fragment<wmma::matrix_a, 16, 16, 16, __nv_bfloat16, ALay> a;
        wmma::fragment<wmma::matrix_b, 16, 16, 16, __nv_bfloat16, BLay> b;
        const __nv_bfloat16* ap = A_COL ? A + (size_t)kk * 16 * lda + mi * 16
                                        : A + (size_t)mi * 16 * lda + kk * 16;
        const __nv_bfloat16* bp = B_ROW ? B + (size_t)kk * 16 * ldb + ni * 16
                                        : B + (size_t)ni * 16 * ldb + kk * 16;
        wmma::load_matrix_sync(a, ap, lda);
        wmma::load_matrix_sync(b, bp, ldb);
        wmma::mma_sync(f[m], a, b, f[m]);
      }
    }
  }
  __device__ __forceinline__ void store(float* C, int ldc) const {
    const int warp = threadIdx.x >> 5;
#pragma unroll
    for (int m = 0; m < NF; ++m) {
      const int t = warp + m * (kBwdThreads / 32);
      const int mi = t / TN, ni = t - mi * TN;
      nvcuda::wmma::store_matrix_sync(C + (size_t)mi * 16 * ldc + ni * 16, f[m], ldc,
                                      nvcuda::wmma::mem_row_major);
    }
  }
};

// acc [64 x D] (row stride BwdLd::A, scaled) added to X[bh, rows[c], :]
// with atomics
template <int D>
__device__ __forceinline__ void bwd_add_rows(float* X, const float* acc, float scale, size_t bh,
                                             int L, const int* rows) {
  for (int x = threadIdx.x; x < kBwdB * D; x += blockDim.x) {
    const int c = x / D, e = x - c * D;
    if (rows[c] >= 0)
      atomicAdd(X + (bh * L + rows[c]) * D + e, acc[c * BwdLd<D>::A + e] * scale);
  }
}

// KIND 1: global keys; 2: global rows.  One CTA per unit (two per SM for
// D = 64, whose shared memory allows it).
template <int D, int KIND>
__global__ void __launch_bounds__(kBwdThreads, D == 64 ? 2 : 1) lf_bwd_kernel(const BwdParams p) {
  extern __shared__ __align__(128) uint8_t bwd_smem_raw[];
  BwdSmem<D>& sm = *reinterpret_cast<BwdSmem<D>*>(bwd_smem_raw);
  using LD = BwdLd<D>;
  const float log2e = 1.4426950408889634f;
  static_assert(KIND == 1 || KIND == 2, "global classes only");
  // the unit: gathered global rows fixed0 .. +63 of head bh against the
  // streamed blocks blk0 .. n_blocks-1 (this CTA's chunk)
  const int n_gt = (p.n_g + kBwdB - 1) / kBwdB;
  const int all_blocks = (p.L + kBwdB - 1) / kBwdB;
  const int n_sc = (all_blocks + kBwdChunk - 1) / kBwdChunk;
  const int sc = (int)(blockIdx.x % n_sc);
  const size_t unit = blockIdx.x / n_sc;
  const size_t bh = unit / n_gt;
  const int fixed0 = (int)(unit % n_gt) * kBwdB;
  const int d = p.head_dil[bh % p.H];
  const int blk0 = sc * kBwdChunk;
  const int n_blocks = min(all_blocks, blk0 + kBwdChunk);
  // the fixed side: keys (global keys) or queries (global rows)
  int* fixed_pos = (KIND == 2) ? sm.qpos : sm.kpos;
  for (int c = threadIdx.x; c < kBwdB; c += blockDim.x)
    fixed_pos[c] = fixed0 + c < p.n_g ? p.gidx[fixed0 + c] : -1;
  // the fixed rows' sums over the streamed blocks: dV, dK of the keys, or
  // dQ of the global rows (fix0 only)
  BwdFragAcc<D> fix0, fix1;
  fix0.zero();
  fix1.zero();
  __syncthreads();
  if (KIND == 2) {
    bwd_load_rows<D>(sm.q, p.q, bh, p.L, sm.qpos);
    bwd_load_rows<D>(sm.dout, p.dout, bh, p.L, sm.qpos);
    for (int c = threadIdx.x; c < kBwdB; c += blockDim.x) {
      sm.lse[c] = sm.qpos[c] >= 0 ? p.lse[bh * p.L + sm.qpos[c]] * log2e : 0.f;
      sm.delta[c] = sm.qpos[c] >= 0 ? p.delta[bh * p.L + sm.qpos[c]] : 0.f;
      sm.qglob[c] = 1;
    }
  } else {
    bwd_load_rows<D>(sm.k, p.k, bh, p.L, sm.kpos);
    bwd_load_rows<D>(sm.v, p.v, bh, p.L, sm.kpos);
  }
  const float sl2 = p.scale * log2e;

  for (int blk = blk0; blk < n_blocks; ++blk) {
    __syncthreads();
    // the streamed side's rows
    int* str_pos = (KIND == 2) ? sm.kpos : sm.qpos;
    for (int c = threadIdx.x; c < kBwdB; c += blockDim.x) {
      const int i = blk * kBwdB + c;
      str_pos[c] = i < p.L ? i : -1;
    }
    __syncthreads();
    if (KIND == 2) {
      bwd_load_rows<D>(sm.k, p.k, bh, p.L, sm.kpos);
      bwd_load_rows<D>(sm.v, p.v, bh, p.L, sm.kpos);
    } else {
      bwd_load_rows<D>(sm.q, p.q, bh, p.L, sm.qpos);
      bwd_load_rows<D>(sm.dout, p.dout, bh, p.L, sm.qpos);
      for (int c = threadIdx.x; c < kBwdB; c += blockDim.x) {
        sm.lse[c] = sm.qpos[c] >= 0 ? p.lse[bh * p.L + sm.qpos[c]] * log2e : 0.f;
        sm.delta[c] = sm.qpos[c] >= 0 ? p.delta[bh * p.L + sm.qpos[c]] : 0.f;
        sm.qglob[c] = sm.qpos[c] >= 0 ? p.is_glob[sm.qpos[c]] : 0;
      }
    }
    __syncthreads();
    // S = Q K^T, dP = dO V^T   [64 queries x 64 keys]
    bwd_gemm<kBwdB, D, false, false>(sm.s, LD::SQ, sm.q, LD::X, sm.k, LD::X);
    bwd_gemm<kBwdB, D, false, false>(sm.dp, LD::SQ, sm.dout, LD::X, sm.v, LD::X);
    __syncthreads();
    // P and dS of the pairs this class owns (0 elsewhere)
    for (int x = threadIdx.x; x < kBwdB * kBwdB; x += blockDim.x) {
      const int a = x / kBwdB, b = x - a * kBwdB;   // query row a, key row b
      const int i = sm.qpos[a], j = sm.kpos[b];
      bool ok = i >= 0 && j >= 0;
      if (ok) {
        if (KIND == 1) {
          const int diff = i - j;
          const bool in_band = abs(diff) <= d * p.w && diff % d == 0;
          ok = sm.qglob[a] == 0 && !in_band;
        }
      }
      float pv = 0.f, dsv = 0.f;
      if (ok) {
        pv = exp2f(sm.s[a * LD::SQ + b] * sl2 - sm.lse[a]);
        dsv = pv * (sm.dp[a * LD::SQ + b] - sm.delta[a]);
      }
      sm.p[a * LD::PQ + b] = __float2bfloat16_rn(pv);
      sm.ds[a * LD::PQ + b] = __float2bfloat16_rn(dsv);
    }
    __syncthreads();
    // dV_keys += P^T dO, dK_keys += scale dS^T Q, dQ_queries += scale dS K:
    // the fixed side's rows sum in shared memory over the streamed blocks,
    // the streamed side's go to global memory with atomics
    if (KIND == 2) {
      bwd_gemm<D, kBwdB, true, true>(sm.acc, LD::A, sm.p, LD::PQ, sm.dout, LD::X);
      __syncthreads();
      bwd_add_rows<D>(p.dv, sm.acc, 1.f, bh, p.L, sm.kpos);
      __syncthreads();
      bwd_gemm<D, kBwdB, true, true>(sm.acc, LD::A, sm.ds, LD::PQ, sm.q, LD::X);
      __syncthreads();
      bwd_add_rows<D>(p.dk, sm.acc, p.scale, bh, p.L, sm.kpos);
      fix0.template mma<kBwdB, false, true>(sm.ds, LD::PQ, sm.k, LD::X);
    } else {
      fix0.template mma<kBwdB, true, true>(sm.p, LD::PQ, sm.dout, LD::X);
      fix1.template mma<kBwdB, true, true>(sm.ds, LD::PQ, sm.q, LD::X);
      bwd_gemm<D, kBwdB, false, true>(sm.acc, LD::A, sm.ds, LD::PQ, sm.k, LD::X);
      __syncthreads();
      bwd_add_rows<D>(p.dq, sm.acc, p.scale, bh, p.L, sm.qpos);
    }
  }
  __syncthreads();
  fix0.store(sm.acc, LD::A);
  __syncthreads();
  if (KIND == 2) {
    bwd_add_rows<D>(p.dq, sm.acc, p.scale, bh, p.L, sm.qpos);
  } else {
    bwd_add_rows<D>(p.dv, sm.acc, 1.f, bh, p.L, sm.kpos);
    __syncthreads();
    fix1.store(sm.acc, LD::A);
    __syncthreads();
    bwd_add_rows<D>(p.dk, sm.acc, p.scale, bh, p.L, sm.kpos);
  }
}

}  // namespace lf
