// Small kernels around the attention kernel: fp32 -> bf16 rounding of the
// inputs, gathering of the global rows, merging of the global-row partials
// and the per-query key-list enumerator.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "lf_common.cuh"

namespace lf {

// ---------------------------------------------------------------- cast
// q, k, v rounded to bf16 in one launch: out[x * n4 + i] = bf16_rn(in_x[i])
// for x = 0, 1, 2 (in_0 = q, in_1 = k, in_2 = v); n4 = float4 groups of one
// tensor.
__global__ void lf_cast_f32_bf16_kernel(const float4* __restrict__ q, const float4* __restrict__ k,
                                        const float4* __restrict__ v, uint2* __restrict__ out,
                                        size_t n4) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
#pragma unroll 1
  for (int x = 0; x < 3; ++x) {
    const float4* __restrict__ in = x == 0 ? q : (x == 1 ? k : v);
    uint2* __restrict__ dst = out + x * n4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += stride) {
      const float4 f = in[i];
      __nv_bfloat162 a = __floats2bfloat162_rn(f.x, f.y);
      __nv_bfloat162 b = __floats2bfloat162_rn(f.z, f.w);
      uint2 o;
      o.x = *reinterpret_cast<uint32_t*>(&a);
      o.y = *reinterpret_cast<uint32_t*>(&b);
      dst[i] = o;
    }
  }
}

// ---------------------------------------------------------------- gather
// dst_X[bh][g][:] = X[bh][G[g]][:] for g < n_g, 0 for n_g <= g < NGQ, for
// X = q, k, v and, when `x4` is not null, a fourth tensor x4.
// One thread per 16-byte piece (D/8 pieces per row).
__global__ void lf_gather_globals_kernel(const uint4* __restrict__ q, const uint4* __restrict__ k,
                                         const uint4* __restrict__ v, uint4* __restrict__ qg,
                                         uint4* __restrict__ kg, uint4* __restrict__ vg,
                                         const int32_t* __restrict__ gidx, int n_g, int NGQ, int L,
                                         int D, int BH, const uint4* __restrict__ x4 = nullptr,
                                         uint4* __restrict__ x4g = nullptr) {
  const int pieces = D / 8;
  const size_t total = (size_t)BH * NGQ * pieces;
  for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < total;
       x += (size_t)gridDim.x * blockDim.x) {
    const int pc = (int)(x % pieces);
    const size_t rowi = x / pieces;
    const int g = (int)(rowi % NGQ);
    const size_t bh = rowi / NGQ;
    uint4 a = make_uint4(0, 0, 0, 0), b = a, c = a, e = a;
    if (g < n_g) {
      const size_t src = (bh * L + gidx[g]) * pieces + pc;
      a = q[src];
      b = k[src];
      c = v[src];
      if (x4 != nullptr) e = x4[src];
    }
    qg[x] = a;
    kg[x] = b;
    vg[x] = c;
    if (x4g != nullptr) x4g[x] = e;
  }
}

// ---------------------------------------------------------------- combine
// One warp per (bh, g < n_g): merges the key-chunk partials of a global row,
//   m = max_c m_c,  l = sum_c l_c 2^(m_c - m),  o = sum_c o_c 2^(m_c - m) / l
// (m in log2 units), and writes the row of the output at position G[g] (and
// its log-sum-exp (m + log2 l) ln 2, if lse is given).  The chunks go in
// groups of up to 32: lane c of a group reads chunk c's (m_c, l_c), and the
// group's O rows (D / 32 values per lane and chunk, up to kCombineBatch
// chunks at a time) are loaded before any of the arithmetic, so that the
// warp waits for memory once per batch rather than once per step.
constexpr int kCombineBatch = 16;
template <int D>
__global__ void lf_combine_globals_kernel(const float* __restrict__ part_o,
                                          const float* __restrict__ part_ml,
                                          const int32_t* __restrict__ gidx, void* out, int out_f32,
                                          int n_g, int NGQ, int n_chunks, int L, int BH,
                                          float* __restrict__ lse) {
  constexpr int PER = D / 32;
  const float NEG_INF = -__int_as_float(0x7f800000);
  const unsigned FULL = 0xffffffffu;
  const int warps_per_block = blockDim.x / 32;
  const long long wid = (long long)blockIdx.x * warps_per_block + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (wid >= (long long)BH * n_g) return;
  const int g = (int)(wid % n_g);
  const long long bh = wid / n_g;
  const size_t base = ((size_t)bh * NGQ + g) * n_chunks;
  const int grow = __ldg(gidx + g);
  // running (m, l, o) of the row over the groups merged so far
  float m = NEG_INF, l = 0.f;
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int c0 = 0; c0 < n_chunks; c0 += 32) {
    const int nc = min(32, n_chunks - c0);
    // this group: each lane's chunk statistics, and the first batch of O rows
    float mc = NEG_INF, lc = 0.f;
    if (lane < nc) {
      const float2 ml = *reinterpret_cast<const float2*>(part_ml + (base + c0 + lane) * 2);
      mc = ml.x;
      lc = ml.y;
    }
    float ob[kCombineBatch][PER];
#pragma unroll
    for (int c = 0; c < kCombineBatch; ++c)
#pragma unroll
      for (int e = 0; e < PER; ++e)
        ob[c][e] = c < nc ? part_o[(base + c0 + c) * D + lane + 32 * e] : 0.f;
    float mg = mc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mg = fmaxf(mg, __shfl_xor_sync(FULL, mg, o));
    const float mn = fmaxf(m, mg);
    // rescale what has been merged so far, then add this group
    const float sc = (m == NEG_INF) ? 0.f : ((m == mn) ? 1.f : exp2f(m - mn));
    l *= sc;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= sc;
    m = mn;
    const float wgt = (lane < nc && mc != NEG_INF) ? ((mc == m) ? 1.f : exp2f(mc - m)) : 0.f;
    float lw = wgt * lc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(FULL, lw, o);
    l += lw;
#pragma unroll
    for (int c = 0; c < kCombineBatch; ++c) {
      const float wc = __shfl_sync(FULL, wgt, c);
#pragma unroll
      for (int e = 0; e < PER; ++e) acc[e] = fmaf(ob[c][e], wc, acc[e]);
    }
    for (int cb = kCombineBatch; cb < nc; cb += kCombineBatch) {
#pragma unroll
      for (int c = 0; c < kCombineBatch; ++c)
#pragma unroll
        for (int e = 0; e < PER; ++e)
          ob[c][e] = cb + c < nc ? part_o[(base + c0 + cb + c) * D + lane + 32 * e] : 0.f;
#pragma unroll
      for (int c = 0; c < kCombineBatch; ++c) {
        const float wc = __shfl_sync(FULL, wgt, (cb + c) & 31);
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = fmaf(ob[c][e], cb + c < nc ? wc : 0.f, acc[e]);
      }
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const size_t orow = ((size_t)bh * L + grow) * D;
  if (lse != nullptr && lane == 0) lse[(size_t)bh * L + grow] = (m + __log2f(l)) * 0.69314718f;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const float val = acc[e] * inv;
    if (out_f32)
      static_cast<float*>(out)[orow + lane + 32 * e] = val;
    else
      static_cast<__nv_bfloat16*>(out)[orow + lane + 32 * e] = __float2bfloat16_rn(val);
  }
}

// ---------------------------------------------------------------- key lists
// Row (h, i) of the CSR lists K(i) in increasing key order.

// number of entries of the sorted array G[0..n) that are < x
__device__ __forceinline__ int lower_count(const int32_t* G, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (G[mid] < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ void row_band(int i, int d, int w, int L, int& r, int& tlo, int& thi) {
  r = i % d;
  const int t = i / d;
  band_window(t, w, residue_len(L, d, r), tlo, thi);
}

// counts[h*L + i] = |K(i)|
__global__ void lf_pairs_count_kernel(const int32_t* __restrict__ dil, const int32_t* __restrict__ G,
                                      const uint8_t* __restrict__ is_glob, int n_g, int H, int L,
                                      int w, int64_t* __restrict__ counts) {
  const long long total = (long long)H * L;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const int h = (int)(x / L), i = (int)(x % L);
    if (is_glob[i]) { counts[x] = L; continue; }
    const int d = dil[h];
    int r, tlo, thi;
    row_band(i, d, w, L, r, tlo, thi);
    int64_t c = thi - tlo + 1;
    // globals outside the band: n_g minus those inside it
    const int jlo = r + d * tlo, jhi = r + d * thi;
    const int a = lower_count(G, n_g, jlo), b = lower_count(G, n_g, jhi + 1);
    int inside = 0;
    for (int e = a; e < b; ++e) inside += in_band_abs(i, G[e], d, w) ? 1 : 0;
    counts[x] = c + (n_g - inside);
  }
}

// Exclusive scan of counts[0..n) into row_ptr[0..n] (one block, sequential
// over tiles of blockDim.x elements; this is not on the attention path).
__global__ void lf_pairs_scan_kernel(const int64_t* __restrict__ counts, int64_t* __restrict__ row_ptr,
                                     long long n) {
  __shared__ int64_t buf[1024];
  __shared__ int64_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (long long base = 0; base < n; base += blockDim.x) {
    const long long x = base + threadIdx.x;
    const int64_t v = x < n ? counts[x] : 0;
    buf[threadIdx.x] = v;
    __syncthreads();
    for (int off = 1; off < (int)blockDim.x; off <<= 1) {
      int64_t add = threadIdx.x >= (unsigned)off ? buf[threadIdx.x - off] : 0;
      __syncthreads();
      buf[threadIdx.x] += add;
      __syncthreads();
    }
    if (x < n) row_ptr[x] = carry + buf[threadIdx.x] - v;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry += buf[threadIdx.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) row_ptr[n] = carry;
}

// Fill: merge the band (an arithmetic sequence) with G, dropping globals
// already in the band; global rows list every key.
__global__ void lf_pairs_fill_kernel(const int32_t* __restrict__ dil, const int32_t* __restrict__ G,
                                     const uint8_t* __restrict__ is_glob, int n_g, int H, int L,
                                     int w, const int64_t* __restrict__ row_ptr,
                                     int32_t* __restrict__ col) {
  const long long total = (long long)H * L;
  for (long long x = blockIdx.x * (long long)blockDim.x + threadIdx.x; x < total;
       x += (long long)gridDim.x * blockDim.x) {
    const int h = (int)(x / L), i = (int)(x % L);
    int32_t* dst = col + row_ptr[x];
    if (is_glob[i]) {
      for (int j = 0; j < L; ++j) dst[j] = j;
      continue;
    }
    const int d = dil[h];
    int r, tlo, thi;
    row_band(i, d, w, L, r, tlo, thi);
    int t = tlo, e = 0;
    long long o = 0;
    while (t <= thi || e < n_g) {
      const int jb = t <= thi ? r + d * t : 0x7fffffff;
      int jg = e < n_g ? G[e] : 0x7fffffff;
      if (e < n_g && in_band_abs(i, jg, d, w)) { ++e; continue; }   // counted with the band
      if (jb < jg) { dst[o++] = jb; ++t; }
      else { dst[o++] = jg; ++e; }
    }
  }
}

// The bias table as the BIAS attention kernel reads it: four copies per
// head, copy c of head h at (4h + c) * bias_row_len(w), whose entry x holds
// rel_bias[h, x + c - kBiasPad] * inv_scale where that index is in [0, 2w]
// and 0 elsewhere.  A row whose values start at index I of the padded table
// reads copy I % 4 from I - I % 4, a 16-byte aligned address.
__global__ void lf_bias_pad_kernel(const float* __restrict__ rb, float* __restrict__ out, int H,
                                   int w, float inv_scale) {
  const int rl = bias_row_len(w);
  const int n = 4 * H * rl;
  for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < n; x += gridDim.x * blockDim.x) {
    const int row = x / rl, h = row >> 2, c = (x - row * rl) + (row & 3) - kBiasPad;
    out[x] = (c >= 0 && c <= 2 * w) ? rb[static_cast<size_t>(h) * (2 * w + 1) + c] * inv_scale : 0.f;
  }
}

}  // namespace lf
