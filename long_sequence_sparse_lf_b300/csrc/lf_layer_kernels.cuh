// The first residual + LayerNorm of the Longformer layer forward
// ("基于Block-Sparse Attention的Longformer" (block-sparse Longformer), §6
// "Longformer的整体架构"), between the attention and the feed-forward map:
//   merge_ln1   x1 = bf16(LN1(x + merge_heads(a)))
// reading and writing its tensors once.  (The q, k, v maps and the
// feed-forward map with its residual + LayerNorm are tcgen05 GEMMs with fused
// epilogues, lf_gemm_kernel.cuh.)
// LayerNorm (over the hidden axis, biased variance):
//   LN(v) = (v - mean(v)) / sqrt(var(v) + eps) * gamma + beta.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

namespace lf {

__device__ __forceinline__ uint32_t layer_pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// bf16 <-> fp32 vectors of VW elements (VW = 2, 4 or 8: 4, 8 or 16 bytes)
template <int VW>
__device__ __forceinline__ void layer_load_bf16(const uint16_t* p, float (&v)[VW]) {
  if (VW == 8) {
    const uint4 u = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[(2 * i + 1) % VW] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else if (VW == 4) {
    const uint2 u = *reinterpret_cast<const uint2*>(p);
    v[0] = __uint_as_float(u.x << 16);
    v[1 % VW] = __uint_as_float(u.x & 0xffff0000u);
    v[2 % VW] = __uint_as_float(u.y << 16);
    v[3 % VW] = __uint_as_float(u.y & 0xffff0000u);
  } else {
    const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
    v[0] = __uint_as_float(u << 16);
    v[1 % VW] = __uint_as_float(u & 0xffff0000u);
  }
}

template <int VW>
__device__ __forceinline__ void layer_store_bf16(uint16_t* p, const float (&v)[VW]) {
  if (VW == 8) {
    *reinterpret_cast<uint4*>(p) =
        make_uint4(layer_pack_bf16x2(v[0], v[1 % VW]), layer_pack_bf16x2(v[2 % VW], v[3 % VW]),
                   layer_pack_bf16x2(v[4 % VW], v[5 % VW]), layer_pack_bf16x2(v[6 % VW], v[7 % VW]));
  } else if (VW == 4) {
    *reinterpret_cast<uint2*>(p) =
        make_uint2(layer_pack_bf16x2(v[0], v[1 % VW]), layer_pack_bf16x2(v[2 % VW], v[3 % VW]));
  } else {
    *reinterpret_cast<uint32_t*>(p) = layer_pack_bf16x2(v[0], v[1 % VW]);
  }
}

// VW consecutive fp32 values (16-byte loads for VW = 4, 8; 8-byte for VW = 2;
// p aligned to VW floats)
template <int VW>
__device__ __forceinline__ void layer_load_f32(const float* p, float (&v)[VW]) {
  if (VW % 4 == 0) {
#pragma unroll
    for (int i = 0; i < VW / 4; ++i) {
      const float4 t = reinterpret_cast<const float4*>(p)[i];
      v[4 * i] = t.x;
      v[(4 * i + 1) % VW] = t.y;
      v[(4 * i + 2) % VW] = t.z;
      v[(4 * i + 3) % VW] = t.w;
    }
  } else {
    const float2 t = *reinterpret_cast<const float2*>(p);
    v[0] = t.x;
    v[1 % VW] = t.y;
  }
}

// LayerNorm of one token row held by one warp: lane t holds the VW
// consecutive columns VW*t + 32*VW*j, j < NJ (hidden = 32 * VW * NJ).
template <int VW, int NJ>
__device__ __forceinline__ void layer_norm_row(float (&v)[NJ][VW], float eps,
                                               const float* __restrict__ gamma,
                                               const float* __restrict__ beta, int lane,
                                               uint16_t* __restrict__ out_row) {
  constexpr int hidden = 32 * VW * NJ;
  // gamma and beta first: their loads overlap the reductions
  float g[NJ][VW], bt[NJ][VW];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = VW * lane + 32 * VW * j;
    layer_load_f32<VW>(gamma + c, g[j]);
    layer_load_f32<VW>(beta + c, bt[j]);
  }
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int e = 0; e < VW; ++e) s += v[j][e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s * (1.0f / hidden);
  float q = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j)
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const float dv = v[j][e] - mean;
      q = fmaf(dv, dv, q);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q * (1.0f / hidden) + eps);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = VW * lane + 32 * VW * j;
    float y[VW];
#pragma unroll
    for (int e = 0; e < VW; ++e) y[e] = (v[j][e] - mean) * rstd * g[j][e] + bt[j][e];
    layer_store_bf16<VW>(out_row + c, y);
  }
}

// x1 = bf16(LN1(x + a)), a = the attention output [B, H, L, D] merged back to
// [B, L, H*D].  ln1: gamma then beta, fp32 [2*hidden].  One warp per row.
template <int VW, int NJ>
__global__ void lf_layer_merge_ln1_kernel(const uint16_t* __restrict__ x,
                                          const uint16_t* __restrict__ attn,
                                          const float* __restrict__ ln1, uint16_t* __restrict__ x1,
                                          int B, int H, int L, int D, float eps) {
  constexpr int hidden = 32 * VW * NJ;
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * L) return;
  const int b = (int)(row / L), l = (int)(row % L);
  float v[NJ][VW];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int c = VW * lane + 32 * VW * j;
    const int h = c / D, e = c - h * D;
    float xa[VW], aa[VW];
    layer_load_bf16<VW>(x + (size_t)row * hidden + c, xa);
    layer_load_bf16<VW>(attn + (((size_t)b * H + h) * L + l) * D + e, aa);
#pragma unroll
    for (int i = 0; i < VW; ++i) v[j][i] = xa[i] + aa[i];
  }
  layer_norm_row<VW, NJ>(v, eps, ln1, ln1 + hidden, lane, x1 + (size_t)row * hidden);
}

}  // namespace lf
