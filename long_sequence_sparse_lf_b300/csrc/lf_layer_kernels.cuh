// Kernels of the Longformer layer forward around the attention kernel
// ("基于Block-Sparse Attention的Longformer" (block-sparse Longformer), §6
// "Longformer的整体架构": q, k, v linear maps of x, the attention, residual +
// LayerNorm, a linear feed-forward map, residual + LayerNorm).  The two linear
// maps are plain GEMMs (cuBLASLt, fp32 results); these kernels do the
// memory-bound steps between them, each reading and writing its tensors once:
//   split_qkv   q, k, v = bf16(Y + b) split into heads [B, H, L, D]
//   merge_ln1   x1 = bf16(LN1(x + merge_heads(a)))
//   ln2         y  = bf16(LN2(x1 + F + b_f))
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

// Y: fp32 [M = B*L, 3*hidden] (row = token, columns q | k | v features, head
// h of each at h*D .. h*D + D-1); bias fp32 [3*hidden].  qkv: bf16, three
// consecutive [B, H, L, D] tensors.  One thread per 4 output elements.
__global__ void lf_layer_split_qkv_kernel(const float4* __restrict__ Y,
                                          const float4* __restrict__ bias,
                                          uint2* __restrict__ qkv, int B, int H, int L, int D) {
  const int hidden = H * D;
  const size_t per = (size_t)B * H * L * D / 4;   // 4-element groups per tensor
  const size_t total = 3 * per;
  for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < total;
       x += (size_t)gridDim.x * blockDim.x) {
    const int s = (int)(x / per);
    size_t r = x % per;
    const int e4 = (int)(r % (D / 4));
    r /= (D / 4);
    const int l = (int)(r % L);
    r /= L;
    const int h = (int)(r % H);
    const int b = (int)(r / H);
    const int col4 = (s * hidden + h * D) / 4 + e4;
    const float4 y = Y[((size_t)b * L + l) * (3 * hidden / 4) + col4];
    const float4 c = bias[col4];
    qkv[x] = make_uint2(layer_pack_bf16x2(y.x + c.x, y.y + c.y),
                        layer_pack_bf16x2(y.z + c.z, y.w + c.w));
  }
}

// One warp per token row: lane t holds the bf16 pairs at columns
// 2t + 64j, j < hidden/64.  PER2 = hidden / 64 pairs per lane.
template <int PER2>
__device__ __forceinline__ void layer_norm_row(float (&v)[2 * PER2], float eps,
                                               const float* __restrict__ gamma,
                                               const float* __restrict__ beta, int lane,
                                               uint32_t* __restrict__ out_row) {
  constexpr int hidden = 64 * PER2;
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 2 * PER2; ++e) s += v[e];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  const float mean = s * (1.0f / hidden);
  float q = 0.f;
#pragma unroll
  for (int e = 0; e < 2 * PER2; ++e) {
    const float dv = v[e] - mean;
    q = fmaf(dv, dv, q);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
  const float rstd = rsqrtf(q * (1.0f / hidden) + eps);
#pragma unroll
  for (int j = 0; j < PER2; ++j) {
    const int c = 2 * lane + 64 * j;
    const float y0 = (v[2 * j] - mean) * rstd * gamma[c] + beta[c];
    const float y1 = (v[2 * j + 1] - mean) * rstd * gamma[c + 1] + beta[c + 1];
    out_row[c / 2] = layer_pack_bf16x2(y0, y1);
  }
}

// x1 = bf16(LN1(x + a)), a = the attention output [B, H, L, D] merged back to
// [B, L, H*D].  ln1: gamma then beta, fp32 [2*hidden].  One warp per row.
template <int PER2>
__global__ void lf_layer_merge_ln1_kernel(const uint32_t* __restrict__ x,
                                          const uint32_t* __restrict__ attn,
                                          const float* __restrict__ ln1, uint32_t* __restrict__ x1,
                                          int B, int H, int L, int D, float eps) {
  constexpr int hidden = 64 * PER2;
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= (long long)B * L) return;
  const int b = (int)(row / L), l = (int)(row % L);
  float v[2 * PER2];
#pragma unroll
  for (int j = 0; j < PER2; ++j) {
    const int c = 2 * lane + 64 * j;
    const int h = c / D, e = c % D;
    const uint32_t xw = x[(size_t)row * (hidden / 2) + c / 2];
    const uint32_t aw = attn[((((size_t)b * H + h) * L + l) * D + e) / 2];
    v[2 * j] = __uint_as_float(xw << 16) + __uint_as_float(aw << 16);
    v[2 * j + 1] = __uint_as_float(xw & 0xffff0000u) + __uint_as_float(aw & 0xffff0000u);
  }
  layer_norm_row<PER2>(v, eps, ln1, ln1 + hidden, lane, x1 + (size_t)row * (hidden / 2));
}

// y = bf16(LN2(x1 + F + b_f)), F: fp32 [M, hidden] (the feed-forward GEMM),
// b_f fp32 [hidden], ln2: gamma then beta.  One warp per row.
template <int PER2>
__global__ void lf_layer_ln2_kernel(const uint32_t* __restrict__ x1, const float2* __restrict__ F,
                                    const float2* __restrict__ bf, const float* __restrict__ ln2,
                                    uint32_t* __restrict__ y, long long M, float eps) {
  constexpr int hidden = 64 * PER2;
  const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= M) return;
  float v[2 * PER2];
#pragma unroll
  for (int j = 0; j < PER2; ++j) {
    const int c2 = lane + 32 * j;   // pair index
    const uint32_t xw = x1[(size_t)row * (hidden / 2) + c2];
    const float2 f = F[(size_t)row * (hidden / 2) + c2];
    const float2 bb = bf[c2];
    v[2 * j] = __uint_as_float(xw << 16) + f.x + bb.x;
    v[2 * j + 1] = __uint_as_float(xw & 0xffff0000u) + f.y + bb.y;
  }
  layer_norm_row<PER2>(v, eps, ln2, ln2 + hidden, lane, y + (size_t)row * (hidden / 2));
}

}  // namespace lf
