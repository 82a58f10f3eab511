// Per-head RMSNorm of q / k followed by the split-halves rotation, for 8 channel pairs of
// one row (Difflet PR #153, FLUX and Wan split-RoPE commits: the per-head qk RMSNorm weights
// are permuted with the q/k channels, so the norm acts in the split-halves layout, just
// before the rotation):
//   n = x / sqrt(mean_d(x_d^2) + eps) * w,
//   y[i] = n[i] cos - n[i + D/2] sin,  y[i + D/2] = n[i] sin + n[i + D/2] cos.
// The caller reduces the row's sum of squares (sumsq16 over its 16 values, then across the
// D/16 threads that share the row) and passes inv = 1 / sqrt(sumsq / D + eps).
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace dit {

// Sum of squares of 16 bf16 values: 8 of the first half (a) and the 8 matching values of the
// second half (b), accumulated in fp32 in a fixed order.
__device__ __forceinline__ float sumsq16(const uint4 a, const uint4 b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float x1l = bf16lo_to_f32(aw[w]), x1h = bf16hi_to_f32(aw[w]);
    const float x2l = bf16lo_to_f32(bw[w]), x2h = bf16hi_to_f32(bw[w]);
    s = fmaf(x1l, x1l, s);
    s = fmaf(x1h, x1h, s);
    s = fmaf(x2l, x2l, s);
    s = fmaf(x2h, x2h, s);
  }
  return s;
}

// Normalises and rotates 8 channel pairs in place: a holds channels c..c+7 of the first half,
// b the matching channels of the second half (bf16 in; fp16, saturating, when kF16, else
// bf16 out); wa / wb the norm weights of those channels, cs / sn the 8 cos / sin values.
template <bool kF16>
__device__ __forceinline__ void norm_rotate8(uint4& a, uint4& b, float inv, const float (&wa)[8],
                                             const float (&wb)[8], const float (&cs)[8],
                                             const float (&sn)[8]) {
  uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int l = 2 * w, h = 2 * w + 1;
    const float x1l = bf16lo_to_f32(aw[w]) * inv * wa[l], x1h = bf16hi_to_f32(aw[w]) * inv * wa[h];
    const float x2l = bf16lo_to_f32(bw[w]) * inv * wb[l], x2h = bf16hi_to_f32(bw[w]) * inv * wb[h];
    const float y1l = fmaf(x1l, cs[l], -x2l * sn[l]), y1h = fmaf(x1h, cs[h], -x2h * sn[h]);
    const float y2l = fmaf(x1l, sn[l], x2l * cs[l]), y2h = fmaf(x1h, sn[h], x2h * cs[h]);
    aw[w] = kF16 ? pack_f16x2_satfinite(y1l, y1h) : pack_bf16x2(y1l, y1h);
    bw[w] = kF16 ? pack_f16x2_satfinite(y2l, y2h) : pack_bf16x2(y2l, y2h);
  }
  a = make_uint4(aw[0], aw[1], aw[2], aw[3]);
  b = make_uint4(bw[0], bw[1], bw[2], bw[3]);
}

// Loads 8 consecutive fp32 values (16-byte aligned) into an array.
__device__ __forceinline__ void load8f(const float* __restrict__ p, float (&v)[8]) {
  const float4 x = __ldg(reinterpret_cast<const float4*>(p));
  const float4 y = __ldg(reinterpret_cast<const float4*>(p + 4));
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}

}  // namespace dit
