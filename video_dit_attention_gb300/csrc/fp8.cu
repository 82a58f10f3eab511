// FP8 (e4m3) preparation for the FP8 attention: the split-halves rotation of q and k, then
// quantisation of q~ with one scale per 128-row tile of a head, and of k~ and v with one
// scale per head (b, h), each scale = amax / 448 over the valid rows (1 when the amax is 0);
// x8 = e4m3(x / scale), round to nearest even, saturating. v is written transposed,
// [B, H, D, S] (keys contiguous), so that the attention's P.V product reads it K-major. Pad
// rows become 0. Two launches: the tile maxima, then the quantisation.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kD = 128;           // head dimension of the FP8 path
constexpr float kE4m3Max = 448.f;

// Block (b, h, tile, tensor) of a launch over B * H * (nt_q + 2 * nt_k) blocks: tensor 0 = q
// (tiles over Sq), 1 = k, 2 = v (tiles over Skv).
struct Fp8Block {
  int kind, b, h, t;
};
__device__ __forceinline__ Fp8Block fp8_block(int B, int H, int nt_q, int nt_k) {
  int idx = blockIdx.x;
  const int nq = B * H * nt_q, nk = B * H * nt_k;
  Fp8Block r;
  int nt;
  if (idx < nq) {
    r.kind = 0;
    nt = nt_q;
  } else if (idx < nq + nk) {
    r.kind = 1;
    idx -= nq;
    nt = nt_k;
  } else {
    r.kind = 2;
    idx -= nq + nk;
    nt = nt_k;
  }
  r.t = idx % nt;
  const int bh = idx / nt;
  r.h = bh % H;
  r.b = bh / H;
  return r;
}

// The sixteen channels of a row that lane unit u (0..7) holds: 8u .. 8u+7 of the first half
// and the matching eight of the second half, rotated when cos/sin rows are given (pair i is
// channels (i, i + 64)). Eight lanes cover a row with two 128-byte segments.
__device__ __forceinline__ void load_unit(const uint16_t* __restrict__ xr, const float* ct, const float* st,
                                          int u, float (&y)[16]) {
  const uint4 a = *reinterpret_cast<const uint4*>(xr + 8 * u);
  const uint4 b = *reinterpret_cast<const uint4*>(xr + kD / 2 + 8 * u);
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
  float x1[8], x2[8];
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    x1[2 * w] = bf16lo_to_f32(aw[w]);
    x1[2 * w + 1] = bf16hi_to_f32(aw[w]);
    x2[2 * w] = bf16lo_to_f32(bw[w]);
    x2[2 * w + 1] = bf16hi_to_f32(bw[w]);
  }
  if (ct != nullptr) {
    const float4 c0 = *reinterpret_cast<const float4*>(ct + 8 * u), c1 = *reinterpret_cast<const float4*>(ct + 8 * u + 4);
    const float4 s0 = *reinterpret_cast<const float4*>(st + 8 * u), s1 = *reinterpret_cast<const float4*>(st + 8 * u + 4);
    const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[i] = fmaf(x1[i], cs[i], -x2[i] * sn[i]);
      y[8 + i] = fmaf(x1[i], sn[i], x2[i] * cs[i]);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      y[i] = x1[i];
      y[8 + i] = x2[i];
    }
  }
}

struct Fp8Args {
  const uint16_t* x[3];    // q, k, v
  const float* cos_t[2];   // q, k tables (null: no rotation)
  const float* sin_t[2];
  int B, Sq, Skv, H, q_valid, kv_valid, nt_q, nt_k;
  float* amax[3];          // [B, H, nt_q], [B, H, nt_k], [B, H, nt_k]
  uint8_t* q8;             // [B, Sq, H, D]
  uint8_t* k8;             // [B, Skv, H, D]
  uint8_t* vt8;            // [B, H, D, Skv]
  float* sq;               // [B, H, nt_q]
  float* sk;               // [B, H]
  float* sv;               // [B, H]
};

// 256 threads: warp w takes rows 4w .. 4w + 3, then 32 further on, ...; eight lanes per row.
__global__ void __launch_bounds__(256) fp8_amax_kernel(const Fp8Args a) {
  const Fp8Block blk = fp8_block(a.B, a.H, a.nt_q, a.nt_k);
  const int S = blk.kind == 0 ? a.Sq : a.Skv, valid = blk.kind == 0 ? a.q_valid : a.kv_valid;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, u = lane & 7;
  const float* ct = blk.kind < 2 ? a.cos_t[blk.kind] : nullptr;
  const float* st = blk.kind < 2 ? a.sin_t[blk.kind] : nullptr;
  float m = 0.f;
  const int n_rows = min(128, valid - blk.t * 128);   // valid rows of this tile (may be <= 0)
#pragma unroll 2
  for (int rr = warp * 4 + (lane >> 3); rr < n_rows; rr += 32) {
    const int row = blk.t * 128 + rr;
    const uint16_t* xr = a.x[blk.kind] + ((static_cast<size_t>(blk.b) * S + row) * a.H + blk.h) * kD;
    float y[16];
    load_unit(xr, ct ? ct + static_cast<size_t>(row) * (kD / 2) : nullptr,
              st ? st + static_cast<size_t>(row) * (kD / 2) : nullptr, u, y);
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(y[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[8];
  if (lane == 0) wm[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = wm[0];
    for (int i = 1; i < 8; ++i) r = fmaxf(r, wm[i]);
    const int nt = blk.kind == 0 ? a.nt_q : a.nt_k;
    a.amax[blk.kind][(blk.b * a.H + blk.h) * nt + blk.t] = r;
  }
}

__device__ __forceinline__ float fp8_scale(float amax) { return amax > 0.f ? amax / kE4m3Max : 1.f; }

__global__ void __launch_bounds__(256) fp8_quantize_kernel(const Fp8Args a) {
  const Fp8Block blk = fp8_block(a.B, a.H, a.nt_q, a.nt_k);
  const int S = blk.kind == 0 ? a.Sq : a.Skv, valid = blk.kind == 0 ? a.q_valid : a.kv_valid;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blk.b * a.H + blk.h;
  float scale;
  if (blk.kind == 0) {
    scale = fp8_scale(a.amax[0][bh * a.nt_q + blk.t]);
  } else {
    float m = 0.f;
    for (int t = 0; t < a.nt_k; ++t) m = fmaxf(m, a.amax[blk.kind][bh * a.nt_k + t]);
    scale = fp8_scale(m);
  }
  if (threadIdx.x == 0) {
    if (blk.kind == 0) a.sq[bh * a.nt_q + blk.t] = scale;
    else if (blk.t == 0) (blk.kind == 1 ? a.sk : a.sv)[bh] = scale;
  }
  const float* ct = blk.kind < 2 ? a.cos_t[blk.kind] : nullptr;
  const float* st = blk.kind < 2 ? a.sin_t[blk.kind] : nullptr;
  // v only: [d][key] for the transposed write, rows padded to 132 bytes (the 16 byte
  // stores of a lane go to channels 8u + i and 64 + 8u + i of one key).
  constexpr int kTS = 132;
  __shared__ __align__(16) uint8_t tile[kD * kTS];
  const int u = lane & 7;
#pragma unroll 2
  for (int rr = warp * 4 + (lane >> 3); rr < 128; rr += 32) {
    const int row = blk.t * 128 + rr;
    uint32_t e[4] = {0u, 0u, 0u, 0u};   // e4m3 of the 16 channels, 4 per word; pads stay 0
    if (row < valid) {
      const uint16_t* xr = a.x[blk.kind] + ((static_cast<size_t>(blk.b) * S + row) * a.H + blk.h) * kD;
      float y[16];
      load_unit(xr, ct ? ct + static_cast<size_t>(row) * (kD / 2) : nullptr,
                st ? st + static_cast<size_t>(row) * (kD / 2) : nullptr, u, y);
#pragma unroll
      for (int w = 0; w < 4; ++w)
        e[w] = pack_e4m3x2(y[4 * w] / scale, y[4 * w + 1] / scale) |
               (pack_e4m3x2(y[4 * w + 2] / scale, y[4 * w + 3] / scale) << 16);
    }
    if (blk.kind < 2) {
      uint8_t* dst = (blk.kind == 0 ? a.q8 : a.k8) + ((static_cast<size_t>(blk.b) * S + row) * a.H + blk.h) * kD;
      *reinterpret_cast<uint2*>(dst + 8 * u) = make_uint2(e[0], e[1]);
      *reinterpret_cast<uint2*>(dst + kD / 2 + 8 * u) = make_uint2(e[2], e[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        tile[(8 * u + i) * kTS + rr] = static_cast<uint8_t>(e[i >> 2] >> (8 * (i & 3)));
        tile[(kD / 2 + 8 * u + i) * kTS + rr] = static_cast<uint8_t>(e[2 + (i >> 2)] >> (8 * (i & 3)));
      }
    }
  }
  if (blk.kind == 2) {
    __syncthreads();
    // 128 rows (channels) of 128 keys: 1024 chunks of 16 bytes, four per thread.
    for (int c = threadIdx.x; c < kD * 8; c += 256) {
      const int d = c >> 3, kc = (c & 7) * 16;
      if (blk.t * 128 + kc < a.Skv) {
        uint8_t* dst = a.vt8 + (static_cast<size_t>(bh) * kD + d) * a.Skv + blk.t * 128 + kc;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + d * kTS + kc);   // 4-byte aligned
        *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
      }
    }
  }
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

}  // namespace

Fp8Layout fp8_layout(int B, int Sq, int Skv, int H, int D) {
  Fp8Layout L{};
  L.nt_q = (Sq + 127) / 128;
  L.nt_k = (Skv + 127) / 128;
  size_t o = 0;
  L.q8 = o;
  o += round256(static_cast<size_t>(B) * Sq * H * D);
  L.k8 = o;
  o += round256(static_cast<size_t>(B) * Skv * H * D);
  L.vt8 = o;
  o += round256(static_cast<size_t>(B) * H * D * Skv);
  L.amax_q = o;
  o += round256(static_cast<size_t>(B) * H * L.nt_q * 4);
  L.amax_k = o;
  o += round256(static_cast<size_t>(B) * H * L.nt_k * 4);
  L.amax_v = o;
  o += round256(static_cast<size_t>(B) * H * L.nt_k * 4);
  L.sq = o;
  o += round256(static_cast<size_t>(B) * H * L.nt_q * 4);
  L.sk = o;
  o += round256(static_cast<size_t>(B) * H * 4);
  L.sv = o;
  o += round256(static_cast<size_t>(B) * H * 4);
  L.total = o;
  return L;
}

cudaError_t launch_fp8_prepare(const AttnArgs& a, const Fp8Layout& L) {
  char* ws = static_cast<char*>(a.workspace);
  Fp8Args f;
  f.x[0] = static_cast<const uint16_t*>(a.q);
  f.x[1] = static_cast<const uint16_t*>(a.k);
  f.x[2] = static_cast<const uint16_t*>(a.v);
  f.cos_t[0] = a.cos_q;
  f.sin_t[0] = a.sin_q;
  f.cos_t[1] = a.cos_k;
  f.sin_t[1] = a.sin_k;
  f.B = a.B;
  f.Sq = a.Sq;
  f.Skv = a.Skv;
  f.H = a.H;
  f.q_valid = a.q_valid;
  f.kv_valid = a.kv_valid;
  f.nt_q = L.nt_q;
  f.nt_k = L.nt_k;
  f.amax[0] = reinterpret_cast<float*>(ws + L.amax_q);
  f.amax[1] = reinterpret_cast<float*>(ws + L.amax_k);
  f.amax[2] = reinterpret_cast<float*>(ws + L.amax_v);
  f.q8 = reinterpret_cast<uint8_t*>(ws + L.q8);
  f.k8 = reinterpret_cast<uint8_t*>(ws + L.k8);
  f.vt8 = reinterpret_cast<uint8_t*>(ws + L.vt8);
  f.sq = reinterpret_cast<float*>(ws + L.sq);
  f.sk = reinterpret_cast<float*>(ws + L.sk);
  f.sv = reinterpret_cast<float*>(ws + L.sv);
  const int blocks = a.B * a.H * (L.nt_q + 2 * L.nt_k);
  fp8_amax_kernel<<<blocks, 256, 0, a.stream>>>(f);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fp8_quantize_kernel<<<blocks, 256, 0, a.stream>>>(f);
  return cudaGetLastError();
}

}  // namespace dit
