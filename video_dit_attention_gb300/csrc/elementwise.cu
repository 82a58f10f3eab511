// Memory-bound kernels: standalone split-halves RoPE, the LSE merge of key-shard partials,
// and the token-row copies used to pad and unpad sequences. All use 16-byte vector accesses,
// are coalesced along the contiguous BSHD rows and use grid-stride loops over a grid sized
// to a multiple of the SM count.

#include <cuda_bf16.h>

#include "common.h"
#include "exp2_fma.cuh"
#include "ptx.cuh"
#include "qknorm.cuh"

namespace dit {
namespace {

// Grid of a grid-stride kernel: enough CTAs for the items, at most 8 per SM of the current
// device (asked per launch, so devices with different SM counts each get their own cap).
int grid_for(long long items, int threads) {
  int dev = 0, sm_count = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sm_count < 1)
    sm_count = 1;   // the loops stride over the grid, so any grid size is correct
  const long long need = (items + threads - 1) / threads;
  const long long cap = static_cast<long long>(sm_count) * 8;
  long long g = need < cap ? need : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

// ------------------------------------------------------------------------------------
// Split-halves RoPE (Difflet PR #153, split RoPE commit): channel i pairs with i + D/2.
// One work item = one (b, s, h) row and one 8-pair chunk: two 16-byte loads of x, four
// 16-byte loads of the table row s (shared by the H heads of that token, so L1/L2 hits),
// two 16-byte stores.
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) rope_split_halves_kernel(const uint16_t* x,
                                                                uint16_t* y,
                                                                const float* __restrict__ cos_t,
                                                                const float* __restrict__ sin_t,
                                                                long long rows, int S, int H) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8;
  const long long items = rows * kChunks;
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = it / kChunks;
    const int ch = static_cast<int>(it % kChunks);
    const int s = static_cast<int>((row / H) % S);
    const uint16_t* xr = x + row * D + ch * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(xr);
    const uint4 bv = *reinterpret_cast<const uint4*>(xr + kHalf);
    const float* ct = cos_t + static_cast<long long>(s) * kHalf + ch * 8;
    const float* st = sin_t + static_cast<long long>(s) * kHalf + ch * 8;
    const float4 c0 = __ldg(reinterpret_cast<const float4*>(ct));
    const float4 c1 = __ldg(reinterpret_cast<const float4*>(ct + 4));
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(st));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(st + 4));
    const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    const uint32_t bw[4] = {bv.x, bv.y, bv.z, bv.w};
    uint32_t ya[4], yb[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float x1l = bf16lo_to_f32(aw[w]), x1h = bf16hi_to_f32(aw[w]);
      const float x2l = bf16lo_to_f32(bw[w]), x2h = bf16hi_to_f32(bw[w]);
      const float cl = cs[2 * w], chh = cs[2 * w + 1], sl = sn[2 * w], sh = sn[2 * w + 1];
      ya[w] = pack_bf16x2(fmaf(x1l, cl, -x2l * sl), fmaf(x1h, chh, -x2h * sh));
      yb[w] = pack_bf16x2(fmaf(x1l, sl, x2l * cl), fmaf(x1h, sh, x2h * chh));
    }
    uint16_t* yr = y + row * D + ch * 8;
    *reinterpret_cast<uint4*>(yr) = make_uint4(ya[0], ya[1], ya[2], ya[3]);
    *reinterpret_cast<uint4*>(yr + kHalf) = make_uint4(yb[0], yb[1], yb[2], yb[3]);
  }
}

// ------------------------------------------------------------------------------------
// Per-head RMSNorm then split-halves RoPE (qknorm.cuh), bf16 in and out. The D/16 threads
// of a row are adjacent lanes of one warp; they reduce the row's sum of squares with
// shuffles. The loop advances whole warps together so that every lane takes part in each
// shuffle (a group of lanes is either a whole row or past the end).
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) qk_rmsnorm_rope_kernel(const uint16_t* x, uint16_t* y,
                                                             const float* __restrict__ w, float eps,
                                                             const float* __restrict__ cos_t,
                                                             const float* __restrict__ sin_t,
                                                             long long rows, int S, int H) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8;
  const long long items = rows * kChunks;
  const int lane = threadIdx.x & 31;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31);
       base < items; base += stride) {
    const long long it = base + lane;
    const bool valid = it < items;
    const long long row = valid ? it / kChunks : 0;
    const int ch = static_cast<int>(it % kChunks);
    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
    // Weights and table rows are loaded together with the data, ahead of the shuffles, so
    // that their latency overlaps the data's.
    float wa[8], wb[8], cs[8], sn[8];
    if (valid) {
      a = *reinterpret_cast<const uint4*>(x + row * D + ch * 8);
      b = *reinterpret_cast<const uint4*>(x + row * D + kHalf + ch * 8);
      const int s = static_cast<int>((row / H) % S);
      load8f(w + ch * 8, wa);
      load8f(w + kHalf + ch * 8, wb);
      load8f(cos_t + static_cast<long long>(s) * kHalf + ch * 8, cs);
      load8f(sin_t + static_cast<long long>(s) * kHalf + ch * 8, sn);
    }
    float ss = sumsq16(a, b);
#pragma unroll
    for (int off = 1; off < kChunks; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (valid) {
      const float inv = rsqrtf(ss * (1.f / D) + eps);
      norm_rotate8<false>(a, b, inv, wa, wb, cs, sn);
      *reinterpret_cast<uint4*>(y + row * D + ch * 8) = a;
      *reinterpret_cast<uint4*>(y + row * D + kHalf + ch * 8) = b;
    }
  }
}

// ------------------------------------------------------------------------------------
// LSE merge (mstar PR #376, attention over sharded keys):
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) O_s.
// D/8 threads per (b, s, h) row, each owning 8 channels (16-byte loads of every partial);
// the n partial LSEs of the row are read by all of its threads (same cache lines).
// ------------------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) lse_merge_kernel(const uint16_t* __restrict__ po,
                                                        const float* __restrict__ pl, int n,
                                                        long long rows, uint16_t* __restrict__ out,
                                                        float* __restrict__ lse) {
  constexpr int kTPR = D / 8;   // threads per row
  const long long items = rows * kTPR;
  const long long part_stride = rows * D;
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = it / kTPR;
    const int ch = static_cast<int>(it % kTPR);
    float m = -INFINITY;
    for (int s = 0; s < n; ++s) m = fmaxf(m, __ldg(pl + s * rows + row));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float lse_row = -INFINITY;
    if (m > -INFINITY) {
      float tot = 0.f;
      for (int s = 0; s < n; ++s) tot += __expf(__ldg(pl + s * rows + row) - m);
      lse_row = m + __logf(tot);
      for (int s = 0; s < n; ++s) {
        const float w = __expf(__ldg(pl + s * rows + row) - lse_row);
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(po + s * part_stride + row * D + ch * 8));
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(w, bf16lo_to_f32(vw[q]), acc[2 * q]);
          acc[2 * q + 1] = fmaf(w, bf16hi_to_f32(vw[q]), acc[2 * q + 1]);
        }
      }
    }
    *reinterpret_cast<uint4*>(out + row * D + ch * 8) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    if (ch == 0) lse[row] = lse_row;
  }
}

// lse_merge_kernel for a fixed number of partials N (1..8): the N partial LSEs and the N
// 16-byte pieces of partial O are all loaded before any arithmetic, so each thread has N + N
// independent loads in flight instead of a chain through the loop.
template <int D, int N>
__global__ void __launch_bounds__(256) lse_merge_fixed_kernel(const uint16_t* __restrict__ po,
                                                              const float* __restrict__ pl, long long rows,
                                                              uint16_t* __restrict__ out,
                                                              float* __restrict__ lse) {
  constexpr int kTPR = D / 8;
  const long long items = rows * kTPR;
  const long long part_stride = rows * D;
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = it / kTPR;
    const int ch = static_cast<int>(it % kTPR);
    float ls[N];
    uint4 v[N];
#pragma unroll
    for (int s = 0; s < N; ++s) {
      ls[s] = __ldg(pl + s * rows + row);
      v[s] = __ldg(reinterpret_cast<const uint4*>(po + s * part_stride + row * D + ch * 8));
    }
    float m = ls[0];
#pragma unroll
    for (int s = 1; s < N; ++s) m = fmaxf(m, ls[s]);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float lse_row = -INFINITY;
    if (m > -INFINITY) {
      float tot = 0.f;
#pragma unroll
      for (int s = 0; s < N; ++s) tot += __expf(ls[s] - m);
      lse_row = m + __logf(tot);
#pragma unroll
      for (int s = 0; s < N; ++s) {
        const float w = __expf(ls[s] - lse_row);
        const uint32_t vw[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          acc[2 * q] = fmaf(w, bf16lo_to_f32(vw[q]), acc[2 * q]);
          acc[2 * q + 1] = fmaf(w, bf16hi_to_f32(vw[q]), acc[2 * q + 1]);
        }
      }
    }
    *reinterpret_cast<uint4*>(out + row * D + ch * 8) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    if (ch == 0) lse[row] = lse_row;
  }
}

// ------------------------------------------------------------------------------------
// Row copies for pad / unpad: rows [0, L) of each batch, row_bytes per token row.
// ------------------------------------------------------------------------------------
template <typename V>
__global__ void __launch_bounds__(256) copy_rows_kernel(const uint8_t* __restrict__ src,
                                                        uint8_t* __restrict__ dst, int L,
                                                        long long src_rows, long long dst_rows,
                                                        long long row_vecs, long long total) {
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < total;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long per_batch = static_cast<long long>(L) * row_vecs;
    const long long bb = it / per_batch;
    const long long rem = it % per_batch;
    const V* s = reinterpret_cast<const V*>(src) + bb * src_rows * row_vecs + rem;
    V* d = reinterpret_cast<V*>(dst) + bb * dst_rows * row_vecs + rem;
    *d = *s;
  }
}

// The attention kernel's FMA-pipe exp2 applied to an array (diagnostic).
__global__ void __launch_bounds__(256) exp2_fma_kernel(const float* __restrict__ x,
                                                       float* __restrict__ y, long long n) {
  for (long long i = 2 * (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x); i < n;
       i += 2 * static_cast<long long>(gridDim.x) * blockDim.x) {
    float y0, y1;
    exp2_fma2(y0, y1, x[i], i + 1 < n ? x[i + 1] : 0.f);
    y[i] = y0;
    if (i + 1 < n) y[i + 1] = y1;
  }
}

}  // namespace

cudaError_t launch_exp2_fma(const float* x, float* y, long long n, cudaStream_t stream) {
  exp2_fma_kernel<<<grid_for((n + 1) / 2, 256), 256, 0, stream>>>(x, y, n);
  return cudaGetLastError();
}

cudaError_t launch_rope_split_halves(const void* x, void* y, const float* cos_tab,
                                     const float* sin_tab, int B, int S, int H, int D,
                                     cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * S * H;
  const long long items = rows * (D / 16);
  const int grid = grid_for(items, 256);
  if (D == 128)
    rope_split_halves_kernel<128><<<grid, 256, 0, stream>>>(
        static_cast<const uint16_t*>(x), static_cast<uint16_t*>(y), cos_tab, sin_tab, rows, S, H);
  else
    rope_split_halves_kernel<64><<<grid, 256, 0, stream>>>(
        static_cast<const uint16_t*>(x), static_cast<uint16_t*>(y), cos_tab, sin_tab, rows, S, H);
  return cudaGetLastError();
}

cudaError_t launch_qk_rmsnorm_rope(const void* x, void* y, const float* w, float eps,
                                   const float* cos_tab, const float* sin_tab, int B, int S, int H,
                                   int D, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * S * H;
  const long long items = rows * (D / 16);
  const int grid = grid_for(items, 256);
  if (D == 128)
    qk_rmsnorm_rope_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x),
                                                          static_cast<uint16_t*>(y), w, eps, cos_tab,
                                                          sin_tab, rows, S, H);
  else
    qk_rmsnorm_rope_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(x),
                                                         static_cast<uint16_t*>(y), w, eps, cos_tab,
                                                         sin_tab, rows, S, H);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(const void* partial_o, const float* partial_lse, int n, int B,
                             int S, int H, int D, void* out, float* lse, cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * S * H;
  const long long items = rows * (D / 8);
  const int grid = grid_for(items, 256);
  const uint16_t* po = static_cast<const uint16_t*>(partial_o);
  uint16_t* o = static_cast<uint16_t*>(out);
  if (n >= 1 && n <= 8) {
    // One instantiation per (D, n): the partials' loads are unrolled.
    using Fn = void (*)(const uint16_t*, const float*, long long, uint16_t*, float*);
    static constexpr Fn k128[8] = {lse_merge_fixed_kernel<128, 1>, lse_merge_fixed_kernel<128, 2>,
                                   lse_merge_fixed_kernel<128, 3>, lse_merge_fixed_kernel<128, 4>,
                                   lse_merge_fixed_kernel<128, 5>, lse_merge_fixed_kernel<128, 6>,
                                   lse_merge_fixed_kernel<128, 7>, lse_merge_fixed_kernel<128, 8>};
    static constexpr Fn k64[8] = {lse_merge_fixed_kernel<64, 1>, lse_merge_fixed_kernel<64, 2>,
                                  lse_merge_fixed_kernel<64, 3>, lse_merge_fixed_kernel<64, 4>,
                                  lse_merge_fixed_kernel<64, 5>, lse_merge_fixed_kernel<64, 6>,
                                  lse_merge_fixed_kernel<64, 7>, lse_merge_fixed_kernel<64, 8>};
    (D == 128 ? k128 : k64)[n - 1]<<<grid, 256, 0, stream>>>(po, partial_lse, rows, o, lse);
    return cudaGetLastError();
  }
  if (D == 128)
    lse_merge_kernel<128><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(partial_o),
                                                    partial_lse, n, rows,
                                                    static_cast<uint16_t*>(out), lse);
  else
    lse_merge_kernel<64><<<grid, 256, 0, stream>>>(static_cast<const uint16_t*>(partial_o),
                                                   partial_lse, n, rows,
                                                   static_cast<uint16_t*>(out), lse);
  return cudaGetLastError();
}

cudaError_t launch_copy_rows(const void* src, void* dst, int B, int L, long long src_rows,
                             long long dst_rows, long long row_bytes, cudaStream_t stream) {
  if (L == 0) return cudaSuccess;
  const uintptr_t align = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                          static_cast<uintptr_t>(row_bytes);
  const uint8_t* s = static_cast<const uint8_t*>(src);
  uint8_t* d = static_cast<uint8_t*>(dst);
  if ((align & 15) == 0) {
    const long long vecs = row_bytes / 16, total = static_cast<long long>(B) * L * vecs;
    copy_rows_kernel<uint4><<<grid_for(total, 256), 256, 0, stream>>>(s, d, L, src_rows, dst_rows, vecs, total);
  } else if ((align & 3) == 0) {
    const long long vecs = row_bytes / 4, total = static_cast<long long>(B) * L * vecs;
    copy_rows_kernel<uint32_t><<<grid_for(total, 256), 256, 0, stream>>>(s, d, L, src_rows, dst_rows, vecs, total);
  } else {
    const long long vecs = row_bytes, total = static_cast<long long>(B) * L * vecs;
    copy_rows_kernel<uint8_t><<<grid_for(total, 256), 256, 0, stream>>>(s, d, L, src_rows, dst_rows, vecs, total);
  }
  return cudaGetLastError();
}

}  // namespace dit
