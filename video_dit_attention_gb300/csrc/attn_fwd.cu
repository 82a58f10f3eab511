// Flash-attention forward for sm_103a on tcgen05 tensor cores, with exact pad-key masking,
// natural-log LSE output and (optionally) split-halves RoPE fused into the q/k tile load.
// This file holds the kernel for RoPE applied per loaded tile (P kept in TMEM); the plain,
// workspace-RoPE, sharded-keys and FP8 modes run attn_sp_kernel (attn_sp.cuh, P staged in
// shared memory), which shares the helpers, work items and parameters defined here. Short-KV
// cross-attention has a kernel of its own (cross_attn.cu).
//
// What it computes (Difflet PR #153: pad keys dropped exactly, pad rows rotated by the
// identity; maxdiffusion PR #491: the real KV length as the ragged tail; mstar PR #376: the
// LSE in natural log returned beside O): for every (batch b, head h, query row i < q_valid)
//   s_j = scale * (R_q(i) q_i) . (R_k(j) k_j)   for j < kv_valid
//   lse_i = ln sum_j exp(s_j),  O_i = sum_j exp(s_j - lse_i) v_j,
// and O = 0, lse = -inf for pad query rows. It is the online-softmax (flash) form of that
// definition: keys are visited in 128-key tiles and the running max/sum are rescaled.
//
// Work items are two 128-row query tiles (Q0, Q1) of one (b, h), which share every K/V tile
// and its rotation; the kernel is persistent (one CTA per SM, items round-robin, see below).
// Warp roles (512 threads):
//   warp 0       TMA producer: Q0/Q1 once, then K_j / V_j into a ring of shared-memory stages.
//   warp 12      single-thread tcgen05.mma issuer (warp 1 allocates TMEM). Per key tile j it
//                issues, in this order, O0 += P0_{j-1} V_{j-1}, S0_j = Q0 K_j^T,
//                O1 += P1_{j-1} V_{j-1}, S1_j = Q1 K_j^T. tcgen05.mma ops of a CTA run in
//                issue order, so S_t,j may reuse the TMEM columns that held P_t,j-1 and its
//                completion also implies that O_t holds P_t,j-1 V_j-1.
//   warps 4-7    softmax of Q0, warps 8-11 softmax of Q1 (thread = query row = TMEM lane).
//                Each reads S_t,j with tcgen05.ld, masks keys >= kv_valid, keeps the running
//                max m and sum l, and writes P_t,j as bf16 over the first 64 columns of S_t,j
//                in TMEM (the A operand of the P V MMA). While one group computes softmax the
//                tensor core works on the other tile (ping-pong). O_t is rescaled in TMEM only
//                when m grows by more than 2^8; the final O / l is exact for any reference m.
//                Epilogue: O / l to bf16, LSE.
//   warps 13-15  auxiliary: RoPE rotation of the landed Q and K tiles in shared memory
//                (pairs (i, i + D/2) sit at the same swizzled offset of the two 64-column
//                halves of a row).
//                The rotation is computed in fp32 from the bf16 inputs and stored as fp16
//                (11-bit significand, 8x finer than bf16; saturating at +-65504), and S =
//                q~ k~^T then runs as an fp16 x fp16 MMA at the same tensor-core rate. Without
//                RoPE, q and k are used as the bf16 values they are.
// Every mbarrier wait is bounded (ptx.cuh); on a timeout the CTA records a status bit,
// drains what it has in flight, frees TMEM and exits.
//
// Shared memory (128-byte swizzle, tiles 1024-byte aligned): Q0, Q1 [128 x D], K and V
// stages [128 x D]. Each [128 x D] tile is D/64 sub-tiles of 128 rows x 128 B.
// TMEM (512 columns): S0/P0 0..127, S1/P1 128..255, O0 256..383, O1 384..511.

#include <cuda_bf16.h>

#include <cstring>
#include <mutex>
#include <type_traits>

#include "common.h"
#include "exp2_fma.cuh"
#include "ptx.cuh"
#include "qknorm.cuh"

namespace dit {

__device__ unsigned int g_dit_status;

namespace {

constexpr int kThreads = 512;
constexpr int kAuxThreads = 96;   // warps 13-15: RoPE rotation, or zeroing of V pad rows
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only if m grows by > 2^8
constexpr int kPrefetchLead = 6;  // key tiles before an item's end at which the next is warmed
constexpr int kPrefetchKV = 4;    // K/V tiles of the next item warmed in L2
// Column pairs (index 0..7 within a 16-column piece) whose exponentials run on the FMA pipe
// (exp2_fma2) instead of the special-function unit. Measured on GB300 at 1/4, 3/8 and 1/2 of
// the pairs this was slower than none (the softmax is not bound by ex2 throughput), so none.
constexpr uint32_t kFmaExpPairs = 0;

template <int D>
struct Cfg {
  static constexpr int kSub = D / 64;               // 64-column sub-tiles per row
  static constexpr int kTileBytes = 128 * D * 2;    // one 128-row q/k/v tile
  static constexpr int kStagesK = (D == 128) ? 2 : 4;
  static constexpr int kStagesV = (D == 128) ? 2 : 4;
  static constexpr int kTabRows = 32;                       // rows per staged table quarter
  static constexpr int kTabBoxBytes = kTabRows * (D / 2) * 4;  // cos (or sin) of a quarter
  static constexpr int kOffQ = 0;                   // Q0, Q1
  static constexpr int kOffK = kOffQ + 2 * kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
  static constexpr int kOffT = kOffV + kStagesV * kTileBytes;   // 2 x (cos, sin) quarters
  static constexpr int kOffBar = kOffT + 2 * 2 * kTabBoxBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;   // barriers + alignment slack
};

struct Bars {
  uint64_t q_full, q_ready;
  uint64_t k_full[4], k_ready[4], k_empty[4];
  uint64_t v_full[4], v_ready[4], v_empty[4];
  uint64_t q_empty;
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t t_full[2], t_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int aux_go;   // outcome of the auxiliary warpgroup's last wait, broadcast to the group
};

struct KParams {
  int Sq, Skv, H;
  int n_pairs, n_items;   // query-tile pairs per (b, h); B * H * n_pairs work items
  int q_valid, kv_valid;
  const float* cos_q;
  const float* sin_q;
  const float* cos_k;
  const float* sin_k;
  float scale_log2;
  uint16_t* out;
  float* lse;
};

// Workspace-mode parameters: the raw keys, their rotated fp16 copy (which the TMA map of k
// points at) and the count of CTAs done rotating (zeroed before launch). Kept apart from
// KParams so the other modes' parameter block stays small.
struct WsParams {
  const uint16_t* k_raw;
  uint16_t* k_rot;
  unsigned int* rotated;
  int B;
  const float* norm_q;   // per-head q/k RMSNorm weights [D] (norm mode only)
  const float* norm_k;
  float norm_eps;
  unsigned int* kmax;      // fixed-m mode: largest squared key norm per (b, h), float bits
  float* qn;               // fixed-m mode: squared norm of each q row [B, Sq, H]
  unsigned int* n_online;  // fixed-m mode: blocks that took the online path (may be null)
  const float* f8_sq;      // FP8 mode: q~ scale per (b, h, 128-row tile) [B, H, f8_nt_q]
  const float* f8_sk;      // FP8 mode: k~ scale per (b, h)
  const float* f8_sv;      // FP8 mode: v scale per (b, h)
  int f8_nt_q;
};

// The RoPE workspace modes (plain, with the q/k RMSNorm, fixed-m softmax, sharded keys).
__host__ __device__ constexpr bool is_ws_mode(int mode) {
  return mode == kModeRopeWs || mode == kModeRopeWsNorm || mode == kModeRopeWsFixedM ||
         mode == kModeRopeWsSharded;
}

// Sharded-keys mode: the keys come in chunks (whole 128-row tiles of one shard each). Chunk c
// has its own raw k rows, rotated copy, table rows, and TMA maps of the rotated k and of v,
// and its own partial output (O_c, LSE_c), merged afterwards through the LSE.
struct KeyChunk {
  const uint16_t* k_raw;   // first row of the chunk in its shard's raw k [B, S_rows, H, D]
  uint16_t* k_rot;         // the same row in the shard's rotated copy (same layout)
  const float* cos_k;      // table rows of the chunk (global key positions)
  const float* sin_k;
  int S_rows;              // rows per batch of the shard (its padded length)
  int valid;               // valid keys in the chunk
};
struct ShardParams {
  CUtensorMap km[kMaxKeyChunks];   // rotated k of each chunk, extent = its valid rows
  CUtensorMap vm[kMaxKeyChunks];   // v of each chunk, extent = its valid rows
  KeyChunk c[kMaxKeyChunks];
  int n_chunks;
  int n_bh;                        // B * H
  long long po_stride, pl_stride;  // elements between consecutive chunks' partial O / LSE
};
struct NoShards {};
template <int kMode>
using ShardArg = typename std::conditional<kMode == kModeRopeWsSharded, ShardParams, NoShards>::type;
// Partial-LSE stride of the sharded mode (0 for the others, which have no ShardParams).
template <int kMode>
struct ShardStride {
  __device__ static long long pl(const ShardArg<kMode>& sh) {
    if constexpr (kMode == kModeRopeWsSharded) return sh.pl_stride;
    else return 0;
  }
};

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// Bounded wait taken by lane 0 of the warp and broadcast, so that every lane leaves with
// the same outcome (the warp then stays converged at .sync.aligned tcgen05 instructions).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* status, unsigned int code) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = bounded_wait(bar, parity, abort_flag, status, code) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  return ok != 0;
}

// Bounded wait taken by one thread of an auxiliary group of NT threads (warps 13-15 by
// default) and broadcast to the group through shared memory and named barrier 1 (all of its
// threads call this).
template <int NT = kAuxThreads>
__device__ __forceinline__ bool group_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned int* status, unsigned int code,
                                           volatile int* go, int at) {
  if (at == 0) *go = bounded_wait(bar, parity, abort_flag, status, code) ? 1 : 0;
  named_bar_sync(1, NT);
  return *go != 0;
}

// Rotates 8 channel pairs: a holds channels c..c+7 of the first half, b the matching
// channels of the second half (bf16x2 words in, f16x2 words out); cs/sn the 8 cos/sin.
__device__ __forceinline__ void rotate8(uint4& a, uint4& b, const float4 c0, const float4 c1,
                                        const float4 s0, const float4 s1) {
  const float cs[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
  uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float x1l = bf16lo_to_f32(aw[w]), x1h = bf16hi_to_f32(aw[w]);
    const float x2l = bf16lo_to_f32(bw[w]), x2h = bf16hi_to_f32(bw[w]);
    const float cl = cs[2 * w], ch = cs[2 * w + 1], sl = sn[2 * w], sh = sn[2 * w + 1];
    aw[w] = pack_f16x2_satfinite(fmaf(x1l, cl, -x2l * sl), fmaf(x1h, ch, -x2h * sh));
    bw[w] = pack_f16x2_satfinite(fmaf(x1l, sl, x2l * cl), fmaf(x1h, sh, x2h * ch));
  }
  a = make_uint4(aw[0], aw[1], aw[2], aw[3]);
  b = make_uint4(bw[0], bw[1], bw[2], bw[3]);
}

// Rotation of one landed [128 x D] tile by the auxiliary group (at = 0 .. kAuxThreads-1),
// one 32-row quarter at a time, with that quarter's cos/sin rows staged in shared memory by
// TMA (fp32, [32][D/2] each, unswizzled). Item i of a quarter is 16-byte chunk i % kChunks of
// row i / kChunks (of the first half and the matching chunk of the second half).
template <int D>
struct Rotator {
  static constexpr int kHalf = D / 2;
  static constexpr int kChunks = kHalf / 8;          // 16-byte chunks per half row
  static constexpr int kItems = 32 * kChunks;        // items per quarter

  __device__ __forceinline__ static void quarter(uint32_t tile, uint32_t tab_cos, uint32_t tab_sin,
                                                 int quarter_idx, int at) {
#pragma unroll
    for (int item = at; item < kItems; item += kAuxThreads) {
      const int rq = item / kChunks, ch = item % kChunks;   // row within the quarter, chunk
      const int row = quarter_idx * 32 + rq;
      const uint32_t toff = static_cast<uint32_t>(rq * kHalf + ch * 8) * 4u;
      const uint4 c0 = lds128(tab_cos + toff), c1 = lds128(tab_cos + toff + 16);
      const uint4 s0 = lds128(tab_sin + toff), s1 = lds128(tab_sin + toff + 16);
      const uint32_t offa = sw128_offset(row, ch);
      const uint32_t offb = (D == 128) ? 16384u + offa : sw128_offset(row, ch + 4);
      uint4 a = lds128(tile + offa), b = lds128(tile + offb);
      rotate8(a, b, make_float4(__uint_as_float(c0.x), __uint_as_float(c0.y), __uint_as_float(c0.z), __uint_as_float(c0.w)),
              make_float4(__uint_as_float(c1.x), __uint_as_float(c1.y), __uint_as_float(c1.z), __uint_as_float(c1.w)),
              make_float4(__uint_as_float(s0.x), __uint_as_float(s0.y), __uint_as_float(s0.z), __uint_as_float(s0.w)),
              make_float4(__uint_as_float(s1.x), __uint_as_float(s1.y), __uint_as_float(s1.z), __uint_as_float(s1.w)));
      sts128(tile + offa, a);
      sts128(tile + offb, b);
    }
  }
};

// O = 0, LSE = -inf for the 128 rows of the query tile starting at q_first (a tile that is
// all pad rows, or a problem with no keys). `tid` ranges over `nthr` cooperating threads.
template <int D>
__device__ __forceinline__ void write_empty_tile(const KParams& p, uint16_t* out, float* lse, int b, int h,
                                                 int q_first, int tid, int nthr) {
  for (int i = tid; i < 128 * (D / 8); i += nthr) {
    const int row = i / (D / 8), ch = i % (D / 8);
    uint16_t* dst = out + ((static_cast<size_t>(b) * p.Sq + q_first + row) * p.H + h) * D + ch * 8;
    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  for (int r = tid; r < 128; r += nthr)
    lse[(static_cast<size_t>(b) * p.Sq + q_first + r) * p.H + h] = -INFINITY;
}

// One unit of work: query rows q0 .. q0 + 255 (two 128-row tiles) of one (b, h).
struct Item {
  int b, h, q0, n_live, n_kv, kv_valid;
  int chunk;      // sharded mode: key chunk of the item
  bool has1;      // tile 1 (rows q0 + 128 ..) lies inside the padded sequence
};

template <int kMode>
__device__ __forceinline__ Item decode_item(const KParams& p, int it) {
  Item w;
  const int pair = it % p.n_pairs, bh = it / p.n_pairs;
  w.h = bh % p.H;
  w.b = bh / p.H;
  w.q0 = pair * 256;
  w.chunk = 0;
  const int kv = p.kv_valid;
  w.kv_valid = kv;
  // Tile t is live if it holds a valid query row and there is at least one key.
  w.has1 = w.q0 + 128 < p.Sq;
  const bool live0 = (w.q0 < p.q_valid) && kv > 0;
  const bool live1 = w.has1 && (w.q0 + 128 < p.q_valid) && kv > 0;
  w.n_live = live1 ? 2 : (live0 ? 1 : 0);
  w.n_kv = (kv + 127) / 128;
  return w;
}

// Sharded mode: items in the order (key chunk, b, h, query-tile pair), so neighbouring CTAs
// share a chunk's K/V; the chunk's valid keys replace the one kv length.
__device__ __forceinline__ Item decode_item_sh(const KParams& p, const ShardParams& sh, int it) {
  Item w;
  const int pair = it % p.n_pairs;
  int bh = it / p.n_pairs;
  w.chunk = bh / sh.n_bh;
  bh -= w.chunk * sh.n_bh;
  w.h = bh % p.H;
  w.b = bh / p.H;
  w.q0 = pair * 256;
  const int kv = sh.c[w.chunk].valid;
  w.kv_valid = kv;
  w.has1 = w.q0 + 128 < p.Sq;
  const bool live0 = (w.q0 < p.q_valid) && kv > 0;
  const bool live1 = w.has1 && (w.q0 + 128 < p.q_valid) && kv > 0;
  w.n_live = live1 ? 2 : (live0 ? 1 : 0);
  w.n_kv = (kv + 127) / 128;
  return w;
}

// Persistent kernel: one CTA per SM walks the items it + k * gridDim.x. Concurrent CTAs thus
// work on neighbouring items of the same heads and share their K/V tiles in L2. Every ring
// and barrier phase runs on counters that continue across items, so the loads, the rotation
// and the first MMAs of the next item overlap the epilogue of the current one.
// Writes the split-halves rotation of rows [0, valid) of x [B, S_rows, H, D] (bf16) as fp16
// into y (same layout), with table rows [S_rows, D/2]. Work items are (row, 8-pair chunk);
// within a batch the valid rows of all heads are contiguous, so consecutive threads read and
// write consecutive 16-byte chunks. Each thread keeps four items in flight.
template <int D>
__device__ __forceinline__ void rotate_rows_fp16(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                 const float* __restrict__ cos_t,
                                                 const float* __restrict__ sin_t, int B, int S_rows,
                                                 int valid, int H, int gtid, int gthreads) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8, kU = 4;
  const int per_b = valid * H * kChunks;
  for (int b = 0; b < B; ++b) {
    const size_t boff = static_cast<size_t>(b) * S_rows * H * D;
    for (int i0 = gtid; i0 < per_b; i0 += kU * gthreads) {
      uint4 a[kU], bb[kU];
      float4 c0[kU], c1[kU], s0[kU], s1[kU];
      size_t off[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = i0 + u * gthreads;
        if (i < per_b) {
          const int ch = i % kChunks, rh = i / kChunks, srow = rh / H;   // rh = srow * H + h
          off[u] = boff + static_cast<size_t>(rh) * D + ch * 8;
          a[u] = *reinterpret_cast<const uint4*>(x + off[u]);
          bb[u] = *reinterpret_cast<const uint4*>(x + off[u] + kHalf);
          const float* ct = cos_t + static_cast<size_t>(srow) * kHalf + ch * 8;
          const float* st = sin_t + static_cast<size_t>(srow) * kHalf + ch * 8;
          c0[u] = __ldg(reinterpret_cast<const float4*>(ct));
          c1[u] = __ldg(reinterpret_cast<const float4*>(ct + 4));
          s0[u] = __ldg(reinterpret_cast<const float4*>(st));
          s1[u] = __ldg(reinterpret_cast<const float4*>(st + 4));
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        if (i0 + u * gthreads < per_b) {
          rotate8(a[u], bb[u], c0[u], c1[u], s0[u], s1[u]);
          *reinterpret_cast<uint4*>(y + off[u]) = a[u];
          *reinterpret_cast<uint4*>(y + off[u] + kHalf) = bb[u];
        }
      }
    }
  }
}

// Rotates, in place and into fp16, a landed [128 x D] bf16 tile in shared memory (128-byte
// swizzle; D = 128: two 64-column sub-tiles, pair (i, i + 64) at the same offset of both;
// D = 64: pair (i, i + 32) in units x and x + 4 of one row) with table rows cos_t / sin_t
// [128, D/2] read from global memory. NT threads, this one is number `at`; each thread has
// kUnroll row units in flight.
template <int D, int NT, int kUnroll = 2>
__device__ __forceinline__ void rotate_tile_smem(uint32_t tile, const float* __restrict__ cos_t,
                                                 const float* __restrict__ sin_t, int at) {
  constexpr int kHalf = D / 2, kUnits = kHalf / 8;   // 8-pair units per row
#pragma unroll kUnroll
  for (int i = at; i < 128 * kUnits; i += NT) {
    const int row = i / kUnits, x = i % kUnits;
    const uint32_t offa = sw128_offset(row, x);
    const uint32_t offb = (D == 128) ? 16384u + offa : sw128_offset(row, x + 4);
    const float* ct = cos_t + row * kHalf + x * 8;
    const float* st = sin_t + row * kHalf + x * 8;
    uint4 a = lds128(tile + offa), b = lds128(tile + offb);
    rotate8(a, b, __ldg(reinterpret_cast<const float4*>(ct)), __ldg(reinterpret_cast<const float4*>(ct + 4)),
            __ldg(reinterpret_cast<const float4*>(st)), __ldg(reinterpret_cast<const float4*>(st + 4)));
    sts128(tile + offa, a);
    sts128(tile + offb, b);
  }
}

// rotate_rows_fp16 with the per-head RMSNorm (weights w [D], eps) applied first. The D/16
// threads of a row are adjacent lanes; they reduce its sum of squares with shuffles, so the
// loop advances whole warps together (gtid's warp-aligned base) and every lane joins each
// shuffle (a group is either a whole row or past the end). gthreads is a multiple of 32.
template <int D>
__device__ __forceinline__ void rotate_rows_fp16_norm(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                      const float* __restrict__ cos_t,
                                                      const float* __restrict__ sin_t,
                                                      const float* __restrict__ w, float eps, int B,
                                                      int S_rows, int valid, int H, int gtid, int gthreads) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8;
  const int per_b = valid * H * kChunks;
  const int lane = gtid & 31;
  for (int b = 0; b < B; ++b) {
    const size_t boff = static_cast<size_t>(b) * S_rows * H * D;
    for (int base = gtid - lane; base < per_b; base += gthreads) {
      const int i = base + lane;
      const bool live = i < per_b;
      const int ch = i % kChunks, rh = live ? i / kChunks : 0, srow = rh / H;
      const size_t off = boff + static_cast<size_t>(rh) * D + ch * 8;
      uint4 a = make_uint4(0, 0, 0, 0), bb = make_uint4(0, 0, 0, 0);
      if (live) {
        a = *reinterpret_cast<const uint4*>(x + off);
        bb = *reinterpret_cast<const uint4*>(x + off + kHalf);
      }
      float ss = sumsq16(a, bb);
#pragma unroll
      for (int o = 1; o < kChunks; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (live) {
        float wa[8], wb[8], cs[8], sn[8];
        load8f(w + ch * 8, wa);
        load8f(w + kHalf + ch * 8, wb);
        load8f(cos_t + static_cast<size_t>(srow) * kHalf + ch * 8, cs);
        load8f(sin_t + static_cast<size_t>(srow) * kHalf + ch * 8, sn);
        norm_rotate8<true>(a, bb, rsqrtf(ss * (1.f / D) + eps), wa, wb, cs, sn);
        *reinterpret_cast<uint4*>(y + off) = a;
        *reinterpret_cast<uint4*>(y + off + kHalf) = bb;
      }
    }
  }
}

// rotate_rows_fp16 that also records, per (b, h), the largest squared norm of the key rows it
// rotates: kmax_s[b * H + h] (shared memory; float bits, which order like unsigned integers
// for non-negative values; zero on entry) through shared-memory atomicMax. The squared norm
// is taken from the bf16 inputs: the rotation preserves it. The loop runs per warp so that
// the D / 16 lanes holding one row can add their partial sums with shuffles.
template <int D>
__device__ __forceinline__ void rotate_rows_fp16_kmax(const uint16_t* __restrict__ x, uint16_t* __restrict__ y,
                                                      const float* __restrict__ cos_t,
                                                      const float* __restrict__ sin_t, int B, int S_rows,
                                                      int valid, int H, int gtid, int gthreads,
                                                      unsigned int* kmax_s) {
  constexpr int kHalf = D / 2, kChunks = kHalf / 8, kU = 4;
  const int per_b = valid * H * kChunks;
  const int lane = gtid & 31;
  for (int b = 0; b < B; ++b) {
    const size_t boff = static_cast<size_t>(b) * S_rows * H * D;
    for (int base = gtid - lane; base < per_b; base += kU * gthreads) {
      uint4 a[kU], bb[kU];
      float4 c0[kU], c1[kU], s0[kU], s1[kU];
      size_t off[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const int i = base + u * gthreads + lane;
        a[u] = make_uint4(0, 0, 0, 0);
        bb[u] = make_uint4(0, 0, 0, 0);
        off[u] = 0;
        if (i < per_b) {
          const int ch = i % kChunks, rh = i / kChunks, srow = rh / H;   // rh = srow * H + h
          off[u] = boff + static_cast<size_t>(rh) * D + ch * 8;
          a[u] = *reinterpret_cast<const uint4*>(x + off[u]);
          bb[u] = *reinterpret_cast<const uint4*>(x + off[u] + kHalf);
          const float* ct = cos_t + static_cast<size_t>(srow) * kHalf + ch * 8;
          const float* st = sin_t + static_cast<size_t>(srow) * kHalf + ch * 8;
          c0[u] = __ldg(reinterpret_cast<const float4*>(ct));
          c1[u] = __ldg(reinterpret_cast<const float4*>(ct + 4));
          s0[u] = __ldg(reinterpret_cast<const float4*>(st));
          s1[u] = __ldg(reinterpret_cast<const float4*>(st + 4));
        }
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        float ss = sumsq16(a[u], bb[u]);
#pragma unroll
        for (int o = 1; o < kChunks; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const int i = base + u * gthreads + lane;
        if (i < per_b) {
          if (i % kChunks == 0) atomicMax(kmax_s + b * H + (i / kChunks) % H, __float_as_uint(ss));
          rotate8(a[u], bb[u], c0[u], c1[u], s0[u], s1[u]);
          *reinterpret_cast<uint4*>(y + off[u]) = a[u];
          *reinterpret_cast<uint4*>(y + off[u] + kHalf) = bb[u];
        }
      }
    }
  }
}

// rotate_tile_smem that also writes each row's squared norm (of the landed bf16 values; the
// rotation preserves it) to qn_rows[row * stride].
// kUnroll row units in flight per thread.
template <int D, int NT, int kUnroll = 1>
__device__ __forceinline__ void rotate_tile_smem_sq(uint32_t tile, const float* __restrict__ cos_t,
                                                    const float* __restrict__ sin_t, int at,
                                                    float* __restrict__ qn_rows, int stride) {
  constexpr int kHalf = D / 2, kUnits = kHalf / 8;
  static_assert(NT % 32 == 0 && (128 * kUnits) % NT == 0, "whole warps, whole rows");
#pragma unroll kUnroll
  for (int i = at; i < 128 * kUnits; i += NT) {
    const int row = i / kUnits, x = i % kUnits;
    const uint32_t offa = sw128_offset(row, x);
    const uint32_t offb = (D == 128) ? 16384u + offa : sw128_offset(row, x + 4);
    const float* ct = cos_t + row * kHalf + x * 8;
    const float* st = sin_t + row * kHalf + x * 8;
    uint4 a = lds128(tile + offa), b = lds128(tile + offb);
    float ss = sumsq16(a, b);
#pragma unroll
    for (int o = 1; o < kUnits; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (x == 0) qn_rows[static_cast<size_t>(row) * stride] = ss;
    rotate8(a, b, __ldg(reinterpret_cast<const float4*>(ct)), __ldg(reinterpret_cast<const float4*>(ct + 4)),
            __ldg(reinterpret_cast<const float4*>(st)), __ldg(reinterpret_cast<const float4*>(st + 4)));
    sts128(tile + offa, a);
    sts128(tile + offb, b);
  }
}

// rotate_tile_smem after a per-row RMSNorm with weights w (eps): kUnroll row units in flight
// per thread.
template <int D, int NT, int kUnroll = 1>
__device__ __forceinline__ void rotate_tile_smem_norm(uint32_t tile, const float* __restrict__ cos_t,
                                                      const float* __restrict__ sin_t,
                                                      const float* __restrict__ w, float eps, int at) {
  constexpr int kHalf = D / 2, kUnits = kHalf / 8;
  static_assert(NT % 32 == 0 && (128 * kUnits) % NT == 0, "whole warps, whole rows");
#pragma unroll kUnroll
  for (int i = at; i < 128 * kUnits; i += NT) {
    const int row = i / kUnits, x = i % kUnits;
    const uint32_t offa = sw128_offset(row, x);
    const uint32_t offb = (D == 128) ? 16384u + offa : sw128_offset(row, x + 4);
    uint4 a = lds128(tile + offa), b = lds128(tile + offb);
    float ss = sumsq16(a, b);
#pragma unroll
    for (int o = 1; o < kUnits; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    float wa[8], wb[8], cs[8], sn[8];
    load8f(w + x * 8, wa);
    load8f(w + kHalf + x * 8, wb);
    load8f(cos_t + row * kHalf + x * 8, cs);
    load8f(sin_t + row * kHalf + x * 8, sn);
    norm_rotate8<true>(a, b, rsqrtf(ss * (1.f / D) + eps), wa, wb, cs, sn);
    sts128(tile + offa, a);
    sts128(tile + offb, b);
  }
}

#include "attn_sp.cuh"

template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_cq,
                    const __grid_constant__ CUtensorMap tm_sq, const __grid_constant__ CUtensorMap tm_ck,
                    const __grid_constant__ CUtensorMap tm_sk, const KParams p) {
  using C = Cfg<D>;
  constexpr int NSK = C::kStagesK, NSV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::kOffQ;
  const uint32_t sK0 = s_base + C::kOffK;
  const uint32_t sV0 = s_base + C::kOffV;
  const uint32_t sT0 = s_base + C::kOffT;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kOffBar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &bars->abort;
  unsigned int* status = &g_dit_status;
  const uint32_t b_q_full = smem_u32(&bars->q_full), b_q_ready = smem_u32(&bars->q_ready);
  const uint32_t b_q_empty = smem_u32(&bars->q_empty);

  if (tid == 0) {
    bars->abort = 0;
    mbar_init(b_q_full, 1);
    mbar_init(b_q_ready, 1);
    mbar_init(b_q_empty, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(smem_u32(&bars->k_full[s]), 1);
      mbar_init(smem_u32(&bars->k_ready[s]), 1);
      mbar_init(smem_u32(&bars->k_empty[s]), 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(smem_u32(&bars->v_full[s]), 1);
      mbar_init(smem_u32(&bars->v_ready[s]), 1);
      mbar_init(smem_u32(&bars->v_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->p_full[t]), 128);
      mbar_init(smem_u32(&bars->o_done[t]), 1);
      mbar_init(smem_u32(&bars->o_free[t]), 128);
      mbar_init(smem_u32(&bars->t_full[t]), 1);
      mbar_init(smem_u32(&bars->t_empty[t]), 1);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
  }
  if (tid == 32) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (kMode == kModeRope) {
      tma_prefetch_desc(&tm_cq);
      tma_prefetch_desc(&tm_sq);
      tma_prefetch_desc(&tm_ck);
      tma_prefetch_desc(&tm_sk);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = bars->tmem_base;
  const int it0 = blockIdx.x, it_step = gridDim.x;

  {
  // Register budgets per warpgroup (40 / 200 / 200 / 72) add up to the launch's 512 x 128;
  // each is set at the top of its role's branch so that the role's code is compiled to it.
  // Warpgroup 0 holds the TMA producers, 1 and 2 the softmax, 3 the MMA issuer and the
  // auxiliary group.
  if (warp < 4) {
    regs_dec<40>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ TMA producer
      int kv_cnt = 0, q_cnt = 0, k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int it = it0; ok && it < p.n_items; it += it_step) {
        const Item w = decode_item<kMode>(p, it);
        if (w.n_live == 0) continue;
        // The Q buffers are free once every S MMA of the previous item has completed.
        if (q_cnt > 0 && !(ok = bounded_wait(b_q_empty, (q_cnt - 1) & 1, abort_flag, status,
                                             kStatusTimeoutLoad)))
          break;
        mbar_arrive_expect_tx(b_q_full, w.n_live * C::kTileBytes);
        for (int t = 0; t < w.n_live; ++t)
#pragma unroll
          for (int c = 0; c < C::kSub; ++c)
            tma_load_4d(sQ + t * C::kTileBytes + c * 16384, &tm_q, b_q_full, c * 64, w.h,
                        w.q0 + 128 * t, w.b);
        ++q_cnt;
        for (int j = 0; j < w.n_kv; ++j) {
          if (j == (w.n_kv > kPrefetchLead ? w.n_kv - kPrefetchLead : 0)) {
            // The next item of this CTA usually starts a head no CTA has read yet, at the same
            // moment as every other CTA: warm L2 with its Q tiles and first K/V tiles now.
            const int nit = it + it_step;
            if (nit < p.n_items) {
              const Item nw = decode_item<kMode>(p, nit);
              for (int t = 0; t < nw.n_live; ++t)
#pragma unroll
                for (int c = 0; c < C::kSub; ++c)
                  tma_prefetch_l2_4d(&tm_q, c * 64, nw.h, nw.q0 + 128 * t, nw.b);
              for (int jj = 0; jj < nw.n_kv && jj < kPrefetchKV; ++jj)
#pragma unroll
                for (int c = 0; c < C::kSub; ++c) {
                  tma_prefetch_l2_4d(&tm_k, c * 64, nw.h, jj * 128, nw.b);
                  tma_prefetch_l2_4d(&tm_v, c * 64, nw.h, jj * 128, nw.b);
                }
            }
          }
          const int g = kv_cnt + j, sk = g % NSK, uk = g / NSK, sv = g % NSV, uv = g / NSV;
          if (uk > 0 && !(ok = bounded_wait(smem_u32(&bars->k_empty[sk]), (uk - 1) & 1, abort_flag,
                                            status, kStatusTimeoutLoad)))
            break;
          const uint32_t kf = smem_u32(&bars->k_full[sk]);
          mbar_arrive_expect_tx(kf, C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kSub; ++c)
            tma_load_4d(sK0 + sk * C::kTileBytes + c * 16384, &tm_k, kf, c * 64, w.h, j * 128, w.b);
          ++k_issued;
          if (uv > 0 && !(ok = bounded_wait(smem_u32(&bars->v_empty[sv]), (uv - 1) & 1, abort_flag,
                                            status, kStatusTimeoutLoad)))
            break;
          const uint32_t vf = smem_u32(&bars->v_full[sv]);
          mbar_arrive_expect_tx(vf, C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kSub; ++c)
            tma_load_4d(sV0 + sv * C::kTileBytes + c * 16384, &tm_v, vf, c * 64, w.h, j * 128, w.b);
          ++v_issued;
        }
        kv_cnt += w.n_kv;
      }
      if (*abort_flag) {
        // Let the copies still in flight land before the CTA gives up its shared memory: the
        // last Q load and the last load of every K and V stage.
        if (q_cnt > 0) drain_wait(b_q_full, (q_cnt - 1) & 1, status);
        for (int g = k_issued - NSK > 0 ? k_issued - NSK : 0; g < k_issued; ++g)
          drain_wait(smem_u32(&bars->k_full[g % NSK]), (g / NSK) & 1, status);
        for (int g = v_issued - NSV > 0 ? v_issued - NSV : 0; g < v_issued; ++g)
          drain_wait(smem_u32(&bars->v_full[g % NSV]), (g / NSV) & 1, status);
      }
    } else if (kMode == kModeRope && warp == 2 && lane == 0) {
      // ------------------------------------------------------------ table producer
      // Streams the cos/sin rows of every tile the auxiliary group rotates (per item: Q0,
      // Q1, then K_0 .. K_n-1), 32 rows at a time, through a 2-buffer ring in shared memory.
      int g = 0;
      bool ok = true;
      for (int it = it0; ok && it < p.n_items; it += it_step) {
        const Item w = decode_item<kMode>(p, it);
        if (w.n_live == 0) continue;
        const int n_rot = w.n_live + w.n_kv;
        for (int r = 0; ok && r < n_rot * 4; ++r, ++g) {
          const int tile_i = r >> 2, qtr = r & 3, buf = g & 1, use = g >> 1;
          const bool is_q = tile_i < w.n_live;
          const int row = (is_q ? w.q0 + 128 * tile_i : (tile_i - w.n_live) * 128) + 32 * qtr;
          if (use > 0 && !(ok = bounded_wait(smem_u32(&bars->t_empty[buf]), (use - 1) & 1,
                                             abort_flag, status, kStatusTimeoutLoad)))
            break;
          const uint32_t tf = smem_u32(&bars->t_full[buf]);
          const uint32_t dst = sT0 + buf * 2 * C::kTabBoxBytes;
          mbar_arrive_expect_tx(tf, 2 * C::kTabBoxBytes);
          tma_load_2d(dst, is_q ? &tm_cq : &tm_ck, tf, 0, row);
          tma_load_2d(dst + C::kTabBoxBytes, is_q ? &tm_sq : &tm_sk, tf, 0, row);
        }
      }
      if (*abort_flag) {
        // The last load of each buffer is the only one that can still be in flight.
        for (int x = g - 2; x < g; ++x)
          if (x >= 0) drain_wait(smem_u32(&bars->t_full[x & 1]), (x >> 1) & 1, status);
      }
    }
  } else if (warp < 12) {
    regs_inc<200>();
    // -------------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;                   // query-tile slot of this warpgroup
    const int r = (tid - 128) & 127;                 // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + t * 128;  // S_t (and P_t in its first 64 columns)
    const uint32_t tO = tbase + lane_off + 256 + t * 128;
    const float sl2 = p.scale_log2;
    int sc = 0, epi = 0;
    bool ok = true;
    for (int it = it0; ok && it < p.n_items; it += it_step) {
      const Item w = decode_item<kMode>(p, it);
      if (t >= w.n_live) {
        if (t == 0 || w.has1) write_empty_tile<D>(p, p.out, p.lse, w.b, w.h, w.q0 + 128 * t, r, 128);
        continue;
      }
      const int n_kv = w.n_kv, kv_valid = w.kv_valid;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < n_kv; ++j) {
        if (!warp_wait(smem_u32(&bars->s_full[t]), (sc + j) & 1, abort_flag, status,
                       kStatusTimeoutSoftmax)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int nv = min(128, kv_valid - j * 128);   // valid keys in this tile (>= 1)
        // The whole S row in registers: four 32-column loads in flight, one wait.
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sr[c]);
        tmem_ld_wait_tied(sr[0]);
        tmem_reg_tie(sr[1]);
        tmem_reg_tie(sr[2]);
        tmem_reg_tie(sr[3]);
        if (nv < 128) {   // keys past the valid length score -inf (whatever S holds there)
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i >= nv) sr[c][i] = 0xff800000u;
        }
        // Row max with four independent three-input chains (one per 32-column chunk).
        float mx4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          mx4[c] = fmaxf(__uint_as_float(sr[c][0]), __uint_as_float(sr[c][1]));
#pragma unroll
          for (int i = 2; i < 32; i += 2)
            mx4[c] = fmax3(mx4[c], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
        }
        const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        const float mt = mx * sl2;
        const bool resc = mt > m_used + kRescaleThreshold;
        const float m_new = resc ? mt : m_used;
        const float alpha = ex2_approx(m_used - m_new);   // 1 if kept; 0 on the first tile
        // S_t,j completing implies P_t,j-1 V_j-1 has completed too (issue order), so O_t is
        // current and nothing else writes it until this group arrives on p_full.
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32(tO + c * 32, orr);
#pragma unroll
            for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
            tmem_st32(tO + c * 32, orr);
          }
        }
        m_used = m_new;
        const float neg_m = -m_used;
        // P = 2^(s * scale * log2 e - m); row sum in four packed partial sums; P (bf16) into
        // the first 64 columns of S_t in TMEM (the row is already in registers).
        float l4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) l4[k] = 0.f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {           // 16 columns at a time
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x0, x1, p0, p1;
            fma2_bc(x0, x1, __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i]),
                    __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i + 1]), sl2, neg_m);
            if ((kFmaExpPairs >> i) & 1u) {
              exp2_fma2(p0, p1, x0, x1);
            } else {
              p0 = ex2_approx(x0);
              p1 = ex2_approx(x1);
            }
            add2(l4[2 * (i & 1)], l4[2 * (i & 1) + 1], p0, p1);
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st8_nowait(tS + c * 8, pk);
        }
        l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(smem_u32(&bars->p_full[t]));
      }
      if (!ok || !warp_wait(smem_u32(&bars->o_done[t]), epi & 1, abort_flag, status,
                            kStatusTimeoutSoftmax)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int qrow = w.q0 + 128 * t + r;
      const bool valid_row = qrow < p.q_valid;
      const float inv_l = 1.f / l;
      uint16_t* dst = p.out + ((static_cast<size_t>(w.b) * p.Sq + qrow) * p.H + w.h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(tO + c * 32, orr);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 o = make_uint4(0, 0, 0, 0);
          if (valid_row) {
            const float* f = reinterpret_cast<const float*>(&orr[8 * q4]);
            o.x = pack_bf16x2(f[0] * inv_l, f[1] * inv_l);
            o.y = pack_bf16x2(f[2] * inv_l, f[3] * inv_l);
            o.z = pack_bf16x2(f[4] * inv_l, f[5] * inv_l);
            o.w = pack_bf16x2(f[6] * inv_l, f[7] * inv_l);
          }
          *reinterpret_cast<uint4*>(dst + c * 32 + q4 * 8) = o;
        }
      }
      // O_t has been read out of TMEM: the next item may overwrite it.
      tc_fence_before_sync();
      mbar_arrive(smem_u32(&bars->o_free[t]));
      p.lse[(static_cast<size_t>(w.b) * p.Sq + qrow) * p.H + w.h] =
          valid_row ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      sc += n_kv;
      ++epi;
    }
  } else {
    regs_dec<72>();
    if (warp == 12) {
     if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      // S = Q K^T: fp16 operands after the fused rotation, the raw bf16 inputs otherwise.
      constexpr uint32_t kIdS = idesc_f16kind_f32(128, 128, kMode == kModePlain,
                                                  false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
      int kv_cnt = 0, q_cnt = 0;
      // Per query-tile slot: S tiles issued so far (p_full phases) and items whose O_t has gone
      // to the epilogue (o_free phases); scalars, so that they stay in registers.
      int sc0 = 0, sc1 = 0, epi0 = 0, epi1 = 0;
      bool ok = true;
      auto wait_k = [&](int g) -> bool {
        const int s = g % NSK;
        const uint32_t kbar = (kMode == kModeRope) ? smem_u32(&bars->k_ready[s]) : smem_u32(&bars->k_full[s]);
        if (!bounded_wait(kbar, (g / NSK) & 1, abort_flag, status, kStatusTimeoutMma)) return false;
        tc_fence_after_sync();
        return true;
      };
      auto wait_v = [&](int g) -> bool {
        const int s = g % NSV;
        const uint32_t vbar = smem_u32(&bars->v_full[s]);
        if (!bounded_wait(vbar, (g / NSV) & 1, abort_flag, status, kStatusTimeoutMma)) return false;
        tc_fence_after_sync();
        return true;
      };
      auto wait_bar = [&](uint32_t bar, int phase) -> bool {
        if (!bounded_wait(bar, phase & 1, abort_flag, status, kStatusTimeoutMma)) return false;
        tc_fence_after_sync();
        return true;
      };
      // Descriptors are built once per tile and advanced by constant offsets (the address
      // field counts 16-byte units), which keeps this thread's register needs small.
      auto issue_s = [&](int t, int g) {
        const uint64_t da = smem_desc_sw128(sQ + t * C::kTileBytes, 16, 1024);
        const uint64_t db = smem_desc_sw128(sK0 + (g % NSK) * C::kTileBytes, 16, 1024);
        const uint32_t d = tbase + t * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
          mma_bf16_ss(d, da + off, db + off, kIdS, kk > 0);
        }
        mma_commit(smem_u32(&bars->s_full[t]));
      };
      // O_t (+)= P_t V_g; the first key tile of an item overwrites O_t, so it waits until the
      // epilogue of the previous item that used this slot has read O_t out of TMEM.
      auto issue_pv = [&](int t, int g, int j) -> bool {
        const int sct = t ? sc1 : sc0, epit = t ? epi1 : epi0;
        if (!wait_bar(smem_u32(&bars->p_full[t]), sct + j)) return false;
        if (j == 0 && epit > 0 && !wait_bar(smem_u32(&bars->o_free[t]), epit - 1)) return false;
        const uint64_t db = smem_desc_sw128(sV0 + (g % NSV) * C::kTileBytes, 16384, 1024);
        const uint32_t a_tmem = tbase + t * 128;          // P_t: bf16 pairs in TMEM
        const uint32_t d = tbase + 256 + t * 128;         // O_t
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(d, a_tmem + kk * 8, db + static_cast<uint64_t>(kk * 2048 >> 4), kIdO,
                      (j > 0 || kk > 0) ? 1u : 0u);
        return true;
      };
      for (int it = it0; ok && it < p.n_items; it += it_step) {
        const Item w = decode_item<kMode>(p, it);
        if (w.n_live == 0) continue;
        if (!(ok = wait_bar(kMode == kModeRope ? b_q_ready : b_q_full, q_cnt))) break;
        if (!(ok = wait_k(kv_cnt))) break;
        issue_s(0, kv_cnt);
        if (w.n_live == 2) issue_s(1, kv_cnt);
        mma_commit(smem_u32(&bars->k_empty[kv_cnt % NSK]));
        for (int j = 1; ok && j < w.n_kv; ++j) {
          const int g = kv_cnt + j;
          if (!(ok = wait_v(g - 1) && issue_pv(0, g - 1, j - 1))) break;
          if (!(ok = wait_k(g))) break;
          issue_s(0, g);
          if (w.n_live == 2) {
            if (!(ok = issue_pv(1, g - 1, j - 1))) break;
            issue_s(1, g);
          }
          mma_commit(smem_u32(&bars->v_empty[(g - 1) % NSV]));
          mma_commit(smem_u32(&bars->k_empty[g % NSK]));
        }
        if (!ok) break;
        const int gl = kv_cnt + w.n_kv - 1;
        if (!(ok = wait_v(gl) && issue_pv(0, gl, w.n_kv - 1))) break;
        mma_commit(smem_u32(&bars->o_done[0]));
        if (w.n_live == 2) {
          if (!(ok = issue_pv(1, gl, w.n_kv - 1))) break;
          mma_commit(smem_u32(&bars->o_done[1]));
        }
        mma_commit(smem_u32(&bars->v_empty[gl % NSV]));
        mma_commit(b_q_empty);
        sc0 += w.n_kv;
        ++epi0;
        if (w.n_live == 2) {
          sc1 += w.n_kv;
          ++epi1;
        }
        kv_cnt += w.n_kv;
        ++q_cnt;
      }
      if (*abort_flag) {
        // Wait for every MMA issued so far before TMEM and shared memory are released.
        mma_commit(smem_u32(&bars->drain));
        drain_wait(smem_u32(&bars->drain), 0, status);
      }
    }
    } else {
    // ------------------------------------------------------------ auxiliary group (96 threads)
    const int at = tid - 416;
    volatile int* go = &bars->aux_go;
    int kv_cnt = 0, q_cnt = 0, g = 0;
    bool ok = true;
    if (kMode == kModeRope) {
      using R = Rotator<D>;
      // Rotates one tile whose four staged table quarters are next in the ring.
      auto rotate_tile = [&](uint32_t sm) -> bool {
        for (int qtr = 0; qtr < 4; ++qtr, ++g) {
          const int buf = g & 1;
          if (!group_wait(smem_u32(&bars->t_full[buf]), (g >> 1) & 1, abort_flag, status,
                          kStatusTimeoutRope, go, at))
            return false;
          const uint32_t tc = sT0 + buf * 2 * C::kTabBoxBytes;
          R::quarter(sm, tc, tc + C::kTabBoxBytes, qtr, at);
          named_bar_sync(1, kAuxThreads);                // every thread is done with the buffer
          if (at == 0) mbar_arrive(smem_u32(&bars->t_empty[buf]));
        }
        return true;
      };
      for (int it = it0; ok && it < p.n_items; it += it_step) {
        const Item w = decode_item<kMode>(p, it);
        if (w.n_live == 0) continue;
        if (!(ok = group_wait(b_q_full, q_cnt & 1, abort_flag, status, kStatusTimeoutRope, go, at)))
          break;
        for (int t = 0; ok && t < w.n_live; ++t) ok = rotate_tile(sQ + t * C::kTileBytes);
        if (!ok) break;
        fence_proxy_async_smem();
        named_bar_sync(1, kAuxThreads);
        if (at == 0) mbar_arrive(b_q_ready);
        for (int j = 0; ok && j < w.n_kv; ++j) {
          const int gk = kv_cnt + j, s = gk % NSK;
          if (!(ok = group_wait(smem_u32(&bars->k_full[s]), (gk / NSK) & 1, abort_flag, status,
                                kStatusTimeoutRope, go, at)))
            break;
          if (!(ok = rotate_tile(sK0 + s * C::kTileBytes))) break;
          fence_proxy_async_smem();
          named_bar_sync(1, kAuxThreads);
          if (at == 0) mbar_arrive(smem_u32(&bars->k_ready[s]));
        }
        kv_cnt += w.n_kv;
        ++q_cnt;
      }
    }
    }
  }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

template <int D, int kMode>
cudaError_t launch_mode(const AttnArgs& a) {
  CUtensorMap mq, mk, mv;
  const int qext = a.q_valid > 0 ? a.q_valid : 1;
  // Workspace mode: the k TMA map reads the rotated fp16 copy (2-byte elements either way);
  // q is loaded raw and rotated in shared memory.
  uint16_t* k_rot = is_ws_mode(kMode) ? static_cast<uint16_t*>(a.workspace) : nullptr;
  const void* q_src = a.q;
  const void* k_src = is_ws_mode(kMode) ? static_cast<const void*>(k_rot) : a.k;
  // Cross-attention reads up to Skv rows and masks per batch on the device; self-attention
  // cuts the key/value extent to the valid length so pad rows are never even loaded.
  const int kvext = a.kv_valid > 0 ? a.kv_valid : 1;
  [[maybe_unused]] Fp8Layout f8{};
  if constexpr (kMode == kModeFp8) {
    // Rotate and quantise q, k, v into the workspace, then read the e4m3 copies: q~ and k~
    // as [B, S, H, D] bytes (one 128-byte row per token and head), v transposed [B, H, D, S].
    f8 = fp8_layout(a.B, a.Sq, a.Skv, a.H, D);
    const cudaError_t e8 = launch_fp8_prepare(a, f8);
    if (e8 != cudaSuccess) return e8;
    char* wsb = static_cast<char*>(a.workspace);
    using u64 = unsigned long long;
    const u64 HD = static_cast<u64>(a.H) * D;
    const u64 dq[4] = {static_cast<u64>(D), static_cast<u64>(a.H), static_cast<u64>(qext), static_cast<u64>(a.B)};
    const u64 sq[3] = {static_cast<u64>(D), HD, HD * a.Sq};
    const u64 dk[4] = {static_cast<u64>(D), static_cast<u64>(a.H), static_cast<u64>(kvext), static_cast<u64>(a.B)};
    const u64 sk[3] = {static_cast<u64>(D), HD, HD * a.Skv};
    const u64 dv[4] = {static_cast<u64>(kvext), static_cast<u64>(D), static_cast<u64>(a.H), static_cast<u64>(a.B)};
    const u64 sv[3] = {static_cast<u64>(a.Skv), static_cast<u64>(D) * a.Skv, HD * a.Skv};
    const unsigned int box_rows[4] = {128, 1, 128, 1}, box_vt[4] = {128, 128, 1, 1};
    if (!encode_u8_map4(&mq, wsb + f8.q8, dq, sq, box_rows) || !encode_u8_map4(&mk, wsb + f8.k8, dk, sk, box_rows) ||
        !encode_u8_map4(&mv, wsb + f8.vt8, dv, sv, box_vt))
      return cudaErrorInvalidValue;
  } else if (!encode_bshd_map(&mq, q_src, a.B, qext, a.Sq, a.H, D) ||
             !encode_bshd_map(&mk, k_src, a.B, kvext, a.Skv, a.H, D) ||
             !encode_bshd_map(&mv, a.v, a.B, kvext, a.Skv, a.H, D)) {
    return cudaErrorInvalidValue;
  }
  // RoPE tables [rows, D/2] fp32, read 32 rows at a time (a copy of the Q map when unused).
  CUtensorMap mcq = mq, msq = mq, mck = mq, msk = mq;
  if (kMode == kModeRope) {
    if (!encode_rows_map_f32(&mcq, a.cos_q, a.Sq, D / 2, Cfg<D>::kTabRows) ||
        !encode_rows_map_f32(&msq, a.sin_q, a.Sq, D / 2, Cfg<D>::kTabRows) ||
        !encode_rows_map_f32(&mck, a.cos_k, a.Skv, D / 2, Cfg<D>::kTabRows) ||
        !encode_rows_map_f32(&msk, a.sin_k, a.Skv, D / 2, Cfg<D>::kTabRows))
      return cudaErrorInvalidValue;
  }
  KParams p;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.H = a.H;
  p.n_pairs = (a.Sq + 255) / 256;
  p.n_items = a.B * a.H * p.n_pairs;
  p.q_valid = a.q_valid;
  p.kv_valid = a.kv_valid;
  p.cos_q = a.cos_q;
  p.sin_q = a.sin_q;
  p.cos_k = a.cos_k;
  p.sin_k = a.sin_k;
  p.scale_log2 = a.scale * kLog2e;
  p.out = static_cast<uint16_t*>(a.out);
  p.lse = a.lse;
  WsParams ws;
  ws.k_raw = static_cast<const uint16_t*>(a.k);
  ws.k_rot = k_rot;
  ws.rotated = nullptr;
  ws.B = a.B;
  ws.norm_q = a.norm_q;
  ws.norm_k = a.norm_k;
  ws.norm_eps = a.norm_eps;
  ws.kmax = nullptr;
  ws.qn = nullptr;
  ws.n_online = a.n_online;
  ws.f8_sq = ws.f8_sk = ws.f8_sv = nullptr;
  ws.f8_nt_q = 0;
  if constexpr (kMode == kModeFp8) {
    const char* wsb = static_cast<const char*>(a.workspace);
    ws.f8_sq = reinterpret_cast<const float*>(wsb + f8.sq);
    ws.f8_sk = reinterpret_cast<const float*>(wsb + f8.sk);
    ws.f8_sv = reinterpret_cast<const float*>(wsb + f8.sv);
    ws.f8_nt_q = f8.nt_q;
  }
  size_t zero_bytes = sizeof(unsigned int);   // what the launch clears: the CTA counter
  if (is_ws_mode(kMode)) {
    const size_t k_bytes = (static_cast<size_t>(a.B) * a.Skv * a.H * D * 2 + 255) / 256 * 256;
    ws.rotated = reinterpret_cast<unsigned int*>(static_cast<char*>(a.workspace) + k_bytes);
    if (kMode == kModeRopeWsFixedM) {
      const size_t kmax_bytes = (static_cast<size_t>(a.B) * a.H * 4 + 255) / 256 * 256;
      ws.kmax = reinterpret_cast<unsigned int*>(static_cast<char*>(a.workspace) + k_bytes + 256);
      ws.qn = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + k_bytes + 256 + kmax_bytes);
      zero_bytes = 256 + kmax_bytes;   // the counter block and the key-norm maxima
    }
  }
  // SM count of the current device, asked on every launch (an attribute query is cheap), so
  // that calls on devices with different SM counts each size their persistent grid right.
  int dev = 0, sm_count = 0;
  cudaError_t qe = cudaGetDevice(&dev);
  if (qe == cudaSuccess) qe = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (qe != cudaSuccess) return qe;
  if (sm_count < 1) return cudaErrorInvalidDevice;
  const int grid = p.n_items < sm_count ? p.n_items : sm_count;   // persistent: one CTA per SM
  if constexpr (kMode == kModeRope) {
    // Per-tile RoPE needs shared memory for its table ring, so it keeps P in TMEM.
    auto kern = attn_fwd_kernel<D, kMode>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, Cfg<D>::kSmemBytes, a.stream>>>(mq, mk, mv, mcq, msq, mck, msk, p);
    return cudaGetLastError();
  } else {
    auto kern = attn_sp_kernel<D, kMode>;
    constexpr int kSmem = CfgSp<D, kMode == kModeFp8>::kSmemBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (!is_ws_mode(kMode)) {
      kern<<<grid, kThreads, kSmem, a.stream>>>(mq, mk, mv, p, ws, NoShards{});
      return cudaGetLastError();
    }
    // CTAs wait for rotated rows that other CTAs produce: launch cooperatively so that every
    // CTA is resident, after zeroing the counter on the same stream.
    e = cudaMemsetAsync(ws.rotated, 0, zero_bytes, a.stream);
    if (e != cudaSuccess) return e;
    NoShards ns{};
    void* args[] = {&mq, &mk, &mv, &p, &ws, &ns};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kThreads),
                                       args, kSmem, a.stream);
  }
}

// Sharded keys in one cooperative launch: every CTA rotates its share of all chunks' k rows
// (the grid counter gates the loads of rotated rows, as in the workspace mode), then the work
// items (chunk, b, h, query-tile pair) run with the chunk's maps and write its partial.
template <int D>
cudaError_t launch_sharded_mode(const AttnArgs& a, const KeyShard* shards, const ShardPlan& plan) {
  constexpr int kMode = kModeRopeWsSharded;
  CUtensorMap mq;
  const int qext = a.q_valid > 0 ? a.q_valid : 1;
  if (!encode_bshd_map(&mq, a.q, a.B, qext, a.Sq, a.H, D)) return cudaErrorInvalidValue;
  char* wsb = static_cast<char*>(a.workspace);
  ShardParams sh;
  std::memset(&sh, 0, sizeof(sh));
  sh.n_chunks = plan.n_chunks;
  sh.po_stride = static_cast<long long>(a.B) * a.Sq * a.H * D;
  sh.pl_stride = static_cast<long long>(a.B) * a.Sq * a.H;
  KParams p;
  std::memset(&p, 0, sizeof(p));
  const size_t row_bytes = static_cast<size_t>(a.H) * D * 2;
  for (int c = 0; c < plan.n_chunks; ++c) {
    const KeyShard& ks = shards[plan.shard[c]];
    const size_t r0 = static_cast<size_t>(plan.row0[c]);
    KeyChunk& kc = sh.c[c];
    kc.k_raw = reinterpret_cast<const uint16_t*>(static_cast<const char*>(ks.k) + r0 * row_bytes);
    kc.k_rot = reinterpret_cast<uint16_t*>(wsb + plan.rot_off[c] + r0 * row_bytes);
    kc.cos_k = ks.cos_k + r0 * (D / 2);
    kc.sin_k = ks.sin_k + r0 * (D / 2);
    kc.S_rows = ks.S_pad;
    kc.valid = plan.valid[c];
    // An empty chunk (every shard empty) is never read: its maps only need to be valid, so
    // they point at the workspace with one row per batch.
    const bool empty = plan.valid[c] == 0;
    const int ext = empty ? 1 : plan.valid[c];
    const int rows = empty ? 1 : ks.S_pad;
    const void* vbase = empty ? static_cast<const void*>(kc.k_rot) : static_cast<const char*>(ks.v) + r0 * row_bytes;
    if (!encode_bshd_map(&sh.km[c], kc.k_rot, a.B, ext, rows, a.H, D) ||
        !encode_bshd_map(&sh.vm[c], vbase, a.B, ext, rows, a.H, D))
      return cudaErrorInvalidValue;
  }
  p.Sq = a.Sq;
  p.Skv = 0;
  p.H = a.H;
  p.n_pairs = (a.Sq + 255) / 256;
  sh.n_bh = a.B * a.H;
  const long long n_items = static_cast<long long>(plan.n_chunks) * a.B * a.H * p.n_pairs;
  if (n_items >= (1ll << 31)) return cudaErrorInvalidValue;
  p.n_items = static_cast<int>(n_items);
  p.q_valid = a.q_valid;
  p.kv_valid = 0;
  p.cos_q = a.cos_q;
  p.sin_q = a.sin_q;
  p.cos_k = p.sin_k = nullptr;
  p.scale_log2 = a.scale * kLog2e;
  p.out = reinterpret_cast<uint16_t*>(wsb + plan.po_off);
  p.lse = reinterpret_cast<float*>(wsb + plan.pl_off);
  WsParams ws;
  std::memset(&ws, 0, sizeof(ws));
  ws.rotated = reinterpret_cast<unsigned int*>(wsb + plan.counter_off);
  ws.B = a.B;
  int dev = 0, sm_count = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (sm_count < 1) return cudaErrorInvalidDevice;
  const int grid = p.n_items < sm_count ? p.n_items : sm_count;
  auto kern = attn_sp_kernel<D, kMode>;
  constexpr int kSmem = CfgSp<D, false>::kSmemBytes;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ws.rotated, 0, sizeof(unsigned int), a.stream);
  if (e != cudaSuccess) return e;
  // the first map arguments are unused in this mode (each chunk has its own)
  void* args[] = {&mq, &mq, &mq, &p, &ws, &sh};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(kThreads), args,
                                     kSmem, a.stream);
}

}  // namespace

bool plan_shards(int B, int Sq, int H, int D, int n_shards, const KeyShard* shards, int sm_count,
                 ShardPlan* plan) {
  std::memset(plan, 0, sizeof(*plan));
  // Rotated k of every shard in the workspace, one after another (each 256-byte aligned).
  size_t off = 0, shard_off[64] = {};
  if (n_shards < 1 || n_shards > 64) return false;
  for (int s = 0; s < n_shards; ++s) {
    shard_off[s] = off;
    off += (static_cast<size_t>(B) * shards[s].S_pad * H * D * 2 + 255) / 256 * 256;
  }
  // Key tiles per shard, and a chunk length (in tiles) that gives at least about six work
  // items per SM: items per chunk = B * H * query-tile pairs.
  const long long items_per_chunk = static_cast<long long>(B) * H * ((Sq + 255) / 256);
  (void)sm_count;   // the plan uses a fixed target so that workspace sizes do not depend on the device
  long long total_tiles = 0;
  int nonempty = 0;
  for (int s = 0; s < n_shards; ++s)
    if (shards[s].valid > 0) {
      total_tiles += (shards[s].valid + 127) / 128;
      ++nonempty;
    }
  if (nonempty > kMaxKeyChunks) return false;
  long long want = (kShardTargetItems + items_per_chunk - 1) / items_per_chunk;   // chunks wanted
  if (want < nonempty) want = nonempty;
  if (want > kMaxKeyChunks) want = kMaxKeyChunks;
  long long chunk_tiles = total_tiles > 0 ? (total_tiles + want - 1) / want : 1;
  if (chunk_tiles < 1) chunk_tiles = 1;
  for (;; ++chunk_tiles) {   // grow the chunks until they fit in kMaxKeyChunks
    int n = 0;
    for (int s = 0; s < n_shards; ++s)
      if (shards[s].valid > 0) n += static_cast<int>(((shards[s].valid + 127) / 128 + chunk_tiles - 1) / chunk_tiles);
    if (n <= kMaxKeyChunks) break;
  }
  int n = 0;
  for (int s = 0; s < n_shards; ++s) {
    if (shards[s].valid <= 0) continue;
    const int tiles = (shards[s].valid + 127) / 128;
    const int parts = static_cast<int>((tiles + chunk_tiles - 1) / chunk_tiles);
    int t0 = 0;
    for (int k = 0; k < parts; ++k) {
      const int nt = tiles / parts + (k < tiles % parts ? 1 : 0);   // near-equal parts
      plan->shard[n] = s;
      plan->row0[n] = t0 * 128;
      const int end = (t0 + nt) * 128 < shards[s].valid ? (t0 + nt) * 128 : shards[s].valid;
      plan->valid[n] = end - t0 * 128;
      plan->rot_off[n] = shard_off[s];
      t0 += nt;
      ++n;
    }
  }
  if (n == 0) {   // no key at all: one empty chunk, whose items write O = 0, LSE = -inf
    plan->shard[0] = 0;
    plan->valid[0] = 0;
    plan->rot_off[0] = shard_off[0];
    n = 1;
  }
  plan->n_chunks = n;
  plan->counter_off = off;
  plan->po_off = off + 256;
  const size_t po = (static_cast<size_t>(n) * B * Sq * H * D * 2 + 255) / 256 * 256;
  plan->pl_off = plan->po_off + po;
  plan->total = plan->pl_off + (static_cast<size_t>(n) * B * Sq * H * 4 + 255) / 256 * 256;
  return true;
}

cudaError_t launch_attn_sharded(const AttnArgs& a, int n_shards, const KeyShard* shards, const ShardPlan& plan) {
  (void)n_shards;
  cudaError_t e = a.D == 128 ? launch_sharded_mode<128>(a, shards, plan) : launch_sharded_mode<64>(a, shards, plan);
  if (e != cudaSuccess) return e;
  char* wsb = static_cast<char*>(a.workspace);
  return launch_lse_merge(wsb + plan.po_off, reinterpret_cast<const float*>(wsb + plan.pl_off), plan.n_chunks, a.B,
                          a.Sq, a.H, a.D, a.out, a.lse, a.stream);
}

size_t attn_workspace_bytes(int B, int Sq, int Skv, int H, int D) {
  (void)Sq;   // q is rotated in shared memory, tile by tile
  const size_t k = (static_cast<size_t>(B) * Skv * H * D * 2 + 255) / 256 * 256;
  return k + 256;   // + the counter of CTAs done rotating
}

size_t attn_fixed_m_workspace_bytes(int B, int Sq, int Skv, int H, int D) {
  const size_t kmax = (static_cast<size_t>(B) * H * 4 + 255) / 256 * 256;
  const size_t qn = (static_cast<size_t>(B) * Sq * H * 4 + 255) / 256 * 256;
  return attn_workspace_bytes(B, Sq, Skv, H, D) + kmax + qn;
}

cudaError_t launch_attn_fwd(const AttnArgs& a, AttnMode mode) {
  if (a.D == 128) {
    if (mode == kModeRopeWs) return launch_mode<128, kModeRopeWs>(a);
    if (mode == kModeRopeWsNorm) return launch_mode<128, kModeRopeWsNorm>(a);
    if (mode == kModeRopeWsFixedM) return launch_mode<128, kModeRopeWsFixedM>(a);
    if (mode == kModeFp8) return launch_mode<128, kModeFp8>(a);
    if (mode == kModeRope) return launch_mode<128, kModeRope>(a);
    return launch_mode<128, kModePlain>(a);
  }
  if (mode == kModeRopeWs) return launch_mode<64, kModeRopeWs>(a);
  if (mode == kModeRopeWsNorm) return launch_mode<64, kModeRopeWsNorm>(a);
  if (mode == kModeRopeWsFixedM) return launch_mode<64, kModeRopeWsFixedM>(a);
  if (mode == kModeFp8) return cudaErrorInvalidValue;   // built for D = 128 only
  if (mode == kModeRope) return launch_mode<64, kModeRope>(a);
  return launch_mode<64, kModePlain>(a);
}

cudaError_t device_status_ptr(unsigned int** out) {
  // Device address of this device's status word, looked up once per device (kernels in other
  // translation units receive it as a parameter).
  static std::mutex mu;
  static unsigned int* ptrs[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dit_status);
    if (e != cudaSuccess) return e;
    ptrs[dev] = static_cast<unsigned int*>(p);
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

cudaError_t read_device_status(unsigned int* out, bool clear) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(out, g_dit_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_dit_status, &zero, sizeof(unsigned int));
  }
  return e;
}

}  // namespace dit

#ifdef DIT_TEST_HOOKS
#include "../../include/dit_attn_test_hooks.h"

extern "C" int dit_test_set_wait_hooks(unsigned long long wait_limit_ns, int skip_load) {
  if (wait_limit_ns == 0) return -1;
  cudaError_t e = cudaMemcpyToSymbol(dit::g_dit_test_wait_limit_ns, &wait_limit_ns, sizeof(wait_limit_ns));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(dit::g_dit_test_skip_load, &skip_load, sizeof(skip_load));
  if (e == cudaSuccess) e = dit::cross_attn_set_test_hooks(wait_limit_ns, skip_load);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? 0 : -4;
}
#endif
