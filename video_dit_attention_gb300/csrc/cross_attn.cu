// Short-KV cross-attention of video queries against a text sequence, with the text keys and
// values of one (batch, head) resident in shared memory (maxdiffusion PR #491: the fused
// short-KV cross-attention kernel of the Wan fast-inference work; the pages give no design).
//
// What it computes (the plain definition of masked softmax attention, exactly as the
// self-attention kernels, without RoPE): for batch b, head h and query row i < q_valid,
//   s_j = scale * q_i . k_j   for j < L_b = kv_valid_dev[b]
//   lse_i = ln sum_j exp(s_j),  O_i = sum_j exp(s_j - lse_i) v_j,
// with O = 0, lse = -inf for pad query rows and for every row of a batch with L_b = 0. A
// batch whose L_b lies outside [0, Skv] is treated as having no keys, and the kernel sets
// kStatusBadKvLength in the device status word (fail closed, no clamping).
//
// Design (one GPU, sm_103a). The text is short (at most 512 keys), so the work per query
// tile is small (one or two 128-key tiles at the drawn lengths) and the query/output stream
// dominates: 97 MB of Q in and 97 MB of O out at B2 H40, against 21 MB of K and V.
//   - Work is a flat list of 128-row query tiles over (b, h, tile). CTA c of a persistent grid
//     takes the contiguous range [c T / G, (c + 1) T / G), so every CTA has the same number of
//     tiles and walks one or two heads.
//   - The keys and values of the current (b, h) are loaded once into shared memory (a "fill")
//     and stay there for all of the CTA's query tiles of that head: K as one 256-row operand
//     (two 128-row tiles, so S = Q K^T is one N = 256 product per K step), V as two 128-row
//     tiles. When L_b > 256 a query tile visits its keys in two halves of up to 256 with the
//     online softmax, and the fill is reloaded per half (consecutive tiles alternate the order
//     of the halves, so each tile reloads only one).
//   - TMEM: S (256 columns, 128 lanes = query rows), P (bf16, 128 columns) and O (D columns).
//     P has columns of its own, so the S columns are free as soon as the softmax has loaded
//     them: S of tile t + 1 is computed while the softmax of tile t runs, and P_t V while
//     the softmax of tile t + 1 starts. O is read out to registers before P of the next tile
//     is released, then staged in shared memory and written with one TMA store per tile
//     while the next P.V runs. (Writing each thread's row straight to global memory, 32
//     scattered 16-byte pieces per warp store, took about 4,300 cycles per tile and slowed
//     the MMA issue and the Q loads beside it.)
//   - One thread issues every MMA, in the order S_0, S_1, P_0 V, S_2, P_1 V, ... (S of the next
//     step goes first unless that step needs a new fill, which must wait for the release of
//     the current one).
//   - Two softmax warpgroups share each tile: warpgroup A owns key columns 0-127 of the S
//     block, warpgroup B columns 128-255, one thread per query row. The row maximum and the
//     row sum are exchanged between the two threads of a row through shared memory (a named
//     barrier per pair of warps that share a TMEM lane quarter). Warpgroup A normalises and
//     stages O columns [0, D/2), warpgroup B [D/2, D); warpgroup A writes the LSE.
//   - Warp 3 zeroes the V rows past L_b of the fill's last V tile, so that 0 * (pad contents)
//     cannot reach O. K pad rows need nothing: their score columns are masked to -inf.
//   - Q is double-buffered; the producer also warms L2 with the next two query tiles.
// Every wait is bounded (ptx.cuh); on a timeout the CTA records a status bit, drains its
// copies and MMAs, frees TMEM and exits.

#include <cuda_bf16.h>

#include "common.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kXThreads = 384;   // warps 0-3: load / TMEM / MMA / V zeroing; 4-11: softmax
constexpr float kXLn2 = 0.69314718055994530942f;
constexpr float kXLog2e = 1.44269504088896340736f;
constexpr float kXRescale = 8.0f;   // log2 units: O is rescaled only if the maximum grows by > 2^8
constexpr int kLenCache = 128;      // per-batch key lengths kept in shared memory
constexpr uint32_t kXColP = 256;    // TMEM columns: S [0, 256), P [256, 384), O [384, 384 + D)
constexpr uint32_t kXColO = 384;

template <int D>
struct XCfg {
  static constexpr int kSub = D / 64;              // 64-column (128-byte) chunks per row
  static constexpr int kTile = 128 * D * 2;        // one 128-row bf16 tile
  static constexpr int kChunk = 128 * 128;         // one 128-row chunk (16 KB)
  static constexpr int kOffQ = 0;                  // two Q buffers
  static constexpr int kOffK = kOffQ + 2 * kTile;  // K: chunk c holds rows 0..255 at c * 2 kChunk
  static constexpr int kOffV = kOffK + 2 * kTile;  // V: two 128-row tiles
  static constexpr int kOffO = kOffV + 2 * kTile;  // O staging tile (TMA store source)
  static constexpr int kOffX = kOffO + kTile;      // row maximum / sum exchange [2][128] fp32
  static constexpr int kOffLen = kOffX + 2 * 128 * 4;   // key lengths of the first kLenCache batches
  static constexpr int kOffBar = kOffLen + kLenCache * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;   // barriers + alignment slack
};
static_assert(XCfg<128>::kSmem <= 232448, "shared memory of the D = 128 cross kernel");

struct XBars {
  uint64_t q_full[2], q_empty[2];
  uint64_t kv_full, kv_ready, kv_empty;
  uint64_t s_full, s_free, p_full, pv_done;
  uint64_t o_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct XParams {
  int B, Sq, Skv, H, q_valid;
  int n_qt;          // 128-row query tiles per (b, h)
  int n_tiles;       // B * H * n_qt
  const int32_t* kv_len;
  float scale_log2;
  float* lse;
  uint16_t* out;     // for the direct writes of empty tiles
  unsigned int* status;
};

// One query tile of the CTA's range and where it sits in its (b, h) run.
struct XTile {
  int b, h, qt;
  int L;        // valid keys (0 for a bad or empty length)
  int n_kv;     // 128-key tiles holding them
  bool live;    // has a valid query row and at least one key
  bool bad;     // the batch's length was outside [0, Skv]
  int i;        // index of this tile among the live tiles of its (b, h) run in this CTA
  bool last;    // last live tile of that run
};

// Every role decodes every tile of its range; the key lengths of the first kLenCache batches
// are read from shared memory (a global load per tile sat on the MMA issuer's critical path).
__device__ __forceinline__ XTile x_decode(const XParams& p, const int* len_s, int g, int g0, int g1) {
  XTile t;
  const int bh = g / p.n_qt;
  t.qt = g - bh * p.n_qt;
  t.b = bh / p.H;
  t.h = bh - t.b * p.H;
  const int raw = t.b < kLenCache ? len_s[t.b] : p.kv_len[t.b];
  t.bad = raw < 0 || raw > p.Skv;
  t.L = t.bad ? 0 : raw;
  t.n_kv = (t.L + 127) >> 7;
  const int n_live_qt = (p.q_valid + 127) >> 7;   // live tiles are a prefix of each head
  t.live = t.L > 0 && t.qt < n_live_qt;
  const int qt_first = (g0 / p.n_qt == bh) ? g0 - bh * p.n_qt : 0;
  const int qt_end = (min(g1, (bh + 1) * p.n_qt) - bh * p.n_qt);   // one past the run's last tile
  t.i = t.qt - qt_first;
  t.last = t.qt == min(qt_end, n_live_qt) - 1;
  return t;
}

// The key steps of a live tile: one step of up to 256 keys when L <= 256; else two halves
// (key tiles {0, 1} and {2, n_kv - 1}), in the order (0, 1) for even i and (1, 0) for odd i,
// so that a tile's first half is the previous tile's last one.
struct XStep {
  int kt0, nkt;     // first key tile and number of key tiles (1 or 2)
  bool new_fill;    // this step loads a new fill (the previous one is released first)
  bool release;     // the fill is released after this step's products
};

__device__ __forceinline__ int x_n_steps(const XTile& t) { return t.n_kv > 2 ? 2 : 1; }

__device__ __forceinline__ XStep x_step(const XTile& t, int s) {
  XStep st;
  if (t.n_kv <= 2) {
    st.kt0 = 0;
    st.nkt = t.n_kv;
    st.new_fill = t.i == 0;
    st.release = t.last;
    return st;
  }
  const int half = ((t.i & 1) == 0) ? s : 1 - s;
  st.kt0 = half ? 2 : 0;
  st.nkt = half ? t.n_kv - 2 : 2;
  st.new_fill = s == 1 || t.i == 0;
  st.release = s == 0 || t.last;
  return st;
}

// O = 0 and LSE = -inf for one tile's rows (columns [c0, c0 + D/2) of O by this warpgroup;
// the LSE by warpgroup A), written directly.
template <int D>
__device__ __forceinline__ void x_write_empty(const XParams& p, const XTile& t, int wg, int r) {
  const int row = t.qt * 128 + r;
  uint16_t* dst = p.out + ((static_cast<size_t>(t.b) * p.Sq + row) * p.H + t.h) * D + wg * (D / 2);
#pragma unroll
  for (int u = 0; u < D / 16; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
  if (wg == 0) p.lse[(static_cast<size_t>(t.b) * p.Sq + row) * p.H + t.h] = -INFINITY;
}

// Position in a CTA's sequence of key steps (live tiles only, each with one or two steps).
struct XPos {
  int g;        // tile index in the flat list (the CTA's range is [g0, g1))
  int s;        // step within the tile
  XTile t;
  XStep st;
  int ns;       // steps of the tile
  int tcnt;     // live tiles before this one (O buffer tcnt & 1)
  int fill;     // index of the fill this step reads
  int step;     // steps before this one
};

// Advances `pos` to the next key step of the CTA's live tiles; false at the end. Start with
// pos.g = g0 - 1, pos.s = pos.ns = 0, pos.tcnt = pos.fill = pos.step = -1 (first call moves
// to the first step, with tcnt = step = 0 and fill = 0).
__device__ __forceinline__ bool x_next(const XParams& p, const int* len_s, int g0, int g1, XPos& pos) {
  if (pos.g >= g0 && pos.s + 1 < pos.ns) {
    ++pos.s;
  } else {
    int g = pos.g + 1;
    XTile t{};
    for (; g < g1; ++g) {
      t = x_decode(p, len_s, g, g0, g1);
      if (t.live) break;
    }
    if (g >= g1) return false;
    pos.g = g;
    pos.t = t;
    pos.s = 0;
    pos.ns = x_n_steps(t);
    ++pos.tcnt;
  }
  pos.st = x_step(pos.t, pos.s);
  if (pos.st.new_fill) ++pos.fill;
  ++pos.step;
  return true;
}

template <int D>
__global__ void __launch_bounds__(kXThreads, 1)
    cross_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const XParams p) {
  using C = XCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::kOffQ, sK = s_base + C::kOffK, sV = s_base + C::kOffV;
  const uint32_t sO = s_base + C::kOffO;
  float* xch = reinterpret_cast<float*>(smem + C::kOffX);   // [wg][row]
  XBars* bars = reinterpret_cast<XBars*>(smem + C::kOffBar);
  int* len_s = reinterpret_cast<int*>(smem + C::kOffLen);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &bars->abort;
  unsigned int* status = p.status;

  const int G = gridDim.x;
  const int g0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.n_tiles / G);
  const int g1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.n_tiles / G);

  if (tid < kLenCache && tid < p.B) len_s[tid] = p.kv_len[tid];
  if (tid == 0) {
    bars->abort = 0;
    mbar_init(smem_u32(&bars->q_full[0]), 1);
    mbar_init(smem_u32(&bars->q_full[1]), 1);
    mbar_init(smem_u32(&bars->q_empty[0]), 1);
    mbar_init(smem_u32(&bars->q_empty[1]), 1);
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->kv_ready), 1);
    mbar_init(smem_u32(&bars->kv_empty), 1);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), 8);
    mbar_init(smem_u32(&bars->p_full), 8);
    mbar_init(smem_u32(&bars->pv_done), 1);
    mbar_init(smem_u32(&bars->o_free), 8);
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
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = bars->tmem_base;
  const uint32_t b_kv_full = smem_u32(&bars->kv_full), b_kv_ready = smem_u32(&bars->kv_ready);
  const uint32_t b_kv_empty = smem_u32(&bars->kv_empty);
  const uint32_t b_s_full = smem_u32(&bars->s_full), b_s_free = smem_u32(&bars->s_free);
  const uint32_t b_p_full = smem_u32(&bars->p_full), b_pv_done = smem_u32(&bars->pv_done);
  auto start_pos = [&]() {
    XPos pos;
    pos.g = g0 - 1;
    pos.s = pos.ns = 0;
    pos.tcnt = pos.fill = pos.step = -1;
    return pos;
  };

  if (warp < 4) {
    regs_dec<64>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------------ producer
      int q_cnt = 0, fill = 0;
      bool ok = true;
      for (int g = g0; ok && g < g1; ++g) {
        const XTile t = x_decode(p, len_s, g, g0, g1);
        if (!t.live) continue;
        // Q buffer q_cnt & 1: free once every S product of the tile before last has completed
        const int buf = q_cnt & 1;
        if (q_cnt >= 2 && !(ok = bounded_wait(smem_u32(&bars->q_empty[buf]), ((q_cnt - 2) >> 1) & 1, abort_flag,
                                              status, kStatusTimeoutLoad)))
          break;
        const uint32_t qb = smem_u32(&bars->q_full[buf]);
        mbar_arrive_expect_tx(qb, C::kTile);
#pragma unroll
        for (int c = 0; c < C::kSub; ++c)
          tma_load_4d(sQ + buf * C::kTile + c * C::kChunk, &tm_q, qb, c * 64, t.h, t.qt * 128, t.b);
        ++q_cnt;
        // Warm L2 with the next two query tiles, so that each refill of the buffer is an L2 hit.
        for (int ga = g + 1; ga <= g + 2 && ga < g1; ++ga) {
          const XTile ta = x_decode(p, len_s, ga, g0, g1);
          if (ta.live)
#pragma unroll
            for (int c = 0; c < C::kSub; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, ta.h, ta.qt * 128, ta.b);
        }
        for (int s = 0; ok && s < x_n_steps(t); ++s) {
          const XStep st = x_step(t, s);
          if (!st.new_fill) continue;
          if (fill > 0 && !(ok = bounded_wait(b_kv_empty, (fill - 1) & 1, abort_flag, status, kStatusTimeoutLoad)))
            break;
          mbar_arrive_expect_tx(b_kv_full, 2 * st.nkt * C::kTile);
          for (int j = 0; j < st.nkt; ++j) {
            const int key0 = (st.kt0 + j) * 128;
#pragma unroll
            for (int c = 0; c < C::kSub; ++c) {
              tma_load_4d(sK + c * 2 * C::kChunk + j * C::kChunk, &tm_k, b_kv_full, c * 64, t.h, key0, t.b);
              tma_load_4d(sV + j * C::kTile + c * C::kChunk, &tm_v, b_kv_full, c * 64, t.h, key0, t.b);
            }
          }
          ++fill;
        }
      }
      // Let the copies in flight land before the CTA releases its shared memory (on the
      // normal path each has been waited for already, and these return at once).
      for (int n = q_cnt - 2 > 0 ? q_cnt - 2 : 0; n < q_cnt; ++n)
        drain_wait(smem_u32(&bars->q_full[n & 1]), (n >> 1) & 1, status);
      if (fill > 0) drain_wait(b_kv_full, (fill - 1) & 1, status);
    } else if (warp == 2 && lane == 0) {
      // ------------------------------------------------------------------ MMA issuer
      constexpr uint32_t kIdS1 = idesc_f16kind_f32(128, 128, true, false, false);
      constexpr uint32_t kIdS2 = idesc_f16kind_f32(128, 256, true, false, false);
      constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
      bool ok = true;
      auto wait = [&](uint32_t bar, int phase) -> bool {
        if (!bounded_wait(bar, phase & 1, abort_flag, status, kStatusTimeoutMma)) return false;
        tc_fence_after_sync();
        return true;
      };
      // S = Q K^T of one step into the S columns.
      auto issue_s = [&](const XPos& x) -> bool {
        const int buf = x.tcnt & 1;
        if (x.s == 0 && !wait(smem_u32(&bars->q_full[buf]), x.tcnt >> 1)) return false;   // Q of the tile
        if (!wait(b_kv_full, x.fill)) return false;                                       // its keys
        if (x.step > 0 && !wait(b_s_free, x.step - 1)) return false;                       // previous S taken out
        const uint64_t da = smem_desc_sw128(sQ + buf * C::kTile, 16, 1024);
        const uint64_t db = smem_desc_sw128(sK, 16, 1024);
        const uint32_t idS = x.st.nkt == 2 ? kIdS2 : kIdS1;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t offa = ((kk / 4) * C::kChunk + (kk % 4) * 32) >> 4;
          const uint64_t offb = ((kk / 4) * 2 * C::kChunk + (kk % 4) * 32) >> 4;
          mma_bf16_ss(tbase, da + offa, db + offb, idS, kk > 0);
        }
        mma_commit(b_s_full);
        if (x.s == x.ns - 1) mma_commit(smem_u32(&bars->q_empty[buf]));   // the tile's last S: Q may be reloaded
        return true;
      };
      // O (+)= P V of one step, P from TMEM (bf16 pairs; keys 128 j .. of the step at columns
      // 256 + 64 j ..).
      auto issue_pv = [&](const XPos& x) -> bool {
        if (!wait(b_p_full, x.step)) return false;
        // the first step of a tile overwrites O: the previous tile's O has been read out
        if (x.s == 0 && x.tcnt >= 1 && !wait(smem_u32(&bars->o_free), x.tcnt - 1)) return false;
        if (!wait(b_kv_ready, x.fill)) return false;
        const uint32_t d_o = tbase + kXColO;
        for (int j = 0; j < x.st.nkt; ++j) {
          const uint64_t dv = smem_desc_sw128(sV + j * C::kTile, C::kChunk, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(d_o, tbase + kXColP + j * 64 + kk * 8, dv + static_cast<uint64_t>(kk * 2048 >> 4), kIdO,
                        (x.s > 0 || j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(b_pv_done);
        if (x.st.release) mma_commit(b_kv_empty);
        return true;
      };
      XPos cur = start_pos();
      if (x_next(p, len_s, g0, g1, cur)) {
        ok = issue_s(cur);
        while (ok) {
          XPos nxt = cur;
          const bool more = x_next(p, len_s, g0, g1, nxt);
          // S of the next step first when it reads keys already in shared memory
          const bool early = more && !nxt.st.new_fill;
          if (early && !(ok = issue_s(nxt))) break;
          if (!(ok = issue_pv(cur))) break;
          if (!more) break;
          if (!early && !(ok = issue_s(nxt))) break;
          cur = nxt;
        }
      }
      // Every MMA of this thread completes before TMEM and shared memory are released.
      mma_commit(smem_u32(&bars->drain));
      drain_wait(smem_u32(&bars->drain), 0, status);
    } else if (warp == 3) {
      // ------------------------------------------------------------------ V pad rows
      int fill = 0;
      bool ok = true;
      for (int g = g0; ok && g < g1; ++g) {
        const XTile t = x_decode(p, len_s, g, g0, g1);
        if (!t.live) continue;
        for (int s = 0; ok && s < x_n_steps(t); ++s) {
          const XStep st = x_step(t, s);
          if (!st.new_fill) continue;
          int got = 0;
          if (lane == 0) got = bounded_wait(b_kv_full, fill & 1, abort_flag, status, kStatusTimeoutRope) ? 1 : 0;
          if (!(ok = __shfl_sync(0xffffffffu, got, 0) != 0)) break;
          const int jl = st.nkt - 1;                            // the fill's last V tile
          const int nv = min(128, t.L - (st.kt0 + jl) * 128);   // its valid rows (>= 1)
          if (nv < 128) {
            const uint32_t tile = sV + jl * C::kTile;
            const int n16 = (128 - nv) * 8;                     // 16-byte units per chunk
            for (int c = 0; c < C::kSub; ++c)
              for (int u = lane; u < n16; u += 32)
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(tile + c * C::kChunk + nv * 128 + u * 16),
                             "r"(0u)
                             : "memory");
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_kv_ready);
          ++fill;
        }
      }
    }
  } else {
    regs_inc<216>();
    // -------------------------------------------------------------------- softmax + epilogue
    // The 256 threads of both warpgroups meet at named barriers (the row exchanges of a pair
    // of warps, the end of each tile). So that a timeout can never leave a thread waiting at
    // one of them, a thread whose bounded wait fails still runs every barrier of the current
    // tile (skipping the tensor-memory work), and all 256 decide together, at the barrier that
    // ends each tile, whether to go on.
    const int wg = (warp - 4) >> 2;           // 0: key columns 0-127 of the S block, 1: 128-255
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;         // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tbase + lane_off + wg * 128;
    const int pair_bar = 2 + quarter;          // named barrier of warps (4 + q, 8 + q)
    float* x_mine = xch + wg * 128 + r;
    const float* x_other = xch + (1 - wg) * 128 + r;
    const float sl2 = p.scale_log2;
    const uint32_t tP = tbase + lane_off + kXColP + wg * 64;   // this warpgroup's P columns
    const uint32_t tO = tbase + lane_off + kXColO + wg * (D / 2);   // its O columns
    const uint32_t p_sw = static_cast<uint32_t>(r & 7);
    // Bounded wait by lane 0, outcome broadcast to the warp.
    auto wwait = [&](uint32_t bar, int phase) -> bool {
      int got = 0;
      if (lane == 0) got = bounded_wait(bar, phase & 1, abort_flag, status, kStatusTimeoutSoftmax) ? 1 : 0;
      return __shfl_sync(0xffffffffu, got, 0) != 0;
    };
    // The previous tile's output, read out of TMEM before P of the next tile is released.
    bool pend = false;
    int pend_b = 0, pend_h = 0, pend_qt = 0;
    float pend_m = 0.f, pend_l = 1.f;
    auto read_o = [&](uint32_t (&orr)[D / 2]) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t part[32];
        tmem_ld32(tO + c * 32, part);
#pragma unroll
        for (int i = 0; i < 32; ++i) orr[c * 32 + i] = part[i];
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->o_free));   // O may be overwritten
    };
    // Normalise the read-out O, stage it in the 128-byte swizzle of the tile's TMA map and
    // store the tile (one thread), and the LSE. All 256 threads call this.
    auto store_o = [&](const uint32_t (&orr)[D / 2], bool ok_now) {
      const int qrow = pend_qt * 128 + r;
      const bool valid_row = qrow < p.q_valid;
      const float inv_l = 1.f / pend_l;
      if (tid == 128) bulk_wait_read();   // the previous store has read the staging tile
      named_bar_sync(1, 256);
#pragma unroll
      for (int u = 0; u < D / 16; ++u) {
        uint4 o = make_uint4(0, 0, 0, 0);
        if (valid_row) {
          const uint32_t* f = &orr[8 * u];
          o.x = pack_bf16x2(__uint_as_float(f[0]) * inv_l, __uint_as_float(f[1]) * inv_l);
          o.y = pack_bf16x2(__uint_as_float(f[2]) * inv_l, __uint_as_float(f[3]) * inv_l);
          o.z = pack_bf16x2(__uint_as_float(f[4]) * inv_l, __uint_as_float(f[5]) * inv_l);
          o.w = pack_bf16x2(__uint_as_float(f[6]) * inv_l, __uint_as_float(f[7]) * inv_l);
        }
        const int cu = wg * (D / 16) + u;   // 16-byte unit of the full row
        const uint32_t addr = sO + static_cast<uint32_t>(cu >> 3) * C::kChunk + static_cast<uint32_t>(r) * 128u +
                              ((static_cast<uint32_t>(cu & 7) ^ p_sw) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      named_bar_sync(1, 256);
      if (tid == 128 && ok_now) {
#pragma unroll
        for (int c = 0; c < C::kSub; ++c) tma_store_4d(&tm_o, sO + c * C::kChunk, c * 64, pend_h, pend_qt * 128, pend_b);
        bulk_commit_group();
      }
      if (wg == 0 && ok_now)
        p.lse[(static_cast<size_t>(pend_b) * p.Sq + qrow) * p.H + pend_h] =
            valid_row ? (pend_m + log2f(pend_l)) * kXLn2 : -INFINITY;
      pend = false;
    };
    int step = 0;
    bool ok = true;
    for (int g = g0; g < g1; ++g) {
      const XTile t = x_decode(p, len_s, g, g0, g1);
      if (!t.live) {
        x_write_empty<D>(p, t, wg, r);
        if (t.bad && wg == 0 && r == 0) atomicOr(status, kStatusBadKvLength);
        continue;
      }
      float m_run = -INFINITY, l_mine = 0.f;
      const int ns = x_n_steps(t);
      for (int s = 0; s < ns; ++s, ++step) {
        const XStep st = x_step(t, s);
        const bool mine = wg < st.nkt;
        const int nv = mine ? min(128, t.L - (st.kt0 + wg) * 128) : 0;   // my valid keys
        ok = ok && wwait(b_s_full, step);
        if (ok) tc_fence_after_sync();
        uint32_t sr[4][32];
        float mx = -INFINITY;
        if (ok && mine) {
#pragma unroll
          for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sr[c]);
          tmem_ld_wait_tied(sr[0]);
          tmem_reg_tie(sr[1]);
          tmem_reg_tie(sr[2]);
          tmem_reg_tie(sr[3]);
        } else {
          // No key tile of mine in this step (or the wait failed): defined values, all masked.
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) sr[c][i] = 0xff800000u;
        }
        if (ok) {
          // S is in registers: the next S product may overwrite the columns.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(b_s_free);
        }
        if (ok && mine) {
          if (nv < 128) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (c * 32 + i >= nv) sr[c][i] = 0xff800000u;
          }
          float mx4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            mx4[c] = fmaxf(__uint_as_float(sr[c][0]), __uint_as_float(sr[c][1]));
#pragma unroll
            for (int i = 2; i < 32; i += 2)
              mx4[c] = fmax3(mx4[c], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
          }
          mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        }
        // Row maximum over both column blocks: exchange with the partner thread of this row
        // (the first barrier: the partner has read the previous exchange).
        named_bar_sync(pair_bar, 64);
        *x_mine = mx;
        named_bar_sync(pair_bar, 64);
        const float mt = fmaxf(mx, *x_other) * sl2;
        const bool resc = mt > m_run + kXRescale;
        const float m_new = resc ? mt : m_run;
        const float alpha = ex2_approx(m_run - m_new);   // 1 if kept; 0 on the first step
        // The previous step's P V must be complete before P is rewritten and before O is read
        // out or rescaled; both warpgroups take the same decision (same maxima).
        if (step > 0) {
          ok = ok && wwait(b_pv_done, step - 1);
          if (ok) tc_fence_after_sync();
        }
        if (ok && s > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            uint32_t o32[32];
            tmem_ld32(tO + c * 32, o32);
#pragma unroll
            for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
            tmem_st32(tO + c * 32, o32);
          }
        }
        m_run = m_new;
        float ls = 0.f;
        if (ok && mine) {
          const float neg_m = -m_run;
          float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int c = 0; c < 8; ++c) {   // 16 keys at a time: 8 bf16 pairs, 8 TMEM columns
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float x0, x1;
              fma2_bc(x0, x1, __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i]),
                      __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i + 1]), sl2, neg_m);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              add2(l4[2 * (i & 1)], l4[2 * (i & 1) + 1], p0, p1);
              pk[i] = pack_bf16x2(p0, p1);
            }
            tmem_st8_nowait(tP + c * 8, pk);
          }
          ls = (l4[0] + l4[1]) + (l4[2] + l4[3]);
          tmem_st_wait();
        }
        l_mine = l_mine * alpha + ls;
        // The previous tile's O is complete (its last P V was waited for above): take it out
        // of TMEM before this step's P is released, since this P V overwrites O.
        if (s == 0 && pend) {
          uint32_t orr[D / 2];
          if (ok) {
            read_o(orr);
          } else {
#pragma unroll
            for (int i = 0; i < D / 2; ++i) orr[i] = 0u;
          }
          if (ok) {
            tc_fence_before_sync();   // P (tcgen05.st) before the P V
            __syncwarp();
            if (lane == 0) mbar_arrive(b_p_full);
          }
          store_o(orr, ok);   // staged and stored while this P V runs
        } else if (ok) {
          tc_fence_before_sync();   // P and the O rescale (tcgen05.st) before the P V
          __syncwarp();
          if (lane == 0) mbar_arrive(b_p_full);
        }
      }
      // Row sum over both column blocks.
      named_bar_sync(pair_bar, 64);
      *x_mine = l_mine;
      named_bar_sync(pair_bar, 64);
      pend = true;
      pend_b = t.b;
      pend_h = t.h;
      pend_qt = t.qt;
      pend_m = m_run;
      pend_l = l_mine + *x_other;
      // Every one of the 256 threads got through this tile's waits.
      if (!named_bar_and(1, 256, ok)) {
        ok = false;
        break;
      }
    }
    if (ok && pend) {
      // the last tile: every thread passed the last tile-end barrier with ok
      uint32_t orr[D / 2];
      const bool got = wwait(b_pv_done, step - 1);
      if (got) {
        tc_fence_after_sync();
        read_o(orr);
      } else {
#pragma unroll
        for (int i = 0; i < D / 2; ++i) orr[i] = 0u;
      }
      store_o(orr, got);
    }
    if (tid == 128) bulk_wait_all();
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

}  // namespace

cudaError_t launch_cross_attn(const AttnArgs& a) {
  CUtensorMap mq, mk, mv, mo;
  const int qext = a.q_valid > 0 ? a.q_valid : 1;
  // Q rows past q_valid read as zeros; K and V are read up to Skv rows and masked per batch
  // on the device.
  if (!encode_bshd_map(&mq, a.q, a.B, qext, a.Sq, a.H, a.D) || !encode_bshd_map(&mk, a.k, a.B, a.Skv, a.Skv, a.H, a.D) ||
      !encode_bshd_map(&mv, a.v, a.B, a.Skv, a.Skv, a.H, a.D) || !encode_bshd_map(&mo, a.out, a.B, a.Sq, a.Sq, a.H, a.D))
    return cudaErrorInvalidValue;
  XParams p;
  p.B = a.B;
  p.Sq = a.Sq;
  p.Skv = a.Skv;
  p.H = a.H;
  p.q_valid = a.q_valid;
  p.n_qt = a.Sq / 128;
  const long long n_tiles = static_cast<long long>(a.B) * a.H * p.n_qt;
  if (n_tiles >= (1ll << 31)) return cudaErrorInvalidValue;
  p.n_tiles = static_cast<int>(n_tiles);
  p.kv_len = a.kv_valid_dev;
  p.scale_log2 = a.scale * kXLog2e;
  p.lse = a.lse;
  p.out = static_cast<uint16_t*>(a.out);
  cudaError_t e = device_status_ptr(&p.status);
  if (e != cudaSuccess) return e;
  int dev = 0, sm_count = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (sm_count < 1) return cudaErrorInvalidDevice;
  const int grid = p.n_tiles < sm_count ? p.n_tiles : sm_count;
  // Both head sizes request the D = 128 amount of shared memory: one CTA per SM, so that no
  // CTA waits for another's tensor memory (each allocates all 512 columns).
  constexpr int kSmem = XCfg<128>::kSmem;
  static_assert(XCfg<64>::kSmem <= kSmem, "shared memory of the D = 64 cross kernel");
  if (a.D == 128) {
    e = cudaFuncSetAttribute(cross_attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    cross_attn_kernel<128><<<grid, kXThreads, kSmem, a.stream>>>(mq, mk, mv, mo, p);
  } else {
    e = cudaFuncSetAttribute(cross_attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    cross_attn_kernel<64><<<grid, kXThreads, kSmem, a.stream>>>(mq, mk, mv, mo, p);
  }
  return cudaGetLastError();
}

}  // namespace dit
