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
// dominates: 97 MB of Q in and 97 MB of O out at B2 H40, against 21 MB of K and V. What
// limits such a kernel is the chain of dependent steps per query tile (S product, softmax,
// P.V product, read-out of O), so the CTA runs its tiles one after another through all eight
// softmax warps, and the products of a tile's neighbours run while its softmax does.
//   - Work is a flat list of 128-row query tiles over (b, h, tile). CTA c of a persistent grid
//     takes the contiguous range [c T / G, (c + 1) T / G). The live tiles of the range (a
//     valid query row and at least one key) are numbered n = 0, 1, ...; tile n uses TMEM
//     region n & 1 (256 columns) and Q buffer n & 1.
//   - Softmax: the two warps of a lane quarter (w and w + 4) share its 32 query rows. Warp-
//     group 0 takes the first half of a product's keys, warpgroup 1 the second. Each thread
//     finds its half's row maximum; the pair exchange it through shared memory (a slot per
//     row and warpgroup, double-buffered, and an mbarrier per quarter), take the larger as
//     the row's reference m (its ceiling, an integer in log2 units) and exponentiate their
//     halves against it. The two partial row sums go across at the next exchange.
//   - TMEM, per region: S of up to 256 keys in columns [0, 128 nkt). Each half's P (bf16
//     pairs) goes over S columns its own warpgroup has read already: warpgroup 0's to
//     [0, 32 nkt) in key order, warpgroup 1's to [96 nkt, 128 nkt), its 32-key chunks taken
//     from the last to the first. O = P V (tensor-memory A operand) goes to [64, 64 + D) for a
//     product of two key tiles and to [128, 128 + D) for one of one key tile: S columns that
//     are dead once the softmax is done.
//   - Overlap: the softmax warps read tile n - 1's O out of its region in the middle of tile
//     n's exponentials (of its last product), as soon as tile n - 1's P V is complete; the
//     read-out frees the region, and tile n + 1's S is issued into it at once. While the
//     softmax warps work on tile n, the tensor pipe runs tile n - 1's P V and tile n + 1's S.
//   - Q and O: tile n's Q lands in buffer n & 1. Once its S has completed the buffer is dead,
//     and the softmax stages tile n - 1's normalised O there (128-byte swizzle); the Q loader
//     writes it out with one TMA store and, once the store has read the buffer, loads tile
//     n + 2's Q into it. (A scattered store of O from registers, 32 rows per instruction,
//     measured far slower.)
//   - The keys and values of the current (b, h) stay in shared memory (a "fill", 256 rows of
//     K and of V) for all of the CTA's tiles of that head. When L_b > 256 a tile visits its
//     keys in two halves (key tiles {0, 1} and {2, n_kv - 1}), one product per key tile, with
//     the online softmax across products: the reference moves only when a product's maximum
//     exceeds it by more than kXRescale, and O and the sums are then scaled by the power of
//     two 2^(m_old - m_new), which is exact. Tile i of a run visits half i & 1 first, so
//     consecutive tiles share the fill at their boundary and a run of P tiles reads P + 1
//     fills. A fill's K lands on a barrier of its own, ahead of its V, so that the first S
//     product of a head waits only for K. A fill is released when both MMA issuers have
//     committed their last product on it.
//   - Roles: warp 0 loads Q and stores O (two buffers; the tile two ahead is warmed in L2);
//     warp 1 owns TMEM, loads the fills and zeroes the V rows past L_b of a fill's last V
//     tile (so that 0 * (pad contents) cannot reach O; K pad rows need nothing, their score
//     columns are masked to -inf); warp 2 issues the S products, warp 3 the P V products;
//     warps 4-11 are the softmax.
// Every wait is bounded (ptx.cuh); on a timeout the CTA records a status bit, raises its
// abort flag (the other roles' waits then give up at once), drains its copies and MMAs,
// frees TMEM and exits. No named barrier is used after the set-up, so no thread can be left
// waiting at one.

#include <cuda.h>
#include <cuda_bf16.h>

#include <type_traits>

#include "common.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kXThreads = 384;   // warps 0-3: Q loads, TMEM + fills, S issuer, P V issuer; 4-11: softmax
constexpr float kXLn2 = 0.69314718055994530942f;
constexpr float kXLog2e = 1.44269504088896340736f;
constexpr float kXRescale = 8.0f;   // log2 units: the reference may trail the maximum by up to 8
constexpr int kLenCache = 128;      // per-batch key lengths kept in shared memory
constexpr int kXQBufs = 2;          // Q buffers (tile n in buffer n & 1)
constexpr uint32_t kXRegion = 256;  // TMEM columns per region (tile n in region n & 1)

template <int D>
struct XCfg {
  static constexpr int kSub = D / 64;              // 64-column (128-byte) chunks per row
  static constexpr int kTile = 128 * D * 2;        // one 128-row bf16 tile
  static constexpr int kChunk = 128 * 128;         // one 128-row chunk (16 KB)
  static constexpr int kOffQ = 0;                  // kXQBufs Q buffers
  static constexpr int kOffK = kOffQ + kXQBufs * kTile;  // K: chunk c holds rows 0..255 at c * 2 kChunk
  static constexpr int kOffV = kOffK + 2 * kTile;  // V: two 128-row tiles
  static constexpr int kOffX = kOffV + 2 * kTile;  // exchange slots: float2 [2 buffers][2 warpgroups][128 rows]
  static constexpr int kOffLen = kOffX + 2 * 2 * 128 * 8;  // key lengths of the first kLenCache batches
  static constexpr int kOffBar = kOffLen + kLenCache * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;     // barriers + alignment slack
};
static_assert(XCfg<128>::kSmem <= 232448, "shared memory of the D = 128 cross kernel");

struct XBars {
  uint64_t q_full[kXQBufs], q_empty[kXQBufs], o_staged[kXQBufs];
  uint64_t kv_full, kv_ready, kv_empty, k_full;   // kv_full: V of a fill; k_full: its K
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];   // per TMEM region
  uint64_t xch[4];                                       // per lane quarter: the softmax exchange
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(XBars) <= 256, "barrier block");

struct XParams {
  int B, Sq, Skv, H, q_valid;
  int n_qt;          // 128-row query tiles per (b, h)
  int n_tiles;       // B * H * n_qt
  const int32_t* kv_len;
  float scale_log2;
  float* lse;
  uint16_t* out;
  unsigned int* status;
};

// One live query tile of the CTA's range and where it sits in its run (the live tiles of its
// (b, h) inside the range, which are consecutive).
struct XTile {
  int b, h, qt;
  int L;        // valid keys (>= 1)
  int n_kv;     // 128-key tiles holding them
  int i;        // index of this tile in its run
  int len;      // live tiles in the run
};

// Walks the CTA's range [g0, g1) of flat tiles head by head, with the coordinates kept
// incrementally (the threads that issue MMAs and loads share their schedulers with busy
// softmax warps, so a per-tile decode with divisions sat on the critical path). The key
// lengths of the first kLenCache batches are read from shared memory.
struct XWalk {
  int g, g1;          // next flat tile and the end of the range
  int b, h, qt;       // coordinates of flat tile g
  int L, n_kv;        // key length of batch b (0 for a bad or empty length)
  bool bad;           // batch b's length lies outside [0, Skv]
  int qt_first;       // first tile of the current head inside the range
  int run_len;        // live tiles of the current head inside the range
};
__device__ __forceinline__ void x_walk_head(XWalk& w, const XParams& p, const int* len_s) {
  const int raw = w.b < kLenCache ? len_s[w.b] : p.kv_len[w.b];
  w.bad = raw < 0 || raw > p.Skv;
  w.L = w.bad ? 0 : raw;
  w.n_kv = (w.L + 127) >> 7;
  w.qt_first = w.qt;
  const int n_live_qt = (p.q_valid + 127) >> 7;   // live tiles are a prefix of each head
  const int end_qt = min(p.n_qt, w.qt + (w.g1 - w.g));
  w.run_len = w.L > 0 ? max(0, min(end_qt, n_live_qt) - w.qt) : 0;
}
__device__ __forceinline__ void x_walk_init(XWalk& w, const XParams& p, const int* len_s, int g0, int g1) {
  w.g = g0;
  w.g1 = g1;
  const int bh = g0 / p.n_qt;
  w.qt = g0 - bh * p.n_qt;
  w.b = bh / p.H;
  w.h = bh - w.b * p.H;
  if (g0 < g1) x_walk_head(w, p, len_s);
}
// To the first tile of the next head.
__device__ __forceinline__ void x_walk_next_head(XWalk& w, const XParams& p, const int* len_s) {
  w.g += p.n_qt - w.qt;
  w.qt = 0;
  if (++w.h == p.H) {
    w.h = 0;
    ++w.b;
  }
  if (w.g < w.g1) x_walk_head(w, p, len_s);
}
// The next live tile of the range; false at its end.
__device__ __forceinline__ bool x_walk_next(XWalk& w, const XParams& p, const int* len_s, XTile& t) {
  while (w.g < w.g1) {
    if (w.qt - w.qt_first < w.run_len) {
      t.b = w.b;
      t.h = w.h;
      t.qt = w.qt;
      t.L = w.L;
      t.n_kv = w.n_kv;
      t.i = w.qt - w.qt_first;
      t.len = w.run_len;
      ++w.g;
      if (++w.qt == p.n_qt) {
        w.qt = 0;
        if (++w.h == p.H) {
          w.h = 0;
          ++w.b;
        }
        if (w.g < w.g1) x_walk_head(w, p, len_s);
      }
      return true;
    }
    x_walk_next_head(w, p, len_s);
  }
  return false;
}

// Fills of a run: one when n_kv <= 2, else len + 1 (fill k holds key half k & 1).
__device__ __forceinline__ int x_run_fills(const XTile& t) { return t.n_kv <= 2 ? 1 : t.len + 1; }
// Key tiles of fill k of the run: first tile and count.
__device__ __forceinline__ void x_fill_tiles(const XTile& t, int k, int& kt0, int& cnt) {
  if (t.n_kv <= 2) {
    kt0 = 0;
    cnt = t.n_kv;
  } else {
    const int half = k & 1;
    kt0 = 2 * half;
    cnt = half ? t.n_kv - 2 : 2;
  }
}

// The products of a live tile. n_kv <= 2: one product over all its keys. n_kv > 2: one
// product per key tile, the tiles of the half visited first (half i & 1, in fill i), then
// those of the other (in fill i + 1).
struct XStep {
  int fill;      // fill of the run it reads (0-based within the run)
  int j0;        // first slot of the fill it reads
  int kt;        // first key tile
  int nkt;       // key tiles in the product (1 or 2)
  bool release;  // the last product of the run that reads this fill
};
__device__ __forceinline__ int x_n_steps(const XTile& t) { return t.n_kv <= 2 ? 1 : t.n_kv; }
__device__ __forceinline__ XStep x_step(const XTile& t, int s) {
  XStep st;
  if (t.n_kv <= 2) {
    st.fill = 0;
    st.j0 = 0;
    st.kt = 0;
    st.nkt = t.n_kv;
    st.release = t.i == t.len - 1;
    return st;
  }
  const int h0 = t.i & 1;
  const int c0 = h0 ? t.n_kv - 2 : 2;   // key tiles of the half visited first
  const bool first = s < c0;
  const int half = first ? h0 : 1 - h0;
  st.j0 = first ? s : s - c0;
  st.kt = 2 * half + st.j0;
  st.nkt = 1;
  st.fill = first ? t.i : t.i + 1;
  // Fill i is read by tile i - 1's second half and tile i's first half; the run's last
  // fill by its last tile's second half.
  st.release = first ? s == c0 - 1 : (s == t.n_kv - 1 && t.i == t.len - 1);
  return st;
}

// 16-key groups holding a product's valid keys (1 .. 8 nkt).
__device__ __forceinline__ int x_groups(const XTile& t, const XStep& st) {
  return (min(128 * st.nkt, t.L - 128 * st.kt) + 15) >> 4;
}
// First TMEM column of O within a region: [64, 64 + D) after a product of two key tiles,
// [128, 128 + D) after products of one.
__device__ __forceinline__ uint32_t x_ocol(const XTile& t) { return t.n_kv == 2 ? 64u : 128u; }

// O = 0 and LSE = -inf for one tile's rows (columns [c0, c0 + D/2) of O by this warpgroup;
// the LSE by warpgroup 0), written directly.
template <int D>
__device__ __forceinline__ void x_write_empty(const XParams& p, int b, int h, int qt, int wg, int r) {
  const int row = qt * 128 + r;
  uint16_t* dst = p.out + ((static_cast<size_t>(b) * p.Sq + row) * p.H + h) * D + wg * (D / 2);
#pragma unroll
  for (int u = 0; u < D / 16; ++u) reinterpret_cast<uint4*>(dst)[u] = make_uint4(0, 0, 0, 0);
  if (wg == 0) p.lse[(static_cast<size_t>(b) * p.Sq + row) * p.H + h] = -INFINITY;
}

// Non-blocking test of a phase (the thread is never suspended): true once the phase with this
// parity has completed.
__device__ __forceinline__ bool x_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded_wait (ptx.cuh) by polling: the MMA issuers wait this way, so that each resumes as
// soon as the phase completes.
__device__ __forceinline__ bool x_poll(uint32_t bar, uint32_t parity, volatile int* cta_abort, unsigned int* dev_status,
                                       unsigned int code) {
  if (x_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (x_test_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*cta_abort) return false;
      if (globaltimer_ns() - t0 > wait_limit_ns()) {
        *cta_abort = 1;
        atomicOr(dev_status, code);
        return false;
      }
    }
  }
}

// Scales the fp32 columns [taddr, taddr + 32) of this thread's lane by a (warp-collective).
__device__ __forceinline__ void x_scale_f32_cols(uint32_t taddr, float a) {
  uint32_t v[32];
  tmem_ld32(taddr, v);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * a);
  tmem_st32(taddr, v);
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
    for (int i = 0; i < kXQBufs; ++i) {
      mbar_init(smem_u32(&bars->q_full[i]), 1);
      mbar_init(smem_u32(&bars->q_empty[i]), 1);
      mbar_init(smem_u32(&bars->o_staged[i]), 8);   // one arrival per softmax warp
    }
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->k_full), 1);
    mbar_init(smem_u32(&bars->kv_ready), 1);
    mbar_init(smem_u32(&bars->kv_empty), 2);   // one commit per MMA issuer
    for (int r = 0; r < 2; ++r) {
      mbar_init(smem_u32(&bars->s_full[r]), 1);
      mbar_init(smem_u32(&bars->p_full[r]), 8);   // one arrival per softmax warp
      mbar_init(smem_u32(&bars->pv_done[r]), 1);
      mbar_init(smem_u32(&bars->o_free[r]), 8);
      mbar_init(smem_u32(&bars->drain[r]), 1);
    }
    for (int q = 0; q < 4; ++q) mbar_init(smem_u32(&bars->xch[q]), 2);   // one arrival per warp of the pair
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
  const uint32_t b_k_full = smem_u32(&bars->k_full);
  const uint32_t b_kv_empty = smem_u32(&bars->kv_empty);

  if (warp < 4) {
    regs_dec<72>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------------ Q loads, O stores
      // Buffer b holds, in turn, Q of tile m (m & 1 == b) and, once that tile's last S has
      // completed, the O of tile m - 1, which the softmax stages there during tile m's last
      // product. Step m of this thread stores O(m - 3) out of buffer m & 1 and, once the store
      // has read it, loads Q(m) into it. After the last of the N live tiles, step N hands
      // buffer N & 1 to the softmax for O(N - 1) (a plain arrival on its q_full), and steps
      // N + 1 and N + 2 store the last two O.
      int m = 0;
      bool ok = true;
      // Coordinates (b, h, first row) of tiles m - 1, m - 2 and m - 3, shifted at every step.
      int b1 = 0, h1 = 0, q1 = 0, b2 = 0, h2 = 0, q2 = 0, b3 = 0, h3 = 0, q3 = 0;
      auto shift = [&](int b, int h, int q) {
        b3 = b2; h3 = h2; q3 = q2;
        b2 = b1; h2 = h1; q2 = q1;
        b1 = b; h1 = h; q1 = q;
      };
      int n_live = 1 << 30;   // live tiles: known once the walk has ended
      auto free_buffer = [&]() -> bool {   // buffer m & 1, for step m
        const int b = m & 1;
        if (m >= 3) {
          const int j = m - 3;   // staged in buffer (j + 1) & 1 == b during tile j + 1
          if (!bounded_wait(smem_u32(&bars->o_staged[b]), (j >> 1) & 1, abort_flag, status, kStatusTimeoutLoad))
            return false;
#pragma unroll
          for (int c = 0; c < C::kSub; ++c)
            tma_store_4d(&tm_o, sQ + b * C::kTile + c * C::kChunk, c * 64, h3, q3, b3);
          bulk_commit_group();
          bulk_wait_read();   // the buffer has been read out
        }
        // The buffer's previous Q (tile m - 2, if there is one) has been read by its last S.
        return m < kXQBufs || m - 2 >= n_live ||
               bounded_wait(smem_u32(&bars->q_empty[b]), ((m >> 1) - 1) & 1, abort_flag, status, kStatusTimeoutLoad);
      };
      XWalk w, ahead;
      x_walk_init(w, p, len_s, g0, g1);
      ahead = w;
      XTile t, ta;
      for (int i = 0; i < 2; ++i) x_walk_next(ahead, p, len_s, ta);   // two tiles ahead of w
      while (ok && x_walk_next(w, p, len_s, t)) {
        const int buf = m & 1;
        if (!(ok = free_buffer())) break;
        const uint32_t qb = smem_u32(&bars->q_full[buf]);
        mbar_arrive_expect_tx(qb, C::kTile);
#pragma unroll
        for (int c = 0; c < C::kSub; ++c)
          tma_load_4d(sQ + buf * C::kTile + c * C::kChunk, &tm_q, qb, c * 64, t.h, t.qt * 128, t.b);
        shift(t.b, t.h, t.qt * 128);
        ++m;
        // Warm L2 with the tile two ahead.
        if (x_walk_next(ahead, p, len_s, ta))
#pragma unroll
          for (int c = 0; c < C::kSub; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, ta.h, ta.qt * 128, ta.b);
      }
      n_live = m;
      bool handed = false;   // buffer n_live & 1 went to the softmax (its q_full moved on)
      for (; ok && n_live > 0 && m < n_live + 3; ++m) {
        if (!(ok = free_buffer())) break;
        if (m == n_live) {
          mbar_arrive(smem_u32(&bars->q_full[m & 1]));
          handed = true;
        }
        shift(0, 0, 0);
      }
      bulk_wait_all();
      // Let the loads in flight land before the CTA releases its shared memory (on the
      // normal path each has been waited for already, and these return at once). Once the
      // buffer was handed over, tile n_live - 2's load had landed (its S had completed).
      for (int j = n_live > kXQBufs ? n_live - kXQBufs : 0; j < n_live; ++j)
        if (!(handed && j == n_live - 2)) drain_wait(smem_u32(&bars->q_full[j & 1]), (j >> 1) & 1, status);
    } else if (warp == 1) {
      // ------------------------------------------------------------------ fills + V pad rows
      int e = 0;
      bool ok = true;
      XWalk w;
      x_walk_init(w, p, len_s, g0, g1);
      XTile t;
      while (ok && x_walk_next(w, p, len_s, t)) {
        if (t.i != 0) continue;   // once per run, at its first tile
        const int nf = x_run_fills(t);
        for (int k = 0; k < nf; ++k, ++e) {
          int kt0, cnt;
          x_fill_tiles(t, k, kt0, cnt);
          // 0: the previous fill was not released (nothing issued); 1: issued, not landed;
          // 2: landed.
          int got = 1;
          if (lane == 0) {
#ifdef DIT_TEST_HOOKS
            const bool skip = e == g_dit_test_skip_load;   // test build only: counted, never issued
#else
            constexpr bool skip = false;
#endif
            if (e > 0 && !bounded_wait(b_kv_empty, (e - 1) & 1, abort_flag, status, kStatusTimeoutLoad)) {
              got = 0;
            } else {
              if (!skip) {
                // K first (the S products need only K), then V on a barrier of its own.
                mbar_arrive_expect_tx(b_k_full, cnt * C::kTile);
                mbar_arrive_expect_tx(b_kv_full, cnt * C::kTile);
                for (int j = 0; j < cnt; ++j)
#pragma unroll
                  for (int c = 0; c < C::kSub; ++c)
                    tma_load_4d(sK + c * 2 * C::kChunk + j * C::kChunk, &tm_k, b_k_full, c * 64, t.h, (kt0 + j) * 128, t.b);
                for (int j = 0; j < cnt; ++j)
#pragma unroll
                  for (int c = 0; c < C::kSub; ++c)
                    tma_load_4d(sV + j * C::kTile + c * C::kChunk, &tm_v, b_kv_full, c * 64, t.h, (kt0 + j) * 128, t.b);
              }
              if (bounded_wait(b_kv_full, e & 1, abort_flag, status, kStatusTimeoutRope) &&
                  bounded_wait(b_k_full, e & 1, abort_flag, status, kStatusTimeoutRope)) {
                got = 2;
              } else if (!skip) {   // the copies land before the CTA exits
                drain_wait(b_kv_full, e & 1, status);
                drain_wait(b_k_full, e & 1, status);
              }
            }
          }
          if (__shfl_sync(0xffffffffu, got, 0) != 2) {
            ok = false;
            break;
          }
          const int jl = cnt - 1;                           // the fill's last V tile
          const int nv = min(128, t.L - (kt0 + jl) * 128);  // its valid rows (>= 1)
          if (nv < 128) {
            const uint32_t tile = sV + jl * C::kTile;
            const int n16 = (128 - nv) * 8;                 // 16-byte units per chunk
            for (int c = 0; c < C::kSub; ++c)
              for (int u = lane; u < n16; u += 32)
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(tile + c * C::kChunk + nv * 128 + u * 16),
                             "r"(0u)
                             : "memory");
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(b_kv_ready);
        }
      }
    } else if (lane == 0) {
      // ------------------------------------------------------------------ MMA issuers
      // Warp 2 issues every S = Q K^T, warp 3 every O += P V, each in tile order.
      const bool is_s = warp == 2;
      bool ok = true;
      // Polled waits: the issuer resumes as soon as the phase completes.
      auto wait = [&](uint32_t bar, int phase) -> bool {
        if (!x_poll(bar, phase & 1, abort_flag, status, kStatusTimeoutMma)) return false;
        tc_fence_after_sync();
        return true;
      };
      constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
      int n = -1, e_run = 0, e_total = 0;
      int ks0 = 0, ks1 = 0;   // products so far in regions 0 and 1 (scalars: no local memory)
      XWalk wk;
      x_walk_init(wk, p, len_s, g0, g1);
      XTile t;
      while (ok && x_walk_next(wk, p, len_s, t)) {
        ++n;
        if (t.i == 0) {
          e_run = e_total;
          e_total += x_run_fills(t);
        }
        const int rg = n & 1;
        const uint32_t region = tbase + static_cast<uint32_t>(rg) * kXRegion;
        const int ns = x_n_steps(t);
        for (int s = 0; ok && s < ns; ++s) {
          const XStep st = x_step(t, s);
          const int e = e_run + st.fill;
          const int ng = x_groups(t, st);
          const int kr = rg ? ks1 : ks0;   // this product's index in its region
          if (is_s) {
            if (s == 0) {
              if (!(ok = wait(smem_u32(&bars->q_full[rg]), n >> 1))) break;
              // The region's previous tile has been read out (its P V complete, O read).
              if (n >= 2 && !(ok = wait(smem_u32(&bars->o_free[rg]), (n >> 1) - 1))) break;
            } else if (!(ok = wait(smem_u32(&bars->pv_done[rg]), kr - 1))) {
              break;   // (above: the previous product's P has been read; S goes over it)
            }
            if (!(ok = wait(b_k_full, e))) break;
            const uint64_t da = smem_desc_sw128(sQ + rg * C::kTile, 16, 1024);
            const uint64_t db = smem_desc_sw128(sK + st.j0 * C::kChunk, 16, 1024);
            // N covers the product's valid keys in whole 16-key groups (the softmax never
            // reads the columns past them, and P V never reads the keys past them).
            const uint32_t idS = idesc_f16kind_f32(128, 16u * static_cast<uint32_t>(ng), true, false, false);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t offa = ((kk / 4) * C::kChunk + (kk % 4) * 32) >> 4;
              const uint64_t offb = ((kk / 4) * 2 * C::kChunk + (kk % 4) * 32) >> 4;
              mma_bf16_ss(region, da + offa, db + offb, idS, kk > 0);
            }
            mma_commit(smem_u32(&bars->s_full[rg]));
            if (s == ns - 1) mma_commit(smem_u32(&bars->q_empty[rg]));   // Q is read
          } else {
            if (!(ok = wait(smem_u32(&bars->p_full[rg]), kr))) break;
            if (!(ok = wait(b_kv_ready, e))) break;
            // Group gi (keys 16 gi ..) reads P columns 8 gi .. (warpgroup 1's half, from group
            // 4 nkt on, lies 64 nkt columns further) and rows 16 (gi % 8) .. of V tile gi / 8.
            const int hb = 4 * st.nkt;
            const uint32_t hoff = 64u * static_cast<uint32_t>(st.nkt);
            const uint32_t dO = region + x_ocol(t);
            const uint64_t dv0 = smem_desc_sw128(sV + st.j0 * C::kTile, C::kChunk, 1024);
#pragma unroll 1
            for (int gi = 0; gi < ng; ++gi)
              mma_bf16_ts(dO, region + 8u * static_cast<uint32_t>(gi) + (gi >= hb ? hoff : 0u),
                          dv0 + static_cast<uint64_t>(((gi >> 3) * C::kTile + (gi & 7) * 2048) >> 4), kIdO,
                          (s > 0 || gi > 0) ? 1u : 0u);
            mma_commit(smem_u32(&bars->pv_done[rg]));
          }
          if (st.release) mma_commit(b_kv_empty);
          if (rg) ++ks1;
          else ++ks0;
        }
      }
      // Every MMA of this thread completes before TMEM and shared memory are released.
      const uint32_t b_drain = smem_u32(&bars->drain[is_s ? 0 : 1]);
      mma_commit(b_drain);
      drain_wait(b_drain, 0, status);
    }
  } else {
    regs_inc<208>();
    // -------------------------------------------------------------------- softmax + epilogue
    const int wg = (warp - 4) >> 2;            // 0: first half of each product's keys; 1: second
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;         // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t b_x = smem_u32(&bars->xch[quarter]);
    float2* xslot = reinterpret_cast<float2*>(smem + C::kOffX);
    const float sl2 = p.scale_log2;
    auto wwait = [&](uint32_t bar, int phase) -> bool {
      int got = 0;
      if (lane == 0) got = bounded_wait(bar, phase & 1, abort_flag, status, kStatusTimeoutSoftmax) ? 1 : 0;
      return __shfl_sync(0xffffffffu, got, 0) != 0;
    };
    XWalk w;
    x_walk_init(w, p, len_s, g0, g1);
    // Tiles of the range with no valid query row or no key: O = 0, LSE = -inf, written
    // directly while the first products are on their way; a bad key length is reported.
    while (w.g < w.g1) {
      const int end_qt = min(p.n_qt, w.qt + (w.g1 - w.g));
      if (w.bad && wg == 0 && r == 0) atomicOr(status, kStatusBadKvLength);
      for (int qt = w.qt_first + w.run_len; qt < end_qt; ++qt) x_write_empty<D>(p, w.b, w.h, qt, wg, r);
      x_walk_next_head(w, p, len_s);
    }
    x_walk_init(w, p, len_s, g0, g1);
    bool ok = true;
    int n = -1, xc = 0;
    int ks0 = 0, ks1 = 0;   // products so far in regions 0 and 1 (scalars: no local memory)
    // Exchange with the partner thread (same row, other warpgroup): (a, b) out, theirs in.
    auto exchange = [&](float a, float b, float& pa, float& pb) {
      xslot[((xc & 1) * 2 + wg) * 128 + r] = make_float2(a, b);
      __syncwarp();                            // the warp's slots, before its arrival releases them
      if (lane == 0) mbar_arrive(b_x);
      ok = ok && wwait(b_x, xc);
      __syncwarp();                            // lane 0's acquire, before the warp reads
      const float2 v = xslot[((xc & 1) * 2 + (wg ^ 1)) * 128 + r];
      pa = v.x;
      pb = v.y;
      ++xc;
    };
    // The previous tile, whose O is read out and written during this one.
    bool pend = false;
    int pv_n = 0, pv_rg = 0, pv_k = 0, pv_b = 0, pv_h = 0, pv_qt = 0;
    uint32_t pv_ocol = 0;
    float pv_m = 0.f, pv_l = 0.f, pv_lt = 1.f;
    // Reads this thread's half of the previous tile's O (once its P V has completed), frees
    // the region, stages the normalised O in Q buffer (pv_n + 1) & 1 (the current tile's,
    // whose last S has completed) for the Q loader's store, and writes (warpgroup 0) the LSE.
    auto finish_prev = [&]() {
      uint32_t o[D / 64][32];
      if (ok) {
        const uint32_t src = tbase + lane_off + static_cast<uint32_t>(pv_rg) * kXRegion + pv_ocol + wg * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tmem_ld32_nowait(src + c * 32, o[c]);
        tmem_ld_wait_tied(o[0]);
#pragma unroll
        for (int c = 1; c < D / 64; ++c) tmem_reg_tie(o[c]);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->o_free[pv_rg]));   // the region may be reused
        const int qrow = pv_qt * 128 + r;
        const bool valid_row = qrow < p.q_valid;
        const float inv_l = 1.f / pv_lt;
        const uint32_t sO = sQ + static_cast<uint32_t>((pv_n + 1) & 1) * C::kTile;
#pragma unroll
        for (int u = 0; u < D / 16; ++u) {   // 16-byte units of this thread's half row
          uint4 v = make_uint4(0, 0, 0, 0);
          if (valid_row) {
            const uint32_t* f = &o[u >> 2][(u & 3) * 8];
            v.x = pack_bf16x2(__uint_as_float(f[0]) * inv_l, __uint_as_float(f[1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(f[2]) * inv_l, __uint_as_float(f[3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(f[4]) * inv_l, __uint_as_float(f[5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(f[6]) * inv_l, __uint_as_float(f[7]) * inv_l);
          }
          const uint32_t uu = static_cast<uint32_t>(wg * (D / 16) + u);   // unit within the row
          const uint32_t addr = sO + (uu >> 3) * C::kChunk + static_cast<uint32_t>(r) * 128u +
                                (((uu & 7u) ^ static_cast<uint32_t>(r & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                       : "memory");
        }
        fence_proxy_async_smem();   // the staged rows, before the store (async proxy) reads them
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->o_staged[(pv_n + 1) & 1]));
        if (wg == 0)
          p.lse[(static_cast<size_t>(pv_b) * p.Sq + qrow) * p.H + pv_h] =
              valid_row ? (pv_m + log2f(pv_lt)) * kXLn2 : -INFINITY;
      }
      pend = false;
    };
    XTile t;
    // One pass per live tile, and a last one (no tile) that reads out the last tile's O.
    for (;;) {
      const bool have = x_walk_next(w, p, len_s, t);
      if (!have && !pend) break;
      ++n;
      const int rg = n & 1;
      const uint32_t tR = tbase + lane_off + static_cast<uint32_t>(rg) * kXRegion;   // this row's region
      const uint32_t ocol = have ? x_ocol(t) : 0u;
      float m_run = 0.f, l_run = 0.f;   // reference (an integer) and this thread's partial sum
      const int ns = have ? x_n_steps(t) : 0;
      for (int s = 0; s < ns; ++s) {
        const XStep st = x_step(t, s);
        const int rg_k = rg ? ks1++ : ks0++;
        ok = ok && wwait(smem_u32(&bars->s_full[rg]), rg_k);
        if (ok) tc_fence_after_sync();
        const int half = 64 * st.nkt;                                   // keys per warpgroup
        const int lim0 = min(128 * st.nkt, t.L - st.kt * 128);          // valid keys of the product
        const int mine = max(0, min(half, lim0 - wg * half));           // of them in this half
        const int nch = (mine + 31) >> 5;                               // its 32-key chunks
        const uint32_t sS = tR + static_cast<uint32_t>(wg * half);      // its S columns
        const uint32_t sP = tR + static_cast<uint32_t>(wg * 96 * st.nkt);   // its P columns
        // Maximum of this half (log2 units).
        float mx = -INFINITY;
        if (ok) {
          const int nfull = mine >> 5;
          int j = 0;
#pragma unroll 1
          for (; j + 1 < nfull; j += 2) {   // two full chunks per wait
            uint32_t v[32], u[32];
            tmem_ld32_nowait(sS + 32 * j, v);
            tmem_ld32_nowait(sS + 32 * j + 32, u);
            tmem_ld_wait_tied(v);
            tmem_reg_tie(u);
            float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              m0 = fmax3(m0, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
              m1 = fmax3(m1, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
              m2 = fmax3(m2, __uint_as_float(u[i]), __uint_as_float(u[i + 1]));
              m3 = fmax3(m3, __uint_as_float(u[i + 2]), __uint_as_float(u[i + 3]));
            }
            mx = fmax3(mx, fmax3(m0, m1, m2), m3);
          }
#pragma unroll 1
          for (; j < nch; ++j) {
            uint32_t v[32];
            tmem_ld32(sS + 32 * j, v);
            const int lim = mine - 32 * j;
            float m0 = -INFINITY, m1 = -INFINITY;
            if (lim >= 32) {
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                m0 = fmax3(m0, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                m1 = fmax3(m1, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                m0 = fmaxf(m0, i < lim ? __uint_as_float(v[i]) : -INFINITY);
                m1 = fmaxf(m1, i + 1 < lim ? __uint_as_float(v[i + 1]) : -INFINITY);
              }
            }
            mx = fmax3(mx, m0, m1);
          }
          mx *= sl2;
        }
        // The pair's maximum; with the first product of a tile, the previous tile's partial
        // sums go across too.
        float pmx = -INFINITY, pl = 0.f;
        if (ok) exchange(mx, pend && s == 0 ? pv_l : 0.f, pmx, pl);
        if (pend && s == 0) pv_lt = pv_l + pl;
        const float mt = fmaxf(mx, pmx);
        const bool grow = s > 0 && mt > m_run + kXRescale;   // the same in both threads of the pair
        if (s == 0) m_run = ceilf(mt);                          // the product has a valid key
        // The rescale reads and writes TMEM with warp-collective instructions, so the whole
        // warp takes the branch (a = 1 in the rows whose reference stays). O of the earlier
        // products is complete (this product's S was issued after their P V); P of this one
        // is not written yet.
        if (__any_sync(0xffffffffu, grow)) {
          const float m_new = grow ? ceilf(mt) : m_run;
          const float a = ex2_approx(m_run - m_new);   // a power of two; 1 where m stays
          l_run *= a;
          m_run = m_new;
          if (ok) {
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) x_scale_f32_cols(tR + ocol + wg * (D / 2) + c * 32, a);
          }
        }
        // Exponentials: chunk j (S columns 32 j .. of this half) to P columns 16 j .. of this
        // half's P range. Warpgroup 1 walks its chunks from the last, so that each P lands on
        // S columns it has read already.
        const float neg_m = -m_run;
        float l_step = 0.f;
        auto chunk = [&](int j, int lim, auto masked_tag) {
          constexpr bool kMasked = decltype(masked_tag)::value;
          uint32_t v[32];
          tmem_ld32(sS + 32 * j, v);
          float l4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float x0, x1;
            fma2_bc(x0, x1, __uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]), sl2, neg_m);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if (kMasked) {
              p0 = 2 * i < lim ? p0 : 0.f;
              p1 = 2 * i + 1 < lim ? p1 : 0.f;
            }
            add2(l4[2 * (i & 1)], l4[2 * (i & 1) + 1], p0, p1);
            pk[i] = pack_bf16x2(p0, p1);
          }
          tmem_st16_nowait(sP + 16 * j, pk);
          l_step += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        };
        // The previous tile's O is read out during this tile's last product (whose Q buffer,
        // dead then, takes it), as soon as its P V has completed: the chunk loop stops when
        // it has, the O goes out, and the loop resumes.
        bool poll = pend && s == ns - 1;
        int idx = 0;
        if (ok) {
#pragma unroll 1
          for (;;) {
            bool hit = false;
#pragma unroll 1
            for (; idx < nch; ++idx) {
              const int j = wg ? nch - 1 - idx : idx;
              const int lim = mine - 32 * j;
              if (lim >= 32) chunk(j, 32, std::false_type{});
              else chunk(j, lim, std::true_type{});
              if (poll) {
                int got = 0;
                if (lane == 0) got = x_test_wait(smem_u32(&bars->pv_done[pv_rg]), pv_k & 1) ? 1 : 0;
                if (__shfl_sync(0xffffffffu, got, 0)) {
                  ++idx;
                  hit = true;
                  break;
                }
              }
            }
            if (!hit) break;
            tc_fence_after_sync();
            finish_prev();
            poll = false;
          }
        }
        l_run += l_step;
        if (ok) {
          tmem_st_wait();
          tc_fence_before_sync();   // P (tcgen05.st) and any O rescale before the P V
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->p_full[rg]));
        }
      }
      if (!have) {
        // The last tile's partial sums, and the buffer for its O: the Q loader hands over
        // buffer n & 1 with a plain arrival.
        float unused, pl = 0.f;
        if (ok) exchange(0.f, pv_l, unused, pl);
        pv_lt = pv_l + pl;
        ok = ok && wwait(smem_u32(&bars->q_full[n & 1]), n >> 1);
      }
      if (pend) {   // not read out during the tile
        ok = ok && wwait(smem_u32(&bars->pv_done[pv_rg]), pv_k);
        if (ok) tc_fence_after_sync();
        finish_prev();
      }
      if (!have) break;
      pend = true;
      pv_n = n;
      pv_rg = rg;
      pv_k = (rg ? ks1 : ks0) - 1;   // its last product's P V
      pv_b = t.b;
      pv_h = t.h;
      pv_qt = t.qt;
      pv_ocol = ocol;
      pv_m = m_run;
      pv_l = l_run;
    }
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

#ifdef DIT_TEST_HOOKS
cudaError_t cross_attn_set_test_hooks(unsigned long long wait_limit_ns, int skip_fill) {
  cudaError_t e = cudaMemcpyToSymbol(g_dit_test_wait_limit_ns, &wait_limit_ns, sizeof(wait_limit_ns));
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_dit_test_skip_load, &skip_fill, sizeof(skip_fill));
  return e;
}
#endif

}  // namespace dit
