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
// limits such a kernel is the chain of dependent steps per query tile (Q load, S product,
// softmax, P.V product, read-out of O, store), not any one unit, so the design keeps two of
// these chains in flight per SM and gives them nothing to wait for from each other.
//   - Work is a flat list of 128-row query tiles over (b, h, tile). CTA c of a persistent grid
//     takes the contiguous range [c T / G, (c + 1) T / G). The live tiles of the range (a
//     valid query row and at least one key) are numbered n = 0, 1, ...; tile n belongs to
//     softmax warpgroup n & 1 and to Q buffer n % 3. Each warpgroup owns its tiles outright:
//     one thread per query row holds every key column of that row, so the row maximum and
//     sum need no exchange between warpgroups.
//   - The keys and values of the current (b, h) stay in shared memory (a "fill", 256 rows of
//     K and of V) for all of the CTA's tiles of that head. When L_b > 256 a tile visits its
//     keys in two halves (key tiles {0, 1} and {2, n_kv - 1}); the two tiles of a pair
//     (in-run indices 2p and 2p + 1, one per warpgroup) visit the halves in the order
//     (p & 1, 1 - (p & 1)), so a pair's second half is the next pair's first and a run of
//     P pairs needs P + 1 fills. A fill is released when both MMA issuers have arrived on it:
//     by a commit after their last product on it, or, for an issuer with no product on it, by
//     a plain arrival once it has landed.
//   - TMEM: each warpgroup has 256 columns. With n_kv <= 2, S = Q K^T is one product of N =
//     128 n_kv keys into columns [0, 128 n_kv); the softmax writes P (bf16 pairs) over the
//     columns it has already read, [0, 64 n_kv); O = P V (tensor-memory A operand) goes to
//     columns [128, 128 + D), over S columns that are dead by then. With n_kv > 2 each key
//     tile is a step of its own (S in [0, 128), P in [0, 64)), with the online softmax across
//     steps. A warpgroup's next S is issued once its previous P.V is complete (and, when it
//     covers O's columns, once O has been read out).
//   - The softmax reads S once, 32 columns at a time, and keeps a reference m that trails the
//     running maximum by at most kXRescale (log2 units) and is an integer: when a chunk's
//     maximum exceeds m + kXRescale, m becomes its ceiling, and what the row has accumulated
//     (P of the product's earlier chunks, O of earlier steps, the sum) is scaled by the power
//     of two 2^(m_old - m_new), which is exact.
//   - Epilogue: O is read out of TMEM, normalised and staged in the tile's own Q buffer (Q is
//     dead once the tile's products have completed) in the 128-byte swizzle. The Q loader
//     writes it with one TMA store and, once the store has read the buffer, loads tile n + 3's
//     Q into it; the softmax warps never wait for a store.
//   - Warpgroup 1's first S waits for warpgroup 0's first S to complete, which puts the two
//     chains out of phase: while one warpgroup exponentiates, the other's products run.
//   - Roles: warp 0 loads Q and stores O (three buffers; the next two tiles are warmed in L2); warp 1 owns
//     TMEM, loads the fills and zeroes the V rows past L_b of a fill's last V tile (so that
//     0 * (pad contents) cannot reach O; K pad rows need nothing, their score columns are
//     masked to -inf); warps 2 and 3 issue the MMAs of softmax warpgroups 0 and 1; warps 4-7
//     and 8-11 are the two softmax warpgroups.
// Every wait is bounded (ptx.cuh); on a timeout the CTA records a status bit, raises its
// abort flag (the other roles' waits then give up at once), drains its copies and MMAs,
// frees TMEM and exits. No named barrier is used after the set-up, so no thread can be left
// waiting at one.

#include <cuda_bf16.h>

#include <type_traits>

#include "common.h"
#include "ptx.cuh"

namespace dit {
namespace {

constexpr int kXThreads = 384;   // warps 0-3: Q loads, TMEM + fills, two MMA issuers; 4-11: softmax
constexpr float kXLn2 = 0.69314718055994530942f;
constexpr float kXLog2e = 1.44269504088896340736f;
constexpr float kXRescale = 8.0f;   // log2 units: the reference may trail the maximum by up to 8
constexpr int kLenCache = 128;      // per-batch key lengths kept in shared memory
constexpr int kXQBufs = 3;          // Q buffers (each also stages its tile's O)
constexpr uint32_t kXRegion = 256;  // TMEM columns per softmax warpgroup
constexpr uint32_t kXColO = 128;    // O within a region: columns [128, 128 + D)

template <int D>
struct XCfg {
  static constexpr int kSub = D / 64;              // 64-column (128-byte) chunks per row
  static constexpr int kTile = 128 * D * 2;        // one 128-row bf16 tile
  static constexpr int kChunk = 128 * 128;         // one 128-row chunk (16 KB)
  static constexpr int kOffQ = 0;                  // kXQBufs Q buffers
  static constexpr int kOffK = kOffQ + kXQBufs * kTile;  // K: chunk c holds rows 0..255 at c * 2 kChunk
  static constexpr int kOffV = kOffK + 2 * kTile;  // V: two 128-row tiles
  static constexpr int kOffLen = kOffV + 2 * kTile;      // key lengths of the first kLenCache batches
  static constexpr int kOffBar = kOffLen + kLenCache * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;     // barriers + alignment slack
};
static_assert(XCfg<128>::kSmem <= 232448, "shared memory of the D = 128 cross kernel");

struct XBars {
  uint64_t q_full[kXQBufs], o_staged[kXQBufs];
  uint64_t kv_full, kv_ready, kv_empty;
  uint64_t s_full[2], p_full[2], pv_done[2], o_free[2];
  uint64_t drain[2];
  uint64_t started;   // warpgroup 0's first S is complete (one phase only)
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
  uint16_t* out;     // for the direct writes of empty tiles
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

// Fills of a run: one when n_kv <= 2, else pairs + 1 (fill k holds key half k & 1).
__device__ __forceinline__ int x_run_fills(const XTile& t) { return t.n_kv <= 2 ? 1 : ((t.len + 1) >> 1) + 1; }
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

// The products of a live tile. n_kv <= 2: one step over all its keys. n_kv > 2: one step per
// key tile, the tiles of the first half visited, then those of the second.
struct XStep {
  int fill;         // fill of the run it reads (0-based within the run)
  int j0;           // first slot of the fill it reads
  int kt;           // first key tile
  int nkt;          // key tiles in the product (1 or 2)
  bool group_end;   // last step of the tile that reads this fill
  bool first_half;  // n_kv > 2: the step reads the pair's first half
};
__device__ __forceinline__ int x_n_steps(const XTile& t) { return t.n_kv <= 2 ? 1 : t.n_kv; }
__device__ __forceinline__ XStep x_step(const XTile& t, int s) {
  XStep st;
  if (t.n_kv <= 2) {
    st.fill = 0;
    st.j0 = 0;
    st.kt = 0;
    st.nkt = t.n_kv;
    st.group_end = true;
    st.first_half = false;
    return st;
  }
  const int pair = t.i >> 1;
  const int h0 = pair & 1;
  const int c0 = h0 ? t.n_kv - 2 : 2;   // key tiles of the half visited first
  st.first_half = s < c0;
  const int half = st.first_half ? h0 : 1 - h0;
  st.j0 = st.first_half ? s : s - c0;
  st.kt = 2 * half + st.j0;
  st.nkt = 1;
  st.fill = st.first_half ? pair : pair + 1;
  st.group_end = st.first_half ? (s == c0 - 1) : (s == t.n_kv - 1);
  return st;
}

// 16-key groups holding a step's valid keys (1 .. 8 nkt).
__device__ __forceinline__ int x_groups(const XTile& t, const XStep& st) {
  return (min(128 * st.nkt, t.L - 128 * st.kt) + 15) >> 4;
}

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
// Scales 16 columns of bf16 pairs by a (a power of two, so exactly; warp-collective).
__device__ __forceinline__ void x_scale_bf16_cols16(uint32_t taddr, float a) {
  uint32_t v[16];
  tmem_ld16(taddr, v);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = pack_bf16x2(bf16lo_to_f32(v[i]) * a, bf16hi_to_f32(v[i]) * a);
  tmem_st16(taddr, v);
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
      mbar_init(smem_u32(&bars->o_staged[i]), 4);   // the four warps of the tile's warpgroup
    }
    mbar_init(smem_u32(&bars->kv_full), 1);
    mbar_init(smem_u32(&bars->kv_ready), 1);
    mbar_init(smem_u32(&bars->kv_empty), 2);   // one arrival per MMA issuer
    for (int w = 0; w < 2; ++w) {
      mbar_init(smem_u32(&bars->s_full[w]), 1);
      mbar_init(smem_u32(&bars->p_full[w]), 4);
      mbar_init(smem_u32(&bars->pv_done[w]), 1);
      mbar_init(smem_u32(&bars->o_free[w]), 4);
      mbar_init(smem_u32(&bars->drain[w]), 1);
    }
    mbar_init(smem_u32(&bars->started), 1);
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

  if (warp < 4) {
    regs_dec<64>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------------ Q loads, O stores
      // Tile n's Q lands in buffer n % 3, and its O is staged there by its warpgroup; this
      // thread stores it, and once the store has read the buffer, loads tile n + 3's Q into it.
      int n = -1, issued = 0, stored = 0;
      int cb[kXQBufs] = {}, ch[kXQBufs] = {}, cq[kXQBufs] = {};   // coordinates of each buffer's tile
      bool ok = true;
      auto store = [&](int m) -> bool {   // tile m's O, once its warpgroup has staged it
        const int b = m % kXQBufs;
        if (!bounded_wait(smem_u32(&bars->o_staged[b]), (m / kXQBufs) & 1, abort_flag, status, kStatusTimeoutLoad))
          return false;
#pragma unroll
        for (int c = 0; c < C::kSub; ++c) tma_store_4d(&tm_o, sQ + b * C::kTile + c * C::kChunk, c * 64, ch[b], cq[b], cb[b]);
        bulk_commit_group();
        stored = m + 1;
        return true;
      };
      XWalk w, ahead;
      x_walk_init(w, p, len_s, g0, g1);
      ahead = w;
      XTile t, ta;
      for (int i = 0; i < 2; ++i) x_walk_next(ahead, p, len_s, ta);   // two tiles ahead of w
      while (ok && x_walk_next(w, p, len_s, t)) {
        ++n;
        const int buf = n % kXQBufs;
        if (n >= kXQBufs) {
          if (!(ok = store(n - kXQBufs))) break;
          bulk_wait_read();   // the buffer has been read out
        }
        const uint32_t qb = smem_u32(&bars->q_full[buf]);
        mbar_arrive_expect_tx(qb, C::kTile);
#pragma unroll
        for (int c = 0; c < C::kSub; ++c)
          tma_load_4d(sQ + buf * C::kTile + c * C::kChunk, &tm_q, qb, c * 64, t.h, t.qt * 128, t.b);
        cb[buf] = t.b;
        ch[buf] = t.h;
        cq[buf] = t.qt * 128;
        issued = n + 1;
        // Warm L2 with the tile two ahead, so that each refill of a buffer is an L2 hit.
        if (x_walk_next(ahead, p, len_s, ta))
#pragma unroll
          for (int c = 0; c < C::kSub; ++c) tma_prefetch_l2_4d(&tm_q, c * 64, ta.h, ta.qt * 128, ta.b);
      }
      for (int m = stored; ok && m < issued; ++m) ok = store(m);
      bulk_wait_all();
      // Let the loads in flight land before the CTA releases its shared memory (on the
      // normal path each has been waited for already, and these return at once).
      for (int m = issued > kXQBufs ? issued - kXQBufs : 0; m < issued; ++m)
        drain_wait(smem_u32(&bars->q_full[m % kXQBufs]), (m / kXQBufs) & 1, status);
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
            if (e > 0 && !bounded_wait(b_kv_empty, (e - 1) & 1, abort_flag, status, kStatusTimeoutLoad)) {
              got = 0;
            } else {
              mbar_arrive_expect_tx(b_kv_full, 2 * cnt * C::kTile);
              for (int j = 0; j < cnt; ++j) {
                const int key0 = (kt0 + j) * 128;
#pragma unroll
                for (int c = 0; c < C::kSub; ++c) {
                  tma_load_4d(sK + c * 2 * C::kChunk + j * C::kChunk, &tm_k, b_kv_full, c * 64, t.h, key0, t.b);
                  tma_load_4d(sV + j * C::kTile + c * C::kChunk, &tm_v, b_kv_full, c * 64, t.h, key0, t.b);
                }
              }
              if (bounded_wait(b_kv_full, e & 1, abort_flag, status, kStatusTimeoutRope)) got = 2;
              else drain_wait(b_kv_full, e & 1, status);   // the copies land before the CTA exits
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
      // ------------------------------------------------------------------ MMA issuers (warps 2, 3)
      const int w = warp - 2;   // the softmax warpgroup served
      constexpr uint32_t kIdO = idesc_bf16_f32(128, D, false, true);
      const uint32_t region = tbase + static_cast<uint32_t>(w) * kXRegion;
      const uint32_t b_s_full = smem_u32(&bars->s_full[w]), b_p_full = smem_u32(&bars->p_full[w]);
      const uint32_t b_pv_done = smem_u32(&bars->pv_done[w]), b_o_free = smem_u32(&bars->o_free[w]);
      bool ok = true;
      // Polled waits: the issuer resumes as soon as the phase completes.
      auto wait = [&](uint32_t bar, int phase) -> bool {
        if (!x_poll(bar, phase & 1, abort_flag, status, kStatusTimeoutMma)) return false;
        tc_fence_after_sync();
        return true;
      };
      int n = -1, k = 0, tcnt = 0, e_run = 0, e_total = 0, released = 0;
      XWalk wk;
      x_walk_init(wk, p, len_s, g0, g1);
      XTile t;
      while (ok && x_walk_next(wk, p, len_s, t)) {
        ++n;
        if (t.i == 0) {
          e_run = e_total;
          e_total += x_run_fills(t);
        }
        if ((n & 1) != w) continue;
        const int buf = n % kXQBufs;
        const int ns = x_n_steps(t);
        for (int s = 0; ok && s < ns; ++s, ++k) {
          const XStep st = x_step(t, s);
          const int e = e_run + st.fill;
          // Fills before e that this warpgroup does not read: arrive once each has landed.
          while (ok && released < e) {
            if (!(ok = wait(b_kv_full, released))) break;
            mbar_arrive(b_kv_empty);
            ++released;
          }
          if (!ok) break;
          if (s == 0 && !(ok = wait(smem_u32(&bars->q_full[buf]), n / kXQBufs))) break;
          if (!(ok = wait(b_kv_full, e))) break;
          // The previous P V of this warpgroup is complete: its P columns may be overwritten.
          if (k > 0 && !(ok = wait(b_pv_done, k - 1))) break;
          // An S of 256 keys covers O's columns: the previous tile's O has been read out.
          const bool s_over_o = st.nkt == 2;
          if (s == 0 && tcnt > 0 && s_over_o && !(ok = wait(b_o_free, tcnt - 1))) break;
          // Warpgroup 1 starts once warpgroup 0's first S is complete, so that the two chains
          // run out of phase: one warpgroup's softmax while the other's products run.
          if (w == 1 && k == 0 && !(ok = wait(smem_u32(&bars->started), 0))) break;
          {
            const uint64_t da = smem_desc_sw128(sQ + buf * C::kTile, 16, 1024);
            const uint64_t db = smem_desc_sw128(sK + st.j0 * C::kChunk, 16, 1024);
            // N covers the step's valid keys in whole 16-key groups (the softmax never reads
            // the columns past them, and P V never reads the keys past them).
            const uint32_t idS = idesc_f16kind_f32(128, 16u * static_cast<uint32_t>(x_groups(t, st)), true, false, false);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t offa = ((kk / 4) * C::kChunk + (kk % 4) * 32) >> 4;
              const uint64_t offb = ((kk / 4) * 2 * C::kChunk + (kk % 4) * 32) >> 4;
              mma_bf16_ss(region, da + offa, db + offb, idS, kk > 0);
            }
            mma_commit(b_s_full);
            if (w == 0 && k == 0) mma_commit(smem_u32(&bars->started));
          }
          if (!(ok = wait(b_p_full, k))) break;
          // The first P V of a tile overwrites O: the previous tile's O has been read out.
          if (s == 0 && tcnt > 0 && !s_over_o && !(ok = wait(b_o_free, tcnt - 1))) break;
          if (!(ok = wait(b_kv_ready, e))) break;
          // The 16-key groups holding the step's valid keys: group gi reads P columns 8 gi ..
          // and rows 16 (gi % 8) .. of V tile gi / 8.
          const int ng = x_groups(t, st);
          const uint64_t dv0 = smem_desc_sw128(sV + st.j0 * C::kTile, C::kChunk, 1024);
#pragma unroll 1
          for (int gi = 0; gi < ng; ++gi)
            mma_bf16_ts(region + kXColO, region + gi * 8,
                        dv0 + static_cast<uint64_t>(((gi >> 3) * C::kTile + (gi & 7) * 2048) >> 4), kIdO,
                        (s > 0 || gi > 0) ? 1u : 0u);
          mma_commit(b_pv_done);
          // Release the fill after this warpgroup's last product on it: a pair's first half is
          // the previous pair's second, read already; otherwise this warpgroup's next tile of
          // the run (i + 2), if there is one, reads the same fill.
          if (st.group_end && (st.first_half || t.i + 2 >= t.len)) {
            mma_commit(b_kv_empty);
            released = e + 1;
          }
        }
        ++tcnt;
      }
      while (ok && released < e_total) {
        if (!(ok = wait(b_kv_full, released))) break;
        mbar_arrive(b_kv_empty);
        ++released;
      }
      // Every MMA of this thread completes before TMEM and shared memory are released.
      mma_commit(smem_u32(&bars->drain[w]));
      drain_wait(smem_u32(&bars->drain[w]), 0, status);
    }
  } else {
    regs_inc<216>();
    // -------------------------------------------------------------------- softmax + epilogue
    const int wg = (warp - 4) >> 2;            // warpgroup: tiles n with n & 1 == wg
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;         // query row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tR = tbase + lane_off + static_cast<uint32_t>(wg) * kXRegion;   // this row's region
    const uint32_t b_s_full = smem_u32(&bars->s_full[wg]), b_p_full = smem_u32(&bars->p_full[wg]);
    const uint32_t b_pv_done = smem_u32(&bars->pv_done[wg]), b_o_free = smem_u32(&bars->o_free[wg]);
    const float sl2 = p.scale_log2;
    const uint32_t p_sw = static_cast<uint32_t>(r & 7);
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
    int n = -1, k = 0, tcnt = 0;
    bool ok = true;
    XTile t;
    while (x_walk_next(w, p, len_s, t)) {
      ++n;
      if ((n & 1) != wg) continue;
      const int buf = n % kXQBufs;
      float m_run = -INFINITY, l_run = 0.f;   // reference (an integer once set) and row sum
      const int ns = x_n_steps(t);
      for (int s = 0; s < ns; ++s, ++k) {
        const XStep st = x_step(t, s);
        ok = ok && wwait(b_s_full, k);
        if (ok) tc_fence_after_sync();
        // One pass over the step's S columns, 32 at a time (a small loop keeps the code that
        // the softmax warps run between tiles in the instruction cache). Each chunk's maximum
        // may move the reference: when it lies more than kXRescale above it, what the row has
        // accumulated (P of the step's earlier chunks, O of the earlier steps, the sum) is
        // scaled by the exact power of two 2^(m_old - m_new) first. P of chunk q goes to
        // columns 16 q .. 16 q + 15, which hold S this thread has already read (chunk q / 2).
        float l_step = 0.f;   // sum of this step's P so far
        // Chunk q of the step: S columns 32 q .. + 31 (of which `lim` are valid keys); its
        // maximum, a rescale if the reference has to move, the exponentials and P. MASKED:
        // the chunk has fewer than 32 valid keys (only the step's last chunk can).
        auto chunk = [&](int q, int lim, auto masked_tag) {
          constexpr bool kMasked = decltype(masked_tag)::value;
          uint32_t v[32];
          tmem_ld32(tR + q * 32, v);
          auto sv = [&](int i) -> float {
            return (kMasked && i >= lim) ? -INFINITY : __uint_as_float(v[i]);
          };
          float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
          for (int i = 0; i < 32; i += 4) {
            m0 = fmax3(m0, sv(i), sv(i + 1));
            m1 = fmax3(m1, sv(i + 2), sv(i + 3));
          }
          const float mt = fmaxf(m0, m1) * sl2;
          const bool first = s == 0 && q == 0;
          const bool grow = !first && mt > m_run + kXRescale;
          if (first) m_run = ceilf(mt);   // the tile's first chunk has a valid column
          if (__any_sync(0xffffffffu, grow)) {
            const float m_new = grow ? ceilf(mt) : m_run;
            const float a = ex2_approx(m_run - m_new);   // a power of two; 1 where m stays
            l_run = (l_run + l_step) * a;
            l_step = 0.f;
            m_run = m_new;
            tmem_st_wait();
#pragma unroll 1
            for (int g = 0; g < q; ++g) x_scale_bf16_cols16(tR + g * 16, a);
            // O of the earlier steps: their P V is complete (this step's S was issued after it).
            if (s > 0) {
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) x_scale_f32_cols(tR + kXColO + c * 32, a);
            }
          }
          const float neg_m = -m_run;
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
          tmem_st16_nowait(tR + q * 16, pk);
          l_step += (l4[0] + l4[1]) + (l4[2] + l4[3]);
        };
        if (ok) {
          const int lim0 = min(128 * st.nkt, t.L - st.kt * 128);   // valid keys of the step
          const int nfull = lim0 >> 5;                               // chunks with 32 of them
#pragma unroll 1
          for (int q = 0; q < nfull; ++q) chunk(q, 32, std::false_type{});
          // The last chunk with valid keys, if partial. P V reads only the step's valid keys
          // in whole 16-key groups, so no P column past them is read.
          if ((lim0 & 31) != 0) chunk(nfull, lim0 & 31, std::true_type{});
        }
        l_run += l_step;
        if (ok) {
          tmem_st_wait();
          tc_fence_before_sync();   // P (tcgen05.st) and any rescale before the P V
          __syncwarp();
          if (lane == 0) mbar_arrive(b_p_full);
        }
      }
      // Epilogue: O out of TMEM, normalised, staged in this tile's Q buffer (the Q loader
      // stores it).
      uint32_t orr[D / 32][32];
      ok = ok && wwait(b_pv_done, k - 1);
      if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tmem_ld32_nowait(tR + kXColO + c * 32, orr[c]);
        tmem_ld_wait_tied(orr[0]);
#pragma unroll
        for (int c = 1; c < D / 32; ++c) tmem_reg_tie(orr[c]);
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_o_free);   // O may be overwritten
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[c][i] = 0u;
      }
      const int qrow = t.qt * 128 + r;
      const bool valid_row = qrow < p.q_valid;
      const float inv_l = 1.f / l_run;
      const uint32_t sO = sQ + buf * C::kTile;
#pragma unroll
      for (int u = 0; u < D / 8; ++u) {   // 16-byte units of the row
        uint4 o = make_uint4(0, 0, 0, 0);
        if (valid_row) {
          const uint32_t* f = &orr[u >> 2][(u & 3) * 8];
          o.x = pack_bf16x2(__uint_as_float(f[0]) * inv_l, __uint_as_float(f[1]) * inv_l);
          o.y = pack_bf16x2(__uint_as_float(f[2]) * inv_l, __uint_as_float(f[3]) * inv_l);
          o.z = pack_bf16x2(__uint_as_float(f[4]) * inv_l, __uint_as_float(f[5]) * inv_l);
          o.w = pack_bf16x2(__uint_as_float(f[6]) * inv_l, __uint_as_float(f[7]) * inv_l);
        }
        const uint32_t addr = sO + static_cast<uint32_t>(u >> 3) * C::kChunk + static_cast<uint32_t>(r) * 128u +
                              ((static_cast<uint32_t>(u & 7) ^ p_sw) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                     : "memory");
      }
      fence_proxy_async_smem();   // the staged row, before the store (async proxy) reads it
      __syncwarp();
      if (!ok) break;
      if (lane == 0) mbar_arrive(smem_u32(&bars->o_staged[buf]));
      p.lse[(static_cast<size_t>(t.b) * p.Sq + qrow) * p.H + t.h] =
          valid_row ? (m_run + log2f(l_run)) * kXLn2 : -INFINITY;
      ++tcnt;
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

}  // namespace dit
