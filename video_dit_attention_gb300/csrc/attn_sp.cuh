// Attention kernel with P staged in shared memory: the plain, workspace-RoPE (with the q/k
// RMSNorm, fixed-m, sharded-keys variants) and FP8 modes. Included by attn_fwd.cu inside its namespace, after the helpers it
// uses (KParams, WsParams, Item, decode_item, write_empty_tile,
// rotate_rows_fp16, warp_wait, group_wait, sts128).
//
// Same mathematics, work items, persistence and warp roles as attn_fwd_kernel. What changes
// is where P lives. There, P_t,j is written as bf16 over S_t,j in TMEM, so S_t,j+1 can only
// be computed after P_t,j V_j has read P_t,j. Each query tile then runs a serial chain per
// key tile: softmax, then the PV product, then the next S product. Here each softmax thread
// writes its P row into shared memory (128-byte swizzle, the K-major A operand of an SS
// MMA). As soon as the softmax has loaded S_t,j into registers it releases the TMEM columns
// (s_free), and S_t,j+1 is computed while the softmax is still exponentiating; a softmax
// only waits for work that was issued a full step earlier.
// The MMAs come from two threads: warp 12 issues every S_t = Q_t K_j^T, warp 13 every
// O_t += P_t V_j. A single issuing thread spends about 60 cycles per tcgen05.mma plus its
// commits and barrier polls, close to the 64 cycles a 128 x 128 x 16 product takes, and left
// the tensor core idle between groups; two issuers overlap that cost. They touch disjoint
// TMEM columns and every commit covers only its own thread's MMAs, so they need no ordering
// between them beyond the barriers below.
// Workspace modes: warps 14-15 rotate the first item's Q tiles; each later item's tile t is
// rotated by softmax warpgroup t once it has written its last P_t of the item before.
// Synchronisation per query-tile slot t (all waits bounded):
//   s_full[t]  S_t,j computed (commit)          -> softmax t
//   s_free[t]  S_t,j loaded into registers       -> issuer may overwrite S_t (4 warp arrivals)
//   p_full[t]  P_t,j stored in shared memory     -> issuer may run P_t,j V_j (4 warp arrivals)
//   pv_done[t] P_t,j V_j complete (commit)       -> softmax may rescale O_t / overwrite P_t;
//                                                    the epilogue may read O_t
//   o_free[t]  O_t read out by the epilogue      -> the next item's first PV may overwrite it
//   q_ready    (workspace modes) Q rotated       -> S products of the item (8 warp arrivals)
// Shared memory at D = 128: Q0, Q1 (64 KB), a ring of three K/V slots (96 KB), P0, P1
// (64 KB). K and V share the ring, K one tile ahead of V, which gives a K load about two key
// steps and a V load about one to land (two K and one V stage would leave V a fraction).

// Fixed-m softmax: a warp keeps its rows' bounds m as the maximum when every valid row has
// 2 m <= kFixedMSpanLog2 (log2 units). The bound is widened by kFixedMSlack to cover the
// fp16 rounding of the rotated q and k (2^-11 each) and the fp32 norms.
constexpr float kFixedMSpanLog2 = 64.f;

// FP8 softmax: the running maximum may lag by up to kFp8RescaleThreshold (log2 units), so
// p <= 4, and P is stored as e4m3(kFp8PScale * p) with kFp8PScale = 448 / 4 (no saturation).
constexpr float kFp8RescaleThreshold = 2.f;
constexpr float kFp8PScale = 112.f;
constexpr float kFixedMSlack = 1.f + 1.f / 256.f;

// Shared-memory layout. bf16 modes: K/V tiles of 128 rows x D bf16 (D / 64 chunks of 128-byte
// swizzled rows), P of 128 x 128 bf16 in two chunks. FP8 mode (D = 128): every operand tile
// is 128 rows x 128 bytes (one chunk), so the ring has six slots, and O is staged for its
// bf16 store in an area of its own.
template <int D, bool kFp8 = false>
struct CfgSp {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kSub = D * kElem / 128;          // 128-byte chunks per operand row
  static constexpr int kTileBytes = 128 * D * kElem;
  static constexpr int kRing = (kFp8 || D != 128) ? 6 : 3;   // K/V ring slots
  static constexpr int kPBytes = 128 * 128 * kElem;     // P tile: 128 query rows x 128 keys
  static constexpr int kOBytes = kFp8 ? 128 * D * 2 : 0;   // FP8: bf16 O staging per query tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffR = kOffQ + 2 * kTileBytes;
  static constexpr int kOffP = kOffR + kRing * kTileBytes;
  static constexpr int kOffO = kOffP + 2 * kPBytes;
  static constexpr int kOffBar = kOffO + 2 * kOBytes;
  static constexpr int kSmemBytes = kOffBar + 512 + 1024;  // barriers + alignment slack
};

struct BarsSp {
  uint64_t q_full, q_ready, q_empty;
  uint64_t r_full[6], r_empty[6];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2], o_free[2];
  uint64_t drain[2];
  uint32_t tmem_base;
  int abort;
  int aux_go;
};

// The key tiles a CTA visits, flattened over its items: tile g (g = 0 .. G-1) needs K_g for
// the S products and V_g for the PV products. One ring of shared-memory slots holds both,
// loaded in the order K_0, K_1, V_0, K_2, V_1, ..., K_G-1, V_G-2, V_G-1 (K one tile ahead of
// V, as S_g+1 is computed before P_g V_g). Load number n goes to slot n % kRing.
__device__ __forceinline__ int ring_load_k(int g) { return g == 0 ? 0 : 2 * g - 1; }
__device__ __forceinline__ int ring_load_v(int g, int G) { return g == G - 1 ? 2 * G - 1 : 2 * g + 2; }

template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    attn_sp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const KParams p, const WsParams ws,
                   const __grid_constant__ ShardArg<kMode> sh) {
  static_assert(kMode == kModePlain || kMode == kModeFp8 || is_ws_mode(kMode), "mode");
  constexpr bool kFp8 = kMode == kModeFp8;
  static_assert(!kFp8 || D == 128, "the FP8 path is built for D = 128");
  constexpr bool kWs = is_ws_mode(kMode), kNorm = kMode == kModeRopeWsNorm;
  constexpr bool kFixedM = kMode == kModeRopeWsFixedM;
  constexpr bool kShard = kMode == kModeRopeWsSharded;
  using C = CfgSp<D, kFp8>;
  constexpr int R = C::kRing;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t s_base = smem_u32(smem);
  const uint32_t sQ = s_base + C::kOffQ;
  const uint32_t sR = s_base + C::kOffR;
  const uint32_t sP = s_base + C::kOffP;
  const uint32_t sO = s_base + C::kOffO;   // FP8: O staging (the bf16 modes stage O in P)
  BarsSp* bars = reinterpret_cast<BarsSp*>(smem + C::kOffBar);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &bars->abort;
  unsigned int* status = &g_dit_status;
  const uint32_t b_q_full = smem_u32(&bars->q_full), b_q_empty = smem_u32(&bars->q_empty);
  const uint32_t b_q_ready = smem_u32(&bars->q_ready);

  if (tid == 0) {
    bars->abort = 0;
    mbar_init(b_q_full, 1);
    mbar_init(b_q_ready, kWs ? 8 : 1);   // workspace modes: the 8 softmax warps
    mbar_init(b_q_empty, 1);
    for (int s = 0; s < R; ++s) {
      mbar_init(smem_u32(&bars->r_full[s]), 1);
      mbar_init(smem_u32(&bars->r_empty[s]), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&bars->s_full[t]), 1);
      mbar_init(smem_u32(&bars->s_free[t]), 4);
      mbar_init(smem_u32(&bars->p_full[t]), 4);
      mbar_init(smem_u32(&bars->pv_done[t]), 1);
      mbar_init(smem_u32(&bars->o_free[t]), 4);
    }
    mbar_init(smem_u32(&bars->drain[0]), 1);
    mbar_init(smem_u32(&bars->drain[1]), 1);
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
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = bars->tmem_base;
  const int it0 = blockIdx.x, it_step = gridDim.x;
  // Work item `it` (the sharded mode decodes its key chunk too).
  auto dec = [&](int it) -> Item {
    if constexpr (kShard) return decode_item_sh(p, sh, it);
    else return decode_item<kMode>(p, it);
  };
  // TMA maps of an item's keys and values (per key chunk in the sharded mode).
  auto kmap = [&](const Item& w) -> const CUtensorMap* {
    if constexpr (kShard) return &sh.km[w.chunk];
    else return &tm_k;
  };
  auto vmap = [&](const Item& w) -> const CUtensorMap* {
    if constexpr (kShard) return &sh.vm[w.chunk];
    else return &tm_v;
  };
  // First item at or after `it` (in this CTA's sequence) that has work.
  auto first_live = [&](int it) -> int {
    while (it < p.n_items && dec(it).n_live == 0) it += it_step;
    return it;
  };
  // Workspace mode: items whose Q was loaded and rotated before the roles start (0 or 1).
  int pre_q = 0;
  if (kWs) {
    // ------------------------------------------------- rotate k once; the first Q meanwhile
    // Warps 0-13 rotate this CTA's share of the k rows. The rotated rows are published through
    // a counter: each thread's generic-proxy stores are fenced against the async proxy (the
    // TMA loads that read them), then the CTA counts itself in with a device-scope release;
    // only the K/V producer waits for the count. Meanwhile warps 14-15 rotate the first
    // item's Q tiles in shared memory (the softmax warpgroups rotate later ones).
    const int fit = first_live(it0);
    Item fw{};
    if (fit < p.n_items) {
      fw = dec(fit);
      pre_q = 1;
    }
    if (pre_q && tid == 0) {
      mbar_arrive_expect_tx(b_q_full, fw.n_live * C::kTileBytes);
      for (int t = 0; t < fw.n_live; ++t)
#pragma unroll
        for (int c = 0; c < C::kSub; ++c)
          tma_load_4d(sQ + t * C::kTileBytes + c * 16384, &tm_q, b_q_full, c * 64, fw.h,
                      fw.q0 + 128 * t, fw.b);
    }
    constexpr int kRotK = kThreads - 64;   // threads of warps 0-13
    if (warp >= 14) {
      const int at = tid - kRotK;
      if (pre_q && group_wait<64>(b_q_full, 0, abort_flag, status, kStatusTimeoutRope, &bars->aux_go, at)) {
        for (int t = 0; t < fw.n_live; ++t) {
          const size_t row0 = static_cast<size_t>(fw.q0 + 128 * t) * (D / 2);
          if (kNorm)
            rotate_tile_smem_norm<D, 64>(sQ + t * C::kTileBytes, p.cos_q + row0, p.sin_q + row0, ws.norm_q,
                                         ws.norm_eps, at);
          else if (kFixedM)
            rotate_tile_smem_sq<D, 64>(sQ + t * C::kTileBytes, p.cos_q + row0, p.sin_q + row0, at,
                                       ws.qn + (static_cast<size_t>(fw.b) * p.Sq + fw.q0 + 128 * t) * p.H + fw.h, p.H);
          else
            rotate_tile_smem<D, 64>(sQ + t * C::kTileBytes, p.cos_q + row0, p.sin_q + row0, at);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 64);
        if (at == 0)
          for (int x = 0; x < 8; ++x) mbar_arrive(b_q_ready);   // stands in for the 8 softmax warps
      }
    } else {
      // Fixed-m mode: the largest squared key norm of each (b, h) among this CTA's rows is
      // gathered in the (still unused) K/V ring, then merged into the workspace below.
      unsigned int* kmax_s = reinterpret_cast<unsigned int*>(smem + C::kOffR);
      if (kFixedM) {
        for (int i = tid; i < ws.B * p.H; i += kRotK) kmax_s[i] = 0u;
        named_bar_sync(2, kRotK);
      }
      if (kNorm)
        rotate_rows_fp16_norm<D>(ws.k_raw, ws.k_rot, p.cos_k, p.sin_k, ws.norm_k, ws.norm_eps, ws.B, p.Skv,
                                 p.kv_valid, p.H, blockIdx.x * kRotK + tid, gridDim.x * kRotK);
      else if (kFixedM)
        rotate_rows_fp16_kmax<D>(ws.k_raw, ws.k_rot, p.cos_k, p.sin_k, ws.B, p.Skv, p.kv_valid, p.H,
                                 blockIdx.x * kRotK + tid, gridDim.x * kRotK, kmax_s);
      else if constexpr (kShard) {
        for (int c = 0; c < sh.n_chunks; ++c)
          rotate_rows_fp16<D>(sh.c[c].k_raw, sh.c[c].k_rot, sh.c[c].cos_k, sh.c[c].sin_k, ws.B, sh.c[c].S_rows,
                              sh.c[c].valid, p.H, blockIdx.x * kRotK + tid, gridDim.x * kRotK);
      } else
        rotate_rows_fp16<D>(ws.k_raw, ws.k_rot, p.cos_k, p.sin_k, ws.B, p.Skv, p.kv_valid, p.H,
                            blockIdx.x * kRotK + tid, gridDim.x * kRotK);
      fence_proxy_async_all();
    }
    __syncthreads();
    if (kFixedM) {
      // Merge this CTA's maxima before it counts itself in: the release below covers them.
      if (warp < 14) {
        const unsigned int* kmax_s = reinterpret_cast<const unsigned int*>(smem + C::kOffR);
        for (int i = tid; i < ws.B * p.H; i += kRotK)
          if (kmax_s[i] != 0u) atomicMax(ws.kmax + i, kmax_s[i]);
      }
      __syncthreads();
    }
    if (tid == 0) {
      __threadfence();
      atomicAdd(ws.rotated, 1u);
    }
  }
  // Workspace mode: a producer waits, before its first load, until every CTA has counted in
  // its share of the rotation (`ready` remembers that it has).
  auto wait_rotated = [&](bool& ready) -> bool {
    if (!kWs || ready) return true;
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_gpu(ws.rotated) < gridDim.x) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > wait_limit_ns()) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeoutGrid);
        return false;
      }
      __nanosleep(128);
    }
    fence_proxy_async_all();   // the TMA loads that follow read what the other CTAs wrote
    ready = true;
    return true;
  };
  // Fixed-m mode: a warp waits until every CTA has counted in its rotation (and with it its
  // key-norm maxima), with a device-scope acquire.
  auto wait_grid = [&]() -> bool {
    int ok = 1;
    if (lane == 0) {
      const uint64_t t0 = globaltimer_ns();
      while (ld_acquire_gpu(ws.rotated) < gridDim.x) {
        if (*abort_flag) { ok = 0; break; }
        if (globaltimer_ns() - t0 > wait_limit_ns()) {
          *abort_flag = 1;
          atomicOr(status, kStatusTimeoutGrid);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __syncwarp();
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
  };
  // G: key tiles over all of this CTA's items.
  auto count_tiles = [&]() -> int {
    int G = 0;
    for (int it = it0; it < p.n_items; it += it_step) {
      const Item w = dec(it);
      if (w.n_live > 0) G += w.n_kv;
    }
    return G;
  };

  // Two MMA issuers, one thread each: S products (warp 12) and PV products (warp 13). They
  // share no TMEM columns and each commit covers only the issuing thread's own MMAs, so they
  // need no ordering between them; two issuers keep the tensor core fed where one thread's
  // per-instruction issue cost (plus commits and waits) would leave it idle between groups.
  auto wait_bar = [&](uint32_t bar, int phase) -> bool {
    if (!bounded_wait(bar, phase & 1, abort_flag, status, kStatusTimeoutMma)) return false;
    tc_fence_after_sync();
    return true;
  };
  auto s_issuer = [&]() {
    // ------------------------------------------------------------ S_t = Q_t K_g^T
    // bf16 (or fp16 when q/k were rotated) operands, or e4m3 in the FP8 path (format 0 in
    // both cases: f16 for kind::f16, e4m3 for kind::f8f6f4).
    constexpr uint32_t kIdS = idesc_f16kind_f32(128, 128, !kWs && !kFp8, false, false);
    constexpr int kKStep = kFp8 ? 32 : 16;   // K elements per MMA (32 bytes of each row)
    int g0 = 0, q_cnt = 0, ns0 = 0, ns1 = 0;
    bool ok = true;
    for (int it = it0; ok && it < p.n_items; it += it_step) {
      const Item w = dec(it);
      if (w.n_live == 0) continue;
      // Workspace modes: Q is used once it is rotated in shared memory (q_ready).
      if (!(ok = wait_bar(kWs ? b_q_ready : b_q_full, q_cnt))) break;
      for (int j = 0; ok && j < w.n_kv; ++j) {
        const int g = g0 + j;
        const int n = ring_load_k(g), slot = n % R;
        if (!(ok = wait_bar(smem_u32(&bars->r_full[slot]), n / R))) break;
        const uint64_t db = smem_desc_sw128(sR + slot * C::kTileBytes, 16, 1024);
        for (int t = 0; t < w.n_live; ++t) {
          // S_t may be overwritten once the softmax has taken the previous S_t out of TMEM.
          const int ns = t ? ns1 : ns0;
          if (ns > 0 && !(ok = wait_bar(smem_u32(&bars->s_free[t]), ns - 1))) break;
          const uint64_t da = smem_desc_sw128(sQ + t * C::kTileBytes, 16, 1024);
          const uint32_t d = tbase + t * 128;
#pragma unroll
          for (int kk = 0; kk < D / kKStep; ++kk) {
            const uint64_t off = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
            if constexpr (kFp8)
              mma_e4m3_ss(d, da + off, db + off, kIdS, kk > 0);
            else
              mma_bf16_ss(d, da + off, db + off, kIdS, kk > 0);
          }
          mma_commit(smem_u32(&bars->s_full[t]));
          if (t) ++ns1; else ++ns0;
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->r_empty[slot]));
      }
      if (!ok) break;
      mma_commit(b_q_empty);   // every S product of the item is issued: Q may be reloaded
      g0 += w.n_kv;
      ++q_cnt;
    }
    // Wait for every MMA this thread issued before TMEM and shared memory are released. On
    // the normal path the softmax has already waited for each of them; after an abort some
    // may still be running when the other roles reach the final barrier.
    mma_commit(smem_u32(&bars->drain[0]));
    drain_wait(smem_u32(&bars->drain[0]), 0, status);
  };
  auto pv_issuer = [&]() {
    // ------------------------------------------------------------ O_t (+)= P_t V_g
    // bf16: A = P (K-major), B = V tile (MN-major). FP8: both e4m3 and K-major (V transposed).
    constexpr uint32_t kIdO = kFp8 ? idesc_f16kind_f32(128, D, false, false, false) : idesc_bf16_f32(128, D, false, true);
    int g0 = 0, np0 = 0, np1 = 0, epi0 = 0, epi1 = 0;
    const int G = count_tiles();
    bool ok = true;
    for (int it = it0; ok && it < p.n_items; it += it_step) {
      const Item w = dec(it);
      if (w.n_live == 0) continue;
      for (int j = 0; ok && j < w.n_kv; ++j) {
        const int g = g0 + j, n = ring_load_v(g, G), slot = n % R;
        if (!(ok = wait_bar(smem_u32(&bars->r_full[slot]), n / R))) break;
        const uint64_t db = smem_desc_sw128(sR + slot * C::kTileBytes, kFp8 ? 16 : 16384, 1024);
        for (int t = 0; t < w.n_live; ++t) {
          const int np = t ? np1 : np0, epi = t ? epi1 : epi0;
          if (!(ok = wait_bar(smem_u32(&bars->p_full[t]), np))) break;
          // The first key tile of an item overwrites O_t, once the epilogue of the slot's
          // previous item has read it.
          if (j == 0 && epi > 0 && !(ok = wait_bar(smem_u32(&bars->o_free[t]), epi - 1))) break;
          const uint64_t da = smem_desc_sw128(sP + t * C::kPBytes, 16, 1024);
          const uint32_t d = tbase + 256 + t * 128;
          if constexpr (kFp8) {
            // 128 keys in four K steps of 32 bytes, within the one 128-byte row of P and of V^T.
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_e4m3_ss(d, da + static_cast<uint64_t>(kk * 2), db + static_cast<uint64_t>(kk * 2), kIdO,
                          (j > 0 || kk > 0) ? 1u : 0u);
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t offa = ((kk / 4) * 16384 + (kk % 4) * 32) >> 4;
              mma_bf16_ss(d, da + offa, db + static_cast<uint64_t>(kk * 2048 >> 4), kIdO,
                          (j > 0 || kk > 0) ? 1u : 0u);
            }
          }
          mma_commit(smem_u32(&bars->pv_done[t]));
          if (t) ++np1; else ++np0;
        }
        if (!ok) break;
        mma_commit(smem_u32(&bars->r_empty[slot]));
      }
      if (!ok) break;
      ++epi0;
      if (w.n_live == 2) ++epi1;
      g0 += w.n_kv;
    }
    mma_commit(smem_u32(&bars->drain[1]));   // as for the S issuer
    drain_wait(smem_u32(&bars->drain[1]), 0, status);
  };

  {
  if (warp < 4) {
    regs_dec<40>();
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------------------ producer: Q
      int q_cnt = pre_q;
      bool skip = pre_q != 0;   // the first item's Q is already loaded
      bool ok = true;
      for (int it = it0; ok && it < p.n_items; it += it_step) {
        const Item w = dec(it);
        if (w.n_live == 0) continue;
        if (skip) {
          skip = false;
          continue;
        }
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
      }
      // The last Q load has landed before the CTA exits (it has already on the normal path).
      if (q_cnt > 0) drain_wait(b_q_full, (q_cnt - 1) & 1, status);
    } else if (warp == 2 && lane == 0) {
      // ------------------------------------------------------------ producer: K/V ring
      const int G = count_tiles();
      int n = 0;   // loads issued
      bool ok = true;
      auto load = [&](const CUtensorMap* map, const Item& w, int j) -> bool {
        const int slot = n % R, use = n / R;
        if (use > 0 && !bounded_wait(smem_u32(&bars->r_empty[slot]), (use - 1) & 1, abort_flag,
                                     status, kStatusTimeoutLoad))
          return false;
#ifdef DIT_TEST_HOOKS
        if (n == g_dit_test_skip_load) {   // test build only: counted, never issued
          ++n;
          return true;
        }
#endif
        const uint32_t bar = smem_u32(&bars->r_full[slot]);
        mbar_arrive_expect_tx(bar, C::kTileBytes);
        if (kFp8 && map == &tm_v) {
          // FP8 V is stored transposed, [B, H, D, S]: the tile is D rows of 128 keys.
          tma_load_4d(sR + slot * C::kTileBytes, map, bar, j * 128, 0, w.h, w.b);
        } else {
#pragma unroll
          for (int c = 0; c < C::kSub; ++c)
            tma_load_4d(sR + slot * C::kTileBytes + c * 16384, map, bar, c * 64, w.h, j * 128, w.b);
        }
        ++n;
        return true;
      };
      // Separate cursors (item, tile) for the K stream and the V stream.
      int kit = first_live(it0), kj = 0, vit = kit, vj = 0;
      bool k_ready = false;
      Item kw{}, vw{};
      if (kit < p.n_items) kw = vw = dec(kit);
      auto load_next_k = [&]() -> bool {
        if (kj == (kw.n_kv > kPrefetchLead ? kw.n_kv - kPrefetchLead : 0)) {
          // Warm L2 with the next item's Q tiles and first K/V tiles.
          const int nit = first_live(kit + it_step);
          if (nit < p.n_items) {
            const Item nw = dec(nit);
            for (int t = 0; t < nw.n_live; ++t)
#pragma unroll
              for (int c = 0; c < C::kSub; ++c)
                tma_prefetch_l2_4d(&tm_q, c * 64, nw.h, nw.q0 + 128 * t, nw.b);
            for (int jj = 0; jj < nw.n_kv && jj < kPrefetchKV; ++jj)
#pragma unroll
              for (int c = 0; c < C::kSub; ++c) {
                tma_prefetch_l2_4d(kmap(nw), c * 64, nw.h, jj * 128, nw.b);
                if (kFp8)
                  tma_prefetch_l2_4d(&tm_v, jj * 128, 0, nw.h, nw.b);
                else
                  tma_prefetch_l2_4d(vmap(nw), c * 64, nw.h, jj * 128, nw.b);
              }
          }
        }
        if (!wait_rotated(k_ready) || !load(kmap(kw), kw, kj)) return false;
        if (++kj == kw.n_kv) {
          kj = 0;
          kit = first_live(kit + it_step);
          if (kit < p.n_items) kw = dec(kit);
        }
        return true;
      };
      auto load_next_v = [&]() -> bool {
        if (!load(vmap(vw), vw, vj)) return false;
        if (++vj == vw.n_kv) {
          vj = 0;
          vit = first_live(vit + it_step);
          if (vit < p.n_items) vw = dec(vit);
        }
        return true;
      };
      if (G > 0) ok = load_next_k();
      for (int g = 0; ok && g < G; ++g) {
        if (g + 1 < G && !(ok = load_next_k())) break;
        ok = load_next_v();
      }
      {
        // Let the copies still in flight land before the CTA releases its shared memory (on the
        // normal path every load has been consumed, so these waits return at once).
        for (int x = n - R > 0 ? n - R : 0; x < n; ++x) {
#ifdef DIT_TEST_HOOKS
          if (x == g_dit_test_skip_load) continue;   // never issued: nothing to land
#endif
          drain_wait(smem_u32(&bars->r_full[x % R]), (x / R) & 1, status);
        }
      }
    }
  } else if (warp < 12) {
    regs_inc<200>();
    // -------------------------------------------------------------- softmax + epilogue
    const int t = (warp - 4) >> 2;                   // query-tile slot of this warpgroup
    const int r = (tid - 128) & 127;                 // row within the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + t * 128;
    const uint32_t tO = tbase + lane_off + 256 + t * 128;
    // This thread's P row: 16-byte unit x of 64-key chunk c sits at c * 16384 + r * 128 +
    // ((x ^ (r & 7)) * 16), the 128-byte swizzle the MMA's K-major descriptor reads.
    const uint32_t p_row = sP + t * C::kPBytes + r * 128;
    const uint32_t p_sw = static_cast<uint32_t>(r & 7);
    const uint32_t b_s_full = smem_u32(&bars->s_full[t]), b_s_free = smem_u32(&bars->s_free[t]);
    const uint32_t b_p_full = smem_u32(&bars->p_full[t]), b_pv_done = smem_u32(&bars->pv_done[t]);
    const float sl2 = p.scale_log2;
    int sc = 0;   // S_t tiles consumed so far (= P_t tiles produced = PV_t products issued)
    int qi = 0;   // live items seen so far
    // Workspace modes: once its last P_t of live item qi is out, each softmax warpgroup
    // rotates (and, per mode, normalises or takes the row norms of) its tile t of the next
    // live item's Q in shared memory, and each warp arrives on q_ready, so that the next
    // item's S products start while this item's epilogue runs.
    // (Warps 14-15 alone took about 16K cycles per item for the whole Q; the 256 softmax
    // threads take the tile they will use, with nothing else to do until the last P_t V.)
    auto rotate_next = [&](int it_cur) -> bool {
      if constexpr (kWs) {
        const int nit = first_live(it_cur + it_step);
        if (nit >= p.n_items) return true;
        const Item nw = dec(nit);
        if (!warp_wait(b_q_full, (qi + 1) & 1, abort_flag, status, kStatusTimeoutRope)) return false;
        if (t < nw.n_live) {
          const size_t row0 = static_cast<size_t>(nw.q0 + 128 * t) * (D / 2);
          // Unroll depths as measured best per mode (code placement: with one unit in flight
          // the norm and fixed-m modes ran 13-15 % slower at 720p too).
          if constexpr (kNorm)
            rotate_tile_smem_norm<D, 128, 4>(sQ + t * C::kTileBytes, p.cos_q + row0, p.sin_q + row0, ws.norm_q,
                                             ws.norm_eps, r);
          else if constexpr (kFixedM)
            rotate_tile_smem_sq<D, 128, 2>(sQ + t * C::kTileBytes, p.cos_q + row0, p.sin_q + row0, r,
                                           ws.qn + (static_cast<size_t>(nw.b) * p.Sq + nw.q0 + 128 * t) * p.H + nw.h,
                                           p.H);
          else
            rotate_tile_smem<D, 128, 4>(sQ + t * C::kTileBytes, p.cos_q + row0, p.sin_q + row0, r);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_q_ready);
      }
      return true;
    };
    bool ok = true;
    for (int it = it0; ok && it < p.n_items; it += it_step) {
      const Item w = dec(it);
      if (t >= w.n_live) {
        if (t == 0 || w.has1) {
          if constexpr (kShard)   // the partial (O, LSE) of the item's key chunk
            write_empty_tile<D>(p, p.out + w.chunk * sh.po_stride, p.lse + w.chunk * sh.pl_stride, w.b, w.h,
                                w.q0 + 128 * t, r, 128);
          else
            write_empty_tile<D>(p, p.out, p.lse, w.b, w.h, w.q0 + 128 * t, r, 128);
        }
        if (w.n_live > 0) {
          if (!(ok = rotate_next(it))) break;
          ++qi;
        }
        continue;
      }
      const int n_kv = w.n_kv, kv_valid = w.kv_valid;
      float m_used = -INFINITY, l = 0.f;
      // FP8: scores come out of the MMA in units of the q tile's and the head's k scales.
      const float sl2e = kFp8 ? sl2 * ws.f8_sq[(w.b * p.H + w.h) * ws.f8_nt_q + (w.q0 >> 7) + t] *
                                    ws.f8_sk[w.b * p.H + w.h]
                              : sl2;
      bool fixed = false;   // fixed-m mode: this warp's 32 rows skip the running maximum
      if constexpr (kFixedM) {
        // Row bound m = scale * |q_row| * max_j |k_j| (log2 units here): no valid score of the
        // row exceeds it (Cauchy-Schwarz; the rotation keeps norms). The warp keeps m fixed,
        // with no maximum and no rescaling, when every valid row has 2 m <= 64: then the
        // row's largest term exp2(s - m) is at least 2^-64. Pad rows (zero q, bound 0) and
        // pad keys (never in the maximum) cannot move a warp onto the online path.
        // The q row norms of this item were written before q_ready's phase qi completed (by
        // warps 14-15 for the first item, else by this warpgroup in rotate_next); the wait's
        // acquire makes them visible. The phase after it needs this warp's own arrival.
        if (!(ok = warp_wait(b_q_ready, qi & 1, abort_flag, status, kStatusTimeoutSoftmax))) break;
        if (qi == 0 && !(ok = wait_grid())) break;
        const int qrow0 = w.q0 + 128 * t + r;
        const float kq = __uint_as_float(ws.kmax[w.b * p.H + w.h]);
        const float qn = ws.qn[(static_cast<size_t>(w.b) * p.Sq + qrow0) * p.H + w.h];
        const float mb = sl2 * sqrtf(qn * kq) * kFixedMSlack;
        fixed = __all_sync(0xffffffffu, qrow0 >= p.q_valid || mb <= 0.5f * kFixedMSpanLog2);
        if (fixed)
          m_used = mb;
        else if (lane == 0 && ws.n_online != nullptr)
          atomicAdd(ws.n_online, 1u);
      }
      for (int j = 0; j < n_kv; ++j, ++sc) {
        if (!warp_wait(b_s_full, sc & 1, abort_flag, status, kStatusTimeoutSoftmax)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32_nowait(tS + c * 32, sr[c]);
        tmem_ld_wait_tied(sr[0]);
        tmem_reg_tie(sr[1]);
        tmem_reg_tie(sr[2]);
        tmem_reg_tie(sr[3]);
        // S_t is in registers: the issuer may compute S_t,j+1 into the same columns.
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(b_s_free);
        const int nv = min(128, kv_valid - j * 128);   // valid keys in this tile (>= 1)
        if (nv < 128) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i >= nv) sr[c][i] = 0xff800000u;
        }
        float mt = -INFINITY;   // a fixed warp keeps m_used: no rescale, alpha = 1
        if (!fixed) {
          float mx4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            mx4[c] = fmaxf(__uint_as_float(sr[c][0]), __uint_as_float(sr[c][1]));
#pragma unroll
            for (int i = 2; i < 32; i += 2)
              mx4[c] = fmax3(mx4[c], __uint_as_float(sr[c][i]), __uint_as_float(sr[c][i + 1]));
          }
          const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
          mt = mx * sl2e;
        }
        // FP8 lets the maximum lag by at most 2 (p <= 4), so that 112 p fits e4m3.
        const bool resc = mt > m_used + (kFp8 ? kFp8RescaleThreshold : kRescaleThreshold);
        const float m_new = resc ? mt : m_used;
        const float alpha = ex2_approx(m_used - m_new);   // 1 if kept; 0 on the first tile
        if constexpr (kFp8) {
          // FP8: P_t,j is computed into registers first; only its store into the P_t buffer (and
          // the rescale of O_t) waits for P_t,j-1 V_j-1, so the exponentials overlap that
          // product (861 -> 1009 TFLOP/s at Wan 480; the bf16 modes measured 10 % slower this way).
          const float neg_m = -m_new;
          float l4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) l4[k] = 0.f;
          uint32_t pk[8][4];   // 16 keys per c: four e4m3 quads
#pragma unroll
          for (int c = 0; c < 8; ++c) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float x0, x1;
              fma2_bc(x0, x1, __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i]),
                      __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i + 1]), sl2e, neg_m);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              add2(l4[2 * (i & 1)], l4[2 * (i & 1) + 1], p0, p1);
              const uint32_t e = pack_e4m3x2(kFp8PScale * p0, kFp8PScale * p1);
              if (i & 1)
                pk[c][i >> 1] |= e << 16;
              else
                pk[c][i >> 1] = e;
            }
          }
          if (j > 0) {
            // P_t,j-1 V_j-1 must be complete before O_t is rescaled and before P_t is rewritten.
            if (!warp_wait(b_pv_done, (sc - 1) & 1, abort_flag, status, kStatusTimeoutSoftmax)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(tO + c * 32, orr);
#pragma unroll
                for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                tmem_st32(tO + c * 32, orr);
              }
            }
          }
          m_used = m_new;
#pragma unroll
          for (int c = 0; c < 8; ++c)   // 16 e4m3 keys: one 16-byte unit of the single 128-byte P row
            sts128(p_row + ((static_cast<uint32_t>(c) ^ p_sw) << 4), make_uint4(pk[c][0], pk[c][1], pk[c][2], pk[c][3]));
          l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
        } else {
          if (j > 0) {
            // P_t,j-1 V_j-1 must be complete before O_t is rescaled and before P_t is rewritten.
            if (!warp_wait(b_pv_done, (sc - 1) & 1, abort_flag, status, kStatusTimeoutSoftmax)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
              for (int c = 0; c < D / 32; ++c) {
                uint32_t orr[32];
                tmem_ld32(tO + c * 32, orr);
#pragma unroll
                for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
                tmem_st32(tO + c * 32, orr);
              }
            }
          }
          m_used = m_new;
          const float neg_m = -m_used;
          float l4[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) l4[k] = 0.f;
#pragma unroll
          for (int c = 0; c < 8; ++c) {           // 16 keys at a time: two 16-byte units (bf16)
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float x0, x1;
              fma2_bc(x0, x1, __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i]),
                      __uint_as_float(sr[c >> 1][(c & 1) * 16 + 2 * i + 1]), sl2e, neg_m);
              const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
              add2(l4[2 * (i & 1)], l4[2 * (i & 1) + 1], p0, p1);
              pk[i] = pack_bf16x2(p0, p1);
            }
            const uint32_t chunk = static_cast<uint32_t>(c >> 2) * 16384u;
            const uint32_t x0 = static_cast<uint32_t>((2 * c) & 7), x1 = static_cast<uint32_t>((2 * c + 1) & 7);
            sts128(p_row + chunk + ((x0 ^ p_sw) << 4), make_uint4(pk[0], pk[1], pk[2], pk[3]));
            sts128(p_row + chunk + ((x1 ^ p_sw) << 4), make_uint4(pk[4], pk[5], pk[6], pk[7]));
          }
          l = l * alpha + ((l4[0] + l4[1]) + (l4[2] + l4[3]));
        }
        fence_proxy_async_smem();   // P (generic stores) before the MMA's async-proxy reads
        tc_fence_before_sync();     // and the O rescale (tcgen05.st) before the next PV
        __syncwarp();
        if (lane == 0) mbar_arrive(b_p_full);   // one arrival per warp
      }
      if (!ok) break;
      if (!(ok = rotate_next(it))) break;
      // Epilogue. Wait for the last P_t V of this item and take O_t out of TMEM, which then
      // belongs to the next item (its first P_t V may start), then normalise and store.
      if (!warp_wait(b_pv_done, (sc - 1) & 1, abort_flag, status, kStatusTimeoutSoftmax)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int qrow = w.q0 + 128 * t + r;
      const bool valid_row = qrow < p.q_valid;
      // FP8: O came out in units of kFp8PScale (P) and of the head's v scale.
      const float inv_l = kFp8 ? ws.f8_sv[w.b * p.H + w.h] / (kFp8PScale * l) : 1.f / l;
      const uint32_t st_row = kFp8 ? sO + t * C::kOBytes + r * 128 : p_row;   // staging row
      // The warp stages its 32 normalised rows in its own rows of the P_t buffer, in the P
      // layout (row r, 16-byte unit x of 64-column chunk c at c * 16384 + r * 128 +
      // ((x ^ (r & 7)) * 16)), so no other warp reads or writes those bytes. It then writes
      // them out as whole rows, 16 bytes per lane, instead of 32 scattered pieces per row.
      // O_t is read 32 columns at a time and released once the last piece is in registers.
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tmem_ld32(tO + c * 32, orr);
        if (c == D / 32 - 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->o_free[t]));
        }
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {         // columns 32c + 8q4 .. + 7: 16-byte unit 4c + q4
          const int u = 4 * c + q4;
          uint4 o = make_uint4(0, 0, 0, 0);
          if (valid_row) {
            const uint32_t* f = &orr[8 * q4];
            o.x = pack_bf16x2(__uint_as_float(f[0]) * inv_l, __uint_as_float(f[1]) * inv_l);
            o.y = pack_bf16x2(__uint_as_float(f[2]) * inv_l, __uint_as_float(f[3]) * inv_l);
            o.z = pack_bf16x2(__uint_as_float(f[4]) * inv_l, __uint_as_float(f[5]) * inv_l);
            o.w = pack_bf16x2(__uint_as_float(f[6]) * inv_l, __uint_as_float(f[7]) * inv_l);
          }
          sts128(st_row + static_cast<uint32_t>(u >> 3) * 16384u + ((static_cast<uint32_t>(u & 7) ^ p_sw) << 4), o);
        }
      }
      __syncwarp();
      {
        // 16 bytes per lane: D / 8 lanes cover one row, so one store instruction writes
        // 32 / (D / 8) whole rows.
        constexpr int kLPR = D / 8, kRPI = 32 / kLPR;
        const int r0 = r & ~31, lu = lane % kLPR, lr = lane / kLPR;   // r0: first row of this warp
        const uint32_t chunk = static_cast<uint32_t>(lu >> 3) * 16384u, unit = static_cast<uint32_t>(lu & 7);
        // Stores in flight per lane: more helps short items and plain
        // attention slightly; the workspace mode measured best at one.
        constexpr int kStoreUnroll = kWs ? 1 : 4;
#pragma unroll kStoreUnroll
        for (int i = 0; i < 32 / kRPI; ++i) {
          const int rr = r0 + i * kRPI + lr;
          const uint32_t src = (kFp8 ? sO + t * C::kOBytes : sP + t * C::kPBytes) + chunk + static_cast<uint32_t>(rr) * 128u +
                               ((unit ^ static_cast<uint32_t>(rr & 7)) << 4);
          uint16_t* dst = p.out + ((static_cast<size_t>(w.b) * p.Sq + w.q0 + 128 * t + rr) * p.H + w.h) * D;
          if constexpr (kShard) dst += w.chunk * sh.po_stride;
          *reinterpret_cast<uint4*>(dst + lu * 8) = lds128(src);
        }
      }
      __syncwarp();
      (kShard ? p.lse + w.chunk * ShardStride<kMode>::pl(sh) : p.lse)[(static_cast<size_t>(w.b) * p.Sq + qrow) * p.H + w.h] =
          valid_row ? (m_used + log2f(l)) * kLn2 : -INFINITY;
      ++qi;
    }
  } else {
    regs_dec<72>();
    if (warp == 12) {
      if (lane == 0) s_issuer();
    } else if (warp == 13) {
      if (lane == 0) pv_issuer();
    }
  }
  }
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tbase, 512);
}
