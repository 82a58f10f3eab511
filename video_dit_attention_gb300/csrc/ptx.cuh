// Inline-PTX layer for sm_103a: mbarriers with bounded waits, TMA tensor loads,
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads/stores) and the shared-memory
// and instruction descriptors the tcgen05 MMA consumes.
//
// Everything here is written from the public PTX ISA description of these
// instructions; there is no library code underneath.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace dit {

// ---------------------------------------------------------------------------
// Device status word. Bit values are OR-ed in by kernels that give up on a wait
// (see bounded_wait below); the host reads and clears it through the C-ABI.
// ---------------------------------------------------------------------------
enum : unsigned int {
  kStatusTimeoutLoad = 1u << 0,   // a TMA producer gave up waiting for a free stage
  kStatusTimeoutMma = 1u << 1,    // the MMA issuer gave up waiting for operands
  kStatusTimeoutSoftmax = 1u << 2,// a softmax/epilogue thread gave up waiting for S or O
  kStatusTimeoutRope = 1u << 3,   // a rotation thread gave up waiting for a landed tile
  kStatusTimeoutDrain = 1u << 4,  // cleanup after an abort did not see in-flight work finish
  kStatusTimeoutGrid = 1u << 5,   // a CTA gave up waiting at the grid-wide barrier
  kStatusBadKvLength = 1u << 6,   // cross-attention: a device-side key length outside [0, Skv]
};

// Upper bound on any single wait, in nanoseconds of %globaltimer. Every wait in
// these kernels normally completes in microseconds; after this long the kernel
// records a status bit, lets its other roles fall through and exits cleanly.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

#ifdef DIT_TEST_HOOKS
// Test-only build (libdit_attn_testhooks.so, never the product library): the limit is a
// device variable that a test shortens, so that a wait it makes run out gives up within
// milliseconds instead of seconds. Each translation unit compiled for the test library has
// its own copy of these (internal linkage) and its own setter.
static __device__ unsigned long long g_dit_test_wait_limit_ns = kWaitLimitNs;
// Number of the load that a kernel's K/V producer counts but never issues (-1: none): a K/V
// ring load of the attention kernel, a fill of the cross-attention kernel. The consumers of
// that load then wait until the limit runs out.
static __device__ int g_dit_test_skip_load = -1;
__device__ __forceinline__ uint64_t wait_limit_ns() { return g_dit_test_wait_limit_ns; }
#else
__device__ __forceinline__ constexpr uint64_t wait_limit_ns() { return kWaitLimitNs; }
#endif

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete. Returns false if the CTA
// is aborting (another role gave up) or if this wait itself ran past
// wait_limit_ns(); in the latter case it raises the CTA abort flag and ORs `code`
// into the device status word. Never spins forever.
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity,
                                             volatile int* cta_abort,
                                             unsigned int* dev_status, unsigned int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
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

// Same bound, for cleanup after an abort: waits for work already in flight (TMA
// copies, MMAs) to land before the CTA releases its shared and tensor memory.
// Ignores the abort flag.
__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity,
                                           unsigned int* dev_status) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > wait_limit_ns()) {
      atomicOr(dev_status, kStatusTimeoutDrain);
      return false;
    }
  }
}

// Load with acquire semantics at device scope (pairs with a fence + atomic on another SM).
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Proxy fences and named barriers
// ---------------------------------------------------------------------------
// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tcgen05.mma) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's generic-proxy accesses (all state spaces) with its later async-proxy
// (TMA) accesses; used around data written with plain stores and read back by TMA.
__device__ __forceinline__ void fence_proxy_async_all() {
  asm volatile("fence.proxy.async;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ANDs a predicate over the participating threads: every thread
// leaves with the same answer (all of them had `pred` set).
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tiled mode, completion on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Stores one tile from shared memory to global memory (tiled TMA store, bulk-group
// completion). The shared-memory source must not be overwritten before bulk_wait_read().
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Warms L2 with one tile of a tensor (no shared-memory destination, no completion).
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory
// ---------------------------------------------------------------------------
// One full warp executes alloc/dealloc. The allocated column base is written to
// shared memory at `dst_smem`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TMEM address: lane in bits 31:16, column in bits 15:0.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

// ---------------------------------------------------------------------------
// tcgen05: MMA issue and completion
// ---------------------------------------------------------------------------
// D[tmem] (+)= A[smem desc] * B[smem desc]; kind::f16 (bf16 inputs here), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc] for e4m3 operands (kind::f8f6f4; both formats
// 0 = e4m3 in the instruction descriptor, which then has the layout of idesc_f16kind_f32 with
// its format fields at 0). One instruction covers K = 32 (32 bytes of each operand row).
__device__ __forceinline__ void mma_e4m3_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]; A holds two bf16 per 32-bit TMEM cell.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor for kind::f16 with an fp32 accumulator.
// Bit fields: [4,6) D format (1 = f32), [7,10) A format, [10,13) B format (0 = f16,
// 1 = bf16; A and B must have the same format), [15] A major (0 = K-major, 1 = MN-major),
// [16] B major, [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_f16kind_f32(uint32_t M, uint32_t N, bool bf16,
                                                         bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, bool a_mn_major,
                                                      bool b_mn_major) {
  return idesc_f16kind_f32(M, N, true, a_mn_major, b_mn_major);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
// Fields: [0,14) start address >> 4, [16,30) leading byte offset >> 4,
// [32,46) stride byte offset >> 4, [46,48) descriptor version (1),
// [49,52) base offset (0: tiles are 1024-byte aligned), [61,64) layout (2 = 128B swizzle).
//
// K-major operand (rows of 64 bf16 = 128 B, 8-row groups of 1024 B): SBO = 1024,
//   LBO unused; stepping K by 16 elements adds 32 B to the start address.
// MN-major operand (64 MN-contiguous elements per 128-B row, rows along K):
//   LBO = byte distance between consecutive 64-element MN blocks,
//   SBO = byte distance between consecutive 8-row K groups (1024 when packed).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM <-> registers. A warp may touch only lanes 32*(warp%4) .. +31.
// ---------------------------------------------------------------------------
#define DIT_R8(i) "=r"(r[i + 0]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define DIT_W8(i) "+r"(r[i + 0]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                  "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])
#define DIT_S8(i) "r"(r[i + 0]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                  "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])

// Loads 32 consecutive 32-bit columns of this thread's lane into r[0..31], then
// waits for the load; the wait names every register so no use can move above it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : DIT_R8(0), DIT_R8(8), DIT_R8(16), DIT_R8(24)
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : DIT_W8(0), DIT_W8(8), DIT_W8(16), DIT_W8(24)
               :
               : "memory");
}

// Issues the load of 32 columns without waiting; the registers are valid only after a
// later tmem_ld_wait_tied() / tmem_reg_tie() pair names them.
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : DIT_R8(0), DIT_R8(8), DIT_R8(16), DIT_R8(24)
      : "r"(taddr)
      : "memory");
}
// Waits for every outstanding tcgen05.ld of this thread; names r so no use moves above it.
__device__ __forceinline__ void tmem_ld_wait_tied(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : DIT_W8(0), DIT_W8(8), DIT_W8(16), DIT_W8(24)
               :
               : "memory");
}
// Orders uses of r after the preceding volatile asm (an empty statement that "writes" r).
__device__ __forceinline__ void tmem_reg_tie(uint32_t (&r)[32]) {
  asm volatile("" : DIT_W8(0), DIT_W8(8), DIT_W8(16), DIT_W8(24) : : "memory");
}

// 16 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : DIT_R8(0), DIT_R8(8)
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" : DIT_W8(0), DIT_W8(8) : : "memory");
}

// Stores r[0..31] into 32 consecutive columns of this thread's lane and waits.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      DIT_S8(0), DIT_S8(8), DIT_S8(16), DIT_S8(24)
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      DIT_S8(0), DIT_S8(8)
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Stores without waiting; pair with tmem_st_wait() after the last store of a batch.
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      DIT_S8(0), DIT_S8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_st8_nowait(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
      DIT_S8(0)
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

#undef DIT_R8
#undef DIT_W8
#undef DIT_S8

// ---------------------------------------------------------------------------
// Per-warpgroup register budgets (all 128 threads of a warpgroup execute these).
// ---------------------------------------------------------------------------
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// ---------------------------------------------------------------------------
// Small numeric helpers
// ---------------------------------------------------------------------------
// (d0, d1) = (a0, a1) * (b, b) + (c, c) with one packed fp32x2 FMA.
__device__ __forceinline__ void fma2_bc(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 A, B, C, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 B, {%4, %4};\n\tmov.b64 C, {%5, %5};\n\t"
      "fma.rn.f32x2 D, A, B, C;\n\tmov.b64 {%0, %1}, D;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) += (a0, a1) with one packed fp32x2 add.
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1) {
  asm("{\n\t.reg .b64 A, D;\n\t"
      "mov.b64 A, {%2, %3};\n\tmov.b64 D, {%0, %1};\n\t"
      "add.f32x2 D, D, A;\n\tmov.b64 {%0, %1}, D;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// 2^x on the special-function unit (PTX ex2.approx.ftz.f32; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> two e4m3 (round to nearest even, saturating to +-448): `lo` in bits 7:0.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Packs two fp32 into bf16x2 (round to nearest even): `lo` in bits 15:0.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

// Packs two fp32 into f16x2 (round to nearest even, saturating to +-65504): `lo` in 15:0.
__device__ __forceinline__ uint32_t pack_f16x2_satfinite(float lo, float hi) {
  uint32_t out;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a tile of 128-byte
// rows stored with the 128-byte swizzle (tile base 1024-byte aligned).
__host__ __device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace dit
