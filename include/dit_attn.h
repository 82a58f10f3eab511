/*
 * dit_attn.h -- C-ABI of the GB300 (sm_103a) video-DiT attention library.
 *
 * The library computes the data-parallel hot path of video diffusion-transformer
 * attention over token sequences padded to whole 128-row tiles:
 *   - split-halves rotary embedding (RoPE) on q and k,
 *   - self-attention with the pad keys masked out and the RoPE rotation fused into the
 *     q/k tile load, emitting O and the log-sum-exp (LSE),
 *   - short-KV cross-attention of video queries against a text sequence,
 *   - the merge of partial attention results over key shards through their LSEs,
 * and three variants of the self-attention: with a per-head q/k RMSNorm ahead of the
 * rotation, with the fixed-m softmax (norm-bounded maximum per 32-row block), and with
 * e4m3 (FP8) tensor-core products.
 * Sources: Difflet PR #153 "TPU sequence parallelism: ... Wan padding + split RoPE"
 * (row padding to whole tiles, pad keys dropped exactly, identity rotation for pad rows,
 * split-halves RoPE); maxdiffusion PR #491 (Wan fast inference: lane padding to a
 * multiple of 128, pad keys masked through the real KV length, fused short-KV
 * cross-attention); mstar PR #376 (LTX-2.5 TP/SP: attention that also returns the LSE in
 * natural log, attention over sharded keys merged through the LSE; rowwise FP8 linears as
 * the motivation for the FP8 variant).
 *
 * Conventions for every call
 *   - Tensors are contiguous BSHD: q/k/v/out [B, S, H, D] bf16 (raw 16-bit storage passed
 *     as void*), LSE [B, S, H] fp32, natural log of the sum of exp of the SCALED scores.
 *   - Pointers are device pointers unless marked "host". The caller owns every buffer;
 *     the library allocates no device memory and keeps no state other than one per-device
 *     status word (see dit_device_status).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream). Device
 *     calls are asynchronous on that stream and never synchronize the host.
 *   - Padded lengths (Sq, Skv, S) are multiples of 128. D is 64 or 128. Valid lengths are
 *     runtime arguments, so one compiled kernel serves every length.
 *   - The library fails closed: invalid or unsupported arguments return an error status
 *     before any device work is queued; it never runs unpadded or unmasked instead.
 *   - Calls are thread-safe. The last CUDA error code seen by a call on the calling thread
 *     is available through dit_last_cuda_error().
 */
#ifndef DIT_ATTN_H_
#define DIT_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every call. */
#define DIT_OK 0
#define DIT_ERR_INVALID_ARG (-1) /* null pointer, length out of range, bad count or scale   */
#define DIT_ERR_UNSUPPORTED (-2) /* D not in {64, 128}, padded length not a multiple of 128 */
#define DIT_ERR_ALIGNMENT (-3)   /* a device pointer not 16-byte aligned (TMA / 16-B loads) */
#define DIT_ERR_CUDA (-4)        /* a CUDA call or launch failed; see dit_last_cuda_error() */
#define DIT_ERR_TIMEOUT (-5)     /* a kernel gave up on a bounded wait (dit_device_status)  */

/* Human-readable name of a status code (static string; never NULL). */
const char* dit_status_string(int status);

/* cudaError_t value of the last failing CUDA call made by this thread inside the library
 * (0 if none). */
int dit_last_cuda_error(void);

/* Reads the current device's status word into *status_out (host pointer) and clears it if
 * `clear` is non-zero. Bits 0-5 are set by kernels that gave up on a bounded internal wait
 * (each wait is limited to about two seconds, after which the kernel records the bit,
 * releases its resources and exits instead of hanging); bit 6 by a cross-attention call
 * that was given a key length outside its range (see dit_cross_attn_shortkv).
 * Synchronizes the current device.
 * Returns DIT_OK, DIT_ERR_INVALID_ARG (null pointer) or DIT_ERR_CUDA. */
#define DIT_STATUS_TIMEOUT_LOAD 0x01u    /* a TMA producer waited too long for a free slot    */
#define DIT_STATUS_TIMEOUT_MMA 0x02u     /* an MMA issuer waited too long for its operands    */
#define DIT_STATUS_TIMEOUT_SOFTMAX 0x04u /* a softmax / epilogue thread waited too long       */
#define DIT_STATUS_TIMEOUT_AUX 0x08u     /* a rotation / zeroing thread waited too long       */
#define DIT_STATUS_TIMEOUT_DRAIN 0x10u   /* cleanup after a timeout did not see work finish   */
#define DIT_STATUS_TIMEOUT_GRID 0x20u    /* a CTA waited too long at a grid-wide barrier      */
#define DIT_STATUS_BAD_KV_LENGTH 0x40u   /* a device-side key length outside [0, Skv]          */
int dit_device_status(unsigned int* status_out, int clear);

/* ---------------------------------------------------------------------------------------
 * RoPE cos/sin tables (host). Difflet PR #153: split-halves rotary pairs channel i with
 * channel i + D/2; pad rows get the identity rotation.
 *
 * cos, sin: host arrays [S_pad, D/2] fp32, row r = token r. Angles are computed in fp64 and
 * rounded to fp32. Rows r >= L (1-D) or r >= T*Hh*W (3-D) hold cos = 1, sin = 0.
 * ------------------------------------------------------------------------------------- */

/* 1-D: angle[r][i] = (pos_offset + r) * theta^(-2 i / D) for r < L.
 * Errors: DIT_ERR_INVALID_ARG (null, L < 0, L > S_pad, theta <= 0), DIT_ERR_UNSUPPORTED
 * (D odd or < 2). */
int dit_rope_table_1d(float* cos_out, float* sin_out, int S_pad, int L, int D, double theta,
                      int pos_offset);

/* 3-D over a T x Hh x W latent grid, tokens in row-major order (t slowest). The D/2 pairs
 * are cut into consecutive blocks of d_t/2, d_h/2, d_w/2 pairs (Wan: 44/42/42 channels);
 * pair j of an axis block rotates by coord_axis * theta^(-2 j / d_axis).
 * Errors: DIT_ERR_INVALID_ARG (null, T*Hh*W > S_pad, negative sizes, theta <= 0),
 * DIT_ERR_UNSUPPORTED (d_t + d_h + d_w != D or an odd axis width). */
int dit_rope_table_3d(float* cos_out, float* sin_out, int S_pad, int T, int Hh, int W, int D,
                      int d_t, int d_h, int d_w, double theta);

/* ---------------------------------------------------------------------------------------
 * Standalone split-halves RoPE (Difflet PR #153, split RoPE commit; maxdiffusion PR #491,
 * fused RoPE kernel):
 *   y[.., i]       = x[.., i] cos - x[.., i + D/2] sin
 *   y[.., i + D/2] = x[.., i] sin + x[.., i + D/2] cos,   (cos, sin) = table row s, col i.
 * x, y: [B, S, H, D] bf16 (y may equal x for in place); cos, sin: [S, D/2] fp32 (device).
 * Math in fp32, result rounded to nearest-even bf16.
 * Errors: DIT_ERR_INVALID_ARG (null, B/S/H < 1), DIT_ERR_UNSUPPORTED (D not 64/128),
 * DIT_ERR_ALIGNMENT (x, y, cos, sin not 16-byte aligned), DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
int dit_rope_split_halves(const void* x, void* y, const float* cos_tab, const float* sin_tab,
                          int B, int S, int H, int D, void* stream);

/* ---------------------------------------------------------------------------------------
 * Self-attention forward over padded sequences (also used for one key shard).
 * Difflet PR #153 (pad keys dropped exactly), maxdiffusion PR #491 (real KV length as the
 * ragged tail), mstar PR #376 (LSE returned in natural log).
 *
 * For batch b, head h and query row i < q_valid_len:
 *   q~_i = R(cos_q, sin_q row i) q_i,  k~_j = R(cos_k, sin_k row j) k_j   (if tables given)
 *   s_j = softmax_scale * q~_i . k~_j,  j < kv_valid_len only
 *   lse[b,i,h] = ln sum_j exp(s_j),  out[b,i,h,:] = sum_j exp(s_j - lse) v_j
 * Query rows i >= q_valid_len get out = 0 and lse = -inf. If kv_valid_len == 0 every row
 * does. Pad rows of q, k and v (rows >= the valid length) are never read, so their
 * contents (even NaN/Inf) cannot change any output.
 *
 * q: [B, Sq, H, D]; k, v: [B, Skv, H, D]; out: [B, Sq, H, D] (bf16); lse: [B, Sq, H] fp32.
 * cos_q/sin_q: [Sq, D/2], cos_k/sin_k: [Skv, D/2] fp32 device tables; all four NULL = no
 * RoPE (all four or none must be given). With RoPE, q~ and k~ are computed in fp32 and
 * rounded to fp16 (saturating) for the tensor-core product; without it q and k enter as
 * their bf16 values. P is rounded to bf16 before P.V; accumulation and softmax are fp32.
 * Constraints: Sq, Skv multiples of 128; D in {64, 128}; 0 <= q_valid_len <= Sq;
 * 0 <= kv_valid_len <= Skv; softmax_scale > 0 and finite (callers normally pass 1/sqrt(D)).
 * Errors: DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_ALIGNMENT (q, k, v, out, tables
 * not 16-byte aligned; lse not 4-byte aligned), DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
int dit_attn_fwd(const void* q, const void* k, const void* v, int B, int Sq, int Skv, int H,
                 int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                 const float* sin_q, const float* cos_k, const float* sin_k,
                 float softmax_scale, void* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------------------
 * dit_attn_fwd with RoPE, rotating every q and k row exactly once per call (same inputs,
 * outputs and numerics as dit_attn_fwd with tables). The launch first rotates the valid rows
 * of k with the given tables into an fp16 copy in `workspace` (all CTAs; the loads of the
 * rotated rows wait until every CTA has finished, so the launch is cooperative). It then runs
 * the attention on that copy; each q tile, loaded once per CTA that uses it, is rotated in
 * shared memory as it lands. Without a workspace, dit_attn_fwd rotates each k tile again in
 * every CTA that loads it.
 *
 * workspace: device buffer of at least dit_attn_workspace_bytes(B, Sq, Skv, H, D) bytes,
 * 256-byte aligned, owned by the caller; its contents on entry do not matter and are
 * overwritten. Calls that share a workspace must not overlap on the GPU.
 * All four tables are required. Errors as dit_attn_fwd, plus DIT_ERR_INVALID_ARG for a
 * missing or too small workspace, DIT_ERR_ALIGNMENT for a misaligned one, DIT_ERR_UNSUPPORTED
 * when max(Sq, Skv) * H * D / 16 >= 2^30 (one batch of rows indexed in 32 bits), and
 * DIT_ERR_CUDA if the GPU cannot run the cooperative launch.
 * ------------------------------------------------------------------------------------- */
size_t dit_attn_workspace_bytes(int B, int Sq, int Skv, int H, int D);
int dit_attn_fwd_ws(const void* q, const void* k, const void* v, int B, int Sq, int Skv, int H,
                    int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                    const float* sin_q, const float* cos_k, const float* sin_k,
                    float softmax_scale, void* out, float* lse, void* workspace,
                    size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * dit_attn_fwd_ws with a per-head RMSNorm of q and k ahead of the rotation (Difflet PR #153,
 * FLUX and Wan split-RoPE commits: the per-head q/k RMSNorm weights are permuted with the
 * q/k channels into the split-halves order, so the norm acts in that layout just before the
 * rotation). For each (b, s, h) row of q (weights norm_q) and of k (norm_k):
 *   n = x / sqrt(mean_d(x_d^2) + eps) * w,  then the split-halves rotation of n,
 * computed in fp32 from the bf16 inputs and rounded to fp16 for the tensor-core product, as
 * in dit_attn_fwd_ws. norm_q, norm_k: device fp32 [D], 16-byte aligned, in the same channel
 * order as q and k. eps >= 0 and finite (models normally use 1e-6). Workspace, tables,
 * layouts, outputs and the remaining errors as dit_attn_fwd_ws; DIT_ERR_INVALID_ARG also for a
 * missing weight vector or a bad eps, DIT_ERR_ALIGNMENT for a misaligned weight vector.
 * ------------------------------------------------------------------------------------- */
int dit_attn_fwd_ws_qknorm(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                           int H, int D, int q_valid_len, int kv_valid_len, const float* norm_q,
                           const float* norm_k, float eps, const float* cos_q, const float* sin_q,
                           const float* cos_k, const float* sin_k, float softmax_scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * dit_attn_fwd_ws with the fixed-m softmax (maxdiffusion PR #491, Wan fast inference: a
 * "fixed-m per Q block" attention kernel takes per-block metadata from norm reductions over
 * q and k, with pad rows excluded, and lets a block whose metadata allows it skip the online
 * softmax). The pages give no formula; this library's metadata and proof:
 *   bound of query row i:  m_i = softmax_scale * |q_i| * max_{j < kv_valid_len} |k_j|.
 * By Cauchy-Schwarz no valid score s_ij = softmax_scale * q~_i . k~_j exceeds m_i, and the
 * rotation preserves norms, so the raw rows give the bound of the rotated ones. A block of
 * 32 consecutive query rows of one head (one warp) uses p_ij = exp(s_ij - m_i) with m_i
 * fixed -- no running maximum, no rescaling of the accumulator -- when every valid row of
 * the block has 2 m_i <= 64 ln 2: all its scores then lie in [-m_i, m_i], so its largest
 * term is at least 2^-64 and no term exceeds 1. Other blocks take the online softmax. The
 * key maximum runs over valid keys only and pad query rows take no part in the decision, so
 * pad contents never move a block onto the online path. In exact arithmetic both paths give
 * the plain softmax; O and LSE match dit_attn_fwd_ws within the same tolerances.
 *
 * workspace: device buffer of at least dit_attn_fixed_m_workspace_bytes(B, Sq, Skv, H, D)
 * bytes, 256-byte aligned, owned by the caller, contents on entry irrelevant (the call clears
 * what needs clearing on `stream`). n_online: NULL, or a device unsigned int (4-byte
 * aligned) to which the call adds the number of 32-row blocks that took the online path;
 * the caller zeroes it. Calls sharing a workspace or an n_online counter must not overlap.
 * Everything else (arguments, layouts, tables, outputs, numerics) as dit_attn_fwd_ws.
 * Errors: as dit_attn_fwd_ws (workspace checked against the size above), plus
 * DIT_ERR_UNSUPPORTED when B * H > 24576 and DIT_ERR_ALIGNMENT for a misaligned n_online.
 * ------------------------------------------------------------------------------------- */
size_t dit_attn_fixed_m_workspace_bytes(int B, int Sq, int Skv, int H, int D);
int dit_attn_fwd_ws_fixed_m(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                            int H, int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                            const float* sin_q, const float* cos_k, const float* sin_k,
                            float softmax_scale, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, unsigned int* n_online, void* stream);

/* ---------------------------------------------------------------------------------------
 * FP8 (e4m3) attention. The pages measure FP8 only for linear layers (mstar PR #376: a sizing
 * experiment with rowwise FP8 linears cut the SP2 step by about a quarter); this applies the
 * e4m3 format (OCP 8-bit floating point: 4 exponent bits, bias 7, 3 mantissa bits, largest
 * value 448) to the attention of dit_attn_fwd. Steps:
 *   1. q and k are rotated (split-halves RoPE; no rotation when the four tables are NULL) in
 *      fp32; q~ is quantised per 128-row tile of a head, k~ and v per head: scale = amax /
 *      448 over the valid rows (1 when 0), x8 = e4m3(x / scale), round to nearest even,
 *      saturating. v is stored transposed. All of it goes to `workspace`.
 *   2. S = q8 k8^T on the tensor cores (e4m3 operands, fp32 accumulation), times
 *      softmax_scale * s_q * s_k. Softmax over key tiles of 128 with a running maximum m that
 *      lags by at most 2 in log2 units (so p = 2^(s log2 e - m) <= 4); P8 = e4m3(112 p),
 *      O += P8 v8 (e4m3, fp32).
 *   3. O = O * s_v / (112 l) with l = sum p in fp32, LSE = m + ln l; pad rows O = 0, LSE = -inf.
 * Results differ from exact attention by the e4m3 rounding (about 0.04 max-abs on O and 0.02
 * on the LSE for unit-variance inputs, one rounding per operand); against a reference doing
 * the same steps they agree to fp32 accumulation and rare one-step rounding differences.
 * D must be 128. workspace: at least dit_attn_fp8_workspace_bytes(B, Sq, Skv, H, 128) bytes,
 * 256-byte aligned, caller-owned, contents on entry irrelevant; calls sharing one must not
 * overlap. Three launches on `stream` (two preparation kernels, then the attention).
 * Everything else (arguments, layouts, pad handling) as dit_attn_fwd. Errors: as dit_attn_fwd;
 * DIT_ERR_UNSUPPORTED for D != 128; DIT_ERR_INVALID_ARG for a missing or too small workspace
 * or some but not all tables; DIT_ERR_ALIGNMENT for a misaligned workspace (256) or table (16).
 * ------------------------------------------------------------------------------------- */
size_t dit_attn_fp8_workspace_bytes(int B, int Sq, int Skv, int H, int D);
int dit_attn_fwd_fp8(const void* q, const void* k, const void* v, int B, int Sq, int Skv, int H,
                     int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                     const float* sin_q, const float* cos_k, const float* sin_k,
                     float softmax_scale, void* out, float* lse, void* workspace,
                     size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * Standalone per-head RMSNorm then split-halves RoPE (the prologue dit_attn_fwd_ws_qknorm
 * fuses): y[b,s,h,:] = rotate(x[b,s,h,:] / sqrt(mean(x^2) + eps) * w) with table row s.
 * x, y: [B, S, H, D] bf16 (y may equal x); w: device fp32 [D]; cos, sin: [S, D/2] fp32.
 * Arithmetic in fp32, one rounding to bf16 at the end.
 * Errors: DIT_ERR_INVALID_ARG (null, sizes < 1, bad eps), DIT_ERR_UNSUPPORTED (D not 64/128),
 * DIT_ERR_ALIGNMENT (any pointer not 16-byte aligned), DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
int dit_qk_rmsnorm_rope(const void* x, void* y, const float* w, float eps, const float* cos,
                        const float* sin, int B, int S, int H, int D, void* stream);

/* ---------------------------------------------------------------------------------------
 * dit_attn_fwd_ws without a caller-supplied workspace. The pages have no counterpart: this
 * is a library convenience, not part of the method.
 *
 * Who needs it: callers that cannot hand in device memory at the call site. Examples are a
 * plain C caller with no allocator of its own, and code inside a framework whose caching
 * allocator already holds the device memory. There a cudaMalloc can fail for lack of
 * memory, and a cudaMalloc or cudaFree per call can synchronise the device. This function
 * allocates nothing and calls no allocating routine.
 *
 * Scratch: a fixed array of DIT_ATTN_STATIC_SCRATCH_BYTES (96 MiB) of device memory,
 * declared in the library at file scope. The CUDA runtime reserves it on each device where
 * it loads the library's device code. The workspace holds the rotated keys: the Wan 480p
 * self-attention (B1, 4736 key rows, H40, D128) needs 46.25 MiB, and the array fits up to
 * 9728 key rows at H40, D128.
 *
 * Set-up: the first call on each device looks up the array's device address with that
 * device current, once, under a lock. Make that first call outside any stream capture.
 *
 * Zero state: nothing in the array has to start at zero. Each call clears the grid-barrier
 * word on `stream` before its kernel starts, and the rotated k copy is written before
 * it is read.
 *
 * Overlap: there is one array per device per process. Two calls in flight on the same
 * device at the same time share it. That happens with calls on two streams, or from two
 * host threads with no ordering between them. Such calls race: they overwrite each other's
 * rotated k copies and barrier word, and their results are wrong. Order such calls on one
 * stream, or use dit_attn_fwd_ws with one workspace per stream.
 *
 * Arguments, outputs and numerics are those of dit_attn_fwd_ws; all four tables are
 * required. Errors: as dit_attn_fwd_ws. DIT_ERR_UNSUPPORTED also when
 * dit_attn_workspace_bytes(B, Sq, Skv, H, D) > DIT_ATTN_STATIC_SCRATCH_BYTES, or when the
 * current device's ordinal is 64 or more. DIT_ERR_CUDA if the set-up lookup fails.
 * ------------------------------------------------------------------------------------- */
#define DIT_ATTN_STATIC_SCRATCH_BYTES ((size_t)96 << 20)
int dit_attn_fwd_ws_static(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                           int H, int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                           const float* sin_q, const float* cos_k, const float* sin_k,
                           float softmax_scale, void* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------------------
 * Short-KV cross-attention (maxdiffusion PR #491: fused short-KV cross-attention of the video
 * queries against the text sequence). As dit_attn_fwd without RoPE, with one valid key
 * length per batch read on the device: kv_valid_len_dev[b] in [0, Skv] (int32, device
 * array of B entries). Skv <= 512.
 * Fails closed on the device: a batch whose length lies outside [0, Skv] is not clamped
 * into range. All of its query rows get out = 0 and lse = -inf, and the kernel sets
 * DIT_STATUS_BAD_KV_LENGTH in the device status word (read it with dit_device_status). The
 * lengths live in device memory, so the call cannot check them before it returns without
 * a host synchronisation; the status bit keeps the call asynchronous.
 * Errors as dit_attn_fwd; DIT_ERR_UNSUPPORTED also for Skv > 512.
 * ------------------------------------------------------------------------------------- */
int dit_cross_attn_shortkv(const void* q, const void* k, const void* v, int B, int Sq,
                           int Skv, int H, int D, int q_valid_len,
                           const int32_t* kv_valid_len_dev, float softmax_scale, void* out,
                           float* lse, void* stream);

/* ---------------------------------------------------------------------------------------
 * Attention of one query block over keys held in shards, in one call (mstar PR #376:
 * attention over sharded keys, each shard's partial output and log-sum-exp merged through
 * the LSE; Difflet PR #153: every token keeps its rotary angle, so shard s rotates its keys
 * at their global positions). Computes exactly what dit_attn_fwd with RoPE would over the
 * concatenation of the shards' valid keys:
 *   for query row i < q_valid_len:  lse_i = ln sum_{s, j < valid_s} exp(score_sj),
 *   out_i = sum_{s, j} exp(score_sj - lse_i) v_sj,  score_sj = softmax_scale q~_i . k~_sj,
 * with q~ rotated by (cos_q, sin_q) and the keys of shard s by (cos_k[s], sin_k[s]).
 * Pad query rows and rows with no valid key at all get out = 0, lse = -inf.
 *
 * One cooperative launch rotates every shard's valid k rows into an fp16 copy in the
 * workspace and runs the attention of all shards at once: the shards are cut into key chunks
 * of whole 128-row tiles of near-equal length, so that chunks x B x H x (256-row query blocks)
 * gives enough work items to fill the GPU; each chunk writes a partial (O, LSE) to the
 * workspace. A second launch merges the partials (dit_attn_lse_merge's kernel).
 *
 * q: [B, Sq, H, D] bf16; out: [B, Sq, H, D] bf16; lse: [B, Sq, H] fp32; cos_q, sin_q:
 * [Sq, D/2] fp32. k_shards[s], v_shards[s]: [B, shard_padded[s], H, D] bf16 (device pointers
 * held in host arrays of n_shards entries); cos_k[s], sin_k[s]: [shard_padded[s], D/2] fp32
 * at the shard's global key positions; shard_valid[s] in [0, shard_padded[s]] (host int
 * arrays). 1 <= n_shards <= 64, at most 16 of them non-empty; shard_padded[s] a multiple of
 * 128 (0 allowed for an empty shard, whose pointers are then not used). Numerics as dit_attn_fwd_ws (fp16 rotated q~, k~; bf16 P; fp32 accumulation); the
 * partials are bf16, merged in fp32.
 * workspace: at least dit_attn_sharded_workspace_bytes(...) bytes (same B, Sq, H, D and shard
 * lengths), 256-byte aligned, caller-owned, contents on entry irrelevant; calls sharing one
 * must not overlap. The chunk plan, and with it the workspace size, depends only on the
 * arguments, not on the device.
 * Errors: DIT_ERR_INVALID_ARG (null pointer, bad length or scale, workspace too small),
 * DIT_ERR_UNSUPPORTED (D not 64/128, a length not a multiple of 128, more than 16 non-empty
 * shards, sizes past 32-bit row indexing), DIT_ERR_ALIGNMENT, DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
size_t dit_attn_sharded_workspace_bytes(int B, int Sq, int H, int D, int n_shards,
                                        const int* shard_padded, const int* shard_valid);
int dit_attn_fwd_sharded(const void* q, int B, int Sq, int H, int D, int q_valid_len,
                         int n_shards, const void* const* k_shards, const void* const* v_shards,
                         const int* shard_padded, const int* shard_valid, const float* cos_q,
                         const float* sin_q, const float* const* cos_k, const float* const* sin_k,
                         float softmax_scale, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------
 * LSE merge of partial results over key shards (mstar PR #376, attention over sharded keys):
 *   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * O_s.
 * A row whose n partial LSEs are all -inf (no shard saw a key) gets out = 0, lse = -inf.
 * partial_o: [n][B, S, H, D] bf16, contiguous; partial_lse: [n][B, S, H] fp32;
 * out: [B, S, H, D] bf16 (rounded to nearest even from fp32); lse: [B, S, H] fp32.
 * S need not be padded here. 1 <= n <= 64.
 * Errors: DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED (D not 64/128), DIT_ERR_ALIGNMENT
 * (partial_o, out not 16-byte aligned; lse arrays not 4-byte aligned), DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
int dit_attn_lse_merge(const void* partial_o, const float* partial_lse, int n, int B, int S,
                       int H, int D, void* out, float* lse, void* stream);

/* ---------------------------------------------------------------------------------------
 * Token padding at the boundary (Difflet PR #153: the first block pads the patch sequence,
 * the last cuts the pad; maxdiffusion PR #491: pad the tokens at the tail, unpad the output).
 *
 * dit_pad_tokens copies rows [0, L) of x [B, L, row_bytes] into x_pad [B, S_pad, row_bytes];
 * pad rows of x_pad are left untouched (attention never reads them).
 * dit_unpad_tokens copies rows [0, L) of x_pad [B, S_pad, row_bytes] into x [B, L, row_bytes].
 * row_bytes is the size of one token row (H*D*2 for q/k/v/O, H*4 for LSE), any value >= 1.
 * Errors: DIT_ERR_INVALID_ARG (null, B < 1, L < 0, L > S_pad, row_bytes < 1), DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
int dit_pad_tokens(const void* x, void* x_pad, int B, int L, int S_pad, long long row_bytes,
                   void* stream);
int dit_unpad_tokens(const void* x_pad, void* x, int B, int L, int S_pad, long long row_bytes,
                     void* stream);

/* ---------------------------------------------------------------------------------------
 * Diagnostic: the FMA-pipe exponential the attention softmax uses for part of its
 * exponentials (the rest go to the special-function unit), applied elementwise:
 * y[i] ~ 2^x[i] for x[i] <= 126, max relative error 2.6e-6 (degree-4 minimax polynomial
 * after Cody-Waite range reduction); inputs below -125 give 2^-125 (the kernel only feeds it
 * arguments where that is negligible). x, y: device fp32 arrays of n elements. No page
 * defines this; it exists so the approximation can be tested against exp2f.
 * Errors: DIT_ERR_INVALID_ARG, DIT_ERR_ALIGNMENT (not 4-byte aligned), DIT_ERR_CUDA.
 * ------------------------------------------------------------------------------------- */
int dit_exp2_fma_eval(const float* x, float* y, long long n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DIT_ATTN_H_ */
