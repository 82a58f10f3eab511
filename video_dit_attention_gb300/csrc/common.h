// Internal declarations shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dit {

// One attention call: self-attention (optionally with RoPE), short-KV cross-attention or
// sharded keys. Pointers are device pointers; shapes as in include/dit_attn.h.
struct AttnArgs {
  const void* q;
  const void* k;
  const void* v;
  int B, Sq, Skv, H, D;
  int q_valid;
  int kv_valid;                 // self-attention: one length for every batch
  const int32_t* kv_valid_dev;  // cross-attention: per-batch lengths on the device
  const float* cos_q;
  const float* sin_q;
  const float* cos_k;
  const float* sin_k;
  float scale;
  void* out;
  float* lse;
  void* workspace;              // RoPE workspace modes: rotated fp16 k and a CTA counter
  const float* norm_q;          // per-head q/k RMSNorm weights [D] (kModeRopeWsNorm)
  const float* norm_k;
  float norm_eps;
  cudaStream_t stream;
  unsigned int* n_online;       // fixed-m mode: count of 32-row blocks on the online path (may be null)
};

enum AttnMode : int {
  kModePlain = 0,  // no RoPE, one kv length
  kModeRope = 1,   // RoPE fused into the q/k tile load
  kModeRopeWs = 3, // RoPE applied once per q/k tile into a workspace, then attention on it
  kModeRopeWsNorm = 4,  // as kModeRopeWs, with per-head q/k RMSNorm before the rotation
  kModeRopeWsFixedM = 5,  // as kModeRopeWs; 32-row blocks whose norm bound allows it skip the
                          // running maximum (fixed-m softmax)
  kModeFp8 = 6,           // e4m3 q~, k~ (rotated) and v (transposed) prepared in the workspace;
                          // e4m3 tensor-core products, exact running maximum
  kModeRopeWsSharded = 7, // as kModeRopeWs over several key chunks in one launch, one partial
                          // (O, LSE) per chunk
};

// Sharded keys: at most this many key chunks per launch (the partials are merged through
// their LSEs afterwards).
constexpr int kMaxKeyChunks = 16;
// One key shard as the caller hands it in: raw k and v [B, S_pad, H, D] bf16, its RoPE tables
// [S_pad, D/2] at the shard's global key positions, its padded and valid lengths.
struct KeyShard {
  const void* k;
  const void* v;
  const float* cos_k;
  const float* sin_k;
  int S_pad, valid;
};
// How the shards are cut into key chunks of whole 128-row tiles, and where the workspace puts
// the rotated k of each shard, the CTA counter and the partial outputs.
struct ShardPlan {
  int n_chunks;
  int shard[kMaxKeyChunks], row0[kMaxKeyChunks], valid[kMaxKeyChunks];
  size_t rot_off[kMaxKeyChunks];   // byte offset of each chunk's shard's rotated copy
  size_t counter_off, po_off, pl_off, total;
};
// Cuts the shards into chunks of near-equal length so that there are about kShardTargetItems
// work items (six per SM of a 152-SM GB300; a fixed number, so that the plan and the workspace
// size do not depend on the device); returns false if the shards cannot be planned (more than
// kMaxKeyChunks non-empty shards, or more than 64 shards).
constexpr long long kShardTargetItems = 6 * 152;
bool plan_shards(int B, int Sq, int H, int D, int n_shards, const KeyShard* shards, int sm_count,
                 ShardPlan* plan);
cudaError_t launch_attn_sharded(const AttnArgs& a, int n_shards, const KeyShard* shards,
                                const ShardPlan& plan);

// Workspace layout of the RoPE workspace modes: rotated k [B, Skv, H, D] fp16, then a
// 256-byte block holding the count of CTAs done rotating; both 256-byte aligned.
size_t attn_workspace_bytes(int B, int Sq, int Skv, int H, int D);

// Fixed-m mode: the layout above, then the per-(b, h) largest squared key norm [B * H] (u32
// float bits, zeroed before the launch) and the per-row squared q norm [B, Sq, H] fp32, each
// 256-byte aligned. The shared-memory reduction needs B * H <= kFixedMMaxHeads.
size_t attn_fixed_m_workspace_bytes(int B, int Sq, int Skv, int H, int D);
constexpr int kFixedMMaxHeads = 24576;

// FP8 path workspace (D = 128): e4m3 q~ [B, Sq, H, D], k~ [B, Skv, H, D], v transposed
// [B, H, D, Skv]; tile maxima of q~, k~, v; scales of q~ per tile [B, H, nt_q], of k~ and v per
// head [B, H]. Offsets in bytes, each 256-byte aligned.
struct Fp8Layout {
  size_t q8, k8, vt8, amax_q, amax_k, amax_v, sq, sk, sv, total;
  int nt_q, nt_k;
};
Fp8Layout fp8_layout(int B, int Sq, int Skv, int H, int D);
// Rotation and quantisation of q, k, v into the workspace (two launches on a.stream).
cudaError_t launch_fp8_prepare(const AttnArgs& a, const Fp8Layout& L);

cudaError_t launch_attn_fwd(const AttnArgs& a, AttnMode mode);

cudaError_t launch_qk_rmsnorm_rope(const void* x, void* y, const float* w, float eps,
                                   const float* cos_tab, const float* sin_tab, int B, int S, int H,
                                   int D, cudaStream_t stream);
cudaError_t launch_rope_split_halves(const void* x, void* y, const float* cos_tab,
                                     const float* sin_tab, int B, int S, int H, int D,
                                     cudaStream_t stream);

cudaError_t launch_lse_merge(const void* partial_o, const float* partial_lse, int n, int B,
                             int S, int H, int D, void* out, float* lse, cudaStream_t stream);

cudaError_t launch_copy_rows(const void* src, void* dst, int B, int L, long long src_rows,
                             long long dst_rows, long long row_bytes, cudaStream_t stream);

cudaError_t launch_exp2_fma(const float* x, float* y, long long n, cudaStream_t stream);

cudaError_t read_device_status(unsigned int* out, bool clear);
// Device address of the current device's status word.
cudaError_t device_status_ptr(unsigned int** out);

// Short-KV cross-attention (Skv <= 512, per-batch key lengths on the device): the kernel in
// cross_attn.cu, which keeps a head's keys and values resident in shared memory.
cudaError_t launch_cross_attn(const AttnArgs& a);
#ifdef DIT_TEST_HOOKS
// Test library only: the wait limit and skipped fill of the cross-attention kernel's unit.
cudaError_t cross_attn_set_test_hooks(unsigned long long wait_limit_ns, int skip_fill);
#endif

// Encodes a TMA descriptor for a BSHD bf16 tensor [B, S_rows, H, D] whose sequence extent is
// cut to `s_extent` rows (reads past it return zeros), with a box of 64 channels x 1 head x
// 128 rows x 1 batch and the 128-byte swizzle. Returns false if the driver rejects it.
bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int s_extent, int s_rows, int H,
                     int D);

// Encodes a 4-D TMA descriptor for a uint8 tensor (dims innermost first, strides in bytes of
// dims 1..3) with the 128-byte swizzle; box[0] * 1 byte must be a multiple of 16.
bool encode_u8_map4(CUtensorMap* map, const void* base, const unsigned long long dims[4],
                    const unsigned long long strides[3], const unsigned int box[4]);

// Encodes a TMA descriptor for a row-major fp32 matrix [rows, cols] (cols * 4 a multiple of
// 16 bytes) read in unswizzled boxes of box_rows full rows.
bool encode_rows_map_f32(CUtensorMap* map, const float* base, int rows, int cols, int box_rows);

}  // namespace dit
