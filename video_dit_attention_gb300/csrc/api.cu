// C-ABI entry points (include/dit_attn.h): argument validation, TMA descriptor encoding and
// kernel launches. No device memory is allocated at call time; every buffer belongs to the
// caller, except one fixed file-scope device array (end of this file) that only
// dit_attn_fwd_ws_static uses as its workspace.

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/dit_attn.h"
#include "common.h"

namespace dit {
namespace {

thread_local int t_last_cuda_error = 0;

int cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DIT_OK;
  t_last_cuda_error = static_cast<int>(e);
  return DIT_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Shared checks of the attention entry points.
int check_attn_shapes(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                      int H, int D, int q_valid, float scale, const void* out, const float* lse) {
  if (!q || !k || !v || !out || !lse) return DIT_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Sq < 1 || Skv < 1) return DIT_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DIT_ERR_INVALID_ARG;
  if (q_valid < 0 || q_valid > Sq) return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  if ((Sq % 128) != 0 || (Skv % 128) != 0) return DIT_ERR_UNSUPPORTED;
  if (H > 65535 || B > 65535) return DIT_ERR_UNSUPPORTED;   // grid.y / grid.z limits
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return DIT_ERR_ALIGNMENT;
  return DIT_OK;
}

}  // namespace

bool encode_bshd_map(CUtensorMap* map, const void* base, int B, int s_extent, int s_rows, int H,
                     int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(s_extent), static_cast<cuuint64_t>(B)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(H) * D * 2,
                                 static_cast<cuuint64_t>(s_rows) * H * D * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u8_map4(CUtensorMap* map, const void* base, const unsigned long long dims[4],
                    const unsigned long long strides[3], const unsigned int box[4]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), d, st, bx, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_rows_map_f32(CUtensorMap* map, const float* base, int rows, int cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 4};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem_strides[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dit

using namespace dit;

extern "C" const char* dit_status_string(int status) {
  switch (status) {
    case DIT_OK: return "DIT_OK";
    case DIT_ERR_INVALID_ARG: return "DIT_ERR_INVALID_ARG: null pointer or value out of range";
    case DIT_ERR_UNSUPPORTED: return "DIT_ERR_UNSUPPORTED: head dim or padded length not supported";
    case DIT_ERR_ALIGNMENT: return "DIT_ERR_ALIGNMENT: device pointer not aligned";
    case DIT_ERR_CUDA: return "DIT_ERR_CUDA: CUDA call or launch failed";
    case DIT_ERR_TIMEOUT: return "DIT_ERR_TIMEOUT: a kernel gave up on a bounded wait";
    default: return "unknown status";
  }
}

extern "C" int dit_last_cuda_error(void) { return t_last_cuda_error; }

extern "C" int dit_device_status(unsigned int* status_out, int clear) {
  if (!status_out) return DIT_ERR_INVALID_ARG;
  return cuda_status(read_device_status(status_out, clear != 0));
}

extern "C" int dit_rope_split_halves(const void* x, void* y, const float* cos_tab,
                                     const float* sin_tab, int B, int S, int H, int D,
                                     void* stream) {
  if (!x || !y || !cos_tab || !sin_tab || B < 1 || S < 1 || H < 1) return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(cos_tab, 16) || !aligned(sin_tab, 16))
    return DIT_ERR_ALIGNMENT;
  return cuda_status(launch_rope_split_halves(x, y, cos_tab, sin_tab, B, S, H, D,
                                              static_cast<cudaStream_t>(stream)));
}

extern "C" int dit_attn_fwd(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                            int H, int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                            const float* sin_q, const float* cos_k, const float* sin_k,
                            float softmax_scale, void* out, float* lse, void* stream) {
  int st = check_attn_shapes(q, k, v, B, Sq, Skv, H, D, q_valid_len, softmax_scale, out, lse);
  if (st != DIT_OK) return st;
  if (kv_valid_len < 0 || kv_valid_len > Skv) return DIT_ERR_INVALID_ARG;
  const int n_tables = (cos_q != nullptr) + (sin_q != nullptr) + (cos_k != nullptr) + (sin_k != nullptr);
  if (n_tables != 0 && n_tables != 4) return DIT_ERR_INVALID_ARG;
  if (n_tables == 4 && (!aligned(cos_q, 16) || !aligned(sin_q, 16) || !aligned(cos_k, 16) ||
                        !aligned(sin_k, 16)))
    return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, k, v, B, Sq, Skv, H, D, q_valid_len, kv_valid_len, nullptr,
             cos_q, sin_q, cos_k, sin_k, softmax_scale, out, lse, nullptr, nullptr, nullptr, 0.f,
             static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_attn_fwd(a, n_tables == 4 ? kModeRope : kModePlain));
}

extern "C" size_t dit_attn_workspace_bytes(int B, int Sq, int Skv, int H, int D) {
  if (B < 1 || Sq < 1 || Skv < 1 || H < 1 || (D != 64 && D != 128)) return 0;
  return attn_workspace_bytes(B, Sq, Skv, H, D);
}

extern "C" int dit_attn_fwd_ws(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                               int H, int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                               const float* sin_q, const float* cos_k, const float* sin_k,
                               float softmax_scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream) {
  int st = check_attn_shapes(q, k, v, B, Sq, Skv, H, D, q_valid_len, softmax_scale, out, lse);
  if (st != DIT_OK) return st;
  if (kv_valid_len < 0 || kv_valid_len > Skv) return DIT_ERR_INVALID_ARG;
  if (!cos_q || !sin_q || !cos_k || !sin_k || !workspace) return DIT_ERR_INVALID_ARG;
  if (workspace_bytes < attn_workspace_bytes(B, Sq, Skv, H, D)) return DIT_ERR_INVALID_ARG;
  // The rotation phase indexes (row, head, 8-pair chunk) of one batch in 32 bits.
  if (static_cast<long long>(Sq > Skv ? Sq : Skv) * H * (D / 16) >= (1ll << 30)) return DIT_ERR_UNSUPPORTED;
  if (!aligned(cos_q, 16) || !aligned(sin_q, 16) || !aligned(cos_k, 16) || !aligned(sin_k, 16) ||
      !aligned(workspace, 256))
    return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, k, v, B, Sq, Skv, H, D, q_valid_len, kv_valid_len, nullptr,
             cos_q, sin_q, cos_k, sin_k, softmax_scale, out, lse, workspace, nullptr, nullptr, 0.f,
             static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_attn_fwd(a, kModeRopeWs));
}

extern "C" size_t dit_attn_fixed_m_workspace_bytes(int B, int Sq, int Skv, int H, int D) {
  if (B < 1 || Sq < 1 || Skv < 1 || H < 1 || (D != 64 && D != 128)) return 0;
  return attn_fixed_m_workspace_bytes(B, Sq, Skv, H, D);
}

extern "C" int dit_attn_fwd_ws_fixed_m(const void* q, const void* k, const void* v, int B, int Sq,
                                       int Skv, int H, int D, int q_valid_len, int kv_valid_len,
                                       const float* cos_q, const float* sin_q, const float* cos_k,
                                       const float* sin_k, float softmax_scale, void* out, float* lse,
                                       void* workspace, size_t workspace_bytes,
                                       unsigned int* n_online, void* stream) {
  int st = check_attn_shapes(q, k, v, B, Sq, Skv, H, D, q_valid_len, softmax_scale, out, lse);
  if (st != DIT_OK) return st;
  if (kv_valid_len < 0 || kv_valid_len > Skv) return DIT_ERR_INVALID_ARG;
  if (!cos_q || !sin_q || !cos_k || !sin_k || !workspace) return DIT_ERR_INVALID_ARG;
  if (workspace_bytes < attn_fixed_m_workspace_bytes(B, Sq, Skv, H, D)) return DIT_ERR_INVALID_ARG;
  if (static_cast<long long>(Sq > Skv ? Sq : Skv) * H * (D / 16) >= (1ll << 30)) return DIT_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > kFixedMMaxHeads) return DIT_ERR_UNSUPPORTED;
  if (!aligned(cos_q, 16) || !aligned(sin_q, 16) || !aligned(cos_k, 16) || !aligned(sin_k, 16) ||
      !aligned(workspace, 256) || !aligned(n_online, 4))
    return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, k, v, B, Sq, Skv, H, D, q_valid_len, kv_valid_len, nullptr,
             cos_q, sin_q, cos_k, sin_k, softmax_scale, out, lse, workspace, nullptr, nullptr, 0.f,
             static_cast<cudaStream_t>(stream), n_online};
  return cuda_status(launch_attn_fwd(a, kModeRopeWsFixedM));
}

extern "C" size_t dit_attn_fp8_workspace_bytes(int B, int Sq, int Skv, int H, int D) {
  if (B < 1 || Sq < 1 || Skv < 1 || H < 1 || D != 128) return 0;
  return fp8_layout(B, Sq, Skv, H, D).total;
}

extern "C" int dit_attn_fwd_fp8(const void* q, const void* k, const void* v, int B, int Sq, int Skv,
                                int H, int D, int q_valid_len, int kv_valid_len, const float* cos_q,
                                const float* sin_q, const float* cos_k, const float* sin_k,
                                float softmax_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  int st = check_attn_shapes(q, k, v, B, Sq, Skv, H, D, q_valid_len, softmax_scale, out, lse);
  if (st != DIT_OK) return st;
  if (D != 128) return DIT_ERR_UNSUPPORTED;
  if (kv_valid_len < 0 || kv_valid_len > Skv || !workspace) return DIT_ERR_INVALID_ARG;
  const int n_tab = (cos_q != nullptr) + (sin_q != nullptr) + (cos_k != nullptr) + (sin_k != nullptr);
  if (n_tab != 0 && n_tab != 4) return DIT_ERR_INVALID_ARG;
  if (workspace_bytes < fp8_layout(B, Sq, Skv, H, D).total) return DIT_ERR_INVALID_ARG;
  if (n_tab == 4 && (!aligned(cos_q, 16) || !aligned(sin_q, 16) || !aligned(cos_k, 16) || !aligned(sin_k, 16)))
    return DIT_ERR_ALIGNMENT;
  if (!aligned(workspace, 256)) return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, k, v, B, Sq, Skv, H, D, q_valid_len, kv_valid_len, nullptr,
             cos_q, sin_q, cos_k, sin_k, softmax_scale, out, lse, workspace, nullptr, nullptr, 0.f,
             static_cast<cudaStream_t>(stream), nullptr};
  return cuda_status(launch_attn_fwd(a, kModeFp8));
}

extern "C" int dit_attn_fwd_ws_qknorm(const void* q, const void* k, const void* v, int B, int Sq,
                                      int Skv, int H, int D, int q_valid_len, int kv_valid_len,
                                      const float* norm_q, const float* norm_k, float eps,
                                      const float* cos_q, const float* sin_q, const float* cos_k,
                                      const float* sin_k, float softmax_scale, void* out, float* lse,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  int st = check_attn_shapes(q, k, v, B, Sq, Skv, H, D, q_valid_len, softmax_scale, out, lse);
  if (st != DIT_OK) return st;
  if (kv_valid_len < 0 || kv_valid_len > Skv) return DIT_ERR_INVALID_ARG;
  if (!cos_q || !sin_q || !cos_k || !sin_k || !workspace || !norm_q || !norm_k) return DIT_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return DIT_ERR_INVALID_ARG;
  if (workspace_bytes < attn_workspace_bytes(B, Sq, Skv, H, D)) return DIT_ERR_INVALID_ARG;
  if (static_cast<long long>(Sq > Skv ? Sq : Skv) * H * (D / 16) >= (1ll << 30)) return DIT_ERR_UNSUPPORTED;
  if (!aligned(cos_q, 16) || !aligned(sin_q, 16) || !aligned(cos_k, 16) || !aligned(sin_k, 16) ||
      !aligned(norm_q, 16) || !aligned(norm_k, 16) || !aligned(workspace, 256))
    return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, k, v, B, Sq, Skv, H, D, q_valid_len, kv_valid_len, nullptr,
             cos_q, sin_q, cos_k, sin_k, softmax_scale, out, lse, workspace, norm_q, norm_k, eps,
             static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_attn_fwd(a, kModeRopeWsNorm));
}

extern "C" int dit_qk_rmsnorm_rope(const void* x, void* y, const float* w, float eps,
                                   const float* cos_tab, const float* sin_tab, int B, int S, int H,
                                   int D, void* stream) {
  if (!x || !y || !w || !cos_tab || !sin_tab || B < 1 || S < 1 || H < 1) return DIT_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !std::isfinite(eps)) return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(w, 16) || !aligned(cos_tab, 16) || !aligned(sin_tab, 16))
    return DIT_ERR_ALIGNMENT;
  return cuda_status(launch_qk_rmsnorm_rope(x, y, w, eps, cos_tab, sin_tab, B, S, H, D,
                                            static_cast<cudaStream_t>(stream)));
}

extern "C" int dit_cross_attn_shortkv(const void* q, const void* k, const void* v, int B, int Sq,
                                      int Skv, int H, int D, int q_valid_len,
                                      const int32_t* kv_valid_len_dev, float softmax_scale,
                                      void* out, float* lse, void* stream) {
  int st = check_attn_shapes(q, k, v, B, Sq, Skv, H, D, q_valid_len, softmax_scale, out, lse);
  if (st != DIT_OK) return st;
  if (!kv_valid_len_dev) return DIT_ERR_INVALID_ARG;
  if (Skv > 512) return DIT_ERR_UNSUPPORTED;
  if (!aligned(kv_valid_len_dev, 4)) return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, k, v, B, Sq, Skv, H, D, q_valid_len, Skv, kv_valid_len_dev,
             nullptr, nullptr, nullptr, nullptr, softmax_scale, out, lse, nullptr, nullptr, nullptr,
             0.f, static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_cross_attn(a));
}

namespace {
// Shared checks and the plan of the sharded entry points.
int sharded_setup(int B, int Sq, int H, int D, int n_shards, const void* const* k_shards,
                  const void* const* v_shards, const int* shard_padded, const int* shard_valid,
                  const float* const* cos_k, const float* const* sin_k, bool need_ptrs, KeyShard* ks,
                  ShardPlan* plan) {
  if (B < 1 || Sq < 1 || H < 1 || n_shards < 1 || n_shards > 64 || !shard_padded || !shard_valid)
    return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  if ((Sq % 128) != 0 || H > 65535 || B > 65535) return DIT_ERR_UNSUPPORTED;
  if (need_ptrs && (!k_shards || !v_shards || !cos_k || !sin_k)) return DIT_ERR_INVALID_ARG;
  for (int s = 0; s < n_shards; ++s) {
    // an empty shard may have no rows at all (padded length 0); it is never read
    if (shard_padded[s] < 0 || (shard_padded[s] % 128) != 0) return DIT_ERR_UNSUPPORTED;
    if (shard_valid[s] < 0 || shard_valid[s] > shard_padded[s]) return DIT_ERR_INVALID_ARG;
    if (static_cast<long long>(shard_padded[s]) * H * (D / 16) >= (1ll << 30)) return DIT_ERR_UNSUPPORTED;
    ks[s].S_pad = shard_padded[s];
    ks[s].valid = shard_valid[s];
    if (need_ptrs && shard_padded[s] > 0) {
      if (!k_shards[s] || !v_shards[s] || !cos_k[s] || !sin_k[s]) return DIT_ERR_INVALID_ARG;
      if (!aligned(k_shards[s], 16) || !aligned(v_shards[s], 16) || !aligned(cos_k[s], 16) || !aligned(sin_k[s], 16))
        return DIT_ERR_ALIGNMENT;
      ks[s].k = k_shards[s];
      ks[s].v = v_shards[s];
      ks[s].cos_k = cos_k[s];
      ks[s].sin_k = sin_k[s];
    }
  }
  if (static_cast<long long>(Sq) * H * (D / 16) >= (1ll << 30)) return DIT_ERR_UNSUPPORTED;
  if (!plan_shards(B, Sq, H, D, n_shards, ks, 0, plan)) return DIT_ERR_UNSUPPORTED;
  return DIT_OK;
}
}  // namespace

extern "C" size_t dit_attn_sharded_workspace_bytes(int B, int Sq, int H, int D, int n_shards,
                                                   const int* shard_padded, const int* shard_valid) {
  KeyShard ks[64] = {};
  ShardPlan plan;
  if (sharded_setup(B, Sq, H, D, n_shards, nullptr, nullptr, shard_padded, shard_valid, nullptr, nullptr, false,
                    ks, &plan) != DIT_OK)
    return 0;
  return plan.total;
}

extern "C" int dit_attn_fwd_sharded(const void* q, int B, int Sq, int H, int D, int q_valid_len,
                                    int n_shards, const void* const* k_shards, const void* const* v_shards,
                                    const int* shard_padded, const int* shard_valid, const float* cos_q,
                                    const float* sin_q, const float* const* cos_k,
                                    const float* const* sin_k, float softmax_scale, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (!q || !out || !lse || !cos_q || !sin_q || !workspace) return DIT_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return DIT_ERR_INVALID_ARG;
  if (q_valid_len < 0 || q_valid_len > Sq) return DIT_ERR_INVALID_ARG;
  KeyShard ks[64] = {};
  ShardPlan plan;
  const int st = sharded_setup(B, Sq, H, D, n_shards, k_shards, v_shards, shard_padded, shard_valid, cos_k,
                               sin_k, true, ks, &plan);
  if (st != DIT_OK) return st;
  if (workspace_bytes < plan.total) return DIT_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(cos_q, 16) || !aligned(sin_q, 16) ||
      !aligned(workspace, 256))
    return DIT_ERR_ALIGNMENT;
  AttnArgs a{q, nullptr, nullptr, B, Sq, 0, H, D, q_valid_len, 0, nullptr,
             cos_q, sin_q, nullptr, nullptr, softmax_scale, out, lse, workspace, nullptr, nullptr, 0.f,
             static_cast<cudaStream_t>(stream), nullptr};
  return cuda_status(launch_attn_sharded(a, n_shards, ks, plan));
}

extern "C" int dit_attn_lse_merge(const void* partial_o, const float* partial_lse, int n, int B,
                                  int S, int H, int D, void* out, float* lse, void* stream) {
  if (!partial_o || !partial_lse || !out || !lse) return DIT_ERR_INVALID_ARG;
  if (n < 1 || n > 64 || B < 1 || S < 1 || H < 1) return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  if (!aligned(partial_o, 16) || !aligned(out, 16) || !aligned(partial_lse, 4) || !aligned(lse, 4))
    return DIT_ERR_ALIGNMENT;
  return cuda_status(launch_lse_merge(partial_o, partial_lse, n, B, S, H, D, out, lse,
                                      static_cast<cudaStream_t>(stream)));
}

extern "C" int dit_pad_tokens(const void* x, void* x_pad, int B, int L, int S_pad,
                              long long row_bytes, void* stream) {
  if (!x || !x_pad || B < 1 || L < 0 || L > S_pad || row_bytes < 1) return DIT_ERR_INVALID_ARG;
  return cuda_status(launch_copy_rows(x, x_pad, B, L, L, S_pad, row_bytes,
                                      static_cast<cudaStream_t>(stream)));
}

extern "C" int dit_unpad_tokens(const void* x_pad, void* x, int B, int L, int S_pad,
                                long long row_bytes, void* stream) {
  if (!x || !x_pad || B < 1 || L < 0 || L > S_pad || row_bytes < 1) return DIT_ERR_INVALID_ARG;
  return cuda_status(launch_copy_rows(x_pad, x, B, L, S_pad, L, row_bytes,
                                      static_cast<cudaStream_t>(stream)));
}

extern "C" int dit_exp2_fma_eval(const float* x, float* y, long long n, void* stream) {
  if (!x || !y || n < 0) return DIT_ERR_INVALID_ARG;
  if (!aligned(x, 4) || !aligned(y, 4)) return DIT_ERR_ALIGNMENT;
  if (n == 0) return DIT_OK;
  return cuda_status(launch_exp2_fma(x, y, n, static_cast<cudaStream_t>(stream)));
}

// dit_attn_fwd_ws with the workspace taken from a fixed device array instead of the caller.
namespace dit {
namespace {

__device__ __align__(256) unsigned char g_attn_static_scratch[DIT_ATTN_STATIC_SCRATCH_BYTES];

constexpr int kStaticScratchDevices = 64;
std::mutex g_static_scratch_mu;
void* g_static_scratch_ptr[kStaticScratchDevices] = {};

}  // namespace
}  // namespace dit

extern "C" int dit_attn_fwd_ws_static(const void* q, const void* k, const void* v, int B, int Sq,
                                      int Skv, int H, int D, int q_valid_len, int kv_valid_len,
                                      const float* cos_q, const float* sin_q, const float* cos_k,
                                      const float* sin_k, float softmax_scale, void* out,
                                      float* lse, void* stream) {
  if (B < 1 || Sq < 1 || Skv < 1 || H < 1) return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  if (attn_workspace_bytes(B, Sq, Skv, H, D) > DIT_ATTN_STATIC_SCRATCH_BYTES) return DIT_ERR_UNSUPPORTED;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e);
  if (dev < 0 || dev >= kStaticScratchDevices) return DIT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_scratch_mu);
    if (!g_static_scratch_ptr[dev]) {
      // Set-up, once per device, with that device current.
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
      if (e != cudaSuccess) return cuda_status(e);
      g_static_scratch_ptr[dev] = p;
    }
    scratch = g_static_scratch_ptr[dev];
  }
  return dit_attn_fwd_ws(q, k, v, B, Sq, Skv, H, D, q_valid_len, kv_valid_len, cos_q, sin_q, cos_k,
                         sin_k, softmax_scale, out, lse, scratch, DIT_ATTN_STATIC_SCRATCH_BYTES, stream);
}
