// tq_gq.cuh -- host-side interface of the group-quantised KV cache (the comparator that
// SwiftLM's README sets beside TurboQuant: per-request "kv_bits" 4 or 8 with "kv_group_size",
// default 64, MLX's standard group quantization; the lilting.ch article's "TurboQuant
// V2+V3ハイブリッド実装" table calls the linear affine route V2).
//
// Record of one (block, kv head), 16 slots:
//   codes  [16][d bits / 8]      4-bit: element 2j in the low nibble of byte j; 8-bit: one byte each
//   params [16][d / group][2]    fp16 (scale, bias) per group; value = scale * code + bias
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace tq {

inline bool gq_valid(int d, int bits, int group) {
    return (d == 128 || d == 256) && (bits == 4 || bits == 8) &&
           (group == 32 || group == 64 || group == 128) && group <= d;
}
inline size_t gq_region_bytes(int d, int bits, int group) {
    return 16 * ((size_t)d * bits / 8 + 4 * (size_t)(d / group));
}
constexpr int kGqChunk = 128;   // tokens per CTA of the decode pass
inline int gq_nchunk(int max_ctx) { return (max_ctx + kGqChunk - 1) / kGqChunk; }
inline int gq_group_pad(int g) { return g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8; }
inline size_t gq_workspace_bytes(int d, int batch, int hq, int hkv, int max_ctx) {
    return (size_t)batch * hkv * gq_nchunk(max_ctx) * gq_group_pad(hq / hkv) * (d + 4) * sizeof(float);
}

cudaError_t launch_gq_encode(int d, int bits, int group, int dtype, const void *x, int64_t n_tokens, int hkv,
                             const int64_t *slots, uint8_t *pool, int64_t num_blocks, int32_t *status,
                             cudaStream_t st);
cudaError_t launch_gq_decode(int d, int bits, int group, int dtype, const void *q, int batch, int hq, int hkv,
                             const uint8_t *k_pool, const uint8_t *v_pool, int64_t num_blocks,
                             const int32_t *block_table, int max_blocks, const int32_t *ctx_lens, int max_ctx,
                             float *out, float *part, int32_t *status, cudaStream_t st);

}  // namespace tq
