// tq_noalloc.cu -- decode attention for callers that cannot allocate device memory.
//
// tq_decode_attn needs a caller-provided workspace.  Some callers have no way
// to provide one: a serving runtime that hands all free HBM to its KV pool at
// start-up and forbids allocations afterwards, or a decode loop that may not
// call cudaMalloc because that call can synchronise the whole device.  For
// them, tq_decode_attn_noalloc runs the same kernels with their scratch
// in a fixed array compiled into this library (kNoallocScratchBytes per GPU,
// held by every GPU that loads the library until the process exits).
#include <mutex>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr size_t kNoallocScratchBytes = TQ_NOALLOC_SCRATCH_BYTES;   // 16 MiB per GPU
constexpr int kMaxDevices = 64;

// The scratch itself.  Host code must not use this name as an address: on
// the host it is only a stand-in for the symbol, so its device address is
// looked up with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (on the first call made with that device current).
cudaError_t scratch_for_current_device(void **addr) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" int tq_decode_attn_noalloc(const void *params, int d, const void *q, int dtype, int batch, int n_q_heads,
                                      int n_kv_heads, const void *k_pool, const void *v_pool, int64_t num_blocks,
                                      const int32_t *block_table, int max_blocks, const int32_t *ctx_lens,
                                      int max_ctx, float *out, int32_t *status, tq_stream_t stream) {
    if (!valid_d(d)) return TQ_ERR_HEAD_DIM;
    if (dtype != TQ_DTYPE_F32 && dtype != TQ_DTYPE_BF16) return TQ_ERR_DTYPE;
    if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || max_ctx < 0 || max_blocks <= 0 || num_blocks < 0)
        return TQ_ERR_INVALID;
    if (n_q_heads % n_kv_heads != 0 || n_q_heads / n_kv_heads > 8) return TQ_ERR_GQA;
    if (batch == 0) return TQ_OK;
    if (batch > 65535 || n_kv_heads > 65535) return TQ_ERR_INVALID;
    if (!params || !q || !k_pool || !v_pool || !block_table || !ctx_lens || !out) return TQ_ERR_INVALID;
    if (!aligned16(params) || !aligned16(k_pool) || !aligned16(v_pool)) return TQ_ERR_ALIGN;
    // The shape must fit the fixed scratch; nothing is allocated to make room.
    const size_t need = decode_workspace_bytes(d, batch, n_q_heads, max_ctx);
    if (need == 0 || need > kNoallocScratchBytes) return TQ_ERR_WORKSPACE;
    void *ws = nullptr;
    cudaError_t e = scratch_for_current_device(&ws);
    if (e != cudaSuccess) return TQ_ERR_CUDA;
    // Every scratch value the kernels read is written earlier in this same
    // call (the packs by the query prep, the chunk prefix and the partials by
    // the pass), so the contents left by a previous call need no clearing.
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    e = launch_qprep(d, dtype, params, q, batch, 1, n_q_heads, n_kv_heads, ws, st);
    if (e == cudaSuccess)
        e = launch_splitk(d, params, batch, 1, n_q_heads, n_kv_heads, k_pool, v_pool, num_blocks, block_table,
                          max_blocks, ctx_lens, 0, max_ctx, out, ws, status, st, true);
    return e == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}
