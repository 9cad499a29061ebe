// tq_hybrid.cu -- decode attention over a hybrid cache: the compressed history plus a window
// of the most recent tokens kept uncompressed (SwiftLM README: compression starts past 2048
// tokens, and attention covers the compressed history together with the recent "hot window"
// -- the --turbo-kv long-range recall note and the options table).
//
// One softmax runs over both parts.  The compressed pass writes each query row's output and
// the log-sum-exp of its scores; the window pass scores the window's dense K rows against the
// original-domain query (s = q.k / sqrt d, in log2 units) and leaves per-chunk online-softmax
// partials (m, l, acc); the merge combines
//   out = (o_c 2^(lse_c) + sum_chunks acc 2^m) / (2^(lse_c) + sum_chunks l 2^m)
// in log2 units.  Window slots are an unordered set (softmax does not depend on order), so a
// ring buffer of recent tokens can be passed as it is.
//
// Window pass: CTA (chunk, kv head, sequence) of 128 threads over kWinChunk tokens; thread t
// scores token t of the chunk for the group's G heads straight from global memory (one row,
// 16-byte loads), the CTA reduces max and sum per head, then thread c accumulates value column
// c from the chunk's V rows staged in shared memory.  The window is dense and read once, so
// plain FMA keeps pace with memory (G heads share every loaded row).
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kWinThreads = 128;
template <int D> __host__ __device__ constexpr int win_chunk() { return D == 128 ? 128 : 64; }

template <typename T> __device__ __forceinline__ void load8(const T *p, float (&v)[8]);
template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float (&v)[8]) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
template <> __device__ __forceinline__ void load8<float>(const float *p, float (&v)[8]) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Partial of chunk c for (sequence b, kv head kh): part[((b * hkv + kh) * nchunk + c) * G + h]
// = {m (log2), l, 0, 0, acc[D]}.
template <int D, int G, typename TQ, typename TW>
__global__ void __launch_bounds__(kWinThreads)
window_kernel(const TQ *__restrict__ q, const TW *__restrict__ wk, const TW *__restrict__ wv, int batch, int hq,
              int hkv, int win_cap, const int32_t *__restrict__ win_lens, int nchunk, float *__restrict__ part) {
    constexpr int CW = win_chunk<D>(), NT = kWinThreads, TPT = CW / NT == 0 ? 1 : CW / NT;
    constexpr float kLog2e = 1.4426950408889634f;
    extern __shared__ __align__(16) uint8_t smem[];
    float *sq = reinterpret_cast<float *>(smem);                 // [G][D], pre-scaled by log2e / sqrt d
    float *sp = sq + G * D;                                      // [G][CW] weights
    TW *sv = reinterpret_cast<TW *>(sp + G * CW);                // [CW][D] value rows
    __shared__ float sred[2][G][NT / 32];
    const int c = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int wl = win_lens[b];
    wl = wl < 0 ? 0 : (wl > win_cap ? win_cap : wl);
    const int t0 = c * CW, t1 = min(wl, t0 + CW);
    float *pout = part + (((size_t)b * hkv + kh) * nchunk + c) * G * (D + 4);
    if (t0 >= t1) {   // nothing in this chunk: an empty partial
        for (int i = tid; i < G; i += NT) {
            pout[(size_t)i * (D + 4)] = -INFINITY;
            pout[(size_t)i * (D + 4) + 1] = 0.f;
        }
        return;
    }
    const float qs = kLog2e * rsqrtf((float)D);
    for (int i = tid; i < G * D; i += NT) {
        const int h = i / D, dd = i % D;
        sq[i] = to_f32<TQ>(q[((size_t)b * hq + (size_t)kh * G + h) * D + dd]) * qs;
    }
    // stage the chunk's V rows (16-byte copies) while the scores are computed
    constexpr int ROWV = D * (int)sizeof(TW) / 16;
    for (int i = tid; i < (t1 - t0) * ROWV; i += NT) {
        const int r = i / ROWV, o = i % ROWV;
        cp_async16(reinterpret_cast<uint8_t *>(sv) + ((size_t)r * D * sizeof(TW)) + 16 * o,
                   reinterpret_cast<const uint8_t *>(wv + (((size_t)b * win_cap + t0 + r) * hkv + kh) * D) + 16 * o);
    }
    cp_async_commit();
    __syncthreads();
    // scores: thread handles tokens t0 + tid + NT * i
    float s[TPT][G];
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
        const int t = t0 + tid + NT * i;
#pragma unroll
        for (int h = 0; h < G; ++h) s[i][h] = -INFINITY;
        if (t < t1) {
            const TW *row = wk + (((size_t)b * win_cap + t) * hkv + kh) * D;
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) acc[h] = 0.f;
#pragma unroll 4
            for (int d0 = 0; d0 < D; d0 += 8) {
                float kv8[8];
                load8<TW>(row + d0, kv8);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[h] = fmaf(sq[h * D + d0 + e], kv8[e], acc[h]);
            }
#pragma unroll
            for (int h = 0; h < G; ++h) s[i][h] = acc[h];
        }
    }
    // per head: chunk max and sum over the CTA
    float m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float x = s[0][h];
#pragma unroll
        for (int i = 1; i < TPT; ++i) x = fmaxf(x, s[i][h]);
        x = warp_max(x);
        if (lane == 0) sred[0][h][warp] = x;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float x = sred[0][h][0];
#pragma unroll
        for (int w2 = 1; w2 < NT / 32; ++w2) x = fmaxf(x, sred[0][h][w2]);
        m[h] = x;   // finite: the chunk has at least one token
        float ps = 0.f;
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            const int tl = tid + NT * i;
            const float p = exp2f(s[i][h] - m[h]);   // 0 for tokens past the window (s = -inf)
            if (tl < CW) sp[h * CW + tl] = p;
            ps += p;
        }
        ps = warp_sum(ps);
        if (lane == 0) sred[1][h][warp] = ps;
    }
    cp_async_wait_all();
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float x = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NT / 32; ++w2) x += sred[1][h][w2];
        l[h] = x;
    }
    // values: thread handles columns tid + NT * j
    constexpr int CPT = D / NT;
    float acc[CPT][G];
#pragma unroll
    for (int j = 0; j < CPT; ++j)
#pragma unroll
        for (int h = 0; h < G; ++h) acc[j][h] = 0.f;
    const int nt = t1 - t0;
#pragma unroll 4
    for (int t = 0; t < nt; ++t) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const float v = to_f32<TW>(sv[(size_t)t * D + tid + NT * j]);
#pragma unroll
            for (int h = 0; h < G; ++h) acc[j][h] = fmaf(sp[h * CW + t], v, acc[j][h]);
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float *ph = pout + (size_t)h * (D + 4);
        if (tid == 0) {
            ph[0] = m[h];
            ph[1] = l[h];
        }
#pragma unroll
        for (int j = 0; j < CPT; ++j) ph[4 + tid + NT * j] = acc[j][h];
    }
}

// out[b][h] (the compressed pass's normalized output, lse_c its natural log-sum-exp) merged with
// the window partials, in place.  One warp per (sequence, query head).
template <int D>
__global__ void __launch_bounds__(128)
hybrid_merge_kernel(float *__restrict__ out, const float *__restrict__ lse, const float *__restrict__ part, int batch,
                    int hq, int hkv, int nchunk) {
    constexpr int R = D / 32;
    constexpr float kLog2e = 1.4426950408889634f;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= batch * hq) return;
    const int b = row / hq, h = row % hq, G = hq / hkv, kh = h / G, hg = h % G;
    const float lc = lse[row] * kLog2e;   // log2 units; -inf when the history is empty
    const float *pb = part + ((size_t)b * hkv + kh) * nchunk * G * (D + 4);
    float M = lc;
    for (int c = 0; c < nchunk; ++c) M = fmaxf(M, pb[((size_t)c * G + hg) * (D + 4)]);
    float *orow = out + (size_t)row * D;
    if (M == -INFINITY) {   // nothing at all to attend
#pragma unroll
        for (int r = 0; r < R; ++r) orow[32 * r + lane] = 0.f;
        return;
    }
    const float wc = (lc == -INFINITY) ? 0.f : exp2f(lc - M);
    float v[R], den = wc;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = orow[32 * r + lane] * wc;
    for (int c = 0; c < nchunk; ++c) {
        const float *ps = pb + ((size_t)c * G + hg) * (D + 4);
        const float mc = ps[0];
        if (mc == -INFINITY) continue;
        const float w = exp2f(mc - M);
        den = fmaf(ps[1], w, den);
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = fmaf(ps[4 + 32 * r + lane], w, v[r]);
    }
    const float inv = 1.f / den;
#pragma unroll
    for (int r = 0; r < R; ++r) orow[32 * r + lane] = v[r] * inv;
}

template <int D, int G, typename TQ, typename TW>
cudaError_t window_launch(const void *q, const void *wk, const void *wv, int batch, int hq, int hkv, int win_cap,
                          const int32_t *win_lens, int nchunk, float *part, cudaStream_t st) {
    constexpr int CW = win_chunk<D>();
    constexpr size_t smem = (size_t)G * D * 4 + (size_t)G * CW * 4 + (size_t)CW * D * sizeof(TW);
    auto kern = window_kernel<D, G, TQ, TW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(nchunk, hkv, batch), kWinThreads, smem, st>>>((const TQ *)q, (const TW *)wk, (const TW *)wv, batch, hq,
                                                             hkv, win_cap, win_lens, nchunk, part);
    return cudaGetLastError();
}

template <int D, typename TQ, typename TW>
cudaError_t window_any(int G, const void *q, const void *wk, const void *wv, int batch, int hq, int hkv, int win_cap,
                       const int32_t *win_lens, int nchunk, float *part, cudaStream_t st) {
#define TQ_WIN(GG) return window_launch<D, GG, TQ, TW>(q, wk, wv, batch, hq, hkv, win_cap, win_lens, nchunk, part, st)
    switch (G) {
        case 1: TQ_WIN(1);
        case 2: TQ_WIN(2);
        case 3: TQ_WIN(3);
        case 4: TQ_WIN(4);
        case 5: TQ_WIN(5);
        case 6: TQ_WIN(6);
        case 7: TQ_WIN(7);
        default: TQ_WIN(8);
    }
#undef TQ_WIN
}

template <int D>
cudaError_t window_dtypes(int q_dtype, int w_dtype, int G, const void *q, const void *wk, const void *wv, int batch,
                          int hq, int hkv, int win_cap, const int32_t *win_lens, int nchunk, float *part,
                          cudaStream_t st) {
    if (q_dtype == TQ_DTYPE_BF16)
        return w_dtype == TQ_DTYPE_BF16
                   ? window_any<D, __nv_bfloat16, __nv_bfloat16>(G, q, wk, wv, batch, hq, hkv, win_cap, win_lens,
                                                                nchunk, part, st)
                   : window_any<D, __nv_bfloat16, float>(G, q, wk, wv, batch, hq, hkv, win_cap, win_lens, nchunk,
                                                        part, st);
    return w_dtype == TQ_DTYPE_BF16
               ? window_any<D, float, __nv_bfloat16>(G, q, wk, wv, batch, hq, hkv, win_cap, win_lens, nchunk, part,
                                                    st)
               : window_any<D, float, float>(G, q, wk, wv, batch, hq, hkv, win_cap, win_lens, nchunk, part, st);
}

// ---------------------------------------------------------------- window upkeep
// The window is a ring keyed by position: token p of a sequence sits in window slot p mod win_cap
// while it is uncompressed.  Tokens 0 .. ctx - 1 are in the compressed history, ctx .. ctx + wl - 1
// in the window.  The window fills first (ctx = 0, slots 0 .. wl - 1); once it is full, every
// appended token pushes the oldest one, position ctx in slot ctx mod win_cap, into the history.
// A state is valid when 0 <= wl <= win_cap, ctx >= 0 and, unless the window is full,
// ctx mod win_cap = 0 (so that the window's slots are 0 .. wl - 1, the ones attention reads).

// 16-byte copy of n bytes (n a multiple of 16) by the CTA's threads
__device__ __forceinline__ void copy16(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src, size_t n) {
    for (size_t i = threadIdx.x; i < n / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(dst)[i] = reinterpret_cast<const uint4 *>(src)[i];
}

__device__ __forceinline__ bool window_state_ok(int ctx, int wl, int win_cap) {
    return ctx >= 0 && wl >= 0 && wl <= win_cap && (wl == win_cap || ctx % win_cap == 0);
}

// One CTA per sequence: a full window's oldest token (all kv heads) is copied into ek / ev and its
// position into epos (-1: nothing leaves the window); then the new token's rows go into its
// window slot (the freed one when the window was full) and the lengths are updated.  The
// encode of the leaving token reads ek / ev, so it may follow this kernel.  A state this call
// does not produce, or a full window whose leaving token has no block in the history (position
// past the block table, or a block id outside the pool), is flagged TQ_STATUS_BAD_SLOT and left
// as it is: nothing moves and neither length changes.
__global__ void __launch_bounds__(128)
window_step_kernel(const uint8_t *__restrict__ k_new, const uint8_t *__restrict__ v_new, size_t tok_bytes,
                   int win_cap, uint8_t *__restrict__ win_k, uint8_t *__restrict__ win_v, int32_t *ctx_lens,
                   int32_t *win_lens, const int32_t *__restrict__ block_table, int max_blocks, int64_t num_blocks,
                   uint8_t *__restrict__ ek, uint8_t *__restrict__ ev, int32_t *__restrict__ epos, int32_t *status) {
    const int b = blockIdx.x;
    const int ctx = ctx_lens[b], wl = win_lens[b];
    bool ok = window_state_ok(ctx, wl, win_cap);
    if (ok && wl == win_cap) {   // the leaving token goes to history position ctx: it needs a block
        const int lb = ctx / kBlock;
        const int64_t blk = lb < max_blocks ? (int64_t)block_table[(size_t)b * max_blocks + lb] : -1;
        ok = blk >= 0 && blk < num_blocks;
    }
    const bool full = ok && wl == win_cap;
    if (threadIdx.x == 0) {
        epos[b] = full ? ctx : -1;
        if (!ok) flag_status(status, TQ_STATUS_BAD_SLOT);
    }
    if (!ok) return;   // a state this call does not produce is left as it is
    const int slot = full ? ctx % win_cap : wl;
    const size_t at = ((size_t)b * win_cap + slot) * tok_bytes;
    if (full) {
        copy16(ek + (size_t)b * tok_bytes, win_k + at, tok_bytes);
        copy16(ev + (size_t)b * tok_bytes, win_v + at, tok_bytes);
    }
    __syncthreads();   // the leaving rows are copied (and every thread has read ctx and wl)
    copy16(win_k + at, k_new + (size_t)b * tok_bytes, tok_bytes);
    copy16(win_v + at, v_new + (size_t)b * tok_bytes, tok_bytes);
    if (threadIdx.x == 0) {
        ctx_lens[b] = ctx + (full ? 1 : 0);
        win_lens[b] = full ? win_cap : wl + 1;
    }
}

size_t round16(size_t n) { return (n + 15) / 16 * 16; }

}  // namespace

size_t hybrid_append_scratch_bytes(int d, int batch, int hkv, int dtype) {
    const size_t tok = (size_t)hkv * d * (dtype == TQ_DTYPE_BF16 ? 2 : 4);
    return round16((size_t)batch * sizeof(int32_t)) + 2 * round16((size_t)batch * tok);
}

cudaError_t launch_hybrid_append(int d, int dtype, const void *params, const void *k_new, const void *v_new, int batch,
                                 int hkv, void *win_k, void *win_v, int win_cap, int32_t *win_lens,
                                 const int32_t *block_table, int max_blocks, int32_t *ctx_lens, void *k_pool,
                                 void *v_pool, int64_t num_blocks, void *scratch, int32_t *status, cudaStream_t st) {
    const size_t tok = (size_t)hkv * d * (dtype == TQ_DTYPE_BF16 ? 2 : 4);
    uint8_t *sc = static_cast<uint8_t *>(scratch);
    int32_t *epos = reinterpret_cast<int32_t *>(sc);
    uint8_t *ek = sc + round16((size_t)batch * sizeof(int32_t)), *ev = ek + round16((size_t)batch * tok);
    window_step_kernel<<<batch, 128, 0, st>>>(static_cast<const uint8_t *>(k_new), static_cast<const uint8_t *>(v_new),
                                              tok, win_cap, static_cast<uint8_t *>(win_k), static_cast<uint8_t *>(win_v),
                                              ctx_lens, win_lens, block_table, max_blocks, num_blocks, ek, ev, epos,
                                              status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the leaving tokens go into the history at their positions (sequences with epos < 0 are skipped)
    return launch_append(d, dtype, params, ek, ev, batch, hkv, block_table, max_blocks, epos, k_pool, v_pool,
                         num_blocks, status, st);
}

int hybrid_nchunk(int d, int win_cap) {
    const int cw = d == 128 ? win_chunk<128>() : win_chunk<256>();
    return win_cap <= 0 ? 0 : (win_cap + cw - 1) / cw;
}

size_t hybrid_part_bytes(int d, int batch, int hq, int win_cap) {
    return (size_t)batch * hq * hybrid_nchunk(d, win_cap) * (d + 4) * sizeof(float);
}

cudaError_t launch_hybrid_window(int d, int q_dtype, int w_dtype, const void *q, const void *wk, const void *wv,
                                 int batch, int hq, int hkv, int win_cap, const int32_t *win_lens, float *part,
                                 float *out, const float *lse, cudaStream_t st) {
    const int nchunk = hybrid_nchunk(d, win_cap), G = hq / hkv;
    cudaError_t e = cudaSuccess;
    if (nchunk > 0)
        e = d == 128 ? window_dtypes<128>(q_dtype, w_dtype, G, q, wk, wv, batch, hq, hkv, win_cap, win_lens, nchunk,
                                          part, st)
                     : window_dtypes<256>(q_dtype, w_dtype, G, q, wk, wv, batch, hq, hkv, win_cap, win_lens, nchunk,
                                          part, st);
    if (e != cudaSuccess) return e;
    const int rows = batch * hq;
    if (d == 128) hybrid_merge_kernel<128><<<(rows + 3) / 4, 128, 0, st>>>(out, lse, part, batch, hq, hkv, nchunk);
    else hybrid_merge_kernel<256><<<(rows + 3) / 4, 128, 0, st>>>(out, lse, part, batch, hq, hkv, nchunk);
    return cudaGetLastError();
}

}  // namespace tq
