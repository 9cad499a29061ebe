// tq_internal.cuh -- layout constants and device helpers shared by the kernels.
//
// Packed layout of one record (16 token slots of one block, one kv head):
//   K: 4-bit fields, one per (slot, coordinate): cell bits 0..2 and the QJL sign bit 3,
//      8*d bytes, then 16 x {fp16 ||x||, fp16 ||r||}.
//   V: 3-bit cells, 6*d bytes, then 16 x fp16 ||v||.
// The cell region is an array of 32-bit words grouped by a lane L = 4*gid + tig.
//   K: coordinate i = 16*ks + c, c = 2*tig + e + 8*h, of slot t = gid + 8*r is field
//      f = 4*(ks&1) + e + 2*h (bits 4f..4f+3) of word (L*2 + r)*(d/32) + (ks>>1).
//   V: coordinate i = 16*mt + gid + 8*rr has lane slot s = 2*mt + rr, cut into groups of
//      16 (g = s>>4, sg = s&15); slot t has tig = (t&7)>>1, pair P = t>>3, e = t&1.  For
//      sg < 12 the cell is field f = 4*((sg>>1)&1) + 2*e + (sg&1), bits 0..2, of word
//      (L*2 + P)*3*(d/128) + 3*g + (sg>>2); for sg >= 12 its bit p is bit 3 of field
//      f = 4*((sg-12)>>1) + 2*e + (sg&1) of word ... + 3*g + p.
// Every byte belongs to one token slot, so slots are written independently with byte (V) or
// word (K) stores.  Four fields of a word are the PRMT selector of a table lookup in the
// decode kernels; the lookups and byte interleaves give f16x2 operand registers of the
// m16n8k16 mma.sync (K: token rows x coordinate columns; V: coordinate rows x token columns).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

constexpr uint32_t kParamsMagic = 0x31505154u;   // "TQP1"
constexpr int kBlock = 16;

// Device params header (256 bytes); D signs, S and S^T follow.
struct ParamsHeader {
    uint32_t magic;
    int32_t d;
    int32_t reserved[2];
    float centroid[8];     // ascending, unit variance
    float threshold[8];    // 7 used: midpoints of neighbouring centroids
    double centroid64[8];  // the same centroids before rounding to fp32
    uint32_t one16x2;      // 0x3C003C00: f16x2 {1, 1}
    uint32_t lut_lo[2];    // byte j: low byte of the f16 T[j] = f16(alpha * centroid[j]), j = 0..7
    uint32_t lut_hi[2];    // byte j: high byte of T[j]
    float inv_alpha;       // 1 / alpha (T[j] * inv_alpha = centroid[j] within 2e-5)
    uint16_t t16[8];       // T[j] as binary16 bits
    float pad[18];
};
static_assert(sizeof(ParamsHeader) == 256, "params header must be 256 bytes");

// Device params: header, D signs (fp32 +-1), S row-major, S transposed, then the QJL offset
// weights w (fp32, d): w_j = sum of S[k][j] over the coordinates k at field positions 0..2 of
// their K record word (qjl_pos below), so that the decode's offset constant of a query is
// 2^-16 <w, qbar> (the sum of u_k = (S qbar)_k over those coordinates).
__host__ __device__ constexpr size_t params_off_D(int /*d*/) { return 256; }
__host__ __device__ constexpr size_t params_off_S(int d) { return 256 + 4 * (size_t)d; }
__host__ __device__ constexpr size_t params_off_ST(int d) { return params_off_S(d) + 4 * (size_t)d * d; }
__host__ __device__ constexpr size_t params_off_W(int d) { return params_off_ST(d) + 4 * (size_t)d * d; }
__host__ __device__ constexpr size_t params_total(int d) { return params_off_W(d) + 4 * (size_t)d; }

// Field position (0..3) of coordinate k's QJL bit within its K record word's nibble group:
// coordinate 16 s + c sits in field 4 (s & 1) + (c & 1) + 2 (c >> 3), position = field & 3.
__host__ __device__ constexpr int qjl_pos(int k) { return (k & 1) + 2 * ((k & 15) >> 3); }

__host__ __device__ constexpr size_t k_record(int d) { return 8 * (size_t)d + 4 * kBlock; }
__host__ __device__ constexpr size_t v_record(int d) { return 6 * (size_t)d + 2 * kBlock; }

inline bool valid_d(int d) { return d == 128 || d == 256; }

// ---------------------------------------------------------------- value loads

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- lane -> coordinate maps
// Warp-per-vector encoders hold R = d/32 coordinates per lane; coordinate
// kdim(lane, r) / vdim(lane, r) is chosen so that __ballot_sync over register r
// yields one packed word (K) or four packed bytes (V) directly.

template <int D>
__device__ __forceinline__ int kdim(int lane, int r) {
    const int e = lane >> 4, h = (lane >> 3) & 1, s = 8 * (r >> 2) + (lane & 7), tig = r & 3;
    return 16 * s + 8 * h + 2 * tig + e;
}

template <int D>
__device__ __forceinline__ int vdim(int lane, int r) {
    constexpr int NM = D / 128;
    int beta = lane >> 3, q = lane & 7;
    int tau = 4 * r + beta;
    int mhi = tau % NM, rh = (tau / NM) & 1, gid = tau / (2 * NM);
    int mt = 8 * mhi + q;
    return 16 * mt + gid + 8 * rh;
}

// In-register fast Walsh-Hadamard transform (Sylvester order, unnormalised)
// of a d-vector spread over a warp as v[r] at lane l.  Each index bit of the
// coordinate is either a lane bit (butterfly through a shuffle) or a register
// bit (butterfly inside the thread); since H is the Kronecker product of one
// 2x2 butterfly per index bit, any bijective lane/register map is handled by
// running every lane-bit stage and every register-bit stage once.
template <int R>
__device__ __forceinline__ void fwht_warp(float (&v)[R], int lane) {
#pragma unroll
    for (int x = 0; x < 5; ++x) {
        const int m = 1 << x;
        const bool upper = (lane >> x) & 1;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            float w = __shfl_xor_sync(0xffffffffu, v[r], m);
            v[r] = upper ? (w - v[r]) : (v[r] + w);
        }
    }
#pragma unroll
    for (int y = 1; y < R; y <<= 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if ((r & y) == 0) {
                float a = v[r], b = v[r | y];
                v[r] = a + b;
                v[r | y] = a - b;
            }
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, m));
    return x;
}

// Walsh coefficients A0..A3 of the 8 levels (c[k] = sum_m A_m sigma_m(k)).
__device__ __forceinline__ void walsh4(const float *cen, float (&A)[4]) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float s0 = (k & 1) ? 1.f : -1.f, s1 = (k & 2) ? 1.f : -1.f, s2 = (k & 4) ? 1.f : -1.f;
        a0 += cen[k] * s0;
        a1 += cen[k] * s1;
        a2 += cen[k] * s2;
        a3 += cen[k] * s0 * s1 * s2;
    }
    A[0] = a0 * 0.125f;
    A[1] = a1 * 0.125f;
    A[2] = a2 * 0.125f;
    A[3] = a3 * 0.125f;
}

__device__ __forceinline__ void flag_status(int32_t *status, int bits) {
    if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------- async copies

// Programmatic dependent launch.  A prep kernel lets the decode pass launched after it (with
// cudaLaunchAttributeProgrammaticStreamSerialization) start early; the pass waits for the
// prep grid's completion and memory before it reads anything the prep wrote.  Both are no-ops
// for a launch without the attribute.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_n() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---------------------------------------------------------------- projections by S
// out[v][k] = sum_i S[k][i] x[v][i] for NV vectors x[v][*] in shared memory,
// thread t of NT computing rows k = t + NT*u.  S^T (row i = column i of S)
// is read from shared memory: either all of it (resident, d*d floats) or in
// double-buffered chunks of kProjRows rows copied from global memory.
constexpr int kProjRows = 32;

template <int D, int NV, int NT>
__device__ __forceinline__ void project_rows(const float *sST_rows, int i0, int nrows, const float (*x)[D],
                                             float (&acc)[D / NT][NV]) {
    constexpr int KPT = D / NT;
    for (int i = 0; i < nrows; i += 4) {
        float sv[KPT][4];
#pragma unroll
        for (int u = 0; u < KPT; ++u)
#pragma unroll
            for (int c = 0; c < 4; ++c) sv[u][c] = sST_rows[(size_t)(i + c) * D + threadIdx.x + NT * u];
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float4 xv = *reinterpret_cast<const float4 *>(&x[v][i0 + i]);
#pragma unroll
            for (int u = 0; u < KPT; ++u) {
                acc[u][v] = fmaf(sv[u][0], xv.x, acc[u][v]);
                acc[u][v] = fmaf(sv[u][1], xv.y, acc[u][v]);
                acc[u][v] = fmaf(sv[u][2], xv.z, acc[u][v]);
                acc[u][v] = fmaf(sv[u][3], xv.w, acc[u][v]);
            }
        }
    }
}

// Copy rows [i0, i0 + n) of S^T from global to shared memory (one commit group).
template <int D, int NT>
__device__ __forceinline__ void stage_st_rows(float *dst, const float *gST, int i0, int n) {
    const int chunks = n * D / 4;            // 16-byte pieces
    const float *src = gST + (size_t)i0 * D;
    for (int c = threadIdx.x; c < chunks; c += NT) cp_async16(dst + 4 * c, src + 4 * c);
    cp_async_commit();
}

// Streamed projection: S^T passes through sbuf (2 x ROWS x D floats, or
// ROWS x D when one chunk holds all of S^T).  Every thread of the CTA must
// call it (it synchronises the CTA).
template <int D, int NV, int NT, int ROWS = kProjRows>
__device__ __forceinline__ void project_streamed(const float *gST, float *sbuf, const float (*x)[D],
                                                 float (&acc)[D / NT][NV]) {
    constexpr int NCHUNK = D / ROWS;
    stage_st_rows<D, NT>(sbuf, gST, 0, ROWS);
#pragma unroll 1
    for (int c = 0; c < NCHUNK; ++c) {
        if (c + 1 < NCHUNK) {
            stage_st_rows<D, NT>(sbuf + (size_t)((c + 1) & 1) * ROWS * D, gST, (c + 1) * ROWS, ROWS);
            cp_async_wait_1();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        project_rows<D, NV, NT>(sbuf + (size_t)(c & 1) * ROWS * D, c * ROWS, ROWS, x, acc);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- decode work split (stream-K)
__host__ __device__ constexpr int kPartStride(int d) { return d + 4; }   // partial: m, l, pad, pad, acc[d]
constexpr int kMaxSms = 160;               // SMs a decode pass uses at most (GB300 has 152); bounds the workspace

// Stream-K ranges: CTA c of P covers global chunks [sk_begin(c), sk_begin(c+1)).
__host__ __device__ inline int64_t sk_begin(int c, int P, int64_t W) { return (int64_t)c * W / P; }
// the CTA whose range holds chunk x (0 <= x < W)
__device__ inline int sk_cta_of(int64_t x, int P, int64_t W) { return (int)(((x + 1) * P - 1) / W); }
__device__ inline int clamp_len(int L, int max_ctx) { return L < 0 ? 0 : (L > max_ctx ? max_ctx : L); }

// (w & mask) ^ base as a single LOP3 (base held in a register by the caller)
__device__ __forceinline__ uint32_t lop_and_xor(uint32_t w, uint32_t mask, uint32_t base) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(w), "r"(mask), "r"(base));
    return d;
}

// Context length attended for sequence b: the stored length c (plus ctx_add, 1 when the
// step appends a token first), clamped to [0, max_ctx]; c < 0 means nothing to attend.
__device__ inline int attended_len(int c, int ctx_add, int max_ctx) {
    return c < 0 ? 0 : clamp_len(c + ctx_add, max_ctx);
}

__device__ __forceinline__ int64_t warp_sum_i64(int64_t x) {
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
}

// The pass's stream-K schedule, worked out by every CTA of the pass from the lengths alone:
// W = chunks in all (hkv * ceil(len_b / chunk) per sequence b, in (sequence, kv head, chunk)
// order), P = min(W, grid) working CTAs, and for this CTA (if it works) the sequence b0 holding
// its first chunk sk_begin(cta, P, W) and that sequence's first chunk ub0.  A block-wide scan
// over the sequences in tiles of NT threads, stopping at the tile that holds the CTA's first
// chunk; when cpre is given, CTA 0 scans every tile and writes the prefix (cpre[b] = first
// chunk of sequence b, cpre[batch] = W) for the merge kernel.
struct PassSched {
    int64_t W;
    int P;
    int b0;
    int64_t ub0;
};
#ifndef TQ_SCHED_NOINLINE
#define TQ_SCHED_NOINLINE 1   // the schedule as a call: keeps its registers out of the pass loop's allocation
#endif
template <int NT>
#if TQ_SCHED_NOINLINE
__device__ __noinline__
#else
__device__ __forceinline__
#endif
PassSched pass_schedule(const int32_t *__restrict__ ctx_lens, int ctx_add, int batch, int hkv,
                                   int max_ctx, int chunk, int64_t *__restrict__ cpre) {
    constexpr int NWP = NT / 32;
    __shared__ int64_t s_red[NWP];
    __shared__ int64_t s_hit[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto nch = [&](int b) -> int64_t {
        return b < batch ? (int64_t)hkv * ((attended_len(ctx_lens[b], ctx_add, max_ctx) + chunk - 1) / chunk) : 0;
    };
    int64_t x = 0;
    for (int b = tid; b < batch; b += NT) x += nch(b);
    x = warp_sum_i64(x);
    if (lane == 0) s_red[warp] = x;
    if (tid == 0) s_hit[0] = -1;
    __syncthreads();
    PassSched r;
    r.W = 0;
#pragma unroll
    for (int w = 0; w < NWP; ++w) r.W += s_red[w];
    r.P = (int)(r.W < (int64_t)gridDim.x ? r.W : (int64_t)gridDim.x);
    r.b0 = -1;
    r.ub0 = 0;
    __syncthreads();   // s_red is reused below
    const bool all = (blockIdx.x == 0 && cpre != nullptr);
    if ((int)blockIdx.x >= r.P && !all) return r;
    const int64_t g0 = (r.P > 0) ? sk_begin((int)blockIdx.x, r.P, r.W) : 0;
    if (all && tid == 0) cpre[0] = 0;
    int64_t carry = 0;
    for (int base = 0; base < batch; base += NT) {
        const int b = base + tid;
        const int64_t own = nch(b);
        int64_t v = own;   // inclusive scan of the warp
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, v, m);
            if (lane >= m) v += y;
        }
        if (lane == 31) s_red[warp] = v;
        __syncthreads();
        int64_t off = carry, tot = 0;
#pragma unroll
        for (int w = 0; w < NWP; ++w) {
            off += (w < warp) ? s_red[w] : 0;
            tot += s_red[w];
        }
        const int64_t incl = off + v;
        if (b < batch) {
            if (all) cpre[b + 1] = incl;
            if (incl > g0 && incl - own <= g0) {   // the one sequence holding chunk g0
                s_hit[0] = b;
                s_hit[1] = incl - own;
            }
        }
        carry += tot;
        __syncthreads();   // s_red is read, s_hit is written
        if (!all && s_hit[0] >= 0) break;
    }
    r.b0 = (int)s_hit[0];
    r.ub0 = s_hit[1];
    return r;
}

// ---------------------------------------------------------------- launchers (defined in the .cu files)

cudaError_t launch_encode(bool is_k, int d, int dtype, const void *params, const void *x, int64_t n_tokens,
                          int n_heads, const int64_t *slots, void *pool, int64_t num_blocks, int32_t *status,
                          cudaStream_t st);
cudaError_t launch_append(int d, int dtype, const void *params, const void *k_new, const void *v_new, int batch,
                          int n_heads, const int32_t *bt, int max_blocks, const int32_t *ctx, void *kp, void *vp,
                          int64_t num_blocks, int32_t *status, cudaStream_t st);
cudaError_t launch_dequant(bool is_k, int d, int out_dtype, const void *params, const void *pool, int64_t num_blocks,
                           int n_heads, const int32_t *block_ids, int n_ids, void *out, int32_t *status,
                           cudaStream_t st);
size_t decode_workspace_bytes(int d, int batch, int hq, int max_ctx);
// Hybrid attention: the window pass and the merge (tq_hybrid.cu).  `out` holds the compressed
// pass's output and `lse` its log-sum-exp on entry; `part` holds hybrid_part_bytes().
size_t hybrid_part_bytes(int d, int batch, int hq, int win_cap);
cudaError_t launch_hybrid_window(int d, int q_dtype, int w_dtype, const void *q, const void *wk, const void *wv,
                                 int batch, int hq, int hkv, int win_cap, const int32_t *win_lens, float *part,
                                 float *out, const float *lse, cudaStream_t st);
// One CTA whose bounded mbarrier wait runs out (tq_encode.cu): sets TQ_STATUS_TIMEOUT.
cudaError_t launch_wait_timeout_selftest(int32_t *status, cudaStream_t st);
// Window upkeep of the hybrid cache (tq_hybrid.cu): a full window's oldest token into the paged
// history, then the new token into the window; lengths updated on the device.
size_t hybrid_append_scratch_bytes(int d, int batch, int hkv, int dtype);
cudaError_t launch_hybrid_append(int d, int dtype, const void *params, const void *k_new, const void *v_new, int batch,
                                 int hkv, void *win_k, void *win_v, int win_cap, int32_t *win_lens,
                                 const int32_t *block_table, int max_blocks, int32_t *ctx_lens, void *k_pool,
                                 void *v_pool, int64_t num_blocks, void *scratch, int32_t *status, cudaStream_t st);
// Decode launches take q_len queries per sequence (q[b][i][h], out[b][i][h]); query i attends
// the first L - (q_len - 1 - i) of the sequence's L attended tokens.  The workspace is laid
// out for batch sequences of q_len * hq query rows.
// launch_splitk's `early`: the launch before it on the stream is this library's query prep or
// step prep (an ordinary launch that writes neither the lengths nor the block table), so the pass
// may read those before waiting for it.  False after any other kernel.
cudaError_t launch_qprep(int d, int dtype, const void *params, const void *q, int batch, int q_len, int hq, int hkv,
                         void *ws, cudaStream_t st);
cudaError_t launch_splitk(int d, const void *params, int batch, int q_len, int hq, int hkv, const void *k_pool,
                          const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                          const int32_t *ctx_lens, int ctx_add, int max_ctx, float *out, void *ws, int32_t *status,
                          cudaStream_t st, bool early, float *lse = nullptr);
cudaError_t launch_step(int d, int dtype, const void *params, const void *k_new, const void *v_new, const void *q,
                        int batch, int q_len, int hq, int hkv, const int32_t *block_table, int max_blocks,
                        const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool, int64_t num_blocks,
                        float *out, void *ws, int32_t *status, cudaStream_t st);

// PRMT in its default mode: byte k of the result is byte (c >> 4k) & 7 of {b:a} (the
// selector's bit 4k+3 must be clear, or the byte's sign is replicated instead).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

}  // namespace tq
