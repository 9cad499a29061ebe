// tq_gq.cu -- the group-quantised KV comparator: encode K or V into paged records and decode
// attention over them.  (SwiftLM README, per-request parameters "kv_bits" (4 or 8) and
// "kv_group_size" (default 64): standard group quantization from token 0, "~2-4x vs FP16";
// lilting.ch "TurboQuant V2+V3ハイブリッド実装": the V2 route is linear affine quantization.)
//
// Per group of `group` consecutive coordinates: scale = fp16((max - min) / (2^bits - 1)),
// bias = fp16(min), code = clamp(rint((x - bias) / scale), 0, 2^bits - 1), every step in fp32
// round-to-nearest; a group whose fp16 scale is 0 gets code 0.  A decoded coordinate is
// scale * code + bias.  Attention runs in the original domain (no rotation).
//
// Encode: one warp per (token, kv head) vector, d/32 consecutive coordinates per lane, the group
// min and max by xor shuffles among the group's lanes.
// Decode: CTA (chunk of 128 tokens, kv head, sequence).  Thread t scores token t for the G query
// heads straight from its codes in global memory,
//   q.k = sum_g ( scale_g sum_{i in g} q_i code_i + bias_g sum_{i in g} q_i ),
// the CTA reduces max and sum per head, the chunk's value codes are staged in shared memory,
// and thread c accumulates coordinate c as sum_t (w_t scale_t) code_tc + sum_t w_t bias_t.
// Per-chunk partials (m, l, acc) in log2 units are merged per (sequence, query head).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_gq.cuh"
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kGqThreads = 128;
constexpr float kGqLog2e = 1.4426950408889634f;

template <int E>
__device__ __forceinline__ void load_e(const float *p, float (&v)[E]) {
#pragma unroll
    for (int i = 0; i < E; i += 4) {
        const float4 a = *reinterpret_cast<const float4 *>(p + i);
        v[i] = a.x;
        v[i + 1] = a.y;
        v[i + 2] = a.z;
        v[i + 3] = a.w;
    }
}
template <int E>
__device__ __forceinline__ void load_e(const __nv_bfloat16 *p, float (&v)[E]) {
    uint32_t w[E / 2];
    if constexpr (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        w[0] = u.x;
        w[1] = u.y;
    } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        w[0] = u.x;
        w[1] = u.y;
        w[2] = u.z;
        w[3] = u.w;
    }
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// Exact float of a small unsigned integer n < 2^23: 2^23 + n by its bit pattern, minus 2^23.
__device__ __forceinline__ float small_uint_to_float(uint32_t n) {
    return __uint_as_float(0x4B000000u | n) - 8388608.f;
}

template <int D, int BITS, typename T>
__global__ void __launch_bounds__(kGqThreads)
gq_encode_kernel(const T *__restrict__ x, int64_t n_vec, int hkv, int gshift, const int64_t *__restrict__ slots,
                 uint8_t *__restrict__ pool, int64_t num_blocks, int32_t *__restrict__ status) {
    constexpr int E = D / 32, CB = D * BITS / 8, LB = E * BITS / 8;   // per lane: coordinates, code bytes
    constexpr float kTop = (float)((1 << BITS) - 1);
    const int lane = threadIdx.x & 31;
    const int ng = D >> gshift, lpg = (1 << gshift) / E;   // groups per vector, lanes per group
    const size_t region = (size_t)kBlock * (CB + 4 * ng);
    const int64_t stride = (int64_t)gridDim.x * (kGqThreads / 32);
    for (int64_t v = (int64_t)blockIdx.x * (kGqThreads / 32) + (threadIdx.x >> 5); v < n_vec; v += stride) {
        const int64_t tok = v / hkv;
        const int h = (int)(v - tok * hkv);
        const int64_t slot = slots[tok];
        if (slot < 0) continue;   // padding
        if (slot >= num_blocks * kBlock) {
            if (lane == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
            continue;
        }
        float xv[E];
        load_e<E>(x + v * D + lane * E, xv);
        float mn = xv[0], mx = xv[0];
#pragma unroll
        for (int e = 1; e < E; ++e) {
            mn = fminf(mn, xv[e]);
            mx = fmaxf(mx, xv[e]);
        }
        for (int o = 1; o < lpg; o <<= 1) {
            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        }
        const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), kTop));
        const __half z16 = __float2half_rn(mn);
        const float sf = __half2float(s16), zf = __half2float(z16);
        uint64_t pk = 0;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float c = 0.f;
            if (sf > 0.f) c = fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(xv[e], zf), sf)), 0.f), kTop);
            pk |= (uint64_t)(uint32_t)c << (e * BITS);
        }
        uint8_t *reg = pool + ((size_t)(slot / kBlock) * hkv + h) * region;
        const int off = (int)(slot % kBlock);
        uint8_t *cp = reg + (size_t)off * CB + lane * LB;
        if constexpr (LB == 2) {
            *reinterpret_cast<uint16_t *>(cp) = (uint16_t)pk;
        } else if constexpr (LB == 4) {
            *reinterpret_cast<uint32_t *>(cp) = (uint32_t)pk;
        } else {
            *reinterpret_cast<uint2 *>(cp) = make_uint2((uint32_t)pk, (uint32_t)(pk >> 32));
        }
        if ((lane & (lpg - 1)) == 0)
            *reinterpret_cast<__half2 *>(reg + (size_t)kBlock * CB + ((size_t)off * ng + lane / lpg) * 4) =
                __halves2half2(s16, z16);
    }
}

// Partial of chunk c for (sequence b, kv head kh): part[((b * hkv + kh) * nchunk + c) * GP + h]
// = {m (log2), l, 0, 0, acc[D]}; GP = G rounded up to 1, 2, 4 or 8 (rows h >= G are unused).
template <int D, int GP, int BITS>
__global__ void __launch_bounds__(kGqThreads)
gq_chunk_kernel(const void *__restrict__ qv, int q_f32, int hq, int hkv, int G, int gshift,
                const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                int max_ctx, int nchunk, float *__restrict__ part, int32_t *__restrict__ status) {
    constexpr int CW = kGqChunk, NT = kGqThreads, NW = NT / 32, CB = D * BITS / 8, CPT = D / NT;
    constexpr int EPW = 32 / BITS;    // codes per 32-bit word
    constexpr int EPP = 128 / BITS;   // codes per 16-byte piece
    const int ng = D >> gshift, gs = 1 << gshift, ppg = gs / EPP;
    const size_t region = (size_t)kBlock * (CB + 4 * ng);
    extern __shared__ __align__(16) uint8_t smem[];
    float *sq = reinterpret_cast<float *>(smem);                           // [GP][D], times log2 e / sqrt d
    float *sqg = sq + GP * D;                                              // [GP][8] per-group query sums
    float *sws = sqg + GP * 8;                                             // [ng][CW][GP] weight x value scale
    uint8_t *svc = reinterpret_cast<uint8_t *>(sws + (size_t)ng * CW * GP);   // [CW][CB] value codes
    __shared__ float sred[10][GP][NW];                                     // max, sum, bias sums per group
    const int c = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int L = ctx_lens[b];
    L = L < 0 ? 0 : (L > max_ctx ? max_ctx : L);
    const int t0 = c * CW, t1 = min(L, t0 + CW);
    float *pout = part + (((size_t)b * hkv + kh) * nchunk + c) * GP * (D + 4);
    if (t0 >= t1) {   // nothing in this chunk: an empty partial
        if (tid < GP) {
            pout[(size_t)tid * (D + 4)] = -INFINITY;
            pout[(size_t)tid * (D + 4) + 1] = 0.f;
        }
        return;
    }
    const float qs = kGqLog2e * rsqrtf((float)D);
    for (int i = tid; i < GP * D; i += NT) {
        const int h = i / D, dd = i - h * D;
        float v = 0.f;
        if (h < G) {
            const size_t idx = ((size_t)b * hq + (size_t)kh * G + h) * D + dd;
            v = q_f32 ? reinterpret_cast<const float *>(qv)[idx]
                      : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(qv)[idx]);
        }
        sq[i] = v * qs;
    }
    // value codes of the chunk's blocks (16 slots x CB bytes each), copied while the keys are scored
    const int nbk = (t1 - t0 + kBlock - 1) / kBlock;
    for (int i = tid; i < nbk * CB; i += NT) {
        const int j = i / CB, piece = i - j * CB, lb = t0 / kBlock + j;
        if (lb >= max_blocks) continue;
        const int64_t blk = block_table[(size_t)b * max_blocks + lb];
        if (blk < 0 || blk >= num_blocks) continue;
        cp_async16(svc + (size_t)j * kBlock * CB + 16 * piece, v_pool + ((size_t)blk * hkv + kh) * region + 16 * piece);
    }
    cp_async_commit();
    __syncthreads();
    for (int i = tid; i < GP * ng; i += NT) {
        const int h = i / ng, g = i - h * ng;
        float s = 0.f;
        for (int k = 0; k < gs; ++k) s += sq[h * D + g * gs + k];
        sqg[h * 8 + g] = s;
    }
    __syncthreads();

    // scores: thread tid scores token t0 + tid
    const int t = t0 + tid, off = t & (kBlock - 1);
    int64_t blk = -1;
    if (t < t1) {
        const int lb = t / kBlock;
        if (lb < max_blocks) blk = block_table[(size_t)b * max_blocks + lb];
        if (blk < 0 || blk >= num_blocks) {
            blk = -1;
            flag_status(status, TQ_STATUS_BAD_SLOT);
        }
    }
    float s[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) s[h] = -INFINITY;
    if (blk >= 0) {
        const uint8_t *kr = k_pool + ((size_t)blk * hkv + kh) * region;
        const uint4 *kc = reinterpret_cast<const uint4 *>(kr + (size_t)off * CB);
        const __half2 *kp = reinterpret_cast<const __half2 *>(kr + (size_t)kBlock * CB) + (size_t)off * ng;
#pragma unroll
        for (int h = 0; h < GP; ++h) s[h] = 0.f;
        for (int g = 0; g < ng; ++g) {
            float a[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) a[h] = 0.f;
            for (int p = 0; p < ppg; ++p) {
                const int pc = g * ppg + p;
                const uint4 u = __ldg(kc + pc);
                const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float f[EPW];
#pragma unroll
                    for (int e = 0; e < EPW; ++e) f[e] = small_uint_to_float((w4[k] >> (BITS * e)) & ((1u << BITS) - 1u));
                    const float *qrow = sq + pc * EPP + k * EPW;
#pragma unroll
                    for (int h = 0; h < GP; ++h) {
#pragma unroll
                        for (int e = 0; e < EPW; e += 4) {
                            const float4 q4 = *reinterpret_cast<const float4 *>(qrow + h * D + e);
                            a[h] = fmaf(q4.x, f[e], a[h]);
                            a[h] = fmaf(q4.y, f[e + 1], a[h]);
                            a[h] = fmaf(q4.z, f[e + 2], a[h]);
                            a[h] = fmaf(q4.w, f[e + 3], a[h]);
                        }
                    }
                }
            }
            const float2 sz = __half22float2(kp[g]);
#pragma unroll
            for (int h = 0; h < GP; ++h) s[h] = fmaf(sz.x, a[h], fmaf(sz.y, sqg[h * 8 + g], s[h]));
        }
    }
    // per head: chunk max and weights; sum of weights and of weight x value bias per group
    float m[GP], p[GP], l[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        const float x = warp_max(s[h]);
        if (lane == 0) sred[0][h][warp] = x;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        float x = sred[0][h][0];
#pragma unroll
        for (int w2 = 1; w2 < NW; ++w2) x = fmaxf(x, sred[0][h][w2]);
        m[h] = x;
        p[h] = (x == -INFINITY) ? 0.f : exp2f(s[h] - x);   // 0 for tokens not scored (s = -inf)
        const float ps = warp_sum(p[h]);
        if (lane == 0) sred[1][h][warp] = ps;
    }
    const __half2 *vp = blk >= 0 ? reinterpret_cast<const __half2 *>(v_pool + ((size_t)blk * hkv + kh) * region +
                                                                    (size_t)kBlock * CB) + (size_t)off * ng
                                 : nullptr;
    for (int g = 0; g < ng; ++g) {
        const float2 sz = vp ? __half22float2(vp[g]) : make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            sws[((size_t)g * CW + tid) * GP + h] = p[h] * sz.x;
            const float zs = warp_sum(p[h] * sz.y);
            if (lane == 0) sred[2 + g][h][warp] = zs;
        }
    }
    cp_async_wait_all();
    __syncthreads();
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        float x = 0.f;
#pragma unroll
        for (int w2 = 0; w2 < NW; ++w2) x += sred[1][h][w2];
        l[h] = x;
    }
    // values: thread tid accumulates coordinates tid + NT j
    float acc[CPT][GP];
#pragma unroll
    for (int j = 0; j < CPT; ++j)
#pragma unroll
        for (int h = 0; h < GP; ++h) acc[j][h] = 0.f;
    const int nt = t1 - t0;
#pragma unroll 2
    for (int tt = 0; tt < nt; ++tt) {
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int col = tid + NT * j;
            uint32_t code;
            if constexpr (BITS == 8) {
                code = svc[(size_t)tt * CB + col];
            } else {
                code = (svc[(size_t)tt * CB + (col >> 1)] >> ((col & 1) * 4)) & 15u;
            }
            const float f = small_uint_to_float(code);
            const float *wr = sws + ((size_t)(col >> gshift) * CW + tt) * GP;
#pragma unroll
            for (int h = 0; h < GP; ++h) acc[j][h] = fmaf(wr[h], f, acc[j][h]);
        }
    }
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        float *ph = pout + (size_t)h * (D + 4);
        if (tid == 0) {
            ph[0] = m[h];
            ph[1] = l[h];
        }
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int col = tid + NT * j, g = col >> gshift;
            float zs = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NW; ++w2) zs += sred[2 + g][h][w2];
            ph[4 + col] = acc[j][h] + zs;
        }
    }
}

// out[b][h] from the chunk partials of (b, h / G).  One warp per (sequence, query head).
template <int D>
__global__ void __launch_bounds__(128)
gq_merge_kernel(const float *__restrict__ part, float *__restrict__ out, int batch, int hq, int hkv, int GP,
                int nchunk) {
    constexpr int R = D / 32;
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (row >= batch * hq) return;
    const int b = row / hq, h = row % hq, G = hq / hkv, kh = h / G, hg = h % G;
    const float *pb = part + ((size_t)b * hkv + kh) * nchunk * GP * (D + 4);
    float M = -INFINITY;
    for (int c = 0; c < nchunk; ++c) M = fmaxf(M, pb[((size_t)c * GP + hg) * (D + 4)]);
    float v[R], den = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = 0.f;
    if (M != -INFINITY) {
        for (int c = 0; c < nchunk; ++c) {
            const float *ps = pb + ((size_t)c * GP + hg) * (D + 4);
            const float mc = ps[0];
            if (mc == -INFINITY) continue;
            const float w = exp2f(mc - M);
            den = fmaf(w, ps[1], den);
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = fmaf(w, ps[4 + 32 * r + lane], v[r]);
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float *orow = out + (size_t)row * D;
#pragma unroll
    for (int r = 0; r < R; ++r) orow[32 * r + lane] = v[r] * inv;
}

int gshift_of(int group) { return group == 32 ? 5 : group == 64 ? 6 : 7; }

template <int D, int BITS>
cudaError_t gq_encode_d(int dtype, const void *x, int64_t n_vec, int hkv, int gshift, const int64_t *slots,
                        uint8_t *pool, int64_t num_blocks, int32_t *status, cudaStream_t st) {
    const int64_t want = (n_vec + 3) / 4;
    const int grid = (int)(want < 152 * 32 ? want : 152 * 32);
    if (dtype == TQ_DTYPE_F32)
        gq_encode_kernel<D, BITS, float><<<grid, kGqThreads, 0, st>>>(static_cast<const float *>(x), n_vec, hkv,
                                                                       gshift, slots, pool, num_blocks, status);
    else
        gq_encode_kernel<D, BITS, __nv_bfloat16><<<grid, kGqThreads, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(x), n_vec, hkv, gshift, slots, pool, num_blocks, status);
    return cudaGetLastError();
}

template <int D, int GP, int BITS>
cudaError_t gq_decode_g(int gshift, int dtype, const void *q, int batch, int hq, int hkv, const uint8_t *k_pool,
                        const uint8_t *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                        const int32_t *ctx_lens, int max_ctx, float *out, float *part, int32_t *status,
                        cudaStream_t st) {
    const int ng = D >> gshift, nchunk = gq_nchunk(max_ctx);
    const size_t smem = 4 * ((size_t)GP * D + GP * 8 + (size_t)ng * kGqChunk * GP) + (size_t)kGqChunk * (D * BITS / 8);
    cudaError_t e = cudaSuccess;
    if (nchunk > 0) {
        auto kern = gq_chunk_kernel<D, GP, BITS>;
        if (smem > 48 * 1024) e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kern<<<dim3(nchunk, hkv, batch), kGqThreads, smem, st>>>(q, dtype == TQ_DTYPE_F32, hq, hkv, hq / hkv, gshift,
                                                                 k_pool, v_pool, num_blocks, block_table, max_blocks,
                                                                 ctx_lens, max_ctx, nchunk, part, status);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    gq_merge_kernel<D><<<(batch * hq + 3) / 4, 128, 0, st>>>(part, out, batch, hq, hkv, GP, nchunk);
    return cudaGetLastError();
}

template <int D, int BITS>
cudaError_t gq_decode_d(int gshift, int dtype, const void *q, int batch, int hq, int hkv, const uint8_t *k_pool,
                        const uint8_t *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                        const int32_t *ctx_lens, int max_ctx, float *out, float *part, int32_t *status,
                        cudaStream_t st) {
    switch (gq_group_pad(hq / hkv)) {
        case 1: return gq_decode_g<D, 1, BITS>(gshift, dtype, q, batch, hq, hkv, k_pool, v_pool, num_blocks,
                                               block_table, max_blocks, ctx_lens, max_ctx, out, part, status, st);
        case 2: return gq_decode_g<D, 2, BITS>(gshift, dtype, q, batch, hq, hkv, k_pool, v_pool, num_blocks,
                                               block_table, max_blocks, ctx_lens, max_ctx, out, part, status, st);
        case 4: return gq_decode_g<D, 4, BITS>(gshift, dtype, q, batch, hq, hkv, k_pool, v_pool, num_blocks,
                                               block_table, max_blocks, ctx_lens, max_ctx, out, part, status, st);
        default: return gq_decode_g<D, 8, BITS>(gshift, dtype, q, batch, hq, hkv, k_pool, v_pool, num_blocks,
                                                block_table, max_blocks, ctx_lens, max_ctx, out, part, status, st);
    }
}

}  // namespace

cudaError_t launch_gq_encode(int d, int bits, int group, int dtype, const void *x, int64_t n_tokens, int hkv,
                             const int64_t *slots, uint8_t *pool, int64_t num_blocks, int32_t *status,
                             cudaStream_t st) {
    const int64_t n_vec = n_tokens * hkv;
    if (n_vec == 0) return cudaSuccess;
    const int gs = gshift_of(group);
    if (d == 128)
        return bits == 4 ? gq_encode_d<128, 4>(dtype, x, n_vec, hkv, gs, slots, pool, num_blocks, status, st)
                         : gq_encode_d<128, 8>(dtype, x, n_vec, hkv, gs, slots, pool, num_blocks, status, st);
    return bits == 4 ? gq_encode_d<256, 4>(dtype, x, n_vec, hkv, gs, slots, pool, num_blocks, status, st)
                     : gq_encode_d<256, 8>(dtype, x, n_vec, hkv, gs, slots, pool, num_blocks, status, st);
}

cudaError_t launch_gq_decode(int d, int bits, int group, int dtype, const void *q, int batch, int hq, int hkv,
                             const uint8_t *k_pool, const uint8_t *v_pool, int64_t num_blocks,
                             const int32_t *block_table, int max_blocks, const int32_t *ctx_lens, int max_ctx,
                             float *out, float *part, int32_t *status, cudaStream_t st) {
    if (batch == 0) return cudaSuccess;
    const int gs = gshift_of(group);
#define TQ_GQ_DEC(DD, BB)                                                                                         \
    gq_decode_d<DD, BB>(gs, dtype, q, batch, hq, hkv, k_pool, v_pool, num_blocks, block_table, max_blocks, ctx_lens, \
                        max_ctx, out, part, status, st)
    if (d == 128) return bits == 4 ? TQ_GQ_DEC(128, 4) : TQ_GQ_DEC(128, 8);
    return bits == 4 ? TQ_GQ_DEC(256, 4) : TQ_GQ_DEC(256, 8);
#undef TQ_GQ_DEC
}

}  // namespace tq
