// tq_decode.cu -- decode attention over the compressed paged cache.
//
// Method: the scores and the value sum are evaluated in the rotated domain
// straight from the packed cells, signs and fp16 norms (the "fused
// dequantisation" of the SwiftLM README, "TurboQuantization: KV Cache
// Compression"); blocks are found through the block table of the vLLM-MLX
// explainer, "Paged KVキャッシュ".  With qbar = Pi q and u = S qbar:
//   s_j = (n_j/sqrt d) (<qbar, c[cell_j]>/sqrt d + gamma_j sqrt(pi/2)/d <u, 2 sign_j - 1>)
//   a   = sum_j softmax(s)_j nv_j c[vcell_j] / sqrt d,    out = Pi^T a.
//
// Three launches per call: (1) query prep (qbar, u), (2) split-K main pass
// producing an online-softmax partial (m, l, acc[d]) per (seq, q head, split),
// (3) merge of the splits plus one inverse rotation per (seq, q head).
#include "tq_internal.cuh"

namespace tq {

constexpr int kSplitTokens = 512;          // tokens per context split (32 blocks)
__host__ __device__ constexpr int kPartStride(int d) { return d + 4; }   // m, l, pad, pad, acc[d]

size_t decode_workspace_bytes(int d, int batch, int hq, int max_ctx) {
    if (!valid_d(d) || batch <= 0 || hq <= 0 || max_ctx < 0) return 0;
    const size_t nsplit = (size_t)((max_ctx + kSplitTokens - 1) / kSplitTokens);
    const size_t qws = (size_t)batch * hq * 2 * d * sizeof(float);
    const size_t part = (size_t)batch * hq * (nsplit ? nsplit : 1) * kPartStride(d) * sizeof(float);
    return ((qws + 255) & ~(size_t)255) + part;
}

namespace {

// ---------------------------------------------------------------- (1) query prep
template <int D, typename T>
__global__ void __launch_bounds__(128)
qprep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ q, int n_rows, float *__restrict__ qws) {
    constexpr int R = D / 32;
    __shared__ __align__(16) float qb[4][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= n_rows) return;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = to_f32<T>(q[(size_t)row * D + 32 * r + lane]) * __ldg(Dsign + 32 * r + lane);
    fwht_warp<R>(v, lane);
    const float inv_sd = rsqrtf((float)D);
    float *out = qws + (size_t)row * 2 * D;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        v[r] *= inv_sd;                      // qbar = H D q / sqrt d
        qb[warp][32 * r + lane] = v[r];
        out[32 * r + lane] = v[r];
    }
    __syncwarp();
#pragma unroll
    for (int r = 0; r < R; ++r) {            // u_k = sum_i S[k][i] qbar_i
        const int k = 32 * r + lane;
        const float4 *srow = reinterpret_cast<const float4 *>(S + (size_t)k * D);
        const float4 *qq = reinterpret_cast<const float4 *>(qb[warp]);
        float acc = 0.f;
#pragma unroll 8
        for (int i = 0; i < D / 4; ++i) {
            const float4 a = __ldg(srow + i), b = qq[i];
            acc = fmaf(a.x, b.x, acc);
            acc = fmaf(a.y, b.y, acc);
            acc = fmaf(a.z, b.z, acc);
            acc = fmaf(a.w, b.w, acc);
        }
        out[D + k] = acc;
    }
}

// ---------------------------------------------------------------- (2) split-K main pass, SIMT
// grid (splits, Hkv, B), 128 threads.  Per 16-token block: stage both records
// in shared memory, score (thread = (token, head)), online softmax (half-warp
// per head), accumulate values (thread = coordinate, all heads).
template <int D>
__global__ void __launch_bounds__(128)
decode_simt_kernel(const uint8_t *__restrict__ params, const float *__restrict__ qws, int hq, int hkv,
                   const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                   const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                   int max_ctx, float *__restrict__ part, int nsplit, int32_t *status) {
    constexpr int KREC = (int)k_record(D), VREC = (int)v_record(D);
    constexpr int NW = D / 128, NWV = D / 64, DK = D / 128;
    __shared__ __align__(16) float qb[8][D];
    __shared__ __align__(16) float uu[8][D];
    __shared__ __align__(16) uint32_t krec[KREC / 4];
    __shared__ __align__(16) uint32_t vrec[VREC / 4];
    __shared__ float cent[8];
    __shared__ float sc[8][16];
    __shared__ float pr[8][16];
    __shared__ float alpha_s[8], mrun[8], lrun[8];

    const int s = blockIdx.x, kh = blockIdx.y, b = blockIdx.z;
    const int g = hq / hkv;
    const int tid = threadIdx.x;
    int L = ctx_lens[b];
    if (L > max_ctx) L = max_ctx;
    const int t0 = s * kSplitTokens;
    if (t0 >= L) return;                      // the merge only reads splits that hold tokens
    const int t1 = min(L, t0 + kSplitTokens);

    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (tid < 8) { cent[tid] = ph->centroid[tid]; mrun[tid] = -INFINITY; lrun[tid] = 0.f; }
    for (int i = tid; i < g * D; i += 128) {
        const int h = i / D, k = i % D;
        const float *src = qws + ((size_t)b * hq + kh * g + h) * 2 * D;
        qb[h][k] = src[k];
        uu[h][k] = src[D + k];
    }
    float acc[8][DK];
#pragma unroll
    for (int h = 0; h < 8; ++h)
#pragma unroll
        for (int k = 0; k < DK; ++k) acc[h][k] = 0.f;

    const float sd = sqrtf((float)D);
    const float qjl = 1.2533141373155003f / (float)D;     // sqrt(pi/2) / d
    const int t = tid & 15, hh = tid >> 4;

    for (int tb = t0; tb < t1; tb += kBlock) {
        const int lb = tb / kBlock;
        const int64_t phys = (lb < max_blocks) ? (int64_t)block_table[(size_t)b * max_blocks + lb] : -1;
        const bool ok = phys >= 0 && phys < num_blocks;
        __syncthreads();                       // previous block fully consumed
        if (ok) {
            const uint4 *ks = reinterpret_cast<const uint4 *>(k_pool + ((size_t)phys * hkv + kh) * KREC);
            const uint4 *vs = reinterpret_cast<const uint4 *>(v_pool + ((size_t)phys * hkv + kh) * VREC);
            for (int i = tid; i < KREC / 16; i += 128) reinterpret_cast<uint4 *>(krec)[i] = ks[i];
            for (int i = tid; i < VREC / 16; i += 128) reinterpret_cast<uint4 *>(vrec)[i] = vs[i];
        } else if (tid == 0) {
            flag_status(status, TQ_STATUS_BAD_SLOT);
        }
        __syncthreads();
        // scores
        if (hh < g) {
            const int tok = tb + t;
            float sv = -INFINITY;
            if (ok && tok < t1) {
                float dc = 0.f, dq = 0.f;
                for (int i = 0; i < D; ++i) {
                    const int c = i >> 5, wj = c >> 2, q = 2 * (c & 3) + ((i >> 4) & 1), j = i & 3;
                    const int lane4 = 4 * (t & 7) + ((i >> 2) & 3);
                    const int word = (lane4 * 2 + (t >> 3)) * NW + wj;
                    const int bit = 8 * j + q;
                    int code = 0;
#pragma unroll
                    for (int pl = 0; pl < 3; ++pl) code |= ((krec[pl * (D / 2) + word] >> bit) & 1) << pl;
                    const int sg = (krec[3 * (D / 2) + word] >> bit) & 1;
                    dc = fmaf(qb[hh][i], cent[code], dc);
                    dq += sg ? uu[hh][i] : -uu[hh][i];
                }
                const __half2 ng = *reinterpret_cast<const __half2 *>(reinterpret_cast<const uint8_t *>(krec) + 8 * D + 4 * t);
                const float n = __low2float(ng), gm = __high2float(ng);
                sv = (n / sd) * (dc / sd + gm * qjl * dq);
            }
            sc[hh][t] = sv;
        }
        __syncthreads();
        // online softmax, half-warp per head.  Every thread runs the shuffles
        // (full-warp masks); rows hh >= g only compute and store nothing.
        {
            const bool live = hh < g;
            const float sv = live ? sc[hh][t] : -INFINITY;
            float bm = sv;
#pragma unroll
            for (int m = 8; m > 0; m >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, m, 16));
            const float m_old = live ? mrun[hh] : -INFINITY;
            const float m_new = fmaxf(m_old, bm);
            const float alpha = (m_old == -INFINITY) ? 0.f : __expf(m_old - m_new);
            const float p = (sv == -INFINITY) ? 0.f : __expf(sv - m_new);
            float ps = p;
#pragma unroll
            for (int m = 8; m > 0; m >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, m, 16);
            if (live) {
                const float nv = __half2float(*reinterpret_cast<const __half *>(reinterpret_cast<const uint8_t *>(vrec) + 6 * D + 2 * t));
                pr[hh][t] = p * nv / sd;
                if (t == 0) {
                    alpha_s[hh] = alpha;
                    lrun[hh] = lrun[hh] * alpha + ps;
                    mrun[hh] = m_new;
                }
            }
        }
        __syncthreads();
        // value accumulation in the rotated domain
#pragma unroll
        for (int k = 0; k < DK; ++k) {
            const int i = tid + 128 * k;
            const int mt = i >> 4, r16 = i & 15, gid = r16 & 7, rh = r16 >> 3;
#pragma unroll
            for (int h = 0; h < 8; ++h)
                if (h < g) acc[h][k] *= alpha_s[h];
            for (int tt = 0; tt < kBlock; ++tt) {
                const int lane4 = 4 * gid + (tt >> 2);
                const int word = lane4 * NWV + 2 * (mt >> 3) + rh;
                const int bit = 8 * (tt & 3) + (mt & 7);
                int code = 0;
#pragma unroll
                for (int pl = 0; pl < 3; ++pl) code |= ((vrec[pl * (D / 2) + word] >> bit) & 1) << pl;
                const float cv = cent[code];
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (h < g) acc[h][k] = fmaf(pr[h][tt], cv, acc[h][k]);
            }
        }
    }
    // write the partial state
#pragma unroll
    for (int h = 0; h < 8; ++h) {
        if (h >= g) break;
        float *dst = part + (((size_t)b * hq + kh * g + h) * nsplit + s) * kPartStride(D);
#pragma unroll
        for (int k = 0; k < DK; ++k) dst[4 + tid + 128 * k] = acc[h][k];
        if (tid == 0) { dst[0] = mrun[h]; dst[1] = lrun[h]; }
    }
}

// ---------------------------------------------------------------- (3) merge + inverse rotation
template <int D>
__global__ void __launch_bounds__(128)
merge_kernel(const uint8_t *__restrict__ params, const float *__restrict__ part, const int32_t *__restrict__ ctx_lens,
             int max_ctx, int hq, int n_rows, int nsplit, float *__restrict__ out) {
    constexpr int R = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row = blockIdx.x * 4 + warp;
    if (row >= n_rows) return;
    const int b = row / hq;
    int L = ctx_lens[b];
    if (L > max_ctx) L = max_ctx;
    float *o = out + (size_t)row * D;
    if (L <= 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) o[32 * r + lane] = 0.f;
        return;
    }
    const int ns = (L + kSplitTokens - 1) / kSplitTokens;
    const float *p0 = part + (size_t)row * nsplit * kPartStride(D);
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, p0[(size_t)s * kPartStride(D)]);
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = 0.f;
    float l = 0.f;
    for (int s = 0; s < ns; ++s) {
        const float *ps = p0 + (size_t)s * kPartStride(D);
        const float m = ps[0];
        const float w = (m == -INFINITY) ? 0.f : __expf(m - M);
        l = fmaf(ps[1], w, l);
#pragma unroll
        for (int r = 0; r < R; ++r) v[r] = fmaf(ps[4 + 32 * r + lane], w, v[r]);
    }
    const float inv = (l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] *= inv;
    // out = Pi^T a = D (H a) / sqrt d
    fwht_warp<R>(v, lane);
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float inv_sd = rsqrtf((float)D);
#pragma unroll
    for (int r = 0; r < R; ++r) o[32 * r + lane] = v[r] * inv_sd * __ldg(Dsign + 32 * r + lane);
}

}  // namespace

namespace {
struct WsLayout {
    float *qws;
    float *part;
    int nsplit;
};
WsLayout ws_layout(void *ws, int d, int rows, int max_ctx) {
    WsLayout w;
    w.nsplit = max(1, (max_ctx + kSplitTokens - 1) / kSplitTokens);
    w.qws = reinterpret_cast<float *>(ws);
    const size_t qbytes = ((size_t)rows * 2 * d * sizeof(float) + 255) & ~(size_t)255;
    w.part = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(ws) + qbytes);
    return w;
}
}  // namespace

cudaError_t launch_qprep(int d, int dtype, const void *params, const void *q, int batch, int hq, int max_ctx,
                         void *ws, cudaStream_t st) {
    const int rows = batch * hq;
    const WsLayout w = ws_layout(ws, d, rows, max_ctx);
    const uint8_t *P = (const uint8_t *)params;
    const dim3 gq((rows + 3) / 4);
    if (d == 128) {
        if (dtype == TQ_DTYPE_BF16) qprep_kernel<128, __nv_bfloat16><<<gq, 128, 0, st>>>(P, (const __nv_bfloat16 *)q, rows, w.qws);
        else qprep_kernel<128, float><<<gq, 128, 0, st>>>(P, (const float *)q, rows, w.qws);
    } else {
        if (dtype == TQ_DTYPE_BF16) qprep_kernel<256, __nv_bfloat16><<<gq, 128, 0, st>>>(P, (const __nv_bfloat16 *)q, rows, w.qws);
        else qprep_kernel<256, float><<<gq, 128, 0, st>>>(P, (const float *)q, rows, w.qws);
    }
    return cudaGetLastError();
}

cudaError_t launch_partial(int d, const void *params, int batch, int hq, int hkv, const void *k_pool,
                           const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                           const int32_t *ctx_lens, int max_ctx, void *ws, int32_t *status, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch * hq, max_ctx);
    const uint8_t *P = (const uint8_t *)params;
    const dim3 gm(w.nsplit, hkv, batch);
    if (d == 128)
        decode_simt_kernel<128><<<gm, 128, 0, st>>>(P, w.qws, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                                                     num_blocks, block_table, max_blocks, ctx_lens, max_ctx, w.part,
                                                     w.nsplit, status);
    else
        decode_simt_kernel<256><<<gm, 128, 0, st>>>(P, w.qws, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                                                     num_blocks, block_table, max_blocks, ctx_lens, max_ctx, w.part,
                                                     w.nsplit, status);
    return cudaGetLastError();
}

cudaError_t launch_merge(int d, const void *params, int batch, int hq, const int32_t *ctx_lens, int max_ctx,
                         float *out, void *ws, cudaStream_t st) {
    const int rows = batch * hq;
    const WsLayout w = ws_layout(ws, d, rows, max_ctx);
    const uint8_t *P = (const uint8_t *)params;
    const dim3 gq((rows + 3) / 4);
    if (d == 128) merge_kernel<128><<<gq, 128, 0, st>>>(P, w.part, ctx_lens, max_ctx, hq, rows, w.nsplit, out);
    else merge_kernel<256><<<gq, 128, 0, st>>>(P, w.part, ctx_lens, max_ctx, hq, rows, w.nsplit, out);
    return cudaGetLastError();
}

}  // namespace tq
