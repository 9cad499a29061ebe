// tq_decode.cu -- decode attention over the compressed paged cache.
//
// Method: scores and the value sum are evaluated in the rotated domain straight
// from the packed cells, signs and fp16 norms (the "fused dequantisation" of
// the SwiftLM README, "TurboQuantization: KV Cache Compression"); blocks are
// found through the block table of the vLLM-MLX explainer, "Paged KVキャッシュ".
// With qbar = Pi q and u = S qbar:
//   s_j = (n_j/sqrt d) (<qbar, c[cell_j]>/sqrt d + gamma_j sqrt(pi/2)/d <u, 2 sign_j - 1>)
//   a   = sum_j softmax(s)_j nv_j c[vcell_j] / sqrt d,    out = Pi^T a.
//
// Tensor-core formulation (this library's design, not the pages'):
//  * The 8 Lloyd-Max levels are odd in the three cell bits b0,b1,b2, so with
//    sigma_p = 2 b_p - 1 every level is exactly
//      c[cell] = A0 sigma_0 + A1 sigma_1 + A2 sigma_2 + A3 sigma_0 sigma_1 sigma_2,
//    where sigma_0 sigma_1 sigma_2 = 2 (b0^b1^b2) - 1.  A dot product with the
//    levels is therefore four +-1 dot products, and the QJL term a fifth.
//  * A bit plane becomes f16 mma.sync (m16n8k16) operands with one LOP3 per
//    register: for bit position q in 8..15 of each half, (w & bit) ^ base_q is
//    the f16 value alpha_q (bit 0) or alpha_q + delta_q (bit 1), |delta_q| >=
//    1/4; bits at positions 0..7 are first moved up by a shift of the word.
//    The other operand is pre-divided by delta_q and a per-column constant
//    removes alpha_q, so the +-1 product is recovered exactly.
//  * The fp32 query side is carried as f16 hi + lo (relative error about
//    2^-22), the softmax weights as one f16 with a running power-of-two scale;
//    the tensor core accumulates in fp32.
//
// Two launches per call: (1) query prep (qbar, u, f16 operand fragments,
// offset constants, and the work schedule of the pass); (2) the split-K pass,
// persistent: the context of every (sequence, kv head) is cut into 128-token
// chunks (256 for groups of more than 4 query heads), and CTA c of P takes
// the c-th of P equal, contiguous ranges of the chunk sequence ordered by
// (sequence, kv head, chunk) ("stream-K").  A (sequence, kv head) inside one
// CTA's range is finished there; one shared by several CTAs leaves an
// online-softmax partial (m, l, acc[d]) per query head from each, and the last
// of them to finish merges the partials.  Either way one inverse rotation per
// (sequence, query head) is applied at the end.
#include <atomic>

#include "tq_split.cuh"

namespace tq {

size_t decode_workspace_bytes(int d, int batch, int hq, int max_ctx) {
    if (!valid_d(d) || batch <= 0 || hq <= 0 || max_ctx < 0) return 0;
    size_t off[5];
    return ws_sizes(d, batch, hq, off);
}

namespace {

// ---------------------------------------------------------------- (1) query prep (body in tq_prep.cuh)
template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
qprep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch, int q_len, int hq, int hkv,
             const int32_t *__restrict__ ctx_lens, int max_ctx, int chunk, int P, uint8_t *__restrict__ packs,
             unsigned int *__restrict__ counters, int64_t *__restrict__ cpre, int32_t *__restrict__ cta_b) {
    extern __shared__ __align__(16) uint8_t qsm[];
    pdl_launch_dependents();
    if (blockIdx.x == gridDim.x - 1) {   // the last CTA lays out the pass's work
        build_schedule(ctx_lens, 0, batch, hkv, max_ctx, chunk, P, cpre, cta_b);
        return;
    }
    qprep_rows<D, NTK, T>(params, q, batch, q_len, hq, hkv, ctx_lens, 0, max_ctx, chunk, P, packs, counters, cpre, cta_b,
                          blockIdx.x, qsm);
}

// ---------------------------------------------------------------- (2) split-K pass
// grid P (persistent), NWARP warps (4 for G <= 4, else 8).  A CTA walks its
// range of chunks one (sequence, kv head) segment at a time.  The records of a
// chunk of 32*NWARP tokens (2 blocks per warp) are staged in shared memory by
// cp.async one chunk ahead.  Per chunk: warp w scores blocks 2w, 2w+1 against
// all G heads (K side); the warps run the online softmax (warp w owns heads
// w, w+NWARP); warp w accumulates values for its D/NWARP coordinates over the
// whole chunk (V side).

template <int D, int NWARP>
struct SplitCfg {
    static constexpr int NT = NWARP * 32;
    static constexpr int BPW = TQ_SPLITK_BPW;        // blocks scored per warp per chunk
    static constexpr int BPC = NWARP * BPW;          // blocks per chunk
    static constexpr int CH = kBlock * BPC;          // tokens per chunk
    static constexpr int KREC = (int)k_record(D), VREC = (int)v_record(D);
    static constexpr size_t kBytes = 2 * (size_t)BPC * KREC;   // double-buffered K records
    static constexpr size_t vBytes = 2 * (size_t)BPC * VREC;
};

template <int D, int G, int NWARP>
constexpr size_t split_smem_bytes() {
    using C = SplitCfg<D, NWARP>;
    return C::kBytes + C::vBytes + (size_t)8 * (C::CH + 8) * 2 + (size_t)C::CH * G * 4;
}

#ifndef TQ_SPLITK_MINBLOCKS_WIDE
#define TQ_SPLITK_MINBLOCKS_WIDE 3   // resident CTAs for d = 256 or groups of more than 4 heads
#endif
template <int D, int G, int NWARP>
__global__ void __launch_bounds__(NWARP * 32, (NWARP == 4 ? (D == 128 && G <= 4 ? TQ_SPLITK_MINBLOCKS : TQ_SPLITK_MINBLOCKS_WIDE) : 1))
decode_mma_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ packs, int batch, int q_len, int hq, int hkv,
                  const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                  const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                  int ctx_add, int max_ctx, const int64_t *__restrict__ cpre, const int32_t *__restrict__ cta_b,
                  float *__restrict__ part, unsigned int *__restrict__ counters, float *__restrict__ out,
                  float *__restrict__ lse, int32_t *status) {
    using C = SplitCfg<D, NWARP>;
    constexpr int NT_ = C::NT, BPW = C::BPW, BPC = C::BPC, CH = C::CH;
    constexpr int TPL = CH / 32;               // softmax tokens per lane
    constexpr int NTK = (2 * G + 7) / 8;       // K-side n-tiles (hi, lo x G heads)
    constexpr int NKS = D / 16;                // K-side k16 steps
    constexpr int MTW = D / 16 / NWARP;        // V-side m-tiles per warp
    constexpr int NW = D / 128, NWV = D / 64;
    constexpr int KREC = C::KREC, VREC = C::VREC;
    constexpr int HPW = (G + NWARP - 1) / NWARP;   // heads owned per warp in the softmax
    constexpr int PROW = CH + 8;               // halves per sP row (pad: conflict-free fragment reads)
    constexpr int R = D / 32;

    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *sK = smem;                                        // [2][BPC][KREC]
    uint8_t *sV = sK + C::kBytes;                              // [2][BPC][VREC]
    __half *sP = reinterpret_cast<__half *>(sV + C::vBytes);   // [8][PROW] weights, head-major
    float *sS = reinterpret_cast<float *>(sP + 8 * PROW);      // [CH][G] scores
    float *sAcc = reinterpret_cast<float *>(sK);               // [G][D], between segments
    __shared__ int sOk[2][BPC];
    __shared__ float sF[8];
    __shared__ float sM[8], sL[8], sTc[8];
    __shared__ int sE[8];
    __shared__ bool s_last;

    const int cta = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;

    pdl_wait();   // everything before this launch (the prep's schedule, packs, counters) is complete

    // sequences with nothing to attend get out = 0
    for (int b = cta; b < batch; b += gridDim.x)
        if (attended_len(ctx_lens[b], ctx_add, max_ctx) == 0)
        {
            for (int i = tid; i < q_len * hq * D; i += NT_) out[(size_t)b * q_len * hq * D + i] = 0.f;
            if (lse)
                for (int i = tid; i < q_len * hq; i += NT_) lse[(size_t)b * q_len * hq + i] = -INFINITY;
        }

    // P CTAs share the W chunks, at least one chunk each (as in build_schedule)
    const int64_t W = cpre[batch];
    const int P = (int)(W < (int64_t)gridDim.x ? W : (int64_t)gridDim.x);
    if (cta >= P) return;
    const int64_t g0 = sk_begin(cta, P, W), g1 = sk_begin(cta + 1, P, W);

    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    float A[4];
    walsh4(ph->centroid, A);
    const float Asum = A[0] + A[1] + A[2] + A[3];
    const float inv_sd = rsqrtf((float)D);
    const float qjl = 1.2533141373155003f / (float)D;   // sqrt(pi/2) / d
    // f16x2 {1.0, 1.0}, read at run time so that it stays in a register for LOP3
    const uint32_t one16x2 = (uint32_t)ph->one16x2;

    // weight rows of heads >= G stay zero
    for (int i = tid; i < (8 - G) * PROW; i += NT_) sP[G * PROW + i] = __float2half(0.f);
    // V side: operand mask/base of this warp's m-tiles (v_base: no offset, see vop_alpha)
    uint32_t vmask[MTW], vbase[MTW];
#pragma unroll
    for (int i = 0; i < MTW; ++i) {
        const int q = 8 + ((warp * MTW + i) & 7);
        vmask[i] = 0x00010001u << q;
        vbase[i] = vop_base(q);
    }
    const int mhi = (warp * MTW) >> 3;

    // the first segment: sequence b, kv head kh, global chunk g
    int b = cta_b[cta];
    int64_t ub = cpre[b];
    int nchb = (int)((cpre[b + 1] - ub) / hkv);
    int kh = (int)((g0 - ub) / nchb);
    int64_t g = g0;
    bool first_seg = true;

#pragma unroll 1
    while (true) {
        const int64_t us = ub + (int64_t)kh * nchb, ue = us + nchb;
        const int64_t se = (g1 < ue) ? g1 : ue;
        const int L = attended_len(ctx_lens[b], ctx_add, max_ctx);
        const int t0 = (int)(g - us) * CH;
        const int t1 = min(L, (int)(se - us) * CH);

        // stage the K and V records of the chunk starting at token tc into buffer buf
        auto issue_chunk = [&](int tc, int buf) {
            const int k = tid % BPC;
            const bool inrange = tc + kBlock * k < t1;
            const int64_t p = inrange ? block_of(block_table, b, max_blocks, tc / kBlock + k, num_blocks) : -1;
            if (tid < BPC) {
                sOk[buf][k] = p >= 0;
                if (inrange && p < 0) flag_status(status, TQ_STATUS_BAD_SLOT);
            }
            if (p >= 0) {
                const uint8_t *gk = k_pool + ((size_t)p * hkv + kh) * KREC;
                const uint8_t *gv = v_pool + ((size_t)p * hkv + kh) * VREC;
                uint8_t *dk = sK + ((size_t)buf * BPC + k) * KREC;
                uint8_t *dv = sV + ((size_t)buf * BPC + k) * VREC;
                for (int j = tid / BPC; j < KREC / 16; j += NT_ / BPC) cp_async16(dk + 16 * j, gk + 16 * j);
                for (int j = tid / BPC; j < VREC / 16; j += NT_ / BPC) cp_async16(dv + 16 * j, gv + 16 * j);
            }
            cp_async_commit();
        };
        issue_chunk(t0, 0);

        // K-side operand fragments and offset constants of this (sequence, kv head)
        const uint8_t *pack = packs + ((size_t)b * hkv + kh) * kPackBytes(D);
        const float *pf = reinterpret_cast<const float *>(pack) + kPackFloatOff(D);
        uint32_t bq[2][NKS][NTK][2];
#pragma unroll
        for (int qu = 0; qu < 2; ++qu)
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks)
#pragma unroll
                for (int nt = 0; nt < NTK; ++nt) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(
                        pack + (((size_t)(qu * NKS + ks) * NTK + nt) * 64 + lane * 2) * 4);
                    bq[qu][ks][nt][0] = w.x;
                    bq[qu][ks][nt][1] = w.y;
                }
        float cq[NTK], cu[NTK];
        int tlim[NTK];   // tokens column hg attends in this segment (query i: L - (q_len - 1 - i))
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            const int hg = 4 * nt + tig;           // columns 2tig (hi) and 2tig+1 (lo) of n-tile nt
            cq[nt] = hg < G ? pf[hg] * Asum : 0.f;
            cu[nt] = hg < G ? pf[8 + hg] : 0.f;
            tlim[nt] = hg < G ? min(t1, L - (q_len - 1 - hg / (G / q_len))) : 0;
        }

        // value sums of this warp's coordinates, planes combined, in the running weight scale
        float arun[MTW][4];
#pragma unroll
        for (int i = 0; i < MTW; ++i)
#pragma unroll
            for (int k = 0; k < 4; ++k) arun[i][k] = 0.f;
        float m_run[HPW], l_run[HPW], w_ref[HPW];
        int e_run[HPW];
#pragma unroll
        for (int k = 0; k < HPW; ++k) {
            m_run[k] = -INFINITY;
            l_run[k] = 0.f;
            w_ref[k] = 0.f;
            e_run[k] = 0;
        }

        int buf = 0;
#pragma unroll 1
        for (int tc = t0; tc < t1; tc += CH, buf ^= 1) {
            cp_async_wait_all();
            __syncthreads();   // chunk `buf` staged and visible; the other buffer is free
            if (tc + CH < t1) issue_chunk(tc + CH, buf ^ 1);
            const uint8_t *kb_base = sK + (size_t)buf * BPC * KREC;
            const uint8_t *vb_base = sV + (size_t)buf * BPC * VREC;
            // ---- K side: warp scores blocks BPW*warp .. BPW*warp+BPW-1 of the chunk
#pragma unroll 1
            for (int bw = 0; bw < BPW; ++bw) {
                const int k = BPW * warp + bw;
                const bool ok = sOk[buf][k] != 0;
                const uint8_t *rec = kb_base + (size_t)k * KREC;
                uint32_t Wd[4][2][NW];
#pragma unroll
                for (int pl = 0; pl < 4; ++pl) {
                    if (NW == 1) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(rec + pl * 2 * D + lane * 8);
                        Wd[pl][0][0] = w.x;
                        Wd[pl][1][0] = w.y;
                    } else {
                        const uint4 w = *reinterpret_cast<const uint4 *>(rec + pl * 2 * D + lane * 16);
                        Wd[pl][0][0] = w.x;
                        Wd[pl][0][NW - 1] = w.y;
                        Wd[pl][1][0] = w.z;
                        Wd[pl][1][NW - 1] = w.w;
                    }
                }
                float nrm[2], gam[2];
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const __half2 ng = *reinterpret_cast<const __half2 *>(rec + 8 * D + 4 * (gid + 8 * r));
                    nrm[r] = __low2float(ng);
                    gam[r] = __high2float(ng);
                }
                // five masks as independent accumulator chains: code = sum_m A_m (mask m), qjl = mask 4
                uint32_t w[5][2][NW], w8[5][2][NW];
#pragma unroll
                for (int m = 0; m < 5; ++m)
#pragma unroll
                    for (int th = 0; th < 2; ++th)
#pragma unroll
                        for (int wj = 0; wj < NW; ++wj) {
                            w[m][th][wj] = (m < 3) ? Wd[m][th][wj]
                                         : (m == 3) ? (Wd[0][th][wj] ^ Wd[1][th][wj] ^ Wd[2][th][wj]) : Wd[3][th][wj];
                            w8[m][th][wj] = w[m][th][wj] << 8;
                        }
                float acc[5][NTK][4];
#pragma unroll
                for (int m = 0; m < 5; ++m)
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
                        for (int x = 0; x < 4; ++x) acc[m][nt][x] = 0.f;
#pragma unroll
                for (int ks = 0; ks < NKS; ++ks) {
                    const int q = 8 + (ks & 7), wj = ks >> 3;
                    const uint32_t msk = op_mask(q), bas = (q == 14) ? 0u : one16x2;
#pragma unroll
                    for (int m = 0; m < 5; ++m) {
                        const uint32_t a0 = lop_and_xor(w8[m][0][wj], msk, bas), a1 = lop_and_xor(w8[m][1][wj], msk, bas);
                        const uint32_t a2 = lop_and_xor(w[m][0][wj], msk, bas), a3 = lop_and_xor(w[m][1][wj], msk, bas);
                        const int qu = (m == 4) ? 1 : 0;
#pragma unroll
                        for (int nt = 0; nt < NTK; ++nt)
                            mma_f16(acc[m][nt], a0, a1, a2, a3, bq[qu][ks][nt][0], bq[qu][ks][nt][1]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NTK; ++nt) {
                    const int hg = 4 * nt + tig;
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        float code2 = 0.f;
#pragma unroll
                        for (int m = 0; m < 4; ++m) code2 = fmaf(A[m], acc[m][nt][2 * r] + acc[m][nt][2 * r + 1], code2);
                        const float dot_c = code2 - cq[nt];
                        const float dot_q = acc[4][nt][2 * r] + acc[4][nt][2 * r + 1] - cu[nt];
                        const int tl = kBlock * k + gid + 8 * r;           // token within the chunk
                        const bool valid = ok && (tc + tl < tlim[nt]);
                        const float sc = nrm[r] * inv_sd * (dot_c * inv_sd + gam[r] * qjl * dot_q);
                        if (hg < G) sS[tl * G + hg] = valid ? sc : -INFINITY;
                    }
                }
            }
            __syncthreads();   // scores of the chunk are in sS
            // ---- online softmax: warp owns heads warp, warp + NWARP
#pragma unroll
            for (int hk = 0; hk < HPW; ++hk) {
                const int h = warp + NWARP * hk;
                if (h < G) {
                    float sc[TPL], wv[TPL];
                    float cmax = -INFINITY;
#pragma unroll
                    for (int i = 0; i < TPL; ++i) {
                        sc[i] = sS[(lane + 32 * i) * G + h];
                        cmax = fmaxf(cmax, sc[i]);
                    }
                    cmax = warp_max(cmax);
                    const float m_new = fmaxf(m_run[hk], cmax);
                    const float alpha = (m_run[hk] == -INFINITY) ? 0.f : __expf(m_run[hk] - m_new);
                    float psum = 0.f, wmax = 0.f;
#pragma unroll
                    for (int i = 0; i < TPL; ++i) {
                        const int tl = lane + 32 * i;
                        const float p = (sc[i] == -INFINITY) ? 0.f : __expf(sc[i] - m_new);
                        const float nv = __half2float(*reinterpret_cast<const __half *>(
                            vb_base + (size_t)(tl >> 4) * VREC + 6 * D + 2 * (tl & 15)));
                        wv[i] = (p > 0.f) ? p * nv * inv_sd : 0.f;
                        psum += p;
                        wmax = fmaxf(wmax, fabsf(wv[i]));
                    }
                    psum = warp_sum(psum);
                    wmax = warp_max(wmax);
                    const float wr = fmaxf(w_ref[hk] * alpha, wmax);
                    const int e_new = wr > 0.f ? scale_exp(wr) : e_run[hk];
                    const float f = ldexpf(alpha, e_new - e_run[hk]);
                    const float sc2 = ldexpf(1.f, e_new);
                    float tsum = 0.f;
#pragma unroll
                    for (int i = 0; i < TPL; ++i) {
                        const __half hv = __float2half_rn(wv[i] * sc2);
                        sP[h * PROW + lane + 32 * i] = hv;
                        tsum += __half2float(hv);
                    }
                    tsum = warp_sum(tsum);
                    l_run[hk] = l_run[hk] * alpha + psum;
                    m_run[hk] = m_new;
                    w_ref[hk] = wr;
                    e_run[hk] = e_new;
                    if (lane == 0) {
                        sF[h] = f;
                        sTc[h] = tsum;
                    }
                }
            }
            __syncthreads();   // weights of the chunk are in sP, factors in sF, weight sums in sTc
            // ---- V side: coordinates of m-tiles warp*MTW .. warp*MTW+MTW-1 (columns = heads)
            {
                const float f0 = (2 * tig < G) ? sF[2 * tig] : 0.f;
                const float f1 = (2 * tig + 1 < G) ? sF[2 * tig + 1] : 0.f;
#pragma unroll
                for (int i = 0; i < MTW; ++i) {
                    arun[i][0] *= f0;
                    arun[i][1] *= f1;
                    arun[i][2] *= f0;
                    arun[i][3] *= f1;
                }
            }
            // the chunk's plane sums start from zero: chained tensor-core accumulation over a
            // whole context is not accurate enough for the 2 sum(w b) - sum(w) cancellation
            float O[4][MTW][4];
#pragma unroll
            for (int m = 0; m < 4; ++m)
#pragma unroll
                for (int i = 0; i < MTW; ++i)
#pragma unroll
                    for (int k = 0; k < 4; ++k) O[m][i][k] = 0.f;
#pragma unroll 2
            for (int kb = 0; kb < BPC; ++kb) {
                const uint8_t *rec = vb_base + (size_t)kb * VREC;
                uint32_t x[3][2];
#pragma unroll
                for (int pl = 0; pl < 3; ++pl) {
                    const uint2 wv = *reinterpret_cast<const uint2 *>(rec + pl * 2 * D + (lane * NWV + 2 * mhi) * 4);
                    x[pl][0] = wv.x;
                    x[pl][1] = wv.y;
                }
                const __half *prow = sP + gid * PROW + kBlock * kb + 2 * tig;
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(prow);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(prow + 8);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const uint32_t x0 = (m < 3) ? x[m][0] : (x[0][0] ^ x[1][0] ^ x[2][0]);
                    const uint32_t x1 = (m < 3) ? x[m][1] : (x[0][1] ^ x[1][1] ^ x[2][1]);
                    const uint32_t x0s = x0 << 8, x1s = x1 << 8;
#pragma unroll
                    for (int i = 0; i < MTW; ++i) {
                        const uint32_t a0 = lop_and_xor(x0s, vmask[i], vbase[i]), a1 = lop_and_xor(x1s, vmask[i], vbase[i]);
                        const uint32_t a2 = lop_and_xor(x0, vmask[i], vbase[i]), a3 = lop_and_xor(x1, vmask[i], vbase[i]);
                        mma_f16(O[m][i], a0, a1, a2, a3, b0, b1);
                    }
                }
            }
            // combine the planes, undo the operand offsets: sum_m A_m ((O_m - al T) 2/delta - T)
            {
                const float t0 = (2 * tig < G) ? sTc[2 * tig] : 0.f;
                const float t1c = (2 * tig + 1 < G) ? sTc[2 * tig + 1] : 0.f;
#pragma unroll
                for (int i = 0; i < MTW; ++i) {
                    const int q = 8 + ((warp * MTW + i) & 7);
                    const float inv_de = 2.f / vop_delta(q), off = (vop_alpha(q) * inv_de + 1.f) * Asum;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float s4 = fmaf(A[0], O[0][i][k], fmaf(A[1], O[1][i][k], fmaf(A[2], O[2][i][k], A[3] * O[3][i][k])));
                        arun[i][k] += fmaf(s4, inv_de, -off * ((k & 1) ? t1c : t0));
                    }
                }
            }
        }

        // ---- segment epilogue: undo the weight scale
#pragma unroll
        for (int hk = 0; hk < HPW; ++hk) {
            const int h = warp + NWARP * hk;
            if (h < G && lane == 0) {
                sM[h] = m_run[hk];
                sL[h] = l_run[hk];
                sE[h] = e_run[hk];
            }
        }
        __syncthreads();   // the staging buffers are no longer read; sAcc reuses them
#pragma unroll
        for (int i = 0; i < MTW; ++i) {
            const int mt = warp * MTW + i;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * tig + e;
                if (h < G) {
#pragma unroll
                    for (int r = 0; r < 2; ++r) sAcc[h * D + 16 * mt + gid + 8 * r] = ldexpf(arun[i][2 * r + e], -sE[h]);
                }
            }
        }
        __syncthreads();
        const int lo = sk_cta_of(us, P, W), hi = sk_cta_of(ue - 1, P, W);
        // output row of operand column h: query h / gq of head kh * gq + h % gq
        const int gq = G / q_len;
        auto out_row = [&](int h) { return ((size_t)b * q_len + h / gq) * hq + (size_t)kh * gq + h % gq; };
        if (lo == hi) {
            // the whole (sequence, kv head) was in this CTA: finish it here
            for (int h = warp; h < G; h += NWARP) {
                float v[R];
#pragma unroll
                for (int r = 0; r < R; ++r) v[r] = sAcc[h * D + 32 * r + lane];
                finish_row<D>(v, sL[h], params, out + out_row(h) * D, lane);
                if (lse && lane == 0) lse[out_row(h)] = sL[h] > 0.f ? sM[h] + logf(sL[h]) : -INFINITY;
            }
        } else {
            // leave a partial in this CTA's slot (0: its first segment, 1: its last)
            const int slot = first_seg ? 0 : 1;
#pragma unroll 1
            for (int h = 0; h < G; ++h) {
                float *dst = part + (((size_t)cta * 2 + slot) * G + h) * kPartStride(D);
                for (int i = tid; i < D; i += NT_) dst[4 + i] = sAcc[h * D + i];
                if (tid == 0) {
                    dst[0] = sM[h];
                    dst[1] = sL[h];
                }
            }
            __threadfence();                           // every thread publishes its part of the partial
            __syncthreads();
            if (tid == 0) {
                const unsigned int nseg = (unsigned int)(hi - lo + 1);
                const unsigned int done = atomicAdd(&counters[b * hkv + kh], 1u) + 1u;
                s_last = (done == nseg);
                if (s_last) counters[b * hkv + kh] = 0u;   // every segment has arrived
            }
            __syncthreads();
            if (s_last) {
                __threadfence();
                // the partial of CTA c for this unit sits in slot 0, except for the
                // first CTA when the unit does not start its range (then slot 1)
                const int slot_lo = (sk_begin(lo, P, W) >= us) ? 0 : 1;
                for (int h = warp; h < G; h += NWARP) {
                    float M = -INFINITY;
                    for (int c2 = lo; c2 <= hi; ++c2) {
                        const int sl = (c2 == lo) ? slot_lo : 0;
                        M = fmaxf(M, __ldcg(part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D)));
                    }
                    float v[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) v[r] = 0.f;
                    float l = 0.f;
                    for (int c2 = lo; c2 <= hi; ++c2) {
                        const int sl = (c2 == lo) ? slot_lo : 0;
                        const float *ps = part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D);
                        const float m = __ldcg(ps);
                        const float wgt = (m == -INFINITY) ? 0.f : __expf(m - M);
                        l = fmaf(__ldcg(ps + 1), wgt, l);
#pragma unroll
                        for (int r = 0; r < R; ++r) v[r] = fmaf(__ldcg(ps + 4 + 32 * r + lane), wgt, v[r]);
                    }
                    finish_row<D>(v, l, params, out + out_row(h) * D, lane);
                    if (lse && lane == 0) lse[out_row(h)] = l > 0.f ? M + logf(l) : -INFINITY;
                }
            }
        }
        __syncthreads();   // sAcc and the small shared arrays are rewritten by the next segment

        g = se;
        if (g >= g1) break;
        first_seg = false;
        if (++kh == hkv) {         // next sequence with a nonempty context
            kh = 0;
            do {
                ++b;
                ub = cpre[b];
                nchb = (int)((cpre[b + 1] - ub) / hkv);
            } while (nchb == 0);
        }
    }
}

// Persistent CTAs of the pass on the current device: up to kCtasPerSm per SM
// (fewer if the kernel's resources allow fewer), for at most kMaxSms SMs.
template <int D, int G>
int pass_ctas() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    constexpr int NWARP = pass_warps(G);
    constexpr size_t smem = split_smem_bytes<D, G, NWARP>();
    auto kern = decode_mma_kernel<D, G, NWARP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NWARP * 32, smem) != cudaSuccess) return 0;
    occ = occ < 1 ? 1 : (occ > kCtasPerSm ? kCtasPerSm : occ);
    sms = sms > kMaxSms ? kMaxSms : sms;
    return occ * sms;
}

template <int D>
int pass_ctas_g(int G) {
    switch (G) {
        case 1: return pass_ctas<D, 1>();
        case 2: return pass_ctas<D, 2>();
        case 3: return pass_ctas<D, 3>();
        case 4: return pass_ctas<D, 4>();
        case 5: return pass_ctas<D, 5>();
        case 6: return pass_ctas<D, 6>();
        case 7: return pass_ctas<D, 7>();
        default: return pass_ctas<D, 8>();
    }
}

// Cached per (device, d, G): query prep and the pass must agree on it, and the
// occupancy query is not free.
int pass_ctas_any(int d, int G) {
    constexpr int kDevs = 64;
    static std::atomic<int> cache[kDevs][2][9];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || G < 1 || G > 8) return 0;
    if (dev >= kDevs) return d == 128 ? (TQ_DECODE_WARP ? warp_pass_ctas(G) : pass_ctas_g<128>(G)) : pass_ctas_g<256>(G);
    std::atomic<int> &slot = cache[dev][d == 128 ? 0 : 1][G];
    int n = slot.load(std::memory_order_relaxed);
    if (n == 0) {
        n = d == 128 ? (TQ_DECODE_WARP ? warp_pass_ctas(G) : pass_ctas_g<128>(G)) : pass_ctas_g<256>(G);
        slot.store(n, std::memory_order_relaxed);
    }
    return n;
}

template <int D, int NTK, typename T>
cudaError_t qprep_launch_t(const uint8_t *P, const void *q, int batch, int q_len, int hq, int hkv,
                           const int32_t *ctx_lens, int max_ctx, int nctas, const WsLayout &w, cudaStream_t st) {
    constexpr size_t smem = qprep_smem<D>();
    auto kern = qprep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(batch * q_len * hq + kQRows - 1) / kQRows + 1, 128, smem, st>>>(P, (const T *)q, batch, q_len, hq, hkv, ctx_lens,
                                                                       max_ctx, pass_chunk(q_len * hq / hkv), nctas,
                                                                       w.packs, w.counters, w.cpre, w.cta_b);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t qprep_launch(const uint8_t *P, const void *q, int batch, int q_len, int hq, int hkv,
                         const int32_t *ctx_lens, int max_ctx, int nctas, const WsLayout &w, cudaStream_t st) {
    // n-tile count of the K-side operand: (2G + 7) / 8 for G = q_len * hq / hkv columns, as in the passes
    if (q_len * hq / hkv <= 4)
        return qprep_launch_t<D, 1, T>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
    return qprep_launch_t<D, 2, T>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
}

template <int D, int G>
cudaError_t pass_launch_g(int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq, int hkv,
                          const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                          const int32_t *ctx, int ctx_add, int max_ctx, const WsLayout &w, float *out,
                          float *lse, int32_t *status) {
    constexpr int NWARP = pass_warps(G);
    constexpr size_t smem = split_smem_bytes<D, G, NWARP>();
    auto kern = decode_mma_kernel<D, G, NWARP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pass(kern, nctas, NWARP * 32, smem, st, P, w.packs, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx,
                       ctx_add, max_ctx, w.cpre, w.cta_b, w.part, w.counters, out, lse, status);
}

template <int D>
cudaError_t pass_launch(int G, int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq, int hkv,
                        const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                        const int32_t *ctx, int ctx_add, int max_ctx, const WsLayout &w, float *out,
                        float *lse, int32_t *status) {
#define TQ_PASS(GG) return pass_launch_g<D, GG>(nctas, st, P, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx, ctx_add, max_ctx, w, out, lse, status)
    switch (G) {
        case 1: TQ_PASS(1);
        case 2: TQ_PASS(2);
        case 3: TQ_PASS(3);
        case 4: TQ_PASS(4);
        case 5: TQ_PASS(5);
        case 6: TQ_PASS(6);
        case 7: TQ_PASS(7);
        default: TQ_PASS(8);
    }
#undef TQ_PASS
}

}  // namespace

cudaError_t launch_qprep(int d, int dtype, const void *params, const void *q, int batch, int q_len, int hq,
                         int hkv, const int32_t *ctx_lens, int max_ctx, void *ws, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int nctas = pass_ctas_any(d, q_len * hq / hkv);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128)
        return dtype == TQ_DTYPE_BF16
                   ? qprep_launch<128, __nv_bfloat16>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st)
                   : qprep_launch<128, float>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
    return dtype == TQ_DTYPE_BF16
               ? qprep_launch<256, __nv_bfloat16>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st)
               : qprep_launch<256, float>(P, q, batch, q_len, hq, hkv, ctx_lens, max_ctx, nctas, w, st);
}

cudaError_t launch_splitk(int d, const void *params, int batch, int q_len, int hq, int hkv, const void *k_pool,
                          const void *v_pool, int64_t num_blocks, const int32_t *block_table, int max_blocks,
                          const int32_t *ctx_lens, int ctx_add, int max_ctx, float *out, void *ws, int32_t *status,
                          cudaStream_t st, float *lse) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int G = q_len * hq / hkv;   // operand columns per kv head
    const int nctas = pass_ctas_any(d, G);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    if (d == 128 && TQ_DECODE_WARP)
        return warp_pass_launch(G, nctas, st, P, batch, q_len, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                                num_blocks, block_table, max_blocks, ctx_lens, ctx_add, max_ctx, w, out, lse, status);
    if (d == 128)
        return pass_launch<128>(G, nctas, st, P, batch, q_len, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                                num_blocks, block_table, max_blocks, ctx_lens, ctx_add, max_ctx, w, out, lse, status);
    return pass_launch<256>(G, nctas, st, P, batch, q_len, hq, hkv, (const uint8_t *)k_pool, (const uint8_t *)v_pool,
                            num_blocks, block_table, max_blocks, ctx_lens, ctx_add, max_ctx, w, out, lse, status);
}

// ---------------------------------------------------------------- the decode step: append, then attend
// One launch runs the append of one token per sequence (K tiles, V tiles) and the query prep
// side by side; the pass follows.  pre_lens[b] is the position of the new token, and the pass
// attends pre_lens[b] + 1 tokens.
namespace {
// K append tiles hold one vector (all four warps share its QJL projection: 128 FMA per thread),
// V tiles four (no projection)
constexpr int kAppendTileK = 1, kAppendTileV = 4;

template <int D, int NTK, typename T>
__global__ void __launch_bounds__(128)
step_prep_kernel(const uint8_t *__restrict__ params, const T *__restrict__ k_new, const T *__restrict__ v_new,
                 const T *__restrict__ q, int batch, int q_len, int hq, int hkv, SlotMap map, uint8_t *__restrict__ k_pool,
                 uint8_t *__restrict__ v_pool, int n_app_k, int n_app_v, int max_ctx, int chunk, int P,
                 uint8_t *__restrict__ packs,
                 unsigned int *__restrict__ counters, int64_t *__restrict__ cpre, int32_t *__restrict__ cta_b,
                 int32_t *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    pdl_launch_dependents();
    const int blk = blockIdx.x;
    if (blk < n_app_k) {
        encode_tiles<D, kAppendTileK, T>(params, k_new, (int64_t)batch * q_len * hkv, map, k_pool, true, true, blk,
                                         n_app_k, smem, status);
    } else if (blk < n_app_k + n_app_v) {
        encode_tiles<D, kAppendTileV, T>(params, v_new, (int64_t)batch * q_len * hkv, map, v_pool, false, false,
                                         blk - n_app_k, n_app_v, smem, status);
    } else if (blk == gridDim.x - 1) {   // the last CTA lays out the pass's work
        build_schedule(map.ctx_lens, q_len, batch, hkv, max_ctx, chunk, P, cpre, cta_b);
    } else {
        qprep_rows<D, NTK, T>(params, q, batch, q_len, hq, hkv, map.ctx_lens, q_len, max_ctx, chunk, P, packs, counters, cpre,
                              cta_b, blk - n_app_k - n_app_v, smem);
    }
}

template <int D, int NTK, typename T>
cudaError_t step_prep_launch(const uint8_t *P, const void *k_new, const void *v_new, const void *q, int batch,
                             int q_len, int hq, int hkv, const SlotMap &map, void *kp, void *vp, int max_ctx,
                             int nctas, const WsLayout &w, int32_t *status, cudaStream_t st) {
    constexpr size_t ek = EncSmem<D, kAppendTileK>::kBytes, ev = EncSmem<D, kAppendTileV>::kBytes;
    constexpr size_t es = ek > ev ? ek : ev, qs = qprep_smem<D>();
    constexpr size_t smem = es > qs ? es : qs;
    auto kern = step_prep_kernel<D, NTK, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int n_app_k = (batch * q_len * hkv + kAppendTileK - 1) / kAppendTileK;
    const int n_app_v = (batch * q_len * hkv + kAppendTileV - 1) / kAppendTileV;
    const int n_q = (batch * q_len * hq + kQRows - 1) / kQRows;
    kern<<<n_app_k + n_app_v + n_q + 1, 128, smem, st>>>(P, (const T *)k_new, (const T *)v_new, (const T *)q, batch, q_len, hq,
                                             hkv, map, (uint8_t *)kp, (uint8_t *)vp, n_app_k, n_app_v, max_ctx,
                                             pass_chunk(q_len * hq / hkv), nctas, w.packs, w.counters, w.cpre, w.cta_b,
                                             status);
    return cudaGetLastError();
}

template <int D, typename T>
cudaError_t step_prep_any(const uint8_t *P, const void *k_new, const void *v_new, const void *q, int batch, int q_len,
                          int hq, int hkv, const SlotMap &map, void *kp, void *vp, int max_ctx, int nctas,
                          const WsLayout &w, int32_t *status, cudaStream_t st) {
    if (q_len * hq / hkv <= 4)
        return step_prep_launch<D, 1, T>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, max_ctx, nctas, w,
                                         status, st);
    return step_prep_launch<D, 2, T>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, kp, vp, max_ctx, nctas, w,
                                     status, st);
}
}  // namespace

cudaError_t launch_step(int d, int dtype, const void *params, const void *k_new, const void *v_new, const void *q,
                        int batch, int q_len, int hq, int hkv, const int32_t *block_table, int max_blocks,
                        const int32_t *pre_lens, int max_ctx, void *k_pool, void *v_pool, int64_t num_blocks,
                        float *out, void *ws, int32_t *status, cudaStream_t st) {
    const WsLayout w = ws_layout(ws, d, batch, q_len * hq);
    const int nctas = pass_ctas_any(d, q_len * hq / hkv);
    if (nctas <= 0) return cudaErrorInvalidConfiguration;
    const uint8_t *P = (const uint8_t *)params;
    SlotMap map{nullptr, block_table, pre_lens, max_blocks, num_blocks, hkv};
    map.q_len = q_len;
    cudaError_t e;
    if (d == 128)
        e = dtype == TQ_DTYPE_BF16
                ? step_prep_any<128, __nv_bfloat16>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool,
                                                    max_ctx, nctas, w, status, st)
                : step_prep_any<128, float>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool, max_ctx,
                                            nctas, w, status, st);
    else
        e = dtype == TQ_DTYPE_BF16
                ? step_prep_any<256, __nv_bfloat16>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool,
                                                    max_ctx, nctas, w, status, st)
                : step_prep_any<256, float>(P, k_new, v_new, q, batch, q_len, hq, hkv, map, k_pool, v_pool, max_ctx,
                                            nctas, w, status, st);
    if (e != cudaSuccess) return e;
    return launch_splitk(d, params, batch, q_len, hq, hkv, k_pool, v_pool, num_blocks, block_table, max_blocks,
                         pre_lens, q_len, max_ctx, out, ws, status, st);
}

}  // namespace tq
