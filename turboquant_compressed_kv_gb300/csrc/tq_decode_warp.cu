// tq_decode_warp.cu -- the decode pass: every warp scores, weighs and sums its own 16-token
// blocks end to end (d = 128 and d = 256).
//
// Method as in tq_decode.cu (scores and value sums in the rotated domain, straight from the
// packed cells, signs and fp16 norms: the "fused dequantisation" of the SwiftLM README,
// "TurboQuantization: KV Cache Compression"; blocks through the block table of the vLLM-MLX
// explainer, "Paged KVキャッシュ"), with the stream-K schedule, workspace and merge described
// there.  Inside a CTA:
//  * A CTA of 4 warps takes 128-token chunks; warp w owns blocks 2w, 2w+1 of each chunk and
//    stages them itself (cp.async, one pair ahead), so the chunk loop has no CTA-wide barrier.
//  * Operands by table lookup.  The codebook is read as eight binary16 values T[j] =
//    f16(alpha c[j]) (alpha from the params header, worst level error under 2e-5 after
//    dividing by alpha).  A record word holds eight 4-bit fields; masked to their cell bits,
//    four fields are the selector of two PRMTs over byte tables of T (low bytes, high bytes),
//    and two more PRMTs interleave the bytes into two f16x2 registers: an mma.sync A operand
//    with the codebook value of each (token, coordinate) (K side) or (coordinate, token)
//    (V side).  One operand plane replaces four +-1 planes of the codebook's Walsh
//    decomposition, so the pass issues 24 mma per block instead of 76.
//  * K side: the codebook plane against q-bar / alpha, the QJL plane (bit 3 of each K field,
//    one LOP3 per register: 0 / delta or +-2^-14 by bit position) against u, both f16 hi/lo.
//  * Online softmax in registers, per warp and head, with a lazily moved reference:
//    weights are 2^(s - m) * nv with s in log2 units, and m only moves when a block's
//    maximum passes m + 8 (or a weight would leave the f16 range), so the accumulators
//    are rescaled rarely.
//  * V side: one mma per m-tile and block, against the weights (f16 hi in columns 0..3 and
//    f16 lo in 4..7 for up to 4 heads, f16 for 5..8), each block's sum started from zero and
//    added to fp32 running sums (chained tensor-core accumulation over thousands of tokens is
//    not accurate enough).
//  * At the end of a (sequence, kv head) segment the 4 warps' (m, l, acc) are merged in
//    shared memory, then the segment is finished, or, when other CTAs hold parts of it, left as
//    a partial (m in log2 units) for the merge kernel that follows the pass.
#include "tq_split.cuh"

#ifndef TQ_WARP_BQ_SMEM
#define TQ_WARP_BQ_SMEM 0        // 1: K-side query fragments read from shared memory for every shape
#endif
#ifndef TQ_WARP_MINBLOCKS
#define TQ_WARP_MINBLOCKS 3      // resident CTAs per SM the register budget is sized for (d = 128)
#endif
#ifndef TQ_WARP_NBUF
#define TQ_WARP_NBUF 3           // staging buffers per warp: chunks in flight = NBUF - 1 ahead of the one in use
#endif
#ifndef TQ_WARP_MINBLOCKS_256
#define TQ_WARP_MINBLOCKS_256 2  // the same at d = 256
#endif

namespace tq {
namespace {

constexpr int kWWarps = 4, kWBpw = TQ_SPLITK_BPW, kWBuf = TQ_WARP_NBUF;
constexpr float kTau = 8.f;          // the reference moves when a block's maximum passes it by this (log2)
constexpr float kWLimit = 32768.f;   // largest weight held (f16 max is 65504)
constexpr float kNoRef = -1e30f;     // softmax reference before the first unmasked score

template <int G>
__host__ __device__ constexpr int w_ntk() { return (2 * G + 7) / 8; }
// K-side query fragments in shared memory rather than registers: above 4 heads (two n-tiles)
// and at d = 256 (16 k-steps), where registers would hold 64 of them
template <int D, int G>
__host__ __device__ constexpr bool w_bq_smem() { return TQ_WARP_BQ_SMEM || G > 4 || D > 128; }
template <int D>
__host__ __device__ constexpr int w_rec() { return (int)(k_record(D) + v_record(D)); }

template <int D, int G>
__host__ __device__ constexpr size_t warp_smem_bytes() {
    const size_t stage = (size_t)kWWarps * kWBuf * kWBpw * w_rec<D>();   // per warp: NBUF buffers x BPW blocks
    const size_t merge = (size_t)(kWWarps + 1) * G * D * 4;              // sAccW + sAcc
    const size_t bq = w_bq_smem<D, G>() ? (size_t)2 * (D / 16) * w_ntk<G>() * 64 * 4 : 0;
    return stage + merge + bq;
}

// ld.shared of a query fragment at each use: a plain load would be hoisted out of the block
// loop by the compiler and pin the fragments in registers
__device__ __forceinline__ uint2 lds_u2(const uint32_t *p) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y) : "r"((uint32_t)__cvta_generic_to_shared(p)));
    return v;
}

// 2^x for a per-token softmax weight (x <= 8 in log2 units, or -inf): the hardware approximation
// with results below 2^-126 flushed to 0, which drops the subnormal range handling of exp2f (a
// weight that small is below the fp32 resolution of the sum it joins)
__device__ __forceinline__ float weight_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

template <int D, int G>
__global__ void __launch_bounds__(kWWarps * 32, D == 128 ? TQ_WARP_MINBLOCKS : TQ_WARP_MINBLOCKS_256)
decode_warp_kernel(const uint8_t *__restrict__ params, const uint8_t *__restrict__ packs, int batch, int q_len, int hq, int hkv,
                   const uint8_t *__restrict__ k_pool, const uint8_t *__restrict__ v_pool, int64_t num_blocks,
                   const int32_t *__restrict__ block_table, int max_blocks, const int32_t *__restrict__ ctx_lens,
                   int ctx_add, int max_ctx, int early, int64_t *__restrict__ cpre, float *__restrict__ part,
                   float *__restrict__ out, float *__restrict__ lse, int32_t *status) {
    constexpr int NT = kWWarps * 32, NWARP = kWWarps, BPW = kWBpw, NBUF = kWBuf;
    static_assert(NBUF * BPW <= 30, "buffer validity bits");
    constexpr int CH = kBlock * NWARP * BPW;    // tokens per chunk (the schedule's unit)
    constexpr int NTK = w_ntk<G>();             // K-side n-tiles; thread holds heads 4*nt + tig
    constexpr int NKS = D / 16, MT = D / 16, R = D / 32;
    constexpr int NW = D / 32;                  // K words per (lane, token row)
    constexpr int NG = D / 128;                 // V slot groups per lane (3 words per pair each)
    constexpr int KREC = (int)k_record(D), VREC = (int)v_record(D), REC = KREC + VREC;
    constexpr size_t kStage = (size_t)NWARP * NBUF * BPW * REC;
    constexpr size_t kMerge = (size_t)(NWARP + 1) * G * D * 4;
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.6931471805599453f;
    constexpr bool BQS = w_bq_smem<D, G>();

    extern __shared__ __align__(16) uint8_t smem[];
    const int cta = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, gid = lane >> 2, tig = lane & 3;
    uint8_t *sStage = smem + (size_t)warp * NBUF * BPW * REC;  // this warp's [NBUF][BPW][K record | V record]
    float *sAccW = reinterpret_cast<float *>(smem + kStage);     // [NWARP][G][D], segment end only
    float *sAcc = sAccW + NWARP * G * D;                         // [G][D]
    uint32_t *sBq = reinterpret_cast<uint32_t *>(smem + kStage + kMerge);
    __shared__ float sMW[NWARP][8], sLW[NWARP][8];
    __shared__ float sM[8], sL[8];

    // what depends on no earlier kernel of the stream runs before the wait: the params header's
    // table and the staging area, zeroed so that slots of blocks that are not copied always hold
    // finite values (old records or zeros), whose weight is exactly 0
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    const uint32_t L0 = ph->lut_lo[0], L1 = ph->lut_lo[1], H0 = ph->lut_hi[0], H1 = ph->lut_hi[1];
    const float inv_alpha = ph->inv_alpha;
    for (int i = tid; i < (int)(kStage / 16); i += NT) reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    // The schedule, the first segment and its first block ids depend only on the lengths and the
    // block table, which the prep launch before this one does not write: with `early` they are
    // worked out before the wait, overlapping that launch (the prep is an ordinary launch, so
    // every kernel before it has completed).  The packs and the records (the step's appended
    // token) are read after it.
    if (!early) pdl_wait();
    const PassSched sc = pass_schedule<NT>(ctx_lens, ctx_add, batch, hkv, max_ctx, CH, cpre);
    const int64_t W = sc.W;
    const int P = sc.P;
    const bool works = cta < P;
    const int64_t g0 = works ? sk_begin(cta, P, W) : 0, g1 = works ? sk_begin(cta + 1, P, W) : 0;
    const float inv_sd = rsqrtf((float)D);
    const float c_sc = inv_sd * kLog2e;                             // scores in log2 units
    const float qjl = 1.2533141373155003f / (float)D * 65536.f;    // sqrt(pi/2) / d, and 1 / 2^-16 of the operands

    // The CTA's range [g0, g1) of global chunks, walked one (sequence, kv head) segment at a time.
    struct Seg {
        int b, kh, t0, t1, L;
        int64_t us, ue, se;   // chunks [us, ue) of the segment's (sequence, kv head); the CTA's part ends at se
    };
    // chunks per kv head of sequence b
    auto nchunks = [&](int b) { return (attended_len(ctx_lens[b], ctx_add, max_ctx) + CH - 1) / CH; };
    auto make_seg = [&](int b, int kh, int64_t ub, int nchb, int64_t g) {
        Seg s;
        s.b = b;
        s.kh = kh;
        s.us = ub + (int64_t)kh * nchb;
        s.ue = s.us + nchb;
        s.se = (g1 < s.ue) ? g1 : s.ue;
        s.t0 = (int)(g - s.us) * CH;
        s.L = attended_len(ctx_lens[b], ctx_add, max_ctx);
        s.t1 = min(s.L, (int)(s.se - s.us) * CH);
        return s;
    };
    // the segment after s, if the range has one
    auto next_seg = [&](const Seg &s, Seg &n) -> bool {
        if (s.se >= g1) return false;
        int nb = s.b, nkh = s.kh + 1, nn = (int)(s.ue - s.us);
        int64_t nub = s.us - (int64_t)s.kh * nn;   // the sequence's first chunk
        if (nkh == hkv) {   // the next sequence with chunks (one exists: s.se < g1 <= W)
            nkh = 0;
            nub += (int64_t)hkv * nn;
            do {
                ++nb;
                nn = nchunks(nb);
            } while (nn == 0 && nb + 1 < batch);
        }
        n = make_seg(nb, nkh, nub, nn, s.se);
        return true;
    };
    // stage this warp's blocks of the chunk at token tc of segment s into buffer buf; bit bw
    // of the result is set when block bw is in range and has a valid physical id.  Blocks past
    // the context are not copied; a block with a bad id is replaced by block 0 (its scores are
    // masked), so the copies need no per-lane branch.
    // The block ids of a position are read one prefetch step before they are used, so that their
    // load overlaps a chunk of work instead of delaying the copies: id -2 = past the context.
    auto load_ids = [&](const Seg &s, int tc, int64_t (&ids)[BPW]) {
#pragma unroll
        for (int bw = 0; bw < BPW; ++bw) {
            const int tb = tc + kBlock * (BPW * warp + bw);
            ids[bw] = (tb < s.t1) ? block_of(block_table, s.b, max_blocks, tb / kBlock, num_blocks) : -2;
        }
    };
    auto stage = [&](const Seg &s, const int64_t (&ids)[BPW], int buf) -> int {
        int okm = 0;
#pragma unroll
        for (int bw = 0; bw < BPW; ++bw) {
            const int64_t p = ids[bw];
            if (p != -2) {
                if (p < 0 && lane == 0) flag_status(status, TQ_STATUS_BAD_SLOT);
                okm |= (p >= 0) << bw;
                const size_t row = (size_t)(p < 0 ? 0 : p) * hkv + s.kh;
                const uint8_t *gk = k_pool + row * KREC, *gv = v_pool + row * VREC;
                uint8_t *dk = sStage + (size_t)(buf * BPW + bw) * REC, *dv = dk + KREC;
#pragma unroll
                for (int j0 = 0; j0 < KREC / 16; j0 += 32)
                    if (j0 + 32 <= KREC / 16 || j0 + lane < KREC / 16) cp_async16(dk + 16 * (j0 + lane), gk + 16 * (j0 + lane));
#pragma unroll
                for (int j0 = 0; j0 < VREC / 16; j0 += 32)
                    if (j0 + 32 <= VREC / 16 || j0 + lane < VREC / 16) cp_async16(dv + 16 * (j0 + lane), gv + 16 * (j0 + lane));
            }
        }
        cp_async_commit();
        return okm;
    };

    Seg s{};
    if (works) {
        const int n0 = nchunks(sc.b0);
        s = make_seg(sc.b0, (int)((g0 - sc.ub0) / n0), sc.ub0, n0, g0);
    }
    bool first_seg = true;
    // Prefetch cursor: the chunks of the CTA's range in order, NBUF - 1 ahead of the one in use,
    // across segment boundaries.  Every step commits one cp.async group (empty past the range),
    // so waiting for all but the newest NBUF - 1 groups completes the chunk in use.
    Seg ps = s;
    int ptc = s.t0;
    bool pmore = true;
    int okm = 0;   // bit NBUF-slot * BPW + bw: block bw of the buffer is in range with a valid id
    int buf = 0, pbuf = 0;
    int64_t pids[BPW];
    if (works) load_ids(ps, ptc, pids);
    auto prefetch = [&]() {
        int bits = 0;
        if (pmore) {
            bits = stage(ps, pids, pbuf);
            ptc += CH;
            if (ptc >= ps.t1) {
                Seg n2;
                pmore = next_seg(ps, n2);
                if (pmore) {
                    ps = n2;
                    ptc = ps.t0;
                }
            }
            if (pmore) load_ids(ps, ptc, pids);   // for the next step
        } else {
            cp_async_commit();
        }
        okm = (okm & ~(((1 << BPW) - 1) << (pbuf * BPW))) | (bits << (pbuf * BPW));
        pbuf = (pbuf + 1 == NBUF) ? 0 : pbuf + 1;
    };
    // With `early`, the first chunks are staged before the wait too, as long as they hold no
    // position the step appends (tokens from the stored length ctx_lens[b] on): the prep writes
    // only those records (and the packs, read after the wait).
    int npre = 0;
    if (early && works)
        while (npre < NBUF - 1 && pmore && ptc + CH <= ctx_lens[ps.b]) {
            prefetch();
            ++npre;
        }
    if (early) pdl_wait();
    pdl_launch_dependents();   // the merge kernel's CTAs may be placed as this pass's CTAs exit

    for (int b = cta; b < batch; b += gridDim.x)
        if (attended_len(ctx_lens[b], ctx_add, max_ctx) == 0)
        {
            for (int i = tid; i < q_len * hq * D; i += NT) out[(size_t)b * q_len * hq * D + i] = 0.f;
            if (lse)
                for (int i = tid; i < q_len * hq; i += NT) lse[(size_t)b * q_len * hq + i] = -INFINITY;
        }
    if (!works) return;
    for (int k = npre; k < NBUF - 1; ++k) prefetch();

#pragma unroll 1
    while (true) {
        const int b = s.b, kh = s.kh, t0 = s.t0, t1 = s.t1;
        const int64_t us = s.us, ue = s.ue;
        Seg ns;
        const bool more_segs = next_seg(s, ns);

        // K-side query fragments and the QJL offset constants of this (sequence, kv head)
        const uint8_t *pack = packs + ((size_t)b * hkv + kh) * kPackBytes(D);
        const float *pf = reinterpret_cast<const float *>(pack) + kPackFloatOff(D);
        uint32_t bq[BQS ? 1 : 2][BQS ? 1 : NKS][NTK][2];
        if constexpr (BQS) {
            __syncthreads();   // the previous segment's reads of sBq are done
            for (int i = tid; i < 2 * NKS * NTK * 64 / 4; i += NT)
                reinterpret_cast<uint4 *>(sBq)[i] = reinterpret_cast<const uint4 *>(pack)[i];
            __syncthreads();
        } else {
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
        }
        auto bfrag = [&](int qu, int ks, int nt) -> uint2 {
            if constexpr (BQS) return lds_u2(sBq + ((qu * NKS + ks) * NTK + nt) * 64 + lane * 2);
            else return make_uint2(bq[qu][ks][nt][0], bq[qu][ks][nt][1]);
        };
        float cu[NTK];
        // tokens column 4 nt + tig attends in this segment (query i: L - (q_len - 1 - i)); tmin: all
        // columns attend the tokens below it
        int tlim[NTK];
        const int tmin = min(t1, s.L - (q_len - 1));
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            const int hg = 4 * nt + tig;
            cu[nt] = hg < G ? pf[8 + hg] : 0.f;
            tlim[nt] = hg < G ? min(t1, s.L - (q_len - 1 - hg / (G / q_len))) : 0;
        }

        // running value sums (fp32 adds of the per-block mma results)
        float arun[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int k = 0; k < 4; ++k) arun[mt][k] = 0.f;
        float mref[NTK], lpart[NTK];
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            mref[nt] = kNoRef;   // finite: exp2(s - mref) is 0 for masked scores (s = -inf) at any time
            lpart[nt] = 0.f;
        }

        // multiply the accumulators and row sums of head h (= 4 nt + tig) by f[nt]
        auto rescale = [&](const float (&f)[NTK]) {
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt) lpart[nt] *= f[nt];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                // accumulator column c holds head c (G > 4) or head c & 3 (G <= 4: hi, then lo parts)
                const int c = 2 * tig + e, hc = (G <= 4) ? (c & 3) : c;
                float fc = 1.f;
#pragma unroll
                for (int nt = 0; nt < NTK; ++nt) {
                    const float v = __shfl_sync(0xffffffffu, f[nt], (lane & ~3) | (hc & 3));
                    if ((hc >> 2) == nt) fc = v;
                }
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    arun[mt][e] *= fc;
                    arun[mt][2 + e] *= fc;
                }
            }
        };

        // this lane's V words: pair 0 (tokens 2tig, 2tig+1), pair 1 (+8)
        auto load_vw = [&](const uint8_t *vrec, uint32_t (&vw)[2][3 * NG]) {
            if constexpr (NG == 1) {
#pragma unroll
                for (int c = 0; c < 3; ++c) {
                    const uint2 v = reinterpret_cast<const uint2 *>(vrec + lane * 24)[c];
                    vw[(2 * c) / 3][(2 * c) % 3] = v.x;
                    vw[(2 * c + 1) / 3][(2 * c + 1) % 3] = v.y;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 3 * NG / 2; ++c) {
                    const uint4 v = reinterpret_cast<const uint4 *>(vrec + lane * 24 * NG)[c];
                    const uint32_t x4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) vw[(4 * c + k) / (3 * NG)][(4 * c + k) % (3 * NG)] = x4[k];
                }
            }
        };
#pragma unroll 1
        for (int tc = t0; tc < t1; tc += CH, buf = (buf + 1 == NBUF) ? 0 : buf + 1) {
            prefetch();                      // into the buffer the previous chunk used
            cp_async_wait_n<NBUF - 1>();     // the chunk in `buf` has arrived
            __syncwarp();
            const int tbw = tc + kBlock * BPW * warp;   // first token of this warp's blocks
            if (tbw < t1) {
                // ---- K side of the warp's blocks: scores of tokens tb + gid + 8r, heads 4 nt + tig (log2 units)
                float s2[BPW][NTK][2];
#pragma unroll
                for (int bw = 0; bw < BPW; ++bw) {
                    const int tb = tbw + kBlock * bw;
                    const bool ok = (okm >> (buf * BPW + bw)) & 1;
                    const bool full = ok && tb + kBlock <= tmin;   // every score of the block is attended
                    const uint8_t *krec = sStage + (size_t)(buf * BPW + bw) * REC;
                    uint32_t kw[2][NW];   // this lane's words: token rows gid (r = 0) and gid + 8 (r = 1)
#pragma unroll
                    for (int c = 0; c < NW / 2; ++c) {
                        const uint4 v = reinterpret_cast<const uint4 *>(krec + lane * 8 * NW)[c];
                        const int r = (4 * c) / NW, w0 = (4 * c) % NW;
                        kw[r][w0] = v.x;
                        kw[r][w0 + 1] = v.y;
                        kw[r][w0 + 2] = v.z;
                        kw[r][w0 + 3] = v.w;
                    }
                    float nrm[2], gam[2];
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const __half2 ng = *reinterpret_cast<const __half2 *>(krec + 8 * D + 4 * (gid + 8 * r));
                        nrm[r] = __low2float(ng) * c_sc;
                        gam[r] = __high2float(ng) * qjl;
                    }
                    float accc[NTK][4], accq[NTK][4];   // started by the first k-step's zero-accumulator mma
#pragma unroll
                    for (int ks = 0; ks < NKS; ++ks) {
                        // codebook plane: fields 4h .. 4h+3 of word ks/2 are the columns 2tig, 2tig+1,
                        // 2tig+8, 2tig+9 of k-step ks
                        uint32_t a01[2], a23[2];
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const uint32_t m = kw[r][ks >> 1] & 0x77777777u;
                            const uint32_t sel = (ks & 1) ? (m >> 16) : m;
                            const uint32_t pl = prmt(L0, L1, sel), phb = prmt(H0, H1, sel);
                            a01[r] = prmt(pl, phb, 0x5140u);
                            a23[r] = prmt(pl, phb, 0x7362u);
                        }
#pragma unroll
                        for (int nt = 0; nt < NTK; ++nt) {
                            const uint2 bb = bfrag(0, ks, nt);
                            if (ks == 0) mma_f16_z(accc[nt], a01[0], a01[1], a23[0], a23[1], bb.x, bb.y);
                            else mma_f16(accc[nt], a01[0], a01[1], a23[0], a23[1], bb.x, bb.y);
                        }
                        // QJL plane, k-step ks: field positions i0 = 2 (ks & 1) (columns 2tig, 2tig+1)
                        // and i0 + 1 (2tig+8, 2tig+9) of word ks/2, the two halves being the columns' pair
                        const int i0 = 2 * (ks & 1), i1 = i0 + 1;
                        const uint32_t m0 = 0x00010001u << (4 * i0 + 3), m1 = 0x00010001u << (4 * i1 + 3);
                        const uint32_t q0 = lop_and_xor(kw[0][ks >> 1], m0, qjl_base(i0));
                        const uint32_t q1 = lop_and_xor(kw[1][ks >> 1], m0, qjl_base(i0));
                        const uint32_t q2 = lop_and_xor(kw[0][ks >> 1], m1, qjl_base(i1));
                        const uint32_t q3 = lop_and_xor(kw[1][ks >> 1], m1, qjl_base(i1));
#pragma unroll
                        for (int nt = 0; nt < NTK; ++nt) {
                            const uint2 bb = bfrag(1, ks, nt);
                            if (ks == 0) mma_f16_z(accq[nt], q0, q1, q2, q3, bb.x, bb.y);
                            else mma_f16(accq[nt], q0, q1, q2, q3, bb.x, bb.y);
                        }
                    }
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const float dot_c = accc[nt][2 * r] + accc[nt][2 * r + 1];
                            const float dot_q = accq[nt][2 * r] + accq[nt][2 * r + 1] - cu[nt];
                            const float sc = nrm[r] * fmaf(dot_c, inv_sd, gam[r] * dot_q);
                            s2[bw][nt][r] = (full || (ok && tb + gid + 8 * r < tlim[nt])) ? sc : -INFINITY;
                        }
                }

                // ---- online softmax over the warp's blocks: move the reference when their maximum passes it
                {
                    float f[NTK];
                    bool need = false;
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt) {
                        float bm = -INFINITY;
#pragma unroll
                        for (int bw = 0; bw < BPW; ++bw) bm = fmaxf(bm, fmaxf(s2[bw][nt][0], s2[bw][nt][1]));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
                        bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
                        const bool up = bm > mref[nt] + kTau;
                        f[nt] = up ? exp2f(mref[nt] - bm) : 1.f;
                        if (up) mref[nt] = bm;
                        need |= up;
                    }
                    if (__any_sync(0xffffffffu, need)) rescale(f);
                }
                float wv[BPW][NTK][2];
                {
                    float pr[BPW][NTK][2];
                    float wmax = 0.f;
#pragma unroll
                    for (int bw = 0; bw < BPW; ++bw) {
                        const uint8_t *vrec = sStage + (size_t)(buf * BPW + bw) * REC + KREC;
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const float nv = __half2float(*reinterpret_cast<const __half *>(vrec + 6 * D + 2 * (gid + 8 * r)));
#pragma unroll
                            for (int nt = 0; nt < NTK; ++nt) {
                                const float p = weight_exp2(s2[bw][nt][r] - mref[nt]);
                                pr[bw][nt][r] = p;
                                wv[bw][nt][r] = p * nv;
                                wmax = fmaxf(wmax, wv[bw][nt][r]);
                            }
                        }
                    }
                    if (__any_sync(0xffffffffu, wmax > kWLimit)) {
                        // a weight would leave the f16 range: raise the reference of that head
                        float f[NTK];
#pragma unroll
                        for (int nt = 0; nt < NTK; ++nt) {
                            float hm = 0.f;
#pragma unroll
                            for (int bw = 0; bw < BPW; ++bw) hm = fmaxf(hm, fmaxf(wv[bw][nt][0], wv[bw][nt][1]));
                            hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 4));
                            hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 8));
                            hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, 16));
                            const float sh = hm > kWLimit ? ceilf(log2f(hm / kWLimit)) : 0.f;
                            f[nt] = exp2f(-sh);
                            mref[nt] += sh;
#pragma unroll
                            for (int bw = 0; bw < BPW; ++bw)
#pragma unroll
                                for (int r = 0; r < 2; ++r) {
                                    pr[bw][nt][r] *= f[nt];
                                    wv[bw][nt][r] *= f[nt];
                                }
                        }
                        rescale(f);
                    }
#pragma unroll
                    for (int nt = 0; nt < NTK; ++nt)
#pragma unroll
                        for (int bw = 0; bw < BPW; ++bw) lpart[nt] += pr[bw][nt][0] + pr[bw][nt][1];
                }

                // ---- weights to the V-side B layout.  Thread (gid, tig) holds column gid: head gid & 3
                // (G <= 4; columns 4..7 carry the f16 lo parts of heads 0..3) or head gid (G > 4), at
                // tokens 2tig, 2tig+1 (b0) and 2tig+8, 2tig+9 (b1) of each block.  The weights of tokens
                // t, t+8 of head h sit in lane 4 (t & 7) + (h & 3), n-tile h >> 2, packed as one f16x2.
                uint32_t bf0[BPW], bf1[BPW];
                {
                    const int hcol = (G <= 4) ? (gid & 3) : gid;
                    const int srcX = 8 * tig + (hcol & 3), srcY = srcX + 4;
#pragma unroll
                    for (int bw = 0; bw < BPW; ++bw) {
                        uint32_t X = 0u, Y = 0u;
#pragma unroll
                        for (int nt = 0; nt < NTK; ++nt) {
                            const __half2 hh = __floats2half2_rn(wv[bw][nt][0], wv[bw][nt][1]);
                            const uint32_t wh = *reinterpret_cast<const uint32_t *>(&hh);
                            if constexpr (G <= 4) {
                                const float2 fh = __half22float2(hh);
                                const uint32_t wl = pack_h2(wv[bw][nt][0] - fh.x, wv[bw][nt][1] - fh.y);
                                const uint32_t xh = __shfl_sync(0xffffffffu, wh, srcX), yh = __shfl_sync(0xffffffffu, wh, srcY);
                                const uint32_t xl = __shfl_sync(0xffffffffu, wl, srcX), yl = __shfl_sync(0xffffffffu, wl, srcY);
                                X = gid >= 4 ? xl : xh;
                                Y = gid >= 4 ? yl : yh;
                            } else {
                                const uint32_t x = __shfl_sync(0xffffffffu, wh, srcX), y = __shfl_sync(0xffffffffu, wh, srcY);
                                if ((hcol >> 2) == nt) {
                                    X = x;
                                    Y = y;
                                }
                            }
                        }
                        if (hcol >= G) X = Y = 0u;
                        bf0[bw] = prmt(X, Y, 0x5410u);
                        bf1[bw] = prmt(X, Y, 0x7632u);
                    }
                }

                // ---- V side: per pair of m-tiles, the operands of both token pairs of every block; the
                // blocks' mma chained, then one fp32 add
                {
                    uint32_t vw[BPW][2][3 * NG];
#pragma unroll
                    for (int bw = 0; bw < BPW; ++bw)
                        load_vw(sStage + (size_t)(buf * BPW + bw) * REC + KREC, vw[bw]);
#pragma unroll
                    for (int g = 0; g < NG; ++g)
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint32_t A[BPW][2][4];   // [block][pair][slot 4k + j of the group]
#pragma unroll
                            for (int bw = 0; bw < BPW; ++bw)
#pragma unroll
                                for (int pp = 0; pp < 2; ++pp) {
                                    const uint32_t w0 = vw[bw][pp][3 * g], w1 = vw[bw][pp][3 * g + 1], w2 = vw[bw][pp][3 * g + 2];
                                    const uint32_t sw = k == 3 ? (((w0 >> 3) & 0x11111111u) | ((w1 >> 2) & 0x22222222u) |
                                                                  ((w2 >> 1) & 0x44444444u))
                                                               : (vw[bw][pp][3 * g + k] & 0x77777777u);
#pragma unroll
                                    for (int hf = 0; hf < 2; ++hf) {
                                        const uint32_t sel = hf ? (sw >> 16) : sw;
                                        const uint32_t pl = prmt(L0, L1, sel), phb = prmt(H0, H1, sel);
                                        A[bw][pp][2 * hf] = prmt(pl, phb, 0x6240u);
                                        A[bw][pp][2 * hf + 1] = prmt(pl, phb, 0x7351u);
                                    }
                                }
#pragma unroll
                            for (int hf = 0; hf < 2; ++hf) {
                                const int mt = 8 * g + 2 * k + hf;
                                float o[4];
#pragma unroll
                                for (int bw = 0; bw < BPW; ++bw) {
                                    if (bw == 0)
                                        mma_f16_z(o, A[bw][0][2 * hf], A[bw][0][2 * hf + 1], A[bw][1][2 * hf],
                                                  A[bw][1][2 * hf + 1], bf0[bw], bf1[bw]);
                                    else
                                        mma_f16(o, A[bw][0][2 * hf], A[bw][0][2 * hf + 1], A[bw][1][2 * hf],
                                                A[bw][1][2 * hf + 1], bf0[bw], bf1[bw]);
                                }
#pragma unroll
                                for (int e = 0; e < 4; ++e) arun[mt][e] += o[e];
                            }
                        }
                }
            }
            __syncwarp();   // buffer `buf` is restaged NBUF - 1 chunks later
        }

        // ---- segment end: merge the warps' (m, l, acc) in shared memory
        float lh[NTK];
#pragma unroll
        for (int nt = 0; nt < NTK; ++nt) {
            float l = lpart[nt];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            lh[nt] = l;
        }
        __syncthreads();   // the previous segment's merge is done with sAccW / sAcc
        if (gid == 0) {
#pragma unroll
            for (int nt = 0; nt < NTK; ++nt) {
                const int h = 4 * nt + tig;
                if (h < G) {
                    sMW[warp][h] = mref[nt];
                    sLW[warp][h] = lh[nt];
                }
            }
        }
        if constexpr (G <= 4) {
            // columns 4..7 (tig 2, 3) carry the lo parts of heads 0..3 (tig 0, 1): add them in
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const float o = __shfl_xor_sync(0xffffffffu, arun[mt][k], 2);
                    if (tig < 2) arun[mt][k] += o;
                }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = 2 * tig + e;
                if (h < G && (G > 4 || tig < 2)) {
#pragma unroll
                    for (int r = 0; r < 2; ++r)
                        sAccW[(warp * G + h) * D + 16 * mt + gid + 8 * r] = arun[mt][2 * r + e] * inv_alpha;
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < G * D; i += NT) {
            const int h = i / D;
            float M = -INFINITY;
#pragma unroll
            for (int w2 = 0; w2 < NWARP; ++w2) M = fmaxf(M, sMW[w2][h]);
            float v = 0.f, l = 0.f;
#pragma unroll
            for (int w2 = 0; w2 < NWARP; ++w2) {
                const float fw = (sMW[w2][h] == -INFINITY) ? 0.f : exp2f(sMW[w2][h] - M);
                v = fmaf(fw, sAccW[(w2 * G + h) * D + (i % D)], v);
                l = fmaf(fw, sLW[w2][h], l);
            }
            sAcc[i] = v * inv_sd;
            if (i % D == 0) {
                sM[h] = M;
                sL[h] = l;
            }
        }
        __syncthreads();

        const int lo = sk_cta_of(us, P, W), hi = sk_cta_of(ue - 1, P, W);
        // output row of operand column h: query h / gq of head kh * gq + h % gq
        const int gq = G / q_len;
        auto out_row = [&](int h) { return ((size_t)b * q_len + h / gq) * hq + (size_t)kh * gq + h % gq; };
        if (lo == hi) {
            for (int h = warp; h < G; h += NWARP) {
                float v[R];
#pragma unroll
                for (int r = 0; r < R; ++r) v[r] = sAcc[h * D + 32 * r + lane];
                finish_row<D>(v, sL[h], params, out + out_row(h) * D, lane);
                if (lse && lane == 0) lse[out_row(h)] = sL[h] > 0.f ? sM[h] * kLn2 + logf(sL[h]) : -INFINITY;
            }
        } else {
            const int slot = first_seg ? 0 : 1;
#pragma unroll 1
            for (int h = 0; h < G; ++h) {
                float *dst = part + (((size_t)cta * 2 + slot) * G + h) * kPartStride(D);
                for (int i = tid; i < D; i += NT) dst[4 + i] = sAcc[h * D + i];
                if (tid == 0) {
                    dst[0] = sM[h];
                    dst[1] = sL[h];
                }
            }
        }
        if (!more_segs) break;
        first_seg = false;
        s = ns;   // its first chunks are already staged
    }
}

// Merge of the (sequence, kv head) segments that the pass left as partials: CTA = segment, warp h
// merges operand column h by log-sum-exp over the partials of the pass CTAs lo..hi that share the
// segment, then applies the inverse rotation.  Launched as a programmatic dependent of the pass:
// its CTAs are placed as the pass's CTAs exit and wait for the whole pass to complete.
template <int D>
__global__ void __launch_bounds__(256)
merge_kernel(const uint8_t *__restrict__ params, int batch, int q_len, int hq, int hkv, int G,
             const int64_t *__restrict__ cpre, int nctas, const float *__restrict__ part, float *__restrict__ out,
             float *__restrict__ lse) {
    constexpr int R = D / 32;
    constexpr int UN = 32 / R;
    constexpr float kLn2 = 0.6931471805599453f;
    pdl_wait();
    const int b = blockIdx.x / hkv, kh = blockIdx.x % hkv, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = warp;
    if (h >= G) return;
    const int64_t W = cpre[batch];
    const int P = (int)(W < (int64_t)nctas ? W : (int64_t)nctas);
    const int64_t ub = cpre[b];
    const int64_t nch = (cpre[b + 1] - ub) / hkv;
    if (nch == 0 || P == 0) return;
    const int64_t us = ub + kh * nch, ue = us + nch;
    const int lo = sk_cta_of(us, P, W), hi = sk_cta_of(ue - 1, P, W);
    if (lo == hi) return;   // finished by the pass
    // the CTA lo wrote this segment as its second partial slot when its range began earlier
    const int slot_lo = (sk_begin(lo, P, W) >= us) ? 0 : 1;
    const int np = hi - lo + 1;
    auto part_of = [&](int j) {
        const int c2 = lo + j, sl = (c2 == lo) ? slot_lo : 0;
        return part + (((size_t)c2 * 2 + sl) * G + h) * kPartStride(D);
    };
    // (m, l) of up to 32 partials per lane pass, one load each
    float M = -INFINITY, l = 0.f;
    for (int j0 = 0; j0 < np; j0 += 32) {
        const int j = j0 + lane;
        const float2 ml = j < np ? *reinterpret_cast<const float2 *>(part_of(j)) : make_float2(-INFINITY, 0.f);
        const float Mn = fmaxf(M, warp_max(ml.x));
        const float lc = (ml.x == -INFINITY) ? 0.f : ml.y * exp2f(ml.x - Mn);
        l = (M == -INFINITY ? 0.f : l * exp2f(M - Mn)) + warp_sum(lc);
        M = Mn;
    }
    float v[R];
#pragma unroll
    for (int r = 0; r < R; ++r) v[r] = 0.f;
#pragma unroll 1
    for (int j0 = 0; j0 < np; j0 += UN) {
        float vv[UN][R], ww[UN];
#pragma unroll
        for (int u = 0; u < UN; ++u) {
            ww[u] = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) vv[u][r] = 0.f;
            if (j0 + u < np) {
                const float *ps = part_of(j0 + u);
                const float m = ps[0];
#pragma unroll
                for (int r = 0; r < R; ++r) vv[u][r] = ps[4 + 32 * r + lane];
                ww[u] = (m == -INFINITY) ? 0.f : exp2f(m - M);
            }
        }
#pragma unroll
        for (int u = 0; u < UN; ++u)
#pragma unroll
            for (int r = 0; r < R; ++r) v[r] = fmaf(vv[u][r], ww[u], v[r]);
    }
    const int gq = G / q_len;
    const size_t orow = ((size_t)b * q_len + h / gq) * hq + (size_t)kh * gq + h % gq;
    finish_row<D>(v, l, params, out + orow * D, lane);
    if (lse && lane == 0) lse[orow] = l > 0.f ? M * kLn2 + logf(l) : -INFINITY;
}

template <int D, int G>
int warp_ctas_g() {
    int dev = 0, sms = 0, occ = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    constexpr size_t smem = warp_smem_bytes<D, G>();
    auto kern = decode_warp_kernel<D, G>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWWarps * 32, smem) != cudaSuccess) return 0;
    occ = occ < 1 ? 1 : (occ > kCtasPerSm ? kCtasPerSm : occ);
    sms = sms > kMaxSms ? kMaxSms : sms;
    return occ * sms;
}

template <int D, int G>
cudaError_t warp_launch_g(int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq, int hkv,
                          const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                          const int32_t *ctx, int ctx_add, int max_ctx, bool early, const WsLayout &w, float *out,
                          float *lse, int32_t *status) {
    constexpr size_t smem = warp_smem_bytes<D, G>();
    auto kern = decode_warp_kernel<D, G>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pass(kern, nctas, kWWarps * 32, smem, st, P, w.packs, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx,
                    ctx_add, max_ctx, early ? 1 : 0, w.cpre, w.part, out, lse, status);
    if (e != cudaSuccess) return e;
    return launch_pass(merge_kernel<D>, batch * hkv, 256, 0, st, P, batch, q_len, hq, hkv, G, (const int64_t *)w.cpre,
                       nctas, (const float *)w.part, out, lse);
}

template <int D>
int warp_ctas_d(int G) {
    switch (G) {
        case 1: return warp_ctas_g<D, 1>();
        case 2: return warp_ctas_g<D, 2>();
        case 3: return warp_ctas_g<D, 3>();
        case 4: return warp_ctas_g<D, 4>();
        case 5: return warp_ctas_g<D, 5>();
        case 6: return warp_ctas_g<D, 6>();
        case 7: return warp_ctas_g<D, 7>();
        default: return warp_ctas_g<D, 8>();
    }
}

template <int D>
cudaError_t warp_launch_d(int G, int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq, int hkv,
                          const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                          const int32_t *ctx, int ctx_add, int max_ctx, bool early, const WsLayout &w, float *out,
                          float *lse, int32_t *status) {
#define TQ_WPASS(GG) return warp_launch_g<D, GG>(nctas, st, P, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx, ctx_add, max_ctx, early, w, out, lse, status)
    switch (G) {
        case 1: TQ_WPASS(1);
        case 2: TQ_WPASS(2);
        case 3: TQ_WPASS(3);
        case 4: TQ_WPASS(4);
        case 5: TQ_WPASS(5);
        case 6: TQ_WPASS(6);
        case 7: TQ_WPASS(7);
        default: TQ_WPASS(8);
    }
#undef TQ_WPASS
}

}  // namespace

int warp_pass_ctas(int d, int G) { return d == 128 ? warp_ctas_d<128>(G) : warp_ctas_d<256>(G); }

cudaError_t warp_pass_launch(int d, int G, int nctas, cudaStream_t st, const uint8_t *P, int batch, int q_len, int hq,
                             int hkv, const uint8_t *kp, const uint8_t *vp, int64_t nb, const int32_t *bt, int mb,
                             const int32_t *ctx, int ctx_add, int max_ctx, bool early, const WsLayout &w, float *out,
                             float *lse, int32_t *status) {
    if (d == 128)
        return warp_launch_d<128>(G, nctas, st, P, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx, ctx_add, max_ctx,
                                  early, w, out, lse, status);
    return warp_launch_d<256>(G, nctas, st, P, batch, q_len, hq, hkv, kp, vp, nb, bt, mb, ctx, ctx_add, max_ctx, early,
                              w, out, lse, status);
}

}  // namespace tq
