// tq_prep.cuh -- the two small kernels that precede the decode pass, as device functions so
// that they can run in one launch: the paged append's encode (tiles of vectors) and the
// query prep (rotation, S projection, operand packs, work schedule).
#pragma once

#include "tq_internal.cuh"

namespace tq {

constexpr int kEncWarps = 4;               // warps per encode CTA

// Where vector v of a launch goes: slot (or -1 to skip) and its input row.
struct SlotMap {
    const int64_t *slots;                  // bulk: slots[token]
    const int32_t *block_table;            // append: slot from the block table and length
    const int32_t *ctx_lens;
    int max_blocks;
    int64_t num_blocks;
    int n_heads;
    int q_len = 1;                         // append: tokens per sequence (token t is number t % q_len of sequence t / q_len)
    __device__ int64_t slot(int64_t token, int32_t *status, bool report) const {
        if (!slots) {
            const int L0 = len_of(token);
            return slot_of_block(token, L0, block_at(token, L0), status, report);
        }
        return slot_check(slots[token], status, report);
    }
    // The slot-mapping lookup in two steps, so that the load is issued long before its value is
    // needed (a branch on it would wait for it): slot_raw reads slots[token], slot_check turns the
    // value into a slot or -1 (skipped; flagged when outside the pool).
    __device__ int64_t slot_raw(int64_t token) const { return slots[token]; }
    __device__ int64_t slot_check(int64_t s, int32_t *status, bool report) const {
        if (s < 0) return -1;
        if (s / kBlock >= num_blocks) {
            if (report) flag_status(status, TQ_STATUS_BAD_SLOT);
            return -1;
        }
        return s;
    }
    // The block-table lookup in steps, so that each load is issued long before its value is
    // used: len_of reads the sequence's length, block_at the block table entry of the token's
    // position (-1 when there is none), slot_of_block checks the entry and forms the slot.
    __device__ int len_of(int64_t token) const { return ctx_lens[token / q_len]; }
    __device__ int64_t block_at(int64_t token, int L0) const {
        const int64_t seq = token / q_len;
        const int lb = (L0 + (int)(token - seq * q_len)) / kBlock;
        return (L0 >= 0 && lb < max_blocks) ? (int64_t)block_table[(size_t)seq * max_blocks + lb] : -1;
    }
    __device__ int64_t slot_of_block(int64_t token, int L0, int64_t blk, int32_t *status, bool report) const {
        if (L0 < 0) return -1;
        if (blk < 0 || blk >= num_blocks) {   // no block for this position, or one outside the pool
            if (report) flag_status(status, TQ_STATUS_BAD_SLOT);
            return -1;
        }
        return blk * kBlock + (L0 + (int)(token % q_len)) % kBlock;
    }
};

// TILE vectors per CTA: 16 for bulk encodes (each S^T read serves 16
// vectors), 4 for the one-token append (more CTAs, shorter latency chains).
template <int D, int TILE>
struct EncSmem {
    static constexpr bool kResident = (D == 128);
    static constexpr size_t kST = kResident ? (size_t)D * D * 4 : (size_t)2 * kProjRows * D * 4;
    static constexpr size_t kRho = (size_t)TILE * D * 4;
    static constexpr size_t kSgn = (size_t)TILE * D;
    static constexpr size_t kCode = (size_t)TILE * D;
    static constexpr size_t kBytes = kST + kRho + kSgn + kCode;
};


// Encode tiles blk, blk + nblk, ... of TILE vectors (K if is_k, else V) with one CTA of
// 4 warps; `smem` holds EncSmem<D, TILE>::kBytes.  A bad slot is reported by the K tiles
// (or, without K tiles, by the V tiles) when report_bad is set.
template <int D, int TILE, typename T>
__device__ __forceinline__ void encode_tiles(const uint8_t *__restrict__ params, const T *__restrict__ x,
                                             int64_t n_vec, const SlotMap &map, uint8_t *__restrict__ pool, bool is_k,
                                             bool report_bad, int blk, int nblk, uint8_t *smem, int32_t *status) {
    constexpr int R = D / 32;
    constexpr int kTile = TILE, kPerWarp = (TILE + kEncWarps - 1) / kEncWarps;   // tiles below 4 leave warps idle in 1 and 3
    using SM = EncSmem<D, TILE>;
    float *sST = reinterpret_cast<float *>(smem);
    float (*s_rho)[D] = reinterpret_cast<float (*)[D]>(smem + SM::kST);
    uint8_t (*s_sgn)[D] = reinterpret_cast<uint8_t (*)[D]>(smem + SM::kST + SM::kRho);
    uint8_t (*s_code)[D] = reinterpret_cast<uint8_t (*)[D]>(smem + SM::kST + SM::kRho + SM::kSgn);
    __shared__ float s_cent[8], s_thr[8];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    const float *gST = reinterpret_cast<const float *>(params + params_off_ST(D));
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blk == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    if (threadIdx.x < 8) {
        s_cent[threadIdx.x] = ph->centroid[threadIdx.x];
        s_thr[threadIdx.x] = ph->threshold[threadIdx.x];
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const int64_t ntiles = (n_vec + kTile - 1) / kTile;

#pragma unroll 1
    for (int64_t tile = blk; tile < ntiles; tile += nblk) {
        const int64_t v0 = tile * kTile;
        float nrm[kPerWarp], gam[kPerWarp];
        int64_t slot[kPerWarp];
        // ---- 1. norm, rotation, cells, residual
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            const int tv = warp + kEncWarps * j;              // vector within the tile
            const bool mine = tv < kTile;                     // warp-uniform
            const int64_t v = v0 + tv;
            float val[R];
            int dims[R];
#pragma unroll
            for (int r = 0; r < R; ++r) {   // the input row does not depend on the slot: load it first
                dims[r] = is_k ? kdim<D>(lane, r) : vdim<D>(lane, r);
                val[r] = (mine && v < n_vec) ? to_f32<T>(x[v * D + dims[r]]) : 0.f;
            }
            // the slot (block-table lookups) is needed only by the stores: a vector without one is
            // encoded from whatever it holds and not stored, so nothing here waits for the lookup
            slot[j] = -1;
            if (mine && v < n_vec)   // a bad slot is reported once per token
                slot[j] = map.slot(v / map.n_heads, status, report_bad && lane == 0 && (v % map.n_heads) == 0);
            // S^T (64 KB at d = 128) is copied once, after the first rows are requested, so that
            // those small loads are not queued behind it; it is waited for before the projection
            if (is_k && SM::kResident && j == 0 && tile == blk) stage_st_rows<D, kEncWarps * 32>(sST, gST, 0, D);
            nrm[j] = 0.f;
            gam[j] = 0.f;
            if (!mine) continue;
            float ss = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) ss = fmaf(val[r], val[r], ss);
            const float n = sqrtf(warp_sum(ss));
#pragma unroll
            for (int r = 0; r < R; ++r) val[r] *= __ldg(Dsign + dims[r]);
            fwht_warp<R>(val, lane);                       // z = H(D x) / n = sqrt(d) Pi (x/n)
            float g2 = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float z = (n > 0.f) ? val[r] / n : 0.f;
                int k = 0;
#pragma unroll
                for (int t = 0; t < 7; ++t) k += (z >= s_thr[t]) ? 1 : 0;
                s_code[tv][dims[r]] = (uint8_t)k;
                if (is_k) {
                    const float rho = z - s_cent[k];     // residual, rotated unit-variance domain
                    g2 = fmaf(rho, rho, g2);
                    s_rho[tv][dims[r]] = rho;
                }
            }
            nrm[j] = n;
            gam[j] = is_k ? sqrtf(warp_sum(g2)) / sqrtf((float)D) : 0.f;   // ||y - c/sqrt d|| = ||rho|| / sqrt d
        }
        // ---- 2. QJL projections of the tile (K only): bit k = [(S rho)_k >= 0]
        if (is_k) {
            constexpr int KPT = D / (kEncWarps * 32);
            float acc[KPT][kTile];
#pragma unroll
            for (int u = 0; u < KPT; ++u)
#pragma unroll
                for (int t = 0; t < kTile; ++t) acc[u][t] = 0.f;
            if (SM::kResident) {
                cp_async_wait_all();
                __syncthreads();
                project_rows<D, kTile, kEncWarps * 32>(sST, 0, D, s_rho, acc);
            } else {
                __syncthreads();
                project_streamed<D, kTile, kEncWarps * 32>(gST, sST, s_rho, acc);
            }
#pragma unroll
            for (int u = 0; u < KPT; ++u)
#pragma unroll
                for (int t = 0; t < kTile; ++t) s_sgn[t][threadIdx.x + 128 * u] = acc[u][t] >= 0.f ? 1 : 0;
            __syncthreads();
        }
        // ---- 3. pack and store (the layout of tq_internal.cuh); a warp packs the vectors it encoded
        __syncwarp();
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            if (slot[j] < 0) continue;                     // warp-uniform (also for a warp without a vector)
            const int tv = warp + kEncWarps * j;
            const int head = (int)((v0 + tv) % map.n_heads);
            const int64_t blk = slot[j] / kBlock;
            const int off = (int)(slot[j] % kBlock);
            const uint8_t *cd = s_code[tv];
            if (is_k) {
                // 4 D/32 words of 8 fields: word (tig, w) holds columns 2tig, 2tig+1, 2tig+8, 2tig+9 of
                // k-steps 2w (fields 0..3) and 2w+1 (fields 4..7)
                constexpr int NW = D / 32;
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * k_record(D);
                const uint8_t *sg = s_sgn[tv];
                const int gid = off & 7, rr = off >> 3;
                for (int wi = lane; wi < 4 * NW; wi += 32) {
                    const int tg = wi / NW, w = wi % NW;
                    uint32_t word = 0;
#pragma unroll
                    for (int f = 0; f < 8; ++f) {
                        const int cs = f & 3, x = 16 * (2 * w + (f >> 2)) + 2 * tg + (cs & 1) + 8 * (cs >> 1);
                        word |= (uint32_t)(cd[x] | (sg[x] << 3)) << (4 * f);
                    }
                    reinterpret_cast<uint32_t *>(rec)[((4 * gid + tg) * 2 + rr) * NW + w] = word;
                }
                if (lane == 0)
                    *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * off) =
                        __halves2half2(__float2half_rn(nrm[j]), __float2half_rn(gam[j]));
            } else {
                // the slot's bytes: per lane gid, group g, word k and half hf, the cells of lane slots
                // 16g + 4k + 2hf + ab (ab = 0, 1: the byte's two fields) with bit k of the cells of lane
                // slots 16g + 12 + 2hf + ab in bit 3 of the fields
                constexpr int NG = D / 128;
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * v_record(D);
                const int tg = (off & 7) >> 1, pr = off >> 3, e = off & 1;
                for (int bi = lane; bi < 48 * NG; bi += 32) {
                    const int hf = bi & 1, k = (bi >> 1) % 3, g = ((bi >> 1) / 3) % NG, gid = (bi >> 1) / (3 * NG);
                    uint32_t byte = 0;
#pragma unroll
                    for (int ab = 0; ab < 2; ++ab) {
                        const int sd = 16 * g + 4 * k + 2 * hf + ab, ss = 16 * g + 12 + 2 * hf + ab;
                        const int xd = 16 * (sd >> 1) + gid + 8 * (sd & 1), xs = 16 * (ss >> 1) + gid + 8 * (ss & 1);
                        byte |= (uint32_t)(cd[xd] | (((cd[xs] >> k) & 1) << 3)) << (4 * ab);
                    }
                    rec[((size_t)((4 * gid + tg) * 2 + pr) * 3 * NG + 3 * g + k) * 4 + 2 * hf + e] = (uint8_t)byte;
                }
                if (lane == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * off) = __float2half_rn(nrm[j]);
            }
        }
        __syncthreads();   // s_rho / s_sgn are rewritten by the next tile
    }
}


// ---------------------------------------------------------------- f16 operand helpers

// QJL operand of field position i (0..3) of a K record word: bit 4i+3 of each f16 half.
// Positions 3, 7, 11 give 0 or delta_i (2^-21, 2^-17, 2^-13; the first two subnormal, which
// the tensor core keeps); position 15 is the sign bit of 2^-14 (base 0x0400), so that operand
// is -2^-14 sigma.  The B operand is u * qjl_bscale(i), so that every product is
// 2^-16 (u sigma + u) for i < 3 and 2^-16 u sigma for i = 3; the 2^-16 sum of u over the i < 3
// coordinates, 2^-16 <w, qbar> with the params' offset weights w, is removed afterwards.
__host__ __device__ constexpr uint32_t qjl_base(int i) { return i == 3 ? 0x04000400u : 0u; }
__host__ __device__ constexpr float qjl_bscale(int i) { return i == 0 ? 64.f : i == 1 ? 4.f : i == 2 ? 0.25f : -0.25f; }

__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// d = a b with a zero accumulator.  Long chains of mma.sync accumulation lose precision (the
// tensor core's fp32 accumulation is not rounded to nearest: measured on GB300, 235 ulp of the
// sum after 1024 chained m16n8k16 and 1439 after 4096), so sums over many tokens start each
// block from zero and are added up with FADD.
__device__ __forceinline__ void mma_f16_z(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Per (sequence, kv head) query pack: f16x2 B-operand fragments
// [2 (qbar / alpha, QJL-scaled u)][d/16 k-steps][n-tiles][32 lanes][2 words], then floats:
// [8] unused, [8 heads] the QJL offset constant.
__host__ __device__ constexpr size_t kPackBytes(int d) { return 64 * (size_t)d + 256; }
__host__ __device__ constexpr int kPackFloatOff(int d) { return 16 * d; }   // in floats

// ---------------------------------------------------------------- (1) query prep
// A CTA of 128 threads prepares one 32-coordinate slice sl (k-steps 2 sl and 2 sl + 1) of kQRows
// (sequence, query head) rows, kQRpw rows per warp.  Every load is issued first: the rows, the
// signs D, the offset weights and the slice's columns of S^T (d rows of 128 bytes, copied to
// shared memory).  A warp rotates its rows (qbar = H D q / sqrt d, all d coordinates, in
// registers and shuffles) and leaves them in shared memory; thread (warp, lane) then computes
// u_k = (S qbar)_k, k = 32 sl + lane, for each of its warp's rows and writes the f16 hi and lo
// parts of its coordinate in both planes of the K-side B operand (qbar / alpha in natural order;
// u scaled for the coordinate's QJL field position) into the pack of the row's (sequence, kv
// head).  Slice 0 also writes the row's QJL offset constant 2^-16 <w, qbar>.
constexpr int kQRpw = 2, kQRows = 4 * kQRpw, kQSlice = 32;
template <int D> __host__ __device__ constexpr size_t qprep_smem() {
    return (size_t)kQRows * D * 4 + (size_t)D * kQSlice * 4;
}
__host__ __device__ inline int qprep_ctas(int d, int nrows) { return (nrows + kQRows - 1) / kQRows * (d / kQSlice); }

// The f16 hi and lo parts of B value beta at operand row kr of k-step s of plane qu: operand
// columns 2 hg (hi) and 2 hg + 1 (lo).
template <int NKS, int NTK>
__device__ __forceinline__ void put_bpair(uint16_t *ph, int qu, int s, int kr, int hg, float beta) {
    const __half hi = __float2half_rn(beta);
    const __half lo = __float2half_rn(beta - __half2float(hi));
    const int reg = kr >> 3, tig = (kr & 7) >> 1, e = kr & 1;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int col = 2 * hg + x, nt = col >> 3, gid = col & 7;
        const size_t word = ((size_t)(qu * NKS + s) * NTK + nt) * 64 + (4 * gid + tig) * 2 + reg;
        ph[word * 2 + e] = __half_as_ushort(x == 0 ? hi : lo);
    }
}

// CTA blk of the query prep (qprep_ctas of them); `qsm` holds qprep_smem<D>() bytes.  With
// q_len > 1 queries per sequence (q[b][i][h]), query i of head hg of a kv head is operand
// column i * G + hg of the kv head's pack.
template <int D, int NTK, typename T>
__device__ __forceinline__ void qprep_slice(const uint8_t *__restrict__ params, const T *__restrict__ q, int batch,
                                            int q_len, int hq, int hkv, uint8_t *__restrict__ packs, int blk,
                                            uint8_t *qsm) {
    constexpr int R = D / 32, NKS = D / 16, NSL = D / kQSlice, CPR = kQSlice / 4;   // CPR: 16-byte pieces per S^T row
    float (*qs)[D] = reinterpret_cast<float (*)[D]>(qsm);                    // [kQRows][D] qbar
    float *sST = reinterpret_cast<float *>(qsm + (size_t)kQRows * D * 4);   // [D][32]: S^T[j][32 sl + c]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sl = blk % NSL, row0 = (blk / NSL) * kQRows + kQRpw * warp;
    const int nrows = batch * q_len * hq;
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const float *ST = reinterpret_cast<const float *>(params + params_off_ST(D));
    const float *Wq = reinterpret_cast<const float *>(params + params_off_W(D));
    float v[kQRpw][R];
#pragma unroll
    for (int i = 0; i < kQRpw; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r)
            v[i][r] = (row0 + i < nrows) ? to_f32<T>(q[(size_t)(row0 + i) * D + 32 * r + lane]) : 0.f;
    for (int c = threadIdx.x; c < D * CPR; c += 128)
        cp_async16(sST + 4 * c, ST + (size_t)(c / CPR) * D + kQSlice * sl + 4 * (c % CPR));
    cp_async_commit();
    float dsg[R], wq[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        dsg[r] = __ldg(Dsign + 32 * r + lane);
        wq[r] = (sl == 0) ? __ldg(Wq + 32 * r + lane) : 0.f;
    }
    const float inv_alpha = __ldg(&reinterpret_cast<const ParamsHeader *>(params)->inv_alpha);
    const float inv_sd = rsqrtf((float)D);
    float vk[kQRpw];   // coordinate 32 sl + lane of each row
#pragma unroll
    for (int i = 0; i < kQRpw; ++i) {
#pragma unroll
        for (int r = 0; r < R; ++r) v[i][r] *= dsg[r];
        fwht_warp<R>(v[i], lane);
        vk[i] = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            v[i][r] *= inv_sd;   // qbar = H D q / sqrt d
            qs[kQRpw * warp + i][32 * r + lane] = v[i][r];
            if (r == sl) vk[i] = v[i][r];
        }
    }
    cp_async_wait_all();
    __syncthreads();
    // u_k of the warp's rows, four partial sums each
    float acc[kQRpw][4];
#pragma unroll
    for (int i = 0; i < kQRpw; ++i)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
#pragma unroll 4
    for (int j = 0; j < D; j += 4) {
        float sv[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) sv[c] = sST[(j + c) * kQSlice + lane];
#pragma unroll
        for (int i = 0; i < kQRpw; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(&qs[kQRpw * warp + i][j]);
            acc[i][0] = fmaf(sv[0], x.x, acc[i][0]);
            acc[i][1] = fmaf(sv[1], x.y, acc[i][1]);
            acc[i][2] = fmaf(sv[2], x.z, acc[i][2]);
            acc[i][3] = fmaf(sv[3], x.w, acc[i][3]);
        }
    }
    // operand rows of coordinate k: plane 0 row k & 15 of k-step k >> 4; plane 1 (the K record's
    // field f = 4 (s & 1) + pos) row 2 tg + 8 (pos & 1) + (f >> 2) of k-step 2 (s >> 1) + (pos >> 1)
    const int k = kQSlice * sl + lane, pos = qjl_pos(k);
    const int s = k >> 4, c = k & 15, tg = (c & 7) >> 1, f = 4 * (s & 1) + pos;
    const int kr1 = 2 * tg + 8 * (pos & 1) + (f >> 2), s1 = 2 * (s >> 1) + (pos >> 1);
#pragma unroll
    for (int i = 0; i < kQRpw; ++i) {
        const int row = row0 + i;
        if (row >= nrows) break;   // warp-uniform
        const int b = row / (hq * q_len), qi = (row / hq) % q_len, h = row % hq, G = hq / hkv, kvh = h / G;
        const int hg = qi * G + h % G;   // operand column pair of this query row
        uint8_t *pack = packs + ((size_t)b * hkv + kvh) * kPackBytes(D);
        uint16_t *ph = reinterpret_cast<uint16_t *>(pack);
        put_bpair<NKS, NTK>(ph, 0, s, c, hg, vk[i] * inv_alpha);
        const float u = (acc[i][0] + acc[i][1]) + (acc[i][2] + acc[i][3]);
        put_bpair<NKS, NTK>(ph, 1, s1, kr1, hg, u * qjl_bscale(pos));
        if (sl == 0) {
            float cs = 0.f;
#pragma unroll
            for (int r = 0; r < R; ++r) cs = fmaf(wq[r], v[i][r], cs);
            cs = warp_sum(cs);
            if (lane == 0) reinterpret_cast<float *>(pack)[kPackFloatOff(D) + 8 + hg] = cs * (1.f / 65536.f);
            // columns beyond the group's 2 * G * q_len are zero (written by the group's first row)
            if (hg == 0) {
                uint32_t *pw = reinterpret_cast<uint32_t *>(pack);
                for (int col = 2 * G * q_len; col < 8 * NTK; ++col) {
                    const int nt = col >> 3, gid = col & 7;
                    for (int e = lane; e < 2 * NKS * 8; e += 32) {
                        const int qu = e / (NKS * 8), ks = (e / 8) % NKS, kk = e % 8;
                        pw[((size_t)(qu * NKS + ks) * NTK + nt) * 64 + (4 * gid + (kk >> 1)) * 2 + (kk & 1)] = 0u;
                    }
                }
            }
        }
    }
}

// ---------------------------------------------------------------- paged append of single tokens
// K: a CTA of 128 threads encodes one 32-coordinate slice sl (record word column sl) of one
// vector.  Every load is issued first: the row, the signs, the codebook, the slot (length, then
// block table) and the slice's columns of S^T (to shared memory).  Warp 0 computes the norm, the
// rotation, the cells and the residual rho of the whole vector (cells and rho to shared memory);
// thread (warp w, lane) then sums S^T[j][32 sl + lane] rho_j over the w-th quarter of j, the
// quarters are added in shared memory, and lanes 0..3 of warp 0 assemble and store the slice's
// four record words (one per tig).  Slice 0 also stores fp16(n) and fp16(gamma).
template <int D> __host__ __device__ constexpr size_t append_k_smem() {
    return (size_t)D * 32 * 4 + (size_t)D * 4 + 4 * 32 * 4 + D;
}
// V: a CTA of 4 warps encodes 4 vectors, one per warp (no projection).
template <int D> __host__ __device__ constexpr size_t append_v_smem() { return (size_t)4 * D; }
constexpr int kAppendVPerCta = 4;
__host__ __device__ inline int append_k_ctas(int d, int64_t n_vec) { return (int)(n_vec * (d / 32)); }
__host__ __device__ inline int append_v_ctas(int64_t n_vec) { return (int)((n_vec + kAppendVPerCta - 1) / kAppendVPerCta); }

// Norm, rotation and cells of vector x (one warp, lane map dims): val becomes z = sqrt(d) Pi x / n.
template <int R>
__device__ __forceinline__ float rotate_warp(float (&val)[R], const float (&dsg)[R], int lane) {
    float ss = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) ss = fmaf(val[r], val[r], ss);
    const float n = sqrtf(warp_sum(ss));
#pragma unroll
    for (int r = 0; r < R; ++r) val[r] *= dsg[r];
    fwht_warp<R>(val, lane);   // H (D x): sqrt(d) Pi x
#pragma unroll
    for (int r = 0; r < R; ++r) val[r] = (n > 0.f) ? val[r] / n : 0.f;
    return n;
}

template <int D, typename T>
__device__ __forceinline__ void append_k_slice(const uint8_t *__restrict__ params, const T *__restrict__ x,
                                               int64_t n_vec, const SlotMap &map, uint8_t *__restrict__ pool,
                                               int blk, uint8_t *smem, int32_t *status) {
    constexpr int R = D / 32, NSL = D / 32, NW = D / 32;
    float *sST = reinterpret_cast<float *>(smem);   // [D][32]
    float *s_rho = sST + D * 32;                     // [D]
    float *s_part = s_rho + D;                       // [4][32]
    uint8_t *s_code = reinterpret_cast<uint8_t *>(s_part + 128);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t v = blk / NSL;
    const int sl = blk % NSL;
    if (v >= n_vec) return;   // CTA-uniform
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    const float *ST = reinterpret_cast<const float *>(params + params_off_ST(D));
    float n = 0.f, gam = 0.f;
    int64_t slot = -1;
    bool ok = false;
    const int64_t tok = v / map.n_heads;
    int L0 = 0;
    float val[R], dsg[R];
    int dims[R];
    if (warp == 0) {
        L0 = map.len_of(tok);
        const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
#pragma unroll
        for (int r = 0; r < R; ++r) {
            dims[r] = kdim<D>(lane, r);
            val[r] = to_f32<T>(x[v * D + dims[r]]);
            dsg[r] = __ldg(Dsign + dims[r]);
        }
    }
    for (int c = threadIdx.x; c < D * 8; c += 128)   // the slice of S^T: D rows of 128 bytes
        cp_async16(sST + 4 * c, ST + (size_t)(c >> 3) * D + 32 * sl + 4 * (c & 7));
    cp_async_commit();
    if (warp == 0) {
        float thr[7], cen[8];
#pragma unroll
        for (int t = 0; t < 7; ++t) thr[t] = __ldg(&ph->threshold[t]);
#pragma unroll
        for (int t = 0; t < 8; ++t) cen[t] = __ldg(&ph->centroid[t]);
        ok = __ldg(&ph->magic) == kParamsMagic && __ldg(&ph->d) == D;
        const int64_t bid = map.block_at(tok, L0);   // its load overlaps the rest
        n = rotate_warp<R>(val, dsg, lane);
        float g2 = 0.f;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            int k = 0;
#pragma unroll
            for (int t = 0; t < 7; ++t) k += (val[r] >= thr[t]) ? 1 : 0;
            float ck = cen[0];
#pragma unroll
            for (int t = 1; t < 8; ++t) ck = (k == t) ? cen[t] : ck;
            const float rho = val[r] - ck;   // residual, rotated unit-variance domain
            g2 = fmaf(rho, rho, g2);
            s_code[dims[r]] = (uint8_t)k;
            s_rho[dims[r]] = rho;
        }
        gam = sqrtf(warp_sum(g2)) / sqrtf((float)D);   // ||y - c/sqrt d|| = ||rho|| / sqrt d
        if (!ok && lane == 0 && sl == 0 && v == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        slot = map.slot_of_block(tok, L0, bid, status, ok && lane == 0 && sl == 0 && (v % map.n_heads) == 0);
    }
    cp_async_wait_all();
    __syncthreads();
    {
        float a0 = 0.f, a1 = 0.f;
        const int j0 = warp * (D / 4);
#pragma unroll 8
        for (int j = j0; j < j0 + D / 4; j += 2) {
            a0 = fmaf(sST[j * 32 + lane], s_rho[j], a0);
            a1 = fmaf(sST[(j + 1) * 32 + lane], s_rho[j + 1], a1);
        }
        s_part[warp * 32 + lane] = a0 + a1;
    }
    __syncthreads();
    if (warp != 0 || !ok || slot < 0) return;
    const float p = (s_part[lane] + s_part[32 + lane]) + (s_part[64 + lane] + s_part[96 + lane]);
    const uint32_t bits = __ballot_sync(0xffffffffu, p >= 0.f);   // bit c: sign of coordinate 32 sl + c
    const int64_t blk_id = slot / kBlock;
    const int off = (int)(slot % kBlock), head = (int)(v % map.n_heads);
    uint8_t *rec = pool + ((size_t)blk_id * map.n_heads + head) * k_record(D);
    if (lane < 4) {
        // word (tig, sl) holds columns 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 of k-steps 2 sl
        // (fields 0..3) and 2 sl + 1 (fields 4..7)
        const int tg = lane;
        uint32_t word = 0;
#pragma unroll
        for (int f = 0; f < 8; ++f) {
            const int cs = f & 3, xl = 16 * (f >> 2) + 2 * tg + (cs & 1) + 8 * (cs >> 1);
            word |= (uint32_t)(s_code[32 * sl + xl] | (((bits >> xl) & 1u) << 3)) << (4 * f);
        }
        reinterpret_cast<uint32_t *>(rec)[((4 * (off & 7) + tg) * 2 + (off >> 3)) * NW + sl] = word;
    }
    if (sl == 0 && lane == 0)
        *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * off) = __halves2half2(__float2half_rn(n), __float2half_rn(gam));
}

template <int D, typename T>
__device__ __forceinline__ void append_v_rows(const uint8_t *__restrict__ params, const T *__restrict__ x,
                                              int64_t n_vec, const SlotMap &map, uint8_t *__restrict__ pool,
                                              bool report_bad, int blk, uint8_t *smem, int32_t *status) {
    constexpr int R = D / 32, NG = D / 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t v = (int64_t)blk * kAppendVPerCta + warp;
    if (v >= n_vec) return;   // warp-uniform; no CTA-wide synchronisation follows
    uint8_t *cd = smem + (size_t)warp * D;
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    const float *Dsign = reinterpret_cast<const float *>(params + params_off_D(D));
    const int64_t tok = v / map.n_heads;
    const int L0 = map.len_of(tok);
    float val[R], dsg[R];
    int dims[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        dims[r] = vdim<D>(lane, r);
        val[r] = to_f32<T>(x[v * D + dims[r]]);
        dsg[r] = __ldg(Dsign + dims[r]);
    }
    float thr[7];
#pragma unroll
    for (int t = 0; t < 7; ++t) thr[t] = __ldg(&ph->threshold[t]);
    const bool ok = __ldg(&ph->magic) == kParamsMagic && __ldg(&ph->d) == D;
    const int64_t bid = map.block_at(tok, L0);   // its load overlaps the encode
    const float n = rotate_warp<R>(val, dsg, lane);
#pragma unroll
    for (int r = 0; r < R; ++r) {
        int k = 0;
#pragma unroll
        for (int t = 0; t < 7; ++t) k += (val[r] >= thr[t]) ? 1 : 0;
        cd[dims[r]] = (uint8_t)k;
    }
    if (!ok) {
        if (lane == 0 && v == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int64_t slot = map.slot_of_block(tok, L0, bid, status, report_bad && lane == 0 && (v % map.n_heads) == 0);
    __syncwarp();
    if (slot < 0) return;
    // the slot's bytes: per lane gid, group g, word k and half hf, the cells of lane slots
    // 16g + 4k + 2hf + ab (ab = 0, 1: the byte's two fields) with bit k of the cells of lane
    // slots 16g + 12 + 2hf + ab in bit 3 of the fields
    const int64_t blk_id = slot / kBlock;
    const int off = (int)(slot % kBlock), head = (int)(v % map.n_heads);
    uint8_t *rec = pool + ((size_t)blk_id * map.n_heads + head) * v_record(D);
    const int tg = (off & 7) >> 1, pr = off >> 3, e = off & 1;
    for (int bi = lane; bi < 48 * NG; bi += 32) {
        const int hf = bi & 1, k = (bi >> 1) % 3, g = ((bi >> 1) / 3) % NG, gid = (bi >> 1) / (3 * NG);
        uint32_t byte = 0;
#pragma unroll
        for (int ab = 0; ab < 2; ++ab) {
            const int sd = 16 * g + 4 * k + 2 * hf + ab, ss = 16 * g + 12 + 2 * hf + ab;
            const int xd = 16 * (sd >> 1) + gid + 8 * (sd & 1), xs = 16 * (ss >> 1) + gid + 8 * (ss & 1);
            byte |= (uint32_t)(cd[xd] | (((cd[xs] >> k) & 1) << 3)) << (4 * ab);
        }
        rec[((size_t)((4 * gid + tg) * 2 + pr) * 3 * NG + 3 * g + k) * 4 + 2 * hf + e] = (uint8_t)byte;
    }
    if (lane == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * off) = __float2half_rn(n);
}


}  // namespace tq
