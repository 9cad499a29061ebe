// tq_encode.cu -- TurboQuant K/V encode kernels (bulk prefill and paged append).
//
// Method: "SwiftLM" README, "TurboQuantization: KV Cache Compression" ->
// "The Algorithm", K-Cache steps 1-5 (norm, WHT rotation, 3-bit Lloyd-Max
// cells, residual, QJL sign bits) and the V-Cache paragraph (steps 1-3, no
// QJL); the lilting.ch SwiftLM article, "KVキャッシュ圧縮の内訳", lists the
// same steps.  Slots follow the paged layout of the vLLM-MLX explainer,
// "Paged KVキャッシュ".
//
// A CTA of 4 warps encodes tiles of 16 (bulk) or 4 (append) vectors,
// persistent over tiles:
//  1. one warp per vector: norm, rotation (in registers and shuffles), cells,
//     residual (K) written to shared memory;
//  2. K only, all threads: the 16 QJL projections S rho, thread k computing
//     row k for every vector of the tile from S^T in shared memory (resident
//     for d=128, streamed in chunks for d=256); sign bits to shared memory;
//  3. one warp per vector: ballot-pack cells and signs, byte/word stores.
// One launch may carry K (blockIdx.y == 0) and V (blockIdx.y == 1) tiles.  Bulk encodes at
// d = 128 with 16-byte aligned input take the thread-per-row kernel below instead.
#include <string.h>

#include "tq_internal.cuh"
#include "tq_tc.cuh"
#include "tq_prep.cuh"
#include "tq_tmap.h"

#ifndef TQ_ENC_V_TMA
#define TQ_ENC_V_TMA 1           // bulk bf16 V at d = 128: TMA tiles, packed transform, whole records (encode128v_tma_kernel)
#endif
#ifndef TQ_ENC_SPLIT
#define TQ_ENC_SPLIT 1           // bulk K at d = 128: two threads per row (encode128k_split_kernel)
#endif

namespace tq {
namespace {

// a * b, rounded to nearest (the same as the C++ product), in a form the compiler keeps as one
// value: a threshold times the norm then stays in a register, where the compiler would otherwise
// select among the unscaled thresholds and multiply again at every comparison
__device__ __forceinline__ float held_mul(float a, float b) {
    float y;
    asm("mul.rn.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

// kinds: 1 = K only, 2 = V only, 3 = K (blockIdx.y 0) and V (blockIdx.y 1).
template <int D, int TILE, typename T>
__global__ void __launch_bounds__(kEncWarps * 32)
encode_kernel(const uint8_t *__restrict__ params, const T *__restrict__ xk, const T *__restrict__ xv, int64_t n_vec,
              SlotMap map, uint8_t *__restrict__ k_pool, uint8_t *__restrict__ v_pool, int kinds, int32_t *status) {
    extern __shared__ __align__(16) uint8_t smem[];
    const bool is_k = (kinds == 3) ? (blockIdx.y == 0) : (kinds == 1);
    encode_tiles<D, TILE, T>(params, is_k ? xk : xv, n_vec, map, is_k ? k_pool : v_pool, is_k, kinds != 3 || is_k,
                             blockIdx.x, gridDim.x, smem, status);
}

// ---------------------------------------------------------------- bulk encode at d = 128, thread per row
// Two warpgroups take alternate tiles of 128 vectors; thread r of a warpgroup owns vector r of
// the tile from input to record:
//  1. the tile's rows arrive by one bulk copy per row into a padded row stride (16-byte chunks of
//     the 32 rows a warp reads then fall in distinct bank groups), NX tiles in flight;
//  2. norm, signs D, the 128-point transform in registers (no shuffles), z = H D x / n;
//  3. the cell by a three-level binary search over the thresholds, whose outcomes are the cell's
//     bits b2, b1, b0 (cell >= k iff z >= t_{k-1}; ties go up), packed into the plane words;
//  4. K: the residual rho = z - c[cell] (x 256) as f16 hi and lo goes straight from registers into
//     tensor memory (this row's lane); one thread issues S rho = S rho_hi + S rho_lo (S is held at
//     binary16 precision; 16 f16 MMAs, A in tensor memory, B = S rows reordered so that accumulator
//     column 32 tig + b is sign bit b of sign word tig); the thread reads its row back and packs
//     the signs;
//  5. the record words of the row's slot are stored.
// QJL accumulator column n of the d = 128 tcgen05 encoders -> the coordinate whose sign it is.
// Columns 64 h + 16 tig + 8 wl + f are field f of K word (tig, 2 h + wl) of a slot (the record
// layout of tq_internal.cuh), so a thread's 16-column read back covers two of its words.
__host__ __device__ constexpr int k_col_coord(int n) {
    return 16 * (2 * (2 * (n >> 6) + ((n >> 3) & 1)) + ((n & 7) >> 2)) + 2 * ((n >> 4) & 3) + (n & 1) + 8 * ((n >> 1) & 1);
}
// field position of coordinate n (0..127) of a K record word: (tig, word, field)
__host__ __device__ constexpr int k_tig(int n) { return ((n & 15) & 7) >> 1; }
__host__ __device__ constexpr int k_word(int n) { return n >> 5; }
__host__ __device__ constexpr int k_field(int n) { return 4 * ((n >> 4) & 1) + (n & 1) + 2 * ((n & 15) >> 3); }

namespace encr {
constexpr int D = 128, kRows = 128, kThreads = 256;
template <typename T> __host__ __device__ constexpr int nx() { return sizeof(T) == 2 ? 2 : 1; }   // tiles in flight per warpgroup
template <typename T> __host__ __device__ constexpr int row_bytes() { return D * (int)sizeof(T); }
template <typename T> __host__ __device__ constexpr int row_stride() { return row_bytes<T>() + 16; }
template <typename T> __host__ __device__ constexpr int xbuf_bytes() { return kRows * row_stride<T>(); }
template <bool K> __host__ __device__ constexpr int oX() { return K ? 32768 : 0; }          // after S (f16)
// K: one CTA of 2 warpgroups per SM (tensor memory, S in shared memory); V: CTAs of one warpgroup,
// 3 per SM (no tensor memory: fewer registers and more warps per SM)
template <bool K> __host__ __device__ constexpr int n_wg() { return K ? 2 : 1; }
template <bool K> __host__ __device__ constexpr int n_threads() { return 128 * n_wg<K>(); }
template <bool K> __host__ __device__ constexpr int ctas_per_sm() { return K ? 1 : 3; }
template <typename T, bool K> __host__ __device__ constexpr int smem_bytes() {
    return oX<K>() + n_wg<K>() * nx<T>() * xbuf_bytes<T>();
}
}  // namespace encr

template <typename T, bool IS_K>
__global__ void __launch_bounds__(encr::n_threads<IS_K>(), encr::ctas_per_sm<IS_K>())
encode128_rows_kernel(const uint8_t *__restrict__ params, const T *__restrict__ x, int64_t n_vec, SlotMap map,
                      uint8_t *__restrict__ pool, int32_t *status) {
    using namespace encr;
    constexpr int NX = nx<T>(), RS = row_stride<T>(), RB = row_bytes<T>(), EPC = 16 / (int)sizeof(T);
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t xfull[2][2], xempty[2][2], mmabar[2];
    __shared__ uint32_t tmem_base;
    __shared__ float s_D[D];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, wg = tid >> 7, row = tid & 127, warp = tid >> 5;
    const int64_t ntiles = (n_vec + kRows - 1) / kRows;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&xfull[i][0], 1);
            tc::mbar_init(&xfull[i][1], 1);
            tc::mbar_init(&xempty[i][0], 4);   // one arrival per warp of the warpgroup
            tc::mbar_init(&xempty[i][1], 4);
            tc::mbar_init(&mmabar[i], 1);
        }
    }
    if (IS_K && warp == 0) tc::tmem_alloc(&tmem_base, 512);
    if (tid < D) s_D[tid] = reinterpret_cast<const float *>(params + params_off_D(D))[tid];
    if (IS_K) {   // B row n = S row k_col_coord(n)
        const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
        for (int e = tid; e < D * D; e += n_threads<IS_K>()) {
            const int n = e >> 7, k = e & 127;
            const int sr = k_col_coord(n);
            // S is held at binary16 precision: one exact f16 operand
            *reinterpret_cast<__half *>(smem + tc::sw128_off(n, k, D)) = __float2half_rn(__ldg(S + sr * D + k));
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = IS_K ? tmem_base + 256u * wg : 0u;
    const float t0 = ph->threshold[0], t1 = ph->threshold[1], t2 = ph->threshold[2], t3 = ph->threshold[3];
    const float t4 = ph->threshold[4], t5 = ph->threshold[5], t6 = ph->threshold[6];
    float cen[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) cen[k] = ph->centroid[k];
    const float inv_sd = rsqrtf((float)D);
    bool timed_out = false;

    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)(n_wg<IS_K>() * i + wg) * gridDim.x; };
    // the first warp of the warpgroup: the tile's rows, one bulk copy per row, spread over its lanes
    auto issue = [&](int i, int buf) {
        const int64_t v0 = tile_of(i) * kRows;
        const int rows = (int)min((int64_t)kRows, n_vec - v0);
        uint8_t *dst = smem + oX<IS_K>() + (wg * NX + buf) * xbuf_bytes<T>();
        if (row == 0) tc::mbar_arrive_expect_tx(&xfull[wg][buf], (uint32_t)rows * RB);
        for (int r = row; r < rows; r += 32)
            tc::bulk_g2s(dst + r * RS, x + (v0 + r) * D, RB, &xfull[wg][buf]);
    };
    if (row < 32)
        for (int b2 = 0; b2 < NX; ++b2)
            if (tile_of(b2) < ntiles) issue(b2, b2);
    const int bar_id = 1 + wg;

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int buf = i % NX, use = i / NX;
        const int64_t v0 = tile_of(i) * kRows, v = v0 + row;
        // the slot is needed only for the stores: a row past the input or without a slot is
        // computed on whatever its buffer holds (each row's results depend on that row only); its
        // load is issued here and checked there
        const int64_t sraw = v < n_vec ? map.slot_raw(v / map.n_heads) : -1;
        if (!tc::mbar_wait(&xfull[wg][buf], use & 1)) timed_out = true;
        // ---- 1. the row, in natural coordinate order
        float val[D];
        {
            const uint8_t *xr = smem + oX<IS_K>() + (wg * NX + buf) * xbuf_bytes<T>() + row * RS;
#pragma unroll
            for (int c = 0; c < RB / 16; ++c) {
                const uint4 u = *reinterpret_cast<const uint4 *>(xr + 16 * c);
                if constexpr (sizeof(T) == 2) {
                    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        val[EPC * c + 2 * q] = __uint_as_float(w4[q] << 16);
                        val[EPC * c + 2 * q + 1] = __uint_as_float(w4[q] & 0xFFFF0000u);
                    }
                } else {
                    val[EPC * c] = __uint_as_float(u.x);
                    val[EPC * c + 1] = __uint_as_float(u.y);
                    val[EPC * c + 2] = __uint_as_float(u.z);
                    val[EPC * c + 3] = __uint_as_float(u.w);
                }
            }
        }
        __syncwarp();
        if ((row & 31) == 0) tc::mbar_arrive(&xempty[wg][buf]);   // this warp's rows of the buffer are read
        // the first warp refills the buffer with the tile NX ahead once all four warps have read it:
        // at once when it is the only buffer, else after this tile's work (the other warps are long
        // done by then, so nobody waits)
        auto refill = [&]() {
            if (row < 32 && tile_of(i + NX) < ntiles) {
                if (!tc::mbar_wait(&xempty[wg][buf], use & 1)) timed_out = true;
                issue(i + NX, buf);
            }
        };
        if (NX == 1) refill();
        // ---- 2. norm, signs, transform
        float ss = 0.f;
#pragma unroll
        for (int n = 0; n < D; ++n) ss = fmaf(val[n], val[n], ss);
        const float nrm = sqrtf(ss);
#pragma unroll
        for (int n = 0; n < D; ++n) val[n] *= s_D[n];
#pragma unroll
        for (int st = 1; st < D; st <<= 1)
#pragma unroll
            for (int n = 0; n < D; ++n)
                if ((n & st) == 0) {
                    const float a0 = val[n], a1 = val[n | st];
                    val[n] = a0 + a1;
                    val[n | st] = a0 - a1;
                }
        const float rn = nrm > 0.f ? 1.f / nrm : 0.f;
        // ---- 3. cells: the three bits of the binary search on z = val / nrm.  V compares val
        // with the thresholds times nrm instead (a zero vector keeps the unit thresholds: z = 0 is
        // cell 4); K needs z itself for the residual.
        const float ns = (IS_K || nrm == 0.f) ? 1.f : nrm, zs = IS_K ? rn : 1.f;
        const float T0 = held_mul(t0, ns), T1 = held_mul(t1, ns), T2 = held_mul(t2, ns), T3 = held_mul(t3, ns),
                    T4 = held_mul(t4, ns), T5 = held_mul(t5, ns), T6 = held_mul(t6, ns);
        // K: the 16 words of the slot's fields, [tig][word]; V: the 48 bytes of the slot, byte
        // (gid, k, hf) at q = 6 gid + 2 k + hf of vb (4 per register)
        uint32_t kwd[4][4] = {{0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};
        uint32_t vb[12] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        float g2 = 0.f;
#pragma unroll
        for (int n = 0; n < D; ++n) {
            const float z = IS_K ? val[n] * zs : val[n];
            const bool b2 = z >= T3;
            const bool b1 = z >= (b2 ? T5 : T1);
            const bool b0 = z >= (b2 ? (b1 ? T6 : T4) : (b1 ? T2 : T0));
            const uint32_t cell = (uint32_t)b0 | ((uint32_t)b1 << 1) | ((uint32_t)b2 << 2);
            if (IS_K) {
                kwd[k_tig(n)][k_word(n)] |= cell << (4 * k_field(n));
                const float c = b2 ? (b1 ? (b0 ? cen[7] : cen[6]) : (b0 ? cen[5] : cen[4]))
                                   : (b1 ? (b0 ? cen[3] : cen[2]) : (b0 ? cen[1] : cen[0]));
                const float rho = z - c;
                g2 = fmaf(rho, rho, g2);
                val[n] = rho * 256.f;   // exact scaling; keeps the f16 low parts out of the subnormals
            } else {
                // V: coordinate n = 16 mt + gid + 8 ab; lane slot s = 2 mt + ab.  Slots 0..11 are the
                // field ab (bits 0..2) of byte (gid, k = mt >> 1, hf = mt & 1); slots 12..15 give bit k
                // of their cell to bit 3 of the field ab of byte (gid, k, hf = mt - 6), k = 0..2
                const int mt = n >> 4, gid = n & 7, ab = (n >> 3) & 1;
                if (mt < 6) {
                    const int q = 6 * gid + 2 * (mt >> 1) + (mt & 1);
                    vb[q >> 2] |= cell << (8 * (q & 3) + 4 * ab);
                } else {
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        const int q = 6 * gid + 2 * k + (mt - 6);
                        vb[q >> 2] |= ((cell >> k) & 1u) << (8 * (q & 3) + 4 * ab + 3);
                    }
                }
            }
        }
        if constexpr (IS_K) {
            // ---- 4. rho (x 256) as f16 hi / lo into this row's tensor-memory lane, then S rho
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t hw[32], lw[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float a0 = val[64 * q + 2 * c], a1 = val[64 * q + 2 * c + 1];
                    const __half2 h = __floats2half2_rn(a0, a1);
                    const float2 hf = __half22float2(h);
                    const __half2 l = __floats2half2_rn(a0 - hf.x, a1 - hf.y);
                    hw[c] = *reinterpret_cast<const uint32_t *>(&h);
                    lw[c] = *reinterpret_cast<const uint32_t *>(&l);
                }
                tc::st32(lane_addr + 32 * q, hw);
                tc::st32(lane_addr + 64 + 32 * q, lw);
            }
            tc::wait_st();
            tc::fence_before_sync();
            tc::named_sync(bar_id, 128);
            tc::fence_after_sync();
            if (row == 0) {
                const uint32_t bh = tc::smem_u32(smem);
                constexpr uint32_t id = tc::idesc_f16(kRows, D);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_ts_f16(tmem + 128, tmem + 8 * ks, tc::sw128_desc(bh, ks, D), id, ks > 0);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    tc::mma_ts_f16(tmem + 128, tmem + 64 + 8 * ks, tc::sw128_desc(bh, ks, D), id, true);
                tc::mma_commit(&mmabar[wg]);
            }
            if (!tc::mbar_wait(&mmabar[wg], i & 1)) timed_out = true;
            tc::fence_after_sync();
#pragma unroll
            for (int j = 0; j < D / 16; ++j) {
                float pv[16];
                tc::ld16(lane_addr + 128 + 16 * j, pv);
                tc::wait_ld();
#pragma unroll
                for (int b = 0; b < 16; ++b) asm volatile("" : "+f"(pv[b]));   // no use moves above the wait
#pragma unroll
                for (int b = 0; b < 16; ++b)   // column 16 j + b: field b & 7 of word (tig j & 3, 2 (j >> 2) + (b >> 3))
                    kwd[j & 3][2 * (j >> 2) + (b >> 3)] |= (pv[b] >= 0.f ? 8u : 0u) << (4 * (b & 7));
            }
            tc::fence_before_sync();
        }
        // ---- 5. the record words of this row's slot
        const int64_t slot = map.slot_check(sraw, status, v < n_vec && (v % map.n_heads) == 0);
        if (slot >= 0) {
            const int64_t blk = slot / kBlock;
            const int o = (int)(slot % kBlock), head = (int)(v % map.n_heads);
            if (IS_K) {
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * k_record(D);
                const int gid = o & 7, th = o >> 3;
#pragma unroll
                for (int tig = 0; tig < 4; ++tig)
                    reinterpret_cast<uint4 *>(rec)[(4 * gid + tig) * 2 + th] =
                        make_uint4(kwd[tig][0], kwd[tig][1], kwd[tig][2], kwd[tig][3]);
                const float gam = sqrtf(g2) * inv_sd;
                *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * o) = __halves2half2(__float2half_rn(nrm), __float2half_rn(gam));
            } else {
                uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * v_record(D);
                const int tigv = (o & 7) >> 1, pr = o >> 3, e = o & 1;
#pragma unroll
                for (int q = 0; q < 48; ++q) {   // byte (gid, k, hf) of word 3 (L * 2 + pair) + k, byte 2 hf + e
                    const int gid = q / 6, k = (q % 6) >> 1, hf = q & 1;
                    rec[((size_t)((4 * gid + tigv) * 2 + pr) * 3 + k) * 4 + 2 * hf + e] = (uint8_t)(vb[q >> 2] >> (8 * (q & 3)));
                }
                *reinterpret_cast<__half *>(rec + 6 * D + 2 * o) = __float2half_rn(nrm);
            }
        }
        if (IS_K) tc::named_sync(bar_id, 128);   // the accumulator and A lanes are free for the next tile
        if (NX > 1) refill();
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
    if (IS_K) {
        tc::fence_before_sync();
        __syncthreads();
        if (warp == 0) tc::tmem_dealloc(tmem_base, 512);
    }
}

// ---------------------------------------------------------------- V at d = 128 from bf16, TMA input
// Thread r of a CTA of 128 owns row r of a 128-row tile from input to record:
//  1. the tile arrives as two TMA tensor boxes (columns 0..63 and 64..127, 128 rows x 128 bytes,
//     swizzled: the 16-byte chunk c of row r sits at chunk c ^ (r & 7)), kNX tiles in flight;
//  2. the signs D by an XOR of the input words (bit 15 / 31 of each bf16 pair), then the norm and
//     the 128-point transform on f32x2 pairs (x_k, x_{k+64}): the stage on index bit 6 inside
//     each pair, the other six between pairs, a packed add and a packed subtract for two
//     butterflies at once;
//  3. cells by the three-compare search against the thresholds times the norm;
//  4. a tile whose 16-token blocks are whole (16-aligned slots in token order; the kv heads H
//     divide 8, so the tile is 8 / H blocks of H records) assembles its 8 records in shared
//     memory and writes them with 16-byte stores; any other tile stores its bytes one by one.
namespace encv {
constexpr int D = 128, kRows = 128, kThreads = 128, kNX = 2, kCtasPerSm = 3;
constexpr int kBox = kRows * 128;            // one box: 128 rows x 128 bytes
constexpr int kTile = 2 * kBox;              // bf16 rows of 256 bytes
constexpr int kRec = 6 * D + 2 * kBlock;     // V record bytes
constexpr int kImg = 8 * kRec;               // the 8 records of a whole tile
constexpr int smem_bytes() { return 1024 + kNX * kTile + kImg; }   // 1024: slack to align the boxes
}  // namespace encv

__global__ void __launch_bounds__(encv::kThreads, encv::kCtasPerSm)
encode128v_tma_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t *__restrict__ params, int64_t n_vec,
                      SlotMap map, int whole_ok, uint8_t *__restrict__ pool, int32_t *status) {
    using namespace encv;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *tiles = smem;                  // [kNX][2 boxes][128 rows][128 bytes]
    uint8_t *img = smem + kNX * kTile;      // [8][kRec]
    __shared__ uint64_t full[kNX], empty[kNX];
    __shared__ __align__(16) uint32_t s_sg[D / 2];   // XOR masks of the bf16 pairs
    __shared__ int64_t s_blk[2][8];                  // first-token slot of each block, by tile parity
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31, row = tid;
    const int64_t ntiles = (n_vec + kRows - 1) / kRows;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        for (int i = 0; i < kNX; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], kThreads / 32);   // one arrival per warp
        }
    }
    if (tid < D / 2) {
        const float *Dp = reinterpret_cast<const float *>(params + params_off_D(D));
        s_sg[tid] = (Dp[2 * tid] < 0.f ? 0x8000u : 0u) | (Dp[2 * tid + 1] < 0.f ? 0x80000000u : 0u);
    }
    tc::fence_async_smem();
    __syncthreads();
    const float t0 = ph->threshold[0], t1 = ph->threshold[1], t2 = ph->threshold[2], t3 = ph->threshold[3];
    const float t4 = ph->threshold[4], t5 = ph->threshold[5], t6 = ph->threshold[6];
    const int H = map.n_heads;
    const bool small = n_vec <= (int64_t)0x7fffffff;
    bool timed_out = false;

    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)i * gridDim.x; };
    auto issue = [&](int i, int buf) {   // thread 0: the tile's two boxes
        const int y = (int)(tile_of(i) * kRows);
        tc::mbar_arrive_expect_tx(&full[buf], (uint32_t)kTile);
        tc::tma_load_2d(tiles + buf * kTile, &tmap, 0, y, &full[buf]);
        tc::tma_load_2d(tiles + buf * kTile + kBox, &tmap, 64, y, &full[buf]);
    };
    if (tid == 0)
        for (int b2 = 0; b2 < kNX; ++b2)
            if (tile_of(b2) < ntiles) issue(b2, b2);

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int buf = i % kNX, use = i / kNX;
        const int64_t v0 = tile_of(i) * kRows, v = v0 + row;
        const bool live = v < n_vec;
        const int64_t tok = small ? (int64_t)((uint32_t)v / (uint32_t)H) : v / H;
        const int head = (int)(v - tok * H);
        const int64_t sraw = live ? map.slot_raw(tok) : -1;   // checked at the stores
        if (!tc::mbar_wait(&full[buf], use & 1)) timed_out = true;
        // ---- 1. the row: word p holds coordinates 2p (low half) and 2p + 1 (high half)
        uint32_t w[64];
        {
            const uint8_t *rb = tiles + buf * kTile + row * 128;
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(rb + q * kBox + ((c ^ (row & 7)) << 4));
                    w[32 * q + 4 * c] = u.x;
                    w[32 * q + 4 * c + 1] = u.y;
                    w[32 * q + 4 * c + 2] = u.z;
                    w[32 * q + 4 * c + 3] = u.w;
                }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[buf]);   // this warp's rows of the buffer are read
        // ---- 2. signs, norm, transform on pairs P[k] = (x_k, x_{k+64})
        float2 P[64];
#pragma unroll
        for (int p4 = 0; p4 < 8; ++p4) {
            const uint4 sa = reinterpret_cast<const uint4 *>(s_sg)[p4], sb = reinterpret_cast<const uint4 *>(s_sg)[p4 + 8];
            const uint32_t ma[4] = {sa.x, sa.y, sa.z, sa.w}, mb[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int p = 4 * p4 + e;
                const uint32_t a = w[p] ^ ma[e], b = w[p + 32] ^ mb[e];
                P[2 * p] = make_float2(__uint_as_float(a << 16), __uint_as_float(b << 16));
                P[2 * p + 1] = make_float2(__uint_as_float(a & 0xFFFF0000u), __uint_as_float(b & 0xFFFF0000u));
            }
        }
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 64; ++k) acc = __ffma2_rn(P[k], P[k], acc);
        const float nrm = sqrtf(acc.x + acc.y);
#pragma unroll
        for (int k = 0; k < 64; ++k) P[k] = make_float2(P[k].x + P[k].y, P[k].x - P[k].y);
        const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
        for (int st = 1; st < 64; st <<= 1)
#pragma unroll
            for (int k = 0; k < 64; ++k)
                if ((k & st) == 0) {
                    const float2 a = P[k], b = P[k | st];
                    P[k] = __fadd2_rn(a, b);
                    P[k | st] = __ffma2_rn(b, m1, a);   // a - b
                }
        // ---- 3. cells against the thresholds times the norm (a zero row keeps the unit thresholds)
        const float ns = nrm == 0.f ? 1.f : nrm;
        const float T0 = held_mul(t0, ns), T1 = held_mul(t1, ns), T2 = held_mul(t2, ns), T3 = held_mul(t3, ns),
                    T4 = held_mul(t4, ns), T5 = held_mul(t5, ns), T6 = held_mul(t6, ns);
        // the 48 bytes of the slot, byte (gid, k, hf) at q = 6 gid + 2 k + hf of vb (4 per register)
        uint32_t vb[12] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int n = 0; n < D; ++n) {
            const float z = n < 64 ? P[n].x : P[n - 64].y;
            const bool b2 = z >= T3;
            const bool b1 = z >= (b2 ? T5 : T1);
            const bool b0 = z >= (b2 ? (b1 ? T6 : T4) : (b1 ? T2 : T0));
            const uint32_t cell = (uint32_t)b0 | ((uint32_t)b1 << 1) | ((uint32_t)b2 << 2);
            // coordinate n = 16 mt + gid + 8 ab: slots 0..11 are field ab (bits 0..2) of byte
            // (gid, k = mt >> 1, hf = mt & 1); slots 12..15 give bit k of their cell to bit 3 of
            // field ab of byte (gid, k, hf = mt - 6), k = 0..2
            const int mt = n >> 4, gid = n & 7, ab = (n >> 3) & 1;
            if (mt < 6) {
                const int q = 6 * gid + 2 * (mt >> 1) + (mt & 1);
                vb[q >> 2] |= cell << (8 * (q & 3) + 4 * ab);
            } else {
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int q = 6 * gid + 2 * k + (mt - 6);
                    vb[q >> 2] |= ((cell >> k) & 1u) << (8 * (q & 3) + 4 * ab + 3);
                }
            }
        }
        // ---- 4. stores
        const int64_t slot = map.slot_check(sraw, status, live && head == 0);
        const int rel = row / H, bi = rel >> 4, o = rel & 15;   // token within the tile, its block and offset
        bool whole = false;
        if (whole_ok) {   // CTA-uniform
            if (o == 0 && head == 0) s_blk[i & 1][bi] = sraw;
            __syncthreads();
            const int64_t first = s_blk[i & 1][bi];
            whole = __syncthreads_and(live && slot >= 0 && (int)(slot & 15) == o && (slot >> 4) == (first >> 4));
        }
        if (whole) {
            uint8_t *rec = img + (bi * H + head) * kRec;
            const int tigv = (o & 7) >> 1, pr = o >> 3, e = o & 1;
#pragma unroll
            for (int q = 0; q < 48; ++q) {   // byte (gid, k, hf) of word 3 (L * 2 + pair) + k, byte 2 hf + e
                const int gid = q / 6, k = (q % 6) >> 1, hf = q & 1;
                rec[(((4 * gid + tigv) * 2 + pr) * 3 + k) * 4 + 2 * hf + e] = (uint8_t)(vb[q >> 2] >> (8 * (q & 3)));
            }
            *reinterpret_cast<__half *>(rec + 6 * D + 2 * o) = __float2half_rn(nrm);
            __syncthreads();
            for (int c = tid; c < 8 * (kRec / 16); c += kThreads) {
                const int j = c / (kRec / 16), cc = c % (kRec / 16);
                const int64_t blk = s_blk[i & 1][j / H] >> 4;
                *reinterpret_cast<uint4 *>(pool + ((size_t)blk * H + j % H) * kRec + 16 * cc) =
                    *reinterpret_cast<const uint4 *>(img + j * kRec + 16 * cc);
            }
        } else if (slot >= 0) {
            const int64_t blk = slot / kBlock;
            const int so = (int)(slot % kBlock);
            uint8_t *rec = pool + ((size_t)blk * H + head) * kRec;
            const int tigv = (so & 7) >> 1, pr = so >> 3, e = so & 1;
#pragma unroll
            for (int q = 0; q < 48; ++q) {
                const int gid = q / 6, k = (q % 6) >> 1, hf = q & 1;
                rec[(((4 * gid + tigv) * 2 + pr) * 3 + k) * 4 + 2 * hf + e] = (uint8_t)(vb[q >> 2] >> (8 * (q & 3)));
            }
            *reinterpret_cast<__half *>(rec + 6 * D + 2 * so) = __float2half_rn(nrm);
        }
        // the buffer takes the tile kNX ahead once all four warps have read it (long done by now)
        if (tid == 0 && tile_of(i + kNX) < ntiles) {
            if (!tc::mbar_wait(&empty[buf], use & 1)) timed_out = true;
            issue(i + kNX, buf);
        }
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
}

// ---------------------------------------------------------------- V at d = 256 from bf16, TMA input
// Two threads per row: thread (row, h) owns coordinates 128 h .. 128 h + 127, which are exactly
// slot group g = h of the V record (its 48 bytes), so the halves share only the norm.
//  1. the tile (128 rows x 512 bytes) arrives as four TMA boxes of 64 columns; one tile in
//     flight, the buffer refilled as soon as every warp has read its rows;
//  2. half h takes the transform's stage on index bit 7 on the input (u_m = x_m +- x_{m+128},
//     signs D by XOR), then the 128-point transform of its coordinates on f32x2 pairs
//     (u_k, u_{k+64}); the halves' sums of squares add to twice |x|^2;
//  3. cells against the thresholds times the norm, and the group's bytes;
//  4. whole tiles (as encode128v_tma_kernel) assemble their 8 records in shared memory.
namespace encv2 {
constexpr int D = 256, kRows = 128, kThreads = 256, kCtasPerSm = 1;
constexpr int kBox = kRows * 128;            // one box: 128 rows x 64 bf16
constexpr int kTile = 4 * kBox;
constexpr int kRec = 6 * D + 2 * kBlock;
constexpr int kImg = 8 * kRec;
constexpr int smem_bytes() { return 1024 + kTile + kImg; }
}  // namespace encv2

__global__ void __launch_bounds__(encv2::kThreads, encv2::kCtasPerSm)
encode256v_tma_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t *__restrict__ params, int64_t n_vec,
                      SlotMap map, int whole_ok, uint8_t *__restrict__ pool, int32_t *status) {
    using namespace encv2;
    constexpr int NG = D / 128;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *tile = smem;                   // [4 boxes][128 rows][128 bytes]
    uint8_t *img = smem + kTile;            // [8][kRec]
    __shared__ uint64_t full, empty;
    __shared__ __align__(16) uint32_t s_sg[D / 2];
    __shared__ int64_t s_blk[2][8];
    __shared__ float s_ss[2][kRows];                // the halves' sums of squares
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, h = warp >> 2, row = 32 * (warp & 3) + lane;
    const int64_t ntiles = (n_vec + kRows - 1) / kRows;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        tc::mbar_init(&full, 1);
        tc::mbar_init(&empty, kThreads / 32);
    }
    if (tid < D / 2) {
        const float *Dp = reinterpret_cast<const float *>(params + params_off_D(D));
        s_sg[tid] = (Dp[2 * tid] < 0.f ? 0x8000u : 0u) | (Dp[2 * tid + 1] < 0.f ? 0x80000000u : 0u);
    }
    tc::fence_async_smem();
    __syncthreads();
    const float t0 = ph->threshold[0], t1 = ph->threshold[1], t2 = ph->threshold[2], t3 = ph->threshold[3];
    const float t4 = ph->threshold[4], t5 = ph->threshold[5], t6 = ph->threshold[6];
    const int H = map.n_heads;
    const bool small = n_vec <= (int64_t)0x7fffffff;
    bool timed_out = false;
    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)i * gridDim.x; };
    auto issue = [&](int i) {   // thread 0: the tile's four boxes
        const int y = (int)(tile_of(i) * kRows);
        tc::mbar_arrive_expect_tx(&full, (uint32_t)kTile);
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::tma_load_2d(tile + q * kBox, &tmap, 64 * q, y, &full);
    };
    if (tid == 0) issue(0);

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int64_t v0 = tile_of(i) * kRows, v = v0 + row;
        const bool live = v < n_vec;
        const int64_t tok = small ? (int64_t)((uint32_t)v / (uint32_t)H) : v / H;
        const int head = (int)(v - tok * H);
        const int64_t sraw = live ? map.slot_raw(tok) : -1;   // checked at the stores
        if (!tc::mbar_wait(&full, i & 1)) timed_out = true;
        // ---- 1. pairs P[k] = (u_k, u_{k+64}) of this half: u_m = x_m +- x_{m+128} (signs applied);
        // box q word p holds coordinates 64 q + 2 p, 64 q + 2 p + 1
        float2 P[64];
        {
            const uint8_t *rb = tile + row * 128;
            const float2 sgn = make_float2(h ? -1.f : 1.f, h ? -1.f : 1.f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int off = (c ^ (row & 7)) << 4;
                const uint4 a0 = *reinterpret_cast<const uint4 *>(rb + off);              // x_{8c .. 8c+7}
                const uint4 a1 = *reinterpret_cast<const uint4 *>(rb + kBox + off);       // x_{64+8c ..}
                const uint4 b0 = *reinterpret_cast<const uint4 *>(rb + 2 * kBox + off);   // x_{128+8c ..}
                const uint4 b1 = *reinterpret_cast<const uint4 *>(rb + 3 * kBox + off);   // x_{192+8c ..}
                const uint4 m0 = reinterpret_cast<const uint4 *>(s_sg)[c], m1 = reinterpret_cast<const uint4 *>(s_sg)[8 + c];
                const uint4 m2 = reinterpret_cast<const uint4 *>(s_sg)[16 + c], m3 = reinterpret_cast<const uint4 *>(s_sg)[24 + c];
                const uint32_t wa0[4] = {a0.x ^ m0.x, a0.y ^ m0.y, a0.z ^ m0.z, a0.w ^ m0.w};
                const uint32_t wa1[4] = {a1.x ^ m1.x, a1.y ^ m1.y, a1.z ^ m1.z, a1.w ^ m1.w};
                const uint32_t wb0[4] = {b0.x ^ m2.x, b0.y ^ m2.y, b0.z ^ m2.z, b0.w ^ m2.w};
                const uint32_t wb1[4] = {b1.x ^ m3.x, b1.y ^ m3.y, b1.z ^ m3.z, b1.w ^ m3.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 8 * c + 2 * e;   // pairs k (even) and k + 1 (odd coordinates)
                    const float2 lo_a = make_float2(__uint_as_float(wa0[e] << 16), __uint_as_float(wa1[e] << 16));
                    const float2 hi_a = make_float2(__uint_as_float(wa0[e] & 0xFFFF0000u), __uint_as_float(wa1[e] & 0xFFFF0000u));
                    const float2 lo_b = make_float2(__uint_as_float(wb0[e] << 16), __uint_as_float(wb1[e] << 16));
                    const float2 hi_b = make_float2(__uint_as_float(wb0[e] & 0xFFFF0000u), __uint_as_float(wb1[e] & 0xFFFF0000u));
                    P[k] = __ffma2_rn(lo_b, sgn, lo_a);
                    P[k + 1] = __ffma2_rn(hi_b, sgn, hi_a);
                }
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty);   // this warp's rows of the buffer are read
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 64; ++k) acc = __ffma2_rn(P[k], P[k], acc);
        s_ss[h][row] = acc.x + acc.y;
        // the buffer takes the next tile once every warp has read it
        if (tid == 0 && tile_of(i + 1) < ntiles) {
            if (!tc::mbar_wait(&empty, i & 1)) timed_out = true;
            issue(i + 1);
        }
#pragma unroll
        for (int k = 0; k < 64; ++k) P[k] = make_float2(P[k].x + P[k].y, P[k].x - P[k].y);
        const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
        for (int st = 1; st < 64; st <<= 1)
#pragma unroll
            for (int k = 0; k < 64; ++k)
                if ((k & st) == 0) {
                    const float2 a = P[k], b = P[k | st];
                    P[k] = __fadd2_rn(a, b);
                    P[k | st] = __ffma2_rn(b, m1, a);   // a - b
                }
        __syncthreads();   // both halves' sums of squares are in
        const float nrm = sqrtf(0.5f * (s_ss[0][row] + s_ss[1][row]));
        // ---- 2. cells of coordinates 128 h + n against the thresholds times the norm
        const float ns = nrm == 0.f ? 1.f : nrm;
        const float T0 = held_mul(t0, ns), T1 = held_mul(t1, ns), T2 = held_mul(t2, ns), T3 = held_mul(t3, ns),
                    T4 = held_mul(t4, ns), T5 = held_mul(t5, ns), T6 = held_mul(t6, ns);
        uint32_t vb[12] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int n = 0; n < 128; ++n) {
            const float z = n < 64 ? P[n].x : P[n - 64].y;
            const bool b2 = z >= T3;
            const bool b1 = z >= (b2 ? T5 : T1);
            const bool b0 = z >= (b2 ? (b1 ? T6 : T4) : (b1 ? T2 : T0));
            const uint32_t cell = (uint32_t)b0 | ((uint32_t)b1 << 1) | ((uint32_t)b2 << 2);
            const int mt = n >> 4, gid = n & 7, ab = (n >> 3) & 1;
            if (mt < 6) {
                const int q = 6 * gid + 2 * (mt >> 1) + (mt & 1);
                vb[q >> 2] |= cell << (8 * (q & 3) + 4 * ab);
            } else {
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int q = 6 * gid + 2 * k + (mt - 6);
                    vb[q >> 2] |= ((cell >> k) & 1u) << (8 * (q & 3) + 4 * ab + 3);
                }
            }
        }
        // ---- 3. stores: byte (gid, k, hf) of group g = h in word ((4 gid + tig) 2 + pair) 3 NG + 3 g + k
        const int64_t slot = map.slot_check(sraw, status, live && head == 0 && h == 0);
        const int rel = row / H, bi = rel >> 4, o = rel & 15;
        bool whole = false;
        if (whole_ok) {   // CTA-uniform
            if (o == 0 && head == 0 && h == 0) s_blk[i & 1][bi] = sraw;
            __syncthreads();
            const int64_t first = s_blk[i & 1][bi];
            whole = __syncthreads_and(live && slot >= 0 && (int)(slot & 15) == o && (slot >> 4) == (first >> 4));
        }
        auto put = [&](uint8_t *rec, int so) {
            const int tigv = (so & 7) >> 1, pr = so >> 3, e = so & 1;
#pragma unroll
            for (int q = 0; q < 48; ++q) {
                const int gid = q / 6, k = (q % 6) >> 1, hf = q & 1;
                rec[(((4 * gid + tigv) * 2 + pr) * 3 * NG + 3 * h + k) * 4 + 2 * hf + e] = (uint8_t)(vb[q >> 2] >> (8 * (q & 3)));
            }
            if (h == 0) *reinterpret_cast<__half *>(rec + 6 * D + 2 * so) = __float2half_rn(nrm);
        };
        if (whole) {
            put(img + (bi * H + head) * kRec, o);
            __syncthreads();
            for (int c = tid; c < 8 * (kRec / 16); c += kThreads) {
                const int j = c / (kRec / 16), cc = c % (kRec / 16);
                const int64_t blk = s_blk[i & 1][j / H] >> 4;
                *reinterpret_cast<uint4 *>(pool + ((size_t)blk * H + j % H) * kRec + 16 * cc) =
                    *reinterpret_cast<const uint4 *>(img + j * kRec + 16 * cc);
            }
        } else if (slot >= 0) {
            put(pool + ((size_t)(slot / kBlock) * H + head) * kRec, (int)(slot % kBlock));
        }
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
}

// ---------------------------------------------------------------- K at d = 256 from bf16 on tcgen05
// A CTA of 256 threads per SM walks tiles of 128 rows; thread (row, h) owns coordinates
// 128 h .. 128 h + 127 of its row:
//  1. the tile arrives as four TMA boxes (one tile in flight, refilled once every warp has read
//     it); half h takes the transform's stage on index bit 7 on the input (u_m = x_m +- x_{m+128},
//     signs D by XOR), then its 128-point transform on f32x2 pairs (u_k, u_{k+64});
//  2. the halves' sums of squares give the norm; cells and the residual (x 256) as in the d = 128
//     encoder, the residual's f16 hi and lo going to this row's tensor-memory lane (A operand:
//     hi in columns 0..127, lo in 128..255, coordinate 2c and 2c + 1 in column c);
//  3. one thread issues p = S rho (M = 128 rows, N = 256 projections, K = 256 coordinates) as
//     S rho_hi + S rho_lo: 32 MMAs into columns 256..511.  S is held at binary16 precision, so
//     it is one f16 operand (128 KB of shared memory, rows reordered so that accumulator column
//     64 h2 + 16 tig + 8 wl + f is field f of word (tig, 2 h2 + wl));
//  4. each half reads back its 128 columns (its own four words per tig) and stores them; half 0
//     stores fp16 n and gamma.
namespace enck2 {
constexpr int D = 256, kRows = 128, kThreads = 256;
constexpr int kBox = kRows * 128;
constexpr int kTile = 4 * kBox;                 // 64 KB of bf16 rows
constexpr int oS = 0;                           // S, f16, 128-byte swizzled K-major, 256 rows
constexpr int oX = D * D * 2;                   // the input tile
constexpr int smem_bytes() { return 1024 + oX + kTile; }
}  // namespace enck2

__global__ void __launch_bounds__(enck2::kThreads, 1)
encode256k_tc_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t *__restrict__ params, int64_t n_vec,
                     SlotMap map, uint8_t *__restrict__ pool, int32_t *status) {
    using namespace enck2;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *tile = smem + oX;
    __shared__ uint64_t full, empty, mmabar;
    __shared__ uint32_t tmem_base;
    __shared__ __align__(16) uint32_t s_sg[D / 2];
    __shared__ float s_ss[2][kRows], s_g2[kRows];
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, h = warp >> 2, row = 32 * (warp & 3) + lane;
    const int64_t ntiles = (n_vec + kRows - 1) / kRows;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        tc::mbar_init(&full, 1);
        tc::mbar_init(&empty, kThreads / 32);
        tc::mbar_init(&mmabar, 1);
    }
    if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
    if (tid < D / 2) {
        const float *Dp = reinterpret_cast<const float *>(params + params_off_D(D));
        s_sg[tid] = (Dp[2 * tid] < 0.f ? 0x8000u : 0u) | (Dp[2 * tid + 1] < 0.f ? 0x80000000u : 0u);
    }
    {   // B row n = S row k_col_coord(n), f16 (exact: S is held at binary16 precision)
        const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
        for (int e = tid; e < D * D; e += kThreads) {
            const int n = e >> 8, k = e & 255;
            *reinterpret_cast<__half *>(smem + oS + tc::sw128_off(n, k, D)) =
                __float2half_rn(__ldg(S + k_col_coord(n) * D + k));
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float T0 = 256.f * ph->threshold[0], T1 = 256.f * ph->threshold[1], T2 = 256.f * ph->threshold[2];
    const float T3 = 256.f * ph->threshold[3], T4 = 256.f * ph->threshold[4], T5 = 256.f * ph->threshold[5];
    const float T6 = 256.f * ph->threshold[6];
    const float hw_out = 128.f * (ph->centroid[7] - ph->centroid[6]), hw_in = 128.f * (ph->centroid[5] - ph->centroid[4]);
    const float inv_sd = rsqrtf((float)D);
    const int H = map.n_heads;
    const bool small = n_vec <= (int64_t)0x7fffffff;
    bool timed_out = false;
    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)i * gridDim.x; };
    auto issue = [&](int i) {   // thread 0: the tile's four boxes
        const int y = (int)(tile_of(i) * kRows);
        tc::mbar_arrive_expect_tx(&full, (uint32_t)kTile);
#pragma unroll
        for (int q = 0; q < 4; ++q) tc::tma_load_2d(tile + q * kBox, &tmap, 64 * q, y, &full);
    };
    if (tid == 0) issue(0);

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int64_t v0 = tile_of(i) * kRows, v = v0 + row;
        const bool live = v < n_vec;
        const int64_t tok = small ? (int64_t)((uint32_t)v / (uint32_t)H) : v / H;
        const int head = (int)(v - tok * H);
        const int64_t sraw = live ? map.slot_raw(tok) : -1;   // checked at the stores
        if (!tc::mbar_wait(&full, i & 1)) timed_out = true;
        // ---- 1. pairs P[k] = (u_k, u_{k+64}) of this half (as encode256v_tma_kernel)
        float2 P[64];
        {
            const uint8_t *rb = tile + row * 128;
            const float2 sgn = make_float2(h ? -1.f : 1.f, h ? -1.f : 1.f);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int off = (c ^ (row & 7)) << 4;
                const uint4 a0 = *reinterpret_cast<const uint4 *>(rb + off);
                const uint4 a1 = *reinterpret_cast<const uint4 *>(rb + kBox + off);
                const uint4 b0 = *reinterpret_cast<const uint4 *>(rb + 2 * kBox + off);
                const uint4 b1 = *reinterpret_cast<const uint4 *>(rb + 3 * kBox + off);
                const uint4 m0 = reinterpret_cast<const uint4 *>(s_sg)[c], m1 = reinterpret_cast<const uint4 *>(s_sg)[8 + c];
                const uint4 m2 = reinterpret_cast<const uint4 *>(s_sg)[16 + c], m3 = reinterpret_cast<const uint4 *>(s_sg)[24 + c];
                const uint32_t wa0[4] = {a0.x ^ m0.x, a0.y ^ m0.y, a0.z ^ m0.z, a0.w ^ m0.w};
                const uint32_t wa1[4] = {a1.x ^ m1.x, a1.y ^ m1.y, a1.z ^ m1.z, a1.w ^ m1.w};
                const uint32_t wb0[4] = {b0.x ^ m2.x, b0.y ^ m2.y, b0.z ^ m2.z, b0.w ^ m2.w};
                const uint32_t wb1[4] = {b1.x ^ m3.x, b1.y ^ m3.y, b1.z ^ m3.z, b1.w ^ m3.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 8 * c + 2 * e;
                    const float2 lo_a = make_float2(__uint_as_float(wa0[e] << 16), __uint_as_float(wa1[e] << 16));
                    const float2 hi_a = make_float2(__uint_as_float(wa0[e] & 0xFFFF0000u), __uint_as_float(wa1[e] & 0xFFFF0000u));
                    const float2 lo_b = make_float2(__uint_as_float(wb0[e] << 16), __uint_as_float(wb1[e] << 16));
                    const float2 hi_b = make_float2(__uint_as_float(wb0[e] & 0xFFFF0000u), __uint_as_float(wb1[e] & 0xFFFF0000u));
                    P[k] = __ffma2_rn(lo_b, sgn, lo_a);
                    P[k + 1] = __ffma2_rn(hi_b, sgn, hi_a);
                }
            }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty);
        {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 64; ++k) acc = __ffma2_rn(P[k], P[k], acc);
            s_ss[h][row] = acc.x + acc.y;
        }
        if (tid == 0 && tile_of(i + 1) < ntiles) {
            if (!tc::mbar_wait(&empty, i & 1)) timed_out = true;
            issue(i + 1);
        }
#pragma unroll
        for (int k = 0; k < 64; ++k) P[k] = make_float2(P[k].x + P[k].y, P[k].x - P[k].y);
        {
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int st = 1; st < 64; st <<= 1)
#pragma unroll
                for (int k = 0; k < 64; ++k)
                    if ((k & st) == 0) {
                        const float2 a = P[k], b = P[k | st];
                        P[k] = __fadd2_rn(a, b);
                        P[k | st] = __ffma2_rn(b, m1, a);
                    }
        }
        tc::named_sync(1, kThreads);   // both halves' sums of squares are in
        const float nrm = sqrtf(0.5f * (s_ss[0][row] + s_ss[1][row]));
        const float rs = nrm > 0.f ? 256.f / nrm : 0.f;
        // ---- 2. cells and residual of coordinates 128 h + m (Z = 256 z; see the d = 128 encoder)
        uint32_t kwd[4][4] = {{0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}, {0u, 0u, 0u, 0u}};
        float g2 = 0.f;
#pragma unroll
        for (int m = 0; m < 128; ++m) {
            float &pz = (m < 64) ? P[m].x : P[m - 64].y;
            const float Z = pz * rs;
            const bool b2 = Z >= T3;
            const bool b1 = Z >= (b2 ? T5 : T1);
            const float dz = Z - (b2 ? (b1 ? T6 : T4) : (b1 ? T2 : T0));
            const bool b0 = dz >= 0.f;
            kwd[k_tig(m)][k_word(m)] |= ((uint32_t)b0 | ((uint32_t)b1 << 1) | ((uint32_t)b2 << 2)) << (4 * k_field(m));
            const float hw = (b1 == b2) ? hw_out : hw_in;
            const float rho = b0 ? dz - hw : dz + hw;
            g2 = fmaf(rho, rho, g2);
            pz = rho;
        }
        if (h == 1) s_g2[row] = g2;
        // ---- 3. rho (x 256) as f16 hi / lo into this row's lane: columns 64 h + c (hi) and
        // 128 + 64 h + c (lo) hold coordinates 128 h + 2c, 128 h + 2c + 1
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float hw16[16], lw16[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int m0 = 32 * q + 2 * c;   // this half's coordinates m0, m0 + 1
                const float a0 = m0 < 64 ? P[m0].x : P[m0 - 64].y, a1 = (m0 + 1) < 64 ? P[m0 + 1].x : P[m0 + 1 - 64].y;
                const __half2 hh = __floats2half2_rn(a0, a1);
                const float2 hf = __half22float2(hh);
                const __half2 ll = __floats2half2_rn(a0 - hf.x, a1 - hf.y);
                hw16[c] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&hh));
                lw16[c] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&ll));
            }
            tc::st16(lane_addr + 64 * h + 16 * q, hw16);
            tc::st16(lane_addr + 128 + 64 * h + 16 * q, lw16);
        }
        tc::wait_st();
        tc::fence_before_sync();
        tc::named_sync(1, kThreads);
        tc::fence_after_sync();
        if (tid == 0) {
            const uint32_t bs = tc::smem_u32(smem + oS);
            constexpr uint32_t id = tc::idesc_f16(kRows, D);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_ts_f16(tmem + 256, tmem + 8 * ks, tc::sw128_desc(bs, ks, D), id, ks > 0);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_ts_f16(tmem + 256, tmem + 128 + 8 * ks, tc::sw128_desc(bs, ks, D), id, true);
            tc::mma_commit(&mmabar);
        }
        if (!tc::mbar_wait(&mmabar, i & 1)) timed_out = true;
        tc::fence_after_sync();
        // ---- 4. QJL signs: accumulator column 128 h + 16 j + b is field b & 7 of this half's word
        // (tig j & 3, 2 (j >> 2) + (b >> 3))
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float pv[16];
            tc::ld16(lane_addr + 256 + 128 * h + 16 * j, pv);
            tc::wait_ld();
#pragma unroll
            for (int b = 0; b < 16; ++b) asm volatile("" : "+f"(pv[b]));   // no use moves above the wait
#pragma unroll
            for (int b = 0; b < 16; ++b)
                kwd[j & 3][2 * (j >> 2) + (b >> 3)] |= ((~__float_as_uint(pv[b]) >> 31) << 3) << (4 * (b & 7));
        }
        tc::fence_before_sync();
        tc::named_sync(1, kThreads);   // half 1's residual sum is in; the accumulator and A are free
        const int64_t slot = map.slot_check(sraw, status, live && h == 0 && head == 0);
        if (slot >= 0) {
            const int64_t blk = slot / kBlock;
            const int o = (int)(slot % kBlock);
            uint8_t *rec = pool + ((size_t)blk * H + head) * k_record(D);
            const int gid = o & 7, th = o >> 3;
#pragma unroll
            for (int tig = 0; tig < 4; ++tig)   // words 4 h .. 4 h + 3 of word row (4 gid + tig) * 2 + th
                reinterpret_cast<uint4 *>(rec)[((4 * gid + tig) * 2 + th) * 2 + h] =
                    make_uint4(kwd[tig][0], kwd[tig][1], kwd[tig][2], kwd[tig][3]);
            if (h == 0) {
                const float gam = sqrtf(g2 + s_g2[row]) * (inv_sd * (1.f / 256.f));
                *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * o) = __halves2half2(__float2half_rn(nrm), __float2half_rn(gam));
            }
        }
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 512);
}

// ---------------------------------------------------------------- K at d = 128, two threads per row
// As encode128_rows_kernel for K, with each row split over two threads (halves h = 0, 1), so that
// a thread holds 64 coordinates and an SM runs 16 warps:
//  * the transform's stage on index bit 6 is taken first, on the input: half h holds
//    u_m = (D x)_m + (-1)^h (D x)_{m+64} (m < 64) and finishes the 64-point transform in
//    registers; its outputs are coordinates 64 h + m (the stages of the transform commute);
//  * each half reads the whole row (that first stage needs it; the sums of squares of the two
//    halves' outputs add to twice the squared norm);
//  * the record words of coordinates 64 h .. 64 h + 63 (words 2h, 2h + 1 of each tig, cells and QJL
//    sign bits: accumulator columns 64 h .. 64 h + 63) belong to half h, which stores them; half 1
//    leaves its residual sum in shared memory for half 0, which stores the norms.
// Two tile groups of 256 threads take alternate tiles of 128 rows.  From bf16 the tile arrives as
// two TMA tensor boxes, the signs D are an XOR of the input words and the transform runs on f32x2
// pairs (u_m, u_{m+32}): the stage on index bit 5 inside each pair, the five others between pairs.
namespace encs {
constexpr int D = 128, kRows = 128, kTg = 2, kThreads = 256 * kTg;
template <typename T> __host__ __device__ constexpr int nx() { return sizeof(T) == 2 ? 2 : 1; }
template <typename T> __host__ __device__ constexpr int row_bytes() { return D * (int)sizeof(T); }
template <typename T> __host__ __device__ constexpr int row_stride() { return row_bytes<T>() + 16; }
// bf16 tiles arrive as two TMA boxes (128 rows x 128 bytes, 128-byte swizzle); fp32 rows by one
// bulk copy each into a padded row stride
template <typename T> __host__ __device__ constexpr bool tma() { return sizeof(T) == 2; }
template <typename T> __host__ __device__ constexpr int xbuf_bytes() { return tma<T>() ? 2 * kRows * 128 : kRows * row_stride<T>(); }
constexpr int oX = 32768;   // after S (f16)
template <typename T> __host__ __device__ constexpr int oW() { return oX + kTg * nx<T>() * xbuf_bytes<T>(); }
constexpr int kWStride = 15;   // per row: 12 partial plane words, the residual sum of squares, two norm shares
template <typename T> __host__ __device__ constexpr int smem_bytes() { return oW<T>() + kTg * kRows * kWStride * 4; }
}  // namespace encs

template <typename T>
__global__ void __launch_bounds__(encs::kThreads, 1)
encode128k_split_kernel(const __grid_constant__ CUtensorMap tmap, const uint8_t *__restrict__ params,
                        const T *__restrict__ x, int64_t n_vec, SlotMap map, uint8_t *__restrict__ pool,
                        int32_t *status) {
    using namespace encs;
    constexpr bool TM = tma<T>();
    constexpr int NX = nx<T>(), RS = row_stride<T>(), RB = row_bytes<T>(), EPC = 16 / (int)sizeof(T);
    constexpr int HC = RB / 32;   // 16-byte chunks per half row
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t xfull[kTg][2], mmabar[kTg];
    __shared__ uint32_t tmem_base;
    __shared__ float s_Dh[2][2][64];   // half h: D_m and (-1)^h D_{m+64}, m < 64
    __shared__ __align__(16) uint32_t s_sg[D / 2];   // XOR masks of the bf16 pairs (bit 15 / 31: D_2p / D_2p+1 < 0)
    const ParamsHeader *ph = reinterpret_cast<const ParamsHeader *>(params);
    if (ph->magic != kParamsMagic || ph->d != D) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_status(status, TQ_STATUS_BAD_PARAMS);
        return;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tg = (warp >> 2) & 1, h = warp >> 3, sl = warp & 3, row = 32 * sl + lane;
    const int64_t ntiles = (n_vec + kRows - 1) / kRows;
    if ((int64_t)blockIdx.x >= ntiles) return;
    if (tid == 0) {
        for (int i = 0; i < kTg; ++i) {
            tc::mbar_init(&xfull[i][0], 1);
            tc::mbar_init(&xfull[i][1], 1);
            tc::mbar_init(&mmabar[i], 1);
        }
    }
    if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
    if (tid < 2 * D) {
        const float *Dp = reinterpret_cast<const float *>(params + params_off_D(D));
        const int hh = tid >> 7, k = (tid >> 6) & 1, m = tid & 63;
        s_Dh[hh][k][m] = (k && hh) ? -Dp[64 + m] : Dp[64 * k + m];
        if (tid < D / 2) s_sg[tid] = (Dp[2 * tid] < 0.f ? 0x8000u : 0u) | (Dp[2 * tid + 1] < 0.f ? 0x80000000u : 0u);
    }
    {   // B row n = S row k_col_coord(n)
        const float *S = reinterpret_cast<const float *>(params + params_off_S(D));
        for (int e = tid; e < D * D; e += kThreads) {
            const int n = e >> 7, k = e & 127;
            const int sr = k_col_coord(n);
            // S is held at binary16 precision: one exact f16 operand
            *reinterpret_cast<__half *>(smem + tc::sw128_off(n, k, D)) = __float2half_rn(__ldg(S + sr * D + k));
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = tmem_base + 256u * tg;
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * sl) << 16);
    // thresholds x 256 (exact), and x 256 the half-widths of the cell pairs around the even-index
    // thresholds: cells 2k and 2k + 1 are t_2k -/+ hw_k; the codebook is symmetric, so pairs 0 and 3
    // (the outer ones) share hw_out and pairs 1 and 2 share hw_in
    const float T0 = 256.f * ph->threshold[0], T1 = 256.f * ph->threshold[1], T2 = 256.f * ph->threshold[2];
    const float T3 = 256.f * ph->threshold[3], T4 = 256.f * ph->threshold[4], T5 = 256.f * ph->threshold[5];
    const float T6 = 256.f * ph->threshold[6];
    const float hw_out = 128.f * (ph->centroid[7] - ph->centroid[6]), hw_in = 128.f * (ph->centroid[5] - ph->centroid[4]);
    const float inv_sd = rsqrtf((float)D);
    const bool small = n_vec <= (int64_t)0x7fffffff;
    uint32_t *sW = reinterpret_cast<uint32_t *>(smem + oW<T>()) + ((size_t)tg * kRows + row) * kWStride;
    bool timed_out = false;
    const int bar_id = 1 + tg;
    const bool issuer = warp == 4 * tg;   // the tile group's first warp moves its rows

    auto tile_of = [&](int i) { return (int64_t)blockIdx.x + (int64_t)(kTg * i + tg) * gridDim.x; };
    auto issue = [&](int i, int buf) {   // the issuing warp: the two boxes, or one bulk copy per row
        const int64_t v0 = tile_of(i) * kRows;
        uint8_t *dst = smem + oX + (tg * NX + buf) * xbuf_bytes<T>();
        if constexpr (TM) {
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(&xfull[tg][buf], (uint32_t)xbuf_bytes<T>());
                tc::tma_load_2d(dst, &tmap, 0, (int)v0, &xfull[tg][buf]);
                tc::tma_load_2d(dst + kRows * 128, &tmap, 64, (int)v0, &xfull[tg][buf]);
            }
        } else {
            const int rows = (int)min((int64_t)kRows, n_vec - v0);
            if (lane == 0) tc::mbar_arrive_expect_tx(&xfull[tg][buf], (uint32_t)rows * RB);
            __syncwarp();
            for (int r = lane; r < rows; r += 32) tc::bulk_g2s(dst + r * RS, x + (v0 + r) * D, RB, &xfull[tg][buf]);
        }
    };
    if (issuer)
        for (int b2 = 0; b2 < NX; ++b2)
            if (tile_of(b2) < ntiles) issue(b2, b2);

#pragma unroll 1
    for (int i = 0; tile_of(i) < ntiles; ++i) {
        const int buf = i % NX, use = i / NX;
        const int64_t v0 = tile_of(i) * kRows, v = v0 + row;
        // token and head of row v (32-bit division when the rows fit, as they do in practice)
        const int64_t tok = small ? (int64_t)((uint32_t)v / (uint32_t)map.n_heads) : v / map.n_heads;
        const int head = (int)(v - tok * map.n_heads);
        const int64_t sraw = v < n_vec ? map.slot_raw(tok) : -1;   // checked at the stores
        if (!tc::mbar_wait(&xfull[tg][buf], use & 1)) timed_out = true;
        // ---- 1. the whole row: norm, signs D, and the transform stage on index bit 6
        float u[64];
        float ss = 0.f;
        if constexpr (TM) {
            // pairs P[k] = (u_k, u_{k+32}) of this half; box 0 word p holds x_2p, x_2p+1 and box 1 word p
            // holds x_64+2p, x_65+2p
            const uint8_t *xb = smem + oX + (tg * NX + buf) * xbuf_bytes<T>() + row * 128;
            uint32_t wa[32], wb[32];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 ua = *reinterpret_cast<const uint4 *>(xb + ((c ^ (row & 7)) << 4));
                const uint4 ub = *reinterpret_cast<const uint4 *>(xb + kRows * 128 + ((c ^ (row & 7)) << 4));
                const uint4 ma = reinterpret_cast<const uint4 *>(s_sg)[c], mb = reinterpret_cast<const uint4 *>(s_sg)[c + 8];
                wa[4 * c] = ua.x ^ ma.x; wa[4 * c + 1] = ua.y ^ ma.y; wa[4 * c + 2] = ua.z ^ ma.z; wa[4 * c + 3] = ua.w ^ ma.w;
                wb[4 * c] = ub.x ^ mb.x; wb[4 * c + 1] = ub.y ^ mb.y; wb[4 * c + 2] = ub.z ^ mb.z; wb[4 * c + 3] = ub.w ^ mb.w;
            }
            const float2 sgn = make_float2(h ? -1.f : 1.f, h ? -1.f : 1.f);
            float2 P[32];
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 32; ++k) {   // u_k = x_k +- x_{k+64}, u_{k+32} = x_{k+32} +- x_{k+96}
                const uint32_t a0 = wa[k >> 1], a1 = wa[16 + (k >> 1)], b0 = wb[k >> 1], b1 = wb[16 + (k >> 1)];
                const float2 av = (k & 1) ? make_float2(__uint_as_float(a0 & 0xFFFF0000u), __uint_as_float(a1 & 0xFFFF0000u))
                                          : make_float2(__uint_as_float(a0 << 16), __uint_as_float(a1 << 16));
                const float2 bv = (k & 1) ? make_float2(__uint_as_float(b0 & 0xFFFF0000u), __uint_as_float(b1 & 0xFFFF0000u))
                                          : make_float2(__uint_as_float(b0 << 16), __uint_as_float(b1 << 16));
                P[k] = __ffma2_rn(bv, sgn, av);
                acc = __ffma2_rn(P[k], P[k], acc);   // the halves' sums add to 2 |x|^2
            }
            ss = acc.x + acc.y;
            // the 64-point transform of this half: index bit 5 inside the pairs, bits 0..4 between them
#pragma unroll
            for (int k = 0; k < 32; ++k) P[k] = make_float2(P[k].x + P[k].y, P[k].x - P[k].y);
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int st = 1; st < 32; st <<= 1)
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if ((k & st) == 0) {
                        const float2 a = P[k], b = P[k | st];
                        P[k] = __fadd2_rn(a, b);
                        P[k | st] = __ffma2_rn(b, m1, a);   // a - b
                    }
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                u[k] = P[k].x;
                u[k + 32] = P[k].y;
            }
        } else {
            const uint8_t *xr = smem + oX + (tg * NX + buf) * xbuf_bytes<T>() + row * RS;
#pragma unroll
            for (int c = 0; c < HC; ++c) {
                const uint4 ua = *reinterpret_cast<const uint4 *>(xr + 16 * c);
                const uint4 ub = *reinterpret_cast<const uint4 *>(xr + 16 * (c + HC));
                float a[EPC], b[EPC];
                if constexpr (sizeof(T) == 2) {
                    const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        a[2 * q] = __uint_as_float(wa[q] << 16);
                        a[2 * q + 1] = __uint_as_float(wa[q] & 0xFFFF0000u);
                        b[2 * q] = __uint_as_float(wb[q] << 16);
                        b[2 * q + 1] = __uint_as_float(wb[q] & 0xFFFF0000u);
                    }
                } else {
                    a[0] = __uint_as_float(ua.x); a[1] = __uint_as_float(ua.y);
                    a[2] = __uint_as_float(ua.z); a[3] = __uint_as_float(ua.w);
                    b[0] = __uint_as_float(ub.x); b[1] = __uint_as_float(ub.y);
                    b[2] = __uint_as_float(ub.z); b[3] = __uint_as_float(ub.w);
                }
#pragma unroll
                for (int e = 0; e < EPC; ++e) {
                    const int m = EPC * c + e;
                    u[m] = fmaf(b[e], s_Dh[h][1][m], a[e] * s_Dh[h][0][m]);
                    ss = fmaf(u[m], u[m], ss);   // the halves' sums add to 2 |x|^2
                }
            }
        }
        float *sSS = reinterpret_cast<float *>(sW) + 13;   // the halves' norm shares (words 13, 14)
        sSS[1 - h] = ss;
        tc::named_sync(bar_id, 256);   // every row is read: the buffer takes the tile NX ahead
        if (issuer && tile_of(i + NX) < ntiles) issue(i + NX, buf);
        const float nrm = sqrtf(0.5f * (ss + sSS[h]));   // the same sum in both halves (addition commutes)
        // ---- 2. the 64-point transform of this half (index bits 0..5; done above from bf16)
        if constexpr (!TM) {
#pragma unroll
            for (int st = 1; st < 64; st <<= 1)
#pragma unroll
                for (int m = 0; m < 64; ++m)
                    if ((m & st) == 0) {
                        const float a0 = u[m], a1 = u[m | st];
                        u[m] = a0 + a1;
                        u[m | st] = a0 - a1;
                    }
        }
        // 256 / n (exact scaling of 1 / n): Z = 256 z, and the residual comes out x 256, which keeps
        // its f16 low parts out of the subnormals
        const float rs = nrm > 0.f ? 256.f / nrm : 0.f;
        // ---- 3. cells of coordinates 64 h + m, residual.  The search compares Z with 256 t_j, the
        // same decisions as z against t_j (ties go up); the last comparison's difference Z - 256 t_2k
        // gives the residual: Z - 256 c = (Z - 256 t_2k) -/+ 256 hw_k.
        // the words of this half: coordinates 64 h + m are words 2 h, 2 h + 1 of each tig
        uint32_t kwd[4][2] = {{0u, 0u}, {0u, 0u}, {0u, 0u}, {0u, 0u}};
        float g2 = 0.f;   // sum of squares of the residual x 256
#pragma unroll
        for (int m = 0; m < 64; ++m) {
            const float Z = u[m] * rs;
            const bool b2 = Z >= T3;
            const bool b1 = Z >= (b2 ? T5 : T1);
            const float dz = Z - (b2 ? (b1 ? T6 : T4) : (b1 ? T2 : T0));
            const bool b0 = dz >= 0.f;
            kwd[k_tig(m)][k_word(m)] |= ((uint32_t)b0 | ((uint32_t)b1 << 1) | ((uint32_t)b2 << 2)) << (4 * k_field(m));
            const float hw = (b1 == b2) ? hw_out : hw_in;
            const float rho = b0 ? dz - hw : dz + hw;
            g2 = fmaf(rho, rho, g2);
            u[m] = rho;
        }
        // ---- 4. rho (x 256) as f16 hi / lo into this row's lane: K elements 64 h .. 64 h + 63
#pragma unroll
        for (int q = 0; q < 2; ++q) {   // 16 columns at a time (fewer live registers)
            float hw[16], lw[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float a0 = u[32 * q + 2 * c], a1 = u[32 * q + 2 * c + 1];
                const __half2 hh = __floats2half2_rn(a0, a1);
                const float2 hf = __half22float2(hh);
                const __half2 ll = __floats2half2_rn(a0 - hf.x, a1 - hf.y);
                hw[c] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&hh));
                lw[c] = __uint_as_float(*reinterpret_cast<const uint32_t *>(&ll));
            }
            tc::st16(lane_addr + 32 * h + 16 * q, hw);
            tc::st16(lane_addr + 64 + 32 * h + 16 * q, lw);
        }
        if (h == 1) sW[12] = __float_as_uint(g2);   // half 1's residual sum, for half 0
        tc::wait_st();
        tc::fence_before_sync();
        tc::named_sync(bar_id, 256);
        tc::fence_after_sync();
        if (issuer && lane == 0) {
            const uint32_t bh = tc::smem_u32(smem);
            constexpr uint32_t id = tc::idesc_f16(kRows, D);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_ts_f16(tmem + 128, tmem + 8 * ks, tc::sw128_desc(bh, ks, D), id, ks > 0);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                tc::mma_ts_f16(tmem + 128, tmem + 64 + 8 * ks, tc::sw128_desc(bh, ks, D), id, true);
            // S is held at binary16 precision (exact in f16): S rho_hi + S rho_lo is the product
            tc::mma_commit(&mmabar[tg]);
        }
        if (!tc::mbar_wait(&mmabar[tg], i & 1)) timed_out = true;
        tc::fence_after_sync();
        // ---- 5. QJL sign bits of this half: accumulator columns 64 h + 16 j + b are field b & 7 of
        // word (tig j, 2 h + (b >> 3)); bit 3 of the field is set when the projection is >= 0 (its
        // fp32 sign bit clear; only an exact zero, a tie, could read as -0)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float pv[16];
            tc::ld16(lane_addr + 128 + 64 * h + 16 * j, pv);
            tc::wait_ld();
#pragma unroll
            for (int b = 0; b < 16; ++b) asm volatile("" : "+f"(pv[b]));   // no use moves above the wait
#pragma unroll
            for (int b = 0; b < 16; ++b)
                kwd[j][b >> 3] |= ((~__float_as_uint(pv[b]) >> 31) << 3) << (4 * (b & 7));
        }
        tc::fence_before_sync();
        // ---- 6. the record words of this row's slot
        const int64_t slot = map.slot_check(sraw, status, v < n_vec && h == 0 && head == 0);
        if (slot >= 0) {
            const int64_t blk = slot / kBlock;
            const int o = (int)(slot % kBlock);
            uint8_t *rec = pool + ((size_t)blk * map.n_heads + head) * k_record(D);
            const int gid = o & 7, th = o >> 3;
#pragma unroll
            for (int tig = 0; tig < 4; ++tig)   // words 2 h, 2 h + 1 of word row (4 gid + tig) * 2 + th
                reinterpret_cast<uint2 *>(rec)[((4 * gid + tig) * 2 + th) * 2 + h] = make_uint2(kwd[tig][0], kwd[tig][1]);
            if (h == 0) {
                const float gam = sqrtf(g2 + __uint_as_float(sW[12])) * (inv_sd * (1.f / 256.f));
                *reinterpret_cast<__half2 *>(rec + 8 * D + 4 * o) = __halves2half2(__float2half_rn(nrm), __float2half_rn(gam));
            }
        }
        tc::named_sync(bar_id, 256);   // the accumulator, the A lanes and the merge area are free
    }
    if (timed_out) flag_status(status, TQ_STATUS_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 512);
}

template <typename T>
cudaError_t launch_encs(const void *params, const void *x, int64_t n_vec, const SlotMap &map, void *pool,
                        int32_t *status, cudaStream_t st) {
    const int64_t ntiles = (n_vec + encs::kRows - 1) / encs::kRows;
    if (ntiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = encs::smem_bytes<T>();
    auto kern = encode128k_split_kernel<T>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    CUtensorMap tm;   // the bf16 input's map (unused from fp32)
    memset(&tm, 0, sizeof tm);
    if (encs::tma<T>() && (n_vec > (int64_t)0x7fffffff - encs::kRows || !make_tmap_2d(&tm, x, 2, (unsigned long long)n_vec, encs::D, encs::kRows)))
        return cudaErrorNotSupported;
    const unsigned grid = (unsigned)(ntiles < sms ? ntiles : sms);
    kern<<<grid, encs::kThreads, smem, st>>>(tm, (const uint8_t *)params, (const T *)x, n_vec, map, (uint8_t *)pool, status);
    return cudaGetLastError();
}

// The bf16 V encode through TMA; false in *used when the input cannot be mapped (rows past
// 2^31 - 128, or the driver's tensor-map encoder missing), for the caller to fall back.
cudaError_t launch_encv_tma(const void *params, const void *x, int64_t n_vec, const SlotMap &map, void *pool,
                            int32_t *status, cudaStream_t st, bool *used) {
    *used = false;
    const int64_t ntiles = (n_vec + encv::kRows - 1) / encv::kRows;
    if (ntiles <= 0) {
        *used = true;
        return cudaSuccess;
    }
    if (n_vec > (int64_t)0x7fffffff - encv::kRows) return cudaSuccess;
    CUtensorMap tm;
    if (!make_tmap_2d(&tm, x, 2, (unsigned long long)n_vec, encv::D, encv::kRows)) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = encv::smem_bytes();
    e = cudaFuncSetAttribute(encode128v_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t want = (int64_t)sms * encv::kCtasPerSm;
    const unsigned grid = (unsigned)(ntiles < want ? ntiles : want);
    const int H = map.n_heads;
    const int whole_ok = (H == 1 || H == 2 || H == 4 || H == 8) ? 1 : 0;
    encode128v_tma_kernel<<<grid, encv::kThreads, smem, st>>>(tm, (const uint8_t *)params, n_vec, map, whole_ok,
                                                              (uint8_t *)pool, status);
    *used = true;
    return cudaGetLastError();
}

// The bf16 V encode at d = 256 through TMA (as launch_encv_tma).
cudaError_t launch_encv256_tma(const void *params, const void *x, int64_t n_vec, const SlotMap &map, void *pool,
                               int32_t *status, cudaStream_t st, bool *used) {
    *used = false;
    const int64_t ntiles = (n_vec + encv2::kRows - 1) / encv2::kRows;
    if (ntiles <= 0) {
        *used = true;
        return cudaSuccess;
    }
    if (n_vec > (int64_t)0x7fffffff - encv2::kRows) return cudaSuccess;
    CUtensorMap tm;
    if (!make_tmap_2d(&tm, x, 2, (unsigned long long)n_vec, encv2::D, encv2::kRows)) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = encv2::smem_bytes();
    e = cudaFuncSetAttribute(encode256v_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t want = (int64_t)sms * encv2::kCtasPerSm;
    const unsigned grid = (unsigned)(ntiles < want ? ntiles : want);
    const int H = map.n_heads;
    const int whole_ok = (H == 1 || H == 2 || H == 4 || H == 8) ? 1 : 0;
    encode256v_tma_kernel<<<grid, encv2::kThreads, smem, st>>>(tm, (const uint8_t *)params, n_vec, map, whole_ok,
                                                               (uint8_t *)pool, status);
    *used = true;
    return cudaGetLastError();
}

// The bf16 K encode at d = 256 on tcgen05 (as launch_encv_tma).
cudaError_t launch_enck256_tc(const void *params, const void *x, int64_t n_vec, const SlotMap &map, void *pool,
                              int32_t *status, cudaStream_t st, bool *used) {
    *used = false;
    const int64_t ntiles = (n_vec + enck2::kRows - 1) / enck2::kRows;
    if (ntiles <= 0) {
        *used = true;
        return cudaSuccess;
    }
    if (n_vec > (int64_t)0x7fffffff - enck2::kRows) return cudaSuccess;
    CUtensorMap tm;
    if (!make_tmap_2d(&tm, x, 2, (unsigned long long)n_vec, enck2::D, enck2::kRows)) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = enck2::smem_bytes();
    e = cudaFuncSetAttribute(encode256k_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(ntiles < sms ? ntiles : sms);
    encode256k_tc_kernel<<<grid, enck2::kThreads, smem, st>>>(tm, (const uint8_t *)params, n_vec, map, (uint8_t *)pool,
                                                              status);
    *used = true;
    return cudaGetLastError();
}

template <typename T, bool IS_K>
cudaError_t launch_encr(const void *params, const void *x, int64_t n_vec, const SlotMap &map, void *pool,
                        int32_t *status, cudaStream_t st) {
    const int64_t ntiles = (n_vec + encr::kRows - 1) / encr::kRows;
    if (ntiles <= 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    constexpr int smem = encr::smem_bytes<T, IS_K>();
    auto kern = encode128_rows_kernel<T, IS_K>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t want = (int64_t)sms * encr::ctas_per_sm<IS_K>();
    const unsigned grid = (unsigned)(ntiles < want ? ntiles : want);
    kern<<<grid, encr::n_threads<IS_K>(), smem, st>>>((const uint8_t *)params, (const T *)x, n_vec, map,
                                                      (uint8_t *)pool, status);
    return cudaGetLastError();
}

template <int D, int TILE, typename T>
cudaError_t launch_enc(const void *params, const void *xk, const void *xv, int64_t n_vec, const SlotMap &map,
                       void *kp, void *vp, int kinds, int32_t *status, cudaStream_t st) {
    const int64_t ntiles = (n_vec + TILE - 1) / TILE;
    if (ntiles <= 0) return cudaSuccess;
    const int ny = (kinds == 3) ? 2 : 1;
    const int64_t cap = 152 * 2;               // persistent: two CTAs per SM
    const unsigned gx = (unsigned)(ntiles < cap ? ntiles : cap);
    constexpr size_t smem = EncSmem<D, TILE>::kBytes;
    auto kern = encode_kernel<D, TILE, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(gx, ny), kEncWarps * 32, smem, st>>>((const uint8_t *)params, (const T *)xk, (const T *)xv, n_vec, map,
                                                  (uint8_t *)kp, (uint8_t *)vp, kinds, status);
    return cudaGetLastError();
}

template <int TILE>
cudaError_t launch_any(int d, int dtype, const void *params, const void *xk, const void *xv, int64_t n_vec,
                       const SlotMap &map, void *kp, void *vp, int kinds, int32_t *status, cudaStream_t st) {
    if (d == 128)
        return dtype == TQ_DTYPE_BF16
                   ? launch_enc<128, TILE, __nv_bfloat16>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st)
                   : launch_enc<128, TILE, float>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st);
    return dtype == TQ_DTYPE_BF16
               ? launch_enc<256, TILE, __nv_bfloat16>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st)
               : launch_enc<256, TILE, float>(params, xk, xv, n_vec, map, kp, vp, kinds, status, st);
}

}  // namespace

// Self-test of the bounded device waits: one CTA waits on an mbarrier that nothing arrives at,
// with the same bounded wait the encode and dequant kernels use; the wait gives up after its
// limit and the CTA reports TQ_STATUS_TIMEOUT, leaving the context usable.
namespace {
__global__ void wait_timeout_selftest_kernel(int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) tc::mbar_init(&bar, 1);
    __syncthreads();
    const bool done = tc::mbar_wait(&bar, 0);   // phase 0 never completes
    if (!done && threadIdx.x == 0) flag_status(status, TQ_STATUS_TIMEOUT);
}
}  // namespace

cudaError_t launch_wait_timeout_selftest(int32_t *status, cudaStream_t st) {
    wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(status);
    return cudaGetLastError();
}

cudaError_t launch_encode(bool is_k, int d, int dtype, const void *params, const void *x, int64_t n_tokens,
                          int n_heads, const int64_t *slots, void *pool, int64_t num_blocks, int32_t *status,
                          cudaStream_t st) {
    SlotMap map{slots, nullptr, nullptr, 0, num_blocks, n_heads};
    if (d == 128 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0) {
        const int64_t nv = n_tokens * n_heads;
        if (is_k && TQ_ENC_SPLIT)
        {
            if (dtype != TQ_DTYPE_BF16) return launch_encs<float>(params, x, nv, map, pool, status, st);
            // a bf16 input the tensor map cannot describe takes the thread-per-row kernel
            const cudaError_t e = launch_encs<__nv_bfloat16>(params, x, nv, map, pool, status, st);
            if (e != cudaErrorNotSupported) return e;
            return launch_encr<__nv_bfloat16, true>(params, x, nv, map, pool, status, st);
        }
        if (dtype == TQ_DTYPE_BF16 && !is_k && TQ_ENC_V_TMA) {
            bool used = false;
            const cudaError_t e = launch_encv_tma(params, x, nv, map, pool, status, st, &used);
            if (used || e != cudaSuccess) return e;
        }
        if (dtype == TQ_DTYPE_BF16)
            return is_k ? launch_encr<__nv_bfloat16, true>(params, x, nv, map, pool, status, st)
                        : launch_encr<__nv_bfloat16, false>(params, x, nv, map, pool, status, st);
        return is_k ? launch_encr<float, true>(params, x, nv, map, pool, status, st)
                    : launch_encr<float, false>(params, x, nv, map, pool, status, st);
    }
    if (d == 256 && dtype == TQ_DTYPE_BF16 && (reinterpret_cast<uintptr_t>(x) & 15u) == 0 && TQ_ENC_V_TMA) {
        bool used = false;
        const cudaError_t e = is_k ? launch_enck256_tc(params, x, n_tokens * n_heads, map, pool, status, st, &used)
                                   : launch_encv256_tma(params, x, n_tokens * n_heads, map, pool, status, st, &used);
        if (used || e != cudaSuccess) return e;
    }
    return launch_any<16>(d, dtype, params, is_k ? x : nullptr, is_k ? nullptr : x, n_tokens * n_heads, map,
                          is_k ? pool : nullptr, is_k ? nullptr : pool, is_k ? 1 : 2, status, st);
}

}  // namespace tq
