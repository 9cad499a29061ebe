/*
 * tq_oracle.c -- plain, slow fp64 CPU restatement of TurboQuant KV-cache
 * compression and of decode attention over the compressed, paged cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Tests compare the CUDA library in
 * turboquant_compressed_kv_gb300/csrc against this file.  It shares no code,
 * header, table or constant with that library; only tests, the smoke check
 * and the benchmark's CPU-baseline leg may load it.  No product code path
 * calls it.
 *
 * Sources (cited by page title and section; the pages print prose only):
 *  [README]  "SwiftLM" (nomorevibe.com/p/swiftlm), section
 *            "TurboQuantization: KV Cache Compression" -> "The Algorithm",
 *            K-Cache steps 1-5 and the V-Cache paragraph.
 *  [ART]     "SwiftLM ... Swift製LLM推論サーバー" (lilting.ch), sections
 *            "Lloyd-Maxコードブックとは", "KVキャッシュ圧縮の内訳",
 *            "Walsh-Hadamard Transform（WHT）の役割".
 *  [VLLM]    "論文解説: vLLM-MLX" (0h-n0.github.io), section "Paged KVキャッシュ".
 *
 * Where the pages leave a step open, this file takes these readings:
 *  - rotation Pi = (1/sqrt d) H diag(D), Sylvester H, D applied first;
 *  - codebook: 8-level Lloyd-Max for N(0,1); coordinates are compared as
 *    z = sqrt(d) * y (the pages' N(0,1/d) scaled to unit variance);
 *  - residual r = y - c[code]/sqrt(d) on the unit vector, rotated domain;
 *  - QJL: m = d Gaussian rows S, bit = [ (S r)_k >= 0 ], estimator scale
 *    sqrt(pi/2)/d times gamma = ||r||;
 *  - stored norms are IEEE binary16, round-to-nearest-even;
 *  - a code is decided in fp32 (the precision of the GPU kernels): the fp64
 *    coordinate is rounded to fp32 and compared with the fp32-rounded
 *    thresholds; ties go to the upper cell.
 *
 * Parity pins live in tests/test_oracle_pins.py.  The packed bit layout
 * (tqo_k_bitpos / tqo_v_bitpos) is a convention of this library and is
 * parity unpinned except by agreement with the CUDA path (and by the
 * bijection and round-trip pins).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define TQO_BLOCK 16

/* ------------------------------------------------------------------ */
/* IEEE binary16 conversion, written out from the format definition.  */
/* ------------------------------------------------------------------ */

/* Round a double to the nearest binary16 (ties to even).  Values whose
 * magnitude rounds above 65504 become +-inf; NaN maps to a quiet NaN. */
uint16_t tqo_fp16_rne(double x)
{
    uint16_t sign = 0;
    if (isnan(x)) return 0x7e00;
    if (signbit(x)) { sign = 0x8000; x = -x; }
    if (x == 0.0) return sign;
    /* binary16: subnormal spacing 2^-24, normal exponents -14..15 */
    int e;
    frexp(x, &e);               /* x = f * 2^e, f in [0.5,1) -> unbiased exp of x is e-1 */
    int ex = e - 1;
    if (ex < -14) ex = -14;     /* subnormal range shares the spacing of 2^-14 */
    double ulp = ldexp(1.0, ex - 10);
    double q = x / ulp;          /* exact: ulp is a power of two */
    double fl = floor(q);
    double rem = q - fl;
    double m = fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) m = fl + 1.0;
    double r = m * ulp;
    if (r > 65504.0) return (uint16_t)(sign | 0x7c00);
    /* encode r */
    if (r < ldexp(1.0, -14)) {               /* subnormal */
        return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
    }
    int er;
    double fr = frexp(r, &er);                /* r = fr * 2^er */
    int E = er - 1 + 15;
    uint16_t mant = (uint16_t)((fr * 2.0 - 1.0) * 1024.0);
    return (uint16_t)(sign | (E << 10) | mant);
}

double tqo_fp16_value(uint16_t h)
{
    int s = h >> 15, E = (h >> 10) & 31, m = h & 1023;
    double v;
    if (E == 31) v = m ? NAN : INFINITY;
    else if (E == 0) v = ldexp((double)m, -24);
    else v = ldexp(1.0 + m / 1024.0, E - 15);
    return s ? -v : v;
}

/* ------------------------------------------------------------------ */
/* Codebook: Lloyd-Max for N(0,1), 8 levels  [ART "Lloyd-Maxコードブックとは"] */
/* ------------------------------------------------------------------ */

static double phi(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
static double Phi(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

/* Alternate the two Lloyd-Max conditions until the centroids stop moving:
 *   thresholds are midpoints of neighbouring centroids;
 *   each centroid is the conditional mean of N(0,1) on its cell,
 *   E[X | a<X<b] = (phi(a)-phi(b)) / (Phi(b)-Phi(a)).
 * N(0,1) is symmetric and log-concave, so the 8-level optimum is unique and
 * symmetric: the middle threshold is exactly 0 and c[7-j] = -c[j].  The
 * iteration is therefore run on the four positive cells (0,t4),(t4,t5),
 * (t5,t6),(t6,inf) and mirrored, which keeps t[3] == 0 exactly.
 * MSE = 1 - sum_j c_j (phi(t_{j-1}) - phi(t_j))  (E[X^2]=1 minus E[Q(X)^2]).
 * Returns the iteration count (or -1 if it did not converge). */
int tqo_lloyd_max8(double c[8], double t[7], double *mse)
{
    double cp[4] = {0.25, 0.75, 1.25, 1.75};   /* any ordered positive start */
    double tp[5];                              /* cell edges 0, t4, t5, t6, +inf */
    int it;
    for (it = 1; it <= 200000; it++) {
        tp[0] = 0.0;
        for (int j = 1; j < 4; j++) tp[j] = 0.5 * (cp[j - 1] + cp[j]);
        double delta = 0.0;
        for (int j = 0; j < 4; j++) {
            double a = tp[j];
            double pa = phi(a), pb = (j == 3) ? 0.0 : phi(tp[j + 1]);
            /* Phi(b)-Phi(a) = (erfc(a/sqrt2) - erfc(b/sqrt2))/2, accurate in the tail */
            double mass = 0.5 * (erfc(a / sqrt(2.0)) - ((j == 3) ? 0.0 : erfc(tp[j + 1] / sqrt(2.0))));
            double cn = (pa - pb) / mass;
            double dd = fabs(cn - cp[j]);
            if (dd > delta) delta = dd;
            cp[j] = cn;
        }
        if (delta < 1e-15) break;
    }
    for (int j = 0; j < 4; j++) { c[4 + j] = cp[j]; c[3 - j] = -cp[j]; }
    t[3] = 0.0;
    for (int j = 0; j < 3; j++) { t[4 + j] = 0.5 * (cp[j] + cp[j + 1]); t[2 - j] = -t[4 + j]; }
    double s = 0.0;
    for (int j = 0; j < 8; j++) {
        double pa = (j == 0) ? 0.0 : phi(t[j - 1]);
        double pb = (j == 7) ? 0.0 : phi(t[j]);
        s += c[j] * (pa - pb);
    }
    if (mse) *mse = 1.0 - s;
    return it > 200000 ? -1 : it;
}

/* ------------------------------------------------------------------ */
/* Randomized Walsh-Hadamard rotation, dense definition               */
/* [README step 2; ART "Walsh-Hadamard Transform（WHT）の役割"]           */
/* ------------------------------------------------------------------ */

/* Sylvester Hadamard entry H_ij = (-1)^popcount(i & j). */
int tqo_hadamard_entry(int i, int j) { return (__builtin_popcount((unsigned)(i & j)) & 1) ? -1 : 1; }

/* y = Pi x = (1/sqrt d) H diag(D) x, by the dense O(d^2) sum. */
void tqo_rotate(int d, const int8_t *D, const double *x, double *y)
{
    double s = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; i++) {
        double acc = 0.0;
        for (int j = 0; j < d; j++) acc += tqo_hadamard_entry(i, j) * D[j] * x[j];
        y[i] = acc * s;
    }
}

/* x = Pi^T y = diag(D) H y / sqrt d  (H is symmetric). */
void tqo_rotate_t(int d, const int8_t *D, const double *y, double *x)
{
    double s = 1.0 / sqrt((double)d);
    for (int j = 0; j < d; j++) {
        double acc = 0.0;
        for (int i = 0; i < d; i++) acc += tqo_hadamard_entry(j, i) * y[i];
        x[j] = D[j] * acc * s;
    }
}

/* ------------------------------------------------------------------ */
/* Encode one vector  [README K-Cache steps 1-5 / V-Cache; ART KV内訳]  */
/* ------------------------------------------------------------------ */

/* Encodes x (length d, fp64).  Outputs (unpacked):
 *   codes[d]   3-bit cell index of every rotated coordinate,
 *   signs[d]   (K only) QJL sign bits, 1 where (S r)_k >= 0,
 *   *n         ||x||, *gamma ||r|| (K only),
 *   z[d]       (optional) sqrt(d) * (Pi x/||x||), the value compared with the thresholds,
 *   p[d]       (optional, K only) S r.
 * If codes_in is non-null the cells are taken from it instead of being
 * decided here ("QJL given codes"), so sign bits can be compared even where
 * a coordinate sat on a threshold. */
void tqo_encode_vector(int is_k, int d, const int8_t *D, const float *S,
                       const double c[8], const double t[7], const double *x,
                       const uint8_t *codes_in, uint8_t *codes, uint8_t *signs,
                       double *n_out, double *gamma_out, double *z, double *p)
{
    double *xh = (double *)malloc(sizeof(double) * d);
    double *y = (double *)malloc(sizeof(double) * d);
    double *r = (double *)malloc(sizeof(double) * d);
    double sd = sqrt((double)d);

    /* step 1: L2 norm and normalisation (a zero vector stays zero) */
    double nn = 0.0;
    for (int i = 0; i < d; i++) nn += x[i] * x[i];
    double n = sqrt(nn);
    for (int i = 0; i < d; i++) xh[i] = (n > 0.0) ? x[i] / n : 0.0;

    /* step 2: rotation */
    tqo_rotate(d, D, xh, y);

    /* step 3: 3-bit Lloyd-Max cell of z_i = sqrt(d) y_i, decided in fp32 */
    float tf[7];
    for (int j = 0; j < 7; j++) tf[j] = (float)t[j];
    for (int i = 0; i < d; i++) {
        double zi = sd * y[i];
        if (z) z[i] = zi;
        if (codes_in) {
            codes[i] = codes_in[i];
        } else {
            float zf = (float)zi;
            int k = 0;
            for (int j = 0; j < 7; j++) k += (zf >= tf[j]);
            codes[i] = (uint8_t)k;
        }
    }
    *n_out = n;

    if (is_k) {
        /* step 4: residual against the quantised approximation */
        double g2 = 0.0;
        for (int i = 0; i < d; i++) {
            r[i] = y[i] - c[codes[i]] / sd;
            g2 += r[i] * r[i];
        }
        *gamma_out = sqrt(g2);
        /* step 5: QJL projection of the residual, keep the signs */
        for (int k = 0; k < d; k++) {
            double acc = 0.0;
            for (int i = 0; i < d; i++) acc += (double)S[(size_t)k * d + i] * r[i];
            if (p) p[k] = acc;
            signs[k] = ((float)acc >= 0.0f) ? 1 : 0;
        }
    } else if (gamma_out) {
        *gamma_out = 0.0;
    }
    free(xh); free(y); free(r);
}

/* ------------------------------------------------------------------ */
/* Packed paged layout (a convention of this library; parity unpinned) */
/* ------------------------------------------------------------------ */
/* One pool holds [num_blocks][n_kv_heads][record bytes]; a record holds
 * the 16 token slots of one block for one head.
 *
 * K record (d=128: 1088 B): d/2 bytes of 4-bit fields per slot (3 cell bits
 * and the QJL sign bit of one coordinate), 8*d bytes in all, then
 * 16 x {fp16 n, fp16 gamma}.
 * V record (d=128: 800 B): 3*d/8 bytes of cell bits per slot, 6*d bytes in
 * all, then 16 x fp16 n.
 *
 * The cell bits are addressed as bits of little-endian 32-bit words, which
 * are grouped by a "lane" L = 4*gid + tig (0..31).  Every byte belongs to
 * one token slot, so slots can be written independently. */

size_t tqo_k_record_bytes(int d) { return (size_t)8 * d + TQO_BLOCK * 4; }
size_t tqo_v_record_bytes(int d) { return (size_t)6 * d + TQO_BLOCK * 2; }

/* K: slot t, coordinate i, field bit p (0..2: cell bit p, 3: QJL sign bit)
 * -> (word, bit).  Coordinate i = 16*ks + c with column c = 2*tig + e + 8*h
 * (e = c&1, h = c>>3); slot t = gid + 8*r.  Lane L = 4*gid + tig holds, per
 * slot row r, d/32 words; word w holds the 8 coordinates of columns
 * {2tig, 2tig+1, 2tig+8, 2tig+9} of k-steps 2w and 2w+1 as 4-bit fields:
 * field f = 4*(ks&1) + e + 2*h, at bits 4f .. 4f+3. */
void tqo_k_bitpos(int d, int t, int i, int p, int *word, int *bit)
{
    int nw = d / 32;
    int ks = i >> 4, c = i & 15;
    int tig = (c & 7) >> 1, e = c & 1, h = c >> 3;
    int gid = t & 7, r = t >> 3;
    int f = 4 * (ks & 1) + e + 2 * h;
    *word = ((4 * gid + tig) * 2 + r) * nw + (ks >> 1);
    *bit = 4 * f + p;
}

/* V: slot t, coordinate i, cell bit p (0..2) -> (word, bit).
 * Coordinate i = 16*mt + gid + 8*rr; its slot index within the lane is
 * s = 2*mt + rr (0 .. d/8-1), cut into groups of 16 (g = s/16, sg = s%16).
 * Slot t: tig = (t&7)>>1, pair P = t>>3, e = t&1 (first or second slot of
 * the pair).  Lane L = 4*gid + tig holds, per pair P, 3 words per group.
 * With hf = (sg>>1)&1 and ab = sg&1, the 4-bit field f = 4*hf + 2*e + ab of
 * word 3*g + (sg>>2) holds the cell in bits 0..2 when sg < 12; the fields of
 * sg = 12..15 (hf = (sg-12)>>1, ab = sg&1) keep cell bit p in bit 3 of field
 * f of word 3*g + p.  Field f sits in byte f>>1 = 2*hf + e, so the bytes of
 * a word alternate between the two slots of the pair. */
void tqo_v_bitpos(int d, int t, int i, int p, int *word, int *bit)
{
    int ng = d / 128;
    int mt = i >> 4, rr = (i & 15) >> 3, gid = i & 7;
    int s = 2 * mt + rr, g = s >> 4, sg = s & 15;
    int tig = (t & 7) >> 1, P = t >> 3, e = t & 1;
    int base = ((4 * gid + tig) * 2 + P) * 3 * ng + 3 * g;
    if (sg < 12) {
        int f = 4 * ((sg >> 1) & 1) + 2 * e + (sg & 1);
        *word = base + (sg >> 2);
        *bit = 4 * f + p;
    } else {
        int f = 4 * ((sg - 12) >> 1) + 2 * e + (sg & 1);
        *word = base + p;
        *bit = 4 * f + 3;
    }
}

static void set_bit(uint8_t *rec, int word, int bit, int v)
{
    uint8_t *b = rec + (size_t)word * 4 + (bit >> 3);
    uint8_t m = (uint8_t)(1u << (bit & 7));
    if (v) *b |= m; else *b &= (uint8_t)~m;
}
static int get_bit(const uint8_t *rec, int word, int bit)
{
    return (rec[(size_t)word * 4 + (bit >> 3)] >> (bit & 7)) & 1;
}
static void put16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 255); p[1] = (uint8_t)(v >> 8); }
static uint16_t get16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

void tqo_pack_k(int d, uint8_t *rec, int t, const uint8_t *codes, const uint8_t *signs,
                uint16_t n16, uint16_t g16)
{
    for (int i = 0; i < d; i++) {
        for (int pl = 0; pl < 4; pl++) {
            int w, b;
            tqo_k_bitpos(d, t, i, pl, &w, &b);
            set_bit(rec, w, b, pl < 3 ? (codes[i] >> pl) & 1 : signs[i]);
        }
    }
    uint8_t *nr = rec + (size_t)8 * d + 4 * t;
    put16(nr, n16);
    put16(nr + 2, g16);
}

void tqo_unpack_k(int d, const uint8_t *rec, int t, uint8_t *codes, uint8_t *signs,
                  uint16_t *n16, uint16_t *g16)
{
    for (int i = 0; i < d; i++) {
        int k = 0, w, b;
        for (int pl = 0; pl < 3; pl++) {
            tqo_k_bitpos(d, t, i, pl, &w, &b);
            k |= get_bit(rec, w, b) << pl;
        }
        codes[i] = (uint8_t)k;
        tqo_k_bitpos(d, t, i, 3, &w, &b);
        signs[i] = (uint8_t)get_bit(rec, w, b);
    }
    const uint8_t *nr = rec + (size_t)8 * d + 4 * t;
    *n16 = get16(nr);
    *g16 = get16(nr + 2);
}

void tqo_pack_v(int d, uint8_t *rec, int t, const uint8_t *codes, uint16_t n16)
{
    for (int i = 0; i < d; i++) {
        for (int pl = 0; pl < 3; pl++) {
            int w, b;
            tqo_v_bitpos(d, t, i, pl, &w, &b);
            set_bit(rec, w, b, (codes[i] >> pl) & 1);
        }
    }
    put16(rec + (size_t)6 * d + 2 * t, n16);
}

void tqo_unpack_v(int d, const uint8_t *rec, int t, uint8_t *codes, uint16_t *n16)
{
    for (int i = 0; i < d; i++) {
        int k = 0;
        for (int pl = 0; pl < 3; pl++) {
            int w, b;
            tqo_v_bitpos(d, t, i, pl, &w, &b);
            k |= get_bit(rec, w, b) << pl;
        }
        codes[i] = (uint8_t)k;
    }
    *n16 = get16(rec + (size_t)6 * d + 2 * t);
}

/* ------------------------------------------------------------------ */
/* Batched encode into a paged pool                                   */
/* ------------------------------------------------------------------ */
/* x: [n_tokens][n_heads][d] fp32 (an exact copy of bf16 inputs where the
 * caller has bf16).  slots[n] = block*16 + offset.  Every (token, head)
 * vector is encoded independently (parallel), then packed serially (V
 * words are shared by 4 token slots, so packing is kept single-threaded).
 * Optional per-vector outputs: codes_out/signs_out [n][h][d], norms
 * n_out/g_out [n][h] (fp64, before fp16 rounding), z_out/p_out [n][h][d].
 * Returns 0, or -1 for a slot outside the pool. */
int tqo_encode(int is_k, int d, const int8_t *D, const float *S, const double c[8],
               const double t[7], const float *x, int n_tokens, int n_heads,
               const int64_t *slots, uint8_t *pool, int64_t num_blocks,
               const uint8_t *codes_in, uint8_t *codes_out, uint8_t *signs_out,
               double *n_out, double *g_out, double *z_out, double *p_out)
{
    size_t nv = (size_t)n_tokens * n_heads;
    size_t rec = is_k ? tqo_k_record_bytes(d) : tqo_v_record_bytes(d);
    uint8_t *codes = (uint8_t *)malloc(nv * d);
    uint8_t *signs = (uint8_t *)malloc(nv * d);
    double *ns = (double *)malloc(nv * sizeof(double));
    double *gs = (double *)malloc(nv * sizeof(double));
    for (int64_t k = 0; k < n_tokens; k++)
        if (slots[k] < 0 || slots[k] / TQO_BLOCK >= num_blocks) {
            free(codes); free(signs); free(ns); free(gs);
            return -1;
        }
#pragma omp parallel for schedule(dynamic, 16)
    for (long long v = 0; v < (long long)nv; v++) {
        double *xv = (double *)malloc(sizeof(double) * d);
        for (int i = 0; i < d; i++) xv[i] = (double)x[(size_t)v * d + i];
        tqo_encode_vector(is_k, d, D, S, c, t, xv, codes_in ? codes_in + (size_t)v * d : NULL,
                          codes + (size_t)v * d, signs + (size_t)v * d, &ns[v], &gs[v],
                          z_out ? z_out + (size_t)v * d : NULL,
                          p_out ? p_out + (size_t)v * d : NULL);
        free(xv);
    }
    for (size_t v = 0; v < nv; v++) {
        int64_t tok = (int64_t)(v / n_heads);
        int h = (int)(v % n_heads);
        int64_t blk = slots[tok] / TQO_BLOCK;
        int off = (int)(slots[tok] % TQO_BLOCK);
        uint8_t *r = pool + ((size_t)blk * n_heads + h) * rec;
        if (is_k)
            tqo_pack_k(d, r, off, codes + v * d, signs + v * d, tqo_fp16_rne(ns[v]), tqo_fp16_rne(gs[v]));
        else
            tqo_pack_v(d, r, off, codes + v * d, tqo_fp16_rne(ns[v]));
    }
    if (codes_out) memcpy(codes_out, codes, nv * d);
    if (signs_out) memcpy(signs_out, signs, nv * d);
    if (n_out) memcpy(n_out, ns, nv * sizeof(double));
    if (g_out) memcpy(g_out, gs, nv * sizeof(double));
    free(codes); free(signs); free(ns); free(gs);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Decode attention over the compressed, paged cache                  */
/* ------------------------------------------------------------------ */
/* For query head h of sequence b (kv head h / (Hq/Hkv)), over the ctx[b]
 * cached tokens (logical token j lives in block block_table[b][j/16],
 * slot j%16  [VLLM "Paged KVキャッシュ"]):
 *   qbar = Pi q,  u = S qbar,
 *   s_j  = (n_j/sqrt d) * ( <qbar, c[code_j]>/sqrt d
 *                           + gamma_j * sqrt(pi/2)/d * <u, 2*sign_j-1> ),
 *   P    = softmax(s)   (the 1/sqrt d attention scale is inside s_j),
 *   a    = sum_j P_j * nv_j * c[codev_j] / sqrt d     (rotated domain),
 *   o    = Pi^T a.
 * A sequence with no cached tokens gets o = 0.  out: [B][Hq][d] fp64. */
int tqo_decode(int d, const int8_t *D, const float *S, const double c[8],
               const float *q, int B, int Hq, int Hkv,
               const uint8_t *kpool, const uint8_t *vpool,
               const int32_t *block_table, int max_blocks, const int32_t *ctx,
               double *out)
{
    if (Hkv <= 0 || Hq % Hkv) return -1;
    int g = Hq / Hkv;
    size_t krec = tqo_k_record_bytes(d), vrec = tqo_v_record_bytes(d);
    double sd = sqrt((double)d);
    double qjl = sqrt(M_PI / 2.0) / d;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long bh = 0; bh < (long long)B * Hq; bh++) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq), kh = h / g;
        int L = ctx[b];
        double *o = out + (size_t)bh * d;
        if (L <= 0) { for (int i = 0; i < d; i++) o[i] = 0.0; continue; }
        double *qd = (double *)malloc(sizeof(double) * d);
        double *qb = (double *)malloc(sizeof(double) * d);
        double *u = (double *)malloc(sizeof(double) * d);
        double *a = (double *)calloc(d, sizeof(double));
        double *s = (double *)malloc(sizeof(double) * L);
        uint8_t *codes = (uint8_t *)malloc(d), *signs = (uint8_t *)malloc(d);
        for (int i = 0; i < d; i++) qd[i] = q[(size_t)bh * d + i];
        tqo_rotate(d, D, qd, qb);
        for (int k = 0; k < d; k++) {
            double acc = 0.0;
            for (int i = 0; i < d; i++) acc += (double)S[(size_t)k * d + i] * qb[i];
            u[k] = acc;
        }
        double m = -INFINITY;
        for (int j = 0; j < L; j++) {
            int blk = block_table[(size_t)b * max_blocks + j / TQO_BLOCK];
            const uint8_t *rec = kpool + ((size_t)blk * Hkv + kh) * krec;
            uint16_t n16, g16;
            tqo_unpack_k(d, rec, j % TQO_BLOCK, codes, signs, &n16, &g16);
            double dc = 0.0, dq = 0.0;
            for (int i = 0; i < d; i++) {
                dc += qb[i] * c[codes[i]];
                dq += u[i] * (signs[i] ? 1.0 : -1.0);
            }
            double n = tqo_fp16_value(n16), gm = tqo_fp16_value(g16);
            s[j] = (n / sd) * (dc / sd + gm * qjl * dq);
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < L; j++) {
            double pj = exp(s[j] - m);
            l += pj;
            int blk = block_table[(size_t)b * max_blocks + j / TQO_BLOCK];
            const uint8_t *rec = vpool + ((size_t)blk * Hkv + kh) * vrec;
            uint16_t n16;
            tqo_unpack_v(d, rec, j % TQO_BLOCK, codes, &n16);
            double w = pj * tqo_fp16_value(n16) / sd;
            for (int i = 0; i < d; i++) a[i] += w * c[codes[i]];
        }
        for (int i = 0; i < d; i++) a[i] /= l;
        tqo_rotate_t(d, D, a, o);
        free(qd); free(qb); free(u); free(a); free(s); free(codes); free(signs);
    }
    return 0;
}

/* Second, independent formulation: dequantise every cached key and value
 * back to the original domain and run textbook softmax attention.
 *   k~_j = n_j * Pi^T( c[code_j]/sqrt d + sqrt(pi/2)/d * gamma_j * S^T (2*sign_j-1) ),
 *   v~_j = nv_j * Pi^T( c[codev_j]/sqrt d ),
 *   o    = sum_j softmax_j(<q, k~_j>/sqrt d) v~_j.
 * Used only to pin tqo_decode (the two must agree to rounding). */
int tqo_decode_explicit(int d, const int8_t *D, const float *S, const double c[8],
                        const float *q, int B, int Hq, int Hkv,
                        const uint8_t *kpool, const uint8_t *vpool,
                        const int32_t *block_table, int max_blocks, const int32_t *ctx,
                        double *out)
{
    if (Hkv <= 0 || Hq % Hkv) return -1;
    int g = Hq / Hkv;
    size_t krec = tqo_k_record_bytes(d), vrec = tqo_v_record_bytes(d);
    double sd = sqrt((double)d);
    double qjl = sqrt(M_PI / 2.0) / d;
    for (long long bh = 0; bh < (long long)B * Hq; bh++) {
        int b = (int)(bh / Hq), h = (int)(bh % Hq), kh = h / g;
        int L = ctx[b];
        double *o = out + (size_t)bh * d;
        for (int i = 0; i < d; i++) o[i] = 0.0;
        if (L <= 0) continue;
        double *yk = (double *)malloc(sizeof(double) * d);
        double *kt = (double *)malloc(sizeof(double) * d);
        double *vt = (double *)malloc(sizeof(double) * (size_t)L * d);
        double *s = (double *)malloc(sizeof(double) * L);
        uint8_t *codes = (uint8_t *)malloc(d), *signs = (uint8_t *)malloc(d);
        double m = -INFINITY;
        for (int j = 0; j < L; j++) {
            int blk = block_table[(size_t)b * max_blocks + j / TQO_BLOCK];
            uint16_t n16, g16, nv16;
            tqo_unpack_k(d, kpool + ((size_t)blk * Hkv + kh) * krec, j % TQO_BLOCK, codes, signs, &n16, &g16);
            double n = tqo_fp16_value(n16), gm = tqo_fp16_value(g16);
            for (int i = 0; i < d; i++) {
                double st = 0.0;    /* (S^T b~)_i */
                for (int k = 0; k < d; k++) st += (double)S[(size_t)k * d + i] * (signs[k] ? 1.0 : -1.0);
                yk[i] = c[codes[i]] / sd + qjl * gm * st;
            }
            tqo_rotate_t(d, D, yk, kt);
            double dot = 0.0;
            for (int i = 0; i < d; i++) dot += (double)q[(size_t)bh * d + i] * n * kt[i];
            s[j] = dot / sd;
            if (s[j] > m) m = s[j];
            tqo_unpack_v(d, vpool + ((size_t)blk * Hkv + kh) * vrec, j % TQO_BLOCK, codes, &nv16);
            double nv = tqo_fp16_value(nv16);
            for (int i = 0; i < d; i++) yk[i] = c[codes[i]] / sd;
            tqo_rotate_t(d, D, yk, vt + (size_t)j * d);
            for (int i = 0; i < d; i++) vt[(size_t)j * d + i] *= nv;
        }
        double l = 0.0;
        for (int j = 0; j < L; j++) l += exp(s[j] - m);
        for (int j = 0; j < L; j++) {
            double pj = exp(s[j] - m) / l;
            for (int i = 0; i < d; i++) o[i] += pj * vt[(size_t)j * d + i];
        }
        free(yk); free(kt); free(vt); free(s); free(codes); free(signs);
    }
    return 0;
}
