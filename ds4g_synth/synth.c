/*
 * ds4g_synth: seeded synthetic inputs for the routed-MoE layer.
 *
 * Shared by the tests, the oracle runs and the benchmark.  It holds the
 * input recipes only -- random draws, bf16 rounding of activations, router
 * logit recipes, and the encoders that turn drawn fp32 weights into 2-bit
 * blocks (the offline quantization step the pages attribute to gguf-tools,
 * ds4 README mirror, "More Documentation").  It computes no step of the
 * layer itself: no dequantization, no routing decision, no projection.
 *
 * Random numbers: counter-based splitmix64 (Steele, Lea & Flood, "Fast
 * splittable pseudorandom number generators", OOPSLA 2014).  Draw i of the
 * stream with key K is mix64(K + (i + 1) * GAMMA), i.e. the i-th output of a
 * splitmix64 generator whose state starts at K.  Every value depends only on
 * (seed, tensor, sub-stream, index), so the bytes do not depend on the
 * number of threads that produce them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
#define QK 256

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of the sub-stream `sub` of tensor `tensor` under `seed`. */
uint64_t syn_key(uint64_t seed, uint64_t tensor, uint64_t sub)
{
    uint64_t k = mix64(seed * GAMMA + 0x5851F42D4C957F2DULL);
    k = mix64(k ^ (tensor * GAMMA + 0x14057B7EF767814FULL));
    return mix64(k ^ (sub * GAMMA + 0x2545F4914F6CDD1DULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

/* Uniform on [0, 1) with 24 random bits (exact in fp32). */
static inline double uniform24(uint64_t key, uint64_t i)
{
    return (double)(draw(key, i) >> 40) * (1.0 / 16777216.0);
}

/* Standard normals by Box-Muller in fp32 on the pair of draws (2p, 2p+1):
 * u1 in (0, 1], u2 in [0, 1), both with 24 random bits;
 * r = sqrt(-2 ln u1), theta = 2 pi u2; number 2p is r cos(theta), number
 * 2p+1 is r sin(theta). */
static inline void normal_pair(uint64_t key, uint64_t p, double *z0, double *z1)
{
    float u1 = ((float)(draw(key, 2 * p) >> 40) + 1.0f) * (1.0f / 16777216.0f);
    float u2 = (float)(draw(key, 2 * p + 1) >> 40) * (1.0f / 16777216.0f);
    float r = sqrtf(-2.0f * logf(u1));
    float th = 6.2831853f * u2;
    *z0 = (double)(r * cosf(th));
    *z1 = (double)(r * sinf(th));
}

static inline double normal(uint64_t key, uint64_t i)
{
    double z0, z1;
    normal_pair(key, i >> 1, &z0, &z1);
    return (i & 1) ? z1 : z0;
}

double syn_uniform(uint64_t key, uint64_t i) { return uniform24(key, i); }
double syn_normal(uint64_t key, uint64_t i) { return normal(key, i); }
uint64_t syn_draw(uint64_t key, uint64_t i) { return draw(key, i); }

/* fp32 -> bf16 bits, round to nearest even (NaN -> canonical quiet NaN). */
uint16_t syn_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
    uint32_t bias = 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)((u + bias) >> 16);
}

/* double -> IEEE binary16 bits, round to nearest even, with subnormals and
 * overflow to infinity. */
uint16_t syn_double_to_half(double v)
{
    uint16_t sign = 0;
    if (v != v) return 0x7E00;
    if (v < 0 || (v == 0 && signbit(v))) { sign = 0x8000; v = -v; }
    if (v == 0) return sign;
    if (v >= 65520.0) return sign | 0x7C00;           /* rounds to inf */
    int e;
    frexp(v, &e);                                     /* v = m * 2^e, m in [0.5,1) */
    int expo = e - 1;                                 /* v = 1.f * 2^expo */
    if (expo < -14) {                                 /* subnormal: units of 2^-24 */
        double units = nearbyint(ldexp(v, 24));
        if (units >= 1024.0) return sign | 0x0400;    /* rounded up to min normal */
        return sign | (uint16_t)units;
    }
    double mant = nearbyint(ldexp(v, 10 - expo));     /* in [1024, 2048] */
    if (mant >= 2048.0) { mant = 1024.0; expo += 1; }
    if (expo > 15) return sign | 0x7C00;
    return sign | (uint16_t)(((expo + 15) << 10) | ((int)mant - 1024));
}

static double half_value(uint16_t h)
{
    int expo = (h >> 10) & 31, frac = h & 1023;
    double v = expo ? ldexp(1024.0 + frac, expo - 25) : ldexp((double)frac, -24);
    return (h & 0x8000) ? -v : v;
}

/* ------------------------------------------------------------------------
 * Encoders (reference quantizers).  Any deterministic encoder yields valid
 * inputs: the layer is defined on the stored bytes.
 * --------------------------------------------------------------------- */

/* Round to nearest, ties to even, for |v| < 2^51 (default rounding mode):
 * adding and subtracting 1.5 * 2^52 leaves v rounded to an integer. */
static inline double rne(double v)
{
    volatile double big = 6755399441055744.0;
    return (v + big) - big;
}

static int clamp_int(double v, int lo, int hi)
{
    if (!(v >= lo)) return lo;
    if (v > hi) return hi;
    return (int)v;
}

/* Q2_K encoder for one 256-weight block (84 bytes).  Per 16-weight
 * sub-block s: lo = min(0, min w), hi = max w, a_s = (hi - lo) / 3,
 * m_s = -lo.  d = fp16(max a_s / 15), dmin = fp16(max m_s / 15);
 * sc_s = clamp(rne(a_s / d), 0, 15), mn_s = clamp(rne(m_s / dmin), 0, 15);
 * q = clamp(rne((w + dmin mn_s) / (d sc_s)), 0, 3) (0 when sc_s = 0). */
void syn_q2k_encode_block(const float *w, uint8_t *blk)
{
    double a[16], m[16], amax = 0, mmax = 0;
    for (int s = 0; s < 16; ++s) {
        double lo = 0, hi = -INFINITY;
        for (int j = 0; j < 16; ++j) {
            double v = w[16 * s + j];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        a[s] = (hi - lo) / 3.0;
        m[s] = -lo;
        if (a[s] > amax) amax = a[s];
        if (m[s] > mmax) mmax = m[s];
    }
    uint16_t dh = syn_double_to_half(amax / 15.0);
    uint16_t mh = syn_double_to_half(mmax / 15.0);
    double d = half_value(dh), dmin = half_value(mh);
    uint8_t *scales = blk, *qs = blk + 16;
    memset(blk, 0, 84);
    int sc[16], mn[16];
    for (int s = 0; s < 16; ++s) {
        sc[s] = d > 0 ? clamp_int(rne(a[s] / d), 0, 15) : 0;
        mn[s] = dmin > 0 ? clamp_int(rne(m[s] / dmin), 0, 15) : 0;
        scales[s] = (uint8_t)(sc[s] | (mn[s] << 4));
    }
    for (int j = 0; j < QK; ++j) {
        int s = j / 16;
        int q = 0;
        if (sc[s] > 0)
            q = clamp_int(rne(((double)w[j] + dmin * mn[s]) / (d * sc[s])), 0, 3);
        int h = j / 128, r = j % 128, g = r / 32, l = r % 32;
        qs[32 * h + l] |= (uint8_t)(q << (2 * g));
    }
    blk[80] = (uint8_t)(dh & 0xFF);
    blk[81] = (uint8_t)(dh >> 8);
    blk[82] = (uint8_t)(mh & 0xFF);
    blk[83] = (uint8_t)(mh >> 8);
}

/* Q4_K (levels 15) / Q5_K (levels 31) quantization of one 256-weight block.
 * Per 32-weight sub-block s: lo = min(0, min w), hi = max w,
 * a_s = (hi - lo) / levels, m_s = -lo; d = fp16(max a_s / 63),
 * dmin = fp16(max m_s / 63); sc_s = clamp(rne(a_s / d), 0, 63),
 * mn_s = clamp(rne(m_s / dmin), 0, 63);
 * q = clamp(rne((w + dmin mn_s) / (d sc_s)), 0, levels) (0 when sc_s = 0). */
static void k45_quantize(const float *w, int levels, int *sc, int *mn, int *q, uint16_t *dh,
                         uint16_t *mh)
{
    double a[8], m[8], amax = 0, mmax = 0;
    for (int s = 0; s < 8; ++s) {
        double lo = 0, hi = -INFINITY;
        for (int j = 0; j < 32; ++j) {
            double v = w[32 * s + j];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        a[s] = (hi - lo) / levels;
        m[s] = -lo;
        if (a[s] > amax) amax = a[s];
        if (m[s] > mmax) mmax = m[s];
    }
    *dh = syn_double_to_half(amax / 63.0);
    *mh = syn_double_to_half(mmax / 63.0);
    double d = half_value(*dh), dmin = half_value(*mh);
    for (int s = 0; s < 8; ++s) {
        sc[s] = d > 0 ? clamp_int(rne(a[s] / d), 0, 63) : 0;
        mn[s] = dmin > 0 ? clamp_int(rne(m[s] / dmin), 0, 63) : 0;
    }
    for (int j = 0; j < QK; ++j) {
        int s = j / 32;
        q[j] = sc[s] > 0 ? clamp_int(rne(((double)w[j] + dmin * mn[s]) / (d * sc[s])), 0, levels) : 0;
    }
}

/* The 12 packed bytes of eight 6-bit scales and mins (low six bits of bytes
 * 0..3 / 4..7 for sub-blocks 0..3, low / high nibbles of bytes 8..11 for
 * sub-blocks 4..7, whose top two bits ride in the top bits of bytes 0..7). */
static void k45_pack_scales(const int *sc, const int *mn, uint8_t *p)
{
    for (int s = 0; s < 4; ++s) {
        p[s] = (uint8_t)(sc[s] | ((sc[s + 4] >> 4) << 6));
        p[s + 4] = (uint8_t)(mn[s] | ((mn[s + 4] >> 4) << 6));
        p[s + 8] = (uint8_t)((sc[s + 4] & 15) | ((mn[s + 4] & 15) << 4));
    }
}

/* Q4_K block (144 bytes): d, dmin, packed scales, qs (weight 64c + l in the
 * low nibble of qs[32c + l], weight 64c + 32 + l in its high nibble). */
void syn_q4k_encode_block(const float *w, uint8_t *blk)
{
    int sc[8], mn[8], q[QK];
    uint16_t dh, mh;
    k45_quantize(w, 15, sc, mn, q, &dh, &mh);
    memset(blk, 0, 144);
    blk[0] = (uint8_t)(dh & 0xFF); blk[1] = (uint8_t)(dh >> 8);
    blk[2] = (uint8_t)(mh & 0xFF); blk[3] = (uint8_t)(mh >> 8);
    k45_pack_scales(sc, mn, blk + 4);
    for (int j = 0; j < QK; ++j) {
        int c = j / 64, r = j % 64;
        blk[16 + 32 * c + r % 32] |= (uint8_t)(q[j] << (r < 32 ? 0 : 4));
    }
}

/* Q5_K block (176 bytes): as Q4_K, with bit 4 of weight 32s + l in bit s of
 * qh[l] (bytes 16..47) and the low nibbles at bytes 48..175. */
void syn_q5k_encode_block(const float *w, uint8_t *blk)
{
    int sc[8], mn[8], q[QK];
    uint16_t dh, mh;
    k45_quantize(w, 31, sc, mn, q, &dh, &mh);
    memset(blk, 0, 176);
    blk[0] = (uint8_t)(dh & 0xFF); blk[1] = (uint8_t)(dh >> 8);
    blk[2] = (uint8_t)(mh & 0xFF); blk[3] = (uint8_t)(mh >> 8);
    k45_pack_scales(sc, mn, blk + 4);
    for (int j = 0; j < QK; ++j) {
        int c = j / 64, r = j % 64, l = r % 32;
        blk[48 + 32 * c + l] |= (uint8_t)((q[j] & 15) << (r < 32 ? 0 : 4));
        blk[16 + l] |= (uint8_t)(((q[j] >> 4) & 1) << (j / 32));
    }
}

/* Q6_K block (210 bytes).  Per 16-weight sub-block t: a_t = max |w| / 31;
 * d = fp16(max a_t / 127); sc_t = clamp(rne(a_t / d), -128, 127);
 * q = clamp(rne(w / (d sc_t)), -32, 31) (0 when sc_t = 0), stored as
 * v = q + 32: low nibble of v in nibble (u >> 1) of ql[64h + 32(u&1) + l],
 * its top two bits in bits 2u..2u+1 of qh[32h + l] (h = j/128, u = (j%128)/32,
 * l = j%32); scales at 192..207, d at 208..209. */
void syn_q6k_encode_block(const float *w, uint8_t *blk)
{
    double a[16], amax = 0;
    for (int t = 0; t < 16; ++t) {
        double mx = 0;
        for (int j = 0; j < 16; ++j) {
            double v = fabs((double)w[16 * t + j]);
            if (v > mx) mx = v;
        }
        a[t] = mx / 31.0;
        if (a[t] > amax) amax = a[t];
    }
    uint16_t dh = syn_double_to_half(amax / 127.0);
    double d = half_value(dh);
    int sc[16];
    memset(blk, 0, 210);
    for (int t = 0; t < 16; ++t) {
        sc[t] = d > 0 ? clamp_int(rne(a[t] / d), -128, 127) : 0;
        blk[192 + t] = (uint8_t)(int8_t)sc[t];
    }
    for (int j = 0; j < QK; ++j) {
        int t = j / 16;
        int q = sc[t] != 0 ? clamp_int(rne((double)w[j] / (d * sc[t])), -32, 31) : 0;
        int v = q + 32;
        int h = j / 128, r = j % 128, u = r / 32, l = r % 32;
        blk[64 * h + 32 * (u & 1) + l] |= (uint8_t)((v & 15) << (4 * (u >> 1)));
        blk[128 + 32 * h + l] |= (uint8_t)((v >> 4) << (2 * u));
    }
    blk[208] = (uint8_t)(dh & 0xFF);
    blk[209] = (uint8_t)(dh >> 8);
}

/* MXFP4 unit (eight 17-byte blocks, 256 weights).  Per 32 weights:
 * amax = max |w|; e = clamp(ceil(log2(amax / 6)) + 127, 0, 254) (127 when
 * amax = 0), so |w| / 2^(e-127) <= 6; each weight takes the E2M1 magnitude
 * nearest to |w| / 2^(e-127) (0, 0.5, 1, 1.5, 2, 3, 4, 6; the lower one on a
 * tie) and its sign (bit 3; +0 for zero); weight i of the block goes to the
 * low nibble of byte 1 + i, weight 16 + i to the high nibble. */
void syn_mxfp4_encode_block(const float *w, uint8_t *blk)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    memset(blk, 0, 136);
    for (int b = 0; b < 8; ++b) {
        const float *v = w + 32 * b;
        uint8_t *o = blk + 17 * b;
        double amax = 0;
        for (int j = 0; j < 32; ++j)
            if (fabs((double)v[j]) > amax) amax = fabs((double)v[j]);
        int e = 127;
        if (amax > 0) {
            e = (int)ceil(log2(amax / 6.0)) + 127;
            if (e < 0) e = 0;
            if (e > 254) e = 254;
        }
        o[0] = (uint8_t)e;
        double scale = ldexp(1.0, e - 127);
        for (int j = 0; j < 32; ++j) {
            double x = fabs((double)v[j]) / scale;
            int best = 0;
            for (int c = 1; c < 8; ++c)
                if (fabs(x - mag[c]) < fabs(x - mag[best])) best = c;
            int code = best | ((v[j] < 0 && best != 0) ? 8 : 0);
            o[1 + j % 16] |= (uint8_t)(code << (j < 16 ? 0 : 4));
        }
    }
}

/* Super-block bytes of each weight format (0 Q2_K, 1 codebook, 2 Q4_K,
 * 3 Q5_K, 4 Q6_K, 5 MXFP4 (eight blocks)); 0 for an unknown format. */
static int block_bytes(int format)
{
    static const int bb[6] = {84, 70, 144, 176, 210, 136};
    return format >= 0 && format < 6 ? bb[format] : 0;
}

/* score[i] = D * n2[i] - sum_b (2 |w_b|) * |c_ib|, accumulated over b in
 * order; each i is independent, so the vector clones round exactly like the
 * scalar one (no contraction: built with -ffp-contract=off). */
__attribute__((target_clones("avx2", "default")))
static void cb2_scores(float D, const float *absw, const float *mag_t, const float *n2,
                       float *score)
{
    for (int i = 0; i < 256; ++i) score[i] = D * n2[i];
    for (int b = 0; b < 8; ++b) {
        float twice = 2.0f * absw[b];
        const float *mb = mag_t + 256 * b;
        for (int i = 0; i < 256; ++i) score[i] -= twice * mb[i];
    }
}

/* Codebook-2-bit encoder for one 256-weight block (70 bytes).
 * Per 32-group G: a_G = max |w| / 43; d = fp16(max a_G / 15);
 * s_G = clamp(rne(a_G / d), 0, 15).  Per 8 weights: the codebook row
 * minimising sum_b (|w_b| - D |c_b|)^2 with D = d s_G, evaluated as the
 * fp32 score D * n2[idx] - 2 * dot(|w|, |c_idx|) (same argmin in exact
 * arithmetic), ties -> lower row; sign bit b set when sign(w_b) differs from
 * sign(c_b).  `mag_t` is the codebook's magnitudes transposed [8][256] and
 * `n2` their squared norms (both precomputed by the caller). */
static void cb2_encode_block(const float *w, const float *mag_t, const float *n2,
                             const int8_t *codebook, uint8_t *blk)
{
    double aG[8], amax = 0;
    for (int G = 0; G < 8; ++G) {
        double mx = 0;
        for (int j = 0; j < 32; ++j) {
            double v = fabs((double)w[32 * G + j]);
            if (v > mx) mx = v;
        }
        aG[G] = mx / 43.0;
        if (aG[G] > amax) amax = aG[G];
    }
    uint16_t dh = syn_double_to_half(amax / 15.0);
    double d = half_value(dh);
    memset(blk, 0, 70);
    int sG[8];
    for (int G = 0; G < 8; ++G) {
        sG[G] = d > 0 ? clamp_int(rne(aG[G] / d), 0, 15) : 0;
        blk[64 + G / 2] |= (uint8_t)(sG[G] << (4 * (G % 2)));
    }
    float score[256];
    for (int o = 0; o < 32; ++o) {
        float D = (float)(d * sG[o / 4]);
        float absw[8];
        for (int b = 0; b < 8; ++b) absw[b] = fabsf(w[8 * o + b]);
        cb2_scores(D, absw, mag_t, n2, score);
        int best = 0;
        for (int i = 1; i < 256; ++i)
            if (score[i] < score[best]) best = i;
        uint8_t sgn = 0;
        for (int b = 0; b < 8; ++b) {
            int wneg = w[8 * o + b] < 0;
            int cneg = codebook[8 * best + b] < 0;
            if (wneg != cneg) sgn |= (uint8_t)(1u << b);
        }
        blk[o] = (uint8_t)best;
        blk[32 + o] = sgn;
    }
    blk[68] = (uint8_t)(dh & 0xFF);
    blk[69] = (uint8_t)(dh >> 8);
}

static void codebook_tables(const int8_t *codebook, float *mag_t, float *n2)
{
    for (int i = 0; i < 256; ++i) {
        float s = 0;
        for (int b = 0; b < 8; ++b) {
            float m = (float)abs(codebook[8 * i + b]);
            mag_t[256 * b + i] = m;
            s += m * m;
        }
        n2[i] = s;
    }
}

void syn_cb2_encode_block(const float *w, const int8_t *codebook, uint8_t *blk)
{
    float mag_t[8 * 256], n2[256];
    codebook_tables(codebook, mag_t, n2);
    cb2_encode_block(w, mag_t, n2, codebook, blk);
}

/* Seeded 256 x 8 int8 codebook, entries uniform over {+-8, +-25, +-43}. */
void syn_make_codebook(uint64_t seed, int8_t *cb)
{
    static const int8_t vals[6] = {-43, -25, -8, 8, 25, 43};
    uint64_t key = syn_key(seed, 6, 0);
    for (int i = 0; i < 256 * 8; ++i) {
        uint64_t u = draw(key, (uint64_t)i) >> 40;     /* 24 bits */
        cb[i] = vals[(u * 6) >> 24];
    }
}

/* ------------------------------------------------------------------------
 * Expert weight tensors: E experts x N rows x K logical columns drawn
 * N(0, sd) (tensor id, sub-stream = expert, index n*K + kk), encoded row by
 * row into ceil(K/256) blocks; columns K..pad are zero; row bytes beyond the
 * blocks are zero.  Threads split the rows; bytes are thread-independent.
 * --------------------------------------------------------------------- */
typedef struct {
    uint64_t seed;
    int tensor, E, N, K, format;
    int64_t row_bytes;
    double sd;
    uint8_t *out;
    const int8_t *codebook;
    const float *mag_t, *n2;
    int64_t row_begin, row_end;   /* over E*N rows */
} expert_job;

static void *expert_worker(void *arg)
{
    expert_job *J = (expert_job *)arg;
    int nblk = (J->K + QK - 1) / QK;
    int bb = block_bytes(J->format);
    float *w = (float *)malloc(sizeof(float) * nblk * QK);
    if (!w) return (void *)1;
    for (int64_t r = J->row_begin; r < J->row_end; ++r) {
        int e = (int)(r / J->N);
        int n = (int)(r % J->N);
        uint64_t key = syn_key(J->seed, (uint64_t)J->tensor, (uint64_t)e);
        uint64_t base = (uint64_t)n * J->K;
        for (int kk = 0; kk < nblk * QK; ++kk) {
            if (kk >= J->K) { w[kk] = 0.0f; continue; }
            uint64_t i = base + kk;
            if ((i & 1) == 0 && kk + 1 < J->K) {          /* both halves of a pair */
                double z0, z1;
                normal_pair(key, i >> 1, &z0, &z1);
                w[kk] = (float)(J->sd * z0);
                w[kk + 1] = (float)(J->sd * z1);
                ++kk;
            } else {
                w[kk] = (float)(J->sd * normal(key, i));
            }
        }
        uint8_t *row = J->out + r * J->row_bytes;
        memset(row, 0, (size_t)J->row_bytes);
        for (int b = 0; b < nblk; ++b) {
            uint8_t *blk = row + (int64_t)b * bb;
            switch (J->format) {
            case 0: syn_q2k_encode_block(w + b * QK, blk); break;
            case 1: cb2_encode_block(w + b * QK, J->mag_t, J->n2, J->codebook, blk); break;
            case 2: syn_q4k_encode_block(w + b * QK, blk); break;
            case 3: syn_q5k_encode_block(w + b * QK, blk); break;
            case 4: syn_q6k_encode_block(w + b * QK, blk); break;
            default: syn_mxfp4_encode_block(w + b * QK, blk); break;
            }
        }
    }
    free(w);
    return NULL;
}

int syn_make_experts(uint64_t seed, int tensor, int E, int N, int K, int format,
                     int64_t row_bytes, double sd, const int8_t *codebook,
                     uint8_t *out, int n_threads)
{
    int nblk = (K + QK - 1) / QK;
    int bb = block_bytes(format);
    if (bb == 0 || E < 1 || N < 1 || K < 1 || row_bytes < (int64_t)nblk * bb) return 1;
    if (format == 1 && !codebook) return 1;
    float mag_t[8 * 256], n2[256];
    if (format == 1) codebook_tables(codebook, mag_t, n2);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    int64_t rows = (int64_t)E * N;
    if (rows < n_threads) n_threads = (int)rows;
    pthread_t th[256];
    expert_job jobs[256];
    int rc = 0;
    for (int i = 0; i < n_threads; ++i) {
        expert_job *J = &jobs[i];
        J->seed = seed; J->tensor = tensor; J->E = E; J->N = N; J->K = K;
        J->format = format; J->row_bytes = row_bytes; J->sd = sd; J->out = out;
        J->codebook = codebook; J->mag_t = mag_t; J->n2 = n2;
        J->row_begin = rows * i / n_threads;
        J->row_end = rows * (i + 1) / n_threads;
        if (pthread_create(&th[i], NULL, expert_worker, J) != 0) {
            expert_worker(J);
            th[i] = 0;
        }
    }
    for (int i = 0; i < n_threads; ++i) {
        void *res = NULL;
        if (th[i]) pthread_join(th[i], &res);
        if (res) rc = 1;
    }
    return rc;
}

/* Activations x [T x H]: bf16 of N(0,1) (tensor 1, index t*H + h). */
void syn_make_x(uint64_t seed, int T, int H, uint16_t *x)
{
    uint64_t key = syn_key(seed, 1, 0);
    for (int64_t i = 0; i < (int64_t)T * H; ++i)
        x[i] = syn_f32_to_bf16((float)normal(key, (uint64_t)i));
}

/* ------------------------------------------------------------------------
 * Router logits [T x E].
 *   kind 0: N(0,1);  kind 1: U(0,1);  kind 2: N(0,1) + b_e, b_e ~ N(0, 0.5)
 *   drawn once per expert (tensor 7);  kind 3: Zipf(s)-skewed picks.
 * Kinds 0-2 redraw a whole row (attempt counter in the sub-stream) while the
 * gap between the k-th and (k+1)-th largest logit is below `margin`.
 * Kind 3: per token, k distinct experts drawn Zipf(s) over the ranks of a
 * seeded expert permutation, P(rank r) proportional to (r+1)^-s, duplicates
 * redrawn; picked experts get 2.5 + |N(0,1)|, the others min(N(0,1), 1.5),
 * so the gap is at least 1.
 * --------------------------------------------------------------------- */
static int cmp_desc(const void *a, const void *b)
{
    float x = *(const float *)a, y = *(const float *)b;
    return (x < y) - (x > y);
}

static void zipf_logits(uint64_t seed, int T, int E, int k, double s, float *out)
{
    int perm[256];
    double cum[256];
    for (int e = 0; e < E; ++e) perm[e] = e;
    uint64_t pk = syn_key(seed, 8, 0);
    for (int i = E - 1; i > 0; --i) {
        uint64_t u = draw(pk, (uint64_t)i) >> 11;            /* 53 bits */
        int j = (int)(((double)u * (1.0 / 9007199254740992.0)) * (i + 1));
        if (j > i) j = i;
        int tmp = perm[i]; perm[i] = perm[j]; perm[j] = tmp;
    }
    double run = 0;
    for (int r = 0; r < E; ++r) {
        run += pow((double)(r + 1), -s);
        cum[r] = run;
    }
    for (int t = 0; t < T; ++t) {
        uint64_t zk = syn_key(seed, 9, (uint64_t)t);
        uint64_t lk = syn_key(seed, 10, (uint64_t)t);
        char picked[256];
        memset(picked, 0, sizeof picked);
        int got = 0;
        for (uint64_t c = 0; got < k; ++c) {
            double u = uniform24(zk, c) * run;
            int lo = 0, hi = E - 1;
            while (lo < hi) {                                 /* first r with cum[r] > u */
                int mid = (lo + hi) / 2;
                if (cum[mid] > u) hi = mid; else lo = mid + 1;
            }
            int e = perm[lo];
            if (!picked[e]) { picked[e] = 1; ++got; }
        }
        for (int e = 0; e < E; ++e) {
            double z = normal(lk, (uint64_t)e);
            out[(int64_t)t * E + e] = picked[e] ? (float)(2.5 + fabs(z))
                                                : (float)(z < 1.5 ? z : 1.5);
        }
    }
}

int syn_make_logits(uint64_t seed, int kind, int T, int E, int k, double margin,
                    double zipf_s, float *out)
{
    if (T < 0 || E < 1 || E > 256 || k < 1 || k > E) return 1;
    if (kind == 3) { zipf_logits(seed, T, E, k, zipf_s, out); return 0; }
    double bias[256];
    uint64_t bk = syn_key(seed, 7, 0);
    for (int e = 0; e < E; ++e) bias[e] = kind == 2 ? 0.5 * normal(bk, (uint64_t)e) : 0.0;
    float sorted[256];
    for (int t = 0; t < T; ++t) {
        float *row = out + (int64_t)t * E;
        for (uint64_t attempt = 0;; ++attempt) {
            uint64_t key = syn_key(seed, 2, ((uint64_t)attempt << 32) | (uint64_t)t);
            for (int e = 0; e < E; ++e) {
                if (kind == 1)
                    row[e] = (float)uniform24(key, (uint64_t)e);
                else
                    row[e] = (float)(normal(key, (uint64_t)e) + bias[e]);
            }
            if (k == E) break;
            memcpy(sorted, row, sizeof(float) * E);
            qsort(sorted, E, sizeof(float), cmp_desc);
            if ((double)sorted[k - 1] - (double)sorted[k] >= margin) break;
            if (attempt > 1000000) return 2;
        }
    }
    return 0;
}
