/*
 * ds4g reference oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * Plain, single-threaded C99 restatement of what the routed-MoE expert layer
 * over 2-bit quantized experts computes.  Only the test suite, the package
 * smoke check and the CPU-baseline leg of the benchmark may load this code;
 * the CUDA library never does, and the two share no source, header, table
 * or helper.
 *
 * What the pages fix, and where:
 *   - the layer: routed MoE experts, up/gate and down projections, quantized
 *     at 2 bits while everything else stays untouched
 *     (ds4 README mirror, "Model Weights");
 *   - the formats: GGUF quant layouts retained from llama.cpp
 *     (ds4 README mirror, "Acknowledgements to llama.cpp and GGML"),
 *     an IQ2_XXS / Q2_K mix (DwarfStar 4 on aiany.app, "What Sets It Apart").
 * The pages print no formula for any step.  The block layouts, the SiLU
 * gated FFN, the top-k rule and the weight normalisations below are the
 * readings stated in the project design notes; each function says which.
 *
 * Precision: every weight is dequantized to fp32 exactly as its block
 * definition states; every dot product, the SiLU and the routing weights
 * are computed in fp64.
 *
 * Parity status of each function (what pins it) is listed in the design
 * notes; the layout choices for Q2_K (bit order inside qs) and for the
 * codebook format are pinned against the definitions written here, not
 * against real ds4 files ("parity unpinned" against the pages for those
 * byte orders: the pages print no layout).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_QK 256          /* weights per super-block                      */
#define ORC_Q2K_BYTES 84    /* Q2_K super-block bytes                       */
#define ORC_CB2_BYTES 70    /* codebook-2-bit super-block bytes             */
#define ORC_Q4K_BYTES 144   /* Q4_K super-block bytes                       */
#define ORC_Q5K_BYTES 176   /* Q5_K super-block bytes                       */
#define ORC_Q6K_BYTES 210   /* Q6_K super-block bytes                       */
#define ORC_MX_BYTES 17     /* MXFP4 block bytes (32 weights)               */
#define ORC_MXFP4_BYTES 136 /* eight MXFP4 blocks = 256 weights             */

enum { ORC_OK = 0, ORC_ERR_INVALID = 1, ORC_ERR_NOMEM = 2 };
enum { ORC_SCORE_SOFTMAX = 0, ORC_SCORE_SIGMOID = 1 };
enum { ORC_FMT_Q2K = 0, ORC_FMT_CB2 = 1, ORC_FMT_Q4K = 2, ORC_FMT_Q5K = 3, ORC_FMT_Q6K = 4,
       ORC_FMT_MXFP4 = 5 };

/* ------------------------------------------------------------------------
 * Scalar formats.
 * --------------------------------------------------------------------- */

/* IEEE-754 binary16 -> double, decoded from its sign, 5-bit exponent and
 * 10-bit fraction (bias 15; exponent 0 = subnormal, 31 = inf/nan). */
double orc_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25);
    return sign ? -v : v;
}

/* bfloat16 -> double: a bfloat16 is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ------------------------------------------------------------------------
 * Q2_K super-block (84 bytes, 256 weights), GGUF layout:
 *   bytes  0..15  scales[16]: low nibble = scale sc of 16-weight sub-block s,
 *                             high nibble = min m of sub-block s
 *   bytes 16..79  qs[64]: 2-bit quants, four per byte
 *   bytes 80..81  d    (fp16, little-endian)
 *   bytes 82..83  dmin (fp16, little-endian)
 * Weight j (0..255): half h = j/128, r = j%128, shift group g = r/32,
 * lane l = r%32; q_j = (qs[32h + l] >> 2g) & 3; sub-block s = j/16;
 *   w_j = d * (sc_s & 15) * q_j - dmin * (sc_s >> 4)      (fp32).
 * Both products are exact in fp32 (at most 17 significant bits), so the
 * only rounding is the final subtraction.
 * --------------------------------------------------------------------- */
void orc_q2k_dequant_block(const uint8_t *blk, float *w)
{
    const uint8_t *scales = blk;
    const uint8_t *qs = blk + 16;
    float d = (float)orc_half_to_double(rd16(blk + 80));
    float dmin = (float)orc_half_to_double(rd16(blk + 82));
    for (int j = 0; j < ORC_QK; ++j) {
        int h = j / 128;
        int r = j % 128;
        int g = r / 32;
        int l = r % 32;
        int q = (qs[32 * h + l] >> (2 * g)) & 3;
        int sc = scales[j / 16];
        float scale_part = d * (float)(sc & 15);
        float value = scale_part * (float)q;
        float min_part = dmin * (float)(sc >> 4);
        w[j] = value - min_part;
    }
}

/* ------------------------------------------------------------------------
 * Codebook-2-bit super-block (70 bytes, 256 weights), IQ2_XXS-style
 * (ds4 README mirror, "Model Weights": routed up/gate at IQ2_XXS):
 *   bytes  0..31  idx[32]: codebook row for weights 8o..8o+7
 *   bytes 32..63  sgn[32]: bit b of sgn[o] set => weight 8o+b is negated
 *   bytes 64..67  sc[4]:   4-bit scale of 32-weight group G in nibble
 *                          (G & 1) of byte G >> 1, low nibble first
 *   bytes 68..69  d (fp16, little-endian)
 * codebook: 256 rows x 8 int8 entries.
 *   w_j = d * s_{j/32} * cb[idx[j/8]][j%8] * (sign bit ? -1 : +1)   (fp32,
 * exact: at most 11 + 4 + 6 significant bits).
 * --------------------------------------------------------------------- */
void orc_cb2_dequant_block(const uint8_t *blk, const int8_t *codebook, float *w)
{
    const uint8_t *idx = blk;
    const uint8_t *sgn = blk + 32;
    const uint8_t *sc = blk + 64;
    float d = (float)orc_half_to_double(rd16(blk + 68));
    for (int j = 0; j < ORC_QK; ++j) {
        int group = j / 32;
        int scale = (sc[group / 2] >> (4 * (group % 2))) & 15;
        int o = j / 8;
        int b = j % 8;
        int entry = codebook[8 * idx[o] + b];
        int negate = (sgn[o] >> b) & 1;
        float value = d * (float)scale;
        value = value * (float)entry;
        w[j] = negate ? -value : value;
    }
}

/* ------------------------------------------------------------------------
 * The higher-bit routed-expert formats (ds4 README mirror, "Model Weights":
 * routed gate/up in Q2_K, Q4_K or Q5_K, routed down in Q2_K, Q4_K, Q5_K or
 * Q6_K), GGUF K-quant layouts (ds4 README mirror, "Acknowledgements to
 * llama.cpp and GGML").  256 weights per super-block in every case.
 *
 * Q4_K and Q5_K share the packed 6-bit scales: eight 32-weight sub-blocks,
 * each with a 6-bit scale sc_s and a 6-bit min m_s in 12 bytes p[0..11]:
 *   s < 4:  sc_s = p[s] & 63,                        m_s = p[s+4] & 63
 *   s >= 4: sc_s = (p[s+4] & 15) | (p[s-4] >> 6) << 4,
 *           m_s  = (p[s+4] >> 4) | (p[s]   >> 6) << 4
 * (the top two bits of sub-blocks 4..7 ride in the top bits of bytes 0..7).
 * --------------------------------------------------------------------- */
static void k4_scale_min(const uint8_t *p, int s, int *sc, int *m)
{
    if (s < 4) {
        *sc = p[s] & 63;
        *m = p[s + 4] & 63;
    } else {
        *sc = (p[s + 4] & 15) | ((p[s - 4] >> 6) << 4);
        *m = (p[s + 4] >> 4) | ((p[s] >> 6) << 4);
    }
}

/* Q4_K super-block (144 bytes):
 *   bytes  0..1   d    (fp16)        bytes 2..3  dmin (fp16)
 *   bytes  4..15  the packed 6-bit scales and mins above
 *   bytes 16..143 qs[128]: 4-bit quants
 * Weight j: chunk c = j/64 (two sub-blocks), r = j%64, l = r%32; the quant is
 * the low nibble of qs[32c + l] for r < 32 and its high nibble otherwise;
 * sub-block s = j/32;
 *   w_j = d * sc_s * q_j - dmin * m_s      (fp32).
 * Both products are exact in fp32 (at most 11 + 6 + 4 significant bits), so
 * the only rounding is the subtraction. */
void orc_q4k_dequant_block(const uint8_t *blk, float *w)
{
    float d = (float)orc_half_to_double(rd16(blk));
    float dmin = (float)orc_half_to_double(rd16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int j = 0; j < ORC_QK; ++j) {
        int c = j / 64, r = j % 64, l = r % 32, s = j / 32;
        int byte = qs[32 * c + l];
        int q = r < 32 ? (byte & 15) : (byte >> 4);
        int sc, m;
        k4_scale_min(scales, s, &sc, &m);
        float scale_part = d * (float)sc;
        float value = scale_part * (float)q;
        float min_part = dmin * (float)m;
        w[j] = value - min_part;
    }
}

/* Q5_K super-block (176 bytes): as Q4_K with a fifth bit per weight:
 *   bytes  0..1 d, 2..3 dmin, 4..15 packed scales and mins,
 *   bytes 16..47  qh[32]: bit s of qh[l] is the high bit of weight 32s + l,
 *   bytes 48..175 qs[128]: the low four bits, placed as in Q4_K.
 *   q_j = low_j + 16 * ((qh[j%32] >> (j/32)) & 1),
 *   w_j = d * sc_s * q_j - dmin * m_s      (fp32; products exact, at most
 * 11 + 6 + 5 significant bits). */
void orc_q5k_dequant_block(const uint8_t *blk, float *w)
{
    float d = (float)orc_half_to_double(rd16(blk));
    float dmin = (float)orc_half_to_double(rd16(blk + 2));
    const uint8_t *scales = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    for (int j = 0; j < ORC_QK; ++j) {
        int c = j / 64, r = j % 64, l = r % 32, s = j / 32;
        int byte = qs[32 * c + l];
        int low = r < 32 ? (byte & 15) : (byte >> 4);
        int q = low + 16 * ((qh[l] >> s) & 1);
        int sc, m;
        k4_scale_min(scales, s, &sc, &m);
        float scale_part = d * (float)sc;
        float value = scale_part * (float)q;
        float min_part = dmin * (float)m;
        w[j] = value - min_part;
    }
}

/* Q6_K super-block (210 bytes), symmetric, sixteen 16-weight sub-blocks:
 *   bytes   0..127 ql[128]: low four bits
 *   bytes 128..191 qh[64]:  high two bits
 *   bytes 192..207 scales[16]: int8 scale of sub-block j/16
 *   bytes 208..209 d (fp16)
 * Weight j: half h = j/128, r = j%128, quarter u = r/32, l = r%32;
 *   low  = nibble (u >> 1) of ql[64h + 32(u & 1) + l]   (0 = low nibble),
 *   high = (qh[32h + l] >> 2u) & 3,
 *   q_j  = low + 16 * high - 32                          (-32 .. 31),
 *   w_j  = d * scales[j/16] * q_j      (fp32, exact: the significands of d,
 * the scale and q multiply to less than 2^24). */
void orc_q6k_dequant_block(const uint8_t *blk, float *w)
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *scales = (const int8_t *)(blk + 192);
    float d = (float)orc_half_to_double(rd16(blk + 208));
    for (int j = 0; j < ORC_QK; ++j) {
        int h = j / 128, r = j % 128, u = r / 32, l = r % 32;
        int byte = ql[64 * h + 32 * (u & 1) + l];
        int low = (u >> 1) ? (byte >> 4) : (byte & 15);
        int high = (qh[32 * h + l] >> (2 * u)) & 3;
        int q = low + 16 * high - 32;
        float scale_part = d * (float)scales[j / 16];
        w[j] = scale_part * (float)q;
    }
}

/* ------------------------------------------------------------------------
 * MXFP4 routed experts (README "Model Weights": the ds4f-mxfp4 download keeps
 * DeepSeek's released MXFP4 routed-expert weights), read as the OCP
 * microscaling format in its GGUF block: 32 weights share one E8M0 scale.
 *   byte 0       e: scale 2^(e - 127) (e = 255 is NaN)
 *   bytes 1..16  qs: weight j (0..15) in the low nibble of qs[j], weight
 *                j + 16 in its high nibble; each nibble an E2M1 code: bit 3
 *                the sign, bits 0..2 the magnitude 0, 0.5, 1, 1.5, 2, 3, 4, 6
 *   w_j = 2^(e - 127) * value(code_j)       (fp32: a power of two times a
 *   value of at most 3 significant bits, exact unless it leaves fp32's range)
 * Eight blocks (136 bytes) make the 256-weight unit that rows are counted in.
 * --------------------------------------------------------------------- */
static double e2m1_value(int code)
{
    static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    double v = mag[code & 7];
    return (code & 8) ? -v : v;
}

void orc_mxfp4_dequant_block(const uint8_t *blk, float *w)
{
    for (int j = 0; j < ORC_QK; ++j) {
        const uint8_t *b = blk + (j / 32) * ORC_MX_BYTES;
        int r = j % 32;
        int byte = b[1 + r % 16];
        int code = r < 16 ? (byte & 15) : (byte >> 4);
        int e = b[0];
        double scale = e == 255 ? NAN : ldexp(1.0, e - 127);
        w[j] = (float)(scale * e2m1_value(code));
    }
}

void orc_mxfp4_dequant(const uint8_t *blocks, int64_t n_blocks, float *out)
{
    for (int64_t b = 0; b < n_blocks; ++b)
        orc_mxfp4_dequant_block(blocks + b * ORC_MXFP4_BYTES, out + b * ORC_QK);
}

void orc_q4k_dequant(const uint8_t *blocks, int64_t n_blocks, float *out)
{
    for (int64_t b = 0; b < n_blocks; ++b)
        orc_q4k_dequant_block(blocks + b * ORC_Q4K_BYTES, out + b * ORC_QK);
}

void orc_q5k_dequant(const uint8_t *blocks, int64_t n_blocks, float *out)
{
    for (int64_t b = 0; b < n_blocks; ++b)
        orc_q5k_dequant_block(blocks + b * ORC_Q5K_BYTES, out + b * ORC_QK);
}

void orc_q6k_dequant(const uint8_t *blocks, int64_t n_blocks, float *out)
{
    for (int64_t b = 0; b < n_blocks; ++b)
        orc_q6k_dequant_block(blocks + b * ORC_Q6K_BYTES, out + b * ORC_QK);
}

void orc_q2k_dequant(const uint8_t *blocks, int64_t n_blocks, float *out)
{
    for (int64_t b = 0; b < n_blocks; ++b)
        orc_q2k_dequant_block(blocks + b * ORC_Q2K_BYTES, out + b * ORC_QK);
}

void orc_cb2_dequant(const uint8_t *blocks, int64_t n_blocks,
                     const int8_t *codebook, float *out)
{
    for (int64_t b = 0; b < n_blocks; ++b)
        orc_cb2_dequant_block(blocks + b * ORC_CB2_BYTES, codebook, out + b * ORC_QK);
}

/* ------------------------------------------------------------------------
 * Routing: top-k over the router logits, then the weights of the k picks.
 * Rank: larger fp32 logit first; equal logits -> lower expert id first;
 * a NaN logit counts as -infinity, in the rank and in the weights.
 * Selection is made on the logit, not on
 * the transformed score: softmax and sigmoid are monotone, so the picks are
 * the same and exp rounding cannot change them.
 * Weights (fp64) over the k selected logits l_i:
 *   softmax:  w_i = exp(l_i - l_max) / sum_j exp(l_j - l_max)
 *   sigmoid:  s_i = 1 / (1 + exp(-l_i)),  w_i = s_i / sum_j s_j
 * --------------------------------------------------------------------- */
static double rank_value(float l) { return (l != l) ? -INFINITY : (double)l; }

static int ranks_before(float la, int ia, float lb, int ib)
{
    double a = rank_value(la), b = rank_value(lb);
    if (a > b) return 1;
    if (a < b) return 0;
    return ia < ib;
}

/* Selects the k experts of one token and their weights. */
static void route_one(const float *lg, int E, int k, int score,
                      int32_t *ids, double *w)
{
    char used[256];
    memset(used, 0, sizeof used);
    for (int i = 0; i < k; ++i) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (used[e]) continue;
            if (best < 0 || ranks_before(lg[e], e, lg[best], best)) best = e;
        }
        ids[i] = best;
        used[best] = 1;
    }
    if (score == ORC_SCORE_SOFTMAX) {
        double lmax = rank_value(lg[ids[0]]);
        double sum = 0.0;
        for (int i = 0; i < k; ++i) {
            w[i] = exp(rank_value(lg[ids[i]]) - lmax);
            sum += w[i];
        }
        for (int i = 0; i < k; ++i) w[i] /= sum;
    } else {
        double sum = 0.0;
        for (int i = 0; i < k; ++i) {
            w[i] = 1.0 / (1.0 + exp(-rank_value(lg[ids[i]])));
            sum += w[i];
        }
        for (int i = 0; i < k; ++i) w[i] /= sum;
    }
}

/* Full routing of T tokens.
 *   ids[T*k], weights[T*k]        per token, in rank order
 *   counts[E]                     assignments per expert
 *   offsets[E+1]                  exclusive prefix sum of counts
 *   perm[T*k]                     assignments a = t*k + i grouped by expert
 *                                 (segment e = perm[offsets[e]..offsets[e+1]]),
 *                                 ascending t inside a segment
 * Any output pointer except ids/weights may be NULL. */
int orc_route(const float *logits, int T, int E, int k, int score,
              int32_t *ids, double *weights, int32_t *counts,
              int32_t *offsets, int32_t *perm)
{
    if (T < 0 || E < 1 || E > 256 || k < 1 || k > E || !logits || !ids || !weights)
        return ORC_ERR_INVALID;
    if (score != ORC_SCORE_SOFTMAX && score != ORC_SCORE_SIGMOID)
        return ORC_ERR_INVALID;
    for (int t = 0; t < T; ++t)
        route_one(logits + (int64_t)t * E, E, k, score, ids + (int64_t)t * k,
                  weights + (int64_t)t * k);
    if (counts) {
        for (int e = 0; e < E; ++e) counts[e] = 0;
        for (int64_t a = 0; a < (int64_t)T * k; ++a) counts[ids[a]] += 1;
    }
    if (offsets) {
        int32_t run = 0;
        for (int e = 0; e < E; ++e) {
            int32_t c = 0;
            for (int64_t a = 0; a < (int64_t)T * k; ++a) c += (ids[a] == e);
            offsets[e] = run;
            run += c;
        }
        offsets[E] = run;
    }
    if (perm) {
        int64_t pos = 0;
        for (int e = 0; e < E; ++e)
            for (int t = 0; t < T; ++t)
                for (int i = 0; i < k; ++i)
                    if (ids[(int64_t)t * k + i] == e) perm[pos++] = t * k + i;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------
 * The layer.
 * A quantized matrix [N rows x K] is N rows of ceil(K/256) super-blocks;
 * row n starts at n * row_bytes, expert e at e * expert_stride.  Weight
 * (n, kk) is element kk % 256 of block kk / 256 of row n.  Weights at
 * kk >= K (padding of the last block) are ignored.
 * --------------------------------------------------------------------- */
typedef struct {
    int32_t hidden, inter, n_experts, top_k, score;
    int32_t format;         /* W_gate and W_up                                  */
    int32_t down_format;    /* W_down (the shipping mix: codebook up/gate, Q2_K
                               down -- ds4 README mirror, "Model Weights")      */
    const uint8_t *w_gate, *w_up, *w_down;
    int64_t gate_up_row_bytes, down_row_bytes;
    int64_t gate_up_expert_stride, down_expert_stride;
    const int8_t *codebook;
} orc_layer;

/* Supported formats per matrix (ds4 README mirror, "Model Weights": routed
 * gate/up in Q2_K, Q4_K or Q5_K, routed down also in Q6_K; the codebook
 * format for either); a codebook present when either matrix uses it. */
static int orc_formats_ok(const orc_layer *L)
{
    if (L->format != ORC_FMT_Q2K && L->format != ORC_FMT_CB2 && L->format != ORC_FMT_Q4K &&
        L->format != ORC_FMT_Q5K && L->format != ORC_FMT_MXFP4)
        return 0;
    if (L->down_format != ORC_FMT_Q2K && L->down_format != ORC_FMT_CB2 &&
        L->down_format != ORC_FMT_Q4K && L->down_format != ORC_FMT_Q5K &&
        L->down_format != ORC_FMT_Q6K && L->down_format != ORC_FMT_MXFP4)
        return 0;
    if ((L->format == ORC_FMT_CB2 || L->down_format == ORC_FMT_CB2) && !L->codebook) return 0;
    return 1;
}

/* Dequantizes one row of K logical weights (ceil(K/256) blocks of format
 * fmt) to fp32. */
static void dequant_row(const orc_layer *L, int fmt, const uint8_t *row, int K, float *out)
{
    int nblk = (K + ORC_QK - 1) / ORC_QK;
    for (int b = 0; b < nblk; ++b) {
        if (fmt == ORC_FMT_Q2K)
            orc_q2k_dequant_block(row + (int64_t)b * ORC_Q2K_BYTES, out + b * ORC_QK);
        else if (fmt == ORC_FMT_CB2)
            orc_cb2_dequant_block(row + (int64_t)b * ORC_CB2_BYTES, L->codebook,
                                  out + b * ORC_QK);
        else if (fmt == ORC_FMT_Q4K)
            orc_q4k_dequant_block(row + (int64_t)b * ORC_Q4K_BYTES, out + b * ORC_QK);
        else if (fmt == ORC_FMT_Q5K)
            orc_q5k_dequant_block(row + (int64_t)b * ORC_Q5K_BYTES, out + b * ORC_QK);
        else if (fmt == ORC_FMT_MXFP4)
            orc_mxfp4_dequant_block(row + (int64_t)b * ORC_MXFP4_BYTES, out + b * ORC_QK);
        else
            orc_q6k_dequant_block(row + (int64_t)b * ORC_Q6K_BYTES, out + b * ORC_QK);
    }
}

/* SiLU-gated FFN of one expert on one token, fp64:
 *   g_n = sum_kk Wg[n,kk] x_kk,  u_n = sum_kk Wu[n,kk] x_kk   (n < I)
 *   h_n = g_n / (1 + exp(-g_n)) * u_n
 *   o_m = sum_n Wd[m,n] h_n                                     (m < H)  */
static void expert_ffn(const orc_layer *L, int e, const double *x, double *o,
                       float *rowbuf, double *h)
{
    const int H = L->hidden, I = L->inter;
    const uint8_t *wg = L->w_gate + (int64_t)e * L->gate_up_expert_stride;
    const uint8_t *wu = L->w_up + (int64_t)e * L->gate_up_expert_stride;
    const uint8_t *wd = L->w_down + (int64_t)e * L->down_expert_stride;
    for (int n = 0; n < I; ++n) {
        double g = 0.0, u = 0.0;
        dequant_row(L, L->format, wg + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);
        for (int kk = 0; kk < H; ++kk) g += (double)rowbuf[kk] * x[kk];
        dequant_row(L, L->format, wu + (int64_t)n * L->gate_up_row_bytes, H, rowbuf);
        for (int kk = 0; kk < H; ++kk) u += (double)rowbuf[kk] * x[kk];
        h[n] = g / (1.0 + exp(-g)) * u;
    }
    for (int m = 0; m < H; ++m) {
        double acc = 0.0;
        dequant_row(L, L->down_format, wd + (int64_t)m * L->down_row_bytes, I, rowbuf);
        for (int n = 0; n < I; ++n) acc += (double)rowbuf[n] * h[n];
        o[m] = acc;
    }
}

/* Forward pass for a subset of tokens (all tokens when tokens == NULL):
 *   y[j, m] = sum_{i<k} w[t,i] * o_{t,i}[m],  t = tokens[j], summed in
 *   slot order i = 0..k-1.
 * x: [T x H] bf16 bits; logits: [T x E] fp32; y: [n_tokens x H] fp64.
 * ids_out / w_out (optional): [n_tokens x k]. */
int orc_moe_forward(const orc_layer *L, const uint16_t *x, const float *logits,
                    int T, const int32_t *tokens, int n_tokens, double *y,
                    int32_t *ids_out, double *w_out)
{
    if (!L || !x || !logits || !y || T < 0) return ORC_ERR_INVALID;
    const int H = L->hidden, I = L->inter, E = L->n_experts, k = L->top_k;
    if (H < 1 || I < 1 || E < 1 || E > 256 || k < 1 || k > E) return ORC_ERR_INVALID;
    if (!orc_formats_ok(L)) return ORC_ERR_INVALID;
    if (!tokens) n_tokens = T;
    int kmax = H > I ? H : I;
    int kpad = ((kmax + ORC_QK - 1) / ORC_QK) * ORC_QK;
    float *rowbuf = (float *)malloc(sizeof(float) * kpad);
    double *xt = (double *)malloc(sizeof(double) * H);
    double *h = (double *)malloc(sizeof(double) * I);
    double *o = (double *)malloc(sizeof(double) * H);
    int32_t ids[256];
    double w[256];
    int rc = ORC_OK;
    if (!rowbuf || !xt || !h || !o) { rc = ORC_ERR_NOMEM; goto done; }
    for (int j = 0; j < n_tokens; ++j) {
        int t = tokens ? tokens[j] : j;
        if (t < 0 || t >= T) { rc = ORC_ERR_INVALID; goto done; }
        route_one(logits + (int64_t)t * E, E, k, L->score, ids, w);
        for (int kk = 0; kk < H; ++kk) xt[kk] = orc_bf16_to_double(x[(int64_t)t * H + kk]);
        double *yt = y + (int64_t)j * H;
        for (int m = 0; m < H; ++m) yt[m] = 0.0;
        for (int i = 0; i < k; ++i) {
            expert_ffn(L, ids[i], xt, o, rowbuf, h);
            for (int m = 0; m < H; ++m) yt[m] += w[i] * o[m];
        }
        if (ids_out) memcpy(ids_out + (int64_t)j * k, ids, sizeof(int32_t) * k);
        if (w_out) memcpy(w_out + (int64_t)j * k, w, sizeof(double) * k);
    }
done:
    free(rowbuf);
    free(xt);
    free(h);
    free(o);
    return rc;
}

/* Single-expert SiLU FFN on one token, exposed for the reduction pins
 * (k = 1 layer == one dense FFN). x: [H] bf16 bits; o: [H] fp64. */
int orc_expert_ffn(const orc_layer *L, int e, const uint16_t *x, double *o)
{
    if (!L || !x || !o || e < 0 || e >= L->n_experts) return ORC_ERR_INVALID;
    if (!orc_formats_ok(L)) return ORC_ERR_INVALID;
    const int H = L->hidden, I = L->inter;
    int kmax = H > I ? H : I;
    int kpad = ((kmax + ORC_QK - 1) / ORC_QK) * ORC_QK;
    float *rowbuf = (float *)malloc(sizeof(float) * kpad);
    double *xt = (double *)malloc(sizeof(double) * H);
    double *h = (double *)malloc(sizeof(double) * I);
    int rc = ORC_OK;
    if (!rowbuf || !xt || !h) { rc = ORC_ERR_NOMEM; goto done; }
    for (int kk = 0; kk < H; ++kk) xt[kk] = orc_bf16_to_double(x[kk]);
    expert_ffn(L, e, xt, o, rowbuf, h);
done:
    free(rowbuf);
    free(xt);
    free(h);
    return rc;
}
