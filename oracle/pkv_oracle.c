/*
 * pkv_oracle.c -- plain fp64 CPU oracle for paged, prefix-cached KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference the CUDA
 * library is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or constant with the CUDA library and includes nothing from it.
 *
 * What it computes (sources are the web pages the method is described on):
 *
 *  - KV append ("KV 写入"): each new token's K and V row is stored at the
 *    physical slot the caller assigns it.  Page "vLLM Agentic 推理｜面向 Agent
 *    负载的推理优化", section 5.2 (每层两个 Kernel, K1 writes the KV).
 *  - Block addressing: a request of n tokens owns cdiv(n, block_size) blocks,
 *    listed in its block table.  Page "vLLM/V1 推理调度器", section 源码片段
 *    (KVCacheManager.allocate_slots, block capacity).
 *  - Incremental prefill: l_incr new query tokens attend to the l_hist cached
 *    history tokens and to themselves; decode is the case l_incr = 1.  Page
 *    "AMPD：PD 分离遇上多轮推理，incremental prefill 到底该在哪跑", sections 1
 *    and 3.
 *  - GQA: a few KV heads are shared by groups of query heads.  Page "vLLM
 *    Agentic 推理", section 4.3.1.
 *  - Partial results over disjoint key sets merge through their log-sum-exp.
 *    Page "vLLM Agentic 推理", section 4.3.3 (step 4, online-softmax merge).
 *  - Rotary position embedding applied to q and to K before the KV write
 *    (the pages' first per-layer kernel does both: page "vLLM Agentic 推理",
 *    section 5.2, K1).  The pages do not define RoPE; the reading taken is
 *    the usual one: the 64 pairs of a 128-wide head rotate by the angle whose
 *    cosine and sine the caller's table gives for the token's position, pairs
 *    (i, i + 64) ("neox") or (2i, 2i + 1).
 *  - Decode context parallelism: a request's KV tokens are dealt out to N
 *    ranks in runs of `interleave` tokens (interleave 1: token i on rank
 *    i % N); each rank attends to its own tokens only.  Page "vLLM Agentic
 *    推理", sections 4.3.1 and 4.3.3 (step 3).
 *
 * The pages never print the attention formula.  The reading taken here is
 * the plain one: scaled dot-product softmax attention, key j visible to the
 * query at logical position pos iff j <= pos, query token t of a sequence with
 * context length L and q new tokens sitting at position (L - q) + t, query
 * head h reading KV head h / G (G = query heads per KV head).  All arithmetic
 * on attention values is fp64; bf16 inputs are widened exactly.
 *
 * FP8 KV uses the OCP 8-bit floating point format E4M3 ("FN" variant: bias 7,
 * no infinities, S.1111.111 is NaN, largest finite 448), with one fp32 scale
 * per (block, KV head).  Stored codes are decoded exactly: value = e4m3(code)
 * * scale.  Quantisation on append divides in fp32 and rounds to nearest,
 * ties to even, saturating at +-448.
 *
 * NVFP4 KV (the compressed KV format the pages name, nearly half the size
 * of FP8: page "vLLM 优化 DeepSeek-V4.1-Flash：智能体吞吐提升 5 倍", section
 * Kernels, MegaAttention with NVFP4 KV) is read here as: OCP FP4 E2M1 element codes (sign, two exponent bits
 * with bias 1, one mantissa bit; largest 6, no infinities or NaN), two per
 * byte, low nibble first; one E4M3 scale per 16 consecutive elements of a
 * row; and the per-(block, KV head) fp32 scale as the second level.  An
 * element's value is e2m1(code) * e4m3(micro scale) * scale.  Quantisation
 * (the reading taken; the pages give none): amax = largest |x| of the 16
 * values, micro scale = E4M3(amax / (6 * scale)), and, unless that micro
 * scale is zero (then every code is 0), code = E2M1(x / (scale * micro
 * scale)), every product and quotient rounded to fp32, E2M1 rounding to
 * nearest with ties to even and saturating at +-6.
 *
 * Pool layout: [num_blocks][num_kv_heads][block_size][head_dim], so slot s of
 * KV head h is row ((s / bs) * Hkv + h) * bs + s % bs.  NVFP4 pools hold,
 * per (block, KV head), the block's rows in groups of min(block_size, 64)
 * rows (block_size <= 64 or a multiple of 64): a group is its rows' code
 * bytes (head_dim / 2 per row) followed by their micro-scale bytes
 * (head_dim / 16 per row).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PKO_OK 0
#define PKO_BAD_ARG 1
#define PKO_NO_MEM 2

/* ---- number formats -------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double pko_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a real number to bf16 (8 significant bits, binary32 exponent
 * range), to nearest, ties to even; returns the bf16 bit pattern.  Values
 * at or beyond the largest finite bf16 plus half an ulp become infinities. */
uint16_t pko_bf16_round(double v)
{
    if (isnan(v))
        return 0x7FC0;
    double a = fabs(v);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);                       /* a = f * 2^e, f in [0.5, 1) */
        int ulp_exp = e - 8;                /* 8 significant bits */
        if (ulp_exp < -133)                 /* below the smallest normal: fixed quantum */
            ulp_exp = -133;
        double q = ldexp(1.0, ulp_exp);
        double n = a / q;                   /* exact: q is a power of two */
        double fl = floor(n), fr = n - fl;
        double k = fr > 0.5 ? fl + 1.0 : fr < 0.5 ? fl : (fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0);
        r = k * q;
    }
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    if (r >= ldexp(1.0, 128))
        return sign | 0x7F80;
    float f = (float)r;                     /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | (u >> 16));
}

/* OCP E4M3 decode, written from the format definition. */
double pko_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^-6 */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* Round a real number to the nearest integer, ties to even. */
static double round_half_even(double x)
{
    double f = floor(x);
    double r = x - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* OCP E4M3 encode: round to nearest even, saturate finite values to +-448,
 * NaN -> 0x7F (sign kept). */
uint8_t pko_e4m3_encode(float xf)
{
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isnan(x))
        return (uint8_t)(sign | 0x7F);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);           /* 1.75 * 2^8 */
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; m == 8 is the smallest normal,
         * whose code (exponent field 1, mantissa 0) is also 8 */
        double m = round_half_even(ldexp(a, 9));
        return (uint8_t)(sign | (uint8_t)m);
    }
    int e;
    double fr = frexp(a, &e);                    /* a = fr * 2^e, fr in [0.5,1) */
    e -= 1;                                      /* a = (2*fr) * 2^e */
    double mant = round_half_even((2.0 * fr - 1.0) * 8.0);
    if (mant >= 8.0) {
        mant = 0.0;
        e += 1;
    }
    int field = e + 7;
    if (field > 15 || (field == 15 && mant > 6.0))
        return (uint8_t)(sign | 0x7E);
    return (uint8_t)(sign | (uint8_t)(field << 3) | (uint8_t)mant);
}

/* Quantise one bf16 value with a per-(block, KV head) scale: the quotient is
 * formed in fp32 (one correctly rounded division), then encoded. */
uint8_t pko_e4m3_quantize(uint16_t x_bf16, float scale)
{
    uint32_t u = (uint32_t)x_bf16 << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    volatile float q = x / scale;
    return pko_e4m3_encode(q);
}

/* OCP FP4 E2M1 decode of the low 4 bits of `code`, written from the format
 * definition: exponent field 0 is subnormal (0.m * 2^0), else 1.m * 2^(e-1). */
double pko_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* E2M1 encode: round to nearest, ties to even, saturate at +-6; NaN -> 0
 * (sign kept).  The grid has spacing 1/2 below 2, 1 in [2, 4) and 2 in
 * [4, 6]; on each range the code is an offset plus the rounded multiple, and
 * an even multiple is an even code. */
uint8_t pko_e2m1_encode(float xf)
{
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    double a = fabs(x);
    if (isnan(x))
        return sign;
    if (a >= 6.0)
        return (uint8_t)(sign | 0x7);
    if (a < 2.0)
        return (uint8_t)(sign | (uint8_t)round_half_even(2.0 * a));
    if (a < 4.0)
        return (uint8_t)(sign | (uint8_t)(round_half_even(a) + 2.0));
    return (uint8_t)(sign | (uint8_t)(round_half_even(0.5 * a) + 4.0));
}

static float bf16_to_float(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* NVFP4 quantisation of one row of d bf16 values (d a multiple of 16) with
 * the (block, KV head) scale: d/2 code bytes to `codes` (element 2j in the
 * low nibble of byte j), d/16 E4M3 micro scales to `mscale`. */
void pko_nvfp4_quantize_row(const uint16_t *x, int d, float scale, uint8_t *codes,
                            uint8_t *mscale)
{
    for (int b = 0; b < d / 16; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 16; ++i) {
            float a = fabsf(bf16_to_float(x[16 * b + i]));
            if (a > amax)                        /* NaN never compares greater */
                amax = a;
        }
        volatile float six_s = 6.0f * scale;
        volatile float ratio = amax / six_s;
        uint8_t ms = pko_e4m3_encode(ratio);
        mscale[b] = ms;
        double msv = pko_e4m3_value(ms);
        for (int i = 0; i < 16; i += 2) {
            uint8_t c[2] = {0, 0};
            if (msv != 0.0) {
                volatile float step = scale * (float)msv;   /* msv is exact in fp32 */
                for (int k = 0; k < 2; ++k) {
                    volatile float qv = bf16_to_float(x[16 * b + i + k]) / step;
                    c[k] = pko_e2m1_encode(qv);
                }
            }
            codes[(16 * b + i) / 2] = (uint8_t)(c[0] | (c[1] << 4));
        }
    }
}

/* Byte offsets, inside its (block, KV head) tile, of the codes and of the
 * micro scales of row `off` of an NVFP4 pool (groups of min(bs, 64) rows). */
static void nvfp4_offsets(int bs, int d, int64_t off, size_t *codes, size_t *mscale)
{
    int64_t gs = bs < 64 ? bs : 64;
    size_t group = (size_t)(off / gs) * (size_t)gs * (size_t)(d / 2 + d / 16);
    int64_t r = off % gs;
    *codes = group + (size_t)r * (d / 2);
    *mscale = group + (size_t)gs * (d / 2) + (size_t)r * (d / 16);
}

/* ---- KV append --------------------------------------------------------- */

/*
 * For every new token t with slot_mapping[t] >= 0, copy its K and V rows of
 * every KV head into the pool at that slot.  bf16 pools receive the bits
 * unchanged; FP8 pools receive pko_e4m3_quantize(x, scale[block][head]);
 * NVFP4 pools (kv_fmt 2) the codes and micro scales of
 * pko_nvfp4_quantize_row with that scale.
 * Returns PKO_BAD_ARG (and writes nothing further) on a slot past the pool.
 */
int pko_write_slots(int kv_fmt, int64_t num_tokens, int hkv, int d, int bs,
                    int64_t num_blocks, const uint16_t *k_new,
                    const uint16_t *v_new, const int64_t *slot_mapping,
                    void *k_cache, void *v_cache, const float *k_scale,
                    const float *v_scale)
{
    if (num_tokens < 0 || hkv <= 0 || d <= 0 || bs <= 0 || num_blocks < 0 ||
        kv_fmt < 0 || kv_fmt > 2 ||
        (kv_fmt == 2 && (d % 16 != 0 || (bs > 64 && bs % 64 != 0))))
        return PKO_BAD_ARG;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        int64_t blk = slot / bs;
        int64_t off = slot % bs;
        if (blk >= num_blocks)
            return PKO_BAD_ARG;
        for (int h = 0; h < hkv; ++h) {
            const uint16_t *ks = k_new + ((size_t)t * hkv + h) * d;
            const uint16_t *vs = v_new + ((size_t)t * hkv + h) * d;
            size_t row = ((size_t)blk * hkv + h) * bs + off;
            if (kv_fmt == 2) {
                size_t tile = ((size_t)blk * hkv + h) * (size_t)bs * (size_t)(d / 2 + d / 16);
                size_t codes, msc;
                nvfp4_offsets(bs, d, off, &codes, &msc);
                codes += tile;
                msc += tile;
                float sk = k_scale[(size_t)blk * hkv + h];
                float sv = v_scale[(size_t)blk * hkv + h];
                pko_nvfp4_quantize_row(ks, d, sk, (uint8_t *)k_cache + codes,
                                       (uint8_t *)k_cache + msc);
                pko_nvfp4_quantize_row(vs, d, sv, (uint8_t *)v_cache + codes,
                                       (uint8_t *)v_cache + msc);
            } else if (!kv_fmt) {
                memcpy((uint16_t *)k_cache + row * d, ks, (size_t)d * 2);
                memcpy((uint16_t *)v_cache + row * d, vs, (size_t)d * 2);
            } else {
                float sk = k_scale[(size_t)blk * hkv + h];
                float sv = v_scale[(size_t)blk * hkv + h];
                uint8_t *kd = (uint8_t *)k_cache + row * d;
                uint8_t *vd = (uint8_t *)v_cache + row * d;
                for (int i = 0; i < d; ++i) {
                    kd[i] = pko_e4m3_quantize(ks[i], sk);
                    vd[i] = pko_e4m3_quantize(vs[i], sv);
                }
            }
        }
    }
    return PKO_OK;
}

/* ---- attention ------------------------------------------------------------ */

typedef struct {
    int kv_fmt;                 /* 0 bf16, 1 E4M3, 2 NVFP4 */
    const void *k_cache, *v_cache;
    const float *k_scale, *v_scale;
    int hkv, d, bs;
    int64_t num_blocks;
} pool_t;

/* Value of element i of the key (or value) row at logical position j of a
 * sequence whose block table is bt. */
static double pool_elem(const pool_t *p, int is_v, const int32_t *bt,
                        int64_t j, int kvh, int i)
{
    int64_t blk = bt[j / p->bs];
    size_t off = (size_t)(j % p->bs);
    size_t row = ((size_t)blk * p->hkv + kvh) * p->bs + off;
    const void *base = is_v ? p->v_cache : p->k_cache;
    if (!p->kv_fmt)
        return pko_bf16_value(((const uint16_t *)base)[row * p->d + i]);
    const float *sc = is_v ? p->v_scale : p->k_scale;
    if (p->kv_fmt == 2) {
        const uint8_t *tile = (const uint8_t *)base +
            ((size_t)blk * p->hkv + kvh) * (size_t)p->bs * (size_t)(p->d / 2 + p->d / 16);
        size_t co, mo;
        nvfp4_offsets(p->bs, p->d, (int64_t)off, &co, &mo);
        uint8_t byte = tile[co + i / 2];
        uint8_t code = (i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
        uint8_t ms = tile[mo + i / 16];
        return pko_e2m1_value(code) * pko_e4m3_value(ms) *
               (double)sc[(size_t)blk * p->hkv + kvh];
    }
    return pko_e4m3_value(((const uint8_t *)base)[row * p->d + i]) *
           (double)sc[(size_t)blk * p->hkv + kvh];
}

/*
 * Attention for one (query token, query head) over the keys j in
 * [k_lo, k_hi) of sequence i that the causal rule lets it see.  Writes the
 * softmax-weighted mean of V over those keys to out[0..d) and the natural
 * log-sum-exp of the scaled scores to *lse.  With no visible key the result
 * is out = 0, lse = -inf (the identity of the merge).
 */
/* Does context-parallel rank r of n own key j (runs of k tokens dealt out
 * in turn)?  n <= 1: every key. */
static int owns_key(int64_t j, int64_t n, int64_t r, int64_t k)
{
    return n <= 1 || (j / k) % n == r;
}

static int attend_one(const pool_t *p, const uint16_t *qrow, const int32_t *bt,
                      int64_t pos, int kvh, double softmax_scale, int64_t k_lo,
                      int64_t k_hi, int64_t sn, int64_t sr, int64_t sk,
                      double *scores, double *out, double *lse)
{
    int64_t hi = k_hi < pos + 1 ? k_hi : pos + 1; /* causal: j <= pos */
    int d = p->d;
    for (int i = 0; i < d; ++i)
        out[i] = 0.0;
    if (hi <= k_lo) {
        *lse = -INFINITY;
        return 0;
    }
    double m = -INFINITY;
    for (int64_t j = k_lo; j < hi; ++j) {
        if (!owns_key(j, sn, sr, sk))
            continue;
        double s = 0.0;
        for (int i = 0; i < d; ++i)
            s += pko_bf16_value(qrow[i]) * pool_elem(p, 0, bt, j, kvh, i);
        s *= softmax_scale;
        scores[j - k_lo] = s;
        if (s > m)
            m = s;
    }
    if (m == -INFINITY) { /* no owned key is visible */
        *lse = -INFINITY;
        return 0;
    }
    double l = 0.0;
    for (int64_t j = k_lo; j < hi; ++j) {
        if (!owns_key(j, sn, sr, sk))
            continue;
        double w = exp(scores[j - k_lo] - m);
        l += w;
        for (int i = 0; i < d; ++i)
            out[i] += w * pool_elem(p, 1, bt, j, kvh, i);
    }
    for (int i = 0; i < d; ++i)
        out[i] /= l;
    *lse = m + log(l);
    return 0;
}

/*
 * Varlen paged attention.  Sequence i owns query tokens
 * [qsl[i], qsl[i+1]) of q ([T][hq][d] bf16 bits) and has seq_lens[i] context
 * tokens including those new ones; its block table is
 * block_tables[i * bt_stride ...].  Keys are restricted to [k_lo, k_hi) in
 * logical position (k_lo = 0, k_hi = INT64_MAX for full attention), and to
 * the keys context-parallel rank shard_r of shard_n owns with runs of
 * shard_k tokens (shard_n <= 1: no restriction).
 *
 * rows: indices (token * hq + head) to evaluate, or NULL for all T*hq rows in
 * order.  out receives nrows * d doubles, lse nrows doubles.
 */
int pko_attention(int kv_fmt, const void *k_cache, const void *v_cache,
                  const float *k_scale, const float *v_scale,
                  int64_t num_blocks, int hkv, int d, int bs, int hq,
                  const uint16_t *q, const int32_t *qsl,
                  const int32_t *seq_lens, const int32_t *block_tables,
                  int64_t bt_stride, int num_seqs, int64_t num_tokens,
                  double softmax_scale, int64_t k_lo, int64_t k_hi,
                  int64_t shard_n, int64_t shard_r, int64_t shard_k,
                  const int64_t *rows, int64_t nrows, double *out,
                  double *lse)
{
    if (hkv <= 0 || hq <= 0 || hq % hkv != 0 || d <= 0 || bs <= 0 ||
        num_seqs < 0 || num_tokens < 0 || kv_fmt < 0 || kv_fmt > 2 ||
        (kv_fmt == 2 && (d % 16 != 0 || (bs > 64 && bs % 64 != 0))))
        return PKO_BAD_ARG;
    if (shard_n > 1 && (shard_r < 0 || shard_r >= shard_n || shard_k < 1))
        return PKO_BAD_ARG;
    if (qsl[0] != 0 || qsl[num_seqs] != num_tokens)
        return PKO_BAD_ARG;
    for (int i = 0; i < num_seqs; ++i) {
        int64_t qi = (int64_t)qsl[i + 1] - qsl[i];
        if (qi < 0 || qi > seq_lens[i])
            return PKO_BAD_ARG;
        int64_t nb = (seq_lens[i] + bs - 1) / bs;   /* cdiv */
        if (nb > bt_stride)
            return PKO_BAD_ARG;
        for (int64_t b = 0; b < nb; ++b) {
            int32_t id = block_tables[i * bt_stride + b];
            if (id < 0 || id >= num_blocks)
                return PKO_BAD_ARG;
        }
    }
    if (rows == NULL)
        nrows = num_tokens * hq;
    pool_t p = {kv_fmt, k_cache, v_cache, k_scale, v_scale, hkv, d, bs,
                num_blocks};
    int group = hq / hkv;
    int64_t max_len = 0;
    for (int i = 0; i < num_seqs; ++i)
        if (seq_lens[i] > max_len)
            max_len = seq_lens[i];
    int status = PKO_OK;

#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(max_len + 1));
        if (!scores) {
#pragma omp atomic write
            status = PKO_NO_MEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!scores)
                continue;
            int64_t idx = rows ? rows[r] : r;
            int64_t tok = idx / hq;
            int head = (int)(idx % hq);
            int i = 0;
            while (i < num_seqs && qsl[i + 1] <= tok)
                ++i;
            int64_t qi = (int64_t)qsl[i + 1] - qsl[i];
            int64_t t = tok - qsl[i];
            int64_t hist = (int64_t)seq_lens[i] - qi;
            int64_t pos = hist + t;
            attend_one(&p, q + ((size_t)tok * hq + head) * d,
                       block_tables + (size_t)i * bt_stride, pos, head / group,
                       softmax_scale, k_lo, k_hi, shard_n, shard_r, shard_k,
                       scores, out + (size_t)r * d,
                       lse + r);
        }
        free(scores);
    }
    return status;
}

/*
 * Rotary position embedding of rows x [n][heads][d] (bf16 bits), token t
 * at position positions[t]: for pair (a, b) with angle index i,
 *   y_a = x_a cos_i - x_b sin_i,  y_b = x_b cos_i + x_a sin_i,
 * cos_i = cos_sin[p * d + i], sin_i = cos_sin[p * d + d/2 + i]; pairs are
 * (i, i + d/2) when neox, else (2i, 2i + 1).  fp64 arithmetic; out_f64
 * (optional) receives y, out_bits (optional) y rounded to bf16.
 */
int pko_rope(int64_t n, int heads, int d, const uint16_t *x, const int64_t *positions,
             const float *cos_sin, int64_t max_pos, int neox, double *out_f64,
             uint16_t *out_bits)
{
    if (n < 0 || heads <= 0 || d <= 0 || d % 2 != 0)
        return PKO_BAD_ARG;
    int half = d / 2;
    for (int64_t t = 0; t < n; ++t) {
        int64_t p = positions[t];
        if (p < 0 || p >= max_pos)
            return PKO_BAD_ARG;
        const float *cs = cos_sin + (size_t)p * d;
        for (int h = 0; h < heads; ++h) {
            const uint16_t *row = x + ((size_t)t * heads + h) * d;
            size_t o = ((size_t)t * heads + h) * d;
            for (int i = 0; i < half; ++i) {
                int a = neox ? i : 2 * i;
                int b = neox ? i + half : 2 * i + 1;
                double xa = pko_bf16_value(row[a]), xb = pko_bf16_value(row[b]);
                double c = cs[i], s = cs[half + i];
                double ya = xa * c - xb * s;
                double yb = xb * c + xa * s;
                if (out_f64) {
                    out_f64[o + a] = ya;
                    out_f64[o + b] = yb;
                }
                if (out_bits) {
                    out_bits[o + a] = pko_bf16_round(ya);
                    out_bits[o + b] = pko_bf16_round(yb);
                }
            }
        }
    }
    return PKO_OK;
}

/*
 * Merge partial results computed over disjoint key sets: with partial
 * (o_s, lse_s), lse = ln sum_s exp(lse_s) and o = sum_s exp(lse_s - lse) o_s.
 * Parts with lse_s = -inf contribute nothing.
 */
void pko_lse_merge(int nparts, int d, const double *lse_parts,
                   const double *o_parts, double *o, double *lse)
{
    double m = -INFINITY;
    for (int s = 0; s < nparts; ++s)
        if (lse_parts[s] > m)
            m = lse_parts[s];
    for (int i = 0; i < d; ++i)
        o[i] = 0.0;
    if (m == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int s = 0; s < nparts; ++s)
        sum += exp(lse_parts[s] - m);
    double total = m + log(sum);
    for (int s = 0; s < nparts; ++s) {
        double w = exp(lse_parts[s] - total);
        for (int i = 0; i < d; ++i)
            o[i] += w * o_parts[(size_t)s * d + i];
    }
    *lse = total;
}

int pko_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
