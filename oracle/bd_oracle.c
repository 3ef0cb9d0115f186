/*
 * bd_oracle.c -- plain CPU oracle for the NVFP4 KV-cache page writer, the
 * two-term FP4 query quantizer and the paged FP4 decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path; the two meet only in
 * the byte layout that the public header documents, which each side writes on
 * its own.
 *
 * Arithmetic: every quantizer step is one IEEE-754 binary32 operation with
 * round-to-nearest-even (build with -ffp-contract=off -fno-fast-math so that
 * no multiply-add is fused), because the packed bytes must be reproducible
 * exactly.  The attention itself is evaluated in binary64 on the same
 * quantized operands.
 *
 * Sources (cited by page title and section):
 *  [cfg]  BitDecoding-FP4 "evaluation/config.py": RECIPE,
 *         recipe_additional_config, probability_environment, KV_MODES
 *         ("bitdecoding-nvfp4" / "bitdecoding-mxfp4"), PARITY_ENGINE_KWARGS.
 *  [ab]   kv-landlords "scripts/quant_ab.py": module docstring (freeze-at-fill
 *         pages, BF16 hot page), mem_ratio (4-bit data + one 1-byte scale per
 *         16-element block).
 *  [arch] "How openbitsys/bitdecoding-fp4 works" (architecture digest):
 *         hybrid cache, KV quantization / block scaling / scale modes, paged
 *         attention kernel.
 *  NVFP4 / OCP-MX number formats: E2M1 element {0,.5,1,1.5,2,3,4,6} with a
 *  sign bit; E4M3 (bias 7, max 448, no infinities) block scale per 16
 *  elements times one FP32 per-tensor scale; UE8M0 power-of-two scale per 32
 *  elements for MXFP4.
 *
 * Readings where the pages are silent are listed in the repository's design
 * notes; each function below states the reading it implements.
 *
 * Pins: the CPU tests check every function here against something other than
 * itself -- brute force over the code tables, closed forms, the explicit
 * Sylvester matrix, textbook softmax attention in fp64.  The probability
 * quantizer's reading of the pages (each page's own reference maximum,
 * amax2-or-amax6 by tau on u = c*P, the unquantized denominator) is pinned by
 * its endpoints (tau = 0, tau = 448) and by closed forms: all keys equal, and
 * two pages whose keys are constant at two levels, which tells a per-page
 * maximum from one taken over several pages.  No value printed by the pages
 * pins it further: they print none.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_D 128          /* head_dim */
#define OR_PAGE 128       /* tokens per FP4 page ([cfg] PARITY_ENGINE_KWARGS block_size) */
#define OR_CODE_BYTES 8192 /* 128 tokens x 64 bytes of packed nibbles */

typedef struct {
    int num_q_heads;
    int num_kv_heads;
    int head_dim;     /* must be 128 */
    int page_size;    /* must be 128 */
    int sink_tokens;  /* 16 in [cfg] KV_MODES */
    int format;       /* 0 = NVFP4 (E4M3 per 16 + FP32 per tensor), 1 = MXFP4 (UE8M0 per 32) */
    int key_search;   /* 1 = per-block {4,6} search for K, 0 = amax6 */
    int rotation;     /* 1 = Hadamard rotation of K and Q along head_dim */
    int centering;    /* 1 = subtract the static per-channel key mean */
    int query_terms;  /* 1 or 2 */
    int p_mode;       /* 0 = exact P (no quantization), 1 = amax6, 2 = amax2-or-amax6 */
    int p_c;          /* 1 or 8 */
    int pool_pages;   /* physical pages of a layer's pool; 0 = not declared */
} or_config;

/* A physical page the path may touch: in [0, pool_pages), or any
 * non-negative index when the pool size is not declared.  The library's
 * definition of an out-of-range block-table or destination entry: it is left
 * out (no record read or written). */
static int page_in_pool(const or_config* c, int64_t phys) {
    return phys >= 0 && (c->pool_pages <= 0 || phys < c->pool_pages);
}

/* attention debug flags */
#define OR_FLAG_QUANT_DENOM 1  /* softmax denominator = sum of quantized P instead of exact P */

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                            */
/* ------------------------------------------------------------------------ */

static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float or_bf16_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* E2M1 encode, round to nearest, ties to the even code, saturating at 6.
 * The sign bit is the input's sign bit, so a negative value that rounds to
 * zero keeps code 0x8 (reading: IEEE signed zero). */
uint8_t or_e2m1_encode(float v) {
    uint8_t s = signbit(v) ? 0x8 : 0x0;
    float a = fabsf(v);
    int k;
    if (!(a < 6.0f)) {
        k = 7;
    } else {
        k = 0;
        while (kE2M1[k + 1] <= a) k++;          /* kE2M1[k] <= a < kE2M1[k+1] */
        float mid = 0.5f * (kE2M1[k] + kE2M1[k + 1]);   /* exact */
        if (a > mid || (a == mid && (k & 1))) k++;
    }
    return (uint8_t)(s | (uint8_t)k);
}

float or_e2m1_value(uint8_t c) {
    float m = kE2M1[c & 7];
    return (c & 8) ? -m : m;
}

/* E4M3 (FN variant: no infinities, 0x7F is NaN) value of a byte. */
float or_e4m3_value(uint8_t b) {
    int e = (b >> 3) & 0xF;
    int m = b & 7;
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (b & 0x80) ? (float)-v : (float)v;
}

/* E4M3 encode of a non-negative scale: round to nearest, ties to even
 * mantissa, saturating to 448 (0x7E). */
uint8_t or_e4m3_encode(float s) {
    if (!(s <= 448.0f)) return 0x7E;               /* satfinite (also +inf) */
    if (s < 0.015625f) {                            /* below 2^-6: subnormal, step 2^-9 */
        double q = nearbyint((double)s * 512.0);    /* 0..8; 8 is the smallest normal */
        return (uint8_t)q;
    }
    int e;
    (void)frexp((double)s, &e);
    int E = e - 1;                                  /* s in [2^E, 2^(E+1)) */
    double m = nearbyint(((double)s / ldexp(1.0, E) - 1.0) * 8.0);
    if (m == 8.0) { E += 1; m = 0.0; }
    int b = ((E + 7) << 3) | (int)m;
    if (b > 0x7E) b = 0x7E;
    return (uint8_t)b;
}

/* 2^e as binary32 for e in [-127, 127] (subnormal at -127). */
static float pow2f_exact(int e) { return (float)ldexp(1.0, e); }

void or_e2m1_encode_n(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = or_e2m1_encode(x[i]);
}
void or_e4m3_encode_n(const float* x, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; i++) out[i] = or_e4m3_encode(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Block quantizers                                                          */
/* ------------------------------------------------------------------------ */

/* Sum of squared errors in a fixed pairwise order: w[i] += w[i+n/2] for
 * i < n/2, then halves again down to one term.  n is 16 or 32. */
float or_block_sse(const float* x, const float* xhat, int n) {
    float w[32];
    for (int i = 0; i < n; i++) {
        float e = x[i] - xhat[i];
        w[i] = e * e;
    }
    for (int h = n / 2; h >= 1; h /= 2)
        for (int i = 0; i < h; i++) w[i] = w[i] + w[i + h];
    return w[0];
}

/* NVFP4 block of 16 with scale mode m (amax mapped to m, m in {6,4,2}) and
 * per-tensor scale g:  amax -> t = m*g -> s = amax/t -> E4M3 byte -> S = sd*g
 * -> codes = E2M1(x * (1/S)).  Reconstruction xhat = value(code) * S.
 * [cfg] recipe_additional_config scale modes "amax6" / "four_six";
 * [cfg] probability_environment "amax2_or_amax6". */
void or_nvfp4_block(const float* x, int m, float g, uint8_t* codes, uint8_t* sb, float* xhat) {
    float amax = 0.0f;
    for (int i = 0; i < 16; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float t = (float)m * g;
    float s = amax / t;
    uint8_t b = or_e4m3_encode(s);
    float sd = or_e4m3_value(b);
    float S = sd * g;
    *sb = b;
    float inv = 1.0f / S;
    if (S == 0.0f || isinf(inv)) {
        for (int i = 0; i < 16; i++) { codes[i] = 0; xhat[i] = 0.0f; }
        return;
    }
    for (int i = 0; i < 16; i++) {
        float v = x[i] * inv;
        codes[i] = or_e2m1_encode(v);
        xhat[i] = or_e2m1_value(codes[i]) * S;
    }
}

/* Adaptive {4,6} block-scale search for keys ([cfg] RECIPE
 * outlier_aware_key_quantization.adaptive_block_scale_search, scale mode
 * "four_six"): quantize with amax->6 and amax->4, keep amax->4 only when its
 * squared reconstruction error is strictly lower (ties keep the default
 * amax6).  Returns the chosen m. */
int or_four_six_block(const float* x, float g, uint8_t* codes, uint8_t* sb, float* xhat,
                      float* sse4_out, float* sse6_out) {
    uint8_t c6[16], c4[16], b6, b4;
    float x6[16], x4[16];
    or_nvfp4_block(x, 6, g, c6, &b6, x6);
    or_nvfp4_block(x, 4, g, c4, &b4, x4);
    float e6 = or_block_sse(x, x6, 16);
    float e4 = or_block_sse(x, x4, 16);
    if (sse4_out) *sse4_out = e4;
    if (sse6_out) *sse6_out = e6;
    int use4 = e4 < e6;
    memcpy(codes, use4 ? c4 : c6, 16);
    memcpy(xhat, use4 ? x4 : x6, 16 * sizeof(float));
    *sb = use4 ? b4 : b6;
    return use4 ? 4 : 6;
}

/* Quantize one block of 32 with a given power-of-two exponent e. */
static void mx_block_with_exp(const float* x, int e, uint8_t* codes, float* xhat) {
    float down = pow2f_exact(-e);
    float up = pow2f_exact(e);
    for (int i = 0; i < 32; i++) {
        float v = x[i] * down;
        codes[i] = or_e2m1_encode(v);
        xhat[i] = or_e2m1_value(codes[i]) * up;
    }
}

/* MXFP4 "mxfp4_search" ([cfg] KV_MODES["bitdecoding-mxfp4"].scale_mode):
 * UE8M0 scale per 32 elements.  Reading: E = floor(log2 amax) read from the
 * binary32 exponent; candidates e0 = E-2 (the OCP MX shared-exponent rule,
 * maps amax into [4,8)) and e0+1 (maps amax into [2,4)), each clamped to
 * [-127,127]; keep e0+1 only if its squared error is strictly lower.
 * amax == 0 gives byte 0 and all-zero codes.  Returns the chosen exponent. */
int or_mx_block(const float* x, uint8_t* codes, uint8_t* sb, float* xhat,
                float* sse_a_out, float* sse_b_out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int i = 0; i < 32; i++) { codes[i] = 0; xhat[i] = 0.0f; }
        *sb = 0;
        if (sse_a_out) *sse_a_out = 0.0f;
        if (sse_b_out) *sse_b_out = 0.0f;
        return -127;
    }
    int fe;
    (void)frexp((double)amax, &fe);
    int E = fe - 1;                                 /* 2^E <= amax < 2^(E+1) */
    int ea = E - 2, eb = E - 1;
    if (ea < -127) ea = -127;
    if (ea > 127) ea = 127;
    if (eb < -127) eb = -127;
    if (eb > 127) eb = 127;
    uint8_t ca[32], cb[32];
    float xa[32], xb[32];
    mx_block_with_exp(x, ea, ca, xa);
    mx_block_with_exp(x, eb, cb, xb);
    float sa = or_block_sse(x, xa, 32);
    float sbb = or_block_sse(x, xb, 32);
    if (sse_a_out) *sse_a_out = sa;
    if (sse_b_out) *sse_b_out = sbb;
    int useb = sbb < sa;
    int e = useb ? eb : ea;
    memcpy(codes, useb ? cb : ca, 32);
    memcpy(xhat, useb ? xb : xa, 32 * sizeof(float));
    *sb = (uint8_t)(e + 127);
    return e;
}

/* ------------------------------------------------------------------------ */
/* Hadamard rotation along head_dim                                          */
/* ------------------------------------------------------------------------ */

/* Unnormalized fast Walsh-Hadamard transform of 128 values in binary32,
 * strides 1, 2, 4, ..., 64: (x[i], x[i+h]) <- (x[i]+x[i+h], x[i]-x[i+h]).
 * This is the Sylvester-ordered H_128 ([cfg] nvfp4_rotation "hadamard"). */
void or_fwht128(float* x) {
    for (int h = 1; h < OR_D; h <<= 1)
        for (int i = 0; i < OR_D; i++)
            if ((i & h) == 0) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
}

/* Orthonormal rotation: FWHT then one multiply by r = binary32(1/sqrt(128)). */
void or_rotate128(float* x) {
    const float r = 0.08838834764831845f;
    or_fwht128(x);
    for (int i = 0; i < OR_D; i++) x[i] = x[i] * r;
}

/* ------------------------------------------------------------------------ */
/* Pool record layout                                                        */
/* ------------------------------------------------------------------------ */

static int nblk(const or_config* c) { return c->format == 0 ? 8 : 4; }

int64_t or_record_bytes(const or_config* c) { return OR_CODE_BYTES + (int64_t)OR_PAGE * nblk(c); }

/* Byte offset of record (page, head, kv) in a layer's pool; kv 0 = K, 1 = V. */
static int64_t rec_off(const or_config* c, int64_t page, int h, int kv) {
    return ((page * c->num_kv_heads + h) * 2 + kv) * or_record_bytes(c);
}

/* K record.  Codes: the byte of dims d, d+1 (d even; d in the low nibble)
 * of token t sits at (t/8)*512 + (d/32)*128 + (t%8)*16 + (d%32)/2, i.e. in
 * groups of 8 tokens x 32 dims, each group 128 contiguous bytes.  Scales: the
 * byte of block b of token t sits at 8192 + (b/4)*512 + (t%32)*16 + (t/32)*4
 * + b%4 (512-byte groups of 32 lines of 16 bytes; line i holds tokens i,
 * i+32, i+64, i+96, four blocks each). */
static int64_t k_code_off(int tok, int d) {
    return (int64_t)(tok / 8) * 512 + (d / 32) * 128 + (tok % 8) * 16 + (d % 32) / 2;
}
static int64_t k_scale_off(int tok, int b) {
    return OR_CODE_BYTES + (int64_t)(b / 4) * 512 + (tok % 32) * 16 + (tok / 32) * 4 + b % 4;
}

static void put_k(const or_config* c, uint8_t* rec, int tok, const uint8_t* codes128, const uint8_t* sbs) {
    for (int d = 0; d < OR_D; d += 2)
        rec[k_code_off(tok, d)] = (uint8_t)((codes128[d] & 0xF) | ((codes128[d + 1] & 0xF) << 4));
    for (int b = 0; b < nblk(c); b++) rec[k_scale_off(tok, b)] = sbs[b];
}

/* V record: tokens are paired (tau, tau+1) inside each 16-token group i
 * (tau = 16 i + 2 p, p = 0..7).  Row (i, p) is 128 bytes: the byte of head
 * dim d holds token tau in the low nibble and token tau+1 in the high
 * nibble, and the 16 bytes of dims 16c..16c+15 sit at 16-byte slot
 * c XOR 2(p mod 4) of the row.  scales[i][p][b][2] holds the two tokens'
 * scale bytes of block b, token tau first. */
static int v_code_off(int i, int p, int d) {
    return (i * 8 + p) * OR_D + (((d >> 4) ^ (2 * (p & 3))) << 4) + (d & 15);
}

static void put_v(const or_config* c, uint8_t* rec, int tok, const uint8_t* codes128, const uint8_t* sbs) {
    int i = tok / 16, r = tok % 16, p = r / 2, hi = r % 2;
    for (int d = 0; d < OR_D; d++) {
        uint8_t* byte = &rec[v_code_off(i, p, d)];
        if (hi) *byte = (uint8_t)((*byte & 0x0F) | ((codes128[d] & 0xF) << 4));
        else *byte = (uint8_t)((*byte & 0xF0) | (codes128[d] & 0xF));
    }
    for (int b = 0; b < nblk(c); b++) rec[OR_CODE_BYTES + ((i * 8 + p) * nblk(c) + b) * 2 + hi] = sbs[b];
}

static uint8_t get_k_code(const uint8_t* rec, int tok, int d) {
    uint8_t byte = rec[k_code_off(tok, d & ~1)];
    return (d & 1) ? (byte >> 4) : (byte & 0xF);
}
static uint8_t get_k_scale(const or_config* c, const uint8_t* rec, int tok, int b) {
    (void)c;
    return rec[k_scale_off(tok, b)];
}
static uint8_t get_v_code(const uint8_t* rec, int tok, int d) {
    int i = tok / 16, r = tok % 16, p = r / 2, hi = r % 2;
    uint8_t byte = rec[v_code_off(i, p, d)];
    return hi ? (byte >> 4) : (byte & 0xF);
}
static uint8_t get_v_scale(const or_config* c, const uint8_t* rec, int tok, int b) {
    int i = tok / 16, r = tok % 16, p = r / 2, hi = r % 2;
    return rec[OR_CODE_BYTES + ((i * 8 + p) * nblk(c) + b) * 2 + hi];
}

/* Value of a dequantized element given its code and scale byte.  NVFP4:
 * value(code) * E4M3(byte) (the per-tensor scale is applied by the caller);
 * MXFP4: value(code) * 2^(byte-127). */
static double deq(const or_config* c, uint8_t code, uint8_t sbyte) {
    double v = (double)or_e2m1_value(code);
    if (c->format == 0) return v * (double)or_e4m3_value(sbyte);
    return v * ldexp(1.0, (int)sbyte - 127);
}

/* ------------------------------------------------------------------------ */
/* Page writer                                                               */
/* ------------------------------------------------------------------------ */

/* Quantize one token's head vector (128 values, already transformed) into
 * codes and scale bytes with the tensor's scale rule. */
static void quantize_vec(const or_config* c, const float* y, int is_key, float g,
                         uint8_t* codes128, uint8_t* sbs) {
    float xhat[32];
    if (c->format == 0) {
        for (int b = 0; b < 8; b++) {
            if (is_key && c->key_search)
                or_four_six_block(y + 16 * b, g, codes128 + 16 * b, &sbs[b], xhat, NULL, NULL);
            else
                or_nvfp4_block(y + 16 * b, 6, g, codes128 + 16 * b, &sbs[b], xhat);
        }
    } else {
        for (int b = 0; b < 4; b++) or_mx_block(y + 32 * b, codes128 + 32 * b, &sbs[b], xhat, NULL, NULL);
    }
}

/* Freeze-at-fill page quantization ([ab] docstring: each page is quantized
 * once when it fills; [arch] KV cache writer -> KV quantization).
 * k, v: n pages of [128 tokens][Hkv][128] bf16.  dst_pages[n]: physical page
 * of each.  mu: [Hkv][128] key mean of this layer (NULL = zero).
 * K: x = bf16 - mu (centering), rotated (rotation), then {4,6} / amax6 / MX.
 * V: amax6 (NVFP4) or MX search, no centering, no rotation.
 * A destination outside the pool is skipped; returns the number skipped. */
int or_quantize_kv_pages(const or_config* c, const uint16_t* k, const uint16_t* v,
                         const int32_t* dst_pages, int n, const float* mu,
                         float k_gscale, float v_gscale, uint8_t* pool) {
    int H = c->num_kv_heads;
    float x[OR_D];
    uint8_t codes[OR_D], sbs[8];
    int skipped = 0;
    for (int pg = 0; pg < n; pg++) {
        if (!page_in_pool(c, dst_pages[pg])) {
            skipped++;
            continue;
        }
        for (int h = 0; h < H; h++) {
            uint8_t* krec = pool + rec_off(c, dst_pages[pg], h, 0);
            uint8_t* vrec = pool + rec_off(c, dst_pages[pg], h, 1);
            for (int tok = 0; tok < OR_PAGE; tok++) {
                const uint16_t* ks = k + (((int64_t)pg * OR_PAGE + tok) * H + h) * OR_D;
                const uint16_t* vs = v + (((int64_t)pg * OR_PAGE + tok) * H + h) * OR_D;
                for (int d = 0; d < OR_D; d++) {
                    x[d] = or_bf16_to_float(ks[d]);
                    if (c->centering && mu) x[d] = x[d] - mu[h * OR_D + d];
                }
                if (c->rotation) or_rotate128(x);
                quantize_vec(c, x, 1, k_gscale, codes, sbs);
                put_k(c, krec, tok, codes, sbs);
                for (int d = 0; d < OR_D; d++) x[d] = or_bf16_to_float(vs[d]);
                quantize_vec(c, x, 0, v_gscale, codes, sbs);
                put_v(c, vrec, tok, codes, sbs);
            }
        }
    }
    return skipped;
}

/* ------------------------------------------------------------------------ */
/* Query                                                                     */
/* ------------------------------------------------------------------------ */

int64_t or_qpack_stride(const or_config* c) {
    int64_t raw = (int64_t)c->num_q_heads * (2 * 64 + 2 * 8 + 4) + 16;
    return (raw + 255) / 256 * 256;
}
static int64_t qp_codes(const or_config* c, int term, int j) { return ((int64_t)term * c->num_q_heads + j) * 64; }
static int64_t qp_scales(const or_config* c, int term, int j) {
    return (int64_t)2 * c->num_q_heads * 64 + ((int64_t)term * c->num_q_heads + j) * nblk(c);
}
static int64_t qp_g(const or_config* c) { return (int64_t)2 * c->num_q_heads * 64 + (int64_t)2 * c->num_q_heads * 8; }
static int64_t qp_qmu(const or_config* c) { return qp_g(c) + 16; }

/* Quantize one term over all Hq*128 values in xs (rotated query or residual)
 * and write its codes and scales; also returns the reconstruction. */
static float quantize_query_term(const or_config* c, const float* xs, int term, uint8_t* out, float* xhat_all) {
    int Hq = c->num_q_heads;
    float g = 1.0f;
    if (c->format == 0) {
        float amax = 0.0f;
        for (int i = 0; i < Hq * OR_D; i++) {
            float a = fabsf(xs[i]);
            if (a > amax) amax = a;
        }
        g = (amax == 0.0f) ? 1.0f : amax / 2688.0f;   /* 2688 = 6 * 448 */
    }
    for (int j = 0; j < Hq; j++) {
        const float* x = xs + j * OR_D;
        uint8_t codes[OR_D], sbs[8];
        float* xh = xhat_all + j * OR_D;
        if (c->format == 0) {
            for (int b = 0; b < 8; b++) or_nvfp4_block(x + 16 * b, 6, g, codes + 16 * b, &sbs[b], xh + 16 * b);
        } else {
            for (int b = 0; b < 4; b++) or_mx_block(x + 32 * b, codes + 32 * b, &sbs[b], xh + 32 * b, NULL, NULL);
        }
        for (int d = 0; d < OR_D; d += 2)
            out[qp_codes(c, term, j) + d / 2] = (uint8_t)((codes[d] & 0xF) | ((codes[d + 1] & 0xF) << 4));
        for (int b = 0; b < nblk(c); b++) out[qp_scales(c, term, j) + b] = sbs[b];
    }
    return g;
}

/* Dual-residual query quantization ([cfg] RECIPE
 * dual_residual_query_quantization, nvfp4_query_terms 2, query scale mode
 * "amax6"): q -> rotate -> Q1 (amax6, per-tensor scale g1 = amax/2688 over
 * the token's Hq*128 values) -> R = q_rot - Q1hat -> Q2 (amax6, g2).  MXFP4
 * uses the mxfp4_search rule for both terms and no per-tensor scale.
 * Also stores q.mu (unrotated bf16 q, this layer's key mean) per head in fp32
 * for the on-device path; the oracle's own attention recomputes it in fp64.
 * q: [B][Hq][128] bf16.  out: B records of or_qpack_stride bytes. */
int or_quantize_query(const or_config* c, const uint16_t* q, int B, const float* mu, uint8_t* out) {
    int Hq = c->num_q_heads, G = c->num_q_heads / c->num_kv_heads;
    int64_t stride = or_qpack_stride(c);
    float* xs = (float*)malloc(sizeof(float) * Hq * OR_D);
    float* xh = (float*)malloc(sizeof(float) * Hq * OR_D);
    float* rs = (float*)malloc(sizeof(float) * Hq * OR_D);
    for (int bi = 0; bi < B; bi++) {
        uint8_t* o = out + bi * stride;
        memset(o, 0, (size_t)stride);
        for (int j = 0; j < Hq; j++) {
            for (int d = 0; d < OR_D; d++) xs[j * OR_D + d] = or_bf16_to_float(q[((int64_t)bi * Hq + j) * OR_D + d]);
            if (c->rotation) or_rotate128(xs + j * OR_D);
        }
        float g1 = quantize_query_term(c, xs, 0, o, xh);
        float g2 = 0.0f;
        if (c->query_terms == 2) {
            for (int i = 0; i < Hq * OR_D; i++) rs[i] = xs[i] - xh[i];
            g2 = quantize_query_term(c, rs, 1, o, xh);
        }
        float gs[2] = {g1, g2};
        memcpy(o + qp_g(c), gs, 8);
        for (int j = 0; j < Hq; j++) {
            double acc = 0.0;
            if (c->centering && mu) {
                int h = j / G;
                for (int d = 0; d < OR_D; d++)
                    acc += (double)or_bf16_to_float(q[((int64_t)bi * Hq + j) * OR_D + d]) * (double)mu[h * OR_D + d];
            }
            float f = (float)acc;
            memcpy(o + qp_qmu(c) + 4 * j, &f, 4);
        }
    }
    free(xs);
    free(xh);
    free(rs);
    return 0;
}

/* Dequantized query row (sum of its terms) in fp64, rotated domain. */
static void query_hat(const or_config* c, const uint8_t* qp, int j, double* qh) {
    float gs[2];
    memcpy(gs, qp + qp_g(c), 8);
    for (int d = 0; d < OR_D; d++) qh[d] = 0.0;
    for (int term = 0; term < c->query_terms; term++) {
        double g = (c->format == 0) ? (double)gs[term] : 1.0;
        for (int d = 0; d < OR_D; d++) {
            uint8_t byte = qp[qp_codes(c, term, j) + d / 2];
            uint8_t code = (d & 1) ? (byte >> 4) : (byte & 0xF);
            uint8_t sbyte = qp[qp_scales(c, term, j) + d / (c->format == 0 ? 16 : 32)];
            qh[d] += deq(c, code, sbyte) * g;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

typedef struct { double m, l; double o[OR_D]; int empty; } seg_t;

static void seg_init(seg_t* s) { s->m = -INFINITY; s->l = 0.0; s->empty = 1; for (int d = 0; d < OR_D; d++) s->o[d] = 0.0; }

/* Exact-P segment over BF16 tokens (sink or tail; [cfg] KV_MODES sink_tokens
 * 16 and the BF16 partial page of the hybrid cache): scores from raw bf16 q
 * and raw bf16 k, P = exp(s - m_seg), O = sum P v, l = sum P. */
static void bf16_segment(const uint16_t* qrow, const uint16_t* kbase, const uint16_t* vbase,
                         int ntok, int H, int h, double sm, seg_t* out) {
    seg_init(out);
    if (ntok <= 0) return;
    double* s = (double*)malloc(sizeof(double) * ntok);
    double m = -INFINITY;
    for (int t = 0; t < ntok; t++) {
        const uint16_t* kt = kbase + ((int64_t)t * H + h) * OR_D;
        double acc = 0.0;
        for (int d = 0; d < OR_D; d++) acc += (double)or_bf16_to_float(qrow[d]) * (double)or_bf16_to_float(kt[d]);
        s[t] = sm * acc;
        if (s[t] > m) m = s[t];
    }
    out->m = m;
    out->empty = 0;
    for (int t = 0; t < ntok; t++) {
        double p = exp(s[t] - m);
        out->l += p;
        const uint16_t* vt = vbase + ((int64_t)t * H + h) * OR_D;
        for (int d = 0; d < OR_D; d++) out->o[d] += p * (double)or_bf16_to_float(vt[d]);
    }
    free(s);
}

/* Probability quantization of one 16-token block ([cfg]
 * probability_environment: "amax6", or "amax2_or_amax6" with c in {1, 8}
 * and a threshold tau in [0, 448]).  Reading: u = fp32(c * P); a = max u;
 * scale mode 2 if a < tau else 6 (always 6 and c = 1 for "amax6"); NVFP4
 * block quantization of u with per-tensor scale 1; Phat = value * E4M3 / c.
 * ptil: exact probabilities (fp64).  Returns Phat in fp64 and the mode. */
void or_p_block(const double* ptil, int p_mode, int p_c, float tau, double* phat, int* mode_out) {
    int cc = (p_mode == 2) ? p_c : 1;
    float u[16], xh[16];
    uint8_t codes[16], sb;
    float a = 0.0f;
    for (int i = 0; i < 16; i++) {
        u[i] = (float)((double)cc * ptil[i]);
        if (u[i] > a) a = u[i];
    }
    int mode = (p_mode == 2 && a < tau) ? 2 : 6;
    or_nvfp4_block(u, mode, 1.0f, codes, &sb, xh);
    double sd = (double)or_e4m3_value(sb);
    for (int i = 0; i < 16; i++) phat[i] = (double)or_e2m1_value(codes[i]) * sd / (double)cc;
    if (mode_out) *mode_out = mode;
}

/* One FP4 page as one segment.  Scores s = sm * (Qhat . Khat * gK + q.mu)
 * with Khat in the rotated, centered domain (q.mu restores the key mean's
 * contribution so that FP4 and BF16 segments share one logit origin).
 * Probabilities ([cfg] underflow_aware_probability_scaling): reading --
 * the reference max m_p is the page's own max, P = exp(s - m_p), and each
 * 16-token block is quantized by or_p_block.  O_p = sum Phat * Vhat * gV;
 * l_p = sum P (exact) unless OR_FLAG_QUANT_DENOM. */
static void fp4_page_segment(const or_config* c, const uint8_t* krec, const uint8_t* vrec,
                             const double* qh, double qmu, double sm, float tau, float gk, float gv,
                             int flags, seg_t* out) {
    double s[OR_PAGE], phat[OR_PAGE], ptil[OR_PAGE];
    double gK = (c->format == 0) ? (double)gk : 1.0;
    double gV = (c->format == 0) ? (double)gv : 1.0;
    int kb = (c->format == 0) ? 16 : 32;
    double m = -INFINITY;
    for (int t = 0; t < OR_PAGE; t++) {
        double acc = 0.0;
        for (int d = 0; d < OR_D; d++)
            acc += qh[d] * deq(c, get_k_code(krec, t, d), get_k_scale(c, krec, t, d / kb));
        s[t] = sm * (acc * gK + (c->centering ? qmu : 0.0));
        if (s[t] > m) m = s[t];
    }
    for (int t = 0; t < OR_PAGE; t++) ptil[t] = exp(s[t] - m);
    if (c->p_mode == 0) {
        for (int t = 0; t < OR_PAGE; t++) phat[t] = ptil[t];
    } else {
        for (int b = 0; b < OR_PAGE / 16; b++) or_p_block(ptil + 16 * b, c->p_mode, c->p_c, tau, phat + 16 * b, NULL);
    }
    seg_init(out);
    out->m = m;
    out->empty = 0;
    for (int t = 0; t < OR_PAGE; t++) {
        out->l += (flags & OR_FLAG_QUANT_DENOM) ? phat[t] : ptil[t];
        if (phat[t] == 0.0) continue;
        int vb = (c->format == 0) ? 16 : 32;
        for (int d = 0; d < OR_D; d++)
            out->o[d] += phat[t] * deq(c, get_v_code(vrec, t, d), get_v_scale(c, vrec, t, d / vb)) * gV;
    }
}

/* Merge segments: M = max m_seg; O = sum e^(m-M) O / sum e^(m-M) l. */
static void merge(const seg_t* segs, int n, double* o) {
    double M = -INFINITY;
    for (int i = 0; i < n; i++) if (!segs[i].empty && segs[i].m > M) M = segs[i].m;
    double L = 0.0;
    for (int d = 0; d < OR_D; d++) o[d] = 0.0;
    if (M == -INFINITY) return;
    for (int i = 0; i < n; i++) {
        if (segs[i].empty) continue;
        double w = exp(segs[i].m - M);
        L += w * segs[i].l;
        for (int d = 0; d < OR_D; d++) o[d] += w * segs[i].o[d];
    }
    for (int d = 0; d < OR_D; d++) o[d] = o[d] / L;
}

/* Paged single-token decode attention over the hybrid cache ([arch] paged
 * attention kernel; [cfg] sink_tokens 16, block_size 128).  For a sequence of
 * length L: sink = tokens [0, min(L,16)); FP4 pages p = 0..npages-1 with
 * npages = max(0, L-16) div 128 holding tokens 16+128p ..; tail = the
 * remaining max(0, L-16) - 128 npages tokens.  Query head j reads KV head
 * j div (Hq/Hkv); softmax scale 1/sqrt(128).  Out-of-range arguments, as the
 * library defines them: a negative L counts as 0; only the first max_blocks
 * pages exist; a page whose block-table entry lies outside the pool is left
 * out of the attention.
 * out: [B][Hq][128] fp64. */
int or_decode_attention(const or_config* c, const uint8_t* q_packed, const uint16_t* q, const float* mu,
                        const uint8_t* pool, const int32_t* block_table, int max_blocks,
                        const int32_t* seq_lens, const uint16_t* sink_k, const uint16_t* sink_v,
                        const uint16_t* tail_k, const uint16_t* tail_v, int B, float tau,
                        float gk, float gv, int flags, double* out) {
    int Hq = c->num_q_heads, H = c->num_kv_heads, G = Hq / H;
    int SINK = c->sink_tokens;
    double sm = 1.0 / sqrt((double)OR_D);
    int64_t stride = or_qpack_stride(c);
    double qh[OR_D];
    for (int b = 0; b < B; b++) {
        int L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        int nsink = L < SINK ? L : SINK;
        int rest = L - SINK > 0 ? L - SINK : 0;
        int npages = rest / OR_PAGE;
        int ntail = rest - npages * OR_PAGE;
        if (npages > max_blocks) npages = max_blocks;
        seg_t* segs = (seg_t*)malloc(sizeof(seg_t) * (size_t)(npages + 2));
        const uint8_t* qp = q_packed + b * stride;
        for (int j = 0; j < Hq; j++) {
            int h = j / G;
            const uint16_t* qrow = q + ((int64_t)b * Hq + j) * OR_D;
            double qmu = 0.0;
            if (c->centering && mu)
                for (int d = 0; d < OR_D; d++) qmu += (double)or_bf16_to_float(qrow[d]) * (double)mu[h * OR_D + d];
            query_hat(c, qp, j, qh);
            bf16_segment(qrow, sink_k + (int64_t)b * SINK * H * OR_D, sink_v + (int64_t)b * SINK * H * OR_D,
                         nsink, H, h, sm, &segs[0]);
            bf16_segment(qrow, tail_k + (int64_t)b * OR_PAGE * H * OR_D, tail_v + (int64_t)b * OR_PAGE * H * OR_D,
                         ntail, H, h, sm, &segs[1]);
            for (int p = 0; p < npages; p++) {
                int64_t phys = block_table[(int64_t)b * max_blocks + p];
                if (!page_in_pool(c, phys)) {
                    seg_init(&segs[2 + p]);   /* empty: left out of the merge */
                    continue;
                }
                fp4_page_segment(c, pool + rec_off(c, phys, h, 0), pool + rec_off(c, phys, h, 1), qh, qmu, sm,
                                 tau, gk, gv, flags, &segs[2 + p]);
            }
            merge(segs, npages + 2, out + ((int64_t)b * Hq + j) * OR_D);
        }
        free(segs);
    }
    return 0;
}

/* Attention with every quantizer replaced by the identity: the method's
 * transforms (centering, rotation, q.mu restore) applied to all L tokens of
 * one sequence in binary32 exactly as the writer and query quantizer apply
 * them, then one softmax over all tokens in fp64.  With centering and
 * rotation both off this is textbook attention.
 * q: [Hq][128]; k, v: [L][Hkv][128] bf16; out: [Hq][128]. */
int or_attention_identity_quant(const or_config* c, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                int L, const float* mu, double* out) {
    int Hq = c->num_q_heads, H = c->num_kv_heads, G = Hq / H;
    double sm = 1.0 / sqrt((double)OR_D);
    float qr[OR_D], kr[OR_D];
    double* s = (double*)malloc(sizeof(double) * (L > 0 ? L : 1));
    for (int j = 0; j < Hq; j++) {
        int h = j / G;
        double qmu = 0.0;
        for (int d = 0; d < OR_D; d++) {
            qr[d] = or_bf16_to_float(q[j * OR_D + d]);
            if (c->centering && mu) qmu += (double)qr[d] * (double)mu[h * OR_D + d];
        }
        if (c->rotation) or_rotate128(qr);
        double m = -INFINITY;
        for (int t = 0; t < L; t++) {
            for (int d = 0; d < OR_D; d++) {
                kr[d] = or_bf16_to_float(k[((int64_t)t * H + h) * OR_D + d]);
                if (c->centering && mu) kr[d] = kr[d] - mu[h * OR_D + d];
            }
            if (c->rotation) or_rotate128(kr);
            double acc = 0.0;
            for (int d = 0; d < OR_D; d++) acc += (double)qr[d] * (double)kr[d];
            s[t] = sm * (acc + qmu);
            if (s[t] > m) m = s[t];
        }
        double l = 0.0;
        double* o = out + (int64_t)j * OR_D;
        for (int d = 0; d < OR_D; d++) o[d] = 0.0;
        for (int t = 0; t < L; t++) {
            double p = exp(s[t] - m);
            l += p;
            for (int d = 0; d < OR_D; d++) o[d] += p * (double)or_bf16_to_float(v[((int64_t)t * H + h) * OR_D + d]);
        }
        for (int d = 0; d < OR_D; d++) o[d] = (L > 0) ? o[d] / l : 0.0;
    }
    free(s);
    return 0;
}

/* Memory ratio of a packed page vs BF16 ([ab] mem_ratio): bytes of one
 * token-head in BF16 (K and V) over the packed record bytes for it. */
double or_mem_ratio(const or_config* c) {
    double bf16 = 2.0 * 2.0 * OR_D;
    double packed = 2.0 * (double)or_record_bytes(c) / OR_PAGE;
    return bf16 / packed;
}
