/*
 * pkv_oracle.c -- plain CPU oracle for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls, links or includes
 * this file; only the tests, the smoke check and the CPU-baseline leg of the
 * benchmark load it.  It shares no code, header, table or constant with the
 * CUDA path.
 *
 * It is written to be read against the pages it follows, not to be fast:
 * scalar loops, fp64 for attention, and for the quantisers exactly the IEEE
 * fp32 operation sequence the method states (compiled with
 * -ffp-contract=off, no fast-math, default round-to-nearest-even mode).
 *
 * Sources (cited by page title and section):
 *   [APPEND]  "Write Triton Kv Cache Append Kernel" (skill guide):
 *             "Inputs the agent should gather first" items 1, 4-8;
 *             "Required reasoning process" steps 3, 5, 6, 9;
 *             "Correctness requirements".
 *   [PAGED]   "10. Triton KV Cache and PagedAttention" (llm-algo-leetcode):
 *             Step 1 (pool layout and block table), Step 4 (PyTorch gather
 *             reference), reference-code TODO 1-5 (lookup, masking, softmax).
 *   [3BIT]    "triton-3bit-kv-cache-kernel" README: section 1.A (24-bit octet
 *             layout and formulas), section 1.B (96-bit word layout and lane
 *             formula), section 2 item 3 (affine dequant round trip).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes):
 *   - context_lens counts the tokens to attend, the newest token included.
 *   - GQA maps q head h to kv head h / (num_heads / num_kv_heads).
 *   - e4m3 is the OCP "fn" variant (bias 7, max 448, no infinities,
 *     S.1111.111 = NaN); encoding rounds to nearest even and saturates finite
 *     overflow and infinities to +-448; every NaN encodes to 0x7F.
 *   - e5m2 (the second fp8 cache format of "Write Triton Kv Cache Append
 *     Kernel", inputs item 4) is the OCP E5M2 format (bias 15, 2 mantissa
 *     bits, infinities and NaNs at exponent 31, max 57344); encoding rounds
 *     to nearest even and saturates finite overflow and infinities to
 *     +-57344, like e4m3; every NaN encodes to 0x7F.
 *   - scale granularity of fp8 / int8 caches (inputs item 4: per tensor,
 *     per token, per head or per block): a row's scale is the kv head's
 *     (per head; per tensor is equal per-head scales), the physical block's
 *     scale for that head ([num_blocks, num_kv_heads]), or the row's own
 *     scale ([num_blocks, block_size, num_kv_heads], per token: the append
 *     takes each new token's scale per kv head from the caller and stores it
 *     at the token's slot).
 *   - int8 caches ("Write Triton Kv Cache Append Kernel", inputs item 4 and
 *     reasoning step 6: (x / scale) cast to the cache dtype) store
 *     clamp(rint(x / scale), -127, 127) with x / scale in fp32 and rint
 *     rounding half to even (symmetric range); NaN stores 0; the stored code
 *     c means c * scale.
 *   - 3-bit quantiser: s = fp16_rn((max-min)/7), z = clamp(rint(-min/s),0,7),
 *     q = clamp(rint(x/s)+z,0,7), all fp32; s == 0 gives z = 0, q = 0; an s
 *     that overflows fp16 saturates to 65504.  Element d of a head row sits at
 *     bit 3d of a little-endian bit stream (octet j = elements 8j..8j+7).
 *   - a context of length 0 gives an all-zero output row.
 *
 * Parity pins: every function here is pinned by a test against something
 * other than itself (closed forms, the pages' figures, library routines,
 * brute force); the quantiser's formula itself is a reading (see above), so
 * only its properties are pinned: range, round trip, error bound.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* dtype codes used by this oracle's interface (its own numbering). */
#define O_F16 1
#define O_BF16 2
#define O_E4M3 3
#define O_U3 4
#define O_E5M2 9
#define O_I8 10

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                           */
/* ------------------------------------------------------------------------ */

/* IEEE 754 binary16 -> double: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 = subnormal (m * 2^-24), 31 = inf/NaN. */
double pkvo_f16_to_f64(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);
    return s ? -v : v;
}

/* bfloat16 -> double: the upper 16 bits of an IEEE binary32. */
double pkvo_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

static double elem16_to_f64(uint16_t x, int dtype)
{
    return dtype == O_F16 ? pkvo_f16_to_f64(x) : pkvo_bf16_to_f64(x);
}

/* binary32 -> binary16, round to nearest even.  Written from the format
 * definition: pick the quantum of the binade (2^-24 below 2^-14), round the
 * exact quotient a/quantum to an integer (nearbyint in the default mode is
 * round-half-even), then encode.  |a| >= 65520 (max + half an ulp, a tie that
 * goes to the even neighbour 2^16) overflows to infinity. */
uint16_t pkvo_f32_to_f16_rn(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
    if (isnan(f))
        return sign | 0x7e00;
    double a = fabs((double)f);
    if (a >= 65520.0)
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);           /* a = fr * 2^e, fr in [0.5,1) */
    int ex = e - 1;         /* floor(log2 a) */
    if (ex < -14)
        ex = -14;           /* subnormal binade shares the 2^-24 quantum */
    double quantum = ldexp(1.0, ex - 10);
    double r = nearbyint(a / quantum) * quantum;
    if (r < ldexp(1.0, -14)) /* subnormal (or rounded up to 2^-14 = 0x0400) */
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    int e2;
    frexp(r, &e2);
    int E = e2 - 1;
    uint16_t mant = (uint16_t)(r / ldexp(1.0, E - 10) - 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | mant;
}

/* OCP FP8 E4M3 ("fn") decode: bias 7; exponent field 0 = subnormal
 * (m * 2^-9); S.1111.111 = NaN; no infinities; max finite 448. */
double pkvo_e4m3_to_f64(uint8_t c)
{
    int s = c >> 7, E = (c >> 3) & 0xf, m = c & 7;
    double v;
    if (E == 15 && m == 7)
        return NAN;
    if (E == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), E - 10);
    return s ? -v : v;
}

/* binary32 -> E4M3, round to nearest even, saturating to +-448. */
/* OCP E5M2: S.EEEEE.MM, bias 15; E = 31 holds the infinities (M = 0) and
 * NaNs; E = 0 the subnormals M/4 * 2^-14. */
double pkvo_e5m2_to_f64(uint8_t c)
{
    int s = c >> 7, E = (c >> 2) & 0x1f, m = c & 3;
    double v;
    if (E == 31)
        v = m ? NAN : INFINITY;
    else if (E == 0)
        v = ldexp((double)m, -16);
    else
        v = ldexp((double)(4 + m), E - 17);
    return s ? -v : v;
}

/* Nearest even, finite overflow and infinities to +-57344 (S.11110.11), NaN
 * to 0x7F: the value's binade sets the quantum (2^-16 in the subnormal
 * range), the rounded multiple of it is re-encoded. */
uint8_t pkvo_f32_to_e5m2(float f)
{
    uint8_t sign = signbit(f) ? 0x80 : 0;
    if (isnan(f))
        return 0x7f;
    double a = fabs((double)f);
    if (a >= 57344.0)
        return sign | 0x7b;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1;                     /* a in [2^ex, 2^(ex+1)) */
    if (ex < -14)
        ex = -14;
    double quantum = ldexp(1.0, ex - 2);
    double r = nearbyint(a / quantum) * quantum; /* a < 57344 => r <= 57344 */
    if (r < ldexp(1.0, -14))
        return sign | (uint8_t)(r / ldexp(1.0, -16));
    int e2;
    frexp(r, &e2);
    int E = e2 - 1;
    uint8_t mant = (uint8_t)(r / ldexp(1.0, E - 2) - 4.0);
    return sign | (uint8_t)((E + 15) << 2) | mant;
}

/* int8 code of x (already divided by the scale, in fp32): nearest integer,
 * half to even, saturated to +-127; NaN -> 0. */
int8_t pkvo_f32_to_i8(float f)
{
    if (isnan(f))
        return 0;
    if (f >= 127.0f)
        return 127;
    if (f <= -127.0f)
        return -127;
    return (int8_t)nearbyintf(f);
}

uint8_t pkvo_f32_to_e4m3(float f)
{
    uint8_t sign = signbit(f) ? 0x80 : 0;
    if (isnan(f))
        return 0x7f;
    double a = fabs((double)f);
    if (a >= 448.0)
        return sign | 0x7e;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < -6)
        ex = -6;            /* subnormal binade: quantum 2^-9 */
    double quantum = ldexp(1.0, ex - 3);
    double r = nearbyint(a / quantum) * quantum; /* a < 448 => r <= 448 */
    if (r < ldexp(1.0, -6))
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    int e2;
    frexp(r, &e2);
    int E = e2 - 1;
    uint8_t mant = (uint8_t)(r / ldexp(1.0, E - 3) - 8.0);
    return sign | (uint8_t)((E + 7) << 3) | mant;
}

/* ------------------------------------------------------------------------ */
/* 3-bit packing: [3BIT] section 1.A (octets) and 1.B (96-bit words)         */
/* ------------------------------------------------------------------------ */

/* Pack 8 values (only their low 3 bits are used) into 3 bytes. */
void pkvo_pack3_octet(const uint8_t v[8], uint8_t b[3])
{
    b[0] = (uint8_t)((v[0] & 7) | ((v[1] & 7) << 3) | ((v[2] & 3) << 6));
    b[1] = (uint8_t)(((v[2] >> 2) & 1) | ((v[3] & 7) << 1) | ((v[4] & 7) << 4) |
                     ((v[5] & 1) << 7));
    b[2] = (uint8_t)(((v[5] >> 1) & 3) | ((v[6] & 7) << 2) | ((v[7] & 7) << 5));
}

/* Unpack 3 bytes into 8 values; v2 and v5 straddle byte boundaries. */
void pkvo_unpack3_octet(const uint8_t b[3], uint8_t v[8])
{
    v[0] = b[0] & 7;
    v[1] = (b[0] >> 3) & 7;
    v[2] = (uint8_t)(((b[0] >> 6) & 3) | ((b[1] & 1) << 2));
    v[3] = (b[1] >> 1) & 7;
    v[4] = (b[1] >> 4) & 7;
    v[5] = (uint8_t)(((b[1] >> 7) & 1) | ((b[2] & 3) << 1));
    v[6] = (b[2] >> 2) & 7;
    v[7] = (b[2] >> 5) & 7;
}

void pkvo_pack3(const uint8_t *values, uint8_t *packed, int64_t n_octets)
{
    for (int64_t i = 0; i < n_octets; ++i)
        pkvo_pack3_octet(values + 8 * i, packed + 3 * i);
}

void pkvo_unpack3(const uint8_t *packed, uint8_t *values, int64_t n_octets)
{
    for (int64_t i = 0; i < n_octets; ++i)
        pkvo_unpack3_octet(packed + 3 * i, values + 8 * i);
}

/* 96-bit group (3 x uint32) -> 32 lanes.  Lane i starts at bit 3i, in word
 * w = 3i/32 at shift s = 3i%32; lanes with s > 29 (i = 10, 21) take their
 * high bits from the next word. */
void pkvo_unpack3_words(const uint32_t *words, uint8_t *values, int64_t n_groups)
{
    for (int64_t g = 0; g < n_groups; ++g) {
        const uint32_t *W = words + 3 * g;
        for (int i = 0; i < 32; ++i) {
            int w = (3 * i) / 32, s = (3 * i) % 32;
            uint32_t lo = W[w] >> s;
            uint32_t hi = 0;
            if (s > 29)
                hi = W[w + 1] << (32 - s);
            values[32 * g + i] = (uint8_t)((lo | hi) & 7);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* 3-bit affine quantiser of one head row (reading stated in the header)     */
/* ------------------------------------------------------------------------ */

void pkvo_u3_quantize_row(const float *x, int D, uint16_t *s_bits, uint8_t *z_out,
                          uint8_t *q_out)
{
    float mn = x[0], mx = x[0];
    for (int d = 1; d < D; ++d) {
        if (x[d] < mn)
            mn = x[d];
        if (x[d] > mx)
            mx = x[d];
    }
    float s32 = (mx - mn) / 7.0f;
    uint16_t sh = pkvo_f32_to_f16_rn(s32);
    if ((sh & 0x7fff) == 0x7c00)
        sh = 0x7bff; /* saturate: 65504 */
    float s = (float)pkvo_f16_to_f64(sh);
    if (s == 0.0f) {
        *s_bits = sh;
        *z_out = 0;
        for (int d = 0; d < D; ++d)
            q_out[d] = 0;
        return;
    }
    float zf = rintf(-mn / s);
    if (zf < 0.0f)
        zf = 0.0f;
    if (zf > 7.0f)
        zf = 7.0f;
    for (int d = 0; d < D; ++d) {
        float t = rintf(x[d] / s) + zf;
        if (t < 0.0f)
            t = 0.0f;
        if (t > 7.0f)
            t = 7.0f;
        q_out[d] = (uint8_t)t;
    }
    *s_bits = sh;
    *z_out = (uint8_t)zf;
}

/* Quantise and pack a batch of rows: x [n_rows, D] fp16/bf16 bits ->
 * packed [n_rows, 3D/8], scale bits [n_rows], zero [n_rows]. */
void pkvo_u3_quantize_pack_rows(const uint16_t *x, int src_dtype, int64_t n_rows, int D,
                                uint8_t *packed, uint16_t *s_bits, uint8_t *zeros)
{
    float xf[1024];
    uint8_t q[1024];
    for (int64_t r = 0; r < n_rows; ++r) {
        for (int d = 0; d < D; ++d)
            xf[d] = (float)elem16_to_f64(x[r * D + d], src_dtype);
        pkvo_u3_quantize_row(xf, D, &s_bits[r], &zeros[r], q);
        pkvo_pack3(q, packed + r * (int64_t)(3 * D / 8), D / 8);
    }
}

/* ------------------------------------------------------------------------ */
/* slot_mapping builder: [APPEND] step 9                                     */
/* ------------------------------------------------------------------------ */

/* One new token per listed (request, position):
 * slot = block_table[req][pos / BS] * BS + pos % BS; a negative position
 * marks padding and yields slot -1. */
void pkvo_build_slot_mapping(const int32_t *block_tables, int max_blocks, int block_size,
                             const int32_t *req, const int32_t *pos, int64_t n,
                             int64_t *slot_mapping)
{
    for (int64_t t = 0; t < n; ++t) {
        if (pos[t] < 0) {
            slot_mapping[t] = -1;
            continue;
        }
        int64_t logical = pos[t] / block_size;
        int64_t in_block = pos[t] % block_size;
        int64_t block_id = block_tables[(int64_t)req[t] * max_blocks + logical];
        slot_mapping[t] = block_id * block_size + in_block;
    }
}

/* ------------------------------------------------------------------------ */
/* Append (scatter): [APPEND] steps 3, 5, 6                                  */
/* ------------------------------------------------------------------------ */

/* Cache arrays are contiguous [num_blocks, block_size, num_kv_heads, row]
 * with row = head_dim elements (16-bit or e4m3 bytes) or 3*head_dim/8 bytes
 * (3-bit); 3-bit metadata is [num_blocks, block_size, num_kv_heads].
 * New K/V are contiguous [num_tokens, num_kv_heads, head_dim] 16-bit bits.
 * Tokens are applied in order (a duplicated slot keeps the last write).
 * Returns the number of tokens whose slot was out of range (skipped). */
/* Scale of cache row (blk, off, h) for fp8 / int8 caches, by granularity. */
#define SCALE_PER_HEAD 0
#define SCALE_PER_BLOCK 1
#define SCALE_PER_TOKEN 2
static double row_scale(int mode, const float *per_head, const float *arr, int64_t blk, int64_t off,
                        int h, int num_kv_heads, int block_size)
{
    if (mode == SCALE_PER_BLOCK)
        return arr[blk * num_kv_heads + h];
    if (mode == SCALE_PER_TOKEN)
        return arr[(blk * block_size + off) * num_kv_heads + h];
    return per_head ? per_head[h] : 1.0;
}

/* The append with a scale granularity: per head (k_scale / v_scale),
 * per block (k_scales / v_scales [num_blocks, Hkv], read), or per token
 * (k_new_scale / v_new_scale [num_tokens, Hkv] given with the new rows and
 * stored into k_scales / v_scales [num_blocks, block_size, Hkv]). */
int64_t pkvo_kv_append_scaled(int cache_dtype, int src_dtype, int64_t num_tokens, int num_kv_heads,
                              int head_dim, const uint16_t *k_new, const uint16_t *v_new,
                              const int64_t *slot_mapping, int64_t num_blocks, int block_size,
                              void *k_cache, void *v_cache, const float *k_scale,
                              const float *v_scale, uint16_t *k_qscale, uint8_t *k_qzero,
                              uint16_t *v_qscale, uint8_t *v_qzero, int scale_mode,
                              const float *k_new_scale, const float *v_new_scale, float *k_scales,
                              float *v_scales)
{
    int64_t bad = 0;
    const int D = head_dim;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue; /* padding token: no load, no store */
        if (slot >= num_blocks * block_size) {
            ++bad;
            continue;
        }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            int64_t row = (blk * block_size + off) * num_kv_heads + h; /* row index */
            const uint16_t *ks = k_new + (t * num_kv_heads + h) * D;
            const uint16_t *vs = v_new + (t * num_kv_heads + h) * D;
            float ksc = 1.0f, vsc = 1.0f;             /* the row's fp8 / int8 scales */
            if (scale_mode == SCALE_PER_TOKEN && (cache_dtype == O_E4M3 || cache_dtype == O_E5M2 ||
                                                  cache_dtype == O_I8)) {
                ksc = k_new_scale[t * num_kv_heads + h];
                vsc = v_new_scale[t * num_kv_heads + h];
                k_scales[row] = ksc;
                v_scales[row] = vsc;
            } else if (scale_mode == SCALE_PER_BLOCK) {
                ksc = k_scales[blk * num_kv_heads + h];
                vsc = v_scales[blk * num_kv_heads + h];
            } else if (k_scale) {
                ksc = k_scale[h];
                vsc = v_scale[h];
            }
            if (cache_dtype == O_F16 || cache_dtype == O_BF16) {
                memcpy((uint16_t *)k_cache + row * D, ks, (size_t)D * 2);
                memcpy((uint16_t *)v_cache + row * D, vs, (size_t)D * 2);
            } else if (cache_dtype == O_I8) {
                int8_t *kd = (int8_t *)k_cache + row * D;
                int8_t *vd = (int8_t *)v_cache + row * D;
                for (int d = 0; d < D; ++d) {
                    float xk = (float)elem16_to_f64(ks[d], src_dtype) / ksc;
                    float xv = (float)elem16_to_f64(vs[d], src_dtype) / vsc;
                    kd[d] = pkvo_f32_to_i8(xk);
                    vd[d] = pkvo_f32_to_i8(xv);
                }
            } else if (cache_dtype == O_E4M3 || cache_dtype == O_E5M2) {
                uint8_t *kd = (uint8_t *)k_cache + row * D;
                uint8_t *vd = (uint8_t *)v_cache + row * D;
                for (int d = 0; d < D; ++d) {
                    /* scale division in fp32, then the cast */
                    float xk = (float)elem16_to_f64(ks[d], src_dtype) / ksc;
                    float xv = (float)elem16_to_f64(vs[d], src_dtype) / vsc;
                    kd[d] = cache_dtype == O_E4M3 ? pkvo_f32_to_e4m3(xk) : pkvo_f32_to_e5m2(xk);
                    vd[d] = cache_dtype == O_E4M3 ? pkvo_f32_to_e4m3(xv) : pkvo_f32_to_e5m2(xv);
                }
            } else { /* O_U3 */
                int64_t rb = 3 * D / 8;
                pkvo_u3_quantize_pack_rows(ks, src_dtype, 1, D, (uint8_t *)k_cache + row * rb,
                                           &k_qscale[row], &k_qzero[row]);
                pkvo_u3_quantize_pack_rows(vs, src_dtype, 1, D, (uint8_t *)v_cache + row * rb,
                                           &v_qscale[row], &v_qzero[row]);
            }
        }
    }
    return bad;
}

int64_t pkvo_kv_append(int cache_dtype, int src_dtype, int64_t num_tokens, int num_kv_heads,
                       int head_dim, const uint16_t *k_new, const uint16_t *v_new,
                       const int64_t *slot_mapping, int64_t num_blocks, int block_size,
                       void *k_cache, void *v_cache, const float *k_scale,
                       const float *v_scale, uint16_t *k_qscale, uint8_t *k_qzero,
                       uint16_t *v_qscale, uint8_t *v_qzero)
{
    return pkvo_kv_append_scaled(cache_dtype, src_dtype, num_tokens, num_kv_heads, head_dim, k_new,
                                 v_new, slot_mapping, num_blocks, block_size, k_cache, v_cache,
                                 k_scale, v_scale, k_qscale, k_qzero, v_qscale, v_qzero,
                                 SCALE_PER_HEAD, NULL, NULL, NULL, NULL);
}

/* ------------------------------------------------------------------------ */
/* Paged decode: [PAGED] Step 1 + Step 4 reference, in fp64                  */
/* ------------------------------------------------------------------------ */

/* Dequantised element d of cache row `row` (row = (blk*BS + off)*Hkv + h). */
static double cache_elem(int cache_dtype, const void *cache, int64_t row, int D, int d,
                         double scale_h, const uint16_t *qs, const uint8_t *qz)
{
    if (cache_dtype == O_F16)
        return pkvo_f16_to_f64(((const uint16_t *)cache)[row * D + d]);
    if (cache_dtype == O_BF16)
        return pkvo_bf16_to_f64(((const uint16_t *)cache)[row * D + d]);
    if (cache_dtype == O_E4M3)
        return pkvo_e4m3_to_f64(((const uint8_t *)cache)[row * D + d]) * scale_h;
    if (cache_dtype == O_E5M2)
        return pkvo_e5m2_to_f64(((const uint8_t *)cache)[row * D + d]) * scale_h;
    if (cache_dtype == O_I8)
        return (double)((const int8_t *)cache)[row * D + d] * scale_h;
    /* O_U3: bit 3d of the row's little-endian bit stream */
    const uint8_t *p = (const uint8_t *)cache + row * (int64_t)(3 * D / 8);
    uint8_t v[8];
    pkvo_unpack3_octet(p + 3 * (d / 8), v);
    double s = pkvo_f16_to_f64(qs[row]);
    return ((double)v[d % 8] - (double)qz[row]) * s;
}

/* out[b, h, :] = softmax_t(sm_scale * q[b,h,:] . k_t) @ v_t over t < ctx_b,
 * K/V gathered through block_tables.  `pairs` (optional) lists the flattened
 * b*num_heads + h rows to compute; other rows of `out` are left untouched.
 * Returns the number of rows that met an out-of-range block id or context
 * length (those rows are set to NaN). */
int64_t pkvo_paged_decode_scaled(int cache_dtype, int q_dtype, int B, int Hq, int Hkv, int D, int BS,
                                 const uint16_t *q, const void *k_cache, const void *v_cache,
                                 int64_t num_blocks, const int32_t *block_tables, int max_blocks,
                                 const int32_t *context_lens, double sm_scale, const float *k_scale,
                                 const float *v_scale, const uint16_t *k_qscale,
                                 const uint8_t *k_qzero, const uint16_t *v_qscale,
                                 const uint8_t *v_qzero, const int32_t *pairs, int64_t n_pairs,
                                 double *out, int nthreads, int scale_mode, const float *k_scales,
                                 const float *v_scales)
{
    int64_t n_rows = pairs ? n_pairs : (int64_t)B * Hq;
    int64_t bad = 0;
    int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(+ : bad)
#endif
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t bh = pairs ? pairs[r] : r;
        int b = (int)(bh / Hq), h = (int)(bh % Hq);
        int kvh = h / G;
        int ctx = context_lens[b];
        double *o = out + bh * D;
        if (ctx == 0) {
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            continue;
        }
        if (ctx < 0 || ctx > (int64_t)max_blocks * BS) {
            for (int d = 0; d < D; ++d)
                o[d] = NAN;
            ++bad;
            continue;
        }
        double qd[1024];
        for (int d = 0; d < D; ++d)
            qd[d] = elem16_to_f64(q[bh * D + d], q_dtype);
        /* pass 1: scores and their maximum */
        double *score = (double *)malloc(sizeof(double) * (size_t)ctx);
        double m = -INFINITY;
        int ok = 1;
        for (int t = 0; t < ctx; ++t) {
            int32_t pb = block_tables[(int64_t)b * max_blocks + t / BS];
            if (pb < 0 || pb >= num_blocks) {
                ok = 0;
                break;
            }
            int64_t row = ((int64_t)pb * BS + t % BS) * Hkv + kvh;
            double ks = row_scale(scale_mode, k_scale, k_scales, pb, t % BS, kvh, Hkv, BS);
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += qd[d] * cache_elem(cache_dtype, k_cache, row, D, d, ks, k_qscale, k_qzero);
            score[t] = acc * sm_scale;
            if (score[t] > m)
                m = score[t];
        }
        if (!ok) {
            for (int d = 0; d < D; ++d)
                o[d] = NAN;
            ++bad;
            free(score);
            continue;
        }
        /* pass 2: exp-normalised weights and the weighted sum of values */
        double l = 0.0;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int t = 0; t < ctx; ++t) {
            int32_t pb = block_tables[(int64_t)b * max_blocks + t / BS];
            int64_t row = ((int64_t)pb * BS + t % BS) * Hkv + kvh;
            double vs = row_scale(scale_mode, v_scale, v_scales, pb, t % BS, kvh, Hkv, BS);
            double p = exp(score[t] - m);
            l += p;
            for (int d = 0; d < D; ++d)
                o[d] += p * cache_elem(cache_dtype, v_cache, row, D, d, vs, v_qscale, v_qzero);
        }
        for (int d = 0; d < D; ++d)
            o[d] /= l;
        free(score);
    }
    return bad;
}

int64_t pkvo_paged_decode(int cache_dtype, int q_dtype, int B, int Hq, int Hkv, int D, int BS,
                          const uint16_t *q, const void *k_cache, const void *v_cache,
                          int64_t num_blocks, const int32_t *block_tables, int max_blocks,
                          const int32_t *context_lens, double sm_scale, const float *k_scale,
                          const float *v_scale, const uint16_t *k_qscale,
                          const uint8_t *k_qzero, const uint16_t *v_qscale,
                          const uint8_t *v_qzero, const int32_t *pairs, int64_t n_pairs,
                          double *out, int nthreads)
{
    return pkvo_paged_decode_scaled(cache_dtype, q_dtype, B, Hq, Hkv, D, BS, q, k_cache, v_cache,
                                    num_blocks, block_tables, max_blocks, context_lens, sm_scale,
                                    k_scale, v_scale, k_qscale, k_qzero, v_qscale, v_qzero, pairs,
                                    n_pairs, out, nthreads, SCALE_PER_HEAD, NULL, NULL);
}

int pkvo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Array forms of the scalar conversions (for the tests' sweeps)             */
/* ------------------------------------------------------------------------ */

void pkvo_f32_to_e4m3_n(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_f32_to_e4m3(x[i]);
}

void pkvo_f32_to_f16_n(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_f32_to_f16_rn(x[i]);
}

void pkvo_f16_to_f64_n(const uint16_t *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_f16_to_f64(x[i]);
}

void pkvo_bf16_to_f64_n(const uint16_t *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_bf16_to_f64(x[i]);
}

void pkvo_e4m3_to_f64_n(const uint8_t *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_e4m3_to_f64(x[i]);
}

void pkvo_f32_to_e5m2_n(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_f32_to_e5m2(x[i]);
}

void pkvo_f32_to_i8_n(const float *x, int8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_f32_to_i8(x[i]);
}

void pkvo_e5m2_to_f64_n(const uint8_t *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = pkvo_e5m2_to_f64(x[i]);
}
