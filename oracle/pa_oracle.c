/*
 * pa_oracle.c -- plain, slow, single-threaded CPU oracle for FP8 paged decode
 * attention and the FP8 paged-cache append scatter.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; it exists so that the CUDA library can be checked against an
 * independent statement of what the pages compute. It shares no code, header,
 * table or constant with the CUDA sources.
 *
 * Sources (web pages, cited by title and section):
 *  [PA]  "PyPTO 实现 GLM-4.5 Paged Attention FP8 量化算子 ... Kernel 实战解析":
 *        sections 计算流程 (steps 1-10), Kernel 签名与源码对应关系,
 *        Dtype 转换流程与量化策略, 量化策略, 注意事项.
 *  [SC]  "CANN ops-transformer 中的 FP8 KV Cache 更新算子
 *        scatter_pa_kv_cache_with_k_scale 使用指南": sections
 *        功能说明与计算公式, 参数说明, 约束说明, Kernel 实现 (边界防御).
 *  [KC]  "CANN ops-transformer aclnnKvCompressEpilog 算子详解": section
 *        计算公式, 场景 1 (scale_g = max|x_g| / FP8_MAX, q = round(x / scale_g)),
 *        and the FP8_E4M3FN max value 448 quoted there.
 *  [MS]  "PyPTO-Gym 算子实战：DeepSeek V32 MLA 的 Sparse Attention FP8
 *        反量化算子（Ascend 950PR）解析与验证": sections 核心参数与 KV Cache
 *        布局, API 签名与 Decode / Prefill 差异, 计算流程：5 层嵌套循环,
 *        关键实现细节, 在线反量化与 Online Softmax 的实现细节.
 *
 * Precision: every step is done in the precision the pages fix (FP32 for
 * dequant, softmax and accumulation; E4M3 for Q/K/V/P; BF16 output). The two
 * FP8 matmuls have no fixed summation order on the pages; here each dot
 * product is summed in double, which is exact for E4M3 x E4M3 products of up
 * to 2^15 terms, and rounded once to float: the exactly rounded FP32 result.
 *
 * Parity pins (tests/): E4M3 decode/encode against torch.float8_e4m3fn, the
 * scatter worked example of [SC], brute-force FP64 attention, closed forms
 * (all-equal K, one-token context), block-table permutation invariance and a
 * separately written single-pass softmax for one-tile contexts.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------------- */
/* E4M3 (float8_e4m3fn) codec, written from the format definition:         */
/* 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinity,   */
/* S.1111.111 is NaN, largest finite 448 = 1.75 * 2^8 ([KC] FP8_E4M3FN_MAX),*/
/* subnormals m * 2^-9.                                                     */
/* ---------------------------------------------------------------------- */

double or_e4m3_decode(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(8.0 + (double)m, e - 7 - 3); /* (1 + m/8) * 2^(e-7)   */
    return s ? -v : v;
}

/* Round-half-to-even of a non-negative double y that is exactly a float
 * scaled by a power of two (so y - floor(y) is exact). */
static double rne_nonneg(double y)
{
    double f = floor(y);
    double r = y - f;
    if (r > 0.5)
        return f + 1.0;
    if (r < 0.5)
        return f;
    return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* float -> E4M3, round to nearest even, saturating to +-448 ("satfinite");
 * NaN -> 0x7F. The sign of zero is kept. */
uint8_t or_e4m3_encode(float x)
{
    uint8_t sign;
    double a, q;
    int e;
    if (isnan(x))
        return 0x7F;
    sign = signbit(x) ? 0x80 : 0x00;
    a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: multiples of 2^-9; q == 8 is the smallest normal,
         * whose code (exponent field 1, mantissa 0) is also 8 */
        q = rne_nonneg(ldexp(a, 9));
        return sign | (uint8_t)q;
    }
    frexp(a, &e);          /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                /* a = (1 + frac) * 2^e        */
    q = rne_nonneg(ldexp(a, 3 - e)); /* in [8, 16]         */
    if (q >= 16.0) {
        q = 8.0;
        e += 1;
    }
    {
        int code = ((e + 7) << 3) | ((int)q - 8);
        if (code > 0x7E)
            code = 0x7E;
        return sign | (uint8_t)code;
    }
}

/* BF16 <-> float. Rounding is to nearest even on the float bit pattern. */
uint16_t or_bf16_from_float(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if (isnan(x))
        return 0x7FC0;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

float or_bf16_to_float(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Array forms of the codec (element by element, same functions). */
void or_e4m3_encode_array(const float* x, int64_t n, uint8_t* out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_e4m3_encode(x[i]);
}

void or_bf16_from_float_array(const float* x, int64_t n, uint16_t* out)
{
    int64_t i;
    for (i = 0; i < n; ++i)
        out[i] = or_bf16_from_float(x[i]);
}

/* ---------------------------------------------------------------------- */
/* Quantisers.                                                             */
/* ---------------------------------------------------------------------- */

/* One quantisation group: dequant scale = amax / 448 in FP32 ([KC] 场景 1,
 * the per-token Q/K strategy of [PA] 量化策略), codes = E4M3(x / scale).
 * amax == 0 (excluded by [PA] 注意事项, "scale must be non-zero") is read as
 * scale 0 with all-zero codes, so no Inf/NaN is produced. */
static float quant_group(const float* x, ptrdiff_t stride, int n, uint8_t* codes,
                         ptrdiff_t cstride)
{
    float amax = 0.0f, scale;
    int i;
    for (i = 0; i < n; ++i) {
        float a = fabsf(x[i * stride]);
        if (a > amax)
            amax = a;
    }
    scale = amax / 448.0f;
    for (i = 0; i < n; ++i)
        codes[i * cstride] = (scale == 0.0f) ? 0 : or_e4m3_encode(x[i * stride] / scale);
    return scale;
}

/* Per-row quantiser: x[rows][D] (float) -> codes[rows][D], scale[rows].
 * Used for Q and K "per-token" (per token and head) quantisation. */
void or_quant_rows(const float* x, int64_t rows, int D, uint8_t* codes, float* scale)
{
    int64_t r;
    for (r = 0; r < rows; ++r)
        scale[r] = quant_group(x + r * D, 1, D, codes + r * D, 1);
}

/* Per-channel V dequant scale ([PA] 量化策略, "Value 量化 (per-channel)":
 * one scale per head_dim channel, max taken over the sequence of each
 * batch). v[Ttot][H][D] holds the tokens of batch b at rows
 * cu_seqlens[b] .. cu_seqlens[b+1]-1. vscale[B][H][D] = amax / 448. */
void or_value_channel_scale(const float* v, const int64_t* cu_seqlens, int B, int H,
                            int D, float* vscale)
{
    int b, h, d;
    int64_t t;
    for (b = 0; b < B; ++b)
        for (h = 0; h < H; ++h)
            for (d = 0; d < D; ++d) {
                float amax = 0.0f;
                for (t = cu_seqlens[b]; t < cu_seqlens[b + 1]; ++t) {
                    float a = fabsf(v[(t * H + h) * D + d]);
                    if (a > amax)
                        amax = a;
                }
                vscale[((int64_t)b * H + h) * D + d] = amax / 448.0f;
            }
}

/* V codes against a given per-channel dequant scale: E4M3(v / scale),
 * saturating; scale 0 gives code 0. token_batch[t] names the batch of token t. */
void or_quant_channels(const float* v, const int32_t* token_batch, int64_t T, int H,
                       int D, const float* vscale, uint8_t* codes)
{
    int64_t t;
    int h, d;
    for (t = 0; t < T; ++t)
        for (h = 0; h < H; ++h)
            for (d = 0; d < D; ++d) {
                float s = vscale[((int64_t)token_batch[t] * H + h) * D + d];
                float x = v[(t * H + h) * D + d];
                codes[(t * H + h) * D + d] = (s == 0.0f) ? 0 : or_e4m3_encode(x / s);
            }
}

/* ---------------------------------------------------------------------- */
/* Paged cache addressing. Layout 0 = PA_BSND [num_blocks, BS, H, D] ([PA]  */
/* Kernel 签名: k [num_blocks, block_size, NKV, D]); layout 1 = BNBD        */
/* [num_blocks, H, BS, D] ([SC] 参数说明, cache_layout "BNBD"). Scale caches */
/* have the same shapes with D = 1.                                        */
/* ---------------------------------------------------------------------- */

static int64_t cache_row(int layout, int64_t blk, int64_t off, int64_t h, int BS, int H)
{
    if (layout == 0)
        return (blk * BS + off) * H + h;
    return (blk * H + h) * BS + off;
}

/* ---------------------------------------------------------------------- */
/* Cache append scatter ([SC] 功能说明与计算公式): for token i, head j,     */
/*   block_idx = slot[i] / block_size, block_offset = slot[i] % block_size, */
/*   key_cache[block_idx][j][block_offset][:] = key[i][j][:], same for value,*/
/*   key_scale_cache[block_idx][j][block_offset][0] = key_scale[i][j].      */
/* Slots outside [0, num_blocks*block_size) are skipped ([SC] Kernel 实现,   */
/* 边界防御). Bytes are copied as they are (E4M3 or E5M2 alike).            */
/* key_scale may have a non-contiguous tail: element (i, j) sits at         */
/* key_scale[i * ks_stride0 + j * ks_stride1] ([SC] 参数说明).              */
/* ---------------------------------------------------------------------- */
void or_cache_scatter(const uint8_t* key, const uint8_t* value, uint8_t* key_cache,
                      uint8_t* value_cache, const int64_t* slot, const float* key_scale,
                      int64_t ks_stride0, int64_t ks_stride1, float* key_scale_cache,
                      int64_t T, int H, int Dk, int Dv, int64_t num_blocks, int BS,
                      int layout)
{
    int64_t i;
    int j;
    int64_t nslots = num_blocks * BS;
    for (i = 0; i < T; ++i) {
        int64_t s = slot[i], blk, off;
        if (s < 0 || s >= nslots)
            continue;
        blk = s / BS;
        off = s % BS;
        for (j = 0; j < H; ++j) {
            int64_t row = cache_row(layout, blk, off, j, BS, H);
            memcpy(key_cache + row * Dk, key + (i * H + j) * Dk, (size_t)Dk);
            memcpy(value_cache + row * Dv, value + (i * H + j) * Dv, (size_t)Dv);
            key_scale_cache[row] = key_scale[i * ks_stride0 + j * ks_stride1];
        }
    }
}

/* Quantise-on-append: key/value given in float (already rounded from BF16 by
 * the caller where the source is BF16). Key: per (token, head) dequant scale
 * amax/448 and codes E4M3(k / scale) ([KC] 场景 1 with the whole head as one
 * group; the per-token-head key_scale of [SC]). Value: codes against the
 * static per-channel scale of the token's batch, vscale[B][H][Dv] (the cache
 * of [SC] stores no value scale). Then scattered as in or_cache_scatter. */
void or_cache_quant_scatter(const float* key, const float* value, uint8_t* key_cache,
                            uint8_t* value_cache, const int64_t* slot,
                            float* key_scale_cache, const float* vscale,
                            const int32_t* token_batch, int64_t T, int H, int Dk, int Dv,
                            int64_t num_blocks, int BS, int layout)
{
    int64_t i;
    int j, d;
    int64_t nslots = num_blocks * BS;
    for (i = 0; i < T; ++i) {
        int64_t s = slot[i], blk, off;
        if (s < 0 || s >= nslots)
            continue;
        blk = s / BS;
        off = s % BS;
        for (j = 0; j < H; ++j) {
            int64_t row = cache_row(layout, blk, off, j, BS, H);
            key_scale_cache[row] =
                quant_group(key + (i * H + j) * Dk, 1, Dk, key_cache + row * Dk, 1);
            for (d = 0; d < Dv; ++d) {
                float sc = vscale[((int64_t)token_batch[i] * H + j) * Dv + d];
                float x = value[(i * H + j) * Dv + d];
                value_cache[row * Dv + d] = (sc == 0.0f) ? 0 : or_e4m3_encode(x / sc);
            }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* KV compress epilog, modes 0 and 1 ([KC] 功能说明与计算公式 场景 1 / 场景 2, */
/* 约束说明 headDim, kvCacheCol 的源码级解读).                              */
/* A BF16 row x[d] (d % 64 == 0, d > 64) is split into the nope part        */
/* x[0, d-64) and the rope part x[d-64, d). The cache row (head_dim bytes)  */
/* receives [rope as BF16, 128 B][nope as E4M3, d-64 B][one scale per group */
/* of 64 nope values: BF16 (mode 0) or E8M0 (mode 1)]; its other bytes and  */
/* rows whose slot is -1 or out of range are left as they are.              */
/* ---------------------------------------------------------------------- */

/* Bytes written per row. */
int64_t or_kvc_concat_bytes(int d, int quant_mode)
{
    int64_t groups = (d - 64 + 63) / 64;
    return (int64_t)(d - 64) + 64 * 2 + groups * (quant_mode == 0 ? 2 : 1);
}

/* Smallest head_dim (row pitch) the cache must have: the written bytes,
 * rounded up to 32 for mode 0 and not rounded for mode 1. */
int64_t or_kvc_min_head_dim(int d, int quant_mode)
{
    int64_t c = or_kvc_concat_bytes(d, quant_mode);
    return quant_mode == 0 ? (c + 31) / 32 * 32 : c;
}

/* Exponent k of the E8M0 scale 2^k for a group scale s > 0: with
 * round_scale the power of two at or above s (the scale rounded up, [KC]
 * roundScale), without it the power of two at or below s (the exponent of
 * s, its mantissa dropped); clamped to E8M0's finite range [-127, 127]. */
static int e8m0_exponent(float s, int round_scale)
{
    int e, k;
    frexp((double)s, &e); /* s = f * 2^e, f in [0.5, 1) */
    k = e - 1;            /* 2^k <= s < 2^(k+1)       */
    if (round_scale && ldexp(1.0, k) < (double)s)
        k += 1;
    if (k < -127)
        k = -127;
    if (k > 127)
        k = 127;
    return k;
}

/* x: the BF16 rows as their exact float values [bs][d]; cache: block_num
 * blocks of block_stride bytes, row r of a block at r * head_dim. */
void or_kv_compress_epilog(const float* x, int64_t bs, int d, uint8_t* cache, int64_t block_num,
                           int block_size, int64_t block_stride, int head_dim, const int64_t* slot,
                           int quant_mode, int round_scale)
{
    const int nope = d - 64;
    const int groups = (nope + 63) / 64;
    int64_t i;
    for (i = 0; i < bs; ++i) {
        const float* xr = x + i * d;
        int64_t s = slot[i];
        uint8_t* row;
        int g, j;
        if (s < 0 || s >= block_num * block_size)
            continue;
        row = cache + (s / block_size) * block_stride + (s % block_size) * (int64_t)head_dim;
        for (j = 0; j < 64; ++j) { /* rope part, BF16 little-endian, first */
            uint16_t h = or_bf16_from_float(xr[nope + j]);
            row[2 * j] = (uint8_t)(h & 0xFF);
            row[2 * j + 1] = (uint8_t)(h >> 8);
        }
        for (g = 0; g < groups; ++g) {
            const float* xg = xr + 64 * g;
            const int n = nope - 64 * g < 64 ? nope - 64 * g : 64;
            uint8_t* codes = row + 128 + 64 * g;
            float amax = 0.0f, scale;
            for (j = 0; j < n; ++j)
                if (fabsf(xg[j]) > amax)
                    amax = fabsf(xg[j]);
            scale = amax / 448.0f; /* scale_g = max|x_g| / FP8_MAX */
            if (quant_mode == 0) {
                uint8_t* sc = row + 128 + nope + 2 * g;
                uint16_t h = or_bf16_from_float(scale);
                for (j = 0; j < n; ++j)
                    codes[j] = (scale == 0.0f) ? 0 : or_e4m3_encode(xg[j] / scale);
                sc[0] = (uint8_t)(h & 0xFF);
                sc[1] = (uint8_t)(h >> 8);
            } else {
                uint8_t* sc = row + 128 + nope + g;
                if (scale == 0.0f) {
                    for (j = 0; j < n; ++j)
                        codes[j] = 0;
                    sc[0] = 0;
                } else {
                    const int k = e8m0_exponent(scale, round_scale);
                    const float p = (float)ldexp(1.0, k);
                    for (j = 0; j < n; ++j)
                        codes[j] = or_e4m3_encode(xg[j] / p);
                    sc[0] = (uint8_t)(k + 127);
                }
            }
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Paged FP8 decode attention ([PA] 计算流程 steps 1-10, 循环结构).         */
/*                                                                         */
/* q [B*S1, NQ, D] E4M3, q_scale [B*S1, NQ] (dequant), k/v caches in the   */
/* given layout, k_scale per (block, offset, head), v_scale [B, NKV, D],   */
/* block_table [B, max_blocks] int32, kv_act_seqs [B] int32,               */
/* out [B*S1, NQ, D] BF16 bits; out_f32 (optional) the same before the     */
/* BF16 cast. rows (optional, nrows entries) restricts the work to the     */
/* listed output rows (b*S1 + s)*NQ + h; with rows == NULL every row is    */
/* computed.                                                               */
/*                                                                         */
/* For each row the KV tokens are walked in s2_tile-sized tiles (LOOP_s2): */
/*  2. token j -> block block_table[b][j / BS] (-1 read as 0, [PA] 注意事项),*/
/*     offset j % BS; tokens >= kv_act_seqs[b] take no part (valid_shape).  */
/*  3. MM1: acc_j = q . k_j over E4M3 values, FP32 result.                 */
/*  4. dequant: S_j = (acc_j * q_scale) * k_scale_j.                        */
/*  5. S_j *= softmax_scale; M_new = max(M_old, max_j S_j);                 */
/*     P_j = exp(S_j - M_new); Sum = Sum * exp(M_old - M_new) + sum_j P_j.  */
/*  6. per-row P quant: qs = 448 / max_j P_j, P8_j = E4M3(P_j * qs),        */
/*     P_scale = 1 / qs ([PA] 量化策略, "Attention P 量化 (per-token)").     */
/*  7. MM2: ot_d = sum_j P8_j * v_j[d] over E4M3 values, FP32 result.       */
/*  8. dequant: (ot_d * P_scale) * v_scale[d].                              */
/*  9. O_d = O_d * exp(M_old - M_new) + that.                               */
/* 10. out_d = BF16(O_d / Sum).                                            */
/* A row whose kv_act_seqs is <= 0 gets zeros (the pages are silent).       */
/* Returns 0, or -1 on bad arguments / allocation failure.                 */
/* ---------------------------------------------------------------------- */
int or_pa_decode(const uint8_t* q, const float* q_scale, const uint8_t* k_cache,
                 const float* k_scale, const uint8_t* v_cache, const float* v_scale,
                 const int32_t* block_table, const int32_t* kv_act_seqs,
                 uint16_t* out, float* out_f32, int B, int S1, int NQ, int NKV, int D,
                 int BS, int64_t num_blocks, int max_blocks, int layout, int s2_tile,
                 float softmax_scale, const int64_t* rows, int64_t nrows)
{
    double dq[1024];
    float* S;
    float* P;
    uint8_t* P8;
    float* O;
    int64_t total = (int64_t)B * S1 * NQ, ri;
    int group, d;
    (void)num_blocks;
    if (B <= 0 || S1 <= 0 || NQ <= 0 || NKV <= 0 || NQ % NKV || D <= 0 || D > 1024 ||
        BS <= 0 || s2_tile <= 0)
        return -1;
    group = NQ / NKV;
    S = (float*)malloc(sizeof(float) * (size_t)s2_tile);
    P = (float*)malloc(sizeof(float) * (size_t)s2_tile);
    P8 = (uint8_t*)malloc((size_t)s2_tile);
    O = (float*)malloc(sizeof(float) * (size_t)D);
    if (!S || !P || !P8 || !O) {
        free(S); free(P); free(P8); free(O);
        return -1;
    }
    for (ri = 0; ri < (rows ? nrows : total); ++ri) {
        int64_t row = rows ? rows[ri] : ri;      /* (b*S1 + s)*NQ + h */
        int64_t bs;
        int h, b, n2, n, t, T;
        float qsc, M = -INFINITY, L = 0.0f;
        if (row < 0 || row >= total)
            continue;
        bs = row / NQ;
        h = (int)(row % NQ);
        b = (int)(bs / S1);
        n2 = h / group;                            /* GQA: group = nq // nkv */
        n = kv_act_seqs[b];
        qsc = q_scale[row];
        for (d = 0; d < D; ++d) {
            dq[d] = or_e4m3_decode(q[row * D + d]);
            O[d] = 0.0f;
        }
        if (n <= 0) {
            for (d = 0; d < D; ++d) {
                out[row * D + d] = or_bf16_from_float(0.0f);
                if (out_f32)
                    out_f32[row * D + d] = 0.0f;
            }
            continue;
        }
        T = (n + s2_tile - 1) / s2_tile;
        for (t = 0; t < T; ++t) {
            int j0 = t * s2_tile;
            int j1 = (j0 + s2_tile < n) ? j0 + s2_tile : n;
            int j;
            float m_t = -INFINITY, Mn, alpha, sumP = 0.0f, amax = 0.0f, qs, ps;
            /* steps 2-5a: gather, MM1, dequant, softmax scale */
            for (j = j0; j < j1; ++j) {
                int blk = block_table[(int64_t)b * max_blocks + j / BS];
                int64_t krow;
                double acc = 0.0;
                if (blk < 0)
                    blk = 0;
                krow = cache_row(layout, blk, j % BS, n2, BS, NKV);
                for (d = 0; d < D; ++d)
                    acc += dq[d] * or_e4m3_decode(k_cache[krow * D + d]);
                S[j - j0] = (((float)acc * qsc) * k_scale[krow]) * softmax_scale;
                if (S[j - j0] > m_t)
                    m_t = S[j - j0];
            }
            /* step 5b: online softmax state */
            Mn = (M > m_t) ? M : m_t;
            alpha = expf(M - Mn);
            for (j = 0; j < j1 - j0; ++j) {
                P[j] = expf(S[j] - Mn);
                sumP += P[j];
                if (P[j] > amax)
                    amax = P[j];
            }
            L = L * alpha + sumP;
            /* step 6: per-row FP8 quantisation of P over this tile */
            if (amax > 0.0f) {
                qs = 448.0f / amax;
                ps = 1.0f / qs;
                for (j = 0; j < j1 - j0; ++j)
                    P8[j] = or_e4m3_encode(P[j] * qs);
            } else {
                ps = 0.0f;
                for (j = 0; j < j1 - j0; ++j)
                    P8[j] = 0;
            }
            /* steps 7-9: MM2, dequant, accumulate */
            for (d = 0; d < D; ++d) {
                double acc = 0.0;
                float ot;
                for (j = j0; j < j1; ++j) {
                    int blk = block_table[(int64_t)b * max_blocks + j / BS];
                    int64_t vrow;
                    if (blk < 0)
                        blk = 0;
                    vrow = cache_row(layout, blk, j % BS, n2, BS, NKV);
                    acc += or_e4m3_decode(P8[j - j0]) * or_e4m3_decode(v_cache[vrow * D + d]);
                }
                ot = (float)acc;
                O[d] = O[d] * alpha + (ot * ps) * v_scale[((int64_t)b * NKV + n2) * D + d];
            }
            M = Mn;
        }
        /* step 10 */
        for (d = 0; d < D; ++d) {
            float o = O[d] / L;
            out[row * D + d] = or_bf16_from_float(o);
            if (out_f32)
                out_f32[row * D + d] = o;
        }
    }
    free(S);
    free(P);
    free(P8);
    free(O);
    return 0;
}

/* ---------------------------------------------------------------------- */
/* MLA sparse attention with FP8 anti-quantisation, decode ([MS] 核心参数与 */
/* KV Cache 布局, API 签名, 计算流程: 5 层嵌套循环, 关键实现细节,          */
/* 在线反量化与 Online Softmax 的实现细节).                                 */
/*                                                                         */
/* Fixed sizes: kv_lora_rank 512 (the "nope" part), qk_rope_dim 64, so a   */
/* query/key head is 576 wide; one KV head shared by all NQ query heads.   */
/* Cache row (row_bytes >= 656 bytes apart, [MS] pads them to 672), by    */
/* row_format:                                                             */
/*  0 ([MS] 核心参数与 KV Cache 布局):                                      */
/*   [0, 512)    kn, E4M3 codes;                                            */
/*   [512, 640)  kr, 64 BF16 values (little-endian);                        */
/*   [640, 656)  4 FP32 dequant scales, one per 128 channels of kn.         */
/*  1, 2 (the row the KV compress epilog above writes for d = 576, [KC]    */
/*  计算公式 场景 1 / 场景 2, read back by the same dequantisation):        */
/*   [0, 128)    kr, 64 BF16 values;                                        */
/*   [128, 640)  kn, E4M3 codes;                                            */
/*   [640, ...)  one scale per 64 channels of kn: 8 BF16 values (format 1, */
/*               quant mode 0) or 8 E8M0 bytes e for 2^(e - 127) (format 2, */
/*               quant mode 1).                                            */
/* q_nope [T*NQ][512], q_rope [T*NQ][64] BF16 bits, T = B*S1 query tokens, */
/* token t = b*S1 + s. topk_indices [T][topk] int32: positions in the      */
/* sequence of the selected keys. block_table [B][max_blocks] int32,       */
/* kv_act_seqs [B]. out [T*NQ][512] BF16 bits (out_f32: before the cast).  */
/*                                                                         */
/* For query token t and head h:                                           */
/*  - cur = clamp(kv_act_seqs[b] - S1 + 1 + s, 0, topk): only the first    */
/*    cur selected keys take part ([MS] 关键实现细节, 动态序列裁剪).         */
/*  - those keys are walked in s2_tile-sized tiles; key j of a tile:       */
/*    idx = topk_indices[t][j]; physical row                               */
/*    block_table[b][idx / BS] * BS + idx % BS (a block id of -1, or any   */
/*    id outside the pool, is read as block 0).                            */
/*    An idx outside [0, kv_act_seqs[b]) takes no part (the pages only     */
/*    produce valid positions; masking is the plain reading of "-1" pads). */
/*  - dequant: kn_j[c] = BF16(FP32(E4M3(code)) * scale of c's group);      */
/*    k_j = [kn_j, kr_j] (576), q = [q_nope, q_rope] (576).                */
/*  - C1: s_j = q . k_j, FP32 result (products of BF16 are exact; summed   */
/*    in double and rounded once); S_j = s_j * softmax_scale.              */
/*  - V1 per tile: m = max S_j, p_j = exp(S_j - m), l = sum p_j (FP32),    */
/*    P_j = BF16(p_j).                                                     */
/*  - C2: o[c] = sum_j P_j * kn_j[c] for c < 512 (V reuses kn), FP32.      */
/*  - online update: the first tile sets O = o, L = l, M = m; a later tile */
/*    takes Mn = max(M, m), a = exp(M - Mn), b = exp(m - Mn),              */
/*    O = O * a + o * b, L = L * a + l * b, M = Mn.                         */
/*  - out[c] = BF16(O[c] / L).                                             */
/* A tile with no valid key changes nothing; a row with no valid key at    */
/* all gets zeros (the pages are silent on both).                          */
/* rows (optional) restricts the work to the listed flat rows t*NQ + h.    */
/* Returns 0, or -1 on bad arguments / allocation failure.                 */
/* ---------------------------------------------------------------------- */
int or_mla_sparse_decode(const uint16_t* q_nope, const uint16_t* q_rope, const uint8_t* cache,
                         int64_t row_bytes, const int32_t* topk_indices, int topk,
                         const int32_t* block_table, const int32_t* kv_act_seqs, uint16_t* out,
                         float* out_f32, int B, int S1, int NQ, int BS, int64_t num_blocks,
                         int max_blocks, int s2_tile, float softmax_scale, const int64_t* rows,
                         int64_t nrows, int row_format)
{
    enum { DN = 512, DR = 64, DK = 576 };
    float* kn;   /* [s2_tile][512] dequantised kn of the tile (BF16 values) */
    float* kr;   /* [s2_tile][64]  */
    float* S;
    float* P;
    uint8_t* ok;
    double q[DK];
    float O[DN];
    int64_t total = (int64_t)B * S1 * NQ, ri;
    if (B <= 0 || S1 <= 0 || NQ <= 0 || BS <= 0 || topk < 0 || s2_tile <= 0 ||
        row_bytes < 656 || num_blocks <= 0 || max_blocks <= 0 || row_format < 0 ||
        row_format > 2)
        return -1;
    kn = (float*)malloc(sizeof(float) * (size_t)s2_tile * DN);
    kr = (float*)malloc(sizeof(float) * (size_t)s2_tile * DR);
    S = (float*)malloc(sizeof(float) * (size_t)s2_tile);
    P = (float*)malloc(sizeof(float) * (size_t)s2_tile);
    ok = (uint8_t*)malloc((size_t)s2_tile);
    if (!kn || !kr || !S || !P || !ok) {
        free(kn); free(kr); free(S); free(P); free(ok);
        return -1;
    }
    for (ri = 0; ri < (rows ? nrows : total); ++ri) {
        int64_t row = rows ? rows[ri] : ri; /* t*NQ + h */
        int64_t t;
        int b, s, act, cur, j0, c, any = 0;
        float M = -INFINITY, L = 0.0f;
        if (row < 0 || row >= total)
            continue;
        t = row / NQ;
        b = (int)(t / S1);
        s = (int)(t % S1);
        act = kv_act_seqs[b];
        cur = act - S1 + 1 + s;
        if (cur < 0)
            cur = 0;
        if (cur > topk)
            cur = topk;
        for (c = 0; c < DN; ++c) {
            q[c] = or_bf16_to_float(q_nope[row * DN + c]);
            O[c] = 0.0f;
        }
        for (c = 0; c < DR; ++c)
            q[DN + c] = or_bf16_to_float(q_rope[row * DR + c]);
        for (j0 = 0; j0 < cur; j0 += s2_tile) {
            int n = (cur - j0 < s2_tile) ? cur - j0 : s2_tile, j;
            float m = -INFINITY, l = 0.0f;
            /* gather + dequant + C1 + scale */
            for (j = 0; j < n; ++j) {
                int idx = topk_indices[t * topk + j0 + j];
                const uint8_t* kv;
                const uint8_t* code; /* the 512 kn codes of the row */
                const uint8_t* rope; /* its 64 BF16 kr values       */
                float sc[8];         /* the scale of each 64 channels */
                int blk;
                double acc = 0.0;
                ok[j] = (uint8_t)(idx >= 0 && idx < act);
                if (!ok[j])
                    continue;
                blk = block_table[(int64_t)b * max_blocks + idx / BS];
                if (blk < 0 || blk >= num_blocks)
                    blk = 0;
                kv = cache + ((int64_t)blk * BS + idx % BS) * row_bytes;
                if (row_format == 0) {
                    float s4[4];
                    memcpy(s4, kv + 640, sizeof(s4));
                    for (c = 0; c < 8; ++c)
                        sc[c] = s4[c / 2]; /* one FP32 scale per 128 channels */
                    code = kv;
                    rope = kv + DN;
                } else {
                    for (c = 0; c < 8; ++c)
                        sc[c] = row_format == 1
                                    ? or_bf16_to_float((uint16_t)(kv[640 + 2 * c] |
                                                                  (kv[640 + 2 * c + 1] << 8)))
                                    : (float)ldexp(1.0, (int)kv[640 + c] - 127);
                    code = kv + 2 * DR;
                    rope = kv;
                }
                for (c = 0; c < DN; ++c) {
                    float f = (float)or_e4m3_decode(code[c]) * sc[c / 64];
                    kn[(int64_t)j * DN + c] = or_bf16_to_float(or_bf16_from_float(f));
                }
                for (c = 0; c < DR; ++c)
                    kr[(int64_t)j * DR + c] =
                        or_bf16_to_float((uint16_t)(rope[2 * c] | (rope[2 * c + 1] << 8)));
                for (c = 0; c < DN; ++c)
                    acc += q[c] * (double)kn[(int64_t)j * DN + c];
                for (c = 0; c < DR; ++c)
                    acc += q[DN + c] * (double)kr[(int64_t)j * DR + c];
                S[j] = (float)acc * softmax_scale;
                if (S[j] > m)
                    m = S[j];
            }
            if (m == -INFINITY)
                continue; /* no valid key in this tile */
            /* V1: tile-local softmax numerator, its sum and the BF16 cast */
            for (j = 0; j < n; ++j) {
                float p = ok[j] ? expf(S[j] - m) : 0.0f;
                l += p;
                P[j] = or_bf16_to_float(or_bf16_from_float(p));
            }
            /* C2 and the online update */
            {
                float a = 1.0f, bb = 1.0f, Mn = m;
                if (any) {
                    Mn = (M > m) ? M : m;
                    a = expf(M - Mn);
                    bb = expf(m - Mn);
                }
                for (c = 0; c < DN; ++c) {
                    double acc = 0.0;
                    float o;
                    for (j = 0; j < n; ++j)
                        if (ok[j])
                            acc += (double)P[j] * (double)kn[(int64_t)j * DN + c];
                    o = (float)acc;
                    O[c] = any ? O[c] * a + o * bb : o;
                }
                L = any ? L * a + l * bb : l;
                M = Mn;
                any = 1;
            }
        }
        for (c = 0; c < DN; ++c) {
            float o = any ? O[c] / L : 0.0f;
            out[row * DN + c] = or_bf16_from_float(o);
            if (out_f32)
                out_f32[row * DN + c] = o;
        }
    }
    free(kn);
    free(kr);
    free(S);
    free(P);
    free(ok);
    return 0;
}
