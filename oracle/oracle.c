/*
 * Plain CPU oracle for MoE top-k token dispatch and combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark use this file.  It shares no code, header,
 * table or constant generator with the CUDA library; it is written from the
 * pages' statement of the problem and from the number-format definitions.
 *
 * Sources (cited by page title and section):
 *   [AX]  axolotl docs, integrations.expert_parallel.torch_dispatch:
 *         module description (the DeepEP layout contract), compute_send_counts,
 *         build_send_layout, dispatch, combine, chunk_bounds,
 *         dispatch_chunked_forward.
 *   [UB]  NeMo AutoModel docs, nemo_automodel.components.moe.uccl_ep.buffer:
 *         Buffer.get_dispatch_layout, Buffer.dispatch (fp8 payload: e4m3
 *         [T,H] + fp32 scales [T,H/128]), Buffer.combine (addition without
 *         weights), Buffer.low_latency_dispatch (round_scale, use_ue8m0,
 *         column-major scales), Buffer.low_latency_combine (reduce with
 *         weights).
 *   [VB]  vLLM docs, vllm.model_executor.layers.fused_moe.prepare_finalize:
 *         BatchedPrepareAndFinalize.prepare (hit mask, tokens_per_expert,
 *         slots that preserve token order) and .finalize.
 *   [ND]  NeMo AutoModel docs, ...moe.megatron.token_dispatcher:
 *         TokenDispatcherConfig.moe_router_dtype (weighting in fp32),
 *         moe_expert_capacity_factor, moe_router_expert_pad_multiple.
 *   bfloat16: the upper half of an IEEE-754 binary32.
 *   E4M3: OCP 8-bit Floating Point Specification (OFP8) v1.0, E4M3 format
 *         (bias 7, no infinities, S.1111.111 is NaN, max finite 448).
 *
 * Readings where the pages are silent (each restated where it is used):
 *   - an expert id outside [-1, E) sets error bit 2 and the slot counts as
 *     unrouted;
 *   - tokens_per_expert counts a token once per expert even if two of its
 *     slots name the same expert (the hit mask of [VB] takes `any` over K);
 *   - send_w is +0.0f on slots owned elsewhere; owned slots copy the input;
 *   - combine accumulates in fp32 starting from +0.0f, in ascending rank
 *     order (send layout) or ascending k order with fused multiply-add
 *     (expert-batched layout), and rounds once to bf16 at the end;
 *   - fp8: per 128-element group a = max(max|x|, 1e-4f), inv = 448/a,
 *     q = e4m3_rn_satfinite(x * inv), scale = a / 448, all fp32 with
 *     round-to-nearest-even;
 *   - chunk_bounds: chunk size floor(T / C); the last chunk takes the rest;
 *   - expert-batched capacity: a token past max_num_tokens is dropped (slot
 *     -1, row not written), tokens_per_expert is clipped, error bit 8;
 *   - power-of-two scales (round_scale): the smallest power of two >= a/448,
 *     so x / scale never exceeds 448; the UE8M0 code is its biased exponent;
 *     four codes pack into an int32 with group 4j+i at byte i (least
 *     significant first);
 *   - non-finite inputs to the fp8 quantisers: NaN elements do not enter the
 *     group maximum; a group holding +-inf has a = inf, so scale = +inf and
 *     the reciprocal is +0 in both forms (the plain form by IEEE division;
 *     the power-of-two form by the same choice, UE8M0 code 255): its finite
 *     elements give +-0 codes and its infinities and NaNs NaN codes, whose
 *     sign IEEE leaves to the implementation;
 *   - capacity: an expert keeps its first `capacity` tokens in token order,
 *     later ones are dropped and counted (no error bit); capacity from a
 *     factor is ceil(factor * T * K / E);
 *   - alignment: the kept per-expert count is rounded up to the alignment
 *     (at most M) and the rows in between are zero rows; on the send layout
 *     every rank segment is padded to a multiple of the alignment with rows
 *     that carry no token.
 *
 * Build: plain C11, -O2 -fno-fast-math -ffp-contract=off (no contraction of
 * a*b+c, so every rounding is the one written here).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_ERR_INVALID_EXPERT 2
#define ORC_ERR_CAPACITY 8

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

float orc_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to bfloat16, nearest with ties to even.  Rounding keeps
 * the upper 16 bits after adding half an ulp of the kept part (plus one when
 * the kept part is odd, which sends exact ties to the even neighbour). */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN: keep it a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7fffu + keep_lsb;
    return (uint16_t)(u >> 16);
}

/* Decode one E4M3 code.  Normal: (1 + m/8) * 2^(e-7); subnormal (e == 0):
 * (m/8) * 2^-6; S.1111.111 is NaN. */
float orc_e4m3_to_f32(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 0xf, m = b & 7;
    if (e == 15 && m == 7)
        return NAN;
    float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return s ? -v : v;
}

/* Encode a binary32 as E4M3 with round-to-nearest-even and saturation to the
 * largest finite magnitude (448); NaN stays NaN.
 *
 * Every E4M3 value is an integer multiple of a quantum 2^(E-3), where E is
 * the exponent of the value's binade clamped below at -6 (the subnormal
 * range shares the quantum of the first normal binade).  The value is scaled
 * by the quantum (exact, a power of two), rounded to an integer with ties to
 * even, and re-encoded; a carry into the next binade is handled explicitly. */
uint8_t orc_f32_to_e4m3(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    if (isnan(f))
        return (uint8_t)(sign | 0x7f);
    float a = fabsf(f);
    if (a >= 448.0f)                               /* includes +inf */
        return (uint8_t)(sign | 0x7e);
    int ex;
    (void)frexpf(a, &ex);                          /* a = fr * 2^ex, fr in [0.5,1) */
    int E = ex - 1;                                /* binade: a in [2^E, 2^(E+1)) */
    if (E < -6)
        E = -6;
    float m = ldexpf(a, 3 - E);                    /* exact: a / 2^(E-3), in [0,16) */
    int mi = (int)rintf(m);                        /* nearest, ties to even */
    if (mi == 16) {                                /* carried into the next binade */
        mi = 8;
        E += 1;
    }
    if (E > 8 || (E == 8 && mi > 14))
        return (uint8_t)(sign | 0x7e);
    if (mi < 8)                                    /* subnormal (E == -6) or zero */
        return (uint8_t)(sign | mi);
    return (uint8_t)(sign | ((E + 7) << 3) | (mi - 8));
}

/* Array forms of the conversions above (one call per array). */
void orc_f32_to_bf16_array(const float *f, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_bf16(f[i]);
}

void orc_f32_to_e4m3_array(const float *f, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_f32_to_e4m3(f[i]);
}

void orc_e4m3_to_f32_array(const uint8_t *b, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_to_f32(b[i]);
}

/* ------------------------------------------------------------------------ */
/* [AX] chunk_bounds: C contiguous [start,end) ranges, the last takes the     */
/* remainder (so leading chunks are empty when T < C).                       */
/* ------------------------------------------------------------------------ */
void orc_chunk_bounds(int64_t T, int C, int64_t *bounds)
{
    int64_t size = T / C;
    for (int i = 0; i < C; ++i)
        bounds[i] = (int64_t)i * size;
    bounds[C] = T;
}

/* ------------------------------------------------------------------------ */
/* [AX] compute_send_counts / [UB] Buffer.get_dispatch_layout.               */
/* dest[t,k]      owning rank of slot k (idx / E_local), -1 where unrouted   */
/* is_in_rank[t,p] 1 iff some slot of t is owned by rank p                   */
/* send_counts[p]  number of tokens sent to rank p                           */
/* tokens_per_expert[e] (optional) tokens with some slot naming expert e     */
/* Returns error bits.                                                       */
/* ------------------------------------------------------------------------ */
int orc_compute_send_counts(const int64_t *topk_idx, int64_t T, int K, int P, int E_local,
                            int32_t *dest, uint8_t *is_in_rank, int32_t *send_counts,
                            int32_t *tokens_per_expert)
{
    int err = 0;
    int64_t E = (int64_t)P * E_local;
    for (int p = 0; p < P; ++p)
        send_counts[p] = 0;
    if (tokens_per_expert)
        for (int64_t e = 0; e < E; ++e)
            tokens_per_expert[e] = 0;

    for (int64_t t = 0; t < T; ++t) {
        for (int p = 0; p < P; ++p)
            is_in_rank[t * P + p] = 0;
        for (int k = 0; k < K; ++k) {
            int64_t id = topk_idx[t * K + k];
            int32_t d = -1;
            if (id >= 0 && id < E) {
                d = (int32_t)(id / E_local);
            } else if (id != -1) {
                err |= ORC_ERR_INVALID_EXPERT;
            }
            dest[t * K + k] = d;
            if (d >= 0)
                is_in_rank[t * P + d] = 1;
            if (d >= 0 && tokens_per_expert) {
                int seen = 0;
                for (int j = 0; j < k; ++j)
                    if (topk_idx[t * K + j] == id)
                        seen = 1;
                if (!seen)
                    tokens_per_expert[id] += 1;
            }
        }
        for (int p = 0; p < P; ++p)
            send_counts[p] += is_in_rank[t * P + p];
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* [AX] build_send_layout: rank-major, token-ascending send order.           */
/* For each rank p (ascending) and each token t (ascending) with             */
/* is_in_rank[t,p], one row n:                                               */
/*   send_token_idx[n] = t, send_rank[n] = p, token_pos[t,p] = n,            */
/*   send_idx[n,k] = idx[t,k] - p*E_local if dest[t,k] == p, else -1,        */
/*   send_w[n,k]   = w[t,k]               if dest[t,k] == p, else +0.0f.     */
/* token_pos[t,p] = -1 where t is not sent to p (the combine handle).        */
/* Writes at most num_send rows; returns the number of rows in the layout.   */
/* ------------------------------------------------------------------------ */
int64_t orc_build_send_layout(const int64_t *topk_idx, const float *topk_weights,
                              const int32_t *dest, const uint8_t *is_in_rank,
                              int64_t T, int K, int P, int E_local, int64_t num_send,
                              int32_t *send_token_idx, int32_t *send_rank,
                              int64_t *send_idx, float *send_w, int32_t *token_pos)
{
    for (int64_t i = 0; i < T * P; ++i)
        token_pos[i] = -1;
    int64_t n = 0;
    for (int p = 0; p < P; ++p) {
        for (int64_t t = 0; t < T; ++t) {
            if (!is_in_rank[t * P + p])
                continue;
            if (n < num_send) {
                send_token_idx[n] = (int32_t)t;
                send_rank[n] = p;
                token_pos[t * P + p] = (int32_t)n;
                for (int k = 0; k < K; ++k) {
                    if (dest[t * K + k] == p) {
                        send_idx[n * K + k] = topk_idx[t * K + k] - (int64_t)p * E_local;
                        send_w[n * K + k] = topk_weights[t * K + k];
                    } else {
                        send_idx[n * K + k] = -1;
                        send_w[n * K + k] = 0.0f;
                    }
                }
            }
            ++n;
        }
    }
    return n;
}

/* ------------------------------------------------------------------------ */
/* [AX] dispatch (collective-free local path): recv_x[n] = x[send_token_idx[n]] */
/* bit copy of bf16 rows.                                                    */
/* ------------------------------------------------------------------------ */
void orc_dispatch(const uint16_t *x, int H, const int32_t *send_token_idx, int64_t N,
                  uint16_t *recv_x)
{
    for (int64_t n = 0; n < N; ++n)
        memcpy(recv_x + n * H, x + (int64_t)send_token_idx[n] * H, (size_t)H * sizeof(uint16_t));
}

/* ------------------------------------------------------------------------ */
/* Per-token 1x128-group fp8 e4m3 quantisation of bf16 rows ([UB]            */
/* Buffer.dispatch fp8 payload: e4m3 [T,H] with fp32 scales [T,H/128]).      */
/* For each row and group g of 128 columns:                                  */
/*   a      = max(max_i |x_i|, 1e-4f)                                        */
/*   inv    = 448.0f / a              (fp32, nearest-even)                   */
/*   q_i    = e4m3_rn_satfinite(x_i * inv)                                   */
/*   scale  = a / 448.0f              (fp32, nearest-even)                   */
/* so that q_i * scale approximates x_i.  H must be a multiple of 128.       */
/* ------------------------------------------------------------------------ */
void orc_quantize_fp8_rows(const uint16_t *x, int64_t rows, int H, uint8_t *q, float *scale)
{
    int G = H / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int g = 0; g < G; ++g) {
            const uint16_t *xs = x + r * H + (int64_t)g * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(orc_bf16_to_f32(xs[i]));
                if (v > amax)
                    amax = v;
            }
            float a = amax > 1e-4f ? amax : 1e-4f;
            float inv = 448.0f / a;
            for (int i = 0; i < 128; ++i)
                q[r * H + (int64_t)g * 128 + i] = orc_f32_to_e4m3(orc_bf16_to_f32(xs[i]) * inv);
            scale[r * G + g] = a / 448.0f;
        }
    }
}

/* fp8 dispatch: each token is quantised once (per-token groups), and every  */
/* row sent for it carries the same bytes.                                   */
void orc_dispatch_fp8(const uint16_t *x, int64_t T, int H, const int32_t *send_token_idx,
                      int64_t N, uint8_t *recv_q, float *recv_scale)
{
    int G = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)T * H);
    float *s = (float *)malloc((size_t)T * G * sizeof(float));
    orc_quantize_fp8_rows(x, T, H, q, s);
    for (int64_t n = 0; n < N; ++n) {
        int64_t t = send_token_idx[n];
        memcpy(recv_q + n * H, q + t * H, (size_t)H);
        memcpy(recv_scale + n * G, s + t * G, (size_t)G * sizeof(float));
    }
    free(q);
    free(s);
}

/* ------------------------------------------------------------------------ */
/* Synthetic local expert kernel for the fp8 chunked workload (the           */
/* local_kernel of [AX] dispatch_chunked_forward): expert l maps a token to  */
/* dequant(x) * (1 + l/64) in bf16, and the local kernel weights and sums    */
/* over K ([AX] module description):                                         */
/*   d        = e4m3(q) * scale                     (fp32)                   */
/*   y_k      = bf16(d * (1 + l_k/64))              for slots with l_k >= 0  */
/*   acc      = fma(w_k, y_k, acc), k ascending, from +0.0f                  */
/*   out[n]   = bf16(acc)                                                    */
/* ------------------------------------------------------------------------ */
void orc_local_expert_fp8(const uint8_t *q, const float *scale, const int64_t *send_idx,
                          const float *send_w, int64_t N, int K, int H, uint16_t *out)
{
    int G = H / 128;
    for (int64_t n = 0; n < N; ++n) {
        for (int h = 0; h < H; ++h) {
            float d = orc_e4m3_to_f32(q[n * H + h]) * scale[n * G + h / 128];
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int64_t l = send_idx[n * K + k];
                if (l < 0)
                    continue;
                float y = orc_bf16_to_f32(orc_f32_to_bf16(d * (1.0f + (float)l / 64.0f)));
                acc = fmaf(send_w[n * K + k], y, acc);
            }
            out[n * H + h] = orc_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* [AX] combine / [UB] Buffer.combine (an unweighted sum):                  */
/* out[t] = sum over ranks p ascending with token_pos[t,p] >= 0 of           */
/*          Y[token_pos[t,p]], accumulated in fp32 from +0.0f, then rounded  */
/* once to bf16 (out_f32 == 0) or stored as fp32 (out_f32 == 1).  A token    */
/* that was not sent anywhere combines to +0.                                */
/* ------------------------------------------------------------------------ */
void orc_combine(const uint16_t *y, int64_t T, int H, int P, const int32_t *token_pos,
                 int out_f32, void *out)
{
    float *acc = (float *)malloc((size_t)H * sizeof(float));
    for (int64_t t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h)
            acc[h] = 0.0f;
        for (int p = 0; p < P; ++p) {
            int64_t n = token_pos[t * P + p];
            if (n < 0)
                continue;
            for (int h = 0; h < H; ++h)
                acc[h] = acc[h] + orc_bf16_to_f32(y[n * H + h]);
        }
        for (int h = 0; h < H; ++h) {
            if (out_f32)
                ((float *)out)[t * H + h] = acc[h];
            else
                ((uint16_t *)out)[t * H + h] = orc_f32_to_bf16(acc[h]);
        }
    }
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* [VB] BatchedPrepareAndFinalize.prepare, unquantised branch.               */
/* Local experts are [rank*E_local, (rank+1)*E_local).  For local expert     */
/* e_l and tokens t in ascending order that name it in some slot, the s-th   */
/* such token gets slot s: b_x[e_l, s] = x[t], slot[t,k] = s for each k      */
/* naming it; tokens_per_expert[e_l] is the number of such tokens.  Slots    */
/* of other experts are -1.  Padding rows are left as they are unless        */
/* zero_pad.  A token past max_num_tokens is dropped (error bit 8).          */
/* ------------------------------------------------------------------------ */
int orc_batched_prepare(const uint16_t *x, const int64_t *topk_idx, int64_t T, int K, int H,
                        int E, int E_local, int rank, int M, uint16_t *b_x,
                        int32_t *tokens_per_expert, int32_t *slot, int zero_pad)
{
    int err = 0;
    for (int64_t i = 0; i < T * K; ++i) {
        slot[i] = -1;
        int64_t id = topk_idx[i];
        if (id < -1 || id >= E)
            err |= ORC_ERR_INVALID_EXPERT;
    }
    for (int el = 0; el < E_local; ++el) {
        int64_t e = (int64_t)rank * E_local + el;
        int64_t s = 0;
        for (int64_t t = 0; t < T; ++t) {
            int hit = 0;
            for (int k = 0; k < K; ++k)
                if (topk_idx[t * K + k] == e)
                    hit = 1;
            if (!hit)
                continue;
            if (s < M) {
                memcpy(b_x + ((int64_t)el * M + s) * H, x + t * H, (size_t)H * sizeof(uint16_t));
                for (int k = 0; k < K; ++k)
                    if (topk_idx[t * K + k] == e)
                        slot[t * K + k] = (int32_t)s;
            } else {
                err |= ORC_ERR_CAPACITY;
            }
            ++s;
        }
        int32_t c = (int32_t)(s < M ? s : M);
        tokens_per_expert[el] = c;
        if (zero_pad)
            memset(b_x + ((int64_t)el * M + c) * H, 0, (size_t)(M - c) * H * sizeof(uint16_t));
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* [VB] finalize / [UB] Buffer.low_latency_combine (a weighted reduction):   */
/* out[t] = sum over k ascending with a local expert e_l = idx[t,k] -        */
/*          rank*E_local and slot[t,k] >= 0 of w[t,k] * Y[e_l, slot[t,k]],   */
/* accumulated with fp32 fused multiply-add from +0.0f, rounded once to      */
/* bf16.  This is this rank's partial output; tokens with no local expert    */
/* give +0.                                                                  */
/* ------------------------------------------------------------------------ */
void orc_batched_combine(const uint16_t *y, const int64_t *topk_idx, const float *topk_weights,
                         const int32_t *slot, int64_t T, int K, int H, int E_local, int rank,
                         int M, uint16_t *out)
{
    float *acc = (float *)malloc((size_t)H * sizeof(float));
    for (int64_t t = 0; t < T; ++t) {
        for (int h = 0; h < H; ++h)
            acc[h] = 0.0f;
        for (int k = 0; k < K; ++k) {
            int64_t el = topk_idx[t * K + k] - (int64_t)rank * E_local;
            int32_t s = slot[t * K + k];
            if (el < 0 || el >= E_local || s < 0)
                continue;
            float w = topk_weights[t * K + k];
            const uint16_t *row = y + (el * M + s) * (int64_t)H;
            for (int h = 0; h < H; ++h)
                acc[h] = fmaf(w, orc_bf16_to_f32(row[h]), acc[h]);
        }
        for (int h = 0; h < H; ++h)
            out[t * H + h] = orc_f32_to_bf16(acc[h]);
    }
    free(acc);
}

/* ------------------------------------------------------------------------ */
/* Power-of-two group scales ([UB] Buffer.low_latency_dispatch, round_scale:  */
/* the scales rounded to powers of two; use_ue8m0: the scale stored as an    */
/* UE8M0 code).  Per row and 128-element group g:                            */
/*   a      = max(max_i |x_i|, 1e-4f)                                        */
/*   s0     = a / 448.0f                    (fp32, nearest-even)             */
/*   scale  = the smallest power of two >= s0  (reading: rounding up keeps   */
/*            every |x_i| / scale <= 448, so nothing saturates)              */
/*   q_i    = e4m3_rn_satfinite(x_i * (1 / scale))   (1/scale is exact)      */
/*   code   = e + 127 where scale = 2^e (UE8M0: 8 exponent bits, bias 127,   */
/*            no sign, no mantissa)                                          */
/* A group holding +-inf: scale +inf, 1/scale = +0, code 255.                */
/* ------------------------------------------------------------------------ */
void orc_quantize_fp8_rows_pow2(const uint16_t *x, int64_t rows, int H, uint8_t *q, float *scale,
                                uint8_t *code)
{
    int G = H / 128;
    for (int64_t r = 0; r < rows; ++r) {
        for (int g = 0; g < G; ++g) {
            const uint16_t *xs = x + r * H + (int64_t)g * 128;
            float amax = 0.0f;
            for (int i = 0; i < 128; ++i) {
                float v = fabsf(orc_bf16_to_f32(xs[i]));
                if (v > amax)
                    amax = v;
            }
            float a = amax > 1e-4f ? amax : 1e-4f;
            float s0 = a / 448.0f;
            int e;
            float sc, inv;
            if (isinf(s0)) {                 /* a group holding +-inf: no power of two covers it; */
                e = 128;                     /* scale +inf, reciprocal +0 as 448/a gives the plain */
                sc = INFINITY;               /* form, code 255 (the exponent field of +inf)        */
                inv = 0.0f;
            } else {
                float m = frexpf(s0, &e);    /* s0 = m * 2^e, 0.5 <= m < 1 */
                if (m == 0.5f)
                    e -= 1;                  /* s0 is itself a power of two */
                sc = ldexpf(1.0f, e);
                inv = ldexpf(1.0f, -e);
            }
            for (int i = 0; i < 128; ++i)
                q[r * H + (int64_t)g * 128 + i] = orc_f32_to_e4m3(orc_bf16_to_f32(xs[i]) * inv);
            scale[r * G + g] = sc;
            code[r * G + g] = (uint8_t)(e + 127);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* [VB] BatchedPrepareAndFinalize.prepare, quantised branch, with the scale   */
/* layouts of [UB] Buffer.low_latency_dispatch.  Slots, tokens_per_expert,   */
/* capacity and error bits as orc_batched_prepare; each token is quantised   */
/* once (1x128 groups; plain or power-of-two scales) and every slot it takes */
/* carries the same codes.  With G = H/128 groups per row:                   */
/*   fmt 0: scales [E_local, M, G] fp32, row-major: (e,s,g) at (e*M+s)*G+g;  */
/*   fmt 1: scales [E_local, M, G] fp32, last two dims column-major:         */
/*          (e,s,g) at (e*G+g)*M+s;                                          */
/*   fmt 2: scales [E_local, M, G/4] int32, last two dims column-major:      */
/*          (e,s,j) at (e*(G/4)+j)*M+s; byte (g mod 4) of int (e,s,g/4),     */
/*          little-endian, is group g's UE8M0 code (needs round_scale).      */
/* zero_pad: codes and scale entries of slots >= tokens_per_expert are set   */
/* to zero (the page's zero-initialised outputs); otherwise left as given.   */
/* Returns error bits; 16 (unsupported) for fmt 2 without round_scale or     */
/* H % 512 != 0.                                                             */
/* ------------------------------------------------------------------------ */
int orc_batched_prepare_fp8(const uint16_t *x, const int64_t *topk_idx, int64_t T, int K, int H, int E,
                            int E_local, int rank, int M, uint8_t *b_q, void *b_scale, int fmt,
                            int round_scale, int32_t *tokens_per_expert, int32_t *slot, int zero_pad)
{
    int G = H / 128;
    if (fmt == 2 && (!round_scale || H % 512 != 0))
        return 16;
    uint8_t *q = (uint8_t *)malloc((size_t)(T > 0 ? T : 1) * H);
    float *sc = (float *)malloc((size_t)(T > 0 ? T : 1) * G * sizeof(float));
    uint8_t *code = (uint8_t *)malloc((size_t)(T > 0 ? T : 1) * G);
    if (round_scale)
        orc_quantize_fp8_rows_pow2(x, T, H, q, sc, code);
    else
        orc_quantize_fp8_rows(x, T, H, q, sc);
    float *sf = (float *)b_scale;
    uint8_t *sb = (uint8_t *)b_scale;
    int err = 0;
    for (int64_t i = 0; i < T * K; ++i) {
        slot[i] = -1;
        int64_t id = topk_idx[i];
        if (id < -1 || id >= E)
            err |= ORC_ERR_INVALID_EXPERT;
    }
    for (int el = 0; el < E_local; ++el) {
        int64_t e = (int64_t)rank * E_local + el;
        int64_t s = 0;
        for (int64_t t = 0; t < T; ++t) {
            int hit = 0;
            for (int k = 0; k < K; ++k)
                if (topk_idx[t * K + k] == e)
                    hit = 1;
            if (!hit)
                continue;
            if (s < M) {
                memcpy(b_q + ((int64_t)el * M + s) * H, q + t * H, (size_t)H);
                for (int g = 0; g < G; ++g) {
                    if (fmt == 0)
                        sf[((int64_t)el * M + s) * G + g] = sc[t * G + g];
                    else if (fmt == 1)
                        sf[((int64_t)el * G + g) * M + s] = sc[t * G + g];
                    else
                        sb[(((int64_t)el * (G / 4) + g / 4) * M + s) * 4 + g % 4] = code[t * G + g];
                }
                for (int k = 0; k < K; ++k)
                    if (topk_idx[t * K + k] == e)
                        slot[t * K + k] = (int32_t)s;
            } else {
                err |= ORC_ERR_CAPACITY;
            }
            ++s;
        }
        int32_t c = (int32_t)(s < M ? s : M);
        tokens_per_expert[el] = c;
        if (zero_pad) {
            memset(b_q + ((int64_t)el * M + c) * H, 0, (size_t)(M - c) * H);
            for (int64_t r = c; r < M; ++r)
                for (int g = 0; g < G; ++g) {
                    if (fmt == 0)
                        sf[((int64_t)el * M + r) * G + g] = 0.0f;
                    else if (fmt == 1)
                        sf[((int64_t)el * G + g) * M + r] = 0.0f;
                    else
                        sb[(((int64_t)el * (G / 4) + g / 4) * M + r) * 4 + g % 4] = 0;
                }
        }
    }
    free(q);
    free(sc);
    free(code);
    return err;
}

/* ------------------------------------------------------------------------ */
/* [VB] prepare (both branches) with a per-expert capacity and a receive      */
/* alignment ([ND] TokenDispatcherConfig moe_expert_capacity_factor: a        */
/* per-expert capacity factor, unset meaning that nothing is dropped;         */
/* [UB] Buffer.dispatch expert_alignment: the count each local expert         */
/* receives is made a multiple of it; [ND] moe_router_expert_pad_multiple).   */
/* Local expert e_l keeps the first `capacity` tokens naming it, in token     */
/* order (slots 0 .. capacity-1); later ones are dropped (slot -1, row not    */
/* written) and counted in dropped[e_l]; this is the capacity's purpose, so   */
/* no error bit.  The received count kept = min(hits, capacity) is rounded    */
/* up to a multiple of `alignment` (at most M) and returned as               */
/* tokens_per_expert; rows kept .. aligned-1 are zero rows (codes 0 and zero */
/* scale entries for fp8), rows past that are zeroed only with zero_pad.      */
/* fmt < 0: bf16 rows (b_rows is uint16 [E_local,M,H]); fmt 0..2: fp8 codes   */
/* (b_rows is uint8) with scales as orc_batched_prepare_fp8.                  */
/* Returns error bits (invalid ids 2; 16 for an unsupported fp8 format).     */
/* ------------------------------------------------------------------------ */
int64_t orc_expert_capacity(int64_t T, int K, int E, double factor)
{
    return (int64_t)ceil(factor * (double)T * (double)K / (double)E);
}

int orc_batched_prepare_ex(const uint16_t *x, const int64_t *topk_idx, int64_t T, int K, int H, int E,
                           int E_local, int rank, int M, int capacity, int alignment, void *b_rows,
                           void *b_scale, int fmt, int round_scale, int32_t *tokens_per_expert,
                           int32_t *slot, int32_t *dropped, int zero_pad)
{
    int G = H / 128;
    if (fmt >= 0 && (H % 128 != 0 || (fmt == 2 && (!round_scale || H % 512 != 0))))
        return 16;
    size_t rowb = fmt < 0 ? (size_t)H * 2 : (size_t)H;   /* bytes per row */
    uint8_t *rows = (uint8_t *)b_rows;
    uint8_t *q = NULL, *code = NULL;
    float *sc = NULL;
    if (fmt >= 0) {
        q = (uint8_t *)malloc((size_t)(T > 0 ? T : 1) * H);
        sc = (float *)malloc((size_t)(T > 0 ? T : 1) * G * sizeof(float));
        code = (uint8_t *)malloc((size_t)(T > 0 ? T : 1) * G);
        if (round_scale)
            orc_quantize_fp8_rows_pow2(x, T, H, q, sc, code);
        else
            orc_quantize_fp8_rows(x, T, H, q, sc);
    }
    float *sf = (float *)b_scale;
    uint8_t *sb = (uint8_t *)b_scale;
    int err = 0;
    for (int64_t i = 0; i < T * K; ++i) {
        slot[i] = -1;
        int64_t id = topk_idx[i];
        if (id < -1 || id >= E)
            err |= ORC_ERR_INVALID_EXPERT;
    }
    for (int el = 0; el < E_local; ++el) {
        int64_t e = (int64_t)rank * E_local + el;
        int64_t s = 0;
        for (int64_t t = 0; t < T; ++t) {
            int hit = 0;
            for (int k = 0; k < K; ++k)
                if (topk_idx[t * K + k] == e)
                    hit = 1;
            if (!hit)
                continue;
            if (s < capacity) {
                uint8_t *dst = rows + ((int64_t)el * M + s) * rowb;
                if (fmt < 0)
                    memcpy(dst, x + t * H, rowb);
                else {
                    memcpy(dst, q + t * H, rowb);
                    for (int g = 0; g < G; ++g) {
                        if (fmt == 0)
                            sf[((int64_t)el * M + s) * G + g] = sc[t * G + g];
                        else if (fmt == 1)
                            sf[((int64_t)el * G + g) * M + s] = sc[t * G + g];
                        else
                            sb[(((int64_t)el * (G / 4) + g / 4) * M + s) * 4 + g % 4] = code[t * G + g];
                    }
                }
                for (int k = 0; k < K; ++k)
                    if (topk_idx[t * K + k] == e)
                        slot[t * K + k] = (int32_t)s;
            }
            ++s;
        }
        int64_t kept = s < capacity ? s : capacity;
        int64_t aligned = (kept + alignment - 1) / alignment * alignment;
        if (aligned > M)
            aligned = M;
        tokens_per_expert[el] = (int32_t)aligned;
        if (dropped)
            dropped[el] = (int32_t)(s - kept);
        int64_t zero_end = zero_pad ? M : aligned;
        for (int64_t r = kept; r < zero_end; ++r) {
            memset(rows + ((int64_t)el * M + r) * rowb, 0, rowb);
            for (int g = 0; fmt >= 0 && g < G; ++g) {
                if (fmt == 0)
                    sf[((int64_t)el * M + r) * G + g] = 0.0f;
                else if (fmt == 1)
                    sf[((int64_t)el * G + g) * M + r] = 0.0f;
                else
                    sb[(((int64_t)el * (G / 4) + g / 4) * M + r) * 4 + g % 4] = 0;
            }
        }
    }
    free(q);
    free(sc);
    free(code);
    return err;
}

/* ------------------------------------------------------------------------ */
/* expert_alignment on the send layout ([UB] Buffer.dispatch): every rank's   */
/* segment of the rank-major send buffer starts at a multiple of A rows;     */
/* rank p's rows keep their order, followed by round_up(count_p, A) -        */
/* count_p pad rows that carry no token (send_token_idx -1, send_rank p,     */
/* send_idx -1, send_w +0).  token_pos points at the moved rows.  Input: the  */
/* unaligned layout of orc_build_send_layout and its send_counts.  Output    */
/* arrays hold round-up sizes; returns the aligned row count.                */
/* ------------------------------------------------------------------------ */
int64_t orc_align_send_layout(const int32_t *send_counts, int P, int A, int K, int64_t T,
                              const int32_t *send_token_idx, const int64_t *send_idx, const float *send_w,
                              const int32_t *token_pos, int32_t *rank_offsets, int32_t *a_token_idx,
                              int32_t *a_rank, int64_t *a_idx, float *a_w, int32_t *a_token_pos)
{
    int64_t src = 0, dst = 0;
    for (int p = 0; p < P; ++p) {
        rank_offsets[p] = (int32_t)dst;
        int64_t c = send_counts[p];
        int64_t padded = (c + A - 1) / A * A;
        for (int64_t i = 0; i < padded; ++i, ++dst) {
            if (i < c) {
                a_token_idx[dst] = send_token_idx[src + i];
                a_rank[dst] = p;
                for (int k = 0; k < K; ++k) {
                    a_idx[dst * K + k] = send_idx[(src + i) * K + k];
                    a_w[dst * K + k] = send_w[(src + i) * K + k];
                }
            } else {
                a_token_idx[dst] = -1;
                a_rank[dst] = p;
                for (int k = 0; k < K; ++k) {
                    a_idx[dst * K + k] = -1;
                    a_w[dst * K + k] = 0.0f;
                }
            }
        }
        src += c;
    }
    rank_offsets[P] = (int32_t)dst;
    for (int64_t t = 0; t < T; ++t)
        for (int p = 0; p < P; ++p) {
            int64_t n = token_pos[t * P + p];
            a_token_pos[t * P + p] = -1;
            if (n < 0)
                continue;
            /* row n of rank p moves by the padding of the ranks before p */
            int64_t pad = 0;
            for (int q2 = 0; q2 < p; ++q2)
                pad += (send_counts[q2] + A - 1) / A * A - send_counts[q2];
            a_token_pos[t * P + p] = (int32_t)(n + pad);
        }
    return dst;
}

/* ------------------------------------------------------------------------ */
/* [ND] _DeepepManager._indices_to_multihot / _HybridEPManager.               */
/* _indices_to_multihot: top-k indices [T,K] (-1 = masked) and their          */
/* probabilities [T,K] to a multihot routing map [T,E] and dense              */
/* probabilities [T,E]:                                                      */
/*   routing_map[t,e] = 1 iff some slot k of t names e, else 0;               */
/*   probs[t,e]       = the sum of probs[t,k] over the slots naming e, in     */
/*                      fp32 from +0.0f in ascending k (a single slot copies  */
/*                      its probability; reading for repeated ids: the mass   */
/*                      routed to e), +0.0f where routing_map is 0.           */
/* An id outside [-1, E) sets error bit 2 and its slot is ignored.            */
/* ------------------------------------------------------------------------ */
int orc_indices_to_multihot(const int64_t *topk_idx, const float *topk_probs, int64_t T, int K, int E,
                            uint8_t *routing_map, float *probs)
{
    int err = 0;
    for (int64_t i = 0; i < T * (int64_t)E; ++i) {
        routing_map[i] = 0;
        probs[i] = 0.0f;
    }
    for (int64_t t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            if (e == -1)
                continue;
            if (e < -1 || e >= E) {
                err |= ORC_ERR_INVALID_EXPERT;
                continue;
            }
            routing_map[t * E + e] = 1;
            probs[t * E + e] = probs[t * E + e] + topk_probs[t * K + k];
        }
    return err;
}
