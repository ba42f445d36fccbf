/*
 * Oracle for the W4A8 mixture-of-experts FFN and the block-FP8 dense projection.
 *
 * TEST INFRASTRUCTURE ONLY. This file is plain, slow, single-purpose C that
 * restates the definitions of the method so that the CUDA library can be
 * checked against it. Only tests/, __graft_entry__.smoke() and bench.py's CPU
 * baseline may load it. It shares no code, header or table with the CUDA path
 * in w4a8_moe_gb300/csrc, and the CUDA path never calls it.
 *
 * Sources (web pages the method is taken from):
 *   [P1] "ROCm: enable trillion-parameter MoE models with INT4-FP8 single node"
 *        (sglang PR #4152): Motivation; grok-1-W4A8KV8 config.json,
 *        quantization_config (activation_scheme "static", quant_method "fp8",
 *        int4_experts {bits 4, sym true, group "column"}, pack_method
 *        "reorder", ignored_layers = the MoE gate), Grok-1 shapes.
 *   [P2] "[AMD][Quantization] Add int4fp8_moe online quantization on ROCm"
 *        (sglang PR #7392): description (int4 MoE weights upcast to float8 so
 *        that fp8 math is used) and the review summary, "Core Quantization
 *        Utilities" (tensor-wise FP8, column-wise INT4, INT4 packed in INT32).
 *   [P3] "qwen4_exp: serve the block-FP8 dense projections natively (+25%
 *        decode)" (FreeToken PR #392): description and "What" (FP8_PB_WO
 *        weights kept with weight_scale_inv, one scale per 128-row x 128-col
 *        block; shapes [16384,2560] / [128,20] and [13312,2560] / [104,20]).
 *   OCP 8-bit Floating Point Specification (OFP8), format E4M3: the fp8
 *   format the pages' "fp8" denotes on hardware with /448 saturation.
 *
 * Readings taken where the pages are silent are stated
 * next to each function below.
 *
 * Precision: floating point that only feeds a sum is carried in double;
 * integer dot products are exact (int64). Where floating point decides an
 * integer code (the quantizers), the decision is taken in fp32, the precision
 * the method quantizes in, exactly as the CUDA kernels must.
 *
 * Parity pins: every exported function is pinned by tests/test_oracle_pins.py
 * against closed forms, a library routine (torch float8_e4m3fn, numpy, scipy)
 * or brute force; none is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* OCP E4M3 ("fn") decode: sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (2^-6 * m/8); S.1111.111 is NaN; there
 * is no infinity. Returns NAN for the two NaN codes. */
double orc_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* fp32 -> E4M3, round to nearest, ties to even, saturating to +-448
 * ("satfinite": every finite value and every infinity beyond the largest
 * finite code becomes that code with its sign); NaN -> 0x7F. The value is
 * placed on the grid of its binade: spacing 2^-9 below 2^-6 (subnormals),
 * 2^(E-3) in [2^E, 2^(E+1)). All scalings are exact in double and rint()
 * rounds half to even in the default rounding mode. */
uint8_t orc_e4m3_from_float(float vf)
{
    double v = (double)vf;
    uint8_t sign;
    double a;
    int code;
    if (isnan(vf))
        return 0x7F;
    sign = signbit(vf) ? 0x80 : 0x00;
    a = fabs(v);
    if (a > 448.0)
        return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal binade: value = m * 2^-9, m in 0..8 (8 is the first normal) */
        double q = rint(ldexp(a, 9));
        code = (int)q; /* 0..8; code 8 == 0x08 == 2^-6 */
    } else {
        int ex;
        double f = frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
        int E = ex - 1;           /* a in [2^E, 2^(E+1)) */
        double q = rint(ldexp(a, 3 - E)); /* in [8, 16] */
        (void)f;
        if (q >= 16.0) {
            E += 1;
            q = 8.0;
        }
        code = ((E + 7) << 3) | ((int)q - 8);
        if (code > 0x7E)
            code = 0x7E;
    }
    return (uint8_t)(sign | code);
}

void orc_e4m3_encode_array(const float* v, int64_t n, uint8_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_from_float(v[i]);
}

void orc_e4m3_decode_array(const uint8_t* c, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_to_double(c[i]);
}

/* bfloat16 is the upper half of an IEEE binary32. */
float orc_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* double -> bfloat16 with a single round-to-nearest-even (8 significant
 * bits, exponent range of binary32, subnormals down to 2^-133, overflow to
 * infinity). The model's output dtype is bfloat16 ([P1] config.json,
 * torch_dtype). */
uint16_t orc_double_to_bf16(double d)
{
    uint16_t sign;
    double a;
    int ex, E;
    double q;
    if (isnan(d))
        return 0x7FC0;
    sign = signbit(d) ? 0x8000 : 0x0000;
    a = fabs(d);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80);
    frexp(a, &ex);
    E = ex - 1; /* a in [2^E, 2^(E+1)) */
    if (E < -126) {
        /* subnormal: value = m * 2^-133, m in 0..128 */
        q = rint(ldexp(a, 133));
        return (uint16_t)(sign | (uint16_t)q); /* q == 128 is the first normal */
    }
    q = rint(ldexp(a, 7 - E)); /* in [128, 256] */
    if (q >= 256.0) {
        E += 1;
        q = 128.0;
    }
    if (E > 127)
        return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | (uint16_t)((E + 127) << 7) | (uint16_t)((int)q - 128));
}

void orc_bf16_array_from_double(const double* d, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_double_to_bf16(d[i]);
}

/* ------------------------------------------------------------------------ */
/* INT4 expert weights: column-wise symmetric quantization + int32 packing   */
/* ------------------------------------------------------------------------ */

/* [P1] int4_experts {bits 4, sym true, group "column"}; [P2] "column-wise
 * INT4 quantization" and "packing INT4 values into INT32".
 * Readings: "column" = one scale per output channel n of a weight stored as
 * [N, K] (K is the reduction axis); symmetric range divisor 7; scale 1 for an
 * all-zero channel; code = rint(w / s) (fp32 division, half to even), clamped
 * to [-8, 7]. Packing: 8 codes per int32 along K, code k = 8j + i in bits
 * 4i..4i+3 of word j as a two's-complement nibble.
 *   w    : bf16 bits [E, N, K]
 *   packed: int32 [E, N, K/8]
 *   scale : fp32 [E, N]                                                   */
void orc_quantize_experts(const uint16_t* w, int E, int N, int K, int32_t* packed, float* scale)
{
    for (int64_t row = 0; row < (int64_t)E * N; ++row) {
        const uint16_t* wr = w + row * K;
        float amax = 0.0f, s;
        for (int k = 0; k < K; ++k) {
            float a = fabsf(orc_bf16_to_float(wr[k]));
            if (a > amax)
                amax = a;
        }
        s = (amax == 0.0f) ? 1.0f : amax / 7.0f;
        scale[row] = s;
        for (int j = 0; j < K / 8; ++j) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i) {
                float r = rintf(orc_bf16_to_float(wr[8 * j + i]) / s);
                int q = (int)r;
                if (q < -8)
                    q = -8;
                if (q > 7)
                    q = 7;
                word |= ((uint32_t)q & 0xFu) << (4 * i);
            }
            packed[row * (K / 8) + j] = (int32_t)word;
        }
    }
}

/* Inverse of the packing: nibble -> signed code. */
void orc_unpack_int4(const int32_t* packed, int64_t nwords, int8_t* q)
{
    for (int64_t j = 0; j < nwords; ++j) {
        uint32_t word = (uint32_t)packed[j];
        for (int i = 0; i < 8; ++i) {
            int nib = (int)((word >> (4 * i)) & 0xFu);
            q[8 * j + i] = (int8_t)(nib >= 8 ? nib - 16 : nib);
        }
    }
}

static inline int orc_code_at(const int32_t* row_words, int k)
{
    uint32_t word = (uint32_t)row_words[k >> 3];
    int nib = (int)((word >> (4 * (k & 7))) & 0xFu);
    return nib >= 8 ? nib - 16 : nib;
}

/* ------------------------------------------------------------------------ */
/* FP8 activations, static per-tensor scale                                  */
/* ------------------------------------------------------------------------ */

/* [P1] activation_scheme "static", quant_method "fp8"; [P2] "tensor-wise FP8
 * quantization". Calibration reading: scale = max|x| / 448 over the tensor
 * (1 if the tensor is all zero). */
float orc_act_scale(const uint16_t* x, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(orc_bf16_to_float(x[i]));
        if (a > amax)
            amax = a;
    }
    return amax == 0.0f ? 1.0f : amax / 448.0f;
}

/* xq = E4M3(x / scale), fp32 division. */
void orc_quantize_act(const uint16_t* x, int64_t n, float scale, uint8_t* xq)
{
    for (int64_t i = 0; i < n; ++i)
        xq[i] = orc_e4m3_from_float(orc_bf16_to_float(x[i]) / scale);
}

/* ------------------------------------------------------------------------ */
/* Router: softmax top-k, renormalised; expert histogram; permutation        */
/* ------------------------------------------------------------------------ */

/* [P1] config.json ignored_layers: the MoE gate is not quantized, so its
 * logits are the plain product of the bf16 hidden states and the bf16 gate
 * weight. Computed in double (every bf16 product is exact in double):
 *   hidden bf16 [T, H], gate bf16 [E, H] -> logits double [T, E]          */
void orc_gate_logits(const uint16_t* hidden, const uint16_t* gate, int T, int H, int E, double* logits)
{
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += (double)orc_bf16_to_float(hidden[(int64_t)t * H + h]) *
                       (double)orc_bf16_to_float(gate[(int64_t)e * H + h]);
            logits[(int64_t)t * E + e] = acc;
        }
}

/* [P1] num_local_experts / num_experts_per_tok and the unquantized MoE gate.
 * Readings: experts are ranked on the fp32 logits (softmax is monotone),
 * descending, equal logits ranked by lower expert index; probabilities are
 * the softmax over all E experts (double); with renorm the k selected
 * probabilities are divided by their sum.
 *   logits fp32 [T, E] -> ids int32 [T, k], w double [T, k]              */
void orc_route(const float* logits, int T, int E, int k, int renorm, int32_t* ids, double* w)
{
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (int64_t)t * E;
        double mx = -INFINITY, denom = 0.0, sel = 0.0;
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || l[e] > l[best])
                    best = e; /* strict: the lower index wins ties */
            }
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
        }
        for (int e = 0; e < E; ++e)
            if ((double)l[e] > mx)
                mx = (double)l[e];
        for (int e = 0; e < E; ++e)
            denom += exp((double)l[e] - mx);
        for (int j = 0; j < k; ++j) {
            double p = exp((double)l[ids[(int64_t)t * k + j]] - mx) / denom;
            w[(int64_t)t * k + j] = p;
            sel += p;
        }
        if (renorm)
            for (int j = 0; j < k; ++j)
                w[(int64_t)t * k + j] /= sel;
    }
    free(taken);
}

/* Stable counting sort of the T*k assignments a = t*k + j by expert:
 * counts[e]; offsets = exclusive prefix sum with offsets[E] = T*k;
 * sorted[offsets[e] + (rank of a among earlier assignments of e)] = a;
 * inv[sorted[p]] = p. */
void orc_permute(const int32_t* ids, int T, int k, int E, int32_t* counts, int32_t* offsets,
                 int32_t* sorted, int32_t* inv)
{
    int64_t A = (int64_t)T * k;
    int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t a = 0; a < A; ++a)
        counts[ids[a]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    for (int64_t a = 0; a < A; ++a) {
        int e = ids[a];
        int32_t p = offsets[e] + seen[e]++;
        sorted[p] = (int32_t)a;
        inv[a] = p;
    }
    free(seen);
}

/* ------------------------------------------------------------------------ */
/* W4A8 MoE forward                                                          */
/* ------------------------------------------------------------------------ */

/* Gated activations. Readings: SiLU for Mixtral-shaped layers, the tanh
 * approximation of GELU for Grok-1-shaped layers; no bias. */
static double orc_act(double g, int act)
{
    if (act == 0)
        return g / (1.0 + exp(-g));
    return 0.5 * g * (1.0 + tanh(sqrt(2.0 / acos(-1.0)) * (g + 0.044715 * g * g * g)));
}

/* 512 * E4M3 value as an exact integer: every E4M3 value is a multiple of
 * 2^-9 and |value| <= 448, so 512*v is an integer of magnitude <= 229376. */
static int64_t orc_e4m3_times512(uint8_t c)
{
    double v = orc_e4m3_to_double(c) * 512.0;
    return (int64_t)v;
}

typedef struct {
    const uint8_t* xq;
    float s1;
    int T, H, I, E, k;
    const int32_t* w_gu;
    const float* s_gu;
    const int32_t* w_d;
    const float* s_d;
    float s2;
    int act;
    const int32_t* ids;
    const double* topk_w;
    const int32_t* tokens;
    int ntok;
    double* out;        /* [ntok, H] or NULL */
    uint8_t* hq_out;    /* [ntok, k, I] E4M3 codes of h / s2, or NULL */
    double* h_absmax;   /* per-thread slot or NULL */
    int tid, nthreads;
} orc_moe_job;

/* The definition, token by token (no permutation):
 *   G_i = sum_h dec(xq[t,h]) q_gu[e,i,h],  U_i = sum_h dec(xq[t,h]) q_gu[e,I+i,h]
 *   g = s1 S_gu[e,i] G_i,  u = s1 S_gu[e,I+i] U_i,  h_i = act(g) u
 *   hq_i = E4M3(fp32(h_i / s2))                         (static scale s2)
 *   D_n = sum_i dec(hq_i) q_d[e,n,i],  y_n = s2 S_d[e,n] D_n
 *   out[t,n] = sum_j w[t,j] y_n(e = ids[t,j])
 * Integer sums are exact int64 on 512*dec values. Reading: rows [0, I) of
 * gate_up are the gate, rows [I, 2I) the up projection. */
static void* orc_moe_worker(void* arg)
{
    orc_moe_job* J = (orc_moe_job*)arg;
    const int H = J->H, I = J->I, k = J->k;
    int64_t* x512 = (int64_t*)malloc(sizeof(int64_t) * (size_t)H);
    int64_t* h512 = (int64_t*)malloc(sizeof(int64_t) * (size_t)I);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    double local_max = 0.0;
    for (int it = J->tid; it < J->ntok; it += J->nthreads) {
        int t = J->tokens[it];
        if (J->out)
            for (int n = 0; n < H; ++n)
                J->out[(int64_t)it * H + n] = 0.0;
        for (int h = 0; h < H; ++h)
            x512[h] = orc_e4m3_times512(J->xq[(int64_t)t * H + h]);
        for (int j = 0; j < k; ++j) {
            int e = J->ids[(int64_t)t * k + j];
            double wt = J->out ? J->topk_w[(int64_t)t * k + j] : 0.0;
            const int32_t* Wgu = J->w_gu + (int64_t)e * 2 * I * (H / 8);
            const int32_t* Wd = J->w_d ? J->w_d + (int64_t)e * H * (I / 8) : NULL;
            for (int i = 0; i < I; ++i) {
                const int32_t* rg = Wgu + (int64_t)i * (H / 8);
                const int32_t* ru = Wgu + (int64_t)(I + i) * (H / 8);
                int64_t G = 0, U = 0;
                double g, u, hv;
                for (int h = 0; h < H; ++h) {
                    G += x512[h] * orc_code_at(rg, h);
                    U += x512[h] * orc_code_at(ru, h);
                }
                g = (double)J->s1 * (double)J->s_gu[(int64_t)e * 2 * I + i] * ((double)G / 512.0);
                u = (double)J->s1 * (double)J->s_gu[(int64_t)e * 2 * I + I + i] * ((double)U / 512.0);
                hv = orc_act(g, J->act) * u;
                if (fabs(hv) > local_max)
                    local_max = fabs(hv);
                if (J->out || J->hq_out) {
                    uint8_t code = orc_e4m3_from_float((float)(hv / (double)J->s2));
                    h512[i] = orc_e4m3_times512(code);
                    if (J->hq_out)
                        J->hq_out[((int64_t)it * k + j) * I + i] = code;
                }
            }
            if (!J->out)
                continue;
            for (int n = 0; n < H; ++n) {
                const int32_t* rd = Wd + (int64_t)n * (I / 8);
                int64_t D = 0;
                for (int i = 0; i < I; ++i)
                    D += h512[i] * orc_code_at(rd, i);
                y[n] = (double)J->s2 * (double)J->s_d[(int64_t)e * H + n] * ((double)D / 512.0);
                J->out[(int64_t)it * H + n] += wt * y[n];
            }
        }
    }
    if (J->h_absmax)
        *J->h_absmax = local_max;
    free(x512);
    free(h512);
    free(y);
    return NULL;
}

static void orc_moe_run(orc_moe_job* proto, int nthreads)
{
    pthread_t* th;
    orc_moe_job* jobs;
    if (nthreads < 1)
        nthreads = 1;
    th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    jobs = (orc_moe_job*)malloc(sizeof(orc_moe_job) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].tid = i;
        jobs[i].nthreads = nthreads;
        if (proto->h_absmax)
            jobs[i].h_absmax = proto->h_absmax + i;
        if (nthreads == 1)
            orc_moe_worker(&jobs[i]);
        else
            pthread_create(&th[i], NULL, orc_moe_worker, &jobs[i]);
    }
    if (nthreads > 1)
        for (int i = 0; i < nthreads; ++i)
            pthread_join(th[i], NULL);
    free(th);
    free(jobs);
}

/* out[ti, :] (double) for each token tokens[ti]; threads partition tokens,
 * which leaves every token's arithmetic unchanged. */
void orc_moe_forward(const uint8_t* xq, float s1, int T, int H, int I, int E, int k,
                     const int32_t* w_gu, const float* s_gu, const int32_t* w_d, const float* s_d,
                     float s2, int act, const int32_t* ids, const double* topk_w,
                     const int32_t* tokens, int ntok, double* out, int nthreads)
{
    orc_moe_job J;
    memset(&J, 0, sizeof(J));
    J.xq = xq; J.s1 = s1; J.T = T; J.H = H; J.I = I; J.E = E; J.k = k;
    J.w_gu = w_gu; J.s_gu = s_gu; J.w_d = w_d; J.s_d = s_d; J.s2 = s2; J.act = act;
    J.ids = ids; J.topk_w = topk_w; J.tokens = tokens; J.ntok = ntok; J.out = out;
    orc_moe_run(&J, nthreads);
}

/* The E4M3 codes of the intermediate activation, hq[ti, j, i] =
 * E4M3(fp32(h_i / s2)) for assignment (tokens[ti], j), i in natural order:
 * the quantity the down projection consumes ([P1] quantization_config,
 * static per-tensor FP8 activations), computed exactly as in
 * orc_moe_forward. */
void orc_moe_hidden_codes(const uint8_t* xq, float s1, int T, int H, int I, int E, int k,
                          const int32_t* w_gu, const float* s_gu, float s2, int act, const int32_t* ids,
                          const int32_t* tokens, int ntok, uint8_t* hq, int nthreads)
{
    orc_moe_job J;
    memset(&J, 0, sizeof(J));
    J.xq = xq; J.s1 = s1; J.T = T; J.H = H; J.I = I; J.E = E; J.k = k;
    J.w_gu = w_gu; J.s_gu = s_gu; J.s2 = s2; J.act = act;
    J.ids = ids; J.tokens = tokens; J.ntok = ntok; J.out = NULL; J.hq_out = hq;
    orc_moe_run(&J, nthreads);
}

/* Static-scale calibration for the intermediate activation (reading: the
 * scale is max|h| / 448 over the assignments of the given calibration tokens,
 * 1 if that is zero). Returns max|h|. */
double orc_moe_hidden_absmax(const uint8_t* xq, float s1, int T, int H, int I, int E, int k,
                             const int32_t* w_gu, const float* s_gu, int act, const int32_t* ids,
                             const int32_t* tokens, int ntok, int nthreads)
{
    orc_moe_job J;
    double* slots;
    double m = 0.0;
    if (nthreads < 1)
        nthreads = 1;
    slots = (double*)calloc((size_t)nthreads, sizeof(double));
    memset(&J, 0, sizeof(J));
    J.xq = xq; J.s1 = s1; J.T = T; J.H = H; J.I = I; J.E = E; J.k = k;
    J.w_gu = w_gu; J.s_gu = s_gu; J.s2 = 1.0f; J.act = act;
    J.ids = ids; J.tokens = tokens; J.ntok = ntok; J.out = NULL; J.h_absmax = slots;
    J.topk_w = NULL; /* routing weights are not read when out == NULL */
    orc_moe_run(&J, nthreads);
    for (int i = 0; i < nthreads; ++i)
        if (slots[i] > m)
            m = slots[i];
    free(slots);
    return m;
}

/* ------------------------------------------------------------------------ */
/* Block-FP8 dense projection                                                */
/* ------------------------------------------------------------------------ */

/* [P3] FP8_PB_WO weights: e4m3 [N, K] with weight_scale_inv [N/128, K/128],
 * one scale per 128-row x 128-col block; the per-block scales concatenate
 * along whole 128-row blocks. Reading: weight_scale_inv is the multiplier
 * that dequantizes (w ~ dec(wq) * Wsi). Input preparation (the checkpoint's
 * own quantizer): Wsi = amax/448 over the block (1 if zero), wq = E4M3(w/Wsi). */
void orc_block_quantize_weight(const uint16_t* w, int N, int K, uint8_t* wq, float* wsi)
{
    int NB = N / 128, KB = K / 128;
    for (int nb = 0; nb < NB; ++nb)
        for (int kb = 0; kb < KB; ++kb) {
            float amax = 0.0f, s;
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c) {
                    float a = fabsf(orc_bf16_to_float(w[(int64_t)(nb * 128 + r) * K + kb * 128 + c]));
                    if (a > amax)
                        amax = a;
                }
            s = amax == 0.0f ? 1.0f : amax / 448.0f;
            wsi[nb * KB + kb] = s;
            for (int r = 0; r < 128; ++r)
                for (int c = 0; c < 128; ++c) {
                    int64_t idx = (int64_t)(nb * 128 + r) * K + kb * 128 + c;
                    wq[idx] = orc_e4m3_from_float(orc_bf16_to_float(w[idx]) / s);
                }
        }
}

/* Activation side of the block-FP8 projection. Reading: one scale per token
 * and 128-column group, s = amax/448 (1 if zero), xq = E4M3(x / s).
 *   x bf16 [M, K] -> xq [M, K], xs fp32 [M, K/128] */
void orc_block_quantize_act(const uint16_t* x, int M, int K, uint8_t* xq, float* xs)
{
    int G = K / 128;
    for (int m = 0; m < M; ++m)
        for (int g = 0; g < G; ++g) {
            const uint16_t* xr = x + (int64_t)m * K + g * 128;
            float amax = 0.0f, s;
            for (int c = 0; c < 128; ++c) {
                float a = fabsf(orc_bf16_to_float(xr[c]));
                if (a > amax)
                    amax = a;
            }
            s = amax == 0.0f ? 1.0f : amax / 448.0f;
            xs[(int64_t)m * G + g] = s;
            for (int c = 0; c < 128; ++c)
                xq[(int64_t)m * K + g * 128 + c] = orc_e4m3_from_float(orc_bf16_to_float(xr[c]) / s);
        }
}

typedef struct {
    const uint8_t* xq;
    const float* xs;
    int M, N, K;
    const uint8_t* wq;
    const float* wsi;
    const int32_t* rows;
    int nrows;
    double* y;
    int tid, nthreads;
} orc_blk_job;

/* y[m, n] = sum_g xs[m,g] Wsi[n/128,g] sum_{k in g} dec(xq[m,k]) dec(wq[n,k]).
 * The inner sum is exact: products of E4M3 values are multiples of 2^-18,
 * accumulated as int64 of (512 dec)(512 dec). */
static void* orc_blk_worker(void* arg)
{
    orc_blk_job* J = (orc_blk_job*)arg;
    int G = J->K / 128;
    int64_t* xi = (int64_t*)malloc(sizeof(int64_t) * (size_t)J->K);
    int64_t lut[256];
    for (int c = 0; c < 256; ++c)
        lut[c] = ((c & 0x7F) == 0x7F) ? 0 : orc_e4m3_times512((uint8_t)c);
    for (int r = J->tid; r < J->nrows; r += J->nthreads) {
        int m = J->rows[r];
        for (int kk = 0; kk < J->K; ++kk)
            xi[kk] = lut[J->xq[(int64_t)m * J->K + kk]];
        for (int n = 0; n < J->N; ++n) {
            const uint8_t* wr = J->wq + (int64_t)n * J->K;
            double acc = 0.0;
            for (int g = 0; g < G; ++g) {
                int64_t S = 0;
                for (int c = 0; c < 128; ++c)
                    S += xi[g * 128 + c] * lut[wr[g * 128 + c]];
                acc += (double)J->xs[(int64_t)m * G + g] * (double)J->wsi[(int64_t)(n / 128) * G + g] *
                       ((double)S / 262144.0);
            }
            J->y[(int64_t)r * J->N + n] = acc;
        }
    }
    free(xi);
    return NULL;
}

void orc_block_linear(const uint8_t* xq, const float* xs, int M, int N, int K, const uint8_t* wq,
                      const float* wsi, const int32_t* rows, int nrows, double* y, int nthreads)
{
    orc_blk_job proto;
    pthread_t* th;
    orc_blk_job* jobs;
    if (nthreads < 1)
        nthreads = 1;
    proto.xq = xq; proto.xs = xs; proto.M = M; proto.N = N; proto.K = K;
    proto.wq = wq; proto.wsi = wsi; proto.rows = rows; proto.nrows = nrows; proto.y = y;
    th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    jobs = (orc_blk_job*)malloc(sizeof(orc_blk_job) * (size_t)nthreads);
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = proto;
        jobs[i].tid = i;
        jobs[i].nthreads = nthreads;
        if (nthreads == 1)
            orc_blk_worker(&jobs[i]);
        else
            pthread_create(&th[i], NULL, orc_blk_worker, &jobs[i]);
    }
    if (nthreads > 1)
        for (int i = 0; i < nthreads; ++i)
            pthread_join(th[i], NULL);
    free(th);
    free(jobs);
}

/* ------------------------------------------------------------------------ */
/* Per-tensor FP8 dense linear                                               */
/* ------------------------------------------------------------------------ */

/* [P2] description: the attention projections are quantized online to float8;
 * review summary: QuarkInt4Fp8LinearMethod for linear layers and tensor-wise
 * FP8 quantization. Reading: one scale for the whole weight (sw) and one for
 * the activations (sx), both from the tensor-wise quantizer, so
 *   y[m, n] = sx * sw * sum_k dec(xq[m, k]) * dec(wq[n, k])
 * with the inner sum exact (int64 on 512*dec values; products are multiples
 * of 2^-18).   xq u8 [M, K], wq u8 [N, K] -> y double [rows, N]           */
void orc_fp8_linear(const uint8_t* xq, float sx, int M, int N, int K, const uint8_t* wq, float sw,
                    const int32_t* rows, int nrows, double* y)
{
    int64_t* w512 = (int64_t*)malloc(sizeof(int64_t) * (size_t)K);
    int64_t* x512 = (int64_t*)malloc(sizeof(int64_t) * (size_t)K);
    (void)M;
    for (int ri = 0; ri < nrows; ++ri) {
        int m = rows[ri];
        for (int k = 0; k < K; ++k)
            x512[k] = orc_e4m3_times512(xq[(int64_t)m * K + k]);
        for (int n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int k = 0; k < K; ++k)
                w512[k] = orc_e4m3_times512(wq[(int64_t)n * K + k]);
            for (int k = 0; k < K; ++k)
                acc += x512[k] * w512[k];
            y[(int64_t)ri * N + n] = (double)sx * (double)sw * ((double)acc / 262144.0);
        }
    }
    free(w512);
    free(x512);
}
