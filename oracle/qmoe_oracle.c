/*
 * qmoe_oracle.c -- plain CPU oracle of the qwen3moe MoE FFN over GGUF k-quant
 * expert weights, and of one qwen3moe decoder layer at decode time.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code with the CUDA path.
 *
 * Every quantity is computed in double from the exact stored fields, with no
 * blocking, fusion or reordering beyond the definitions cited next to each
 * function.  Threads (OpenMP) only split independent outer loops (experts,
 * heads); every reduction is a plain serial sum in index order.
 *
 * Sources (web pages, cited by title and section):
 *  [P2] aprender issue "qwen3moe (Qwen3-30B-A3B, Qwen3-Coder-30B-A3B, Q4_K_M)
 *       has NO working CUDA path", sections "File facts" (geometry, 144 B Q4_K /
 *       210 B Q6_K superblocks, 884,736 / 1,290,240 B per expert, base + e*stride
 *       addressing), "Gaps ... G3" (router GEMV, per-qtype expert GEMVs, fused
 *       SwiGLU, weighted sum, residual add, softmax/top-8/renorm).
 *  [P1] aprender issue "Qwen3 GPU inference produces garbage output", section
 *       "Fix Applied" (head_dim 128 independent of hidden/heads, GQA uses head_dim,
 *       per-head Q/K RMSNorm).
 *  [P4] aprender PR "apply per-head Q/K RMSNorm in forward_qwen3_moe", section
 *       "The fix" (Q/K norm after bias, before RoPE).
 *  [P5] SharpInference issue "Forward-pass divergence on Qwen3-Coder 30B-A3B",
 *       closing comment (NEOX RoPE: rotated pairs offset by head_dim/2).
 *  [P3] atlasinference source page "spark_model/weight_loader/qwen3.rs",
 *       function load_layers, branches "Native FP8 MoE" and "Native FP8
 *       Attention" (FP8 block-scaled weights with block size 128, loaded for
 *       FP8-weight / 16-bit-activation GEMMs, the "w8a16" remark) and the
 *       router-precision option (router kept in full precision while the
 *       experts stay FP8).
 *  The bit layout inside a Q4_K / Q6_K superblock is the public GGUF k-quant
 *  format; the pages fix only the superblock sizes and field order.  The FP8
 *  code is the OCP E4M3 ("e4m3fn") format; the pages fix only the block size.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QO_QK 256
#define QO_Q4_K 1
#define QO_Q6_K 2

/* ------------------------------------------------------------------ fp16 */

/* IEEE 754 binary16 -> double, exact for every finite pattern incl. subnormals. */
double qo_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 31;
    int man = h & 1023;
    double v;
    if (ex == 0)
        v = ldexp((double)man, -24);             /* man * 2^-24 */
    else if (ex == 31)
        v = man ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + man), ex - 25); /* (1 + man/1024) * 2^(ex-15) */
    return sign ? -v : v;
}

/* double -> binary16 with round-to-nearest-even (used for the KV-cache write). */
uint16_t qo_double_to_half(double v) {
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (isnan(v)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00;      /* rounds past the largest finite half */
    if (a < ldexp(1.0, -14)) {                    /* subnormal range: multiples of 2^-24 */
        double r = nearbyint(ldexp(a, 24));
        return sign | (uint16_t)r;                /* r == 1024 is the smallest normal */
    }
    int e;
    double f = frexp(a, &e);                      /* a = f * 2^e, f in [0.5, 1) */
    double r = nearbyint(ldexp(f, 11));           /* 11 significant bits, in [1024, 2048] */
    int E = e - 1 + 15;
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(E << 10) | (uint16_t)((int)r - 1024);
}

static double half_at(const uint8_t* p) {
    return qo_half_to_double((uint16_t)(p[0] | (p[1] << 8)));
}

/* ------------------------------------------------------------------ k-quant blocks */

int qo_block_bytes(int qtype) {
    return qtype == QO_Q4_K ? 144 : qtype == QO_Q6_K ? 210 : -1;
}

/* Q4_K sub-block j (0..7) scale s_j and min m_j, both 6-bit, packed in 12 bytes:
 * j < 4 : low 6 bits of byte j (scale) and of byte j+4 (min);
 * j >= 4: low nibble / high nibble of byte j+4 give the 4 low bits of scale /
 *         min, the top 2 bits of byte j-4 / byte j give their 2 high bits. */
static void q4k_scale_min(const uint8_t* sc, int j, int* s, int* m) {
    if (j < 4) {
        *s = sc[j] & 63;
        *m = sc[j + 4] & 63;
    } else {
        *s = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
        *m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
}

/* Element i (0..255) of a 144-byte Q4_K superblock:
 * bytes 0-1 d (fp16), 2-3 dmin (fp16), 4-15 packed scales/mins, 16-143 nibbles.
 * Element i lies in sub-block j = i/32 at position l = i%32; the nibbles form
 * four 32-byte chunks, chunk c holding sub-block 2c in its low nibbles and
 * sub-block 2c+1 in its high nibbles (byte l of the chunk -> position l).
 * value = d * s_j * q - dmin * m_j. */
double qo_q4k_element(const uint8_t* blk, int i) {
    double d = half_at(blk), dmin = half_at(blk + 2);
    const uint8_t* sc = blk + 4;
    const uint8_t* qs = blk + 16;
    int j = i / 32, l = i % 32;
    int q = (qs[32 * (j / 2) + l] >> (4 * (j % 2))) & 15;
    int s, m;
    q4k_scale_min(sc, j, &s, &m);
    return d * s * q - dmin * m;
}

/* Element i (0..255) of a 210-byte Q6_K superblock:
 * bytes 0-127 ql (low 4 bits), 128-191 qh (high 2 bits), 192-207 int8 scales,
 * 208-209 d (fp16).  i = 128n + 32g + l (half n, group g, position l):
 * low 4 bits from ql[64n + l + 32*(g%2)] (low nibble for g<2, high for g>=2),
 * high 2 bits = bits 2g..2g+1 of qh[32n + l], scale sc[8n + l/16 + 2g],
 * value = d * sc * (q6 - 32). */
double qo_q6k_element(const uint8_t* blk, int i) {
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    const int8_t* sc = (const int8_t*)(blk + 192);
    double d = half_at(blk + 208);
    int n = i / 128, g = (i % 128) / 32, l = i % 32;
    int lo = (ql[64 * n + l + 32 * (g % 2)] >> (4 * (g / 2))) & 15;
    int hi = (qh[32 * n + l] >> (2 * g)) & 3;
    int q = (lo | (hi << 4)) - 32;
    return d * (double)sc[8 * n + l / 16 + 2 * g] * (double)q;
}

int qo_dequant_block(int qtype, const uint8_t* blk, double* out) {
    for (int i = 0; i < QO_QK; ++i) {
        if (qtype == QO_Q4_K) out[i] = qo_q4k_element(blk, i);
        else if (qtype == QO_Q6_K) out[i] = qo_q6k_element(blk, i);
        else return -1;
    }
    return 0;
}

/* A matrix with `rows` outputs and `cols` inputs is stored row after row; a row
 * is cols/256 consecutive superblocks ([P2] "File facts"). */
int qo_dequant_matrix(int qtype, const uint8_t* data, long rows, long cols, double* out) {
    int bb = qo_block_bytes(qtype);
    if (bb < 0 || cols % QO_QK) return -1;
    long nb = cols / QO_QK;
    for (long r = 0; r < rows; ++r)
        for (long b = 0; b < nb; ++b)
            if (qo_dequant_block(qtype, data + (r * nb + b) * bb, out + r * cols + b * QO_QK)) return -1;
    return 0;
}

/* Byte stride between experts of a 3-D expert tensor: expert e starts at
 * base + e * rows * (cols/256) * block_bytes ([P2] "File facts"). */
long qo_expert_stride(int qtype, long rows, long cols) {
    int bb = qo_block_bytes(qtype);
    if (bb < 0 || cols % QO_QK) return -1;
    return rows * (cols / QO_QK) * bb;
}

/* ------------------------------------------------------------------ router */

/* Router for one token ([P2] "Gaps ... G3": router GEMV, softmax, top-k, renorm):
 * logit_e = sum_h Wr[e][h] x[h] (+ bias_e), accumulated in double and delivered
 * as an F32 vector (the router output the pages move is 128 x f32);
 * S = the k largest F32 logits, ties to the lower expert index, ordered by
 * descending logit then ascending index;
 * p = softmax(logits) in double; w_j = p_{S_j} / sum_{i in S} p_i (norm_topk)
 * or p_{S_j}.  If `force` is given, S = force (weights still from p). */
static void route_one(int H, int E, int K, int norm_topk, const double* x, const float* wr,
                      const float* bias, const int32_t* force, float* logits, int32_t* ids,
                      double* w, double* probs) {
    for (int e = 0; e < E; ++e) {
        double acc = 0.0;
        for (int h = 0; h < H; ++h) acc += (double)wr[(long)e * H + h] * x[h];
        if (bias) acc += (double)bias[e];
        logits[e] = (float)acc;
    }
    if (force) {
        for (int j = 0; j < K; ++j) ids[j] = force[j];
    } else {
        char* taken = (char*)calloc((size_t)E, 1);
        for (int j = 0; j < K; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || logits[e] > logits[best])) best = e;
            taken[best] = 1;
            ids[j] = best;
        }
        free(taken);
    }
    double mx = logits[0];
    for (int e = 1; e < E; ++e) if (logits[e] > mx) mx = logits[e];
    double z = 0.0;
    for (int e = 0; e < E; ++e) z += exp((double)logits[e] - mx);
    double ps = 0.0;
    for (int j = 0; j < K; ++j) ps += exp((double)logits[ids[j]] - mx) / z;
    for (int j = 0; j < K; ++j) {
        double p = exp((double)logits[ids[j]] - mx) / z;
        w[j] = norm_topk ? p / ps : p;
    }
    if (probs)
        for (int e = 0; e < E; ++e) probs[e] = exp((double)logits[e] - mx) / z;
}

int qo_router(int T, int H, int E, int K, int norm_topk, const double* x, const float* wr,
              const float* bias, const int32_t* force, float* logits, int32_t* ids, double* w,
              double* probs) {
    if (K < 1 || K > E) return -1;
    for (int t = 0; t < T; ++t)
        route_one(H, E, K, norm_topk, x + (long)t * H, wr, bias, force ? force + (long)t * K : NULL,
                  logits + (long)t * E, ids + (long)t * K, w + (long)t * K,
                  probs ? probs + (long)t * E : NULL);
    return 0;
}

/* ------------------------------------------------------------------ MoE FFN */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* y = W x for a dense double matrix [rows][cols]. */
static void matvec(const double* W, long rows, long cols, const double* x, double* y) {
    for (long r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (long c = 0; c < cols; ++c) acc += W[r * cols + c] * x[c];
        y[r] = acc;
    }
}

/* Loader of one used expert's three matrices as dense doubles: Wg, Wu [F][H]
 * and Wd [H][F]. */
typedef void (*qo_expert_loader)(const void* ctx, int e, long H, long F, double* Wg, double* Wu,
                                 double* Wd);

/* The MoE FFN of T tokens ([P2] "Gaps ... G3") once the experts are dense:
 * for each token t and slot j with expert e = ids[t][j]:
 *   g = Wg_e x_t, u = Wu_e x_t           (gate/up, [F][H])
 *   a = silu(g) * u                      (fused SwiGLU)
 *   y_tj = Wd_e a                        (down, [H][F])
 *   out_t = res_t + sum_j w[t][j] y_tj   (weighted sum into the residual,
 *                                         summed in slot order j = 0..K-1)
 * act (nullable) receives a [T][K][F]; ys (nullable) receives y [T][K][H]. */
static int moe_ffn_dense(int T, int H, int F, int E, int K, const double* x, const double* res,
                         const int32_t* ids, const double* w, qo_expert_loader load,
                         const void* ctx, double* out, double* act, double* ys) {
    for (long p = 0; p < (long)T * K; ++p)
        if (ids[p] < 0 || ids[p] >= E) return -2;
    double* Y = (double*)malloc(sizeof(double) * (size_t)T * K * H);
    if (!Y) return -3;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int e = 0; e < E; ++e) {
        int used = 0;
        for (long p = 0; p < (long)T * K; ++p) used |= (ids[p] == e);
        if (!used) continue;
        double* Wg = (double*)malloc(sizeof(double) * (size_t)F * H);
        double* Wu = (double*)malloc(sizeof(double) * (size_t)F * H);
        double* Wd = (double*)malloc(sizeof(double) * (size_t)H * F);
        double* g = (double*)malloc(sizeof(double) * (size_t)F);
        double* u = (double*)malloc(sizeof(double) * (size_t)F);
        double* a = (double*)malloc(sizeof(double) * (size_t)F);
        if (!Wg || !Wu || !Wd || !g || !u || !a) {
#pragma omp atomic write
            err = 1;
        } else {
            load(ctx, e, H, F, Wg, Wu, Wd);
            for (long p = 0; p < (long)T * K; ++p) {
                if (ids[p] != e) continue;
                long t = p / K;
                matvec(Wg, F, H, x + t * H, g);
                matvec(Wu, F, H, x + t * H, u);
                for (long f = 0; f < F; ++f) a[f] = silu(g[f]) * u[f];
                if (act) memcpy(act + p * F, a, sizeof(double) * (size_t)F);
                matvec(Wd, H, F, a, Y + p * H);
            }
        }
        free(Wg); free(Wu); free(Wd); free(g); free(u); free(a);
    }
    if (err) { free(Y); return -3; }
    for (long t = 0; t < T; ++t)
        for (long h = 0; h < H; ++h) {
            double acc = res ? res[t * H + h] : x[t * H + h];
            for (long j = 0; j < K; ++j) acc += w[t * K + j] * Y[(t * K + j) * H + h];
            out[t * H + h] = acc;
        }
    if (ys) memcpy(ys, Y, sizeof(double) * (size_t)T * K * H);
    free(Y);
    return 0;
}

typedef struct {
    const uint8_t *gate, *up, *down;
    int gate_t, up_t, down_t;
    long sg, su, sd;
} kquant_experts;

/* Expert e of each 3-D k-quant tensor is read in place at base + e*stride
 * ([P2] "File facts"). */
static void load_kquant_expert(const void* ctx, int e, long H, long F, double* Wg, double* Wu,
                               double* Wd) {
    const kquant_experts* k = (const kquant_experts*)ctx;
    qo_dequant_matrix(k->gate_t, k->gate + (long)e * k->sg, F, H, Wg);
    qo_dequant_matrix(k->up_t, k->up + (long)e * k->su, F, H, Wu);
    qo_dequant_matrix(k->down_t, k->down + (long)e * k->sd, H, F, Wd);
}

/* MoE FFN over k-quant experts: Q4_K gate/up [F][H], Q6_K or Q4_K down [H][F]. */
int qo_moe_ffn(int T, int H, int F, int E, int K, const double* x, const double* res,
               const int32_t* ids, const double* w,
               const uint8_t* gate, int gate_t, const uint8_t* up, int up_t,
               const uint8_t* down, int down_t, double* out, double* act, double* ys) {
    kquant_experts k = {gate, up, down, gate_t, up_t, down_t,
                        qo_expert_stride(gate_t, F, H), qo_expert_stride(up_t, F, H),
                        qo_expert_stride(down_t, H, F)};
    if (k.sg < 0 || k.su < 0 || k.sd < 0) return -1;
    return moe_ffn_dense(T, H, F, E, K, x, res, ids, w, load_kquant_expert, &k, out, act, ys);
}

/* ------------------------------------------------------------------ FP8 block-scaled experts */

/* One FP8 E4M3 code (the "fn" variant: sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities; S.1111.111 is NaN).  A zero exponent field
 * is subnormal: m/8 * 2^-6.  Largest finite magnitude 1.75 * 2^8 = 448. */
double qo_fp8_e4m3_to_double(uint8_t c) {
    int s = c >> 7, ex = (c >> 3) & 15, m = c & 7;
    double v;
    if (ex == 15 && m == 7) return NAN;
    if (ex == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, ex - 7);
    return s ? -v : v;
}

/* Block-scaled FP8 matrix ([P3]: FP8 weights with block size 128): codes
 * [rows][cols] e4m3 and one fp32 scale per 128 x 128 tile, stored as
 * scale[(r/128) * ceil(cols/128) + c/128]; W[r][c] = e4m3(code) * scale. */
void qo_fp8_dequant_matrix(const uint8_t* codes, const float* scale, long rows, long cols,
                           double* out) {
    long nb = (cols + 127) / 128;
    for (long r = 0; r < rows; ++r)
        for (long c = 0; c < cols; ++c)
            out[r * cols + c] = qo_fp8_e4m3_to_double(codes[r * cols + c]) *
                                (double)scale[(r / 128) * nb + c / 128];
}

long qo_fp8_scale_count(long rows, long cols) { return ((rows + 127) / 128) * ((cols + 127) / 128); }

typedef struct {
    const uint8_t *gate, *up, *down;
    const float *gs, *us, *ds;
} fp8_experts;

/* Expert e of each 3-D tensor at e * rows * cols codes and
 * e * qo_fp8_scale_count(rows, cols) scales. */
static void load_fp8_expert(const void* ctx, int e, long H, long F, double* Wg, double* Wu,
                            double* Wd) {
    const fp8_experts* k = (const fp8_experts*)ctx;
    long nfh = qo_fp8_scale_count(F, H), nhf = qo_fp8_scale_count(H, F);
    qo_fp8_dequant_matrix(k->gate + (long)e * F * H, k->gs + (long)e * nfh, F, H, Wg);
    qo_fp8_dequant_matrix(k->up + (long)e * F * H, k->us + (long)e * nfh, F, H, Wu);
    qo_fp8_dequant_matrix(k->down + (long)e * H * F, k->ds + (long)e * nhf, H, F, Wd);
}

/* MoE FFN over FP8 block-scaled experts: gate/up [E][F][H] codes with
 * [E][ceil(F/128)][ceil(H/128)] scales, down [E][H][F] with
 * [E][ceil(H/128)][ceil(F/128)]. */
int qo_moe_ffn_fp8(int T, int H, int F, int E, int K, const double* x, const double* res,
                   const int32_t* ids, const double* w, const uint8_t* gate, const float* gate_scale,
                   const uint8_t* up, const float* up_scale, const uint8_t* down,
                   const float* down_scale, double* out, double* act, double* ys) {
    if (H <= 0 || F <= 0) return -1;
    fp8_experts k = {gate, up, down, gate_scale, up_scale, down_scale};
    return moe_ffn_dense(T, H, F, E, K, x, res, ids, w, load_fp8_expert, &k, out, act, ys);
}

/* ------------------------------------------------------------------ NVFP4 experts */

/* One FP4 E2M1 code (low 4 bits): sign, 2 exponent bits with bias 1, 1 mantissa
 * bit; a zero exponent field is subnormal (m/2).  Magnitudes 0, 0.5, 1, 1.5,
 * 2, 3, 4, 6; no infinities or NaN. */
double qo_e2m1_to_double(uint8_t c) {
    int s = (c >> 3) & 1, ex = (c >> 1) & 3, m = c & 1;
    double v = ex == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, ex - 1);
    return s ? -v : v;
}

/* NVFP4 matrix ([P3]: dense weights quantised from BF16 to NVFP4 at load, the
 * "nvfp4_global_absmax" / "quantize_bf16_to_nvfp4" kernels): codes [rows][cols/2]
 * bytes, element c in byte c/2, low nibble for even c; one E4M3 scale per 16
 * consecutive elements of a row, bscale[rows][cols/16]; one fp32 global scale.
 * W[r][c] = e2m1(code) * e4m3(bscale[r][c/16]) * global.  cols % 16 == 0. */
void qo_nvfp4_dequant_matrix(const uint8_t* codes, const uint8_t* bscale, float global, long rows,
                             long cols, double* out) {
    for (long r = 0; r < rows; ++r)
        for (long c = 0; c < cols; ++c) {
            uint8_t b = codes[r * (cols / 2) + c / 2];
            uint8_t q = (c & 1) ? (b >> 4) : (b & 15);
            out[r * cols + c] = qo_e2m1_to_double(q) *
                                qo_fp8_e4m3_to_double(bscale[r * (cols / 16) + c / 16]) *
                                (double)global;
        }
}

typedef struct {
    const uint8_t *gate, *up, *down;          /* codes */
    const uint8_t *gbs, *ubs, *dbs;           /* block scales */
    const float *ggs, *ugs, *dgs;             /* global scales, one per expert */
} nvfp4_experts;

static void load_nvfp4_expert(const void* ctx, int e, long H, long F, double* Wg, double* Wu,
                              double* Wd) {
    const nvfp4_experts* k = (const nvfp4_experts*)ctx;
    qo_nvfp4_dequant_matrix(k->gate + (long)e * F * (H / 2), k->gbs + (long)e * F * (H / 16),
                            k->ggs[e], F, H, Wg);
    qo_nvfp4_dequant_matrix(k->up + (long)e * F * (H / 2), k->ubs + (long)e * F * (H / 16),
                            k->ugs[e], F, H, Wu);
    qo_nvfp4_dequant_matrix(k->down + (long)e * H * (F / 2), k->dbs + (long)e * H * (F / 16),
                            k->dgs[e], H, F, Wd);
}

/* MoE FFN over NVFP4 experts: gate/up codes [E][F][H/2], block scales
 * [E][F][H/16], globals [E]; down codes [E][H][F/2], scales [E][H][F/16],
 * globals [E]. */
int qo_moe_ffn_nvfp4(int T, int H, int F, int E, int K, const double* x, const double* res,
                     const int32_t* ids, const double* w, const uint8_t* gate, const uint8_t* gate_bs,
                     const float* gate_gs, const uint8_t* up, const uint8_t* up_bs,
                     const float* up_gs, const uint8_t* down, const uint8_t* down_bs,
                     const float* down_gs, double* out, double* act, double* ys) {
    if (H <= 0 || F <= 0 || H % 16 || F % 16) return -1;
    nvfp4_experts k = {gate, up, down, gate_bs, up_bs, down_bs, gate_gs, up_gs, down_gs};
    return moe_ffn_dense(T, H, F, E, K, x, res, ids, w, load_nvfp4_expert, &k, out, act, ys);
}

/* Round a non-negative float to the nearest E4M3 code (ties to the even code),
 * saturating at 448 (code 0x7E): a scan over the 127 finite non-negative codes
 * in increasing order. */
static uint8_t e4m3_encode_rne(float t) {
    if (!(t > 0.0f)) return 0;
    if (t >= 448.0f) return 0x7E;
    uint8_t best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
        double lo = qo_fp8_e4m3_to_double((uint8_t)(c - 1)), hi = qo_fp8_e4m3_to_double((uint8_t)c);
        if ((double)t >= hi) { best = (uint8_t)c; continue; }
        /* lo <= t < hi */
        double dl = (double)t - lo, dh = hi - (double)t;
        if (dh < dl || (dh == dl && (c & 1) == 0)) best = (uint8_t)c;
        else best = (uint8_t)(c - 1);
        break;
    }
    return best;
}

/* Round v to the nearest E2M1 code (ties to the even code), saturating at 6;
 * the sign bit is v's (so -0 and small negatives give the code 8, minus zero). */
static uint8_t e2m1_encode_rne(float v) {
    float a = fabsf(v);
    uint8_t m;
    if (a <= 0.25f) m = 0;
    else if (a < 0.75f) m = 1;
    else if (a <= 1.25f) m = 2;
    else if (a < 1.75f) m = 3;
    else if (a <= 2.5f) m = 4;
    else if (a < 3.5f) m = 5;
    else if (a <= 5.0f) m = 6;
    else m = 7;
    return (uint8_t)(m | (signbit(v) ? 8 : 0));
}

static float bf16_to_float(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Runtime quantisation of a BF16 matrix [rows][cols] to NVFP4 ([P3]: a global
 * absmax pass, then the per-block quantisation).  Every decision is taken in
 * fp32, in this order:
 *   amax = max |x|;  global = amax / 2688   (2688 = 448 * 6: the largest block
 *                                            scale times the largest E2M1 value)
 *   per 16-element block: s = e4m3_rne(bmax / (6 * global)), d = e4m3(s) * global,
 *   q = e2m1_rne(x / d) (0 where d = 0).
 * An all-zero matrix has global = 0, zero scales and zero codes.  codes gets
 * rows*cols/2 bytes, bscale rows*cols/16, *global one float. */
int qo_nvfp4_quantize(long rows, long cols, const uint16_t* x, uint8_t* codes, uint8_t* bscale,
                      float* global) {
    if (rows <= 0 || cols <= 0 || cols % 16) return -1;
    float amax = 0.0f;
    for (long i = 0; i < rows * cols; ++i) {
        float a = fabsf(bf16_to_float(x[i]));
        if (a > amax) amax = a;
    }
    float g = amax / 2688.0f;
    *global = g;
    for (long r = 0; r < rows; ++r)
        for (long b = 0; b < cols / 16; ++b) {
            const uint16_t* xb = x + r * cols + 16 * b;
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                float a = fabsf(bf16_to_float(xb[i]));
                if (a > bmax) bmax = a;
            }
            uint8_t s = 0;
            if (g > 0.0f) {
                float den = 6.0f * g;
                s = e4m3_encode_rne(bmax / den);
            }
            bscale[r * (cols / 16) + b] = s;
            float d = (float)qo_fp8_e4m3_to_double(s) * g;
            for (int i = 0; i < 16; i += 2) {
                uint8_t lo = 0, hi = 0;
                if (d > 0.0f) {
                    lo = e2m1_encode_rne(bf16_to_float(xb[i]) / d);
                    hi = e2m1_encode_rne(bf16_to_float(xb[i + 1]) / d);
                }
                codes[r * (cols / 2) + (16 * b + i) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    return 0;
}

/* ------------------------------------------------------------------ Q8_K activations */

/* The int8-activation variant ([P2] "Gaps ... G8": the expert GEMVs run as
 * DP4A kernels on 8-bit activations; "The Q8_K point": that path scored 0.8725
 * where FP32 activations scored 1.0).  The pages name the activation format,
 * Q8_K, without defining it; the reading taken is the GGUF 8-bit activation
 * block: 256 values, one fp32 scale d, 256 int8 codes and 16 sums of 16 codes.
 * The block's value of largest magnitude v (the first, on a tie) maps to code
 * -128: s = -128/v, q_i = min(127, rint(s*x_i)), d = 1/s, all in fp32 (the
 * codes are integers decided by floating point, so they are decided in the
 * precision a kernel uses); an all-zero block has d = 0 and q = 0.
 * n is a multiple of 256; x has n floats; d gets n/256, q n, bsums n/16. */
int qo_q8k_quantize(long n, const float* x, float* d, int8_t* q, int16_t* bsums) {
    if (n % QO_QK) return -1;
    for (long b = 0; b < n / QO_QK; ++b) {
        const float* xb = x + b * QO_QK;
        float v = 0.0f, amax = 0.0f;
        for (int i = 0; i < QO_QK; ++i)
            if (fabsf(xb[i]) > amax) {
                amax = fabsf(xb[i]);
                v = xb[i];
            }
        if (amax == 0.0f) {
            d[b] = 0.0f;
            for (int i = 0; i < QO_QK; ++i) q[b * QO_QK + i] = 0;
        } else {
            volatile float s = -128.0f / v;   /* kept in fp32 */
            for (int i = 0; i < QO_QK; ++i) {
                volatile float t = s * xb[i];
                int c = (int)rintf(t);
                q[b * QO_QK + i] = (int8_t)(c > 127 ? 127 : c);
            }
            d[b] = 1.0f / s;
        }
        for (int g = 0; g < QO_QK / 16; ++g) {
            int acc = 0;
            for (int i = 0; i < 16; ++i) acc += q[b * QO_QK + 16 * g + i];
            bsums[b * (QO_QK / 16) + g] = (int16_t)acc;
        }
    }
    return 0;
}

/* Code (0..15) of element i of a Q4_K superblock and its sub-block j = i/32
 * (layout as in qo_q4k_element). */
static int q4k_code(const uint8_t* blk, int i) {
    int j = i / 32, l = i % 32;
    return (blk[16 + 32 * (j / 2) + l] >> (4 * (j % 2))) & 15;
}

/* Signed code q6 - 32 of element i of a Q6_K superblock and its int8 scale
 * (layout as in qo_q6k_element). */
static int q6k_code(const uint8_t* blk, int i, int* scale) {
    int n = i / 128, g = (i % 128) / 32, l = i % 32;
    int lo = (blk[64 * n + l + 32 * (g % 2)] >> (4 * (g / 2))) & 15;
    int hi = (blk[128 + 32 * n + l] >> (2 * g)) & 3;
    *scale = ((const int8_t*)(blk + 192))[8 * n + l / 16 + 2 * g];
    return (lo | (hi << 4)) - 32;
}

/* Dot product of one weight row (cols/256 superblocks of qtype) with a Q8_K
 * vector, in the integer form an int8 kernel evaluates, superblock by
 * superblock in order:
 *   Q4_K: dx * sum_j [ d*s_j * S_j - dmin*m_j * B_j ], with S_j the integer sum
 *         of q4*q8 over sub-block j (32 values) and B_j the sum of its q8 codes
 *         (the two 16-code sums bsums[2j], bsums[2j+1]);
 *   Q6_K: dx * d * sum over the 16 groups of 16 values of sc_g * sum (q6-32)*q8.
 * Integer sums are exact; the scaling is in double. */
double qo_dot_q8k(int qtype, const uint8_t* row, long cols, const float* d8, const int8_t* q8,
                  const int16_t* bs8) {
    int bb = qo_block_bytes(qtype);
    double acc = 0.0;
    for (long b = 0; b < cols / QO_QK; ++b) {
        const uint8_t* blk = row + b * bb;
        const int8_t* qb = q8 + b * QO_QK;
        const int16_t* sb = bs8 + b * (QO_QK / 16);
        double part = 0.0;
        if (qtype == QO_Q4_K) {
            double d = half_at(blk), dmin = half_at(blk + 2);
            for (int j = 0; j < 8; ++j) {
                long S = 0;
                for (int l = 0; l < 32; ++l) S += (long)q4k_code(blk, 32 * j + l) * qb[32 * j + l];
                long B = (long)sb[2 * j] + sb[2 * j + 1];
                int s, m;
                q4k_scale_min(blk + 4, j, &s, &m);
                part += d * s * (double)S - dmin * m * (double)B;
            }
        } else {
            double d = half_at(blk + 208);
            for (int g = 0; g < 16; ++g) {
                long S = 0;
                int sc = 0;
                for (int l = 0; l < 16; ++l) S += (long)q6k_code(blk, 16 * g + l, &sc) * qb[16 * g + l];
                part += d * sc * (double)S;
            }
        }
        acc += (double)d8[b] * part;
    }
    return acc;
}

/* The MoE FFN of qo_moe_ffn with every expert GEMV on Q8_K activations: the
 * token's x (as fp32) is quantised once for gate and up, the SwiGLU output a
 * (as fp32) once for down; the router, SwiGLU and the weighted sum stay as in
 * qo_moe_ffn.  act (nullable) receives a [T][K][F]. */
int qo_moe_ffn_q8k(int T, int H, int F, int E, int K, const double* x, const double* res,
                   const int32_t* ids, const double* w,
                   const uint8_t* gate, int gate_t, const uint8_t* up, int up_t,
                   const uint8_t* down, int down_t, double* out, double* act) {
    long sg = qo_expert_stride(gate_t, F, H), su = qo_expert_stride(up_t, F, H);
    long sd = qo_expert_stride(down_t, H, F);
    if (sg < 0 || su < 0 || sd < 0 || H % QO_QK || F % QO_QK) return -1;
    for (long p = 0; p < (long)T * K; ++p)
        if (ids[p] < 0 || ids[p] >= E) return -2;
    long rbg = sg / F, rbu = su / F, rbd = sd / H;    /* bytes per weight row */
    double* Y = (double*)malloc(sizeof(double) * (size_t)T * K * H);
    if (!Y) return -3;
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long p = 0; p < (long)T * K; ++p) {
        long t = p / K;
        int e = ids[p];
        float* xf = (float*)malloc(sizeof(float) * (size_t)(H > F ? H : F));
        int8_t* q8 = (int8_t*)malloc((size_t)(H > F ? H : F));
        float* d8 = (float*)malloc(sizeof(float) * (size_t)(H > F ? H : F) / QO_QK);
        int16_t* b8 = (int16_t*)malloc(sizeof(int16_t) * (size_t)(H > F ? H : F) / 16);
        double* a = (double*)malloc(sizeof(double) * (size_t)F);
        if (!xf || !q8 || !d8 || !b8 || !a) {
#pragma omp atomic write
            err = 1;
        } else {
            for (long h = 0; h < H; ++h) xf[h] = (float)x[t * H + h];
            qo_q8k_quantize(H, xf, d8, q8, b8);
            for (long f = 0; f < F; ++f) {
                double g = qo_dot_q8k(gate_t, gate + (long)e * sg + f * rbg, H, d8, q8, b8);
                double u = qo_dot_q8k(up_t, up + (long)e * su + f * rbu, H, d8, q8, b8);
                a[f] = silu(g) * u;
            }
            if (act) memcpy(act + p * F, a, sizeof(double) * (size_t)F);
            for (long f = 0; f < F; ++f) xf[f] = (float)a[f];
            qo_q8k_quantize(F, xf, d8, q8, b8);
            for (long h = 0; h < H; ++h)
                Y[p * H + h] = qo_dot_q8k(down_t, down + (long)e * sd + h * rbd, F, d8, q8, b8);
        }
        free(xf); free(q8); free(d8); free(b8); free(a);
    }
    if (err) { free(Y); return -3; }
    for (long t = 0; t < T; ++t)
        for (long h = 0; h < H; ++h) {
            double acc = res ? res[t * H + h] : x[t * H + h];
            for (long j = 0; j < K; ++j) acc += w[t * K + j] * Y[(t * K + j) * H + h];
            out[t * H + h] = acc;
        }
    free(Y);
    return 0;
}

/* ------------------------------------------------------------------ decoder layer pieces */

/* RMSNorm: x / sqrt(mean(x^2) + eps) * w. */
void qo_rmsnorm(long n, const double* x, const float* w, double eps, double* out) {
    double ss = 0.0;
    for (long i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (long i = 0; i < n; ++i) out[i] = x[i] * r * (double)w[i];
}

/* NEOX rotary embedding of one head ([P5] closing comment): the rotated pairs
 * are (i, i + hd/2) for i < hd/2, angle pos * base^(-2i/hd). */
void qo_rope_neox(int hd, double* v, int pos, double base) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double th = (double)pos * pow(base, -2.0 * (double)i / (double)hd);
        double c = cos(th), s = sin(th);
        double a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = b * c + a * s;
    }
}

/* Single-query attention of one q head over cache positions 0..pos of its kv
 * head: softmax(q . K_p / sqrt(hd)) . V_p.  The cache holds fp16. */
void qo_attend(int hd, const double* q, const uint16_t* Kc, const uint16_t* Vc, int pos,
               double* out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(pos + 1));
    double scale = 1.0 / sqrt((double)hd), mx = -INFINITY;
    for (int p = 0; p <= pos; ++p) {
        double acc = 0.0;
        for (int i = 0; i < hd; ++i) acc += q[i] * qo_half_to_double(Kc[(long)p * hd + i]);
        s[p] = acc * scale;
        if (s[p] > mx) mx = s[p];
    }
    double z = 0.0;
    for (int p = 0; p <= pos; ++p) { s[p] = exp(s[p] - mx); z += s[p]; }
    for (int i = 0; i < hd; ++i) out[i] = 0.0;
    for (int p = 0; p <= pos; ++p)
        for (int i = 0; i < hd; ++i) out[i] += (s[p] / z) * qo_half_to_double(Vc[(long)p * hd + i]);
    free(s);
}

/* One qwen3moe decoder layer at decode time (batch 1), on hidden state h (in/out):
 *  B1 x = RMSNorm(h) * attn_norm
 *  B2 q = Wq x [nq*hd], k = Wk x [nkv*hd], v = Wv x [nkv*hd]   (no bias, [P1])
 *  B3 per-head RMSNorm of q (q_norm) and k (k_norm), after bias, before RoPE ([P4])
 *  B4 NEOX RoPE at position pos, base rope_base ([P5])
 *  B5 k, v rounded to fp16 and written to cache slot pos
 *  B6 GQA: q head hq reads kv head hq / (nq/nkv) over positions 0..pos ([P1])
 *  B7 h += Wo attn
 *  B8 x2 = RMSNorm(h) * ffn_norm
 *  B9 h += MoE(x2) (router + experts, as qo_router / qo_moe_ffn)
 * Caches are [nkv][ctx][hd] fp16; entries before pos are used as stored.
 * q_out / att_out (nullable) receive q after norm+RoPE and the attention output. */
int qo_decode_layer(int H, int E, int K, int F, int nq, int nkv, int hd, int ctx, double eps,
                    double rope_base, int pos, double* h,
                    const float* attn_norm, const float* q_norm, const float* k_norm,
                    const float* ffn_norm, const uint8_t* wq, const uint8_t* wk,
                    const uint8_t* wv, const uint8_t* wo, const float* router,
                    const uint8_t* gate, const uint8_t* up, const uint8_t* down, int down_t,
                    uint16_t* k_cache, uint16_t* v_cache, const int32_t* force,
                    float* logits_out, int32_t* ids_out, double* w_out, double* q_out,
                    double* att_out) {
    if (pos < 0 || pos >= ctx || nq % nkv || hd % 2) return -1;
    long qd = (long)nq * hd, kvd = (long)nkv * hd;
    double* x = (double*)malloc(sizeof(double) * H);
    double* q = (double*)malloc(sizeof(double) * qd);
    double* k = (double*)malloc(sizeof(double) * kvd);
    double* v = (double*)malloc(sizeof(double) * kvd);
    double* att = (double*)malloc(sizeof(double) * qd);
    double* Wbuf = (double*)malloc(sizeof(double) * (size_t)(qd > kvd ? qd : kvd) * (size_t)H);
    double* o = (double*)malloc(sizeof(double) * H);
    double* tmp = (double*)malloc(sizeof(double) * hd);
    if (!x || !q || !k || !v || !att || !Wbuf || !o || !tmp) return -3;

    qo_rmsnorm(H, h, attn_norm, eps, x);                              /* B1 */
    qo_dequant_matrix(QO_Q4_K, wq, qd, H, Wbuf); matvec(Wbuf, qd, H, x, q);   /* B2 */
    qo_dequant_matrix(QO_Q4_K, wk, kvd, H, Wbuf); matvec(Wbuf, kvd, H, x, k);
    qo_dequant_matrix(QO_Q4_K, wv, kvd, H, Wbuf); matvec(Wbuf, kvd, H, x, v);
    for (int hh = 0; hh < nq; ++hh) {                                 /* B3 + B4 */
        qo_rmsnorm(hd, q + (long)hh * hd, q_norm, eps, tmp);
        memcpy(q + (long)hh * hd, tmp, sizeof(double) * hd);
        qo_rope_neox(hd, q + (long)hh * hd, pos, rope_base);
    }
    for (int hh = 0; hh < nkv; ++hh) {
        qo_rmsnorm(hd, k + (long)hh * hd, k_norm, eps, tmp);
        memcpy(k + (long)hh * hd, tmp, sizeof(double) * hd);
        qo_rope_neox(hd, k + (long)hh * hd, pos, rope_base);
    }
    for (int hh = 0; hh < nkv; ++hh)                                  /* B5 */
        for (int i = 0; i < hd; ++i) {
            k_cache[((long)hh * ctx + pos) * hd + i] = qo_double_to_half(k[(long)hh * hd + i]);
            v_cache[((long)hh * ctx + pos) * hd + i] = qo_double_to_half(v[(long)hh * hd + i]);
        }
    int group = nq / nkv;
#pragma omp parallel for schedule(static)
    for (int hh = 0; hh < nq; ++hh) {                                 /* B6 */
        int kvh = hh / group;
        qo_attend(hd, q + (long)hh * hd, k_cache + (long)kvh * ctx * hd,
                  v_cache + (long)kvh * ctx * hd, pos, att + (long)hh * hd);
    }
    if (q_out) memcpy(q_out, q, sizeof(double) * qd);
    if (att_out) memcpy(att_out, att, sizeof(double) * qd);
    qo_dequant_matrix(QO_Q4_K, wo, H, qd, Wbuf); matvec(Wbuf, H, qd, att, o);  /* B7 */
    for (int i = 0; i < H; ++i) h[i] += o[i];
    qo_rmsnorm(H, h, ffn_norm, eps, x);                               /* B8 */
    double* w = (double*)malloc(sizeof(double) * K);                  /* B9 */
    int32_t* ids = (int32_t*)malloc(sizeof(int32_t) * K);
    float* lg = (float*)malloc(sizeof(float) * E);
    qo_router(1, H, E, K, 1, x, router, NULL, force, lg, ids, w, NULL);
    double* out = (double*)malloc(sizeof(double) * H);
    int rc = qo_moe_ffn(1, H, F, E, K, x, h, ids, w, gate, QO_Q4_K, up, QO_Q4_K, down, down_t,
                        out, NULL, NULL);
    if (rc == 0) memcpy(h, out, sizeof(double) * H);
    if (logits_out) memcpy(logits_out, lg, sizeof(float) * E);
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * K);
    if (w_out) memcpy(w_out, w, sizeof(double) * K);
    free(x); free(q); free(k); free(v); free(att); free(Wbuf); free(o); free(tmp);
    free(w); free(ids); free(lg); free(out);
    return rc;
}
