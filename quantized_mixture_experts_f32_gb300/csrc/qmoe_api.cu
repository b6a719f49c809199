// qmoe_api.cu -- the C ABI (include/qmoe.h): argument checks, workspace, and the
// launch sequence of one MoE-FFN layer call on the context's stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <new>

#include "../../include/qmoe.h"
#include "qmoe_internal.h"

struct qmoe_ctx {
    qmoe_config cfg;
    cudaStream_t stream;
    int device;
    char err[512];
    void* ws;
    size_t ws_bytes;
    qmoe::Route route;
    float* act;       // [P][F]
    float* y;         // [P][H]
    float* hin;       // [T][H] staging for qmoe_forward_host
    float* hout;      // [T][H]
    int* status;      // device status word
    unsigned* bar;    // decode kernels' control words (exit counter, launch tag, arrival words)
    unsigned* nvq;    // per-matrix amax words of qmoe_nvfp4_quantize
    unsigned* ltctl;  // counters and launch tag of the one-launch FP8 / NVFP4 decode kernel
    unsigned long long* ltlg; // its tagged router logits [E]
    qmoe::FusedBufs fb; // tagged values passed between the fused kernel's CTAs
    __half* xp;       // [P][H] fp16 gathered x (prefill)
    __half* actp;     // [P][F] fp16 SwiGLU output (prefill)
    int32_t* inv_pos; // [P] pair -> position in the expert-sorted list
    qmoe::Q8Bufs q8;  // Q8_K codes of x and act (qmoe_forward_q8k)
    int num_sms;
    // decode-step scratch
    float* xs;        // [H] normed hidden
    float* q;         // [nq*hd]
    float* kv;        // [2*nkv*hd]
    float* att;       // [nq*hd]
    float* attn_part; // split-K partials
    double* inv_freq; // [head_dim/2] RoPE frequencies
    float2* rope_cs;  // [head_dim/2] cos/sin at the current position
    int attn_splits;
    void* pl_scratch; // batched prefill layer scratch (null: shape not served)
    unsigned long long stall_ns; // test hook: the next fused launch stalls for this long (0: off)
};

namespace {

// message of the last failed qmoe_create on this thread (read via qmoe_last_error(NULL))
thread_local char g_create_err[512] = "";
// test hook: the next n workspace allocations of qmoe_create fail as if out of memory
int g_fail_alloc = 0;

void create_fail(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_create_err, sizeof(g_create_err), fmt, ap);
    va_end(ap);
    fprintf(stderr, "qmoe_create: %s\n", g_create_err);
}

constexpr int DECODE_ALIAS_MAX = 8;
constexpr int FP8_GEMV_MAX = 32;         // qmoe_forward_fp8: largest call on the expert GEMVs
constexpr int NVFP4_QUANT_MATS_MAX = 1024;   // matrices per qmoe_nvfp4_quantize call
constexpr int FUSED_GRID_MAX = 1024;     // largest grid of the fused decode kernel

qmoe_status fail(qmoe_ctx* c, qmoe_status s, const char* fmt, ...) {
    if (c) {
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(c->err, sizeof(c->err), fmt, ap);
        va_end(ap);
    }
    return s;
}

qmoe_status cuda_fail(qmoe_ctx* c, cudaError_t e, const char* what) {
    return fail(c, QMOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_qtype(int q) { return q == QMOE_Q4_K || q == QMOE_Q6_K; }

struct Layout {
    size_t logits, ids, wts, n_used, used_expert, used_first, pair_list, act, y, hin, hout,
        status, bar, arrive, nvq, ltctl, ltlg, xp, actp, inv_pos, logits_part, tokmap, jmap, q8, ftag, xs, q, kv, att, attn_part, inv_freq,
        rope_cs, pl, total;
    int attn_splits;
    bool pl_ok;
};

bool config_ok(const qmoe_config* c, char* why, size_t n) {
    if (!c) { snprintf(why, n, "config is NULL"); return false; }
    if (c->hidden <= 0 || c->hidden % 256) { snprintf(why, n, "hidden=%d is not a positive multiple of 256", c->hidden); return false; }
    if (c->ffn <= 0 || c->ffn % 256) { snprintf(why, n, "ffn=%d is not a positive multiple of 256", c->ffn); return false; }
    if (c->n_experts < 1 || c->n_experts > 1024) { snprintf(why, n, "n_experts=%d outside 1..1024", c->n_experts); return false; }
    if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts) { snprintf(why, n, "top_k=%d outside 1..min(n_experts,16)", c->top_k); return false; }
    if (c->max_tokens < 1 || c->max_tokens > (1 << 20)) { snprintf(why, n, "max_tokens=%d outside 1..2^20", c->max_tokens); return false; }
    const bool attn = c->n_heads || c->n_kv_heads || c->head_dim || c->max_ctx;
    if (attn) {
        if (c->n_heads < 1 || c->n_kv_heads < 1 || c->n_heads % c->n_kv_heads) { snprintf(why, n, "n_heads=%d must be a positive multiple of n_kv_heads=%d", c->n_heads, c->n_kv_heads); return false; }
        if (c->head_dim < 64 || c->head_dim > 256 || c->head_dim % 64) { snprintf(why, n, "head_dim=%d must be a multiple of 64 in 64..256", c->head_dim); return false; }
        if ((c->n_heads * c->head_dim) % 256) { snprintf(why, n, "n_heads*head_dim=%d is not a multiple of 256", c->n_heads * c->head_dim); return false; }
        if ((c->n_kv_heads * c->head_dim) % 256 && c->n_kv_heads * c->head_dim % 32) { snprintf(why, n, "bad kv dim"); return false; }
        if (c->max_ctx < 1 || c->max_ctx > (1 << 18)) { snprintf(why, n, "max_ctx=%d outside 1..262144 (the attention merge keeps two floats per 64 positions in shared memory)", c->max_ctx); return false; }
        if (!(c->rope_base > 0.f) || !(c->rms_eps > 0.f)) { snprintf(why, n, "rope_base and rms_eps must be positive"); return false; }
        if (c->hidden > 4096 || c->n_heads * c->head_dim > 4096) { snprintf(why, n, "decode step serves hidden and n_heads*head_dim up to 4096"); return false; }
        if (!qmoe::attention_supported(c->n_heads, c->n_kv_heads, c->head_dim)) { snprintf(why, n, "attention shape n_heads=%d n_kv_heads=%d head_dim=%d not served (at most 32 q heads per kv head)", c->n_heads, c->n_kv_heads, c->head_dim); return false; }
    }
    return true;
}

Layout layout(const qmoe_config* c) {
    Layout L{};
    const size_t T = c->max_tokens, E = c->n_experts, K = c->top_k, F = c->ffn, H = c->hidden;
    const size_t P = T * K;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    L.logits = take(sizeof(float) * T * E);
    L.ids = take(sizeof(int32_t) * P);
    L.wts = take(sizeof(float) * P);
    L.n_used = take(sizeof(int32_t) * 4);
    L.used_expert = take(sizeof(int32_t) * E);
    L.used_first = take(sizeof(int32_t) * (E + 1));
    L.pair_list = take(sizeof(int32_t) * P);
    L.act = take(sizeof(float) * P * F);
    L.y = take(sizeof(float) * P * H);
    L.hin = take(sizeof(float) * T * H);
    L.hout = take(sizeof(float) * T * H);
    L.status = take(sizeof(int) * 16);
    L.bar = take(sizeof(unsigned) * 64);
    L.arrive = take(sizeof(unsigned) * 4);
    L.nvq = take(sizeof(unsigned) * NVFP4_QUANT_MATS_MAX);
    L.ltctl = take(sizeof(unsigned) * 4);
    L.ltlg = take(sizeof(unsigned long long) * E);
    L.xp = take(sizeof(__half) * P * H);
    L.actp = take(sizeof(__half) * P * F);
    L.inv_pos = take(sizeof(int32_t) * P);
    L.logits_part = take(sizeof(float) * qmoe::route_many_part_floats((int)T, (int)H, (int)E));
    L.tokmap = take(sizeof(uint32_t) * qmoe::route_many_tokmap_words((int)T, (int)E));
    L.jmap = take(E * T);
    L.q8 = take(qmoe::q8_bufs_bytes((int)T, (int)H, (int)K, (int)F));
    const int Tf = (int)(T < 8 ? T : 8);                 // the fused decode kernel serves T <= 8
    L.ftag = take(qmoe::fused_bufs_bytes(Tf, (int)H, (int)E, (int)K, (int)F, FUSED_GRID_MAX));
    const size_t qd = (size_t)c->n_heads * c->head_dim, kvd = (size_t)c->n_kv_heads * c->head_dim;
    L.attn_splits = c->max_ctx > 0 ? qmoe::attn_splits(c->max_ctx) : 0;
    L.xs = take(sizeof(float) * H);
    L.q = take(sizeof(float) * (qd ? qd : 1));
    L.kv = take(sizeof(float) * (2 * kvd + 1));
    L.att = take(sizeof(float) * (qd ? qd : 1));
    L.attn_part = take(sizeof(float) * (size_t)c->n_heads * L.attn_splits * (c->head_dim + 2) + 4);
    L.inv_freq = take(sizeof(double) * (c->head_dim > 0 ? c->head_dim / 2 : 1));
    L.rope_cs = take(sizeof(float2) * (c->head_dim > 0 ? c->head_dim / 2 : 1));
    L.pl_ok = c->n_heads > 0 &&
              qmoe::prefill_layer_supported(c->hidden, c->n_heads, c->n_kv_heads, c->head_dim);
    L.pl = take(L.pl_ok ? qmoe::prefill_layer_scratch_bytes(c->max_tokens, c->hidden, c->n_heads,
                                                            c->n_kv_heads, c->head_dim)
                        : 0);
    L.total = off;
    return L;
}

qmoe_status check_forward(qmoe_ctx* c, const float* in, const float* router_w, const void* g,
                          const void* u, const void* d, int gt, int ut, int dt, int T,
                          const float* out) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    if (!in || !router_w || !g || !u || !d || !out)
        return fail(c, QMOE_ERR_INVALID_ARG, "null tensor pointer");
    if (T < 1 || T > c->cfg.max_tokens)
        return fail(c, QMOE_ERR_SHAPE, "n_tokens=%d outside 1..max_tokens=%d", T, c->cfg.max_tokens);
    if (!valid_qtype(gt) || !valid_qtype(ut) || !valid_qtype(dt))
        return fail(c, QMOE_ERR_UNSUPPORTED_QTYPE, "qtypes gate=%d up=%d down=%d (allowed: 1=Q4_K, 2=Q6_K)", gt, ut, dt);
    if (!aligned16(in) || !aligned16(router_w) || !aligned16(g) || !aligned16(u) || !aligned16(d) || !aligned16(out))
        return fail(c, QMOE_ERR_MISALIGNED, "every tensor base pointer must be 16-byte aligned");
    return QMOE_OK;
}

qmoe_status check_layers(qmoe_ctx* c, const qmoe_layer_weights* layers, int n_layers) {
    for (int l = 0; l < n_layers; ++l) {
        const qmoe_layer_weights& w = layers[l];
        if (!w.attn_norm || !w.wq || !w.wk || !w.wv || !w.wo || !w.q_norm || !w.k_norm ||
            !w.ffn_norm || !w.router_w || !w.gate_exps || !w.up_exps || !w.down_exps ||
            !w.k_cache || !w.v_cache)
            return fail(c, QMOE_ERR_INVALID_ARG, "layer %d: null pointer", l);
        if (!aligned16(w.wq) || !aligned16(w.wk) || !aligned16(w.wv) || !aligned16(w.wo) ||
            !aligned16(w.router_w) || !aligned16(w.gate_exps) || !aligned16(w.up_exps) ||
            !aligned16(w.down_exps) || !aligned16(w.k_cache) || !aligned16(w.v_cache) ||
            !aligned16(w.attn_norm) || !aligned16(w.ffn_norm))
            return fail(c, QMOE_ERR_MISALIGNED, "layer %d: a base pointer is not 16-byte aligned", l);
        if (!valid_qtype(w.down_t))
            return fail(c, QMOE_ERR_UNSUPPORTED_QTYPE, "layer %d: down qtype %d", l, (int)w.down_t);
    }
    return QMOE_OK;
}

qmoe_status run_moe(qmoe_ctx* c, const float* x, const float* res, const float* bias,
                    const float* router_w, const void* gate, const void* up, const void* down,
                    int gt, int ut, int dt, int T, float* out, int32_t* ids_out, float* w_out) {
    const qmoe_config& k = c->cfg;
    qmoe::MoeShape s{T, k.hidden, k.n_experts, k.top_k, k.ffn, k.norm_topk_prob ? 1 : 0};
    qmoe::FusedDebug dbg{c->stall_ns, 1};
    qmoe::T1Plan p1;
    if (qmoe::t1_decode_plan(s, gt, ut, dt, c->num_sms, &p1)) {
        // one token: the whole layer is one latency-oriented kernel
        cudaError_t e = qmoe::launch_t1_decode(
            s, p1, dt, x, res, bias, router_w, static_cast<const uint8_t*>(gate),
            static_cast<const uint8_t*>(up), static_cast<const uint8_t*>(down), out, ids_out, w_out,
            c->fb, nullptr, 0.f, c->stream, c->stall_ns ? &dbg : nullptr);
        c->stall_ns = 0;
        if (e != cudaSuccess) return cuda_fail(c, e, "batch-1 decode launch");
        c->err[0] = 0;
        return QMOE_OK;
    }
    qmoe::FusedPlan plan;
    if (qmoe::fused_decode_plan(s, gt, ut, dt, c->num_sms, &plan)) {
        // decode: the whole layer is one cooperative kernel
        cudaError_t e = qmoe::launch_fused_decode(
            s, plan, x, res, bias, router_w, static_cast<const uint8_t*>(gate),
            static_cast<const uint8_t*>(up), static_cast<const uint8_t*>(down), out, ids_out,
            w_out, c->fb, nullptr, 0.f, c->stream, c->stall_ns ? &dbg : nullptr);
        c->stall_ns = 0;
        if (e != cudaSuccess) return cuda_fail(c, e, "fused decode launch");
        c->err[0] = 0;
        return QMOE_OK;
    }
    const bool many = qmoe::prefill_supported(s, gt, ut, dt) && qmoe::route_many_supported(s, c->route);
    cudaError_t e = many ? qmoe::launch_route_many(s, x, router_w, bias, c->route, c->stream)
                         : qmoe::launch_route(s, x, router_w, bias, c->route, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "route launch");
    if (many) {
        // many tokens: grouped GEMMs on the tensor cores
        e = qmoe::launch_prefill(s, x, res ? res : x, static_cast<const uint8_t*>(gate),
                                 static_cast<const uint8_t*>(up), static_cast<const uint8_t*>(down),
                                 dt, c->route, c->xp, c->actp, c->y, c->inv_pos, out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "prefill launch");
        if (ids_out || w_out) {
            e = qmoe::copy_route_out(s, c->route, ids_out, w_out, c->stream);
            if (e != cudaSuccess) return cuda_fail(c, e, "routing copy");
        }
        c->err[0] = 0;
        return QMOE_OK;
    }
    e = qmoe::launch_gateup(s, x, static_cast<const uint8_t*>(gate), gt,
                            static_cast<const uint8_t*>(up), ut, c->route, c->act, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "gate/up launch");
    e = qmoe::launch_down(s, c->act, static_cast<const uint8_t*>(down), dt, c->route, c->y, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "down launch");
    e = qmoe::launch_combine(s, c->y, c->route, res ? res : x, out, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "combine launch");
    if (ids_out || w_out) {
        e = qmoe::copy_route_out(s, c->route, ids_out, w_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "routing copy");
    }
    c->err[0] = 0;
    return QMOE_OK;
}

}  // namespace

extern "C" {

size_t qmoe_workspace_bytes(const qmoe_config* cfg) {
    char why[256];
    if (!config_ok(cfg, why, sizeof(why))) return 0;
    return layout(cfg).total;
}

int qmoe_fused_decode_available(const qmoe_ctx* c, int n_tokens, qmoe_qtype gate_t,
                                qmoe_qtype up_t, qmoe_qtype down_t) {
    if (!c || n_tokens < 1 || n_tokens > c->cfg.max_tokens) return 0;
    if (!valid_qtype(gate_t) || !valid_qtype(up_t) || !valid_qtype(down_t)) return 0;
    const qmoe_config& k = c->cfg;
    qmoe::MoeShape s{n_tokens, k.hidden, k.n_experts, k.top_k, k.ffn, k.norm_topk_prob ? 1 : 0};
    qmoe::T1Plan p1;
    if (qmoe::t1_decode_plan(s, gate_t, up_t, down_t, c->num_sms, &p1)) return 1;
    qmoe::FusedPlan plan;
    return qmoe::fused_decode_plan(s, gate_t, up_t, down_t, c->num_sms, &plan) ? 1 : 0;
}

size_t qmoe_expert_stride(qmoe_qtype qtype, int rows, int cols) {
    if (!valid_qtype(qtype) || rows < 1 || cols < 256 || cols % 256) return 0;
    return (size_t)rows * qmoe::row_bytes(qtype, cols);
}

qmoe_status qmoe_create(const qmoe_config* cfg, qmoe_ctx** out) {
    g_create_err[0] = 0;
    if (!out) {
        create_fail("out is NULL");
        return QMOE_ERR_INVALID_ARG;
    }
    *out = nullptr;
    qmoe_ctx* c = new (std::nothrow) qmoe_ctx();
    if (!c) {
        create_fail("host allocation of the context failed");
        return QMOE_ERR_NO_MEMORY;
    }
    if (!config_ok(cfg, c->err, sizeof(c->err))) {
        create_fail("%s", c->err);
        delete c;
        return QMOE_ERR_INVALID_ARG;
    }
    c->cfg = *cfg;
    c->stream = static_cast<cudaStream_t>(cfg->stream);
    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) {
        create_fail("cudaGetDevice: %s", cudaGetErrorString(e));
        delete c;
        return QMOE_ERR_CUDA;
    }
    const Layout L = layout(cfg);
    size_t free_b = 0, total_b = 0;
    e = cudaMemGetInfo(&free_b, &total_b);
    if (e != cudaSuccess) {
        create_fail("cudaMemGetInfo: %s", cudaGetErrorString(e));
        delete c;
        return QMOE_ERR_CUDA;
    }
    if (L.total > free_b) {
        create_fail("workspace needs %zu bytes (%.1f MiB) but only %zu bytes (%.1f MiB) of %zu are free",
                    L.total, L.total / 1048576.0, free_b, free_b / 1048576.0, total_b);
        delete c;
        return QMOE_ERR_NO_MEMORY;
    }
    e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        create_fail("cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        delete c;
        return QMOE_ERR_CUDA;
    }
    e = qmoe::fused_prepare();
    if (e == cudaSuccess) e = qmoe::t1_prepare();
    if (e == cudaSuccess) e = qmoe::route_prepare();
    if (e == cudaSuccess) e = qmoe::decode_step_prepare();
    if (e == cudaSuccess && L.pl_ok) e = qmoe::prefill_layer_prepare();
    if (e != cudaSuccess) {
        create_fail("kernel set-up: %s", cudaGetErrorString(e));
        delete c;
        return QMOE_ERR_CUDA;
    }
    if (g_fail_alloc > 0) {
        --g_fail_alloc;
        e = cudaErrorMemoryAllocation;
    } else {
        e = cudaMalloc(&c->ws, L.total);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        create_fail("workspace allocation of %zu bytes (%.1f MiB) failed with %zu bytes (%.1f MiB) free: %s",
                    L.total, L.total / 1048576.0, free_b, free_b / 1048576.0, cudaGetErrorString(e));
        delete c;
        return QMOE_ERR_NO_MEMORY;
    }
    c->ws_bytes = L.total;
    char* b = static_cast<char*>(c->ws);
    c->route.logits = reinterpret_cast<float*>(b + L.logits);
    c->route.ids = reinterpret_cast<int32_t*>(b + L.ids);
    c->route.wts = reinterpret_cast<float*>(b + L.wts);
    c->route.n_used = reinterpret_cast<int32_t*>(b + L.n_used);
    c->route.used_expert = reinterpret_cast<int32_t*>(b + L.used_expert);
    c->route.used_first = reinterpret_cast<int32_t*>(b + L.used_first);
    c->route.pair_list = reinterpret_cast<int32_t*>(b + L.pair_list);
    c->route.logits_part = reinterpret_cast<float*>(b + L.logits_part);
    c->route.tokmap = reinterpret_cast<uint32_t*>(b + L.tokmap);
    c->route.jmap = reinterpret_cast<uint8_t*>(b + L.jmap);
    c->route.arrive = reinterpret_cast<unsigned*>(b + L.arrive);
    c->nvq = reinterpret_cast<unsigned*>(b + L.nvq);
    c->ltctl = reinterpret_cast<unsigned*>(b + L.ltctl);
    c->ltlg = reinterpret_cast<unsigned long long*>(b + L.ltlg);
    c->q8 = qmoe::q8_bufs_carve(reinterpret_cast<unsigned char*>(b + L.q8), c->cfg.max_tokens, c->cfg.hidden,
                                c->cfg.top_k, c->cfg.ffn);
    c->act = reinterpret_cast<float*>(b + L.act);
    c->y = reinterpret_cast<float*>(b + L.y);
    c->hin = reinterpret_cast<float*>(b + L.hin);
    c->hout = reinterpret_cast<float*>(b + L.hout);
    c->status = reinterpret_cast<int*>(b + L.status);
    c->bar = reinterpret_cast<unsigned*>(b + L.bar);
    {
        const int Tf = c->cfg.max_tokens < 8 ? c->cfg.max_tokens : 8;
        c->fb = qmoe::fused_bufs_carve(reinterpret_cast<unsigned char*>(b + L.ftag), Tf, c->cfg.hidden, c->cfg.n_experts,
                                       c->cfg.top_k, c->cfg.ffn, FUSED_GRID_MAX, c->bar, c->status);
    }
    c->xp = reinterpret_cast<__half*>(b + L.xp);
    c->actp = reinterpret_cast<__half*>(b + L.actp);
    c->inv_pos = reinterpret_cast<int32_t*>(b + L.inv_pos);
    c->xs = reinterpret_cast<float*>(b + L.xs);
    c->q = reinterpret_cast<float*>(b + L.q);
    c->kv = reinterpret_cast<float*>(b + L.kv);
    c->att = reinterpret_cast<float*>(b + L.att);
    c->attn_part = reinterpret_cast<float*>(b + L.attn_part);
    c->attn_splits = L.attn_splits;
    c->inv_freq = reinterpret_cast<double*>(b + L.inv_freq);
    c->rope_cs = reinterpret_cast<float2*>(b + L.rope_cs);
    c->pl_scratch = L.pl_ok ? b + L.pl : nullptr;
    e = cudaMemsetAsync(c->ws, 0, L.total, c->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) {
        create_fail("workspace clear: %s", cudaGetErrorString(e));
        cudaFree(c->ws);
        delete c;
        return QMOE_ERR_CUDA;
    }
    if (c->cfg.head_dim > 0) {
        // RoPE frequencies base^(-2j/head_dim), j < head_dim/2, in double
        const int half = c->cfg.head_dim / 2;
        double f[128];
        for (int j = 0; j < half; ++j)
            f[j] = pow((double)c->cfg.rope_base, -2.0 * (double)j / (double)c->cfg.head_dim);
        e = cudaMemcpy(c->inv_freq, f, sizeof(double) * half, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            create_fail("RoPE table upload: %s", cudaGetErrorString(e));
            cudaFree(c->ws);
            delete c;
            return QMOE_ERR_CUDA;
        }
    }
    *out = c;
    return QMOE_OK;
}

void qmoe_destroy(qmoe_ctx* c) {
    if (!c) return;
    cudaStreamSynchronize(c->stream);
    cudaFree(c->ws);
    delete c;
}

qmoe_status qmoe_set_stream(qmoe_ctx* c, void* stream) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    c->stream = static_cast<cudaStream_t>(stream);
    c->cfg.stream = stream;
    return QMOE_OK;
}

qmoe_status qmoe_forward(qmoe_ctx* c, const float* hidden_in, const float* router_w,
                         const void* gate_exps, const void* up_exps, const void* down_exps,
                         qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t, int n_tokens,
                         float* hidden_out) {
    qmoe_status s = check_forward(c, hidden_in, router_w, gate_exps, up_exps, down_exps, gate_t,
                                  up_t, down_t, n_tokens, hidden_out);
    if (s != QMOE_OK) return s;
    if (hidden_in == hidden_out && n_tokens > DECODE_ALIAS_MAX)
        return fail(c, QMOE_ERR_INVALID_ARG, "hidden_out may alias hidden_in only for n_tokens <= %d", DECODE_ALIAS_MAX);
    return run_moe(c, hidden_in, nullptr, nullptr, router_w, gate_exps, up_exps, down_exps, gate_t,
                   up_t, down_t, n_tokens, hidden_out, nullptr, nullptr);
}

qmoe_status qmoe_forward_ex(qmoe_ctx* c, const float* ffn_in, const float* residual,
                            const float* router_bias, const float* router_w,
                            const void* gate_exps, const void* up_exps, const void* down_exps,
                            qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t, int n_tokens,
                            float* out, int32_t* ids_out, float* weights_out) {
    qmoe_status s = check_forward(c, ffn_in, router_w, gate_exps, up_exps, down_exps, gate_t,
                                  up_t, down_t, n_tokens, out);
    if (s != QMOE_OK) return s;
    if ((residual && !aligned16(residual)) || (router_bias && !aligned16(router_bias)))
        return fail(c, QMOE_ERR_MISALIGNED, "residual / router_bias must be 16-byte aligned");
    if (out == ffn_in && n_tokens > DECODE_ALIAS_MAX)
        return fail(c, QMOE_ERR_INVALID_ARG, "out may alias ffn_in only for n_tokens <= %d", DECODE_ALIAS_MAX);
    if (residual && out == residual && n_tokens > DECODE_ALIAS_MAX)
        return fail(c, QMOE_ERR_INVALID_ARG, "out may alias residual only for n_tokens <= %d", DECODE_ALIAS_MAX);
    return run_moe(c, ffn_in, residual, router_bias, router_w, gate_exps, up_exps, down_exps,
                   gate_t, up_t, down_t, n_tokens, out, ids_out, weights_out);
}

qmoe_status qmoe_forward_q8k(qmoe_ctx* c, const float* hidden_in, const float* router_w,
                             const void* gate_exps, const void* up_exps, const void* down_exps,
                             qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t, int n_tokens,
                             float* hidden_out, int32_t* ids_out, float* weights_out) {
    qmoe_status s = check_forward(c, hidden_in, router_w, gate_exps, up_exps, down_exps, gate_t,
                                  up_t, down_t, n_tokens, hidden_out);
    if (s != QMOE_OK) return s;
    const qmoe_config& k = c->cfg;
    qmoe::MoeShape ms{n_tokens, k.hidden, k.n_experts, k.top_k, k.ffn, k.norm_topk_prob ? 1 : 0};
    cudaError_t e = qmoe::launch_route(ms, hidden_in, router_w, nullptr, c->route, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "route launch");
    e = qmoe::launch_moe_q8k(ms, hidden_in, hidden_in, static_cast<const uint8_t*>(gate_exps), gate_t,
                             static_cast<const uint8_t*>(up_exps), up_t,
                             static_cast<const uint8_t*>(down_exps), down_t, c->route, c->q8, c->act,
                             c->y, hidden_out, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "Q8_K expert launch");
    if (ids_out || weights_out) {
        e = qmoe::copy_route_out(ms, c->route, ids_out, weights_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "routing copy");
    }
    c->err[0] = 0;
    return QMOE_OK;
}

qmoe_status qmoe_forward_fp8(qmoe_ctx* c, const float* hidden_in, const float* router_w,
                             const void* gate_exps, const float* gate_scale, const void* up_exps,
                             const float* up_scale, const void* down_exps,
                             const float* down_scale, int n_tokens, float* hidden_out,
                             int32_t* ids_out, float* weights_out) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    if (!hidden_in || !router_w || !gate_exps || !gate_scale || !up_exps || !up_scale ||
        !down_exps || !down_scale || !hidden_out)
        return fail(c, QMOE_ERR_INVALID_ARG, "null tensor pointer");
    const qmoe_config& k = c->cfg;
    if (n_tokens < 1 || n_tokens > k.max_tokens)
        return fail(c, QMOE_ERR_SHAPE, "n_tokens=%d outside 1..max_tokens=%d", n_tokens, k.max_tokens);
    if (!qmoe::fp8_supported(k.hidden, k.ffn))
        return fail(c, QMOE_ERR_SHAPE, "FP8 experts serve hidden/256 in {2,4,8,16} and ffn/256 in 1..6 (hidden=%d ffn=%d)", k.hidden, k.ffn);
    if (!aligned16(hidden_in) || !aligned16(router_w) || !aligned16(gate_exps) ||
        !aligned16(up_exps) || !aligned16(down_exps) || !aligned16(hidden_out))
        return fail(c, QMOE_ERR_MISALIGNED, "activation, router and code base pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(gate_scale) | reinterpret_cast<uintptr_t>(up_scale) |
         reinterpret_cast<uintptr_t>(down_scale)) & 3u)
        return fail(c, QMOE_ERR_MISALIGNED, "scale pointers must be 4-byte aligned");
    qmoe::MoeShape ms{n_tokens, k.hidden, k.n_experts, k.top_k, k.ffn, k.norm_topk_prob ? 1 : 0};
    const qmoe::Fp8Experts w{static_cast<const uint8_t*>(gate_exps), gate_scale,
                             static_cast<const uint8_t*>(up_exps), up_scale,
                             static_cast<const uint8_t*>(down_exps), down_scale};
    if (qmoe::lowbit_t1_supported(1, n_tokens, k.hidden, k.n_experts, k.top_k, k.ffn, c->num_sms)) {
        // one token: the whole layer is one kernel
        cudaError_t e = qmoe::launch_lowbit_t1(1, ms, hidden_in, router_w, &w, nullptr, c->act, hidden_out,
                                               ids_out, weights_out, c->ltlg, c->ltctl, c->status,
                                               c->num_sms, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "FP8 decode launch");
        c->err[0] = 0;
        return QMOE_OK;
    }
    // up to FP8_GEMV_MAX tokens: expert GEMVs on the CUDA cores; more: grouped
    // GEMMs on the tensor cores
    const bool many = n_tokens > FP8_GEMV_MAX && qmoe::route_many_supported(ms, c->route) &&
                      qmoe::prefill_fp8_supported(ms);
    cudaError_t e = many ? qmoe::launch_route_many(ms, hidden_in, router_w, nullptr, c->route, c->stream)
                         : qmoe::launch_route(ms, hidden_in, router_w, nullptr, c->route, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "route launch");
    if (many) {
        e = qmoe::launch_prefill_fp8(ms, hidden_in, hidden_in, w, c->route, c->xp, c->actp, c->y,
                                     c->inv_pos, hidden_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "FP8 tensor-core expert launch");
    } else {
        e = qmoe::launch_fp8_experts(ms, hidden_in, w, c->route, c->act, c->y, c->num_sms, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "FP8 expert launch");
        e = qmoe::launch_combine(ms, c->y, c->route, hidden_in, hidden_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "combine launch");
    }
    if (ids_out || weights_out) {
        e = qmoe::copy_route_out(ms, c->route, ids_out, weights_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "routing copy");
    }
    c->err[0] = 0;
    return QMOE_OK;
}

qmoe_status qmoe_forward_nvfp4(qmoe_ctx* c, const float* hidden_in, const float* router_w,
                               const void* gate_exps, const void* gate_bscale, const float* gate_global,
                               const void* up_exps, const void* up_bscale, const float* up_global,
                               const void* down_exps, const void* down_bscale,
                               const float* down_global, int n_tokens, float* hidden_out,
                               int32_t* ids_out, float* weights_out) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    if (!hidden_in || !router_w || !gate_exps || !gate_bscale || !gate_global || !up_exps ||
        !up_bscale || !up_global || !down_exps || !down_bscale || !down_global || !hidden_out)
        return fail(c, QMOE_ERR_INVALID_ARG, "null tensor pointer");
    const qmoe_config& k = c->cfg;
    if (n_tokens < 1 || n_tokens > k.max_tokens)
        return fail(c, QMOE_ERR_SHAPE, "n_tokens=%d outside 1..max_tokens=%d", n_tokens, k.max_tokens);
    if (!qmoe::nvfp4_supported(k.hidden, k.ffn))
        return fail(c, QMOE_ERR_SHAPE, "NVFP4 experts serve hidden/512 in {1,2,4,8} and ffn/256 in 1..6 (hidden=%d ffn=%d)", k.hidden, k.ffn);
    if (!aligned16(hidden_in) || !aligned16(router_w) || !aligned16(gate_exps) ||
        !aligned16(up_exps) || !aligned16(down_exps) || !aligned16(hidden_out))
        return fail(c, QMOE_ERR_MISALIGNED, "activation, router and code base pointers must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(gate_bscale) | reinterpret_cast<uintptr_t>(up_bscale) |
         reinterpret_cast<uintptr_t>(down_bscale)) & 1u)
        return fail(c, QMOE_ERR_MISALIGNED, "block-scale pointers must be 2-byte aligned");
    if ((reinterpret_cast<uintptr_t>(gate_global) | reinterpret_cast<uintptr_t>(up_global) |
         reinterpret_cast<uintptr_t>(down_global)) & 3u)
        return fail(c, QMOE_ERR_MISALIGNED, "global-scale pointers must be 4-byte aligned");
    qmoe::MoeShape ms{n_tokens, k.hidden, k.n_experts, k.top_k, k.ffn, k.norm_topk_prob ? 1 : 0};
    const qmoe::NvExperts w{static_cast<const uint8_t*>(gate_exps), static_cast<const uint8_t*>(gate_bscale),
                            gate_global, static_cast<const uint8_t*>(up_exps),
                            static_cast<const uint8_t*>(up_bscale), up_global,
                            static_cast<const uint8_t*>(down_exps), static_cast<const uint8_t*>(down_bscale),
                            down_global};
    if (qmoe::lowbit_t1_supported(2, n_tokens, k.hidden, k.n_experts, k.top_k, k.ffn, c->num_sms)) {
        // one token: the whole layer is one kernel
        cudaError_t e = qmoe::launch_lowbit_t1(2, ms, hidden_in, router_w, nullptr, &w, c->act, hidden_out,
                                               ids_out, weights_out, c->ltlg, c->ltctl, c->status,
                                               c->num_sms, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "NVFP4 decode launch");
        c->err[0] = 0;
        return QMOE_OK;
    }
    const bool many = n_tokens > FP8_GEMV_MAX && qmoe::route_many_supported(ms, c->route);
    // the tensor-core path copies the block scales by TMA (16-byte aligned rows)
    const bool tc = many && qmoe::prefill_nvfp4_supported(ms) && aligned16(gate_bscale) &&
                    aligned16(up_bscale) && aligned16(down_bscale);
    cudaError_t e = many ? qmoe::launch_route_many(ms, hidden_in, router_w, nullptr, c->route, c->stream)
                         : qmoe::launch_route(ms, hidden_in, router_w, nullptr, c->route, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "route launch");
    if (tc) {
        e = qmoe::launch_prefill_nvfp4(ms, hidden_in, hidden_in, w, c->route, c->xp, c->actp, c->y,
                                       c->inv_pos, hidden_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "NVFP4 tensor-core expert launch");
    } else {
        e = qmoe::launch_nvfp4_experts(ms, hidden_in, w, c->route, c->act, c->y, c->num_sms, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "NVFP4 expert launch");
        e = qmoe::launch_combine(ms, c->y, c->route, hidden_in, hidden_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "combine launch");
    }
    if (ids_out || weights_out) {
        e = qmoe::copy_route_out(ms, c->route, ids_out, weights_out, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "routing copy");
    }
    c->err[0] = 0;
    return QMOE_OK;
}

qmoe_status qmoe_nvfp4_quantize(qmoe_ctx* c, const void* x_bf16, int n_mats, int rows, int cols,
                                void* codes, void* bscale, float* global) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    if (!x_bf16 || !codes || !bscale || !global)
        return fail(c, QMOE_ERR_INVALID_ARG, "null tensor pointer");
    if (n_mats < 1 || n_mats > NVFP4_QUANT_MATS_MAX || rows < 1 || cols < 16 || cols % 16)
        return fail(c, QMOE_ERR_SHAPE, "n_mats=%d (1..%d), rows=%d, cols=%d (a positive multiple of 16)",
                    n_mats, NVFP4_QUANT_MATS_MAX, rows, cols);
    if (!aligned16(x_bf16) || (reinterpret_cast<uintptr_t>(codes) & 7u) ||
        (reinterpret_cast<uintptr_t>(global) & 3u))
        return fail(c, QMOE_ERR_MISALIGNED, "x 16-byte, codes 8-byte and global 4-byte aligned");
    const cudaError_t e = qmoe::launch_nvfp4_quantize(
        static_cast<const uint16_t*>(x_bf16), n_mats, rows, cols, static_cast<uint8_t*>(codes),
        static_cast<uint8_t*>(bscale), global, c->nvq, c->num_sms, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "NVFP4 quantise launch");
    c->err[0] = 0;
    return QMOE_OK;
}

qmoe_status qmoe_forward_host(qmoe_ctx* c, const float* hin, const float* router_w,
                              const void* gate_exps, const void* up_exps, const void* down_exps,
                              qmoe_qtype gate_t, qmoe_qtype up_t, qmoe_qtype down_t, int n_tokens,
                              float* hout) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    if (!hin || !hout) return fail(c, QMOE_ERR_INVALID_ARG, "null host activation pointer");
    qmoe_status s = check_forward(c, c->hin, router_w, gate_exps, up_exps, down_exps, gate_t, up_t,
                                  down_t, n_tokens, c->hout);
    if (s != QMOE_OK) return s;
    const size_t bytes = sizeof(float) * (size_t)n_tokens * c->cfg.hidden;
    cudaError_t e = cudaMemcpyAsync(c->hin, hin, bytes, cudaMemcpyHostToDevice, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "host->device copy");
    s = run_moe(c, c->hin, nullptr, nullptr, router_w, gate_exps, up_exps, down_exps, gate_t, up_t,
                down_t, n_tokens, c->hout, nullptr, nullptr);
    if (s != QMOE_OK) return s;
    e = cudaMemcpyAsync(hout, c->hout, bytes, cudaMemcpyDeviceToHost, c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "device->host copy");
    e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "stream synchronize");
    return QMOE_OK;
}

qmoe_status qmoe_decode_step(qmoe_ctx* c, const qmoe_layer_weights* layers, int n_layers, int pos,
                             float* hidden, int32_t* ids_out) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    const qmoe_config& k = c->cfg;
    if (k.n_heads < 1 || k.max_ctx < 1)
        return fail(c, QMOE_ERR_INVALID_ARG, "context was created without attention geometry");
    if (!layers || n_layers < 1 || !hidden)
        return fail(c, QMOE_ERR_INVALID_ARG, "null layers / hidden or n_layers < 1");
    if (pos < 0 || pos >= k.max_ctx)
        return fail(c, QMOE_ERR_SHAPE, "pos=%d outside 0..max_ctx-1=%d", pos, k.max_ctx - 1);
    if (!aligned16(hidden)) return fail(c, QMOE_ERR_MISALIGNED, "hidden must be 16-byte aligned");
    {
        qmoe_status ls = check_layers(c, layers, n_layers);
        if (ls != QMOE_OK) return ls;
    }
    qmoe::AttnShape a{k.hidden, k.n_heads, k.n_kv_heads, k.head_dim, k.max_ctx, pos, k.rms_eps,
                      k.rope_base, c->inv_freq, c->rope_cs};
    {
        // cos/sin of the RoPE angles at pos: one table for every layer
        cudaError_t e = qmoe::launch_rope_table(c->inv_freq, k.head_dim, pos, c->rope_cs, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "rope table launch");
    }
    // the hidden state alternates between `hidden` and the context's staging
    // row: the fused MoE layer then never writes over its own input (no wait
    // for every CTA to have staged x before the first output row)
    float* cur = hidden;
    float* other = c->hout;
    for (int l = 0; l < n_layers; ++l) {
        const qmoe_layer_weights& w = layers[l];
        qmoe::LayerAttn la{w.attn_norm,
                           static_cast<const uint8_t*>(w.wq),
                           static_cast<const uint8_t*>(w.wk),
                           static_cast<const uint8_t*>(w.wv),
                           static_cast<const uint8_t*>(w.wo),
                           w.q_norm,
                           w.k_norm,
                           static_cast<__half*>(w.k_cache),
                           static_cast<__half*>(w.v_cache)};
        // B1-B7: h += Wo attn(...)
        cudaError_t e = qmoe::launch_attention_block(a, la, cur, c->xs, c->q, c->kv, c->att,
                                                     c->attn_part, cur, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "attention launch");
        // B8 + B9: h = h + MoE(RMSNorm(h) * ffn_norm); the fused decode kernel
        // normalises x itself, other paths take a separate normalisation
        int32_t* ids_l = ids_out ? ids_out + (size_t)l * k.top_k : nullptr;
        qmoe::MoeShape ms{1, k.hidden, k.n_experts, k.top_k, k.ffn, k.norm_topk_prob ? 1 : 0};
        qmoe::T1Plan p1;
        qmoe::FusedPlan plan;
        if (qmoe::t1_decode_plan(ms, QMOE_Q4_K, QMOE_Q4_K, w.down_t, c->num_sms, &p1)) {
            e = qmoe::launch_t1_decode(
                ms, p1, w.down_t, cur, cur, nullptr, w.router_w,
                static_cast<const uint8_t*>(w.gate_exps), static_cast<const uint8_t*>(w.up_exps),
                static_cast<const uint8_t*>(w.down_exps), other, ids_l, nullptr, c->fb,
                w.ffn_norm, k.rms_eps, c->stream);
            if (e != cudaSuccess) return cuda_fail(c, e, "batch-1 decode launch");
            float* t = cur;
            cur = other;
            other = t;
        } else if (qmoe::fused_decode_plan(ms, QMOE_Q4_K, QMOE_Q4_K, w.down_t, c->num_sms, &plan)) {
            e = qmoe::launch_fused_decode(
                ms, plan, cur, cur, nullptr, w.router_w,
                static_cast<const uint8_t*>(w.gate_exps), static_cast<const uint8_t*>(w.up_exps),
                static_cast<const uint8_t*>(w.down_exps), other, ids_l, nullptr, c->fb,
                w.ffn_norm, k.rms_eps, c->stream);
            if (e != cudaSuccess) return cuda_fail(c, e, "fused decode launch");
            float* t = cur;
            cur = other;
            other = t;
        } else {
            e = qmoe::launch_rmsnorm(cur, w.ffn_norm, k.rms_eps, k.hidden, c->xs, c->stream);
            if (e != cudaSuccess) return cuda_fail(c, e, "ffn norm launch");
            qmoe_status st = run_moe(c, c->xs, cur, nullptr, w.router_w, w.gate_exps,
                                     w.up_exps, w.down_exps, QMOE_Q4_K, QMOE_Q4_K, w.down_t, 1,
                                     cur, ids_l, nullptr);
            if (st != QMOE_OK) return st;
        }
    }
    if (cur != hidden) {
        cudaError_t e = cudaMemcpyAsync(hidden, cur, sizeof(float) * k.hidden,
                                        cudaMemcpyDeviceToDevice, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "hidden copy");
    }
    c->err[0] = 0;
    return QMOE_OK;
}

qmoe_status qmoe_prefill(qmoe_ctx* c, const qmoe_layer_weights* layers, int n_layers, int n_tokens,
                         int pos0, float* hidden, int32_t* ids_out) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    const qmoe_config& k = c->cfg;
    if (k.n_heads < 1 || k.max_ctx < 1)
        return fail(c, QMOE_ERR_INVALID_ARG, "context was created without attention geometry");
    if (!c->pl_scratch)
        return fail(c, QMOE_ERR_SHAPE, "batched prefill does not serve n_heads=%d n_kv_heads=%d head_dim=%d "
                    "(needs at most 8 q heads per kv head and 128-row multiples)", k.n_heads, k.n_kv_heads, k.head_dim);
    if (!layers || n_layers < 1 || !hidden)
        return fail(c, QMOE_ERR_INVALID_ARG, "null layers / hidden or n_layers < 1");
    if (n_tokens < 1 || n_tokens > k.max_tokens)
        return fail(c, QMOE_ERR_SHAPE, "n_tokens=%d outside 1..max_tokens=%d", n_tokens, k.max_tokens);
    if (pos0 < 0 || pos0 > k.max_ctx - n_tokens)
        return fail(c, QMOE_ERR_SHAPE, "positions %d..%d outside 0..max_ctx-1=%d", pos0, pos0 + n_tokens - 1,
                    k.max_ctx - 1);
    if (!aligned16(hidden)) return fail(c, QMOE_ERR_MISALIGNED, "hidden must be 16-byte aligned");
    {
        qmoe_status ls = check_layers(c, layers, n_layers);
        if (ls != QMOE_OK) return ls;
    }
    float* x2 = qmoe::prefill_layer_x2(c->pl_scratch, n_tokens, k.hidden, k.n_heads, k.n_kv_heads, k.head_dim);
    for (int l = 0; l < n_layers; ++l) {
        const qmoe_layer_weights& w = layers[l];
        qmoe::PrefillLayerArgs a{n_tokens, k.hidden, k.n_heads, k.n_kv_heads, k.head_dim, k.max_ctx, pos0,
                                 k.rms_eps, c->inv_freq, w.attn_norm,
                                 static_cast<const uint8_t*>(w.wq), static_cast<const uint8_t*>(w.wk),
                                 static_cast<const uint8_t*>(w.wv), static_cast<const uint8_t*>(w.wo),
                                 w.q_norm, w.k_norm, w.ffn_norm,
                                 static_cast<__half*>(w.k_cache), static_cast<__half*>(w.v_cache),
                                 hidden, c->pl_scratch, c->status};
        // B1-B8: h += Wo attn(...), x2 = RMSNorm(h) * ffn_norm
        cudaError_t e = qmoe::launch_prefill_layer_attn(a, c->stream);
        if (e != cudaSuccess) return cuda_fail(c, e, "prefill attention launch");
        // B9: h = h + MoE(x2).  The residual is updated in place: every output
        // element is formed from the same element of the residual by one thread
        int32_t* ids_l = ids_out ? ids_out + (size_t)l * n_tokens * k.top_k : nullptr;
        qmoe_status st = run_moe(c, x2, hidden, nullptr, w.router_w, w.gate_exps, w.up_exps,
                                 w.down_exps, QMOE_Q4_K, QMOE_Q4_K, w.down_t, n_tokens, hidden, ids_l,
                                 nullptr);
        if (st != QMOE_OK) return st;
    }
    c->err[0] = 0;
    return QMOE_OK;
}

qmoe_status qmoe_get_status(qmoe_ctx* c) {
    if (!c) return QMOE_ERR_INVALID_ARG;
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return cuda_fail(c, e, "stream synchronize");
    int st = 0;
    e = cudaMemcpy(&st, c->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "status read");
    if (st != 0) {
        cudaMemset(c->status, 0, sizeof(int) * 16);
        return fail(c, static_cast<qmoe_status>(st), "device reported status %d", st);
    }
    return QMOE_OK;
}

const char* qmoe_last_error(qmoe_ctx* c) { return c ? c->err : g_create_err; }

qmoe_status qmoe_debug_stall_next(qmoe_ctx* c, uint64_t wait_ns) {
    if (!c || wait_ns == 0) return QMOE_ERR_INVALID_ARG;
    c->stall_ns = wait_ns;
    return QMOE_OK;
}

void qmoe_debug_fail_alloc(int n) { g_fail_alloc = n > 0 ? n : 0; }

}  // extern "C"
