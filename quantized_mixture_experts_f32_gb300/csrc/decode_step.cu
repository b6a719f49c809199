// decode_step.cu -- the attention half of a qwen3moe decoder layer at decode
// time (batch 1): RMSNorm, Q/K/V and O projections (Q4_K dequant-GEMV),
// per-head Q/K RMSNorm, NEOX RoPE, fp16 KV-cache append and GQA attention.
//
// Step order and details: aprender issue "Qwen3 GPU inference produces garbage
// output" ("Fix Applied": head_dim 128 is explicit, q_dim = n_heads*head_dim
// != hidden, GQA uses head_dim), aprender PR "apply per-head Q/K RMSNorm in
// forward_qwen3_moe" ("The fix": per-head RMSNorm of q and k after the bias,
// before RoPE), SharpInference issue "Forward-pass divergence on Qwen3-Coder
// 30B-A3B" (closing comment: NEOX rotation, pairs offset by head_dim/2).
#include <cuda_fp16.h>
#include <math.h>

#include "kquant.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

// out = h / sqrt(mean(h^2) + eps) * w   (one CTA)
__global__ void __launch_bounds__(512) rmsnorm_kernel(const float* __restrict__ h,
                                                      const float* __restrict__ w, float eps, int n,
                                                      float* __restrict__ out) {
    __shared__ float part[16];
    float ss = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) ss = fmaf(h[i], h[i], ss);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) tot += part[i];
    const float r = rsqrtf(tot / (float)n + eps);
    for (int i = threadIdx.x; i < n; i += blockDim.x) out[i] = h[i] * r * w[i];
}

constexpr int GV_ROWS = 8;      // rows per CTA (one per warp)

struct GemvSeg {
    const uint8_t* W;   // Q4_K [rows][cols/256 superblocks]
    float* y;
    const float* res;   // nullable: y = W x + res
    int rows;
};

struct GemvArgs {
    GemvSeg seg[3];
    int nseg;
    int cols;
    const float* x;
};

// y = W x (+ res) for up to three Q4_K matrices sharing the same x; one warp per
// row, 16-byte pieces decoded in registers, x and its 16-column sums in smem
__global__ void __launch_bounds__(256) q4k_gemv(const GemvArgs a) {
    extern __shared__ float sx[];
    float* xsum = sx + a.cols;
    for (int i = threadIdx.x; i < a.cols / 4; i += blockDim.x)
        reinterpret_cast<float4*>(sx)[i] = reinterpret_cast<const float4*>(a.x)[i];
    __syncthreads();
    for (int i = threadIdx.x; i < a.cols / 16; i += blockDim.x) {
        const float4* q = reinterpret_cast<const float4*>(sx + 16 * i);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) s += (q[j].x + q[j].y) + (q[j].z + q[j].w);
        xsum[i] = s;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int r = blockIdx.x * GV_ROWS + warp;
    int sidx = 0;
    while (sidx < a.nseg && r >= a.seg[sidx].rows) { r -= a.seg[sidx].rows; ++sidx; }
    if (sidx >= a.nseg) return;
    const GemvSeg& sg = a.seg[sidx];
    const int nsb = a.cols / QK;
    const uint8_t* row = sg.W + (size_t)r * nsb * Q4K_BYTES;
    float acc = 0.f;
    for (int t = lane; t < 8 * nsb; t += 32) {
        const int s = t >> 3, pc = t & 7;
        const uint8_t* sb = row + (size_t)s * Q4K_BYTES;
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(sb));
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(sb + 16 + 16 * pc));
        const int col = QK * s + 64 * (pc >> 1) + 16 * (pc & 1);
        float PA, PB;
        q4_piece_dot(q, reinterpret_cast<const float4*>(sx + col),
                     reinterpret_cast<const float4*>(sx + col + 32), PA, PB);
        acc += q4_piece_finish(hdr, pc, PA, PB, xsum[col / 16], xsum[col / 16 + 2]);
    }
    acc = warp_sum(acc);
    if (lane == 0) sg.y[r] = acc + (sg.res ? sg.res[r] : 0.f);
}

// Per head: RMSNorm (q with q_norm, k with k_norm), NEOX RoPE at pos, then k and
// v rounded to fp16 into cache slot pos.  blocks: nq + nkv, threads: hd
__global__ void qk_norm_rope_append(float* __restrict__ q, const float* __restrict__ k,
                                    const float* __restrict__ v, const float* __restrict__ q_norm,
                                    const float* __restrict__ k_norm, float eps, int pos,
                                    float rope_base, int hd, int nq, int nkv, int max_ctx,
                                    __half* __restrict__ k_cache, __half* __restrict__ v_cache) {
    extern __shared__ float buf[];        // hd values + 32 partials
    float* part = buf + hd;
    const int head = blockIdx.x, i = threadIdx.x;
    const bool is_q = head < nq;
    const int kvh = head - nq;
    const float* src = is_q ? q + (size_t)head * hd : k + (size_t)kvh * hd;
    const float val = src[i];
    float ss = warp_sum(val * val);
    if ((i & 31) == 0) part[i >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int j = 0; j < hd / 32; ++j) tot += part[j];
    const float nv = val * rsqrtf(tot / (float)hd + eps) * (is_q ? q_norm[i] : k_norm[i]);
    buf[i] = nv;
    __syncthreads();
    // NEOX: pairs (j, j + hd/2), angle pos * base^(-2j/hd); the angle and its
    // sine/cosine in double (angles reach thousands of radians)
    const int half = hd / 2;
    const int j = i < half ? i : i - half;
    const double th = (double)pos * pow((double)rope_base, -2.0 * (double)j / (double)hd);
    double sn, cs;
    sincos(th, &sn, &cs);
    const float a = buf[j], b = buf[j + half];
    const float rot = i < half ? (float)((double)a * cs - (double)b * sn)
                               : (float)((double)b * cs + (double)a * sn);
    if (is_q) {
        q[(size_t)head * hd + i] = rot;
    } else {
        k_cache[((size_t)kvh * max_ctx + pos) * hd + i] = __float2half_rn(rot);
        v_cache[((size_t)kvh * max_ctx + pos) * hd + i] = __float2half_rn(v[(size_t)kvh * hd + i]);
    }
}

constexpr int ATT_CHUNK = 128;        // positions per split
constexpr int ATT_THREADS = 256;

// Split-K (flash-decoding) GQA attention: block (kv head, chunk) handles the
// `group` q heads of that kv head over positions [c*CH, min((c+1)*CH, pos+1)).
// Writes per (q head, chunk): running max, sum of exp, unnormalised acc[hd].
__global__ void __launch_bounds__(ATT_THREADS) attn_partial(
    const float* __restrict__ q, const __half* __restrict__ k_cache,
    const __half* __restrict__ v_cache, int pos, int hd, int nq, int nkv, int max_ctx, int nsplit,
    float* __restrict__ part) {
    extern __shared__ float sm[];
    const int kvh = blockIdx.x, c = blockIdx.y;
    const int group = nq / nkv;
    const int p0 = c * ATT_CHUNK, p1 = min(p0 + ATT_CHUNK, pos + 1);
    const int np = p1 - p0;
    float* qs = sm;                        // group * hd
    float* sc = qs + group * hd;           // group * CHUNK
    const float scale = rsqrtf((float)hd);
    for (int i = threadIdx.x; i < group * hd; i += blockDim.x)
        qs[i] = q[(size_t)(kvh * group) * hd + i];
    __syncthreads();
    const __half* K = k_cache + ((size_t)kvh * max_ctx + p0) * hd;
    const __half* V = v_cache + ((size_t)kvh * max_ctx + p0) * hd;
    for (int i = threadIdx.x; i < group * ATT_CHUNK; i += blockDim.x) {
        const int g = i / ATT_CHUNK, pp = i % ATT_CHUNK;
        float s = -INFINITY;
        if (pp < np) {
            const __half2* kr = reinterpret_cast<const __half2*>(K + (size_t)pp * hd);
            const float* qg = qs + g * hd;
            float a = 0.f;
            for (int d = 0; d < hd / 2; ++d) {
                const float2 kv = __half22float2(kr[d]);
                a = fmaf(qg[2 * d], kv.x, a);
                a = fmaf(qg[2 * d + 1], kv.y, a);
            }
            s = a * scale;
        }
        sc[i] = s;
    }
    __syncthreads();
    // per q head (one warp each, warps loop over heads): max and sum of exp
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    __shared__ float mx_s[32], sum_s[32];
    for (int g = warp; g < group; g += nw) {
        float m = -INFINITY;
        for (int pp = lane; pp < np; pp += 32) m = fmaxf(m, sc[g * ATT_CHUNK + pp]);
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float l = 0.f;
        for (int pp = lane; pp < np; pp += 32) {
            const float e = expf(sc[g * ATT_CHUNK + pp] - m);
            sc[g * ATT_CHUNK + pp] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) { mx_s[g] = m; sum_s[g] = l; }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < group * hd; i += blockDim.x) {
        const int g = i / hd, d = i % hd;
        float a = 0.f;
        for (int pp = 0; pp < np; ++pp)
            a = fmaf(sc[g * ATT_CHUNK + pp], __half2float(V[(size_t)pp * hd + d]), a);
        float* o = part + ((size_t)(kvh * group + g) * nsplit + c) * (hd + 2);
        o[2 + d] = a;
        if (d == 0) { o[0] = mx_s[g]; o[1] = sum_s[g]; }
    }
}

// merge the splits of one q head (block per q head, hd threads)
__global__ void attn_merge(const float* __restrict__ part, int nsplit, int nvalid, int hd,
                           float* __restrict__ out) {
    const int h = blockIdx.x, d = threadIdx.x;
    const float* ph = part + (size_t)h * nsplit * (hd + 2);
    float m = -INFINITY;
    for (int c = 0; c < nvalid; ++c) m = fmaxf(m, ph[(size_t)c * (hd + 2)]);
    float l = 0.f, a = 0.f;
    for (int c = 0; c < nvalid; ++c) {
        const float* pc = ph + (size_t)c * (hd + 2);
        const float w = expf(pc[0] - m);
        l = fmaf(w, pc[1], l);
        a = fmaf(w, pc[2 + d], a);
    }
    out[(size_t)h * hd + d] = a / l;
}

}  // namespace

cudaError_t launch_rmsnorm(const float* h, const float* w, float eps, int n, float* out,
                           cudaStream_t st) {
    rmsnorm_kernel<<<1, 512, 0, st>>>(h, w, eps, n, out);
    return cudaGetLastError();
}

cudaError_t launch_attention_block(const AttnShape& a, const LayerAttn& L, const float* h,
                                   float* xs, float* q, float* kv, float* att, float* part,
                                   float* h_out, cudaStream_t st) {
    const int qd = a.nq * a.hd, kvd = a.nkv * a.hd;
    cudaError_t e;
    // B1: x = RMSNorm(h) * attn_norm
    rmsnorm_kernel<<<1, 512, 0, st>>>(h, L.attn_norm, a.eps, a.H, xs);
    // B2: q, k, v = Wq x, Wk x, Wv x  (no bias)
    GemvArgs g{};
    g.seg[0] = GemvSeg{L.wq, q, nullptr, qd};
    g.seg[1] = GemvSeg{L.wk, kv, nullptr, kvd};
    g.seg[2] = GemvSeg{L.wv, kv + kvd, nullptr, kvd};
    g.nseg = 3;
    g.cols = a.H;
    g.x = xs;
    const size_t gsm = sizeof(float) * (a.H + a.H / 16);
    q4k_gemv<<<(qd + 2 * kvd + GV_ROWS - 1) / GV_ROWS, 256, gsm, st>>>(g);
    // B3-B5: per-head Q/K RMSNorm, NEOX RoPE, fp16 KV append at pos
    qk_norm_rope_append<<<a.nq + a.nkv, a.hd, sizeof(float) * (a.hd + 32), st>>>(
        q, kv, kv + kvd, L.q_norm, L.k_norm, a.eps, a.pos, a.rope_base, a.hd, a.nq, a.nkv,
        a.max_ctx, L.k_cache, L.v_cache);
    // B6: GQA attention over positions 0..pos
    const int nsplit = (a.max_ctx + ATT_CHUNK - 1) / ATT_CHUNK;
    const int nvalid = a.pos / ATT_CHUNK + 1;
    const int group = a.nq / a.nkv;
    dim3 ga(a.nkv, nvalid);
    attn_partial<<<ga, ATT_THREADS, sizeof(float) * group * (a.hd + ATT_CHUNK), st>>>(
        q, L.k_cache, L.v_cache, a.pos, a.hd, a.nq, a.nkv, a.max_ctx, nsplit, part);
    attn_merge<<<a.nq, a.hd, 0, st>>>(part, nsplit, nvalid, a.hd, att);
    // B7: h_out = h + Wo att
    GemvArgs go{};
    go.seg[0] = GemvSeg{L.wo, h_out, h, a.H};
    go.nseg = 1;
    go.cols = qd;
    go.x = att;
    q4k_gemv<<<(a.H + GV_ROWS - 1) / GV_ROWS, 256, sizeof(float) * (qd + qd / 16), st>>>(go);
    e = cudaGetLastError();
    return e;
}

int attn_splits(int max_ctx) { return (max_ctx + ATT_CHUNK - 1) / ATT_CHUNK; }

}  // namespace qmoe
