// prefill_layer.cu -- one qwen3moe decoder layer for T tokens at once (batched
// prefill), instead of T decode steps.
//
// The aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path"
// (later gap list, "Prefill is token-by-token": 1,685 prompt tokens in 21.9 s
// on an RTX 4090) names a batched prefill as the fix.  The layer computed is
// the decode layer of the same issue ("Fix Applied" of "Qwen3 GPU inference
// produces garbage output", per-head Q/K RMSNorm of the aprender PR "apply
// per-head Q/K RMSNorm in forward_qwen3_moe", NEOX RoPE of the SharpInference
// issue "Forward-pass divergence on Qwen3-Coder 30B-A3B") applied to T tokens
// at positions pos0 .. pos0+T-1 with causal attention: token t sees the cache
// positions 0 .. pos0-1 as stored and the batch's tokens 0 .. t.  Within one
// layer a token's K and V depend only on its own input, so this equals the
// layer applied token by token.
//
// Launch sequence (all on the context's stream):
//   rmsnorm_rows_f16     x = RMSNorm(h) * attn_norm as fp16 rows (the MMA operand)
//   dense Q4_K GEMM x3   q, k, v = Wq x, Wk x, Wv x (tcgen05, prefill_umma.cu)
//   qk_norm_rope_append  per-head Q/K RMSNorm, NEOX RoPE at pos0 + t; k, v -> fp16
//                        cache slots pos0 + t
//   prefill_attention    causal GQA attention over cache + batch -> fp16 rows
//   dense Q4_K GEMM      h = h + Wo att (in place)
//   rmsnorm_rows_f32     x2 = RMSNorm(h) * ffn_norm
//   MoE FFN              h = h + MoE(x2) (the tensor-core prefill path for T > 8)
#include <cuda_fp16.h>
#include <math.h>

#include "kquant.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

constexpr int NR_THREADS = 256;

__device__ __forceinline__ float block_sum_256(float v, float* red) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < NR_THREADS / 32; ++w) t += red[w];
    __syncthreads();
    return t;
}

// one block per token row: out = RMSNorm(h) * w, as fp16 (f16 = 1) or fp32
template <int F16>
__global__ void __launch_bounds__(NR_THREADS) rmsnorm_rows(const float* __restrict__ h,
                                                           const float* __restrict__ w, float eps,
                                                           int H, void* __restrict__ out) {
    __shared__ float red[NR_THREADS / 32];
    const float* row = h + (size_t)blockIdx.x * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += NR_THREADS) ss = fmaf(row[i], row[i], ss);
    const float r = rsqrtf(block_sum_256(ss, red) / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += NR_THREADS) {
        const float v = row[i] * r * w[i];
        if (F16) reinterpret_cast<__half*>(out)[(size_t)blockIdx.x * H + i] = __float2half_rn(v);
        else reinterpret_cast<float*>(out)[(size_t)blockIdx.x * H + i] = v;
    }
}

// cos/sin of the NEOX RoPE angle of pair j at position pos: the angle
// pos * base^(-2j/hd) is formed and reduced to [-pi, pi] in double (inv_freq
// from the host, double), cos and sin taken in float
__device__ __forceinline__ float2 rope_cs(const double* __restrict__ inv_freq, int j, int pos) {
    constexpr double TWO_PI = 6.283185307179586476925286766559;
    const double th = (double)pos * inv_freq[j];
    const double red = fma(-rint(th * (1.0 / TWO_PI)), TWO_PI, th);
    float sn, c;
    sincosf((float)red, &sn, &c);
    return make_float2(c, sn);
}

// one warp per (token, head): heads 0..nq-1 are q heads (RMSNorm q_norm, RoPE,
// fp32 out), heads nq..nq+nkv-1 are kv heads (k: RMSNorm k_norm, RoPE, fp16 into
// cache slot pos0 + t; v: fp16 into the same slot).  Lane owns dims lane + 32 i,
// so the rotated pairs (d, d + hd/2) sit in the same lane.
__global__ void __launch_bounds__(128) qk_norm_rope_append(
    const float* __restrict__ qkv, int nq, int nkv, int hd, const float* __restrict__ q_norm,
    const float* __restrict__ k_norm, float eps, const double* __restrict__ inv_freq, int pos0,
    int max_ctx, float* __restrict__ qr, __half* __restrict__ k_cache, __half* __restrict__ v_cache,
    int T) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x, hh = blockIdx.y * 4 + warp;
    if (t >= T || hh >= nq + nkv) return;
    const int qd = nq * hd, kvd = nkv * hd, n = hd / 32;
    const float* row = qkv + (size_t)t * (qd + 2 * kvd);
    const bool isq = hh < nq;
    const int g = hh - nq;
    const float* src = isq ? row + hh * hd : row + qd + g * hd;
    const float* nw = isq ? q_norm : k_norm;
    float v[8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = i < n ? src[lane + 32 * i] : 0.f;
        ss = fmaf(v[i], v[i], ss);
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)hd + eps);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < n) v[i] = v[i] * r * nw[lane + 32 * i];
    const int pos = pos0 + t;
    float o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (i < n / 2) {
            const float2 cs = rope_cs(inv_freq, lane + 32 * i, pos);
            const float a = v[i], b = v[i + n / 2];
            o[i] = a * cs.x - b * cs.y;
            o[i + n / 2] = b * cs.x + a * cs.y;
        }
    }
    if (isq) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < n) qr[(size_t)t * qd + hh * hd + lane + 32 * i] = o[i];
    } else {
        __half* kd = k_cache + ((size_t)g * max_ctx + pos) * hd;
        __half* vd = v_cache + ((size_t)g * max_ctx + pos) * hd;
        const float* vs = row + qd + kvd + g * hd;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < n) {
                kd[lane + 32 * i] = __float2half_rn(o[i]);
                vd[lane + 32 * i] = __float2half_rn(vs[lane + 32 * i]);
            }
        }
    }
}

// Causal GQA attention of T query tokens over the fp16 cache (positions
// 0 .. pos0 + t for token t).  Block (kv head g, tokens [QT*b, QT*b + QT)): the
// group = nq/nkv q heads of those tokens (QT*group query vectors) against key
// chunks of 64 positions staged in shared memory; warp w owns query vectors
// w, w + 8, ...; scores by lanes over keys, online softmax, the output as fp16
// rows att[t][h*hd + d] (the O projection's MMA operand).
constexpr int PA_THREADS = 256;
constexpr int PA_CHUNK = 64;
constexpr int PA_QT = 4;

template <int MAXV>
__global__ void __launch_bounds__(PA_THREADS) prefill_attention(
    const float* __restrict__ qr, const __half* __restrict__ k_cache,
    const __half* __restrict__ v_cache, int nq, int nkv, int hd, int pos0, int max_ctx, int T,
    __half* __restrict__ att) {
    extern __shared__ __align__(16) float sm[];
    const int g = blockIdx.x, t0 = blockIdx.y * PA_QT;
    const int group = nq / nkv, nvec = PA_QT * group;         // query vectors of the block
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = PA_THREADS / 32;
    const int qd = nq * hd, n = hd / 32;
    const int kw = hd / 2 + 1;                                 // padded K row, 32-bit words
    float* qs = sm;                                            // nvec * hd
    uint32_t* ks = reinterpret_cast<uint32_t*>(qs + nvec * hd); // CHUNK * kw
    __half* vs = reinterpret_cast<__half*>(ks + ((PA_CHUNK * kw + 3) & ~3));   // CHUNK * hd
    // query vectors: v = (token t0 + v / group, head g*group + v % group)
    for (int i = threadIdx.x; i < nvec * hd; i += PA_THREADS) {
        const int vq = i / hd, d = i - vq * hd;
        const int t = t0 + vq / group, h = g * group + vq % group;
        qs[i] = t < T ? qr[(size_t)t * qd + h * hd + d] : 0.f;
    }
    const int tlast = min(t0 + PA_QT, T) - 1;
    const int kend = pos0 + tlast + 1;                         // keys this block needs
    const float scale = rsqrtf((float)hd);
    // per owned query vector (MAXV = ceil(nvec / 8) at most): running max, sum,
    // accumulator (lane owns dims lane + 32 i)
    float m[MAXV], l[MAXV], acc[MAXV][8];
#pragma unroll
    for (int a = 0; a < MAXV; ++a) {
        m[a] = -INFINITY;
        l[a] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[a][i] = 0.f;
    }
    const uint4* K = reinterpret_cast<const uint4*>(k_cache + (size_t)g * max_ctx * hd);
    const uint4* V = reinterpret_cast<const uint4*>(v_cache + (size_t)g * max_ctx * hd);
    const int vpr = hd / 8;
    for (int c0 = 0; c0 < kend; c0 += PA_CHUNK) {
        const int np = min(PA_CHUNK, kend - c0);
        __syncthreads();                                       // previous chunk consumed
        for (int i = threadIdx.x; i < np * vpr; i += PA_THREADS) {
            const int row = i / vpr, cc = i - row * vpr;
            const uint4 kq = K[(size_t)(c0 + row) * vpr + cc];
            uint32_t* kd = ks + row * kw + 4 * cc;
            kd[0] = kq.x; kd[1] = kq.y; kd[2] = kq.z; kd[3] = kq.w;
            reinterpret_cast<uint4*>(vs)[i] = V[(size_t)(c0 + row) * vpr + cc];
        }
        __syncthreads();
#pragma unroll
        for (int a = 0; a < MAXV; ++a) {
            const int vq = warp + nw * a;
            if (vq >= nvec) continue;
            const int t = t0 + vq / group;
            if (t >= T) continue;
            const int kmax = pos0 + t;                         // last key this token sees
            const float* q = qs + vq * hd;
            // scores of keys c0 + lane and c0 + lane + 32
            float s[2];
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                const int kk = lane + 32 * hk;
                float dot = 0.f;
                if (kk < np && c0 + kk <= kmax) {
                    const uint32_t* kr = ks + kk * kw;
                    for (int d2 = 0; d2 < hd / 2; ++d2) {
                        const float2 kv2 = __half22float2(*reinterpret_cast<const __half2*>(kr + d2));
                        dot = fmaf(q[2 * d2], kv2.x, fmaf(q[2 * d2 + 1], kv2.y, dot));
                    }
                    s[hk] = dot * scale;
                } else {
                    s[hk] = -INFINITY;
                }
            }
            float cmax = fmaxf(s[0], s[1]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
            if (cmax == -INFINITY) continue;                   // no visible key in this chunk
            const float mnew = fmaxf(m[a], cmax);
            const float corr = expf(m[a] - mnew);
            const float p0 = expf(s[0] - mnew), p1 = expf(s[1] - mnew);
            l[a] = l[a] * corr + warp_sum(p0 + p1);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[a][i] *= corr;
            m[a] = mnew;
            // acc[d] += sum_k p_k v_k[d]: broadcast each key's weight from its lane
            for (int kk = 0; kk < np; ++kk) {
                const float pk = __shfl_sync(0xffffffffu, kk < 32 ? p0 : p1, kk & 31);
                if (pk != 0.f) {
                    const __half* vr = vs + (size_t)kk * hd;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (i < n) acc[a][i] = fmaf(pk, __half2float(vr[lane + 32 * i]), acc[a][i]);
                }
            }
        }
    }
#pragma unroll
    for (int a = 0; a < MAXV; ++a) {
        const int vq = warp + nw * a;
        if (vq >= nvec) continue;
        const int t = t0 + vq / group, h = g * group + vq % group;
        if (t >= T) continue;
        const float inv = 1.f / l[a];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < n) att[(size_t)t * qd + h * hd + lane + 32 * i] = __float2half_rn(acc[a][i] * inv);
    }
}

size_t pa_smem(int group, int hd) {
    const int kw = hd / 2 + 1;
    return sizeof(float) * (size_t)PA_QT * group * hd + 4 * (size_t)((PA_CHUNK * kw + 3) & ~3) +
           sizeof(__half) * (size_t)PA_CHUNK * hd;
}

}  // namespace

size_t prefill_layer_scratch_bytes(int T, int H, int nq, int nkv, int hd) {
    const size_t qd = (size_t)nq * hd, kvd = (size_t)nkv * hd;
    auto a = [](size_t v) { return (v + 255) / 256 * 256; };
    const size_t xin = (size_t)T * (H > (int)qd ? H : qd);
    return a(4 * T * (qd + 2 * kvd)) + a(4 * T * qd) + a(2 * xin) + a(2 * T * qd) + a(4 * (size_t)T * H);
}

bool prefill_layer_supported(int H, int nq, int nkv, int hd) {
    const int qd = nq * hd, kvd = nkv * hd;
    if (H % 128 || qd % 128 || kvd % 128 || H % QK || qd % QK) return false;   // dense GEMM tiles
    if (hd % 64 || hd > 256 || nkv < 1 || nq % nkv || nq / nkv > 8) return false;
    return pa_smem(nq / nkv, hd) <= 200 * 1024;
}

cudaError_t prefill_layer_prepare() {
    cudaError_t e = cudaFuncSetAttribute(prefill_attention<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_attention<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_attention<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    return e;
}

cudaError_t launch_prefill_layer_attn(const PrefillLayerArgs& a, cudaStream_t st) {
    const int qd = a.nq * a.hd, kvd = a.nkv * a.hd, T = a.T;
    const size_t xin_cols = a.H > qd ? a.H : qd;
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    unsigned char* b = static_cast<unsigned char*>(a.scratch);
    float* qkv = reinterpret_cast<float*>(b);
    b += al(4 * (size_t)T * (qd + 2 * kvd));
    float* qr = reinterpret_cast<float*>(b);
    b += al(4 * (size_t)T * qd);
    __half* x16 = reinterpret_cast<__half*>(b);
    b += al(2 * (size_t)T * xin_cols);
    __half* att16 = reinterpret_cast<__half*>(b);
    b += al(2 * (size_t)T * qd);
    float* x2 = reinterpret_cast<float*>(b);
    // B1: x = RMSNorm(h) * attn_norm, fp16 rows
    rmsnorm_rows<1><<<T, NR_THREADS, 0, st>>>(a.hidden, a.attn_norm, a.eps, a.H, x16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // B2: q, k, v rows of every token, side by side in one [T][qd + 2 kvd] buffer
    const int ld = qd + 2 * kvd;
    e = launch_dense_q4k_gemm(a.wq, qd, a.H, x16, T, qkv, ld, 0, nullptr, st);
    if (e == cudaSuccess) e = launch_dense_q4k_gemm(a.wk, kvd, a.H, x16, T, qkv, ld, qd, nullptr, st);
    if (e == cudaSuccess) e = launch_dense_q4k_gemm(a.wv, kvd, a.H, x16, T, qkv, ld, qd + kvd, nullptr, st);
    if (e != cudaSuccess) return e;
    // B3-B5: per-head Q/K RMSNorm, NEOX RoPE, fp16 KV append at pos0 + t
    qk_norm_rope_append<<<dim3(T, (a.nq + a.nkv + 3) / 4), 128, 0, st>>>(
        qkv, a.nq, a.nkv, a.hd, a.q_norm, a.k_norm, a.eps, a.inv_freq, a.pos0, a.max_ctx, qr, a.k_cache,
        a.v_cache, T);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // B6: causal GQA attention over cache + batch
    const int group = a.nq / a.nkv;
    const int mv = (PA_QT * group + PA_THREADS / 32 - 1) / (PA_THREADS / 32);   // vectors per warp
    const dim3 ga(a.nkv, (T + PA_QT - 1) / PA_QT);
    const size_t sm = pa_smem(group, a.hd);
    if (mv <= 1)
        prefill_attention<1><<<ga, PA_THREADS, sm, st>>>(qr, a.k_cache, a.v_cache, a.nq, a.nkv, a.hd, a.pos0, a.max_ctx, T, att16);
    else if (mv <= 2)
        prefill_attention<2><<<ga, PA_THREADS, sm, st>>>(qr, a.k_cache, a.v_cache, a.nq, a.nkv, a.hd, a.pos0, a.max_ctx, T, att16);
    else
        prefill_attention<4><<<ga, PA_THREADS, sm, st>>>(qr, a.k_cache, a.v_cache, a.nq, a.nkv, a.hd, a.pos0, a.max_ctx, T, att16);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // B7: h = h + Wo att, in place (every element read and written by one thread)
    e = launch_dense_q4k_gemm(a.wo, a.H, qd, att16, T, a.hidden, a.H, 0, a.hidden, st);
    if (e != cudaSuccess) return e;
    // B8: x2 = RMSNorm(h) * ffn_norm (the MoE input; h stays the residual)
    rmsnorm_rows<0><<<T, NR_THREADS, 0, st>>>(a.hidden, a.ffn_norm, a.eps, a.H, x2);
    return cudaGetLastError();
}

float* prefill_layer_x2(void* scratch, int T, int H, int nq, int nkv, int hd) {
    const size_t qd = (size_t)nq * hd, kvd = (size_t)nkv * hd;
    const size_t xin_cols = (size_t)H > qd ? (size_t)H : qd;
    auto al = [](size_t v) { return (v + 255) / 256 * 256; };
    unsigned char* b = static_cast<unsigned char*>(scratch);
    b += al(4 * (size_t)T * (qd + 2 * kvd)) + al(4 * (size_t)T * qd) + al(2 * (size_t)T * xin_cols) +
         al(2 * (size_t)T * qd);
    return reinterpret_cast<float*>(b);
}

}  // namespace qmoe
