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
#include "pdl.cuh"
#include "qmoe_internal.h"
#include "umma.cuh"

namespace qmoe {

// 2-D fp16 tensor map, box 64 columns x box_rows rows, 128B swizzle (prefill_umma.cu)
bool tensor_map_half(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows);

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
    pdl_wait();
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

// the O projection split over K in two planes: h = h + p0 + p1 (in place),
// then out = RMSNorm(h) * w (fp32), one block per token row
__global__ void __launch_bounds__(NR_THREADS) residual_rmsnorm_rows(float* __restrict__ h,
                                                                    const float* __restrict__ p0,
                                                                    const float* __restrict__ p1,
                                                                    const float* __restrict__ w, float eps,
                                                                    int H, float* __restrict__ out) {
    pdl_wait();
    __shared__ float red[NR_THREADS / 32];
    const size_t base = (size_t)blockIdx.x * H;
    float ss = 0.f;
    for (int i = threadIdx.x; i < H; i += NR_THREADS) {
        const float v = (h[base + i] + p0[base + i]) + p1[base + i];
        h[base + i] = v;
        ss = fmaf(v, v, ss);
    }
    const float r = rsqrtf(block_sum_256(ss, red) / (float)H + eps);
    for (int i = threadIdx.x; i < H; i += NR_THREADS) out[base + i] = h[base + i] * r * w[i];
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

// cos/sin of every (token, pair) of the batch: cs[t][j] for position pos0 + t
__global__ void rope_table_rows(const double* __restrict__ inv_freq, int half, int pos0, int T,
                                float2* __restrict__ cs) {
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T * half) return;
    const int t = i / half, j = i - t * half;
    cs[i] = rope_cs(inv_freq, j, pos0 + t);
}

// one warp per (token, head): heads 0..nq-1 are q heads (RMSNorm q_norm, RoPE,
// fp32 out), heads nq..nq+nkv-1 are kv heads (k: RMSNorm k_norm, RoPE, fp16 into
// cache slot pos0 + t; v: fp16 into the same slot).  Lane owns dims lane + 32 i,
// so the rotated pairs (d, d + hd/2) sit in the same lane.
__global__ void __launch_bounds__(128) qk_norm_rope_append(
    const float* __restrict__ qkv, int nq, int nkv, int hd, const float* __restrict__ q_norm,
    const float* __restrict__ k_norm, float eps, const float2* __restrict__ rcs, int pos0,
    int max_ctx, float* __restrict__ qr, __half* __restrict__ qh, __half* __restrict__ k_cache,
    __half* __restrict__ v_cache, int T) {
    pdl_wait();
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
            const float2 cs = rcs[(size_t)t * (hd / 2) + lane + 32 * i];
            const float a = v[i], b = v[i + n / 2];
            o[i] = a * cs.x - b * cs.y;
            o[i + n / 2] = b * cs.x + a * cs.y;
        }
    }
    if (isq && qh) {
        // fp16 rows for the tensor-core attention: [kv group][token][head of
        // the group][hd], so a block's (token, head) rows are contiguous
        const int group = nq / nkv, gq = hh / group, hq = hh - gq * group;
        __half* dq = qh + (((size_t)gq * T + t) * group + hq) * hd;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < n) dq[lane + 32 * i] = __float2half_rn(o[i]);
    } else if (isq) {
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
    pdl_wait();
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

// Causal GQA attention on the tensor cores.  CTA = (kv head g, 128 / group
// tokens): its 128 query rows (token, head of the group) against key chunks of
// 128 positions, two passes over the chunks.  Pass 1: S = Q K^T (tcgen05, fp32
// in TMEM); row r's scores are read by two threads (columns 0-63 and 64-127,
// TMEM lane r), each keeping the running maximum and sum of exponentials of its
// visible scores; the two halves are merged once, after the pass.  Pass 2: S
// again, P = exp(s - max) / sum as fp16 into shared memory (128B-swizzled,
// K-major: each thread's half of a row is one 64-key k-block), V^T of the chunk
// staged by the threads in the same layout, O += P V^T in TMEM.  Two passes
// instead of rescaling O on every new maximum keep the accumulator in TMEM
// untouched until the end.  P reuses the K buffer (the S MMA that read K has
// completed before P is written), so two CTAs fit an SM.  Epilogue: O rows ->
// fp16 att.  Masking: key p is visible to the row of token t when p <= pos0 + t;
// keys past the block's last visible key are not read (their V^T columns are
// zero).  One thread (tid 0) issues the TMA copies and MMAs.
constexpr int PT_THREADS = 256;
constexpr int PT_KC = 128;                                 // keys per chunk
constexpr int PT_HC = PT_KC / 2;                           // keys per thread (one half of a row)

__device__ __forceinline__ uint32_t h2_pack(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(PT_THREADS, 2) prefill_attention_tc(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __half* __restrict__ v_cache, int nq, int nkv, int hd, int pos0, int max_ctx, int T,
    __half* __restrict__ att, int* __restrict__ status) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const int group = nq / nkv, QB = 128 / group;          // tokens per CTA
    const int g = blockIdx.x, t0 = blockIdx.y * QB;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int nkb = hd / 64;                               // 64-wide k-blocks of hd
    uint8_t* sQ = sm;                                      // nkb x 16 KB (128 rows)
    uint8_t* sK = sQ + nkb * 16384;                        // max(nkb, 2) x 16 KB: K, then P
    uint8_t* sP = sK;                                      // 2 x 16 KB (128 rows x 128 keys)
    uint8_t* sV = sK + (nkb > 2 ? nkb : 2) * 16384;        // 2 x (hd x 128 B): V^T, keys = K
    uint64_t* bars = reinterpret_cast<uint64_t*>(sV + 2 * hd * 128);
    float* xch = reinterpret_cast<float*>(bars + 4);       // [2][128] half-row statistics
    uint32_t* tslot = reinterpret_cast<uint32_t*>(xch + 512);
    uint64_t* tma_bar = bars;
    uint64_t* mma_bar = bars + 1;
    uint64_t* q_bar = bars + 2;
    const int t_last = min(t0 + QB, T) - 1;                // last token of the block
    const int kend = pos0 + t_last + 1;                    // keys the block sees
    const int nchunks = (kend + PT_KC - 1) / PT_KC;
    // this thread's query row and half of the chunk's columns
    const int row = tid & 127, hf = tid >> 7;
    const int tl = row / group, t = t0 + tl;
    const int kmax = pos0 + t;                             // last key of this row
    const float sl2 = rsqrtf((float)hd) * 1.4426950408889634f;   // scale * log2(e)

    if (tid == 0) {
        mbar_init(tma_bar, 1);
        mbar_init(mma_bar, 1);
        mbar_init(q_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tS = tmem, tO = tmem + 128;             // columns: S [0,128), O [128, 128 + hd)
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    uint32_t tpar = 0, mpar = 0;
    bool ok = true;

    // Q rows of the block, one TMA box per 64-wide k-block
    if (tid == 0) {
        mbar_arrive_expect_tx(q_bar, (uint32_t)(nkb * 16384));
        for (int kb = 0; kb < nkb; ++kb)
            tma_load_2d(sQ + kb * 16384, &tm_q, kb * 64, (g * T + t0) * group, q_bar);
        if (!mbar_wait(q_bar, 0)) ok = false;
    }
    // No thread leaves an iteration early: a failed wait only clears ok, and
    // every iteration starts with a block-wide vote, so all threads stop at the
    // same point and every barrier is reached by all of them.
    float m = -INFINITY, l = 0.f;
    for (int pass = 0; pass < 2; ++pass) {
        bool stop = false;
        if (pass == 1) {
            // merge the two half-row statistics of each row
            xch[hf * 128 + row] = m;
            xch[256 + hf * 128 + row] = l;
            __syncthreads();
            const float mo = xch[(hf ^ 1) * 128 + row], lo = xch[256 + (hf ^ 1) * 128 + row];
            const float mn = fmaxf(m, mo);
            l = (m > -INFINITY ? l * exp2f(m - mn) : 0.f) + (mo > -INFINITY ? lo * exp2f(mo - mn) : 0.f);
            m = mn;
        }
        for (int c = 0; c < nchunks; ++c) {
            if (!__syncthreads_and(ok)) {
                ok = false;
                stop = true;
                break;
            }
            const int k0 = c * PT_KC;
            if (tid == 0) {
                // K chunk (the previous chunk's MMAs have completed: every thread
                // waited for them before the vote that starts the iteration)
                mbar_arrive_expect_tx(tma_bar, (uint32_t)(nkb * 16384));
                for (int kb = 0; kb < nkb; ++kb)
                    tma_load_2d(sK + kb * 16384, &tm_k, kb * 64, g * max_ctx + k0, tma_bar);
                if (!mbar_wait(tma_bar, tpar)) ok = false;
                tpar ^= 1u;
                if (ok) {
                    tc_fence_after();
                    const uint32_t idesc = umma_idesc_f16(128, PT_KC);
                    for (int ks = 0; ks < hd / 16; ++ks) {
                        const uint64_t ad = umma_sdesc(smem_u32(sQ + (ks >> 2) * 16384)) + (uint64_t)(2 * (ks & 3));
                        const uint64_t bd = umma_sdesc(smem_u32(sK + (ks >> 2) * 16384)) + (uint64_t)(2 * (ks & 3));
                        umma_f16(tS, ad, bd, idesc, ks != 0);
                    }
                    umma_commit(mma_bar);
                }
            }
            if (pass == 1) {
                // V^T of the chunk: thread -> key pair (2 i, 2 i + 1), a quarter of hd
                const int i = tid & 63, dq = tid >> 6, kk = 2 * i;
                const int qd4 = hd / 4;
                uint8_t* reg = sV + (kk >> 6) * (hd * 128);
                for (int d0 = dq * qd4; d0 < dq * qd4 + qd4; d0 += 8) {
                    uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
                    if (k0 + kk < kend)
                        a = *reinterpret_cast<const uint4*>(v_cache + ((size_t)g * max_ctx + k0 + kk) * hd + d0);
                    if (k0 + kk + 1 < kend)
                        b = *reinterpret_cast<const uint4*>(v_cache + ((size_t)g * max_ctx + k0 + kk + 1) * hd + d0);
                    const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // halves d0 + 2q (low) and d0 + 2q + 1 (high) of keys kk, kk + 1
                        const uint32_t lo = __byte_perm(aw[q], bw[q], 0x5410);
                        const uint32_t hi = __byte_perm(aw[q], bw[q], 0x7632);
                        *reinterpret_cast<uint32_t*>(reg + sw128_offset(d0 + 2 * q, kk & 63)) = lo;
                        *reinterpret_cast<uint32_t*>(reg + sw128_offset(d0 + 2 * q + 1, kk & 63)) = hi;
                    }
                }
            }
            if (!mbar_wait(mma_bar, mpar)) ok = false;
            mpar ^= 1u;
            tc_fence_after();
            // this thread's 64 scores of its row, 16 at a time
            const int kb0 = k0 + PT_HC * hf;
            float cm = -INFINITY;
            float sv[PT_HC];
#pragma unroll
            for (int j0 = 0; j0 < PT_HC; j0 += 16) {
                float v16[16];
                tmem_ld16(tS + lane_off + (uint32_t)(PT_HC * hf + j0), v16);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float s2 = kb0 + j0 + j <= kmax ? v16[j] * sl2 : -INFINITY;
                    sv[j0 + j] = s2;
                    cm = fmaxf(cm, s2);
                }
            }
            if (pass == 0) {
                if (cm > -INFINITY) {
                    const float mn = fmaxf(m, cm);
                    float sum = 0.f;
#pragma unroll
                    for (int j = 0; j < PT_HC; ++j) sum += exp2f(sv[j] - mn);
                    l = l * exp2f(m - mn) + sum;
                    m = mn;
                }
            } else {
                // this half of the P row -> fp16, one 64-key k-block (128B-swizzled K-major)
                const float inv = 1.f / l;
                uint8_t* preg = sP + hf * 16384;
#pragma unroll
                for (int j0 = 0; j0 < PT_HC; j0 += 8) {
                    uint4 w;
                    w.x = h2_pack(exp2f(sv[j0 + 0] - m) * inv, exp2f(sv[j0 + 1] - m) * inv);
                    w.y = h2_pack(exp2f(sv[j0 + 2] - m) * inv, exp2f(sv[j0 + 3] - m) * inv);
                    w.z = h2_pack(exp2f(sv[j0 + 4] - m) * inv, exp2f(sv[j0 + 5] - m) * inv);
                    w.w = h2_pack(exp2f(sv[j0 + 6] - m) * inv, exp2f(sv[j0 + 7] - m) * inv);
                    *reinterpret_cast<uint4*>(preg + sw128_offset(row, j0)) = w;
                }
                fence_proxy_async();
            }
            tc_fence_before();
            __syncthreads();
            if (pass == 1 && tid == 0 && ok) {
                // O += P V^T over the chunk's 128 keys
                tc_fence_after();
                const uint32_t idesc = umma_idesc_f16(128, hd);
                for (int ks = 0; ks < PT_KC / 16; ++ks) {
                    const uint64_t ad = umma_sdesc(smem_u32(sP + (ks >> 2) * 16384)) + (uint64_t)(2 * (ks & 3));
                    const uint64_t bd = umma_sdesc(smem_u32(sV + (ks >> 2) * (hd * 128))) + (uint64_t)(2 * (ks & 3));
                    umma_f16(tO, ad, bd, idesc, (c | ks) != 0);
                }
                umma_commit(mma_bar);
            }
            if (pass == 1) {
                // P (in the K buffer) and V^T are reused by the next chunk: wait for this chunk's MMAs
                if (!mbar_wait(mma_bar, mpar)) ok = false;
                mpar ^= 1u;
            }
        }
        if (stop) break;
    }
    ok = __syncthreads_and(ok) != 0;
    if (!ok && tid == 0) atomicExch(status, ST_TIMEOUT);
    if (ok) {
        tc_fence_after();
        // O row -> fp16 att[t][h * hd + d], h = g * group + (row % group); this
        // thread writes its half of hd
        const int h = g * group + (row - tl * group);
        for (int d0 = hf * (hd / 2); d0 < hf * (hd / 2) + hd / 2; d0 += 16) {
            float v16[16];
            tmem_ld16(tO + lane_off + (uint32_t)d0, v16);
            if (t <= t_last) {
                uint4 w0, w1;
                w0.x = h2_pack(v16[0], v16[1]);
                w0.y = h2_pack(v16[2], v16[3]);
                w0.z = h2_pack(v16[4], v16[5]);
                w0.w = h2_pack(v16[6], v16[7]);
                w1.x = h2_pack(v16[8], v16[9]);
                w1.y = h2_pack(v16[10], v16[11]);
                w1.z = h2_pack(v16[12], v16[13]);
                w1.w = h2_pack(v16[14], v16[15]);
                uint4* dst = reinterpret_cast<uint4*>(att + (size_t)t * nq * hd + (size_t)h * hd + d0);
                dst[0] = w0;
                dst[1] = w1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

size_t pt_smem(int hd) {
    const int nkb = hd / 64;
    return 1024 + (size_t)nkb * 16384 + (size_t)(nkb > 2 ? nkb : 2) * 16384 + 2 * (size_t)hd * 128 + 32 +
           sizeof(float) * 512 + 16;
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
    return a(4 * T * (qd + 2 * kvd)) + a(4 * T * qd) + a(2 * xin) + a(2 * T * qd) + a(4 * (size_t)T * H) +
           a(8 * (size_t)T * H) + a(sizeof(float2) * (size_t)T * (hd / 2));
}

bool prefill_layer_supported(int H, int nq, int nkv, int hd) {
    const int qd = nq * hd, kvd = nkv * hd;
    if (H % 128 || qd % 128 || kvd % 128 || H % QK || qd % QK) return false;   // dense GEMM tiles
    if (hd % 64 || hd > 256 || nkv < 1 || nq % nkv || nq / nkv > 8) return false;
    return pa_smem(nq / nkv, hd) <= 200 * 1024;
}

// the tensor-core attention serves query groups whose rows tile 128 evenly and
// head sizes of one or two 64-wide k-blocks
bool pt_supported(int group, int hd) {
    return (group == 1 || group == 2 || group == 4 || group == 8) && (hd == 64 || hd == 128);
}

cudaError_t prefill_layer_prepare() {
    cudaError_t e = cudaFuncSetAttribute(prefill_attention_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pt_smem(128));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_attention<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
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
    cudaError_t e = launch_pdl(rmsnorm_rows<1>, dim3(T), dim3(NR_THREADS), 0, st, a.hidden, a.attn_norm,
                               a.eps, a.H, x16);
    if (e != cudaSuccess) return e;
    // B2: q, k, v rows of every token, side by side in one [T][qd + 2 kvd]
    // buffer, the three projections in one launch
    const int ld = qd + 2 * kvd;
    {
        const DenseSeg segs[3] = {{a.wq, qd, 0}, {a.wk, kvd, qd}, {a.wv, kvd, qd + kvd}};
        e = launch_dense_q4k_gemm_multi(segs, 3, a.H, x16, T, qkv, ld, nullptr, 1, 0, st);
        if (e != cudaSuccess) return e;
    }
    // B3-B5: per-head Q/K RMSNorm, NEOX RoPE, fp16 KV append at pos0 + t (q as
    // fp16 rows grouped by kv head for the tensor-core attention, else fp32)
    const int group = a.nq / a.nkv;
    const bool tc = pt_supported(group, a.hd);
    __half* qh = tc ? reinterpret_cast<__half*>(qr) : nullptr;
    float2* rcs = reinterpret_cast<float2*>(reinterpret_cast<unsigned char*>(x2) + al(4 * (size_t)T * a.H) +
                                            al(8 * (size_t)T * a.H));
    e = launch_pdl(rope_table_rows, dim3((T * (a.hd / 2) + 255) / 256), dim3(256), 0, st, a.inv_freq,
                   a.hd / 2, a.pos0, T, rcs);
    if (e != cudaSuccess) return e;
    e = launch_pdl(qk_norm_rope_append, dim3(T, (a.nq + a.nkv + 3) / 4), dim3(128), 0, st, qkv, a.nq, a.nkv,
                   a.hd, a.q_norm, a.k_norm, a.eps, rcs, a.pos0, a.max_ctx, qr, qh, a.k_cache, a.v_cache, T);
    if (e != cudaSuccess) return e;
    // B6: causal GQA attention over cache + batch
    if (tc) {
        CUtensorMap tq, tk;
        if (!tensor_map_half(&tq, qh, (uint64_t)a.hd, (uint64_t)a.nkv * T * group, 128) ||
            !tensor_map_half(&tk, a.k_cache, (uint64_t)a.hd, (uint64_t)a.nkv * a.max_ctx, 128))
            return cudaErrorInvalidValue;
        const int QB = 128 / group;
        e = launch_pdl(prefill_attention_tc, dim3(a.nkv, (T + QB - 1) / QB), dim3(PT_THREADS), pt_smem(a.hd),
                       st, tq, tk, a.v_cache, a.nq, a.nkv, a.hd, a.pos0, a.max_ctx, T, att16, a.status);
    } else {
        // other shapes: the CUDA-core kernel
        const int mv = (PA_QT * group + PA_THREADS / 32 - 1) / (PA_THREADS / 32);   // vectors per warp
        const dim3 ga(a.nkv, (T + PA_QT - 1) / PA_QT);
        const size_t sm = pa_smem(group, a.hd);
        auto kern = mv <= 1 ? prefill_attention<1> : mv <= 2 ? prefill_attention<2> : prefill_attention<4>;
        e = launch_pdl(kern, ga, dim3(PA_THREADS), sm, st, qr, a.k_cache, a.v_cache, a.nq, a.nkv, a.hd,
                       a.pos0, a.max_ctx, T, att16);
    }
    if (e != cudaSuccess) return e;
    // B7 + B8: h = h + Wo att, x2 = RMSNorm(h) * ffn_norm (the MoE input; h
    // stays the residual).  With too few row x token tiles to fill the GPU the
    // O projection is split over K into two planes that the norm kernel adds.
    const DenseSeg so{a.wo, a.H, 0};
    if (2 * dense_q4k_items(a.H, T) <= device_sm_count() && (qd / QK) % 2 == 0) {
        float* part = x2 + (size_t)T * a.H;                // two [T][H] planes after x2
        e = launch_dense_q4k_gemm_multi(&so, 1, qd, att16, T, part, a.H, nullptr, 2, (size_t)T * a.H, st);
        if (e != cudaSuccess) return e;
        return launch_pdl(residual_rmsnorm_rows, dim3(T), dim3(NR_THREADS), 0, st, a.hidden, part,
                          part + (size_t)T * a.H, a.ffn_norm, a.eps, a.H, x2);
    } else {
        // in place: every element of h is read and written by one thread
        e = launch_dense_q4k_gemm_multi(&so, 1, qd, att16, T, a.hidden, a.H, a.hidden, 1, 0, st);
        if (e != cudaSuccess) return e;
        return launch_pdl(rmsnorm_rows<0>, dim3(T), dim3(NR_THREADS), 0, st, a.hidden, a.ffn_norm, a.eps, a.H,
                          x2);
    }
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
