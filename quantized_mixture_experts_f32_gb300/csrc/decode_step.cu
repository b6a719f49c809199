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
#include "pdl.cuh"
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

constexpr int GV_WARPS = 8;

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
    const float* norm_w;   // nullable: x is first RMS-normalised and scaled by norm_w
    float eps;
};

// y = W x (+ res) for up to three Q4_K matrices sharing the same x (optionally
// x = RMSNorm(x) * norm_w, recomputed by every CTA).  Each warp owns RPW
// consecutive rows and issues all their loads before any arithmetic (16-byte
// pieces, NT per lane and row), so a CTA keeps ~RPW*9 KB in flight; x and its
// 16-column sums sit in shared memory.
// x sits in shared memory with 4 floats of padding after every 64 (column c
// at c + 4*(c/64)): the 16-float runs the 8 lanes of one superblock read at
// once then fall in 8 different bank groups instead of 2.
__device__ __forceinline__ int xpad(int c) { return c + 4 * (c >> 6); }

// Programmatic dependent launch: every kernel of the decode step is launched so
// that it may start while the previous kernel on the stream drains.  Before
// griddep_wait() a kernel touches only data that no kernel of the current step
// before it writes (weights, KV slots of earlier positions); after it, the
// previous kernel has completed and its writes are visible.  Each kernel lets
// the next one launch only once it has passed its own wait, so a kernel that
// starts early never overlaps the kernel two places before it.
__device__ __forceinline__ void griddep_wait_launch() {
    pdl_wait();
    pdl_launch_dependents();
}

template <int RPW, int NT>
__global__ void __launch_bounds__(GV_WARPS * 32, 2) q4k_gemv(const GemvArgs a) {
    extern __shared__ float sx[];
    float* xsum = sx + xpad(a.cols);
    __shared__ float red[GV_WARPS];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this warp's weight pieces first: they stream in while x is staged
    const int npieces = 8 * (a.cols / QK);
    const int r0 = (blockIdx.x * GV_WARPS + warp) * RPW;
    uint4 hd[RPW][NT], qd[RPW][NT];
    const uint8_t* wp[RPW];
    float* yp[RPW];
    const float* rp[RPW];
    int rr[RPW];
    const int n0 = a.seg[0].rows, n1 = a.nseg > 1 ? a.seg[1].rows : 0,
              n2 = a.nseg > 2 ? a.seg[2].rows : 0;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        // segment of row r0 + i, selected without indexing the parameter array
        const int r_ = r0 + i;
        const int s_ = r_ < n0 ? 0 : r_ < n0 + n1 ? 1 : r_ < n0 + n1 + n2 ? 2 : 3;
        wp[i] = s_ == 0 ? a.seg[0].W : s_ == 1 ? a.seg[1].W : s_ == 2 ? a.seg[2].W : nullptr;
        yp[i] = s_ == 0 ? a.seg[0].y : s_ == 1 ? a.seg[1].y : a.seg[2].y;
        rp[i] = s_ == 0 ? a.seg[0].res : s_ == 1 ? a.seg[1].res : a.seg[2].res;
        rr[i] = r_ - (s_ >= 1 ? n0 : 0) - (s_ >= 2 ? n1 : 0);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int task = lane + 32 * t;
            if (wp[i] && task < npieces) {
                const uint8_t* b = wp[i] + ((size_t)rr[i] * (a.cols / QK) + (task >> 3)) * Q4K_BYTES;
                hd[i][t] = __ldg(reinterpret_cast<const uint4*>(b));
                qd[i][t] = __ldg(reinterpret_cast<const uint4*>(b + 16 + 16 * (task & 7)));
            }
        }
    }
    // x is the previous kernel's output: wait for it only now, with the weight
    // loads already in flight
    griddep_wait_launch();
    // the residual rows, in flight with x (read at the end, they would add a
    // round trip after the dot products)
    float resv[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i) resv[i] = lane == 0 && wp[i] && rp[i] ? rp[i][rr[i]] : 0.f;
    // x (and the norm weights) in flight at once: cols <= 4096, 4 float4 per thread
    constexpr int XLD = 4096 / 4 / (GV_WARPS * 32);
    float4 xv[XLD], wv[XLD];
#pragma unroll
    for (int j = 0; j < XLD; ++j) {
        const int i = threadIdx.x + j * GV_WARPS * 32;
        if (i < a.cols / 4) {
            xv[j] = reinterpret_cast<const float4*>(a.x)[i];
            wv[j] = a.norm_w ? reinterpret_cast<const float4*>(a.norm_w)[i] : make_float4(1.f, 1.f, 1.f, 1.f);
        }
    }
    float r = 1.f;
    if (a.norm_w) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < XLD; ++j) {
            const int i = threadIdx.x + j * GV_WARPS * 32;
            if (i < a.cols / 4) {
                const float4 v = xv[j];
                ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
        for (int i = 0; i < GV_WARPS; ++i) tot += red[i];
        r = rsqrtf(tot / (float)a.cols + a.eps);
    }
#pragma unroll
    for (int j = 0; j < XLD; ++j) {
        const int i = threadIdx.x + j * GV_WARPS * 32;
        if (i < a.cols / 4) {
            float4 v = xv[j];
            if (a.norm_w) {
                const float4 w = wv[j];
                v = make_float4(v.x * r * w.x, v.y * r * w.y, v.z * r * w.z, v.w * r * w.w);
            }
            *reinterpret_cast<float4*>(sx + xpad(4 * i)) = v;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.cols / 16; i += blockDim.x) {
        const float4* q = reinterpret_cast<const float4*>(sx + xpad(16 * i));
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) s += (q[j].x + q[j].y) + (q[j].z + q[j].w);
        xsum[i] = s;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        float acc = 0.f;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int task = lane + 32 * t;
            if (wp[i] && task < npieces) {
                const int pc = task & 7;
                const int col = QK * (task >> 3) + 64 * (pc >> 1) + 16 * (pc & 1);
                float PA, PB;
                q4_piece_dot(qd[i][t], reinterpret_cast<const float4*>(sx + xpad(col)),
                             reinterpret_cast<const float4*>(sx + xpad(col + 32)), PA, PB);
                acc += q4_piece_finish(hd[i][t], pc, PA, PB, xsum[col / 16], xsum[col / 16 + 2]);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0 && wp[i]) yp[i][rr[i]] = acc + resv[i];
    }
}

// launch with RPW rows per warp chosen so that the grid still covers the SMs
// (and the per-lane registers stay bounded: RPW * NT <= 8)
cudaError_t launch_gemv(const GemvArgs& g, int total_rows, cudaStream_t st) {
    const int nt = (8 * (g.cols / QK) + 31) / 32;
    const size_t smem = sizeof(float) * (g.cols + g.cols / 16 + g.cols / 16);
    auto blocks = [&](int rpw) { return (total_rows + GV_WARPS * rpw - 1) / (GV_WARPS * rpw); };
    const int rpw_max = nt <= 2 ? 4 : 2;
    const int rpw = rpw_max >= 4 && blocks(4) >= 148 ? 4 : blocks(2) >= 148 ? 2 : 1;
    dim3 grid(blocks(rpw)), thr(GV_WARPS * 32);
#define QMOE_GEMV(R, N)                                                   \
    do {                                                                  \
        cudaError_t e_ = launch_pdl(q4k_gemv<R, N>, grid, thr, smem, st, g); \
        if (e_ != cudaSuccess) return e_;                                 \
    } while (0)
    if (nt == 1) {
        if (rpw == 4) QMOE_GEMV(4, 1); else if (rpw == 2) QMOE_GEMV(2, 1); else QMOE_GEMV(1, 1);
    } else if (nt == 2) {
        if (rpw == 4) QMOE_GEMV(4, 2); else if (rpw == 2) QMOE_GEMV(2, 2); else QMOE_GEMV(1, 2);
    } else if (nt <= 4) {
        if (rpw == 2) QMOE_GEMV(2, 4); else QMOE_GEMV(1, 4);
    } else {
        return cudaErrorInvalidValue;
    }
#undef QMOE_GEMV
    return cudaGetLastError();
}

constexpr int ATT_CHUNK = 64;         // positions per split
constexpr int ATT_THREADS = 256;
constexpr int ATT_HPT = 8;            // q heads per thread in the score pass, at most
constexpr int ATT_DPL = 8;            // head dims per lane in the norm/RoPE pass, at most

// cos/sin of the NEOX RoPE angles at one position, shared by every head and
// every layer of a decode step: inv_freq[j] = base^(-2j/hd) (host, double);
// the angle pos * inv_freq[j] (thousands of radians) is formed and reduced to
// [-pi, pi] in double, then cos and sin are taken in float.  One block.
__global__ void rope_table(const double* __restrict__ inv_freq, int half, int pos,
                           float2* __restrict__ cs) {
    constexpr double TWO_PI = 6.283185307179586476925286766559;
    griddep_wait_launch();
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        const double th = (double)pos * inv_freq[j];
        const double red = fma(-rint(th * (1.0 / TWO_PI)), TWO_PI, th);
        float sn, c;
        sincosf((float)red, &sn, &c);
        cs[j] = make_float2(c, sn);
    }
}

// One head vector into a warp: lane owns dims lane + 32 i, i < hd/32, so the
// pairs (d, d + hd/2) that RoPE rotates together sit in the same lane.
__device__ __forceinline__ void load_head(const float* __restrict__ src, int hd, float (&v)[ATT_DPL]) {
    const int lane = threadIdx.x & 31, n = hd / 32;
#pragma unroll
    for (int i = 0; i < ATT_DPL; ++i) v[i] = i < n ? src[lane + 32 * i] : 0.f;
}

// Per-head RMSNorm (weights nw) and NEOX RoPE (table cs) of a head vector held
// as load_head leaves it (v is overwritten)
__device__ __forceinline__ void norm_rope_vals(float (&v)[ATT_DPL], const float* __restrict__ nw,
                                               float eps, int hd, const float2* __restrict__ cs,
                                               float (&o)[ATT_DPL]) {
    const int lane = threadIdx.x & 31, n = hd / 32;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < ATT_DPL; ++i) ss = fmaf(v[i], v[i], ss);
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / (float)hd + eps);
#pragma unroll
    for (int i = 0; i < ATT_DPL; ++i)
        if (i < n) v[i] = v[i] * r * nw[lane + 32 * i];
#pragma unroll
    for (int i = 0; i < ATT_DPL / 2; ++i) {
        if (i < n / 2) {
            const float2 t = cs[lane + 32 * i];               // pair (j, j + hd/2)
            const float a = v[i], b = v[i + n / 2];
            o[i] = a * t.x - b * t.y;
            o[i + n / 2] = b * t.x + a * t.y;
        }
    }
}

// both, for a head vector read from src
__device__ __forceinline__ void norm_rope_warp(const float* __restrict__ src,
                                               const float* __restrict__ nw, float eps, int hd,
                                               const float2* __restrict__ cs,
                                               float (&o)[ATT_DPL]) {
    float v[ATT_DPL];
    load_head(src, hd, v);
    norm_rope_vals(v, nw, eps, hd, cs, o);
}

// Split-K (flash-decoding) GQA attention with the per-head Q/K RMSNorm, RoPE
// and the fp16 KV append fused in: block (kv head, chunk) normalises and
// rotates the `group` q heads of that kv head, and the block whose chunk holds
// position pos also normalises and rotates k, rounds k and v to fp16 and writes
// them to cache slot pos (and into its staged tile).  It then attends over
// positions [c*CH, min((c+1)*CH, pos+1)).  The chunk's K and V rows
// (contiguous in the cache) are staged in shared memory with coalesced 16-byte
// loads; K rows padded to an odd number of words so that one thread per
// position reads them without bank conflicts.  Writes per (q head, chunk):
// running max, sum of exp, unnormalised acc[hd].
template <int HPT>
__global__ void __launch_bounds__(ATT_THREADS) attn_partial(
    const float* __restrict__ q_raw, const float* __restrict__ k_raw,
    const float* __restrict__ v_raw, const float* __restrict__ q_norm,
    const float* __restrict__ k_norm, float eps, const float2* __restrict__ rope_cs,
    __half* __restrict__ k_cache, __half* __restrict__ v_cache, int pos, int hd, int nq, int nkv,
    int max_ctx, int nsplit, float* __restrict__ part) {
    extern __shared__ __align__(16) float sm[];
    // chunks in reverse block order: the CTA that owns position pos (and does
    // the KV append on top of its chunk) is among the first to be scheduled
    const int kvh = blockIdx.x, c = gridDim.y - 1 - blockIdx.y;
    const int group = nq / nkv;
    const int p0 = c * ATT_CHUNK, p1 = min(p0 + ATT_CHUNK, pos + 1);
    const int np = p1 - p0;
    const int kw = hd / 2 + 1;                         // padded K row, 32-bit words
    float* qs = sm;                                    // group * hd
    float* sc = qs + group * hd;                       // group * CHUNK
    uint32_t* ks = reinterpret_cast<uint32_t*>(sc + group * ATT_CHUNK);   // CHUNK * kw
    __half* vs = reinterpret_cast<__half*>(ks + ((ATT_CHUNK * kw + 3) & ~3));
    __shared__ float mx_s[32], sum_s[32];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = ATT_THREADS >> 5;
    const uint4* K = reinterpret_cast<const uint4*>(k_cache + ((size_t)kvh * max_ctx + p0) * hd);
    const uint4* V = reinterpret_cast<const uint4*>(v_cache + ((size_t)kvh * max_ctx + p0) * hd);
    const int vpr = hd / 8;                            // uint4 per row
    {
        // every thread's share of the tile in flight at once, then stored
        constexpr int NLD = ATT_CHUNK * 32 / ATT_THREADS;   // uint4 per thread at hd = 256
        uint4 kq[NLD], vq[NLD];
#pragma unroll
        for (int j = 0; j < NLD; ++j) {
            const int i = tid + j * ATT_THREADS;
            if (i < np * vpr) {
                kq[j] = __ldg(K + i);
                vq[j] = __ldg(V + i);
            }
        }
#pragma unroll
        for (int j = 0; j < NLD; ++j) {
            const int i = tid + j * ATT_THREADS;
            if (i < np * vpr) {
                const int row = i / vpr, cc = i - row * vpr;
                uint32_t* kd = ks + row * kw + 4 * cc;
                kd[0] = kq[j].x; kd[1] = kq[j].y; kd[2] = kq[j].z; kd[3] = kq[j].w;
                reinterpret_cast<uint4*>(vs)[i] = vq[j];
            }
        }
    }
    // q, k and v are the previous kernel's output (the tile above holds only
    // slots of earlier positions, and the slot at pos is overwritten below)
    griddep_wait_launch();
    // the chunk owner's warp 0 loads the new token's k and v together with its
    // q head, so the append costs no round trip of its own
    const bool owner = pos >= p0 && pos < p1;
    float knew[ATT_DPL], vnew[ATT_DPL];
    if (owner && warp == 0) {
        load_head(k_raw + (size_t)kvh * hd, hd, knew);
        load_head(v_raw + (size_t)kvh * hd, hd, vnew);
    }
    // q heads of this kv head: RMSNorm + RoPE (warp per head)
    for (int g = warp; g < group; g += nw) {
        float o[ATT_DPL];
        norm_rope_warp(q_raw + (size_t)(kvh * group + g) * hd, q_norm, eps, hd, rope_cs, o);
#pragma unroll
        for (int i = 0; i < ATT_DPL; ++i)
            if (i < hd / 32) qs[g * hd + lane + 32 * i] = o[i];
    }
    __syncthreads();                                   // tile staged (row pos - p0 is stale)
    if (owner && warp == 0) {
        // the new token's k and v: cache slot pos and tile row pos - p0
        float o[ATT_DPL];
        norm_rope_vals(knew, k_norm, eps, hd, rope_cs, o);
        __half* kc = k_cache + ((size_t)kvh * max_ctx + pos) * hd;
        __half* vc = v_cache + ((size_t)kvh * max_ctx + pos) * hd;
        __half* kt = reinterpret_cast<__half*>(ks + (pos - p0) * kw);
        __half* vt = vs + (size_t)(pos - p0) * hd;
#pragma unroll
        for (int i = 0; i < ATT_DPL; ++i) {
            if (i < hd / 32) {
                const int d = lane + 32 * i;
                const __half kh = __float2half_rn(o[i]);
                const __half vh = __float2half_rn(vnew[i]);
                kc[d] = kh;
                vc[d] = vh;
                kt[d] = kh;
                vt[d] = vh;
            }
        }
    }
    __syncthreads();
    // scores: thread -> position pp, heads [hg*HPT, (hg+1)*HPT)
    const float scale = rsqrtf((float)hd);
    {
        const int pp = tid % ATT_CHUNK, hg = tid / ATT_CHUNK;
        float acc[HPT];
#pragma unroll
        for (int g = 0; g < HPT; ++g) acc[g] = 0.f;
        if (hg * HPT < group && pp < np) {
            const uint32_t* kr = ks + pp * kw;
            const float* qh = qs + hg * HPT * hd;
#pragma unroll 4
            for (int d2 = 0; d2 < hd / 2; d2 += 2) {
                const float2 k0 = __half22float2(*reinterpret_cast<const __half2*>(kr + d2));
                const float2 k1 = __half22float2(*reinterpret_cast<const __half2*>(kr + d2 + 1));
#pragma unroll
                for (int g = 0; g < HPT; ++g) {
                    const float4 qv = *reinterpret_cast<const float4*>(qh + g * hd + 2 * d2);
                    acc[g] = fmaf(qv.x, k0.x, fmaf(qv.y, k0.y, fmaf(qv.z, k1.x, fmaf(qv.w, k1.y, acc[g]))));
                }
            }
        }
#pragma unroll
        for (int g = 0; g < HPT; ++g)
            if (hg * HPT + g < group)
                sc[(hg * HPT + g) * ATT_CHUNK + pp] = pp < np ? acc[g] * scale : -INFINITY;
    }
    __syncthreads();
    // per q head (one warp each, warps loop over heads): max and sum of exp
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
    // P V: thread -> (head g, 4 consecutive dims)
    const int dq = hd / 4;
    for (int i = tid; i < group * dq; i += ATT_THREADS) {
        const int g = i / dq, d4 = i - g * dq;
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
        const float* pg = sc + g * ATT_CHUNK;
        for (int pp = 0; pp < np; ++pp) {
            const float w = pg[pp];
            const uint2 vv = *reinterpret_cast<const uint2*>(vs + (size_t)pp * hd + 4 * d4);
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
            a0 = fmaf(w, v01.x, a0);
            a1 = fmaf(w, v01.y, a1);
            a2 = fmaf(w, v23.x, a2);
            a3 = fmaf(w, v23.y, a3);
        }
        float* o = part + ((size_t)(kvh * group + g) * nsplit + c) * (hd + 2);
        *reinterpret_cast<float2*>(o + 2 + 4 * d4) = make_float2(a0, a1);
        *reinterpret_cast<float2*>(o + 4 + 4 * d4) = make_float2(a2, a3);
        if (d4 == 0) { o[0] = mx_s[g]; o[1] = sum_s[g]; }
    }
}

size_t attn_smem(int group, int hd) {
    const size_t kwords = (size_t)ATT_CHUNK * (hd / 2 + 1);
    return sizeof(float) * (group * hd + group * ATT_CHUNK) + 4 * ((kwords + 3) & ~(size_t)3) +
           sizeof(__half) * ATT_CHUNK * hd;
}

// merge the splits of one q head (block per q head).  Every load a thread
// needs is issued before any of them is used, so the merge costs one round
// trip to L2 instead of a chain of them: thread (d2, sl) holds the partial
// accumulators of dims 2*d2, 2*d2+1 for splits sl, sl+S, ... in registers
// while the split statistics (running max, sum of exp) are loaded beside them
// and reduced over the block; the split weights exp(m_c - M) then go through
// shared memory, each thread sums its splits in order and the S slices are
// combined in order.
constexpr int MRG_THREADS = 256;
constexpr int MRG_LD = 16;            // splits per thread held in registers at once

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float w = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, w) : v + w;
    }
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = red[0];
    for (int i = 1; i < MRG_THREADS / 32; ++i) t = is_max ? fmaxf(t, red[i]) : t + red[i];
    return t;
}

__global__ void __launch_bounds__(MRG_THREADS) attn_merge(const float* __restrict__ part,
                                                          int nsplit, int nvalid, int hd,
                                                          float* __restrict__ out) {
    extern __shared__ float wsh[];                     // nvalid m_c (then weights), nvalid l_c,
                                                       // then S * hd slice sums
    __shared__ float red_m[MRG_THREADS / 32], red_l[MRG_THREADS / 32];
    const int h = blockIdx.x, tid = threadIdx.x;
    const int pitch = hd + 2;                          // per split: m, l, acc[hd]
    const int hd2 = hd / 2;
    const int S = MRG_THREADS / hd2;                   // slices of splits (hd <= 256: S >= 2)
    const int d2 = tid % hd2, sl = tid / hd2;
    const bool has = sl < S;                           // hd = 192 leaves 64 threads idle here
    float* ls = wsh + nvalid;
    float* acc_s = ls + nvalid;
    griddep_wait_launch();
    const float* ph = part + (size_t)h * nsplit * pitch;
    // the accumulators of this thread's first MRG_LD splits ...
    float2 av[MRG_LD];
#pragma unroll
    for (int j = 0; j < MRG_LD; ++j) {
        const int c = sl + j * S;
        av[j] = has && c < nvalid ? *reinterpret_cast<const float2*>(ph + (size_t)c * pitch + 2 + 2 * d2)
                                  : make_float2(0.f, 0.f);
    }
    // ... and the split statistics, in flight together
    float m = -INFINITY;
    for (int c = tid; c < nvalid; c += MRG_THREADS) {
        const float2 v = *reinterpret_cast<const float2*>(ph + (size_t)c * pitch);
        wsh[c] = v.x;
        ls[c] = v.y;
        m = fmaxf(m, v.x);
    }
    const float M = block_reduce(m, true, red_m);
    float l = 0.f;
    for (int c = tid; c < nvalid; c += MRG_THREADS) {
        const float w = expf(wsh[c] - M);
        wsh[c] = w;
        l = fmaf(w, ls[c], l);
    }
    const float tot = block_reduce(l, false, red_l);  // its barrier also publishes the weights
    float2 a = make_float2(0.f, 0.f);
    if (has) {
#pragma unroll
        for (int j = 0; j < MRG_LD; ++j) {
            const int c = sl + j * S;
            if (c < nvalid) {
                a.x = fmaf(wsh[c], av[j].x, a.x);
                a.y = fmaf(wsh[c], av[j].y, a.y);
            }
        }
        // splits beyond the first MRG_LD * S (contexts over 4096 at head_dim 128)
        for (int c0 = sl + MRG_LD * S; c0 < nvalid; c0 += MRG_LD * S) {
#pragma unroll
            for (int j = 0; j < MRG_LD; ++j) {
                const int c = c0 + j * S;
                av[j] = c < nvalid ? *reinterpret_cast<const float2*>(ph + (size_t)c * pitch + 2 + 2 * d2)
                                   : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int j = 0; j < MRG_LD; ++j) {
                const int c = c0 + j * S;
                if (c < nvalid) {
                    a.x = fmaf(wsh[c], av[j].x, a.x);
                    a.y = fmaf(wsh[c], av[j].y, a.y);
                }
            }
        }
        acc_s[sl * hd + 2 * d2] = a.x;
        acc_s[sl * hd + 2 * d2 + 1] = a.y;
    }
    __syncthreads();
    if (tid < hd) {
        float r = 0.f;
        for (int k = 0; k < S; ++k) r += acc_s[k * hd + tid];
        out[(size_t)h * hd + tid] = r / tot;
    }
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
    (void)xs;
    const int qd = a.nq * a.hd, kvd = a.nkv * a.hd;
    cudaError_t e;
    // B1 + B2: q, k, v = Wq x, Wk x, Wv x with x = RMSNorm(h) * attn_norm (no bias)
    GemvArgs g{};
    g.seg[0] = GemvSeg{L.wq, q, nullptr, qd};
    g.seg[1] = GemvSeg{L.wk, kv, nullptr, kvd};
    g.seg[2] = GemvSeg{L.wv, kv + kvd, nullptr, kvd};
    g.nseg = 3;
    g.cols = a.H;
    g.x = h;
    g.norm_w = L.attn_norm;
    g.eps = a.eps;
    e = launch_gemv(g, qd + 2 * kvd, st);
    if (e != cudaSuccess) return e;
    // B3-B6: per-head Q/K RMSNorm, NEOX RoPE, fp16 KV append at pos (all fused
    // into the split-K attention), GQA attention over positions 0..pos
    const int nsplit = (a.max_ctx + ATT_CHUNK - 1) / ATT_CHUNK;
    const int nvalid = a.pos / ATT_CHUNK + 1;
    const int group = a.nq / a.nkv;
    dim3 ga(a.nkv, nvalid);
    const int hpt = (group * ATT_CHUNK + ATT_THREADS - 1) / ATT_THREADS;
#define QMOE_ATT(N)                                                                          \
    e = launch_pdl(attn_partial<N>, ga, dim3(ATT_THREADS), attn_smem(group, a.hd), st, q,          \
                   (const float*)kv, (const float*)(kv + kvd), L.q_norm, L.k_norm, a.eps,          \
                   a.rope_cs, L.k_cache, L.v_cache, a.pos, a.hd, a.nq, a.nkv, a.max_ctx, nsplit,   \
                   part)
    if (hpt <= 1) QMOE_ATT(1); else if (hpt <= 2) QMOE_ATT(2); else if (hpt <= 4) QMOE_ATT(4); else QMOE_ATT(8);
#undef QMOE_ATT
    if (e != cudaSuccess) return e;
    e = launch_pdl(attn_merge, dim3(a.nq), dim3(MRG_THREADS), sizeof(float) * (2 * nvalid + 2 * MRG_THREADS), st,
                   (const float*)part, nsplit, nvalid, a.hd, att);
    if (e != cudaSuccess) return e;
    // B7: h_out = h + Wo att
    GemvArgs go{};
    go.seg[0] = GemvSeg{L.wo, h_out, h, a.H};
    go.nseg = 1;
    go.cols = qd;
    go.x = att;
    e = launch_gemv(go, a.H, st);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Shared memory limit of the attention kernel (once per device context) and
// the shapes it serves: at most ATT_HPT * ATT_THREADS / ATT_CHUNK (32) q heads
// per kv head, head_dim a multiple of 64 up to 256 with the staged chunk inside
// ATT_SMEM_MAX.
constexpr int ATT_SMEM_MAX = 200 * 1024;     // dynamic; the kernel also has 256 B static

cudaError_t decode_step_prepare() {
    const void* fns[] = {reinterpret_cast<const void*>(&attn_partial<1>),
                         reinterpret_cast<const void*>(&attn_partial<2>),
                         reinterpret_cast<const void*>(&attn_partial<4>),
                         reinterpret_cast<const void*>(&attn_partial<8>)};
    for (const void* f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ATT_SMEM_MAX);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_rope_table(const double* inv_freq, int hd, int pos, float2* cs,
                              cudaStream_t st) {
    return launch_pdl(rope_table, dim3(1), dim3(128), 0, st, inv_freq, hd / 2, pos, cs);
}

bool attention_supported(int nq, int nkv, int hd) {
    if (nkv < 1 || nq % nkv || (nq / nkv) * ATT_CHUNK > ATT_HPT * ATT_THREADS) return false;
    if (hd < 64 || hd > 32 * ATT_DPL || hd % 64) return false;     // RoPE pairs within a lane
    return attn_smem(nq / nkv, hd) <= (size_t)ATT_SMEM_MAX;
}

int attn_splits(int max_ctx) { return (max_ctx + ATT_CHUNK - 1) / ATT_CHUNK; }

}  // namespace qmoe
