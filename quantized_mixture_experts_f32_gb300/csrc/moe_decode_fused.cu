// moe_decode_fused.cu -- the whole qwen3moe MoE-FFN layer for a few tokens
// (decode, T <= 8) as ONE persistent cooperative kernel, one CTA per SM.
//
// What it computes is the layer of the aprender issue "qwen3moe (Qwen3-30B-A3B,
// ...) has NO working CUDA path" ("File facts", "Gaps ... G3"): F32 router GEMV,
// softmax + top-k + renorm, per selected expert Q4_K gate/up dequant-GEMV with
// SiLU(gate)*up, Q6_K or Q4_K down dequant-GEMV, weighted sum into the residual.
// The page's v1 design spent 48 host syncs per token on host top-k and 2
// launches per expert for the weighted sum; here the layer is one launch with
// no host involvement and is graph-capturable.
//
// Structure (G CTAs of 16 warps):
//  A  every CTA stages x in shared memory; CTA c computes the router logits of
//     experts c, c+G, ... (fixed-order reductions) -> grid barrier 1.
//  B  every CTA redoes the (cheap, deterministic) top-k of all T tokens and
//     builds the same per-expert pair lists; it then owns a contiguous share of
//     the (expert, f) gate/up rows and a contiguous range of down rows of every
//     used expert, cut into chunks of a few KB.
//  C  warp w handles chunks w, w+16, ... and streams them itself with bulk async
//     copies (TMA) into its two shared-memory slots, one chunk ahead of the one
//     it computes (one issuing thread per CTA cannot keep HBM busy; sixteen
//     can).  Gate/up chunks produce act[p][f] = silu(g)*u (fp32); a warp's
//     first down chunks are already in flight while it finishes gate/up.
//  -  grid barrier 2 (all act written).
//  D  down chunks: y = Wd_e act for this CTA's rows of every used expert, then
//     out[t][h] = res[t][h] + sum_j w[t][j] y_j[h] in slot order j = 0..K-1
//     (deterministic, no atomics on values).
// Every wait is bounded (%globaltimer); on expiry the kernel records
// QMOE_ERR_TIMEOUT, stops computing, drains its own copies and exits.
#include <math.h>

#include "kquant.cuh"
#include "ptx_sync.cuh"
#include "qmoe_internal.h"

#ifdef QMOE_PHASE_TRACE
// per-CTA phase timestamps (%globaltimer), compiled only into diagnostic builds
__device__ unsigned long long g_qmoe_trace[1024 * 64];
#define QMOE_TRACE(slot)                                                            \
    do {                                                                            \
        g_qmoe_trace[blockIdx.x * 64 + (slot)] = qmoe::globaltimer();               \
    } while (0)
#else
#define QMOE_TRACE(slot) \
    do {                 \
    } while (0)
#endif

namespace qmoe {

namespace {

constexpr int NCW = 16;                     // warps; each streams its own chunks
constexpr int NTHREADS = NCW * 32;
constexpr int NSLOT = 2 * NCW;              // two ring slots per warp
constexpr int MAXT = 8;
constexpr int MAXP = 128;

// misc int slots
enum { M_NUSED = 0, M_NCH, M_NGU, M_GUDONE, M_ABORT, M_H0, M_NROWS, M_GULO, M_NRC, M_GUWARPS,
       M_COUNT = 16 };

struct SmemLayout {
    int off_bar, off_misc, off_red, off_ids, off_wts, off_used, off_first, off_pairs,
        off_x, off_xsum, off_xscale, off_ybuf, off_ring, total, slot_bytes, rows_max, act_stage;
};

__host__ __device__ inline int al(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline SmemLayout fused_layout(int T, int H, int K, int F, int rows_max,
                                                   int slot_bytes, int asum_bytes, bool stage_act) {
    SmemLayout L;
    const int P = T * K;
    // the x region is reused in the down phase for the act group sums and,
    // when it fits, a copy of act itself
    const int act_bytes = stage_act ? P * F * 4 : 0;
    asum_bytes = al(asum_bytes, 16) + act_bytes;
    int o = 0;
    L.off_bar = o;      o += NSLOT * 8;
    L.off_misc = o;     o += M_COUNT * 4;
    L.off_red = o;      o += NCW * MAXT * 4;
    L.off_ids = o;      o += al(P, 4) * 4;
    L.off_wts = o;      o += al(P, 4) * 4;
    L.off_used = o;     o += al(P, 4) * 4;
    L.off_first = o;    o += al(P + 1, 4) * 4;
    L.off_pairs = o;    o += al(P, 4) * 4;
    o = al(o, 16);
    L.off_x = o;        o += al(T * H * 4 > asum_bytes ? T * H * 4 : asum_bytes, 16);
    L.off_xsum = o;     o += al(T * (H / 16) * 4, 16);
    L.off_xscale = o;   o += al(T * (H / 16) * 4, 16);
    L.off_ybuf = o;     o += al(P * rows_max * 4, 16);
    o = al(o, 128);
    L.off_ring = o;     o += NSLOT * slot_bytes;
    L.total = o;
    L.slot_bytes = slot_bytes;
    L.rows_max = rows_max;
    L.act_stage = act_bytes ? al(asum_bytes - act_bytes, 16) : -1;   // byte offset in the x region
    return L;
}

struct FusedParams {
    const float* x;
    const float* res;
    const float* bias;
    const float* router;
    const uint8_t* gate;
    const uint8_t* up;
    const uint8_t* down;
    float* out;
    int32_t* ids_out;
    float* w_out;
    float* logits;
    float* act;
    unsigned* bar;
    int* status;
    int T, H, E, K, F, norm;
    int cf;          // f rows per gate/up chunk (divides F)
    SmemLayout L;
};

// ----------------------------------------------------------------------------- small helpers

__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// 8 bytes at an even shared-memory address (three aligned words, funnel shift)
__device__ __forceinline__ uint2 lds8_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3) * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2];
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// one 16-byte Q4_K nibble piece against 32 x values held in registers
__device__ __forceinline__ void q4_piece_regs(uint4 q, const float4 (&xa)[4], const float4 (&xb)[4],
                                              float& PA, float& PB) {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0x0F0F0F0Fu;
        const uint32_t hi = (w[i] >> 4) & 0x0F0F0F0Fu;
        fma2(a0, a1, mag<0>(lo), mag<1>(lo), xa[i].x, xa[i].y);
        fma2(a0, a1, mag<2>(lo), mag<3>(lo), xa[i].z, xa[i].w);
        fma2(b0, b1, mag<0>(hi), mag<1>(hi), xb[i].x, xb[i].y);
        fma2(b0, b1, mag<2>(hi), mag<3>(hi), xb[i].z, xb[i].w);
    }
    PA = a0 + a1;
    PB = b0 + b1;
}

// Exact integer form of one 16-byte Q4_K piece.  The 16 x values paired with the
// low nibbles are n_l * scaleA with n_l a 24-bit integer split into three
// signed byte planes (n = p2*2^16 + p1*2^8 + p0); the nibble bytes of the
// piece are the other dp4a operand, so sum_l q_l n_l is formed exactly in
// int32 with no per-weight float conversion.  Returns sum q*x for the low
// (SA) and high (SB) nibbles.
__device__ __forceinline__ void q4_piece_dp4a(uint4 q, const int (&xa)[3][4], const int (&xb)[3][4],
                                              float scaleA, float scaleB, float& SA, float& SB) {
    int a0 = 0, a1 = 0, a2 = 0, b0 = 0, b1 = 0, b2 = 0;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int lo = (int)(w[i] & 0x0F0F0F0Fu), hi = (int)((w[i] >> 4) & 0x0F0F0F0Fu);
        a0 = __dp4a(lo, xa[0][i], a0);
        a1 = __dp4a(lo, xa[1][i], a1);
        a2 = __dp4a(lo, xa[2][i], a2);
        b0 = __dp4a(hi, xb[0][i], b0);
        b1 = __dp4a(hi, xb[1][i], b1);
        b2 = __dp4a(hi, xb[2][i], b2);
    }
    SA = scaleA * fmaf((float)a2, 65536.f, (float)(a1 * 256 + a0));
    SB = scaleB * fmaf((float)b2, 65536.f, (float)(b1 * 256 + b0));
}

// contribution of a piece given the exact sums QA = sum q x, QB, and the x sums
__device__ __forceinline__ float q4_piece_finish_exact(uint4 hdr, int pc, float QA, float QB,
                                                       float XA, float XB) {
    int sA, mA, sB, mB;
    q4_scales(hdr.y, hdr.z, hdr.w, pc >> 1, sA, mA, sB, mB);
    const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
    float r = (d * (float)sA) * QA - (dmin * (float)mA) * XA;
    r = fmaf(d * (float)sB, QB, r) - (dmin * (float)mB) * XB;
    return r;
}

// 24-bit exact-integer quantiser limit: |n| <= 2^23 - 2^16 keeps the top byte
// plane in [-127, 127]
constexpr float XQ_LIM = 8323072.f;

// ----------------------------------------------------------------------------- the kernel

template <int NSB_G, int NSB_D, int DQT>
__global__ void __launch_bounds__(NTHREADS, 1) moe_decode_fused(const FusedParams p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const SmemLayout& L = p.L;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int T = p.T, H = p.H, E = p.E, K = p.K, F = p.F, P = T * K;
    constexpr int RBG = NSB_G * Q4K_BYTES;                        // gate/up row bytes
    constexpr int BBD = DQT == 1 ? Q4K_BYTES : Q6K_BYTES;
    constexpr int RBD = NSB_D * BBD;                              // down row bytes
    constexpr int NTG = (8 * NSB_G + 31) / 32;                    // gate/up tasks per lane

    uint64_t* fullb = reinterpret_cast<uint64_t*>(sm + L.off_bar);
    int* misc = reinterpret_cast<int*>(sm + L.off_misc);
    float* red = reinterpret_cast<float*>(sm + L.off_red);
    int32_t* ids_s = reinterpret_cast<int32_t*>(sm + L.off_ids);
    float* wts_s = reinterpret_cast<float*>(sm + L.off_wts);
    int32_t* used_e = reinterpret_cast<int32_t*>(sm + L.off_used);
    int32_t* used_first = reinterpret_cast<int32_t*>(sm + L.off_first);
    int32_t* pairs = reinterpret_cast<int32_t*>(sm + L.off_pairs);
    float* x_s = reinterpret_cast<float*>(sm + L.off_x);
    float* xsum = reinterpret_cast<float*>(sm + L.off_xsum);
    float* xscale = reinterpret_cast<float*>(sm + L.off_xscale);
    int32_t* xq = reinterpret_cast<int32_t*>(x_s);                 // byte planes, after the router
    float* ybuf = reinterpret_cast<float*>(sm + L.off_ybuf);
    uint8_t* ring = sm + L.off_ring;
    const int SB = L.slot_bytes;

    // ---------------- phase A: stage x, barriers, router slice
    if (tid == 0) QMOE_TRACE(0);
    // this warp's router columns of the first expert row, loaded before x so
    // that both loads are in flight together
    constexpr int RW = 2;                                          // float4 per lane
    float4 wpre[RW];
#pragma unroll
    for (int i = 0; i < RW; ++i) {
        const int h = 4 * (lane + 32 * warp) + i * 4 * 32 * NCW;
        wpre[i] = (c < E && h < H) ? __ldg(reinterpret_cast<const float4*>(p.router + (size_t)c * H + h))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = tid; i < T * H / 4; i += NTHREADS)
        reinterpret_cast<float4*>(x_s)[i] = __ldg(reinterpret_cast<const float4*>(p.x) + i);
    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) mbar_init(&fullb[s], 1);
        for (int i = 0; i < M_COUNT; ++i) misc[i] = 0;
        fence_barrier_init();
    }
    __syncthreads();
    for (int i = tid; i < T * (H / 16); i += NTHREADS) {
        const float4* q = reinterpret_cast<const float4*>(x_s + 16 * i);
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) s += (q[j].x + q[j].y) + (q[j].z + q[j].w);
        xsum[i] = s;
    }
    for (int e = c; e < E; e += G) {
        {
            float acc[MAXT];
#pragma unroll
            for (int t = 0; t < MAXT; ++t) acc[t] = 0.f;
            const float* wr = p.router + (size_t)e * H;
            auto dot4 = [&](const float4 w, int h) {
#pragma unroll
                for (int t = 0; t < MAXT; ++t) {
                    if (t < T) {
                        const float4 xv = *reinterpret_cast<const float4*>(x_s + t * H + h);
                        acc[t] = fmaf(w.x, xv.x, acc[t]);
                        acc[t] = fmaf(w.y, xv.y, acc[t]);
                        acc[t] = fmaf(w.z, xv.z, acc[t]);
                        acc[t] = fmaf(w.w, xv.w, acc[t]);
                    }
                }
            };
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                const int h = 4 * (lane + 32 * warp) + i * 4 * 32 * NCW;
                if (h < H) dot4(e == c ? wpre[i] : __ldg(reinterpret_cast<const float4*>(wr + h)), h);
            }
            for (int h = 4 * (lane + 32 * warp) + RW * 4 * 32 * NCW; h < H; h += 4 * 32 * NCW)
                dot4(__ldg(reinterpret_cast<const float4*>(wr + h)), h);
#pragma unroll
            for (int t = 0; t < MAXT; ++t) {
                if (t < T) {
                    const float s = warp_sum(acc[t]);
                    if (lane == 0) red[warp * MAXT + t] = s;
                }
            }
        }
        __syncthreads();
        if (tid < T) {
            float s = 0.f;
            for (int w = 0; w < NCW; ++w) s += red[w * MAXT + tid];
            p.logits[(size_t)tid * E + e] = s + (p.bias ? p.bias[e] : 0.f);
        }
        __syncthreads();
    }
    // x -> per-16-column scale and three signed byte planes, in place (the
    // router, the only fp32 reader of x_s, is done)
    {
        constexpr int GPT = 2;                                     // 16-col groups per thread
        int pw[GPT][12];
        float psc[GPT];
        const int ng = T * (H / 16);
#pragma unroll
        for (int gi = 0; gi < GPT; ++gi) {
            const int g = tid + gi * NTHREADS;
            if (g < ng) {
                const float* xv = x_s + 16 * g;
                float mx = 0.f;
#pragma unroll
                for (int z = 0; z < 16; ++z) mx = fmaxf(mx, fabsf(xv[z]));
                const float inv = mx > 0.f ? XQ_LIM / mx : 0.f;
                psc[gi] = mx / XQ_LIM;
#pragma unroll
                for (int w4 = 0; w4 < 4; ++w4) {
                    uint32_t p0 = 0, p1 = 0, p2 = 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int n = __float2int_rn(xv[4 * w4 + b] * inv);
                        const int d0 = ((n + 128) & 255) - 128;
                        const int n1 = (n - d0) >> 8;
                        const int d1 = ((n1 + 128) & 255) - 128;
                        const int d2 = (n1 - d1) >> 8;
                        p0 |= (uint32_t)(d0 & 255) << (8 * b);
                        p1 |= (uint32_t)(d1 & 255) << (8 * b);
                        p2 |= (uint32_t)(d2 & 255) << (8 * b);
                    }
                    pw[gi][w4] = (int)p0;
                    pw[gi][4 + w4] = (int)p1;
                    pw[gi][8 + w4] = (int)p2;
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int gi = 0; gi < GPT; ++gi) {
            const int g = tid + gi * NTHREADS;
            if (g < ng) {
#pragma unroll
                for (int z = 0; z < 12; ++z) xq[12 * g + z] = pw[gi][z];
                xscale[g] = psc[gi];
            }
        }
    }
    if (tid == 0) {
        QMOE_TRACE(1);
        grid_arrive(&p.bar[0]);
        if (!grid_wait(&p.bar[0], (unsigned)G)) {
            set_status(p.status, ST_TIMEOUT);
            misc[M_ABORT] = 1;
        }
    }
    __syncthreads();

    // ---------------- phase B: routing (identical in every CTA), all threads in
    // parallel: rank of every logit, softmax weights, pairs sorted by expert
    if (tid == 0) QMOE_TRACE(2);
    const bool abort_b = misc[M_ABORT] != 0;
    float* lg_s = reinterpret_cast<float*>(ring);                 // ring is idle until phase C
    int32_t* sel = reinterpret_cast<int32_t*>(lg_s + T * E);      // [T][K]
    uint32_t* bitmap = reinterpret_cast<uint32_t*>(sel + P);      // used experts, E <= 1024
    int32_t* se = reinterpret_cast<int32_t*>(bitmap + 32);        // experts in pair order
    for (int i = tid; i < T * E; i += NTHREADS) lg_s[i] = __ldcg(p.logits + i);
    if (tid < 32) bitmap[tid] = 0u;
    for (int i = tid; i < P; i += NTHREADS) sel[i] = 0;
    __syncthreads();
    if (!abort_b) {
        // rank of every logit among its token's E (ties: lower index first);
        // tpe consecutive lanes share one logit's E comparisons
        const int nel = T * E;
        int tpe = NTHREADS / nel;
        tpe = tpe >= 32 ? 32 : tpe >= 16 ? 16 : tpe >= 8 ? 8 : tpe >= 4 ? 4 : tpe >= 2 ? 2 : 1;
        if (tpe > 1) {
            const int i = tid / tpe, sub = tid - (tid / tpe) * tpe;
            const bool valid = i < nel;
            const int t = valid ? i / E : 0, e = valid ? i - t * E : 0;
            const float* l = lg_s + t * E;
            const float v = l[e];
            int rank = 0;
            for (int e2 = sub; e2 < E; e2 += tpe) {
                const float w = l[e2];
                rank += (w > v) || (w == v && e2 < e);
            }
            for (int o = tpe >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
            if (valid && sub == 0 && rank < K) sel[t * K + rank] = e;
        } else {
            for (int i = tid; i < nel; i += NTHREADS) {
                const int t = i / E, e = i - t * E;
                const float* l = lg_s + t * E;
                const float v = l[e];
                int rank = 0;
                for (int e2 = 0; e2 < E; ++e2) {
                    const float w = l[e2];
                    rank += (w > v) || (w == v && e2 < e);
                }
                if (rank < K) sel[t * K + rank] = e;
            }
        }
    }
    if (tid == 0) QMOE_TRACE(11);
    __syncthreads();
    // softmax weights (warp t) and, in parallel, each pair's place in the
    // expert-sorted pair list (threads 256.. ; ids are the selection itself)
    if (!abort_b && warp < T) {
        const float* l = lg_s + warp * E;
        const float vmax = l[sel[warp * K]];
        float z = 0.f;
        for (int e = lane; e < E; e += 32) z += expf(l[e] - vmax);
        z = warp_sum(z);
        int id = lane < K ? sel[warp * K + lane] : 0;
        if (id < 0 || id >= E) {                                  // only with NaN logits
            id = 0;
            set_status(p.status, ST_DEVICE_CHECK);
        }
        const float pj = lane < K ? expf(l[id] - vmax) / z : 0.f;
        const float psel = warp_sum(pj);
        if (lane < K) {
            ids_s[warp * K + lane] = id;
            wts_s[warp * K + lane] = p.norm ? pj / psel : pj;
        }
    }
    const int pt = tid - NTHREADS / 2;
    if (!abort_b && pt >= 0 && pt < P) {
        int e = sel[pt];
        e = (e < 0 || e >= E) ? 0 : e;
        int pos = 0;
        for (int q = 0; q < P; ++q) {
            int e2 = sel[q];
            e2 = (e2 < 0 || e2 >= E) ? 0 : e2;
            pos += (e2 < e) || (e2 == e && q < pt);
        }
        pairs[pos] = pt;
        se[pos] = e;
        atomicOr(&bitmap[e >> 5], 1u << (e & 31));
    }
    __syncthreads();
    if (tid == 0) QMOE_TRACE(12);
    if (!abort_b && tid < P) {
        const int e = se[tid];
        if (tid == 0 || se[tid - 1] != e) {
            int u = __popc(bitmap[e >> 5] & ((1u << (e & 31)) - 1u));
            for (int w = 0; w < (e >> 5); ++w) u += __popc(bitmap[w]);
            used_e[u] = e;
            used_first[u] = tid;
        }
    }
    if (warp == NCW - 1) {
        int nu = __popc(bitmap[lane]);
        for (int o = 16; o > 0; o >>= 1) nu += __shfl_xor_sync(0xffffffffu, nu, o);
        if (abort_b) nu = 0;
        if (lane == 0) {
            misc[M_NUSED] = nu;
            used_first[nu] = P;
            // Work of this CTA, in closed form.  Gate/up: the used experts' f rows
            // are cut into global chunks of CF consecutive f (CF divides F); CTA c
            // owns global chunks [c*NG/G, (c+1)*NG/G).  Down: rows [h0, h1) of
            // every used expert, RPC rows per chunk.
            const int CF = p.cf, CPE = F / CF;
            const int NG = nu * CPE;                             // < 2^17, NG * G < 2^31
            const int lo = NG * c / G, hi = NG * (c + 1) / G;
            const int h0 = H * c / G, h1 = H * (c + 1) / G;
            const int RPC = (SB - 32) / RBD;
            const int nrc = (h1 - h0 + RPC - 1) / RPC;
            misc[M_GULO] = lo;
            misc[M_NGU] = hi - lo;
            misc[M_GUWARPS] = hi - lo < NCW ? hi - lo : NCW;      // warps with gate/up work
            misc[M_NRC] = nrc;
            misc[M_NCH] = (hi - lo) + nu * nrc;
            misc[M_H0] = h0;
            misc[M_NROWS] = h1 - h0;
            if (hi - lo == 0) grid_arrive(&p.bar[1]);
        }
    }
    __syncthreads();
    if (tid == 0) QMOE_TRACE(13);
    if (c == 0 && tid < P && !abort_b) {
        if (p.ids_out) p.ids_out[tid] = ids_s[tid];
        if (p.w_out) p.w_out[tid] = wts_s[tid];
    }
    if (tid == 0) QMOE_TRACE(3);
    const int n_ch = misc[M_NCH], n_gu = misc[M_NGU];
    const int gu_lo = misc[M_GULO], nrc = misc[M_NRC];
    const int CPE = F / p.cf, RPC = (SB - 32) / RBD;
    const int H0c = misc[M_H0], H1c = H0c + misc[M_NROWS];
    // chunk k -> (is_gu, used index u, start row, row count)
    auto decode = [&](int k, int& u, int& start, int& cnt) -> bool {
        if (k < n_gu) {
            const int g = gu_lo + k;
            u = g / CPE;
            start = (g - u * CPE) * p.cf;
            cnt = p.cf;
            return true;
        }
        const int kd = k - n_gu;
        u = kd / nrc;
        start = H0c + (kd - u * nrc) * RPC;
        cnt = min(RPC, H1c - start);
        return false;
    };

    // ---------------- phases C and D: warp w streams and computes chunks w, w+16, ...
    // chunk j of this warp lives in slot warp + 16*(j&1); it is issued two
    // chunks ahead, right after the chunk that used the slot before it
    auto issue = [&](int j) {                                    // lane 0 only
        const int k = warp + NCW * j;
        if (k >= n_ch) return;
        const int s = warp + NCW * (j & 1);
        int u, start, cnt;
        const bool is_gu = decode(k, u, start, cnt);
        const int e = used_e[u];
        uint8_t* dst = ring + (size_t)s * SB;
        fence_proxy_async();                                     // earlier reads of the slot
        if (is_gu) {
            const uint32_t bytes = (uint32_t)(cnt * RBG);
            const size_t off = (size_t)e * F * RBG + (size_t)start * RBG;
            mbar_arrive_expect_tx(&fullb[s], 2 * bytes);
            bulk_g2s(dst, p.gate + off, bytes, &fullb[s]);
            bulk_g2s(dst + bytes, p.up + off, bytes, &fullb[s]);
        } else {
            const uint8_t* src = p.down + (size_t)e * H * RBD + (size_t)start * RBD;
            const uintptr_t a0 = reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15);
            const uintptr_t a1 = (reinterpret_cast<uintptr_t>(src) + (size_t)cnt * RBD + 15) & ~uintptr_t(15);
            mbar_arrive_expect_tx(&fullb[s], (uint32_t)(a1 - a0));
            bulk_g2s(dst, reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0), &fullb[s]);
        }
    };
    if (lane == 0) {
        issue(0);
        issue(1);
    }
    {
        // ---------------- phase C: gate/up + SwiGLU
        int xa[NTG][3][4], xb[NTG][3][4];
        float XA[NTG], XB[NTG], SXA[NTG], SXB[NTG];
        int xtok = -1;
        int j = 0;
        for (; warp + NCW * j < n_gu; ++j) {
            const int k = warp + NCW * j;
            const int s = warp + NCW * (j & 1);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&fullb[s], (uint32_t)(j >> 1) & 1u));
            if (lane == 0 && j == 0) QMOE_TRACE(32 + warp);
            if (!ok) { if (lane == 0) { set_status(p.status, ST_TIMEOUT); misc[M_ABORT] = 1; } }
            const bool run = __all_sync(0xffffffffu, ok && misc[M_ABORT] == 0);
            if (run) {
                int u, f0, nf;
                decode(k, u, f0, nf);
                const uint8_t* slot = ring + (size_t)s * SB;
                const int q0 = used_first[u], q1 = used_first[u + 1];
                // two f rows at a time: gate f, gate f+1, up f, up f+1 interleaved
                // per lane (four independent FMA chains), then one transposed
                // butterfly reduces the four sums together
                for (int qi = q0; qi < q1; ++qi) {
                    const int pr = pairs[qi];
                    const int t = pr / K;
                    if (t != xtok) {
                        xtok = t;
#pragma unroll
                        for (int jt = 0; jt < NTG; ++jt) {
                            const int tsk = lane + 32 * jt;
                            const int sb = tsk >> 3, pc = tsk & 7;
                            if (tsk < 8 * NSB_G) {
                                const int col = QK * sb + 64 * (pc >> 1) + 16 * (pc & 1);
                                const int ga = t * (H / 16) + col / 16, gb = ga + 2;
                                const int4* pa = reinterpret_cast<const int4*>(xq + 12 * ga);
                                const int4* pb = reinterpret_cast<const int4*>(xq + 12 * gb);
#pragma unroll
                                for (int pl = 0; pl < 3; ++pl) {
                                    const int4 va = pa[pl], vb = pb[pl];
                                    xa[jt][pl][0] = va.x; xa[jt][pl][1] = va.y; xa[jt][pl][2] = va.z; xa[jt][pl][3] = va.w;
                                    xb[jt][pl][0] = vb.x; xb[jt][pl][1] = vb.y; xb[jt][pl][2] = vb.z; xb[jt][pl][3] = vb.w;
                                }
                                XA[jt] = xsum[ga];
                                XB[jt] = xsum[gb];
                                SXA[jt] = xscale[ga];
                                SXB[jt] = xscale[gb];
                            }
                        }
                    }
                    if (lane == 0 && warp == 0 && j == 0) QMOE_TRACE(10);
                    for (int i = 0; i < nf; ++i) {
                        // gate row i and up row i, all of this lane's pieces at once
                        float g = 0.f, v = 0.f;
                        uint4 hd[2 * NTG], qd[2 * NTG];
#pragma unroll
                        for (int z = 0; z < 2 * NTG; ++z) {
                            const int jt = z >> 1, tsk = lane + 32 * jt;
                            if (tsk < 8 * NSB_G) {
                                const int sb = tsk >> 3, pc = tsk & 7;
                                const int row = (z & 1) ? nf + i : i;
                                const uint8_t* b = slot + row * RBG + sb * Q4K_BYTES;
                                hd[z] = *reinterpret_cast<const uint4*>(b);
                                qd[z] = *reinterpret_cast<const uint4*>(b + 16 + 16 * pc);
                            }
                        }
#pragma unroll
                        for (int z = 0; z < 2 * NTG; ++z) {
                            const int jt = z >> 1, tsk = lane + 32 * jt;
                            if (tsk < 8 * NSB_G) {
                                const int pc = tsk & 7;
                                float QA, QB;
                                q4_piece_dp4a(qd[z], xa[jt], xb[jt], SXA[jt], SXB[jt], QA, QB);
                                const float c = q4_piece_finish_exact(hd[z], pc, QA, QB, XA[jt], XB[jt]);
                                if (z & 1) v += c; else g += c;
                            }
                        }
                        // lanes 0-15 end with the gate sum, lanes 16-31 with the up sum
                        const bool h16 = lane & 16;
                        float m = (h16 ? v : g) + __shfl_xor_sync(0xffffffffu, h16 ? g : v, 16);
                        m += __shfl_xor_sync(0xffffffffu, m, 8);
                        m += __shfl_xor_sync(0xffffffffu, m, 4);
                        m += __shfl_xor_sync(0xffffffffu, m, 2);
                        m += __shfl_xor_sync(0xffffffffu, m, 1);
                        const float upv = __shfl_down_sync(0xffffffffu, m, 16);
                        if (lane == 0) p.act[(size_t)pr * F + f0 + i] = m / (1.f + expf(-m)) * upv;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (warp == 0 && j == 0) QMOE_TRACE(9);
                issue(j + 2);
            }
        }
        // this warp's act rows are written: publish them once (every writing lane
        // fences its own stores), then count the warp in; the last warp of the
        // CTA arrives at the grid barrier
        if (j > 0) {
            __threadfence();
            __syncwarp();
            if (lane == 0 && atomicAdd(&misc[M_GUDONE], 1) == misc[M_GUWARPS] - 1)
                grid_arrive(&p.bar[1]);
        }
        if (lane == 0) QMOE_TRACE(16 + warp);
        named_bar(1, NCW * 32);
        if (tid == 0) QMOE_TRACE(4);
        if (tid == 0 && misc[M_ABORT] == 0) {
            if (!grid_wait(&p.bar[1], (unsigned)G)) {
                set_status(p.status, ST_TIMEOUT);
                misc[M_ABORT] = 1;
            }
        }
        named_bar(1, NCW * 32);
        if (tid == 0) QMOE_TRACE(5);

        // ---------------- phase D prologue: group sums of act (8 for Q6_K, 16 for Q4_K)
        constexpr int GS = DQT == 1 ? 16 : 8;
        float* asum = x_s;                                       // x is no longer needed
        const bool live = misc[M_ABORT] == 0;
        float* act_s = L.act_stage >= 0 ? reinterpret_cast<float*>(sm + L.off_x + L.act_stage) : nullptr;
        if (live)
            for (int i = tid; i < P * (F / GS); i += NCW * 32) {
                const float4* a4 = reinterpret_cast<const float4*>(p.act + (size_t)i * GS);
                float s = 0.f;
#pragma unroll
                for (int z = 0; z < GS / 4; ++z) {
                    const float4 q = a4[z];
                    s += (q.x + q.y) + (q.z + q.w);
                    if (act_s) reinterpret_cast<float4*>(act_s + (size_t)i * GS)[z] = q;
                }
                asum[i] = s;
            }
        named_bar(1, NCW * 32);
        if (tid == 0) QMOE_TRACE(6);

        // ---------------- phase D: down rows of every used expert
        const int H0 = misc[M_H0];
        const int rr = lane >> 3, kk = lane & 7;
        for (; warp + NCW * j < n_ch; ++j) {
            const int k = warp + NCW * j;
            const int s = warp + NCW * (j & 1);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&fullb[s], (uint32_t)(j >> 1) & 1u));
            if (!ok) { if (lane == 0) { set_status(p.status, ST_TIMEOUT); misc[M_ABORT] = 1; } }
            if (__all_sync(0xffffffffu, ok && misc[M_ABORT] == 0)) {
                int u, r0, nr;
                decode(k, u, r0, nr);
                const int e = used_e[u];
                const uintptr_t src = reinterpret_cast<uintptr_t>(p.down + (size_t)e * H * RBD + (size_t)r0 * RBD);
                const uint8_t* slot = ring + (size_t)s * SB + (src & 15);
                const int q0 = used_first[u], q1 = used_first[u + 1];
                for (int qi = q0; qi < q1; ++qi) {
                    const int pr = pairs[qi];
                    const float* a = (act_s ? act_s : p.act) + (size_t)pr * F;
                    const float* as = asum + (size_t)pr * (F / GS);
                    for (int rb = 0; rb < nr; rb += 4) {
                        const int r = rb + rr;
                        float acc = 0.f;
                        if (r < nr) {
                            const uint8_t* row = slot + (size_t)r * RBD;
#pragma unroll
                            for (int sb = 0; sb < NSB_D; ++sb) {
                                if (DQT == 2) {
                                    const int n = kk >> 2, m = kk & 3;
                                    const uint8_t* blk = row + sb * Q6K_BYTES;
                                    const uint2 qa = lds8_a2(blk + 64 * n + 8 * m);
                                    const uint2 qb = lds8_a2(blk + 64 * n + 32 + 8 * m);
                                    const uint2 qh = lds8_a2(blk + 128 + 32 * n + 8 * m);
                                    const uint2 scw = lds8_a2(blk + 192 + 8 * n);
                                    const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                                    const int sb0 = (m >> 1) * 8;
                                    const float* ab = a + QK * sb + 128 * n + 8 * m;
                                    const float* asb = as + (QK * sb + 128 * n + 8 * m) / 8;
#pragma unroll
                                    for (int g = 0; g < 4; ++g) {
                                        const int bo = sb0 + 16 * g;
                                        const uint32_t sw = bo < 32 ? (scw.x >> bo) : (scw.y >> (bo - 32));
                                        const float sc = (float)(int8_t)(sw & 0xFF);
                                        float p0 = 0.f, p1 = 0.f;
#pragma unroll
                                        for (int hf = 0; hf < 2; ++hf) {
                                            const uint32_t A = hf ? qa.y : qa.x, B = hf ? qb.y : qb.x;
                                            const uint32_t Hh = hf ? qh.y : qh.x;
                                            uint32_t q6;
                                            if (g == 0) q6 = (A & 0x0F0F0F0Fu) | ((Hh << 4) & 0x30303030u);
                                            else if (g == 1) q6 = (B & 0x0F0F0F0Fu) | ((Hh << 2) & 0x30303030u);
                                            else if (g == 2) q6 = ((A >> 4) & 0x0F0F0F0Fu) | (Hh & 0x30303030u);
                                            else q6 = ((B >> 4) & 0x0F0F0F0Fu) | ((Hh >> 2) & 0x30303030u);
                                            const float4 xv = *reinterpret_cast<const float4*>(ab + 32 * g + 4 * hf);
                                            fma2(p0, p1, mag<0>(q6), mag<1>(q6), xv.x, xv.y);
                                            fma2(p0, p1, mag<2>(q6), mag<3>(q6), xv.z, xv.w);
                                        }
                                        acc = fmaf(d * sc, fmaf(256.f, p0 + p1, -160.f * asb[4 * g]), acc);
                                    }
                                } else {
                                    const int pc = kk;
                                    const uint8_t* blk = row + sb * Q4K_BYTES;
                                    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                                    const uint4 q = *reinterpret_cast<const uint4*>(blk + 16 + 16 * pc);
                                    const int col = QK * sb + 64 * (pc >> 1) + 16 * (pc & 1);
                                    float4 va[4], vb[4];
#pragma unroll
                                    for (int z = 0; z < 4; ++z) {
                                        va[z] = *reinterpret_cast<const float4*>(a + col + 4 * z);
                                        vb[z] = *reinterpret_cast<const float4*>(a + col + 32 + 4 * z);
                                    }
                                    float PA, PB;
                                    q4_piece_regs(q, va, vb, PA, PB);
                                    acc += q4_piece_finish(hdr, pc, PA, PB, as[col / 16], as[col / 16 + 2]);
                                }
                            }
                        }
                        acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                        if (r < nr && kk == 0) ybuf[pr * L.rows_max + (r0 - H0) + r] = acc;
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && warp == 0) QMOE_TRACE(15);
            if (lane == 0) issue(j + 2);
        }
        if (lane == 0) QMOE_TRACE(48 + warp);
        named_bar(1, NCW * 32);
        if (tid == 0) QMOE_TRACE(7);
        // ---------------- combine into the residual
        if (misc[M_ABORT] == 0) {
            const int nrows = misc[M_NROWS];
            const float* res = p.res ? p.res : p.x;
            for (int i = tid; i < T * nrows; i += NCW * 32) {
                const int t = i / nrows, r = i % nrows, h = H0 + r;
                float acc = res[(size_t)t * H + h];
                for (int jj = 0; jj < K; ++jj)
                    acc = fmaf(wts_s[t * K + jj], ybuf[(t * K + jj) * L.rows_max + r], acc);
                p.out[(size_t)t * H + h] = acc;
            }
        }
    }
    __syncthreads();
    if (tid == 0) QMOE_TRACE(8);
    if (tid == 0) {
        // the last CTA out resets the grid-barrier counters for the next launch
        __threadfence();
        if (atomicAdd(&p.bar[2], 1u) == (unsigned)G - 1) {
            atomicExch(&p.bar[0], 0u);
            atomicExch(&p.bar[1], 0u);
            atomicExch(&p.bar[2], 0u);
        }
    }
}

struct Variant {
    int nsb_g, nsb_d, dqt;
    const void* fn;
};

template <int A, int B, int C>
const void* kfn() { return reinterpret_cast<const void*>(&moe_decode_fused<A, B, C>); }

const Variant kVariants[] = {
    {8, 3, 2, kfn<8, 3, 2>()}, {8, 3, 1, kfn<8, 3, 1>()},
    {1, 1, 2, kfn<1, 1, 2>()}, {1, 1, 1, kfn<1, 1, 1>()},
};

const Variant* find_variant(int H, int F, int down_t) {
    for (const Variant& v : kVariants)
        if (v.nsb_g == H / QK && v.nsb_d == F / QK && v.dqt == down_t) return &v;
    return nullptr;
}

constexpr int SLOT_BYTES_TARGET = 4608;

int slot_bytes_for(int H, int F, int down_t) {
    const int rbg = (H / QK) * Q4K_BYTES;
    const int rbd = (F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    int sb = SLOT_BYTES_TARGET;
    if (sb < 2 * rbg) sb = 2 * rbg;                       // at least one f per gate/up chunk
    if (sb < rbd + 32) sb = al(rbd + 32, 16);
    return al(sb, 128);
}

}  // namespace

// Host side: can the fused kernel run this shape, and with how much shared memory?
bool fused_decode_plan(const MoeShape& s, int gate_t, int up_t, int down_t, int num_sms,
                       FusedPlan* plan) {
    if (s.T < 1 || s.T > MAXT || s.T * s.K > MAXP) return false;
    if (gate_t != 1 || up_t != 1) return false;
    const Variant* v = find_variant(s.H, s.F, down_t);
    if (!v) return false;
    const int G = num_sms;
    const int rows_max = (s.H + G - 1) / G;
    const int sb = slot_bytes_for(s.H, s.F, down_t);
    const int gs = down_t == 1 ? 16 : 8;
    const int asum_bytes = s.T * s.K * (s.F / gs) * 4;
    bool stage = true;
    SmemLayout L = fused_layout(s.T, s.H, s.K, s.F, rows_max, sb, asum_bytes, stage);
    if (L.total > 227 * 1024) {
        stage = false;
        L = fused_layout(s.T, s.H, s.K, s.F, rows_max, sb, asum_bytes, stage);
    }
    if (L.total > 227 * 1024) return false;
    plan->stage_act = stage;
    const int rbg = (s.H / QK) * Q4K_BYTES;
    const int rbd = (s.F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    // f rows per gate/up chunk: one when a row pair is already >= 2 KB (finer
    // split of a CTA's share over its warps), else the largest power of two
    // that fits the slot and divides F
    int cf = sb / (2 * rbg);
    int p2 = 1;
    while (p2 * 2 <= cf && s.F % (p2 * 2) == 0) p2 *= 2;
    cf = rbg >= 1024 ? 1 : p2;
    if (cf < 1 || (sb - 32) / rbd < 1) return false;
    plan->cf = cf;
    if (s.E > 1024) return false;
    if (s.T * (s.H / 16) > 2 * NTHREADS) return false;       // x byte-plane conversion share
    plan->grid = G;
    plan->smem = L.total;
    plan->fn = v->fn;
    plan->rows_max = rows_max;
    plan->slot_bytes = sb;
    plan->asum_bytes = asum_bytes;
    return true;
}

cudaError_t launch_fused_decode(const MoeShape& s, const FusedPlan& plan, const float* x,
                                const float* res, const float* bias, const float* router,
                                const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                                float* out, int32_t* ids_out, float* w_out, float* logits,
                                float* act, unsigned* bar, int* status, cudaStream_t st) {
    FusedParams p;
    p.x = x; p.res = res; p.bias = bias; p.router = router;
    p.gate = gate; p.up = up; p.down = down;
    p.out = out; p.ids_out = ids_out; p.w_out = w_out;
    p.logits = logits; p.act = act; p.bar = bar; p.status = status;
    p.T = s.T; p.H = s.H; p.E = s.E; p.K = s.K; p.F = s.F; p.norm = s.norm_topk;
    p.cf = plan.cf;
    p.L = fused_layout(s.T, s.H, s.K, s.F, plan.rows_max, plan.slot_bytes, plan.asum_bytes,
                       plan.stage_act);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, plan.fn, args);
}

int fused_threads() { return NTHREADS; }

#ifdef QMOE_PHASE_TRACE
extern "C" int qmoe_trace_read(unsigned long long* host, int n) {
    return (int)cudaMemcpyFromSymbol(host, g_qmoe_trace, sizeof(unsigned long long) * n);
}
#endif

// Allow every fused variant the full 227 KB of dynamic shared memory (once per
// device context) and check that one CTA fits on an SM.
cudaError_t fused_prepare() {
    for (const Variant& v : kVariants) {
        cudaError_t e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        int nb = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, v.fn, NTHREADS, 227 * 1024);
        if (e != cudaSuccess) return e;
        if (nb < 1) return cudaErrorInvalidConfiguration;
    }
    return cudaSuccess;
}

}  // namespace qmoe
