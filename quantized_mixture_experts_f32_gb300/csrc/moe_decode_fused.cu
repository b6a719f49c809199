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
// Structure (G CTAs of 16 warps, all co-resident: cooperative launch).  Values
// that cross CTAs travel as 64-bit words {value, launch tag}: a reader polls
// until the word carries this launch's tag, so no grid barrier, fence or
// counter sits between the phases (the tag is one more than the one the last
// CTA of the previous launch published).
//  A  every CTA stages x in shared memory; CTA c computes the router logits of
//     experts c, c+G, ... (fixed-order reductions) and stores them tagged.
//  B  every CTA waits for the T*E logits, redoes the (cheap, deterministic)
//     top-k of all T tokens and builds the same per-expert pair lists; it then
//     owns a contiguous share of the (expert, f) gate/up rows and a contiguous
//     share of the used experts' down rows (rows weighted by 1 + the expert's
//     pair count, so a few experts at most), cut into chunks of a few KB.
//  C  warp w handles chunks w, w+16, ... and streams them itself with bulk async
//     copies (TMA) into its ring slots, several chunks ahead of the one it
//     computes (one issuing thread per CTA cannot keep HBM busy; sixteen can).
//     Gate/up chunks produce act[p][f] = silu(g)*u, stored tagged; the down
//     chunks are already in flight meanwhile.
//  D  the CTA waits for act of its down experts only, then y[p][h] = Wd_e act
//     for its down rows, stored tagged.
//  E  CTA c owns out rows [H*c/G, H*(c+1)/G): out[t][h] = res[t][h] + sum_j
//     w[t][j] y[t*K+j][h] in slot order j = 0..K-1 (deterministic, no atomics
//     on values).
// Every wait is bounded (%globaltimer); on expiry the kernel records
// QMOE_ERR_TIMEOUT, stops computing, drains its own copies and exits.
#include <math.h>

#include "kquant.cuh"
#include "ptx_sync.cuh"
#include "qmoe_internal.h"

#ifdef QMOE_PHASE_TRACE
// per-CTA phase timestamps (%globaltimer), compiled only into diagnostic builds
__device__ unsigned long long g_qmoe_trace[1024 * 128];
#define QMOE_TRACE(slot)                                                            \
    do {                                                                            \
        g_qmoe_trace[blockIdx.x * 128 + (slot)] = qmoe::globaltimer();              \
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
constexpr int NSMAX = 8;                    // ring slots per warp, at most
constexpr int NSLOT = NSMAX * NCW;
constexpr int MAXT = 8;
constexpr int MAXP = 128;

// misc int slots
constexpr int MAXSEG = 8;                   // experts a CTA's down rows may span
enum { M_NUSED = 0, M_NCH, M_NGU, M_ABORT, M_GULO, M_TAG, M_NSEG, M_QBASE, M_NLOC,
       M_SEG = 16,                          // + 4*s: expert slot u, first row, rows, first chunk
       M_COUNT = M_SEG + 4 * MAXSEG };

struct SmemLayout {
    int off_bar, off_misc, off_red, off_ids, off_wts, off_used, off_first, off_pairs,
        off_x, off_xsum, off_xscale, off_ring, total, slot_bytes, ns, asum_off;
};

__host__ __device__ inline int al(int v, int a) { return (v + a - 1) / a * a; }

// Staged act index with 4 floats of padding after every 128: the two
// half-superblocks that the 8 lanes of a down row read at once then use
// different banks.
__host__ __device__ __forceinline__ int apad(int f) { return f + 4 * (f >> 7); }

// nloc_max: pairs of the experts one CTA's down rows can touch
__host__ __device__ inline SmemLayout fused_layout(int T, int H, int K, int F, int nloc_max,
                                                   int slot_bytes, int ns) {
    SmemLayout L;
    const int P = T * K;
    // after gate/up the x region holds act of this CTA's down experts and the
    // group sums of act (groups of 8 or 16; sized for 8)
    const int act_bytes = al(nloc_max * apad(F) * 4, 16);
    const int asum_bytes = al(nloc_max * (F / 8) * 4, 16);
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
    L.off_x = o;        o += al(T * H * 4 > act_bytes + asum_bytes ? T * H * 4 : act_bytes + asum_bytes, 16);
    L.off_xsum = o;     o += al(T * (H / 16) * 4, 16);
    L.off_xscale = o;   o += al(T * (H / 16) * 4, 16);
    o = al(o, 128);
    L.off_ring = o;     o += NCW * ns * slot_bytes;
    L.total = o;
    L.slot_bytes = slot_bytes;
    L.ns = ns;
    L.asum_off = act_bytes;
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
    unsigned long long* lg;     // [T][E] tagged router logits
    unsigned long long* act;    // [P][F] tagged silu(g)*u
    unsigned long long* y;      // [P][H] tagged down outputs
    unsigned long long* xflag;  // [G] tagged "x staged" marks (only when out aliases x)
    unsigned* ctl;              // [0] exit counter, [1] tag of the last completed launch
    int* status;
    const float* norm_w;        // nullable: x is RMS-normalised per token and scaled first
    float eps;
    unsigned long long wait_ns; // limit of every cross-CTA wait
    int stall;                  // test hook: the logits wait expects a tag no CTA writes
    int T, H, E, K, F, norm, x_alias;
    int cf;          // f rows per gate/up chunk (divides F)
    SmemLayout L;
};

// ----------------------------------------------------------------------------- small helpers

__device__ __forceinline__ void set_status(int* status, int code) { atomicCAS(status, 0, code); }

// N tagged values base[first + z*stride] (those below n): all loads in flight
// together, then the ones not yet carrying `tag` are reloaded together until
// they do (bounded).  Missing values read as 0; false if the wait timed out.
template <int N>
__device__ __forceinline__ bool load_tagged(const unsigned long long* base, int n, int first,
                                            int stride, unsigned tag, float (&v)[N],
                                            unsigned long long limit_ns = WAIT_LIMIT_NS) {
    uint32_t pend = 0u;                                   // bit z: value z still to come
#pragma unroll
    for (int z = 0; z < N; ++z) {
        v[z] = 0.f;
        if (first + z * stride < n) pend |= 1u << z;
    }
    unsigned long long t0 = 0ull;
    for (int round = 0; pend; ++round) {
        if (round == 1) t0 = globaltimer();
        if (round > 1) {
            if (globaltimer() - t0 > limit_ns) return false;
            __nanosleep(32);
        }
        unsigned long long w[N];
#pragma unroll
        for (int z = 0; z < N; ++z)
            w[z] = (pend >> z) & 1u ? ld_relaxed_u64(base + first + z * stride) : 0ull;
#pragma unroll
        for (int z = 0; z < N; ++z)
            if (((pend >> z) & 1u) && (unsigned)(w[z] >> 32) == tag) {
                v[z] = __uint_as_float((unsigned)w[z]);
                pend &= ~(1u << z);
            }
    }
    return true;
}

// 8 bytes at an even shared-memory address (three aligned words, funnel shift)
__device__ __forceinline__ uint2 lds8_a2(const uint8_t* p) {
    const uint32_t off = smem_u32(p) & 3u;
    const uint32_t* b = reinterpret_cast<const uint32_t*>(p - off);   // stays a shared pointer
    const uint32_t sh = off * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2];
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// 16 bytes at an even shared-memory address (five aligned words, funnel shift)
__device__ __forceinline__ uint4 lds16_a2(const uint8_t* p) {
    const uint32_t off = smem_u32(p) & 3u;
    const uint32_t* b = reinterpret_cast<const uint32_t*>(p - off);   // stays a shared pointer
    const uint32_t sh = off * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2], w3 = b[3], w4 = b[4];
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                      __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
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
    constexpr int NTG = 2;                                        // 16-byte pieces per lane (one chunk)
    static_assert(NSB_G <= 8, "one 32-byte chunk per lane covers at most 8 superblocks");
    constexpr int GS = DQT == 1 ? 16 : 8;                         // act group of one down scale
    const int FPAD = apad(F);                                     // staged act row (padded)
    constexpr int RPASS = 3;                                      // row passes of 4 per down chunk

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
    float* act_s = x_s;                                            // after gate/up: act, group sums
    float* asum = reinterpret_cast<float*>(sm + L.off_x + L.asum_off);
    uint8_t* ring = sm + L.off_ring;
    const int SB = L.slot_bytes;
    const int NS = L.ns;

    // ---------------- phase A: stage x, router slice -> tagged logits
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
        for (int s = 0; s < NCW * NS; ++s) mbar_init(&fullb[s], 1);
        for (int i = 0; i < M_COUNT; ++i) misc[i] = 0;
        misc[M_TAG] = (int)(ld_acquire_gpu(p.ctl + 1) + 1u);   // this launch's tag
        fence_barrier_init();
    }
    __syncthreads();
    const unsigned tag = (unsigned)misc[M_TAG];
    if (p.x_alias && tid == 0) st_relaxed_u64(p.xflag + c, tag_pack(0.f, tag));   // x is staged
    if (p.norm_w) {
        // x = x / sqrt(mean(x^2) + eps) * norm_w, per token (every CTA redoes it)
        for (int t = 0; t < T; ++t) {
            float ss = 0.f;
            for (int i = tid; i < H; i += NTHREADS) ss = fmaf(x_s[t * H + i], x_s[t * H + i], ss);
            ss = warp_sum(ss);
            if (lane == 0) red[warp * MAXT + t] = ss;
        }
        __syncthreads();
        for (int i = tid; i < T * H; i += NTHREADS) {
            const int t = i / H;
            float tot = 0.f;
            for (int w = 0; w < NCW; ++w) tot += red[w * MAXT + t];
            x_s[i] = x_s[i] * rsqrtf(tot / (float)H + p.eps) * p.norm_w[i - t * H];
        }
        __syncthreads();
    }
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
            st_relaxed_u64(p.lg + (size_t)tid * E + e, tag_pack(s + (p.bias ? p.bias[e] : 0.f), tag));
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
    if (tid == 0) QMOE_TRACE(1);

    // ---------------- phase B: routing (identical in every CTA).  Wait for all
    // logits of this launch, rank every logit, then in parallel the softmax
    // weights (warp t), each pair's place in the expert-sorted pair list
    // (threads 256..) and, in the last warp, the used-expert list and this
    // CTA's share of the work, so that the weight copies start right after.
    float* lg_s = reinterpret_cast<float*>(ring);                 // ring is idle until phase C
    int32_t* sel = reinterpret_cast<int32_t*>(lg_s + T * E);      // [T][K]
    int32_t* keys = sel + P;                                      // [T][E] order keys
    {
        constexpr int LPT = 2;                                     // logits per thread (T*E <= 1024)
        float v[LPT];
        // (the test hook waits for a tag that no CTA writes, so the wait runs out)
        const unsigned want = p.stall ? (tag ^ 0x80000000u) : tag;
        if (!load_tagged<LPT>(p.lg, T * E, tid, NTHREADS, want, v, p.wait_ns)) {
            set_status(p.status, ST_TIMEOUT);
            misc[M_ABORT] = 1;
        }
#pragma unroll
        for (int z = 0; z < LPT; ++z)
            if (tid + z * NTHREADS < T * E) {
                lg_s[tid + z * NTHREADS] = v[z];
                keys[tid + z * NTHREADS] = order_key(v[z]);
            }
    }
    for (int i = tid; i < P; i += NTHREADS) sel[i] = 0;
    __syncthreads();
    if (tid == 0) QMOE_TRACE(2);
    const bool abort_b = misc[M_ABORT] != 0;
    if (!abort_b && E <= 128) {
        // up to 128 experts: warp t selects token t's top-k.  Lane l sorts the
        // (order key, index) pairs of experts l, l + 32, l + 64, l + 96 (larger
        // key first, ties to the lower index); then K tournament rounds over the
        // 32 lane heads: the largest head key by one warp max-reduction, the
        // lowest index holding it by one min-reduction, the owner drops its head
        if (warp < T) {
            const int* l = keys + warp * E;
            int ks[4], is[4];
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                const int i = lane + 32 * z;
                ks[z] = i < E ? l[i] : INT_MIN;
                is[z] = i < E ? i : INT_MAX;
            }
            auto cswap = [&](int x, int y) {
                if (ks[y] > ks[x] || (ks[y] == ks[x] && is[y] < is[x])) {
                    const int tk = ks[x], ti = is[x];
                    ks[x] = ks[y];
                    is[x] = is[y];
                    ks[y] = tk;
                    is[y] = ti;
                }
            };
            cswap(0, 1);
            cswap(2, 3);
            cswap(0, 2);
            cswap(1, 3);
            cswap(1, 2);
            for (int r = 0; r < K; ++r) {
                const int mk = __reduce_max_sync(0xffffffffu, ks[0]);
                const int wi = (int)__reduce_min_sync(0xffffffffu, ks[0] == mk ? (unsigned)is[0] : 0xffffffffu);
                if (lane == 0) sel[warp * K + r] = wi;
                if ((wi & 31) == lane) {
                    ks[0] = ks[1];
                    ks[1] = ks[2];
                    ks[2] = ks[3];
                    ks[3] = INT_MIN;
                    is[0] = is[1];
                    is[1] = is[2];
                    is[2] = is[3];
                    is[3] = INT_MAX;
                }
            }
        }
    } else if (!abort_b) {
        // rank of every logit among its token's E (ties: lower index first);
        // tpe consecutive lanes share one logit's E comparisons
        const int nel = T * E;
        int tpe = NTHREADS / nel;
        tpe = tpe >= 32 ? 32 : tpe >= 16 ? 16 : tpe >= 8 ? 8 : tpe >= 4 ? 4 : tpe >= 2 ? 2 : 1;
        if (tpe > 1) {
            const int i = tid / tpe, sub = tid - (tid / tpe) * tpe;
            const bool valid = i < nel;
            const int t = valid ? i / E : 0, e = valid ? i - t * E : 0;
            const int* l = keys + t * E;
            const int v = l[e];
            int rank = 0;
#pragma unroll 8
            for (int e2 = sub; e2 < E; e2 += tpe) {
                const int w = l[e2];
                rank += (w > v) || (w == v && e2 < e);
            }
            for (int o = tpe >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
            if (valid && sub == 0 && rank < K) sel[t * K + rank] = e;
        } else {
            for (int i = tid; i < nel; i += NTHREADS) {
                const int t = i / E, e = i - t * E;
                const int* l = keys + t * E;
                const int v = l[e];
                int rank = 0;
#pragma unroll 8
                for (int e2 = 0; e2 < E; ++e2) {
                    const int w = l[e2];
                    rank += (w > v) || (w == v && e2 < e);
                }
                if (rank < K) sel[t * K + rank] = e;
            }
        }
    }
    if (tid == 0) QMOE_TRACE(11);
    __syncthreads();
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
    }
    if (warp == NCW - 1) {
        // used experts in ascending id order: lane owns bitmap word `lane` (E <= 1024)
        uint32_t word = 0u;
        if (!abort_b)
            for (int q = 0; q < P; ++q) {
                int e = sel[q];
                e = (e < 0 || e >= E) ? 0 : e;
                if ((e >> 5) == lane) word |= 1u << (e & 31);
            }
        const int cw = __popc(word);
        int incl = cw;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        const int nu = __shfl_sync(0xffffffffu, incl, 31);
        int u = incl - cw;
        for (uint32_t w = word; w; w &= w - 1u) used_e[u++] = lane * 32 + __ffs(w) - 1;
        __syncwarp();
        // Start the selected experts' bytes moving now: CTA c prefetches into L2
        // its 1/G share of the concatenated (gate, up, down) slices of the used
        // experts; the bulk copies issued after the split then find them there.
        {
            const long long gu_b = (long long)F * RBG, dn_b = (long long)H * RBD;
            const long long per = 2 * gu_b + dn_b, tot = per * nu;
            const long long lo = tot * c / G, hi = tot * (c + 1) / G;
            for (int piece = lane; piece < 3 * nu; piece += 32) {
                const int uu = piece / 3, part = piece - 3 * uu;
                const long long p0 = per * uu + (part == 0 ? 0 : part == 1 ? gu_b : 2 * gu_b);
                const long long p1 = p0 + (part == 2 ? dn_b : gu_b);
                const long long a0 = lo > p0 ? lo : p0, a1 = hi < p1 ? hi : p1;
                if (a1 > a0) {
                    const int e = used_e[uu];
                    const uint8_t* base = part == 0 ? p.gate + (size_t)e * gu_b
                                        : part == 1 ? p.up + (size_t)e * gu_b
                                                    : p.down + (size_t)e * dn_b;
                    const long long o0 = (a0 - p0) & ~15ll, o1 = ((a1 - p0) + 15) & ~15ll;
                    const long long len = (o1 < p1 - p0 ? o1 : p1 - p0) - o0;
                    if (len > 0) bulk_prefetch_l2(base + o0, (uint32_t)(len & ~15ll));
                }
            }
        }
        // first pair of used expert u = number of pairs with a smaller expert id
        for (int uu = lane; uu < nu; uu += 32) {
            const int e = used_e[uu];
            int before = 0;
            for (int q = 0; q < P; ++q) {
                int e2 = sel[q];
                e2 = (e2 < 0 || e2 >= E) ? 0 : e2;
                before += e2 < e;
            }
            used_first[uu] = before;
        }
        if (lane == 0) used_first[nu] = P;
        __syncwarp();
        // Work of this CTA, in closed form.  Gate/up: the used experts' f rows
        // are cut into global chunks of CF consecutive f (CF divides F); CTA c
        // owns global chunks [c*NG/G, (c+1)*NG/G).  Down: the used experts'
        // rows in expert order, each weighted by 1 + the expert's pair count
        // (one row load, one dot product per pair); CTA c owns the rows whose
        // weighted position falls in [c*W/G, (c+1)*W/G): a few experts at most.
        const int RPC = min((SB - 32) / RBD, DQT == 2 ? 8 : 4 * RPASS);
        {
            const long long W = (long long)H * (P + nu);
            const long long wlo = W * c / G, whi = W * (c + 1) / G;
            long long base = 0;
            int nseg = 0;
            bool over = false;
            for (int u0 = 0; u0 < nu; u0 += 32) {
                const int u = u0 + lane;
                const int wu = u < nu ? used_first[u + 1] - used_first[u] + 1 : 0;
                const long long len = (long long)H * wu;
                long long incl = len;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long n = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += n;
                }
                const long long U = base + incl - len;
                const bool hit = u < nu && U < whi && U + len > wlo;
                const uint32_t hm = __ballot_sync(0xffffffffu, hit);
                if (hit) {
                    const long long a = (wlo > U ? wlo : U) - U, b = (whi < U + len ? whi : U + len) - U;
                    const int ra = (int)((a + wu - 1) / wu), rb = (int)((b + wu - 1) / wu);
                    const int slot = nseg + __popc(hm & ((1u << lane) - 1u));
                    if (slot < MAXSEG) {
                        int* sg = misc + M_SEG + 4 * slot;
                        sg[0] = u;
                        sg[1] = ra;
                        sg[2] = rb - ra;
                    } else {
                        over = true;
                    }
                }
                nseg += __popc(hm);
                base += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (over) set_status(p.status, ST_DEVICE_CHECK);      // host bound broken
            __syncwarp();
            if (lane == 0) {
                misc[M_NUSED] = nu;
                if (nseg > MAXSEG) nseg = MAXSEG;
                int ndc = 0, keep = 0;
                for (int sgi = 0; sgi < nseg; ++sgi) {
                    int* sg = misc + M_SEG + 4 * sgi;
                    if (sg[2] <= 0) continue;                     // a range too short for a row
                    int* dst = misc + M_SEG + 4 * keep;
                    dst[0] = sg[0]; dst[1] = sg[1]; dst[2] = sg[2];
                    dst[3] = ndc;
                    ndc += (dst[2] + RPC - 1) / RPC;
                    ++keep;
                }
                const int CF = p.cf, CPE = F / CF;
                const int NG = nu * CPE;                             // < 2^17, NG * G < 2^31
                const int lo = NG * c / G, hi = NG * (c + 1) / G;
                misc[M_GULO] = lo;
                misc[M_NGU] = hi - lo;
                misc[M_NCH] = (hi - lo) + ndc;
                misc[M_NSEG] = keep;
                const int qb = keep ? used_first[misc[M_SEG]] : 0;
                const int qe = keep ? used_first[misc[M_SEG + 4 * (keep - 1)] + 1] : 0;
                misc[M_QBASE] = qb;
                misc[M_NLOC] = qe - qb;
            }
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
    const int gu_lo = misc[M_GULO], nseg = misc[M_NSEG];
    const int CPE = F / p.cf, RPC = min((SB - 32) / RBD, DQT == 2 ? 8 : 4 * RPASS);
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
        int sgi = 0;
        while (sgi + 1 < nseg && misc[M_SEG + 4 * (sgi + 1) + 3] <= kd) ++sgi;
        const int* sg = misc + M_SEG + 4 * sgi;
        u = sg[0];
        start = sg[1] + (kd - sg[3]) * RPC;
        cnt = min(RPC, sg[1] + sg[2] - start);
        return false;
    };

    // ---------------- phases C and D: warp w streams and computes chunks w, w+16, ...
    // chunk j of this warp lives in slot warp + 16*(j%NS); it is issued NS
    // chunks ahead, right after the chunk that used the slot before it
    auto issue = [&](int j) {                                    // lane 0 only
        const int k = warp + NCW * j;
        if (k >= n_ch) return;
        const int s = warp + NCW * (j % NS);
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
        for (int j = 0; j < NS; ++j) issue(j);
    }
    {
        // ---------------- phase C: gate/up + SwiGLU
        int xa[NTG][3][4], xb[NTG][3][4];
        float XA[NTG], XB[NTG], SXA[NTG], SXB[NTG];
        int xtok = -1;
        int j = 0;
        for (; warp + NCW * j < n_gu; ++j) {
            const int k = warp + NCW * j;
            const int s = warp + NCW * (j % NS);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&fullb[s], (uint32_t)(j / NS) & 1u));
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
                        // lane -> 32-byte chunk c of superblock sb (both its 16-byte
                        // pieces, which share one scale/min pair)
#pragma unroll
                        for (int jt = 0; jt < NTG; ++jt) {
                            if (lane < 4 * NSB_G) {
                                const int sb = lane >> 2, c = lane & 3;
                                const int col = QK * sb + 64 * c + 16 * jt;
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
                        // gate row i and up row i: this lane's chunk of each
                        float g = 0.f, v = 0.f;
                        if (lane < 4 * NSB_G) {
                            const int sb = lane >> 2, c = lane & 3;
                            uint4 hd[2], qd[2][2];
#pragma unroll
                            for (int gu = 0; gu < 2; ++gu) {
                                const uint8_t* b = slot + (gu ? nf + i : i) * RBG + sb * Q4K_BYTES;
                                hd[gu] = *reinterpret_cast<const uint4*>(b);
                                qd[gu][0] = *reinterpret_cast<const uint4*>(b + 16 + 32 * c);
                                qd[gu][1] = *reinterpret_cast<const uint4*>(b + 32 + 32 * c);
                            }
#pragma unroll
                            for (int gu = 0; gu < 2; ++gu) {
                                float QA0, QB0, QA1, QB1;
                                q4_piece_dp4a(qd[gu][0], xa[0], xb[0], SXA[0], SXB[0], QA0, QB0);
                                q4_piece_dp4a(qd[gu][1], xa[1], xb[1], SXA[1], SXB[1], QA1, QB1);
                                const float cc = q4_piece_finish_exact(hd[gu], 2 * c, QA0 + QA1, QB0 + QB1,
                                                                       XA[0] + XA[1], XB[0] + XB[1]);
                                if (gu) v += cc; else g += cc;
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
                        if (lane == 0)
                            st_relaxed_u64(p.act + (size_t)pr * F + f0 + i,
                                           tag_pack(m / (1.f + expf(-m)) * upv, tag));
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                if (warp == 0 && j == 0) QMOE_TRACE(9);
                issue(j + NS);
            }
        }
        if (lane == 0) QMOE_TRACE(16 + warp);
        named_bar(1, NCW * 32);                                  // x planes no longer read
        if (tid == 0) QMOE_TRACE(4);

        // ---------------- phase D prologue: act of this CTA's down experts (all
        // gate/up work of the grid contributes) and its group sums (8 for Q6_K,
        // 16 for Q4_K)
        const int qbase = misc[M_QBASE], nloc = misc[M_NLOC];
        if (misc[M_ABORT] == 0) {
            bool ok = true;
            for (int i = tid; i < nloc * (F / GS); i += NCW * 32) {
                const int lp = i / (F / GS), g = i - lp * (F / GS);
                const int pr = pairs[qbase + lp];
                float v[GS];
                ok = load_tagged<GS>(p.act + (size_t)pr * F + g * GS, GS, 0, 1, tag, v) && ok;
                float s = 0.f;
#pragma unroll
                for (int z = 0; z < GS; ++z) s += v[z];
#pragma unroll
                for (int z = 0; z < GS; z += 4)
                    *reinterpret_cast<float4*>(act_s + (size_t)lp * FPAD + apad(g * GS + z)) =
                        make_float4(v[z], v[z + 1], v[z + 2], v[z + 3]);
                asum[i] = s;
            }
            if (!ok) {
                set_status(p.status, ST_TIMEOUT);
                misc[M_ABORT] = 1;
            }
        }
        named_bar(1, NCW * 32);
        if (tid == 0) QMOE_TRACE(6);

        // ---------------- phase D: down rows -> tagged y
        const int rr = lane >> 3, kk = lane & 7;
        for (; warp + NCW * j < n_ch; ++j) {
            const int k = warp + NCW * j;
            const int s = warp + NCW * (j % NS);
            const bool ok = __all_sync(0xffffffffu, mbar_wait(&fullb[s], (uint32_t)(j / NS) & 1u));
            if (lane == 0 && warp + NCW * j >= n_gu && warp + NCW * (j - 1) < n_gu) QMOE_TRACE(64 + warp);
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
                    const float* a = act_s + (size_t)(qi - qbase) * FPAD;
                    const float* as = asum + (size_t)(qi - qbase) * (F / GS);
                    if (DQT == 2) {
                        // Q6_K: four lanes per row (lane = 4 r + 2 n + qq): half n of
                        // every superblock, positions l = 16 qq .. 16 qq + 15 of its four
                        // groups; every row of the chunk in one pass, each lane reading
                        // 16-byte runs of its row once; act broadcast across rows
                        const int r = lane >> 2, n = (lane >> 1) & 1, qq = lane & 1;
                        float acc = 0.f;
                        if (r < nr) {
#pragma unroll 1
                            for (int sb = 0; sb < NSB_D; ++sb) {
                                const uint8_t* blk = slot + (size_t)r * RBD + sb * Q6K_BYTES;
                                const uint4 qa = lds16_a2(blk + 64 * n + 16 * qq);
                                const uint4 qb = lds16_a2(blk + 64 * n + 32 + 16 * qq);
                                const uint4 qh = lds16_a2(blk + 128 + 32 * n + 16 * qq);
                                const uint2 scw = lds8_a2(blk + 192 + 8 * n);
                                const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                                const float* ab = a + apad(QK * sb + 128 * n) + 16 * qq;
                                const float* asb = as + (QK * sb + 128 * n + 16 * qq) / 8;
                                const uint32_t A4[4] = {qa.x, qa.y, qa.z, qa.w};
                                const uint32_t B4[4] = {qb.x, qb.y, qb.z, qb.w};
                                const uint32_t H4[4] = {qh.x, qh.y, qh.z, qh.w};
#pragma unroll
                                for (int g = 0; g < 4; ++g) {
                                    const int bo = 8 * (2 * g + qq);         // scale byte of (g, qq)
                                    const uint32_t sw = bo < 32 ? (scw.x >> bo) : (scw.y >> (bo - 32));
                                    const float sc = (float)(int8_t)(sw & 0xFF);
                                    float p0 = 0.f, p1 = 0.f;
#pragma unroll
                                    for (int wq = 0; wq < 4; ++wq) {
                                        const uint32_t Aw = A4[wq], Bw = B4[wq], Hh = H4[wq];
                                        uint32_t q6;
                                        if (g == 0) q6 = (Aw & 0x0F0F0F0Fu) | ((Hh << 4) & 0x30303030u);
                                        else if (g == 1) q6 = (Bw & 0x0F0F0F0Fu) | ((Hh << 2) & 0x30303030u);
                                        else if (g == 2) q6 = ((Aw >> 4) & 0x0F0F0F0Fu) | (Hh & 0x30303030u);
                                        else q6 = ((Bw >> 4) & 0x0F0F0F0Fu) | ((Hh >> 2) & 0x30303030u);
                                        const float4 x4 = *reinterpret_cast<const float4*>(ab + 32 * g + 4 * wq);
                                        fma2(p0, p1, mag<0>(q6), mag<1>(q6), x4.x, x4.y);
                                        fma2(p0, p1, mag<2>(q6), mag<3>(q6), x4.z, x4.w);
                                    }
                                    const float xsg = asb[4 * g] + asb[4 * g + 1];
                                    acc = fmaf(d * sc, fmaf(256.f, p0 + p1, -160.f * xsg), acc);
                                }
                            }
                        }
                        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                        if (r < nr && (lane & 3) == 0)
                            st_relaxed_u64(p.y + (size_t)pr * H + r0 + r, tag_pack(acc, tag));
                    } else {
                        // Q4_K: lane (kk) owns 16-byte piece kk of every superblock;
                        // its 32 act values are loaded once per superblock and reused
                        // for every row pass
                        const int pc = kk;
                        float acc[RPASS];
#pragma unroll
                        for (int rb = 0; rb < RPASS; ++rb) acc[rb] = 0.f;
#pragma unroll 1
                        for (int sb = 0; sb < NSB_D; ++sb) {
                            const int col = QK * sb + 64 * (pc >> 1) + 16 * (pc & 1);
                            const float* ac = a + apad(col);
                            float4 va[4], vb[4];
#pragma unroll
                            for (int z = 0; z < 4; ++z) {
                                va[z] = *reinterpret_cast<const float4*>(ac + 4 * z);
                                vb[z] = *reinterpret_cast<const float4*>(ac + 32 + 4 * z);
                            }
                            const float XA = as[col / 16], XB = as[col / 16 + 2];
#pragma unroll
                            for (int rb = 0; rb < RPASS; ++rb) {
                                const int r = 4 * rb + rr;
                                if (r < nr) {
                                    const uint8_t* blk = slot + (size_t)r * RBD + sb * Q4K_BYTES;
                                    const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                                    const uint4 q = *reinterpret_cast<const uint4*>(blk + 16 + 16 * pc);
                                    float PA, PB;
                                    q4_piece_regs(q, va, vb, PA, PB);
                                    acc[rb] += q4_piece_finish(hdr, pc, PA, PB, XA, XB);
                                }
                            }
                        }
#pragma unroll
                        for (int rb = 0; rb < RPASS; ++rb) {
                            float v = acc[rb];
                            v += __shfl_xor_sync(0xffffffffu, v, 4);
                            v += __shfl_xor_sync(0xffffffffu, v, 2);
                            v += __shfl_xor_sync(0xffffffffu, v, 1);
                            const int r = 4 * rb + rr;
                            if (r < nr && kk == 0)
                                st_relaxed_u64(p.y + (size_t)pr * H + r0 + r, tag_pack(v, tag));
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && warp + NCW * j >= n_gu && warp + NCW * (j - 1) < n_gu) QMOE_TRACE(80 + warp);
            if (lane == 0 && warp == 0) QMOE_TRACE(15);
            if (lane == 0) issue(j + NS);
        }
        if (lane == 0) QMOE_TRACE(48 + warp);
    }

    // ---------------- phase E: out rows [H*c/G, H*(c+1)/G) = residual + sum over
    // slots j (in order) of w[t][j] * y[t*K+j]
    if (p.x_alias) {
        // out aliases x: every CTA must have staged x before any row is written
        bool ok = true;
        for (int i = tid; i < G; i += NCW * 32) {
            float v;
            ok = poll_tagged(p.xflag + i, tag, v) && ok;
        }
        if (!ok) { set_status(p.status, ST_TIMEOUT); misc[M_ABORT] = 1; }
        __syncthreads();
    }
    if (tid == 0) QMOE_TRACE(7);
    if (misc[M_ABORT] == 0) {
        const int h0 = H * c / G, nrows = H * (c + 1) / G - h0;
        const float* res = p.res ? p.res : p.x;
        bool ok = true;
        for (int i = tid; i < T * nrows; i += NCW * 32) {
            const int t = i / nrows, h = h0 + (i - t * nrows);
            float yv[16];
            ok = load_tagged<16>(p.y + (size_t)t * K * H + h, K * H, 0, H, tag, yv) && ok;
            float acc = res[(size_t)t * H + h];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj)
                if (jj < K) acc = fmaf(wts_s[t * K + jj], yv[jj], acc);
            p.out[(size_t)t * H + h] = acc;
        }
        if (!ok) set_status(p.status, ST_TIMEOUT);
    }
    if (tid == 0) QMOE_TRACE(12);
    __syncthreads();
    if (tid == 0) QMOE_TRACE(8);
    if (tid == 0) {
        // the last CTA out resets the exit counter and publishes this launch's
        // tag, which the next launch increments
        if (atomicAdd(&p.ctl[0], 1u) == (unsigned)G - 1) {
            atomicExch(&p.ctl[0], 0u);
            atomicExch(&p.ctl[1], tag);
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

// Ring slot size: 4608 B (two gate+up row pairs at hidden 2048); measured
// against 2304 B slots, which put a one-token CTA's whole share in flight at
// once but double the number of copies and chunk hand-offs.
int slot_bytes_for(int T, int H, int F, int down_t) {
    (void)T;
    const int rbg = (H / QK) * Q4K_BYTES;
    const int rbd = (F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    int sb = 4608;
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
    if (s.E > 1024 || s.T * s.E > 2 * NTHREADS) return false;   // logits per thread in phase B
    if (s.T * (s.H / 16) > 2 * NTHREADS) return false;          // x byte-plane conversion share
    const int G = num_sms;
    if (G < 1 || G > 1024) return false;                      // size of the "x staged" marks
    const int P = s.T * s.K;
    // experts (and their pairs) that one CTA's share of the down rows can touch
    const int nu_max = s.E < P ? s.E : P;
    // a CTA's weighted share is at most ceil(H*(P+nu)/G); an expert weighs at
    // least 2H, so the share touches at most (P+nu)/(2G) + 2 experts
    int span = (P + nu_max + 2 * G - 1) / (2 * G) + 2;
    if (span > nu_max) span = nu_max;
    if (span > MAXSEG) return false;
    // pairs of the touched experts: the two end experts hold at most T each and
    // the fully covered ones weigh H*(pairs+1) each, at most (P+nu)/G pairs in all
    int nloc_max = 2 * s.T + (P + nu_max) / G + 1;
    if (nloc_max > P) nloc_max = P;
    const int sb = slot_bytes_for(s.T, s.H, s.F, down_t);
    // as many ring slots per warp as fit, up to NSMAX
    constexpr int SMEM_MAX = 227 * 1024;
    int ns = NSMAX;
    SmemLayout L = fused_layout(s.T, s.H, s.K, s.F, nloc_max, sb, ns);
    while (L.total > SMEM_MAX && ns > 2) L = fused_layout(s.T, s.H, s.K, s.F, nloc_max, sb, --ns);
    if (L.total > SMEM_MAX) return false;
    if (2 * s.T * s.E * 4 + P * 4 > NCW * ns * sb) return false;   // routing scratch in the ring
    const int rbg = (s.H / QK) * Q4K_BYTES;
    const int rbd = (s.F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    // f rows per gate/up chunk: the largest power of two that fits the slot and
    // divides F; one token keeps single-row chunks (a CTA's share of ~40 rows
    // then spreads over its 16 warps at 2-3 rows each instead of 2-4)
    int cf = 1;
    while (s.T > 1 && 2 * (2 * cf) * rbg <= sb && s.F % (2 * cf) == 0) cf *= 2;
    if (cf < 1 || (sb - 32) / rbd < 1) return false;
    plan->cf = cf;
    plan->ns = ns;
    plan->nloc_max = nloc_max;
    plan->grid = G;
    plan->smem = L.total;
    plan->fn = v->fn;
    plan->slot_bytes = sb;
    return true;
}

size_t fused_bufs_bytes(int T, int H, int E, int K, int F, int grid) {
    const size_t P = (size_t)T * K;
    auto a = [](size_t v) { return (v + 255) / 256 * 256; };
    return a(8 * (size_t)T * E) + a(8 * P * F) + a(8 * P * H) + a(8 * (size_t)grid) +
           a(4 * (size_t)K * F);
}

FusedBufs fused_bufs_carve(unsigned char* base, int T, int H, int E, int K, int F, int grid,
                           unsigned* ctl, int* status) {
    const size_t P = (size_t)T * K;
    auto a = [](size_t v) { return (v + 255) / 256 * 256; };
    FusedBufs b;
    size_t o = 0;
    b.lg = reinterpret_cast<unsigned long long*>(base + o);
    o += a(8 * (size_t)T * E);
    b.act = reinterpret_cast<unsigned long long*>(base + o);
    o += a(8 * P * F);
    b.y = reinterpret_cast<unsigned long long*>(base + o);
    o += a(8 * P * H);
    b.xflag = reinterpret_cast<unsigned long long*>(base + o);
    o += a(8 * (size_t)grid);
    b.plain_act = reinterpret_cast<float*>(base + o);
    b.ctl = ctl;
    b.status = status;
    return b;
}

cudaError_t launch_fused_decode(const MoeShape& s, const FusedPlan& plan, const float* x,
                                const float* res, const float* bias, const float* router,
                                const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                                float* out, int32_t* ids_out, float* w_out, const FusedBufs& b,
                                const float* norm_w, float eps, cudaStream_t st,
                                const FusedDebug* dbg) {
    FusedParams p;
    p.norm_w = norm_w;
    p.eps = eps;
    p.wait_ns = dbg ? dbg->wait_ns : WAIT_LIMIT_NS;
    p.stall = dbg ? dbg->stall : 0;
    p.x = x; p.res = res; p.bias = bias; p.router = router;
    p.gate = gate; p.up = up; p.down = down;
    p.out = out; p.ids_out = ids_out; p.w_out = w_out;
    p.lg = b.lg; p.act = b.act; p.y = b.y; p.xflag = b.xflag; p.ctl = b.ctl; p.status = b.status;
    p.T = s.T; p.H = s.H; p.E = s.E; p.K = s.K; p.F = s.F; p.norm = s.norm_topk;
    const uintptr_t x0 = reinterpret_cast<uintptr_t>(x), o0 = reinterpret_cast<uintptr_t>(out);
    const uintptr_t n = sizeof(float) * (uintptr_t)s.T * s.H;
    p.x_alias = (x0 < o0 + n && o0 < x0 + n) ? 1 : 0;
    p.cf = plan.cf;
    p.L = fused_layout(s.T, s.H, s.K, s.F, plan.nloc_max, plan.slot_bytes, plan.ns);
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
