// moe_decode_t1.cu -- the qwen3moe MoE-FFN layer for ONE token (batch-1
// decode) as one kernel of one CTA per SM, built for latency.
//
// What it computes is the layer of the aprender issue "qwen3moe (Qwen3-30B-A3B,
// ...) has NO working CUDA path" ("File facts", "Gaps ... G3"): F32 router GEMV,
// softmax + top-k + renorm, per selected expert Q4_K gate/up dequant-GEMV with
// SiLU(gate)*up, Q6_K or Q4_K down dequant-GEMV, weighted sum into the residual.
// At one token the layer reads 8 experts x 3 MB: about 4 us of HBM time at this
// GPU's bandwidth, so what decides its speed is the chain of dependent steps
// (router -> selection -> weight bytes -> act -> down), not arithmetic.  The
// kernel keeps that chain as short as it can:
//  * launched as a programmatic dependent of the previous kernel on the stream:
//    its CTAs start while that kernel drains, prefetch their router rows into L2
//    and wait in griddepcontrol.wait; nothing written by earlier work is read
//    before that wait;
//  * A: CTA c computes router logits c, c+G, ... (x and the row in registers,
//    one block reduction) and publishes them as {value, launch tag} words;
//  * B: every CTA reads all E logits, ranks them (order keys: ties to the lower
//    index) and, the moment the k selected ids are known, issues EVERY weight
//    copy it will need at once into shared memory (no buffer is reused, so
//    nothing waits for one to drain): for every slot j, its share of expert
//    e_j's gate and up rows (rows [F*c/G, F*(c+1)/G) of each) and the rows
//    [h0, h1) of e_j's down matrix that this CTA owns;
//  * C: every warp computes this CTA's gate/up rows as their slot's bytes
//    land, two rows at a time -- exact integer dot products (dp4a) of the
//    nibble codes with x split into three byte planes per 16 columns -- and
//    stores SiLU(g)*u; the CTA then counts itself in on one arrival word;
//  * D: once every CTA has counted in (one thread polls that word), every CTA
//    loads the k*F act values and computes y_j[h] for its own output rows and
//    every slot from the down rows already in shared memory (Q6_K rows are
//    first unpacked to one code per byte in column order, while the CTA waits
//    for the others, so that every lane of the dot products does useful work);
//  * finally out[h] = res[h] + sum_j w_j y_j[h] in slot order: a CTA owns whole
//    output rows, so no partial sums cross CTAs and no atomics touch values.
// Every cross-CTA wait is bounded (%globaltimer); on expiry the kernel records
// QMOE_ERR_TIMEOUT, computes nothing further, waits for its own copies and
// exits, and the launch tag still advances.  (Measured on this GPU: polling the
// act values themselves -- every thread of a CTA, or even four warps per CTA --
// floods L2 with requests while other CTAs are still streaming weights; one
// thread per loader polling one arrival word does not.)
#include <limits.h>
#include <math.h>

#include "kquant.cuh"
#include "ptx_sync.cuh"
#include "qmoe_internal.h"

#ifdef QMOE_PHASE_TRACE
// per-CTA phase timestamps (%globaltimer), compiled only into diagnostic builds
__device__ unsigned long long g_qmoe_trace_t1[1024 * 128];
#define T1_TRACE(slot)                                                               \
    do {                                                                             \
        g_qmoe_trace_t1[blockIdx.x * 128 + (slot)] = qmoe::globaltimer();             \
    } while (0)
#else
#define T1_TRACE(slot) \
    do {               \
    } while (0)
#endif

namespace qmoe {

namespace {

constexpr int TW = 16;                       // warps
constexpr int TN = TW * 32;                  // threads
constexpr int ACT_WORD = 3;                  // ctl[3]: CTAs whose act values are stored
constexpr int MAXK = 16;

constexpr float XQ_LIM1 = 8323072.f;         // 2^23 - 2^16: top byte plane stays in [-127, 127]

enum { MS_TAG = 0, MS_ABORT = 1, MS_COUNT = 4 };

__host__ __device__ inline int al1(int v, int a) { return (v + a - 1) / a * a; }
// staged act index: 4 floats of padding after every 128, so the two halves of
// a Q6_K superblock that lanes read together sit in different banks
__host__ __device__ __forceinline__ int apad1(int f) { return f + 4 * (f >> 7); }

struct T1Layout {
    int off_bar, off_misc, off_red, off_lg, off_key, off_sel, off_wts, off_x, off_xq, off_xsum,
        off_xscale, off_ys, off_gu, off_dn, total;
    int nrs_max, nrd_max, dn_seg, act_pitch, uq_row;
};

// x (fp32, phase A) and, later, the staged act values share one region; so do
// the gate/up rows and, once they are consumed, the unpacked Q6_K down rows
// (uq_row bytes each: F six-bit codes, one per byte in column order, then F/16
// floats d * scale; 0 when the down matrix is Q4_K)
__host__ __device__ inline T1Layout t1_layout(int H, int E, int K, int F, int G, int rbg, int rbd,
                                              int uq_row) {
    T1Layout L;
    L.nrs_max = (F + G - 1) / G;                 // gate/up rows per slot and CTA
    L.nrd_max = (H + G - 1) / G;                 // output rows per CTA
    L.dn_seg = al1(L.nrd_max * rbd + 32, 128);
    L.uq_row = uq_row;
    // one staged act row: Q4_K down -- padded as apad1 plus its group sums;
    // Q6_K down -- 16 lanes' column ranges, 4 floats of padding after each
    const int ap4 = apad1(F) + F / 8, ap6 = F + 64;
    L.act_pitch = al1(uq_row ? ap6 : ap4, 4);
    int o = 0;
    L.off_bar = o;    o += 2 * MAXK * 8;
    L.off_misc = o;   o += MS_COUNT * 4;
    L.off_red = o;    o += TW * 4;
    L.off_lg = o;     o += al1(E, 4) * 4;
    L.off_key = o;    o += al1(E, 128) * 4;
    L.off_sel = o;    o += MAXK * 4;
    L.off_wts = o;    o += MAXK * 4;
    o = al1(o, 16);
    L.off_x = o;      o += al1(H * 4 > K * L.act_pitch * 4 ? H * 4 : K * L.act_pitch * 4, 16);
    L.off_xq = o;     o += (H / 16) * 48;
    L.off_xsum = o;   o += (H / 16) * 4;
    L.off_xscale = o; o += (H / 16) * 4;
    L.off_ys = o;     o += al1(K * L.nrd_max * 4, 16);
    o = al1(o, 128);
    L.off_gu = o;
    o += 2 * K * L.nrs_max * rbg > K * L.nrd_max * uq_row ? 2 * K * L.nrs_max * rbg : K * L.nrd_max * uq_row;
    o = al1(o, 128);
    L.off_dn = o;     o += K * L.dn_seg;
    L.total = o;
    return L;
}

struct T1Params {
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
    unsigned long long* lg;     // [E] tagged router logits
    float* act;                 // [K][F] silu(g)*u (readiness: ctl[3])
    unsigned* ctl;              // [0] exit counter, [1] tag of the last completed launch,
                                // [3] CTAs whose act values are stored (reset at exit)
    int* status;
    const float* norm_w;        // nullable: x is RMS-normalised and scaled first
    float eps;
    unsigned long long wait_ns;
    int stall;                  // test hook: the logits wait expects a tag no CTA writes
    int H, E, K, F, norm;
    T1Layout L;
};

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void t1_status(int* status, int code) { atomicCAS(status, 0, code); }

// N tagged values base[first + z*stride] (those below n), all loads in flight
// together, reloaded until each carries `tag` (bounded).  False on timeout.
template <int N>
__device__ __forceinline__ bool t1_load_tagged(const unsigned long long* base, int n, int first,
                                               int stride, unsigned tag, float (&v)[N],
                                               unsigned long long limit_ns) {
    uint32_t pend = 0u;
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
            __nanosleep(20);
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

// bounded mbarrier wait with a caller-given limit: the suspending try_wait,
// during which the warp issues nothing (a spin on the non-blocking test was
// measured to more than double the kernel's issued instructions and slow the
// warps doing the work)
__device__ __forceinline__ bool t1_mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait_sleep(bar, parity, 20000u)) {
        if (globaltimer() - t0 > limit_ns) return false;
    }
    return true;
}

// exact integer form of one 16-byte Q4_K piece against x held as three signed
// byte planes (x = scale * (p2*2^16 + p1*2^8 + p0)): sum q*x for the low (SA)
// and high (SB) nibbles
__device__ __forceinline__ void t1_piece_dp4a(uint4 q, const int (&xa)[3][4], const int (&xb)[3][4],
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

// d*s*Q - dmin*m*X for the two sub-blocks of 32-byte chunk pc/2 of a Q4_K block
__device__ __forceinline__ float t1_piece_finish(uint4 hdr, int pc, float QA, float QB, float XA, float XB) {
    int sA, mA, sB, mB;
    q4_scales(hdr.y, hdr.z, hdr.w, pc >> 1, sA, mA, sB, mB);
    const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
    float r = (d * (float)sA) * QA - (dmin * (float)mA) * XA;
    r = fmaf(d * (float)sB, QB, r) - (dmin * (float)mB) * XB;
    return r;
}

// 16 bytes at an even shared-memory address (five aligned words, funnel shift)
__device__ __forceinline__ uint4 t1_lds16(const uint8_t* p) {
    const uint32_t off = smem_u32(p) & 3u;
    const uint32_t* b = reinterpret_cast<const uint32_t*>(p - off);
    const uint32_t sh = off * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2], w3 = b[3], w4 = b[4];
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                      __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

template <int NSB_G, int NSB_D, int DQT>
__global__ void __launch_bounds__(TN, 1) moe_decode_t1(const __grid_constant__ T1Params p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const T1Layout& L = p.L;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int H = p.H, E = p.E, K = p.K, F = p.F;
    constexpr int RBG = NSB_G * Q4K_BYTES;                        // gate/up row bytes
    constexpr int BBD = DQT == 1 ? Q4K_BYTES : Q6K_BYTES;
    constexpr int RBD = NSB_D * BBD;                              // down row bytes
    constexpr int HQ = NSB_G * QK / 4;                            // float4 of x
    constexpr int NX = (HQ + TN - 1) / TN;                        // x float4 per thread
    constexpr int GS = DQT == 1 ? 16 : 8;                         // act group of one down sub-scale
    const int FPAD = apad1(F);

    uint64_t* gub = reinterpret_cast<uint64_t*>(sm + L.off_bar);  // [K] gate/up rows of slot j landed
    uint64_t* dnb = gub + MAXK;                                    // [K] down rows of slot j landed
    int* misc = reinterpret_cast<int*>(sm + L.off_misc);
    float* red = reinterpret_cast<float*>(sm + L.off_red);
    float* lg_s = reinterpret_cast<float*>(sm + L.off_lg);
    int* key_s = reinterpret_cast<int*>(sm + L.off_key);
    int* sel = reinterpret_cast<int*>(sm + L.off_sel);
    float* wts = reinterpret_cast<float*>(sm + L.off_wts);
    float* x_s = reinterpret_cast<float*>(sm + L.off_x);
    float* act_st = x_s;                                          // [K][act_pitch] after phase A
    int32_t* xq = reinterpret_cast<int32_t*>(sm + L.off_xq);
    float* xsum = reinterpret_cast<float*>(sm + L.off_xsum);
    float* xscale = reinterpret_cast<float*>(sm + L.off_xscale);
    float* ys = reinterpret_cast<float*>(sm + L.off_ys);
    uint8_t* gu_s = sm + L.off_gu;
    uint8_t* dn_s = sm + L.off_dn;

    // this CTA's gate/up rows of every slot and its output rows
    const int f0 = (int)((long long)F * c / G), nrs = (int)((long long)F * (c + 1) / G) - f0;
    const int h0 = (int)((long long)H * c / G), nrd = (int)((long long)H * (c + 1) / G) - h0;

    // ---------------- before the previous kernel has finished: weights only
    if (tid == 0) T1_TRACE(0);
    if (tid < 4) {
        const int e = c + tid * G;
        if (e < E) bulk_prefetch_l2(p.router + (size_t)e * H, (uint32_t)(H * 4));
    }
    if (tid == 0) {
        for (int j = 0; j < K; ++j) {
            mbar_init(&gub[j], 1);
            mbar_init(&dnb[j], 1);
        }
        for (int i = 0; i < MS_COUNT; ++i) misc[i] = 0;
        fence_barrier_init();
    }
    griddep_wait();
    griddep_launch();
    if (tid == 0) T1_TRACE(1);
    if (tid == 0) misc[MS_TAG] = (int)(ld_acquire_gpu(p.ctl + 1) + 1u);   // this launch's tag

    // ---------------- phase A: x (optionally RMS-normalised), router logits.
    // The first router row this CTA owns is loaded together with x (both from
    // L2 by now), so the two loads share one round trip.
    float4 wr0[NX];
#pragma unroll
    for (int i = 0; i < NX; ++i) {
        const int q = tid + i * TN;
        wr0[i] = (c < E && q < HQ) ? __ldg(reinterpret_cast<const float4*>(p.router + (size_t)c * H) + q)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 xr[NX];
#pragma unroll
    for (int i = 0; i < NX; ++i) {
        const int q = tid + i * TN;
        xr[i] = q < HQ ? __ldg(reinterpret_cast<const float4*>(p.x) + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (p.norm_w) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < NX; ++i)
            ss += xr[i].x * xr[i].x + xr[i].y * xr[i].y + xr[i].z * xr[i].z + xr[i].w * xr[i].w;
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < TW; ++w) tot += red[w];
        const float r = rsqrtf(tot / (float)H + p.eps);
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            const int q = tid + i * TN;
            if (q < HQ) {
                const float4 nw = __ldg(reinterpret_cast<const float4*>(p.norm_w) + q);
                xr[i] = make_float4(xr[i].x * r * nw.x, xr[i].y * r * nw.y, xr[i].z * r * nw.z,
                                    xr[i].w * r * nw.w);
            }
        }
        __syncthreads();                                          // red is reused below
    }
#pragma unroll
    for (int i = 0; i < NX; ++i) {
        const int q = tid + i * TN;
        if (q < HQ) reinterpret_cast<float4*>(x_s)[q] = xr[i];
    }
    for (int e = c; e < E; e += G) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            const int q = tid + i * TN;
            if (q < HQ) {
                const float4 w = e == c ? wr0[i] : __ldg(reinterpret_cast<const float4*>(p.router + (size_t)e * H) + q);
                acc = fmaf(w.x, xr[i].x, acc);
                acc = fmaf(w.y, xr[i].y, acc);
                acc = fmaf(w.z, xr[i].z, acc);
                acc = fmaf(w.w, xr[i].w, acc);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (tid == 0) {
            float s = 0.f;
            for (int w = 0; w < TW; ++w) s += red[w];
            if (p.bias) s += p.bias[e];
            st_relaxed_u64(p.lg + e, tag_pack(s, (unsigned)misc[MS_TAG]));
        }
        __syncthreads();
    }
    __syncthreads();
    if (tid == 0) T1_TRACE(2);
    const unsigned tag = (unsigned)misc[MS_TAG];
    // x -> per-16-column scale, fp32 sum and three signed byte planes
    for (int g = tid; g < H / 16; g += TN) {
        const float* xv = x_s + 16 * g;
        float mx = 0.f, s = 0.f;
#pragma unroll
        for (int z = 0; z < 16; ++z) mx = fmaxf(mx, fabsf(xv[z]));
#pragma unroll
        for (int z = 0; z < 16; z += 4) s += (xv[z] + xv[z + 1]) + (xv[z + 2] + xv[z + 3]);
        const float inv = mx > 0.f ? XQ_LIM1 / mx : 0.f;
        int pw[12];
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
            pw[w4] = (int)p0;
            pw[4 + w4] = (int)p1;
            pw[8 + w4] = (int)p2;
        }
#pragma unroll
        for (int z = 0; z < 12; ++z) xq[12 * g + z] = pw[z];
        xscale[g] = mx / XQ_LIM1;
        xsum[g] = s;
    }

    // ---------------- phase B: all logits, top-k by rank on order keys
    {
        const unsigned want = p.stall ? (tag ^ 0x80000000u) : tag;
        float v[2];
        if (!t1_load_tagged<2>(p.lg, E, tid, TN, want, v, p.wait_ns)) {
            t1_status(p.status, ST_TIMEOUT);
            misc[MS_ABORT] = 1;
        }
#pragma unroll
        for (int z = 0; z < 2; ++z) {
            const int i = tid + z * TN;
            if (i < E) {
                lg_s[i] = v[z];
                key_s[i] = order_key(v[z]);
            } else if (i < ((E + 127) & ~127)) {
                key_s[i] = INT_MIN;                               // padding: never outranks a logit
            }
        }
    }
    if (tid < MAXK) sel[tid] = 0;
    __syncthreads();
    if (tid == 0) T1_TRACE(3);
    const bool abort_b = misc[MS_ABORT] != 0;
    if (!abort_b && warp == 0 && E <= 128) {
        // top-k for up to 128 experts: lane l sorts the (order key, index) pairs
        // of experts l, l + 32, l + 64, l + 96 (larger key first, ties to the
        // lower index), then K tournament rounds over the 32 lane heads: the
        // largest head key by one warp max-reduction, the lowest index holding it
        // by one min-reduction, and the owning lane drops its head.  (A warp
        // arg-max over all keys per round was measured 4x slower: a round is a
        // chain of five dependent shuffle steps.)
        int ks[4], is[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) {
            const int i = lane + 32 * z;
            ks[z] = i < E ? key_s[i] : INT_MIN;
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
            if (lane == 0) sel[r] = wi;
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
    } else if (!abort_b && warp == 0) {
        // more experts: K rounds of a warp arg-max over 64-bit keys (order key
        // of the logit, then E - 1 - e): round r takes the largest key below
        // round r - 1's, i.e. the r-th logit in descending order, ties to the
        // lower index
        long long prev = LLONG_MAX;
        for (int r = 0; r < K; ++r) {
            long long best = LLONG_MIN;
            for (int i = lane; i < E; i += 32) {
                const long long key = (long long)key_s[i] * 4294967296LL + (long long)(E - 1 - i);
                if (key < prev && key > best) best = key;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const long long other = __shfl_xor_sync(0xffffffffu, best, o);
                if (other > best) best = other;
            }
            if (lane == 0) sel[r] = E - 1 - (int)(best & 0xffffffffLL);
            prev = best;
        }
    }
    __syncthreads();
    if (tid == 0) T1_TRACE(10);

    // ---------------- the gate/up copies of this CTA, at once: lane 0 of warp j
    // issues slot j's gate rows and up rows (one barrier).  The down rows
    // (another barrier, from the 16-byte boundary below their first byte) are
    // requested later, once the warp has its first gate/up rows: they are not
    // needed before the act exchange, and requested together with the gate/up
    // rows they took a third of the bandwidth the gate/up phase waits on.
    // (Measured on this GPU: with all of a CTA's ~160 KB requested at once,
    // bulk copies, 16-byte cp.async copies and plain 16-byte loads all take
    // ~6 us to bring 24.5 MB into the 152 SMs; bulk copies leave the other
    // threads free; an L2 prefetch in front gains nothing.)
    if (!abort_b && lane == 0 && warp < K) {
        const int j = warp, e = sel[j];
        const uint32_t gbytes = (uint32_t)(nrs * RBG);
        mbar_arrive_expect_tx(&gub[j], 2 * gbytes);
        if (nrs > 0) {
            const size_t off = ((size_t)e * F + f0) * RBG;
            bulk_g2s(gu_s + (size_t)(2 * j) * L.nrs_max * RBG, p.gate + off, gbytes, &gub[j]);
            bulk_g2s(gu_s + (size_t)(2 * j + 1) * L.nrs_max * RBG, p.up + off, gbytes, &gub[j]);
        }
    }
    bool dn_issued = abort_b || warp >= K;
    auto issue_down = [&]() {
        if (lane == 0) {
            const int j = warp, e = sel[j];
            const uintptr_t src = reinterpret_cast<uintptr_t>(p.down) + ((size_t)e * H + h0) * RBD;
            const uintptr_t a0 = src & ~uintptr_t(15), a1 = (src + (size_t)nrd * RBD + 15) & ~uintptr_t(15);
            mbar_arrive_expect_tx(&dnb[j], (uint32_t)(a1 - a0));
            if (a1 > a0)
                bulk_g2s(dn_s + (size_t)j * L.dn_seg, reinterpret_cast<const void*>(a0), (uint32_t)(a1 - a0),
                         &dnb[j]);
        }
        dn_issued = true;
    };
    if (lane == 0) T1_TRACE(64 + warp);
    // routing weights (warp 0) while the copies are in flight
    if (!abort_b && warp == 0) {
        const float vmax = lg_s[sel[0]];
        float z = 0.f;
        for (int e = lane; e < E; e += 32) z += expf(lg_s[e] - vmax);
        z = warp_sum(z);
        const int id = lane < K ? sel[lane] : 0;
        const float pj = lane < K ? expf(lg_s[id] - vmax) / z : 0.f;
        const float psel = warp_sum(pj);
        if (lane < K) {
            const float w = p.norm ? pj / psel : pj;
            wts[lane] = w;
            if (c == 0) {
                if (p.ids_out) p.ids_out[lane] = id;
                if (p.w_out) p.w_out[lane] = w;
            }
        }
    }

    // ---------------- C: every warp, this CTA's gate/up rows of all slots (row
    // t = j * nrs + i), two at a time so that two independent dot products are
    // in flight per lane; SiLU(g)*u stored as plain floats
    {
        // x byte planes of this lane: 32-byte chunk c4 of superblock sb (two
        // 16-byte pieces, each pairing 16 columns with the low nibbles and the
        // 16 columns 32 further on with the high nibbles)
        int xa[2][3][4], xb[2][3][4];
        float XA[2], XB[2], SXA[2], SXB[2];
        const int sb = lane >> 2, c4 = lane & 3;
        const bool lane_on = lane < 4 * NSB_G;
#pragma unroll
        for (int jt = 0; jt < 2; ++jt) {
            XA[jt] = XB[jt] = SXA[jt] = SXB[jt] = 0.f;
#pragma unroll
            for (int pl = 0; pl < 3; ++pl)
#pragma unroll
                for (int z = 0; z < 4; ++z) xa[jt][pl][z] = xb[jt][pl][z] = 0;
            if (lane_on) {
                const int ga = (QK * sb + 64 * c4 + 16 * jt) / 16, gb = ga + 2;
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
        // Jobs of a warp: first a pair of rows (2w, 2w + 1) while pairs last for
        // every warp, then the remaining rows one at a time, spread over all
        // warps (pairs all the way put twice the rows on some warps than on
        // others when the CTA's row count is not a multiple of 2 * TW, and the
        // last warp sets the time of the phase)
        const int nrows = K * nrs;
        const int np = min(nrows / 2, TW);
        bool ok = !abort_b;
        for (int q = 0; ok; ++q) {
            int tr[2];
            if (q == 0 && warp < np) {
                tr[0] = 2 * warp;
                tr[1] = 2 * warp + 1;
            } else {
                const int qs = warp < np ? q - 1 : q;
                tr[0] = 2 * np + warp + qs * TW;
                tr[1] = -1;
            }
            if (tr[0] >= nrows) break;
            float gsum[2], usum[2];
            int jj[2], ii[2];
            bool on[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int t = tr[u];
                on[u] = t >= 0 && t < nrows;
                jj[u] = on[u] ? t / nrs : 0;
                ii[u] = on[u] ? t - jj[u] * nrs : 0;
                if (on[u]) ok = ok && __all_sync(0xffffffffu, t1_mbar_wait(&gub[jj[u]], 0, p.wait_ns));
            }
            if (!ok) break;
            if (lane == 0 && q == 0) T1_TRACE(80 + warp);
            if (!dn_issued) issue_down();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                gsum[u] = usum[u] = 0.f;
                if (lane_on && on[u]) {
#pragma unroll
                    for (int gu = 0; gu < 2; ++gu) {
                        const uint8_t* b = gu_s + ((size_t)(2 * jj[u] + gu) * L.nrs_max + ii[u]) * RBG + sb * Q4K_BYTES;
                        const uint4 hd = *reinterpret_cast<const uint4*>(b);
                        const uint4 q0 = *reinterpret_cast<const uint4*>(b + 16 + 32 * c4);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(b + 32 + 32 * c4);
                        float QA0, QB0, QA1, QB1;
                        t1_piece_dp4a(q0, xa[0], xb[0], SXA[0], SXB[0], QA0, QB0);
                        t1_piece_dp4a(q1, xa[1], xb[1], SXA[1], SXB[1], QA1, QB1);
                        const float cc = t1_piece_finish(hd, 2 * c4, QA0 + QA1, QB0 + QB1, XA[0] + XA[1], XB[0] + XB[1]);
                        if (gu) usum[u] = cc; else gsum[u] = cc;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                // lanes 0-15 end with the gate sum, lanes 16-31 with the up sum
                const bool h16 = lane & 16;
                float m = (h16 ? usum[u] : gsum[u]) + __shfl_xor_sync(0xffffffffu, h16 ? gsum[u] : usum[u], 16);
                m += __shfl_xor_sync(0xffffffffu, m, 8);
                m += __shfl_xor_sync(0xffffffffu, m, 4);
                m += __shfl_xor_sync(0xffffffffu, m, 2);
                m += __shfl_xor_sync(0xffffffffu, m, 1);
                const float upv = __shfl_down_sync(0xffffffffu, m, 16);
                if (lane == 0 && on[u]) p.act[(size_t)jj[u] * F + f0 + ii[u]] = m / (1.f + expf(-m)) * upv;
            }
        }
        if (!ok && lane == 0 && !abort_b) {
            t1_status(p.status, ST_TIMEOUT);
            misc[MS_ABORT] = 1;
        }
        // a warp with no gate/up rows (or one that gave up) still owes its slot's down copy
        if (!dn_issued) issue_down();
        if (lane == 0) T1_TRACE(16 + warp);
    }
    // This CTA's act values are stored: count it in.  Readiness of all act
    // values is then ONE word that one thread per CTA polls (polling the values
    // themselves, from every CTA, was measured to flood L2 with requests while
    // other CTAs were still streaming weights).
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        atomicAdd(p.ctl + ACT_WORD, 1u);
        T1_TRACE(4);
    }
    // ---------------- D prologue: the k x F act values staged in shared memory
    // once every CTA has counted in (and, for a Q6_K down matrix, the down rows
    // unpacked meanwhile)
    const bool run_pre = !abort_b && misc[MS_ABORT] == 0;
    if constexpr (DQT == 2) {
        // Warp 0: one lane polls the act counter, then the warp copies every act
        // value (cp.async through L2) into the staging layout: lane q of a
        // half-warp later reads columns [LQ q, LQ q + LQ) of a slot, so each such
        // range is followed by 4 floats of padding (the 8 lanes of one 16-byte
        // shared load then hit distinct banks).  The act values' L2 round trip
        // thus overlaps the unpacking below.
        if (warp == 0) {
            int okp = 0;
            if (lane == 0 && run_pre) {
                okp = 1;
                const unsigned long long t0 = globaltimer();
                for (int it = 1; ld_acquire_gpu(p.ctl + ACT_WORD) < (unsigned)G; ++it) {
                    __nanosleep(32);
                    if ((it & 15) == 0 && globaltimer() - t0 > p.wait_ns) {
                        t1_status(p.status, ST_TIMEOUT);
                        misc[MS_ABORT] = 1;
                        okp = 0;
                        break;
                    }
                }
                T1_TRACE(5);
            }
            okp = __shfl_sync(0xffffffffu, okp, 0);
            if (okp) {
                constexpr int LQ = 16 * NSB_D, F4 = NSB_D * QK / 4;   // F / 4
                const int n4 = K * F4;
                for (int i = lane; i < n4; i += 32) {
                    const int j = i / F4, c = 4 * (i - j * F4);
                    const int ql = c / LQ;
                    cp_async_cg16(act_st + (size_t)j * L.act_pitch + ql * (LQ + 4) + (c - ql * LQ),
                                  reinterpret_cast<const float4*>(p.act) + i);
                }
                cp_async_wait_all();
            }
        } else {
            // While the other CTAs finish: this CTA's Q6_K down rows, unpacked from
            // their copies into the (consumed) gate/up region as one six-bit code per
            // byte in column order and the float d * scale of each 16 columns.  A unit
            // is (slot, row, superblock s, half n, low-bit pair g01, 16 positions qq):
            // one 16-byte run of low-bit codes, one of high bits, and from them the
            // 16 codes of group g01 (low nibbles) and of group g01 + 2 (high
            // nibbles).  Consecutive threads take consecutive units, so the 8 lanes
            // of one 16-byte store write 8 different 16-byte slots of 128 bytes
            // except for the half bit (two ways, not eight).
            // (warps 1.. only)
            if (!abort_b && misc[MS_ABORT] == 0) {
                bool okd = true;
                for (int j = 0; j < K; ++j) okd = okd && t1_mbar_wait(&dnb[j], 0, p.wait_ns);
                if (tid == 32) T1_TRACE(11);
                if (!okd) {
                    t1_status(p.status, ST_TIMEOUT);
                    misc[MS_ABORT] = 1;
                } else {
                    constexpr int UPR = 8 * NSB_D;
                    uint8_t* uq = gu_s;
                    const int nu = K * nrd * UPR;
                    // rr / nrd as a multiply-high by ceil(2^32 / nrd): exact for rr,
                    // nrd < 2^16 (nrd = 1 needs 2^32 itself and is taken apart)
                    const unsigned magic = nrd > 1 ? (unsigned)((0x100000000ull + nrd - 1) / nrd) : 0u;
                    // UB units per thread per pass, every unit's shared loads issued
                    // before any of its stores (independent work for the scheduler)
                    constexpr int UB = 3;
                    for (int u0 = tid - 32; u0 < nu; u0 += UB * (TN - 32)) {
                        uint4 ql[UB], qh[UB];
                        int sc_lo[UB], sc_hi[UB], sh[UB];
                        float d[UB];
                        uint8_t* run[UB];
                        float* dsc[UB];
#pragma unroll
                        for (int b = 0; b < UB; ++b) {
                            const int u = min(u0 + b * (TN - 32), nu - 1);  // a repeated unit stores the same bytes
                            const int rr = u / UPR, w = u - rr * UPR;
                            const int j = nrd == 1 ? rr : (int)__umulhi((unsigned)rr, magic), r = rr - j * nrd;
                            const int qq = w & 1, g01 = (w >> 1) & 1, n = (w >> 2) & 1, s = w >> 3;
                            const uintptr_t src = reinterpret_cast<uintptr_t>(p.down) + ((size_t)sel[j] * H + h0) * RBD;
                            const uint8_t* blk = dn_s + (size_t)j * L.dn_seg + (src & 15) + (size_t)r * RBD + s * Q6K_BYTES;
                            ql[b] = t1_lds16(blk + 64 * n + 32 * g01 + 16 * qq);
                            qh[b] = t1_lds16(blk + 128 + 32 * n + 16 * qq);
                            sc_lo[b] = (int)*reinterpret_cast<const int8_t*>(blk + 192 + 8 * n + 2 * g01 + qq);
                            sc_hi[b] = (int)*reinterpret_cast<const int8_t*>(blk + 192 + 8 * n + 2 * g01 + qq + 4);
                            d[b] = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                            sh[b] = 2 * g01;                         // high bits of group g at bit 2g
                            uint8_t* dst = uq + (size_t)(j * L.nrd_max + r) * L.uq_row;
                            run[b] = dst + QK * s + 128 * n + 32 * g01 + 16 * qq;
                            dsc[b] = reinterpret_cast<float*>(dst + F) + 16 * s + 8 * n + 2 * g01 + qq;
                        }
#pragma unroll
                        for (int b = 0; b < UB; ++b) {
                            const uint32_t L4[4] = {ql[b].x, ql[b].y, ql[b].z, ql[b].w};
                            const uint32_t H4[4] = {qh[b].x, qh[b].y, qh[b].z, qh[b].w};
                            uint32_t lo[4], hi[4];
#pragma unroll
                            for (int wq = 0; wq < 4; ++wq) {
                                const uint32_t hb = H4[wq] >> sh[b];
                                lo[wq] = (L4[wq] & 0x0F0F0F0Fu) | ((hb << 4) & 0x30303030u);
                                hi[wq] = ((L4[wq] >> 4) & 0x0F0F0F0Fu) | (hb & 0x30303030u);
                            }
                            *reinterpret_cast<uint4*>(run[b]) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                            *reinterpret_cast<uint4*>(run[b] + 64) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                            dsc[b][0] = d[b] * (float)sc_lo[b];
                            dsc[b][4] = d[b] * (float)sc_hi[b];
                        }
                    }
                    if (tid == 32) T1_TRACE(13);
                }
            }
        }
        __syncthreads();
    } else {
        if (tid == 0) {
            if (!abort_b && misc[MS_ABORT] == 0) {
                const unsigned long long t0 = globaltimer();
                for (int it = 1; ld_acquire_gpu(p.ctl + ACT_WORD) < (unsigned)G; ++it) {
                    __nanosleep(32);
                    if ((it & 15) == 0 && globaltimer() - t0 > p.wait_ns) {
                        t1_status(p.status, ST_TIMEOUT);
                        misc[MS_ABORT] = 1;
                        break;
                    }
                }
            }
            T1_TRACE(5);
        }
        __syncthreads();
        if (run_pre && misc[MS_ABORT] == 0) {
            // two groups per thread per round, both groups' loads issued before any
            // store (one L2 round trip per round instead of one per group)
            const int ng = K * (F / GS);
            for (int g0 = tid; g0 < ng; g0 += 2 * TN) {
                float v[2][GS];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int g = g0 + u * TN;
                    const int j = g / (F / GS), gl = g - j * (F / GS);
                    const float4* src = reinterpret_cast<const float4*>(p.act + (size_t)j * F + gl * GS);
#pragma unroll
                    for (int z = 0; z < GS / 4; ++z) {
                        const float4 w = g < ng ? __ldcg(src + z) : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[u][4 * z] = w.x; v[u][4 * z + 1] = w.y; v[u][4 * z + 2] = w.z; v[u][4 * z + 3] = w.w;
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int g = g0 + u * TN;
                    if (g >= ng) continue;
                    const int j = g / (F / GS), gl = g - j * (F / GS);
                    float s = 0.f;
#pragma unroll
                    for (int z = 0; z < GS; ++z) s += v[u][z];
                    float* ast = act_st + (size_t)j * L.act_pitch;
#pragma unroll
                    for (int z = 0; z < GS; z += 4)
                        *reinterpret_cast<float4*>(ast + apad1(gl * GS + z)) =
                            make_float4(v[u][z], v[u][z + 1], v[u][z + 2], v[u][z + 3]);
                    ast[FPAD + gl] = s;
                }
            }
        }
        __syncthreads();
    }
    const bool run_d = !abort_b && misc[MS_ABORT] == 0;
    if (tid == 0) T1_TRACE(12);
    // ---------------- D: y_j[h] for this CTA's rows and every slot.
    if constexpr (DQT == 2) {
        // Q6_K down from the unpacked rows.  Half-warp hw (of 32) serves slot
        // hw / hps (hps = 32 / K half-warps per slot) and rows sub, sub + hps, ...
        // of it; lane q owns columns [LQ q, LQ q + LQ) -- NSB_D groups of 16 --
        // holds their act values and group sums, and for each row takes the dot
        // with the six-bit codes (as 0.5 + code / 256, two fp32x2 FMA chains) and
        // sum_g d s_g (256 P_g - 160 A_g) = sum (code - 32) a; the 16 lanes' parts
        // are summed by a fixed butterfly.
        if (run_d) {
            constexpr int LQ = 16 * NSB_D;
            const int hps = 32 / K;
            const int hw = 2 * warp + (lane >> 4), q = lane & 15;
            const int j = hw / hps, sub = hw - j * hps;
            const unsigned hmask = 0xFFFFu << (lane & 16);
            const uint8_t* uq = gu_s;
            if (j < K) {
                const float* ast = act_st + (size_t)j * L.act_pitch + q * (LQ + 4);
                float4 av[NSB_D][4];
                float A[NSB_D];
#pragma unroll
                for (int t = 0; t < NSB_D; ++t) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) av[t][k] = *reinterpret_cast<const float4*>(ast + 16 * t + 4 * k);
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        a0 += av[t][k].x + av[t][k].y;
                        a1 += av[t][k].z + av[t][k].w;
                    }
                    A[t] = a0 + a1;
                }
                // two rows per pass (rows r and r + hps): twice the independent
                // work between the shared loads and the butterfly
                auto row_dot = [&](int r) {
                    const uint8_t* row = uq + (size_t)(j * L.nrd_max + r) * L.uq_row;
                    const float* dsc = reinterpret_cast<const float*>(row + F) + q * NSB_D;
                    uint4 w[NSB_D];
                    float ds[NSB_D];
#pragma unroll
                    for (int t = 0; t < NSB_D; ++t) {
                        w[t] = *reinterpret_cast<const uint4*>(row + LQ * q + 16 * t);
                        ds[t] = dsc[t];
                    }
                    float part = 0.f;
#pragma unroll
                    for (int t = 0; t < NSB_D; ++t) {
                        const uint32_t W[4] = {w[t].x, w[t].y, w[t].z, w[t].w};
                        float p0 = 0.f, p1 = 0.f;
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            fma2(p0, p1, mag<0>(W[k]), mag<1>(W[k]), av[t][k].x, av[t][k].y);
                            fma2(p0, p1, mag<2>(W[k]), mag<3>(W[k]), av[t][k].z, av[t][k].w);
                        }
                        part = fmaf(ds[t], fmaf(256.f, p0 + p1, -160.f * A[t]), part);
                    }
                    return part;
                };
                for (int r = sub; r < nrd; r += 2 * hps) {
                    const int r2 = r + hps;
                    const bool two = r2 < nrd;
                    float pa = row_dot(r);
                    float pb = row_dot(two ? r2 : r);
#pragma unroll
                    for (int o = 8; o > 0; o >>= 1) {
                        pa += __shfl_xor_sync(hmask, pa, o);
                        pb += __shfl_xor_sync(hmask, pb, o);
                    }
                    if (q == 0) {
                        ys[j * L.nrd_max + r] = pa;
                        if (two) ys[j * L.nrd_max + r2] = pb;
                    }
                }
            }
            if (lane == 0) T1_TRACE(48 + warp);
        }
    } else if (run_d) {
        // Q4_K down from the raw rows.  Warp task (slot j, block of 8 rows); a
        // lane owns one 16-byte piece of a superblock for the 8 rows of the
        // block, and the parts of a row are summed across lanes by a fixed
        // butterfly.
        const int nrb = (nrd + 7) / 8;
        for (int t = warp; t < K * nrb; t += TW) {
            const int j = t / nrb, rb = t - j * nrb;
            if (!__all_sync(0xffffffffu, t1_mbar_wait(&dnb[j], 0, p.wait_ns))) {
                if (lane == 0) { t1_status(p.status, ST_TIMEOUT); misc[MS_ABORT] = 1; }
                break;
            }
            const float* ast = act_st + (size_t)j * L.act_pitch;
            const float* asm_ = ast + FPAD;
            const uintptr_t src = reinterpret_cast<uintptr_t>(p.down) + ((size_t)sel[j] * H + h0) * RBD;
            const uint8_t* seg = dn_s + (size_t)j * L.dn_seg + (src & 15);
            {
                // Q4_K: lane < 8*NSB_D is (superblock s, 16-byte piece pc); rows
                // 8 rb + k, k < 8
                const bool on = lane < 8 * NSB_D;
                const int s = lane >> 3, pc = lane & 7;
                const int col = QK * s + 64 * (pc >> 1) + 16 * (pc & 1);
                float4 va[4], vb[4];
                float XA = 0.f, XB = 0.f;
#pragma unroll
                for (int z = 0; z < 4; ++z) va[z] = vb[z] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (on) {
                    const float* ac = ast + apad1(col);
#pragma unroll
                    for (int z = 0; z < 4; ++z) {
                        va[z] = *reinterpret_cast<const float4*>(ac + 4 * z);
                        vb[z] = *reinterpret_cast<const float4*>(ac + 32 + 4 * z);
                    }
                    XA = asm_[col / 16];
                    XB = asm_[col / 16 + 2];
                }
                float part[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int r = 8 * rb + k;
                    part[k] = 0.f;
                    if (on && r < nrd) {
                        const uint8_t* blk = seg + (size_t)r * RBD + s * Q4K_BYTES;
                        const uint4 hdr = *reinterpret_cast<const uint4*>(blk);
                        const uint4 qv = *reinterpret_cast<const uint4*>(blk + 16 + 16 * pc);
                        float PA, PB;
                        q4_piece_dot(qv, va, vb, PA, PB);
                        part[k] = q4_piece_finish(hdr, pc, PA, PB, XA, XB);
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float v = part[k];
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 4);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    const int r = 8 * rb + k;
                    if (lane == 0 && r < nrd) ys[j * L.nrd_max + r] = v;
                }
            }
        }
        if (lane == 0) T1_TRACE(48 + warp);
    }
    __syncthreads();
    if (tid == 0) T1_TRACE(6);
    if (!abort_b && misc[MS_ABORT] == 0) {
        // out[h] = res[h] + sum_j w_j y_j[h], slot order
        const float* res = p.res ? p.res : p.x;
        for (int r = tid; r < nrd; r += TN) {
            float o = res[h0 + r];
            for (int j = 0; j < K; ++j) o = fmaf(wts[j], ys[j * L.nrd_max + r], o);
            p.out[h0 + r] = o;
        }
    }
    // every copy this CTA issued has landed before it exits (already true
    // unless a wait gave up)
    if (!abort_b && lane == 0 && warp < K) {
        t1_mbar_wait(&gub[warp], 0, p.wait_ns);
        t1_mbar_wait(&dnb[warp], 0, p.wait_ns);
    }
    __syncthreads();
    if (tid == 0) T1_TRACE(7);
    if (tid == 0) {
        // the last CTA out resets the exit counter and the act arrival word
        // and publishes this launch's tag
        __threadfence();
        if (atomicAdd(&p.ctl[0], 1u) == (unsigned)G - 1) {
            atomicExch(&p.ctl[0], 0u);
            atomicExch(&p.ctl[ACT_WORD], 0u);
            atomicExch(&p.ctl[1], tag);
        }
    }
}

struct T1Variant {
    int nsb_g, nsb_d, dqt;
    const void* fn;
};

template <int A, int B, int C>
const void* t1fn() { return reinterpret_cast<const void*>(&moe_decode_t1<A, B, C>); }

const T1Variant kT1[] = {
    {8, 3, 2, t1fn<8, 3, 2>()}, {8, 3, 1, t1fn<8, 3, 1>()},
    {1, 1, 2, t1fn<1, 1, 2>()}, {1, 1, 1, t1fn<1, 1, 1>()},
};

const T1Variant* t1_variant(int H, int F, int down_t) {
    for (const T1Variant& v : kT1)
        if (v.nsb_g == H / QK && v.nsb_d == F / QK && v.dqt == down_t) return &v;
    return nullptr;
}

}  // namespace

bool t1_decode_plan(const MoeShape& s, int gate_t, int up_t, int down_t, int num_sms, T1Plan* plan) {
    if (s.T != 1 || gate_t != 1 || up_t != 1) return false;
    const T1Variant* v = t1_variant(s.H, s.F, down_t);
    if (!v) return false;
    if (s.E < 1 || s.E > 2 * TN || s.K < 1 || s.K > MAXK || s.K > s.E) return false;
    const int G = num_sms;
    if (G < 1 || G > 1024 || s.E > 4 * G) return false;          // router rows per CTA (prefetch)
    // every CTA counts in on every slot after reading x, and no CTA writes an
    // output row before every CTA has counted in on slot 0 (out may alias x)
    if (s.K > TW) return false;
    const int rbg = (s.H / QK) * Q4K_BYTES;
    const int rbd = (s.F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    const T1Layout L = t1_layout(s.H, s.E, s.K, s.F, G, rbg, rbd, down_t == 2 ? s.F + s.F / 4 : 0);
    if (L.total > 227 * 1024) return false;
    plan->grid = G;
    plan->smem = L.total;
    plan->fn = v->fn;
    return true;
}

cudaError_t launch_t1_decode(const MoeShape& s, const T1Plan& plan, int down_t, const float* x,
                             const float* res, const float* bias, const float* router,
                             const uint8_t* gate, const uint8_t* up, const uint8_t* down, float* out,
                             int32_t* ids_out, float* w_out, const FusedBufs& b, const float* norm_w,
                             float eps, cudaStream_t st, const FusedDebug* dbg) {
    T1Params p;
    p.x = x; p.res = res; p.bias = bias; p.router = router;
    p.gate = gate; p.up = up; p.down = down;
    p.out = out; p.ids_out = ids_out; p.w_out = w_out;
    p.lg = b.lg; p.act = b.plain_act; p.ctl = b.ctl; p.status = b.status;
    p.norm_w = norm_w; p.eps = eps;
    p.wait_ns = dbg ? dbg->wait_ns : WAIT_LIMIT_NS;
    p.stall = dbg ? dbg->stall : 0;
    p.H = s.H; p.E = s.E; p.K = s.K; p.F = s.F; p.norm = s.norm_topk;
    const int rbg = (s.H / QK) * Q4K_BYTES;
    const int rbd = (s.F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    p.L = t1_layout(s.H, s.E, s.K, s.F, plan.grid, rbg, rbd, down_t == 2 ? s.F + s.F / 4 : 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(plan.grid);
    cfg.blockDim = dim3(TN);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* args[] = {&p};
    return cudaLaunchKernelExC(&cfg, plan.fn, args);
}

#ifdef QMOE_PHASE_TRACE
extern "C" int qmoe_trace_read_t1(unsigned long long* host, int n) {
    return (int)cudaMemcpyFromSymbol(host, g_qmoe_trace_t1, sizeof(unsigned long long) * n);
}
#endif

cudaError_t t1_prepare() {
    for (const T1Variant& v : kT1) {
        cudaError_t e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace qmoe
