// moe_route.cu -- router GEMV, softmax / top-k / renorm, and the per-expert pair
// lists (the routing half of the qwen3moe MoE FFN).
//
// aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path",
// section "Gaps ... G3": router = F32 GEMV of ffn_gate_inp [E x H]; softmax,
// top-8 and renorm (planned device kernel K1 in G8).  Everything stays on the
// device: no logits copy, no host sync, so the layer is graph-capturable.
#include <climits>
#include <float.h>
#include <math.h>

#include "kquant.cuh"

#include "pdl.cuh"
#include "topk.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

constexpr int RT_TOK = 8;     // tokens per router CTA
constexpr int RT_EXP = 2;     // experts per router CTA (one warp each): E / 2 CTAs keep many SMs loading

// logits[t][e] = sum_h Wr[e][h] x[t][h] (+ bias[e]), fp32 accumulation.
__global__ void __launch_bounds__(32 * RT_EXP) router_kernel(const float* __restrict__ x,
                                                     const float* __restrict__ wr,
                                                     const float* __restrict__ bias, int T,
                                                     int H, int E, float* __restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * RT_EXP + warp;
    const int t0 = blockIdx.y * RT_TOK;
    if (e >= E) return;
    const int nt = min(RT_TOK, T - t0);
    float acc[RT_TOK];
#pragma unroll
    for (int i = 0; i < RT_TOK; ++i) acc[i] = 0.f;
    const float* wrow = wr + (size_t)e * H;
#pragma unroll 4
    for (int h = 4 * lane; h < H; h += 128) {
        const float4 w = __ldg(reinterpret_cast<const float4*>(wrow + h));
#pragma unroll
        for (int i = 0; i < RT_TOK; ++i) {
            if (i < nt) {
                const float4 v = __ldg(reinterpret_cast<const float4*>(x + (size_t)(t0 + i) * H + h));
                acc[i] = fmaf(w.x, v.x, acc[i]);
                acc[i] = fmaf(w.y, v.y, acc[i]);
                acc[i] = fmaf(w.z, v.z, acc[i]);
                acc[i] = fmaf(w.w, v.w, acc[i]);
            }
        }
    }
    const float b = bias ? bias[e] : 0.f;
#pragma unroll
    for (int i = 0; i < RT_TOK; ++i) {
        if (i < nt) {
            const float s = warp_sum(acc[i]);
            if (lane == 0) logits[(size_t)(t0 + i) * E + e] = s + b;
        }
    }
}

__global__ void __launch_bounds__(1024) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                    int K, int norm, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts,
                                                    int32_t* __restrict__ n_used,
                                                    int32_t* __restrict__ used_expert,
                                                    int32_t* __restrict__ used_first,
                                                    int32_t* __restrict__ pair_list) {
    extern __shared__ int32_t sm[];               // counts[E], cursor[E]
    topk_lists(logits, T, E, K, norm, ids, wts, n_used, used_expert, used_first, pair_list, sm);
}

// Router GEMV and top-k in one launch for up to RS_TOK tokens.  CTA e computes
// logits[t][e] for every token, its RS_THREADS threads splitting the row (one
// round trip of loads), and the last CTA to finish (an arrival counter, which it
// resets for the next launch) runs the top-k and the per-expert lists.  The
// router row is loaded before the wait on the previous kernel (weights are
// never written by a kernel), x after it.
constexpr int RS_TOK = 8, RS_THREADS = 256, RS_EMAX = 1024;

__global__ void __launch_bounds__(RS_THREADS) router_topk_small(
    const float* __restrict__ x, const float* __restrict__ wr, const float* __restrict__ bias,
    int T, int H, int E, int K, int norm, float* __restrict__ logits, int32_t* __restrict__ ids,
    float* __restrict__ wts, int32_t* __restrict__ n_used, int32_t* __restrict__ used_expert,
    int32_t* __restrict__ used_first, int32_t* __restrict__ pair_list, unsigned* arrive) {
    __shared__ float red[RS_TOK][RS_THREADS / 32];
    __shared__ int32_t sm[2 * RS_EMAX];
    __shared__ int is_last;
    const int e = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* wrow = wr + (size_t)e * H;
    constexpr int NW = 4;                         // row float4s a thread keeps in registers
    float4 w[NW];
#pragma unroll
    for (int k = 0; k < NW; ++k) {
        const int h = 4 * (threadIdx.x + k * RS_THREADS);
        w[k] = h < H ? __ldg(reinterpret_cast<const float4*>(wrow + h)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    pdl_launch_dependents();
    float acc[RS_TOK];
#pragma unroll
    for (int i = 0; i < RS_TOK; ++i) acc[i] = 0.f;
    for (int h0 = 0; h0 < H; h0 += 4 * NW * RS_THREADS) {
#pragma unroll
        for (int k = 0; k < NW; ++k) {
            const int h = h0 + 4 * (threadIdx.x + k * RS_THREADS);
            if (h >= H) continue;
            const float4 wk = h0 == 0 ? w[k] : __ldg(reinterpret_cast<const float4*>(wrow + h));
#pragma unroll
            for (int i = 0; i < RS_TOK; ++i) {
                if (i < T) {
                    const float4 v = __ldg(reinterpret_cast<const float4*>(x + (size_t)i * H + h));
                    acc[i] = fmaf(wk.x, v.x, acc[i]);
                    acc[i] = fmaf(wk.y, v.y, acc[i]);
                    acc[i] = fmaf(wk.z, v.z, acc[i]);
                    acc[i] = fmaf(wk.w, v.w, acc[i]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < RS_TOK; ++i) {
        if (i < T) {
            const float v = warp_sum(acc[i]);
            if (lane == 0) red[i][warp] = v;
        }
    }
    __syncthreads();
    if (threadIdx.x < T) {
        float v = 0.f;
#pragma unroll
        for (int k = 0; k < RS_THREADS / 32; ++k) v += red[threadIdx.x][k];
        logits[(size_t)threadIdx.x * E + e] = v + (bias ? bias[e] : 0.f);
        __threadfence();
    }
    __syncthreads();
    if (threadIdx.x == 0) is_last = atomicAdd(arrive, 1u) == gridDim.x - 1;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    topk_lists(logits, T, E, K, norm, ids, wts, n_used, used_expert, used_first, pair_list, sm);
    if (threadIdx.x == 0) *arrive = 0u;
}

// ---------------------------------------------------------------------------- many tokens

constexpr int RG_T = 64, RG_E = 64, RG_K = 128;    // router tile: tokens x experts x k-slice
constexpr int RG_THREADS = 256;                    // 4 tokens x 4 experts per thread
constexpr int RG_LD = RG_K + 4;                    // padded smem row (floats)

// Split-k router GEMM: part[z][t][e] = sum over k in slice z of X[t][k] Wr[e][k],
// a slice being KS = H / gridDim.z columns (a multiple of RG_K) walked in chunks
// of RG_K.  Slices are summed in a fixed order by topk_rank, so the result is
// deterministic.  Grid (ceil(E/64), ceil(T/64), S).
__global__ void __launch_bounds__(RG_THREADS) router_gemm(const float* __restrict__ x,
                                                          const float* __restrict__ wr, int T,
                                                          int H, int E,
                                                          float* __restrict__ part,
                                                          uint32_t* __restrict__ clear, int nclear) {
    pdl_wait();
    extern __shared__ float4 rg_smem4[];
    float* xs = reinterpret_cast<float*>(rg_smem4);              // [RG_T][RG_LD]
    float* ws = xs + RG_T * RG_LD;                               // [RG_E][RG_LD]
    const int KS = H / gridDim.z;
    const int e0 = blockIdx.x * RG_E, t0 = blockIdx.y * RG_T;
    const int tid = threadIdx.x;
    // the token bitmap and counts that topk_rank fills start from zero
    {
        const int nb = gridDim.x * gridDim.y * gridDim.z;
        const int b = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        for (int i = b * RG_THREADS + tid; i < nclear; i += nb * RG_THREADS) clear[i] = 0u;
    }
    const int tx = tid & 15, ty = tid >> 4;      // experts tx + 16j, tokens ty + 16i
    float acc[4][4] = {};
    for (int k0 = blockIdx.z * KS; k0 < (blockIdx.z + 1) * KS; k0 += RG_K) {
    // 64 rows x 32 float4 per operand, 8 float4 per thread each, all in flight
    float4 vx[8], vw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int f = tid + i * RG_THREADS, r = f >> 5, c = (f & 31) * 4;
        vx[i] = t0 + r < T ? __ldg(reinterpret_cast<const float4*>(x + (size_t)(t0 + r) * H + k0 + c))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        vw[i] = e0 + r < E ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)(e0 + r) * H + k0 + c))
                           : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();                             // the previous chunk is consumed
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int f = tid + i * RG_THREADS, r = f >> 5, c = (f & 31) * 4;
        *reinterpret_cast<float4*>(xs + r * RG_LD + c) = vx[i];
        *reinterpret_cast<float4*>(ws + r * RG_LD + c) = vw[i];
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < RG_K; k += 4) {
        float4 a[4], w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) a[i] = *reinterpret_cast<const float4*>(xs + (ty + 16 * i) * RG_LD + k);
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = *reinterpret_cast<const float4*>(ws + (tx + 16 * j) * RG_LD + k);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                acc[i][j] = fmaf(a[i].x, w[j].x, acc[i][j]);
                acc[i][j] = fmaf(a[i].y, w[j].y, acc[i][j]);
                acc[i][j] = fmaf(a[i].z, w[j].z, acc[i][j]);
                acc[i][j] = fmaf(a[i].w, w[j].w, acc[i][j]);
            }
    }
    }
    float* dst = part + (size_t)blockIdx.z * T * E;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int t = t0 + ty + 16 * i, e = e0 + tx + 16 * j;
            if (t < T && e < E) dst[(size_t)t * E + e] = acc[i][j];
        }
}

// one warp per token: rank every logit (ties: lower index first), keep the top
// K in descending order, softmax over E, renormalise over the selection
__global__ void __launch_bounds__(256) topk_rank(const float* __restrict__ part, int S,
                                                 const float* __restrict__ bias, int T, int E,
                                                 int K, int norm, float* __restrict__ logits,
                                                 int32_t* __restrict__ ids,
                                                 float* __restrict__ wts,
                                                 uint32_t* __restrict__ tokmap,
                                                 int32_t* __restrict__ counts,
                                                 uint8_t* __restrict__ jmap) {
    pdl_wait();
    extern __shared__ float lsm[];                 // 8 warps x (E logits + 16 selection slots)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    float* l = lsm + warp * (E + 16);
    int* sel = reinterpret_cast<int*>(l + E);
    // S split-k partials summed in slice order; four experts per lane at a
    // time, so the loads of a slice are independent of the running sums
    for (int e0 = 0; e0 < E; e0 += 128) {
        float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
        for (int z = 0; z < S; ++z) {
            const float* pz = part + ((size_t)z * T + t) * E;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int e = e0 + lane + 32 * i;
                if (e < E) v[i] += pz[e];
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = e0 + lane + 32 * i;
            if (e < E) {
                const float w = v[i] + (bias ? bias[e] : 0.f);
                l[e] = w;
                logits[(size_t)t * E + e] = w;
            }
        }
    }
    __syncwarp();
    if (E <= 128) {
        // lane l sorts the (order key, index) pairs of experts l, l + 32, l + 64,
        // l + 96 (larger key first, ties to the lower index); then K tournament
        // rounds over the 32 lane heads: the largest head key by one warp
        // max-reduction, the lowest index holding it by one min-reduction, and
        // the owning lane drops its head
        int ks[4], is[4];
#pragma unroll
        for (int z = 0; z < 4; ++z) {
            const int i = lane + 32 * z;
            ks[z] = i < E ? order_key(l[i]) : INT_MIN;
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
    }
    // more experts: K rounds of a warp arg-max over 64-bit keys (order key of
    // the logit, then E - 1 - e): round r takes the largest key below round
    // r - 1's, which is the r-th logit in descending order, ties to the lower index
    long long prev = LLONG_MAX;
    for (int r = 0; E > 128 && r < K; ++r) {
        long long best = LLONG_MIN;
        for (int e = lane; e < E; e += 32) {
            const long long key = (long long)order_key(l[e]) * 4294967296LL + (long long)(E - 1 - e);
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
    __syncwarp();
    const float vmax = l[sel[0]];
    float z = 0.f;
    for (int e = lane; e < E; e += 32) z += expf(l[e] - vmax);
    z = warp_sum(z);
    const int id = lane < K ? sel[lane] : 0;
    const float pj = lane < K ? expf(l[id] - vmax) / z : 0.f;
    const float psel = warp_sum(pj);
    if (lane < K) {
        ids[(size_t)t * K + lane] = id;
        wts[(size_t)t * K + lane] = norm ? pj / psel : pj;
        // expert id's token bitmap (row of W = ceil(T/32) words) and pair count
        atomicOr(&tokmap[(size_t)id * ((T + 31) >> 5) + (t >> 5)], 1u << (t & 31));
        atomicAdd(&counts[id], 1);
        jmap[(size_t)id * T + t] = (uint8_t)lane;
    }
}

constexpr int EL_THREADS = 256;

// One CTA per expert e: the pairs of e in ascending p.  A token selects an
// expert at most once, so ascending p is ascending token order, and the rank of
// token t in e's list is the number of set bits before t in e's token bitmap:
// the row is staged in shared memory with the running popcount before each
// word (a block scan), then every thread places its tokens independently; the
// slot j of the pair (t, e) comes from the byte map topk_rank wrote.  The list
// starts at the sum of the counts of the experts below e; the used-expert list
// comes from the same prefix over the nonzero counts.
__global__ void __launch_bounds__(EL_THREADS) expert_lists(const uint8_t* __restrict__ jmap,
                                                           const uint32_t* __restrict__ tokmap,
                                                           const int32_t* __restrict__ counts, int T,
                                                           int E, int K, int32_t* __restrict__ n_used,
                                                           int32_t* __restrict__ used_expert,
                                                           int32_t* __restrict__ used_first,
                                                           int32_t* __restrict__ pair_list) {
    pdl_wait();
    extern __shared__ uint32_t el_sm[];             // W words, then W running popcounts
    __shared__ int red[2][EL_THREADS / 32];
    __shared__ int scan[EL_THREADS / 32];
    const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int off = 0, ub = 0;
    for (int i = tid; i < e; i += EL_THREADS) {
        const int c = counts[i];
        off += c;
        ub += c > 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        off += __shfl_xor_sync(0xffffffffu, off, o);
        ub += __shfl_xor_sync(0xffffffffu, ub, o);
    }
    if (lane == 0) {
        red[0][warp] = off;
        red[1][warp] = ub;
    }
    __syncthreads();
    off = 0;
    ub = 0;
#pragma unroll
    for (int w = 0; w < EL_THREADS / 32; ++w) {
        off += red[0][w];
        ub += red[1][w];
    }
    const int cnt = counts[e];
    if (tid == 0) {
        if (cnt > 0) {
            used_expert[ub] = e;
            used_first[ub] = off;
        }
        if (e == E - 1) {
            const int used = ub + (cnt > 0);
            *n_used = used;
            used_first[used] = T * K;
        }
    }
    if (cnt == 0) return;
    const int W = (T + 31) >> 5;
    uint32_t* words = el_sm;
    int* before = reinterpret_cast<int*>(el_sm + W);
    const uint32_t* row = tokmap + (size_t)e * W;
    const int per = (W + EL_THREADS - 1) / EL_THREADS;
    const int w0 = min(W, tid * per), w1 = min(W, w0 + per);
    int mine = 0;
    for (int w = w0; w < w1; ++w) {
        const uint32_t b = row[w];
        words[w] = b;
        mine += __popc(b);
    }
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    int run = off + incl - mine;
    for (int w = 0; w < warp; ++w) run += scan[w];
    for (int w = w0; w < w1; ++w) {
        before[w] = run;
        run += __popc(words[w]);
    }
    __syncthreads();
    const uint8_t* jrow = jmap + (size_t)e * T;
    for (int t = tid; t < T; t += EL_THREADS) {
        const uint32_t b = words[t >> 5];
        const uint32_t bit = 1u << (t & 31);
        if (b & bit) pair_list[before[t >> 5] + __popc(b & (bit - 1u))] = t * K + jrow[t];
    }
}

}  // namespace

// k-slices of the router GEMM: as few as keep about eight CTAs per SM in
// flight (each CTA loads its chunks and computes them in turn, so fewer, longer
// CTAs expose the load latency), each a whole number of RG_K chunks
int route_many_slices(int T, int H, int E) {
    const int tiles = ((E + RG_E - 1) / RG_E) * ((T + RG_T - 1) / RG_T);
    int S = H / RG_K;
    while (S % 2 == 0 && tiles * (S / 2) >= 1200) S /= 2;
    return S;
}

cudaError_t launch_route_many(const MoeShape& s, const float* x, const float* router_w,
                              const float* bias, const Route& r, cudaStream_t st) {
    const size_t rg_smem = sizeof(float) * (RG_T + RG_E) * RG_LD;
    const int S = route_many_slices(s.T, s.H, s.E);
    dim3 g1((s.E + RG_E - 1) / RG_E, (s.T + RG_T - 1) / RG_T, S);
    const int W = (s.T + 31) / 32;
    uint32_t* counts = r.tokmap + (size_t)s.E * W;      // E counters after the bitmap
    cudaError_t e = launch_pdl(router_gemm, g1, dim3(RG_THREADS), rg_smem, st, x, router_w, s.T, s.H,
                               s.E, r.logits_part, r.tokmap, s.E * W + s.E);
    if (e != cudaSuccess) return e;
    e = launch_pdl(topk_rank, dim3((s.T + 7) / 8), dim3(256), sizeof(float) * 8 * (s.E + 16), st,
                   r.logits_part, S, bias, s.T, s.E, s.K, s.norm_topk, r.logits, r.ids, r.wts, r.tokmap,
                   reinterpret_cast<int32_t*>(counts), r.jmap);
    if (e != cudaSuccess) return e;
    return launch_pdl(expert_lists, dim3(s.E), dim3(EL_THREADS), sizeof(uint32_t) * 2 * W, st, r.jmap,
                      r.tokmap, reinterpret_cast<const int32_t*>(counts), s.T, s.E, s.K, r.n_used,
                      r.used_expert, r.used_first, r.pair_list);
}

// workspace for the partial sums of any call with up to T tokens (a call with
// fewer tokens may use more slices, never more than H / RG_K)
size_t route_many_part_floats(int T, int H, int E) { return (size_t)(H / RG_K) * T * E; }

size_t route_many_tokmap_words(int T, int E) { return (size_t)E * ((T + 31) / 32) + E; }

bool route_many_supported(const MoeShape& s, const Route& r) {
    // expert_lists stages a bitmap row and its running counts (8 bytes per 32 tokens)
    return r.logits_part && r.tokmap && r.jmap && s.H % RG_K == 0 && s.K <= 32 &&
           sizeof(uint32_t) * 2 * ((s.T + 31) / 32) <= 48 * 1024;
}

// Raise the dynamic shared-memory limits once per device context.
cudaError_t route_prepare() {
    return cudaFuncSetAttribute(router_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(sizeof(float) * (RG_T + RG_E) * RG_LD));
}

cudaError_t launch_route(const MoeShape& s, const float* x, const float* router_w,
                         const float* bias, const Route& r, cudaStream_t st) {
    if (r.arrive && s.T <= RS_TOK && s.E <= RS_EMAX)
        return launch_pdl(router_topk_small, dim3(s.E), dim3(RS_THREADS), 0, st, x, router_w, bias,
                          s.T, s.H, s.E, s.K, s.norm_topk, r.logits, r.ids, r.wts, r.n_used,
                          r.used_expert, r.used_first, r.pair_list, r.arrive);
    dim3 g1((s.E + RT_EXP - 1) / RT_EXP, (s.T + RT_TOK - 1) / RT_TOK);
    router_kernel<<<g1, 32 * RT_EXP, 0, st>>>(x, router_w, bias, s.T, s.H, s.E, r.logits);
    const int threads = 32 * (s.T >= 32 ? 32 : (s.T > 4 ? s.T : 4));
    topk_kernel<<<1, threads, 2 * s.E * sizeof(int32_t), st>>>(
        r.logits, s.T, s.E, s.K, s.norm_topk, r.ids, r.wts, r.n_used, r.used_expert,
        r.used_first, r.pair_list);
    return cudaGetLastError();
}

cudaError_t copy_route_out(const MoeShape& s, const Route& r, int32_t* ids_out, float* w_out,
                           cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    if (ids_out)
        e = cudaMemcpyAsync(ids_out, r.ids, sizeof(int32_t) * s.T * s.K, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess && w_out)
        e = cudaMemcpyAsync(w_out, r.wts, sizeof(float) * s.T * s.K, cudaMemcpyDeviceToDevice, st);
    return e;
}

}  // namespace qmoe
