// moe_route.cu -- router GEMV, softmax / top-k / renorm, and the per-expert pair
// lists (the routing half of the qwen3moe MoE FFN).
//
// aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path",
// section "Gaps ... G3": router = F32 GEMV of ffn_gate_inp [E x H]; softmax,
// top-8 and renorm (planned device kernel K1 in G8).  Everything stays on the
// device: no logits copy, no host sync, so the layer is graph-capturable.
#include <float.h>
#include <math.h>

#include "kquant.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

constexpr int RT_TOK = 8;     // tokens per router CTA
constexpr int RT_EXP = 8;     // experts per router CTA (one warp each)

// logits[t][e] = sum_h Wr[e][h] x[t][h] (+ bias[e]), fp32 accumulation.
__global__ void __launch_bounds__(256) router_kernel(const float* __restrict__ x,
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

constexpr int TK_MAXV = 32;   // logits per lane (E <= 1024)

// Per token (one warp): top-K of the F32 logits (ties -> lower index), softmax
// over all E, routing weights renormalised over the K selected.  Then one warp
// builds the per-expert pair lists with a stable counting sort.
__global__ void __launch_bounds__(1024) topk_kernel(const float* __restrict__ logits, int T, int E,
                                                    int K, int norm, int32_t* __restrict__ ids,
                                                    float* __restrict__ wts,
                                                    int32_t* __restrict__ n_used,
                                                    int32_t* __restrict__ used_expert,
                                                    int32_t* __restrict__ used_first,
                                                    int32_t* __restrict__ pair_list) {
    extern __shared__ int32_t sm[];               // counts[E], cursor[E]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int nv = (E + 31) / 32;
    for (int t = warp; t < T; t += nwarps) {
        float v[TK_MAXV];
#pragma unroll
        for (int i = 0; i < TK_MAXV; ++i) {
            const int e = lane + 32 * i;
            v[i] = (i < nv && e < E) ? logits[(size_t)t * E + e] : -INFINITY;
        }
        uint32_t taken = 0u;                      // bit i: v[i] selected
        float vmax = 0.f, psel = 0.f;
        int sel_id[16];
        float sel_v[16];
        for (int j = 0; j < K; ++j) {
            // lane-local best among not-taken (ascending index order inside a lane)
            float bv = -INFINITY;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < TK_MAXV; ++i) {
                const int e = lane + 32 * i;
                const bool cand = i < nv && e < E && !((taken >> i) & 1u);
                if (cand && (bi == 0x7fffffff || v[i] > bv)) { bv = v[i]; bi = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            sel_id[j] = bi;
            sel_v[j] = bv;
            if (j == 0) vmax = bv;
        }
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < TK_MAXV; ++i) {
            const int e = lane + 32 * i;
            if (i < nv && e < E) z += expf(v[i] - vmax);
        }
        z = warp_sum(z);
        for (int j = 0; j < K; ++j) psel += expf(sel_v[j] - vmax) / z;
        if (lane < K) {
            float pj = 0.f;
            int idj = 0;
            for (int j = 0; j < K; ++j)
                if (j == lane) { pj = expf(sel_v[j] - vmax) / z; idj = sel_id[j]; }
            ids[(size_t)t * K + lane] = idj;
            wts[(size_t)t * K + lane] = norm ? pj / psel : pj;
        }
    }
    __syncthreads();
    // ---- per-expert pair lists (stable counting sort by expert id) ----
    int32_t* counts = sm;
    int32_t* cursor = sm + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = 0;
    __syncthreads();
    const int P = T * K;
    for (int p = threadIdx.x; p < P; p += blockDim.x) atomicAdd(&counts[ids[p]], 1);
    __syncthreads();
    if (warp == 0) {
        // exclusive scan over experts + compaction of used experts, in order
        int run = 0, used = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            const int c = e < E ? counts[e] : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const uint32_t nz = __ballot_sync(0xffffffffu, c > 0);
            if (e < E) cursor[e] = run + incl - c;
            if (c > 0) {
                const int slot = used + __popc(nz & ((1u << lane) - 1u));
                used_expert[slot] = e;
                used_first[slot] = run + incl - c;
            }
            run += __shfl_sync(0xffffffffu, incl, 31);
            used += __popc(nz);
        }
        if (lane == 0) { *n_used = used; used_first[used] = P; }
        __syncwarp();
        // stable scatter: chunks of 32 pairs in ascending p
        for (int base = 0; base < P; base += 32) {
            const int p = base + lane;
            const bool act = p < P;
            const int e = act ? ids[p] : -1 - lane;
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int start = act ? cursor[e] : 0;
            __syncwarp();
            if (act) pair_list[start + rank] = p;
            if (act && rank == __popc(peers) - 1) cursor[e] = start + rank + 1;
            __syncwarp();
        }
    }
}

}  // namespace

cudaError_t launch_route(const MoeShape& s, const float* x, const float* router_w,
                         const float* bias, const Route& r, cudaStream_t st) {
    dim3 g1((s.E + RT_EXP - 1) / RT_EXP, (s.T + RT_TOK - 1) / RT_TOK);
    router_kernel<<<g1, 256, 0, st>>>(x, router_w, bias, s.T, s.H, s.E, r.logits);
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
