// topk.cuh -- softmax / top-k / renorm of F32 router logits and the per-expert
// pair lists, run by one thread block (the routing of the qwen3moe MoE FFN:
// aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path",
// "Gaps ... G3": softmax, top-8, renorm over the F32 router logits), used by the
// routing kernels of moe_route.cu.
#pragma once
#include <climits>
#include <math.h>

#include "kquant.cuh"

namespace qmoe {
namespace {

// the map is its own inverse
__device__ __forceinline__ float key_value(int k) { return __int_as_float(k ^ ((k >> 31) & 0x7fffffff)); }

constexpr int TK_MAXV = 32;   // logits per lane (E <= 1024)

// One token's top-K of up to 128 F32 logits by one warp (ties to the lower
// index), softmax over all E and the weights renormalised over the K selected
// (norm), lane j < K ending with selection j (id and weight).  Lane l sorts the
// (order key, index) pairs of experts l, l + 32, l + 64, l + 96 (larger key
// first), then K tournament rounds over the 32 lane heads: the largest head key
// by one warp max-reduction, the lowest index holding it by one min-reduction,
// the owner drops its head.  SMEM: logits in shared memory (else global memory,
// read through L2: they may come from other CTAs of the same launch).
template <bool SMEM>
__device__ __forceinline__ void topk_warp128(const float* lt, int E, int K, int norm, int& my_id,
                                             float& my_w) {
    const int lane = threadIdx.x & 31;
    auto ld = [&](int i) { return SMEM ? lt[i] : __ldcg(lt + i); };
    int ks[4], is[4];
#pragma unroll
    for (int z = 0; z < 4; ++z) {
        const int i = lane + 32 * z;
        ks[z] = i < E ? order_key(ld(i)) : INT_MIN;
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
    my_id = 0;
    float my_v = 0.f, vmax = 0.f;
    for (int r = 0; r < K; ++r) {
        const int mk = __reduce_max_sync(0xffffffffu, ks[0]);
        const int wi = (int)__reduce_min_sync(0xffffffffu, ks[0] == mk ? (unsigned)is[0] : 0xffffffffu);
        if (r == 0) vmax = key_value(mk);
        if (lane == r) {
            my_id = wi;
            my_v = key_value(mk);
        }
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
    float z = 0.f;
    for (int i = lane; i < E; i += 32) z += expf(ld(i) - vmax);
    z = warp_sum(z);
    const float pj = lane < K ? expf(my_v - vmax) / z : 0.f;
    const float psel = warp_sum(pj);
    my_w = norm ? pj / psel : pj;
}

// Per token (one warp): top-K of the F32 logits (ties -> lower index), softmax
// over all E, routing weights renormalised over the K selected.  Then one warp
// builds the per-expert pair lists with a stable counting sort.
// The whole top-k / lists step for T tokens, run by one block of any size that
// is a multiple of 32 (blockDim.x <= 1024).  Logits are read through L2 (they
// may come from other CTAs of the same launch).  sm: 2 E ints of shared memory.
__device__ __noinline__ void topk_lists(const float* __restrict__ logits, int T, int E, int K, int norm,
                           int32_t* __restrict__ ids, float* __restrict__ wts,
                           int32_t* __restrict__ n_used, int32_t* __restrict__ used_expert,
                           int32_t* __restrict__ used_first, int32_t* __restrict__ pair_list,
                           int32_t* sm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int nv = (E + 31) / 32;
    for (int t = warp; E <= 128 && t < T; t += nwarps) {
        int my_id;
        float my_w;
        topk_warp128<false>(logits + (size_t)t * E, E, K, norm, my_id, my_w);
        if (lane < K) {
            ids[(size_t)t * K + lane] = my_id;
            wts[(size_t)t * K + lane] = my_w;
        }
    }
    for (int t = warp; E > 128 && t < T; t += nwarps) {
        int v[TK_MAXV];                           // order keys; INT_MIN pads
#pragma unroll
        for (int i = 0; i < TK_MAXV; ++i) {
            const int e = lane + 32 * i;
            v[i] = (i < nv && e < E) ? order_key(__ldcg(logits + (size_t)t * E + e)) : INT_MIN;
        }
        uint32_t taken = 0u;                      // bit i: v[i] selected
        float vmax = 0.f, psel = 0.f;
        int sel_id[16];
        float sel_v[16];
        for (int j = 0; j < K; ++j) {
            // lane-local best among not-taken (ascending index order inside a lane);
            // (key, lower index) is a total order, so every lane agrees on the result
            int bv = INT_MIN;
            int bi = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < TK_MAXV; ++i) {
                const int e = lane + 32 * i;
                const bool cand = i < nv && e < E && !((taken >> i) & 1u);
                if (cand && (bi == 0x7fffffff || v[i] > bv)) { bv = v[i]; bi = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const int ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
            }
            if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
            sel_id[j] = bi;
            sel_v[j] = key_value(bv);
            if (j == 0) vmax = sel_v[0];
        }
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < TK_MAXV; ++i) {
            const int e = lane + 32 * i;
            if (i < nv && e < E) z += expf(key_value(v[i]) - vmax);
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
}  // namespace qmoe
