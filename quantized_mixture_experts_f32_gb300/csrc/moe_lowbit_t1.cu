// moe_lowbit_t1.cu -- the whole MoE layer for one token over FP8 or NVFP4
// experts in one launch of one CTA per SM, a programmatic dependent of the
// previous kernel (its router rows prefetched into L2 before the wait).
//
// The layer's steps (aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working
// CUDA path", "Gaps ... G3") over the formats of the atlasinference source page
// "spark_model/weight_loader/qwen3.rs", load_layers (FP8 block-128 and NVFP4
// experts, full-precision router).  The structure of the k-quant batch-1
// kernel, without grid barriers:
//   A  x staged in shared memory (padded); CTA c computes the router logit of
//      expert c (fixed-order reduction) and publishes it as a tagged word
//      {value, launch tag}.
//   B  every CTA polls the E tagged logits (bounded) and selects the top-K with
//      their weights itself (the same deterministic result in every CTA).
//   C  gate/up items (two rows of one slot) grid-strided over all warps; SiLU(g)*u
//      stored to act [K][F]; one arrival per CTA on a counter.
//   D  after every CTA has arrived (bounded wait), act staged in shared memory;
//      the CTA owns 4-row groups [q0, q1) of the output: y_j for its rows and
//      every slot j into shared memory, then out[h] = x[h] + sum_j w_j y_j[h] in
//      slot order, written directly (no combine pass).
// The last CTA out resets the counters and publishes the launch tag that the
// next launch increments.  Every wait gives up after WAIT_LIMIT_NS, records the
// timeout status and lets the CTA fall through to its arrivals.
#include <math.h>

#include "lowbit_items.cuh"
#include "pdl.cuh"
#include "ptx_sync.cuh"
#include "qmoe_internal.h"
#include "topk.cuh"

namespace qmoe {

namespace {

constexpr int LT_THREADS = 512;
constexpr int LT_WARPS = LT_THREADS / 32;
constexpr int LT_KMAX = 16;

struct LtParams {
    const float* x;       // [H], also the residual
    const float* router;  // [E][H] F32
    int H, E, K, F, norm;
    Fp8Experts f8;
    NvExperts nv;
    float* act;           // [K][F] workspace
    float* out;           // [H] (may alias x: written only after every CTA has read x)
    int32_t* ids_out;     // [K] or null
    float* w_out;         // [K] or null
    unsigned long long* lg;  // [E] tagged logits
    unsigned* ctl;        // [0] exit counter, [1] tag of the last completed launch, [3] act arrivals
    int* status;
};

template <int FMT, int NCG, int NCD>
__global__ void __launch_bounds__(LT_THREADS, 1) lowbit_t1(const LtParams p) {
    extern __shared__ __align__(16) float smf[];
    const int H = p.H, E = p.E, K = p.K, F = p.F, G = gridDim.x;
    const int xld = lowbit::vpad_ld(H), ald = lowbit::vpad_ld(F);
    float* xs = smf;                                   // [xld]
    float* as = xs + xld;                              // [K][ald]
    float* ys = as + (size_t)K * ald;                  // [K][H]
    float* lgs = ys + (size_t)K * H;                   // [E]
    __shared__ float red[LT_WARPS];
    __shared__ int s_sel[LT_KMAX], s_slot[LT_KMAX], s_ok;
    __shared__ float s_w[LT_KMAX];
    __shared__ unsigned s_tag;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // before the previous kernel on the stream has finished: weights only (this
    // CTA's router rows towards L2); x, the control words and the logits after
    if (tid == 0)
        for (int e = blockIdx.x; e < E; e += G) bulk_prefetch_l2(p.router + (size_t)e * H, (uint32_t)(H * 4));
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0) {
        s_tag = ld_acquire_gpu(p.ctl + 1) + 1u;
        s_ok = 1;
    }
    if (tid < LT_KMAX) s_slot[tid] = tid;
    lowbit::vstage(xs, p.x, 1, H);
    __syncthreads();
    const unsigned tag = s_tag;

    // ---- A: the router logit of expert blockIdx.x (and + G, ...)
    for (int e = blockIdx.x; e < E; e += G) {
        const float* wrow = p.router + (size_t)e * H;
        float acc = 0.f;
        for (int h = 4 * tid; h < H; h += 4 * LT_THREADS) {
            const float4 w = __ldg(reinterpret_cast<const float4*>(wrow + h));
            const float4 v = __ldg(reinterpret_cast<const float4*>(p.x + h));
            acc = fmaf(w.x, v.x, acc);
            acc = fmaf(w.y, v.y, acc);
            acc = fmaf(w.z, v.z, acc);
            acc = fmaf(w.w, v.w, acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (tid == 0) {
            float v = 0.f;
            for (int w = 0; w < LT_WARPS; ++w) v += red[w];
            st_relaxed_u64(p.lg + e, tag_pack(v, tag));
        }
        __syncthreads();
    }

    // ---- B: every logit of this launch, then the top-K in every CTA
    if (tid < E) {
        float v;
        if (!poll_tagged(p.lg + tid, tag, v)) s_ok = 0;
        lgs[tid] = v;
    }
    __syncthreads();
    bool ok = s_ok != 0;
    if (ok && warp == 0) {
        int id;
        float wt;
        topk_warp128<true>(lgs, E, K, p.norm, id, wt);
        if (lane < K) {
            s_sel[lane] = id;
            s_w[lane] = wt;
            if (blockIdx.x == 0) {
                if (p.ids_out) p.ids_out[lane] = id;
                if (p.w_out) p.w_out[lane] = wt;
            }
        }
    }
    __syncthreads();

    // ---- C: gate/up items, every warp of the grid.  Warps are numbered warp-major
    // over the CTAs, so the items beyond one per warp fall on a few warps of every
    // CTA rather than on every warp of the first CTAs.
    const int nq = H >> 2;
    const int q0 = (int)((long)nq * blockIdx.x / G), q1 = (int)((long)nq * (blockIdx.x + 1) / G);
    if (ok) {
        const int gw = warp * G + blockIdx.x, nw = G * LT_WARPS;
        const int hw = lane >> 4, hl = lane & 15, per = F >> 1;
        if (lane == 0) {
            // the rows of this warp's later items start towards L2 now, while its
            // first item computes
            for (int i = gw + nw; i < K * per; i += nw) {
                const int j = i / per;
                const size_t row = (size_t)s_sel[j] * F + 2 * (i - j * per);
                if (FMT == 1) {
                    bulk_prefetch_l2(p.f8.gate + row * H, (uint32_t)(2 * H));
                    bulk_prefetch_l2(p.f8.up + row * H, (uint32_t)(2 * H));
                } else {
                    bulk_prefetch_l2(p.nv.gate + row * (H / 2), (uint32_t)H);
                    bulk_prefetch_l2(p.nv.up + row * (H / 2), (uint32_t)H);
                    bulk_prefetch_l2(p.nv.gate_bs + row * (H / 16), (uint32_t)(H / 8));
                    bulk_prefetch_l2(p.nv.up_bs + row * (H / 16), (uint32_t)(H / 8));
                }
            }
        }
        for (int i = gw; i < K * per; i += nw) {
            const int j = i / per, f = 2 * (i - j * per) + hw;
            if (FMT == 1)
                lowbit::f8_gateup_rows<NCG, lowbit::SRC_SMEM>(xs, xld, H, F, K, p.f8, s_sel[j], f, hl, s_slot,
                                                              j, j + 1, p.act);
            else
                lowbit::nv_gateup_rows<NCG, lowbit::SRC_SMEM>(xs, xld, H, F, K, p.nv, s_sel[j], f, hl, s_slot,
                                                              j, j + 1, p.act);
        }
        if (lane == 0 && warp < K) {
            // slot `warp`'s down rows of this CTA start towards L2 once the warp's
            // gate/up bytes are in (they stream while the grid gathers at the
            // act counter)
            const size_t r0 = (size_t)s_sel[warp] * H + 4 * q0;
            const uint32_t nr = (uint32_t)(4 * (q1 - q0));
            if (FMT == 1) {
                bulk_prefetch_l2(p.f8.down + r0 * F, nr * (uint32_t)F);
            } else {
                bulk_prefetch_l2(p.nv.down + r0 * (F / 2), nr * (uint32_t)(F / 2));
                bulk_prefetch_l2(p.nv.down_bs + r0 * (F / 16), nr * (uint32_t)(F / 16));
            }
        }
    }
    __syncthreads();
    if (tid == 0) {
        grid_arrive(p.ctl + 3);
        if (!grid_wait(p.ctl + 3, (unsigned)G)) s_ok = 0;
    }
    __syncthreads();
    ok = ok && s_ok != 0;

    // ---- D: this CTA's output rows, every slot, then the combine
    if (ok) {
        lowbit::vstage(as, p.act, K, F);
        __syncthreads();
        const int sub = FMT == 1 ? (lane >> 4) : (lane >> 3), sl = FMT == 1 ? (lane & 15) : (lane & 7);
        const int nt = K * (q1 - q0);
        for (int t = warp; t < nt; t += LT_WARPS) {
            const int j = t / (q1 - q0), h = 4 * (q0 + t - j * (q1 - q0)) + sub;
            if (FMT == 1) {
                lowbit::F8Down<NCD> d;
                lowbit::f8_down_load<NCD>(d, p.f8, s_sel[j], h, H, F, sl);
                lowbit::f8_down_rows<NCD, lowbit::SRC_SMEM>(d, p.f8, s_sel[j], h, H, F, sl, s_slot, j, j + 1,
                                                            as, ald, ys);
            } else {
                lowbit::NvDown<NCD> d;
                lowbit::nv_down_load<NCD>(d, p.nv, s_sel[j], h, H, F, sl);
                lowbit::nv_down_rows<NCD, lowbit::SRC_SMEM>(d, p.nv, s_sel[j], h, H, F, sl, s_slot, j, j + 1,
                                                            as, ald, ys);
            }
        }
        __syncthreads();
        for (int h = 4 * q0 + tid; h < 4 * q1; h += LT_THREADS) {
            float acc = p.x[h];
            for (int j = 0; j < K; ++j) acc = fmaf(s_w[j], ys[(size_t)j * H + h], acc);
            p.out[h] = acc;
        }
    }
    if (!ok && tid == 0) atomicCAS(p.status, 0, ST_TIMEOUT);
    __syncthreads();
    if (tid == 0 && atomicAdd(p.ctl + 0, 1u) == (unsigned)G - 1) {
        // every CTA is past every wait: reset the counters, publish the tag
        atomicExch(p.ctl + 3, 0u);
        atomicExch(p.ctl + 0, 0u);
        atomicExch(p.ctl + 1, tag);
    }
}

size_t lt_smem(int H, int E, int K, int F) {
    return sizeof(float) * ((size_t)lowbit::vpad_ld(H) + (size_t)K * lowbit::vpad_ld(F) + (size_t)K * H + E);
}

template <int FMT, int NCG, int NCD>
cudaError_t lt_launch(const LtParams& p, int num_sms, cudaStream_t st) {
    const size_t smem = lt_smem(p.H, p.E, p.K, p.F);
    static bool attr = false;   // per instantiation
    if (!attr) {
        const cudaError_t e = cudaFuncSetAttribute(lowbit_t1<FMT, NCG, NCD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    // one CTA per SM (the register file holds one 512-thread CTA at 128 registers),
    // grid = SM count: every CTA is resident once the previous kernel's CTAs have
    // left, and those never wait on this grid
    return launch_pdl(lowbit_t1<FMT, NCG, NCD>, dim3(num_sms), dim3(LT_THREADS), smem, st, p);
}

}  // namespace

bool lowbit_t1_supported(int fmt, int T, int H, int E, int K, int F, int num_sms) {
    // the instantiated shape (hidden 2048, ffn 768); E <= 128 (one warp's
    // top-K, every expert's logit by its own CTA); one output 4-row group per CTA
    // at least
    return (fmt == 1 || fmt == 2) && T == 1 && H == 2048 && F == 768 && E <= 128 && E <= num_sms &&
           K >= 1 && K <= LT_KMAX && num_sms <= H / 4 && lt_smem(H, E, K, F) <= 200 * 1024;
}

cudaError_t launch_lowbit_t1(int fmt, const MoeShape& s, const float* x, const float* router_w,
                             const Fp8Experts* f8, const NvExperts* nv, float* act, float* out,
                             int32_t* ids_out, float* w_out, unsigned long long* lg, unsigned* ctl,
                             int* status, int num_sms, cudaStream_t st) {
    if (!lowbit_t1_supported(fmt, s.T, s.H, s.E, s.K, s.F, num_sms)) return cudaErrorInvalidValue;
    LtParams p{x, router_w, s.H, s.E, s.K, s.F, s.norm_topk, f8 ? *f8 : Fp8Experts{}, nv ? *nv : NvExperts{},
               act, out, ids_out, w_out, lg, ctl, status};
    // hidden 2048, ffn 768: FP8 gate/up 8 chunks a lane, down 3; NVFP4 4 and 3
    return fmt == 1 ? lt_launch<1, 8, 3>(p, num_sms, st) : lt_launch<2, 4, 3>(p, num_sms, st);
}

}  // namespace qmoe
