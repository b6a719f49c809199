// moe_fp8.cu -- expert GEMVs of the MoE FFN over FP8 block-scaled experts.
//
// atlasinference source page "spark_model/weight_loader/qwen3.rs", load_layers:
// experts stored as FP8 with one scale per 128 x 128 block ("Native FP8 MoE"),
// consumed with FP8 weights and 16-bit-or-wider activations (the "w8a16"
// remark), routed by a full-precision router.  Codes are OCP E4M3 ("e4m3fn");
// W[r][c] = e4m3(code[r][c]) * scale[r / 128][c / 128].  Layout per 3-D tensor:
// codes [E][rows][cols] bytes, scales [E][rows/128][cols/128] fp32.
//
// Each E4M3 pair is widened with the hardware e4m3x2 -> f16x2 conversion (exact:
// every E4M3 value is an fp16 value), then to fp32; x, act and every sum are
// fp32.  A 16-byte chunk of a row (16 weights) never straddles a 128-column
// scale block, so a lane multiplies its chunk's partial dot by one scale.
//
// Work is expert-centric and grid-strided: a warp item is two rows (one per
// half-warp) of gate and up, or four rows of down, of one used expert; the
// lane's chunks of every row of the item are loaded before any is used, so a
// lane keeps 16 (gate/up) or 6 (down) 16-byte loads in flight.  Both kernels are programmatic
// dependents of the kernel before them; the down kernel loads its first item's
// weights while the gate/up kernel still runs.
#include <math.h>

#include "lowbit_items.cuh"
#include "pdl.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

constexpr int F8_THREADS = 256;

// Gate/up + SwiGLU.  Item i -> used expert u = i / (F/2), rows f0 = 2 (i % (F/2))
// and f0 + 1 (half-warp hw takes row f0 + hw of both gate and up); NC = H / 256.
// STAGE: the T x rows are first staged in shared memory (padded; few tokens).
template <int NC, bool STAGE>
__global__ void __launch_bounds__(F8_THREADS) fp8_gateup_kernel(
    const float* __restrict__ x, int T, int H, int F, int K, const Fp8Experts w,
    const int32_t* __restrict__ n_used, const int32_t* __restrict__ used_expert,
    const int32_t* __restrict__ used_first, const int32_t* __restrict__ pair_list,
    float* __restrict__ act) {
    extern __shared__ __align__(16) float xs[];
    pdl_wait();                 // the routing of this call
    pdl_launch_dependents();
    if (STAGE) {
        lowbit::vstage(xs, x, T, H);
        __syncthreads();
    }
    const int lane = threadIdx.x & 31, hw = lane >> 4, hl = lane & 15;
    const int gw = (blockIdx.x * F8_THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * F8_THREADS) >> 5;
    const int per = F >> 1;
    const int items = *n_used * per;
    for (int i = gw; i < items; i += nw) {
        const int u = i / per, f = 2 * (i - u * per) + hw;
        if (STAGE)
            lowbit::f8_gateup_rows<NC, lowbit::SRC_SMEM>(xs, lowbit::vpad_ld(H), H, F, K, w, used_expert[u],
                                                         f, hl, pair_list, used_first[u], used_first[u + 1],
                                                         act);
        else
            lowbit::f8_gateup_rows<NC, lowbit::SRC_NC>(x, H, H, F, K, w, used_expert[u], f, hl, pair_list,
                                                       used_first[u], used_first[u + 1], act);
    }
}

// Down projection.  Item i -> used expert u = i / (H/4), rows h0 = 4 (i % (H/4)) ..
// h0 + 3; half-warp hw takes rows h0 + hw and h0 + 2 + hw; NC = F / 256.
// STAGE: the P act rows are first staged in shared memory (padded).
template <int NC, bool STAGE>
__global__ void __launch_bounds__(F8_THREADS) fp8_down_kernel(
    const float* __restrict__ act, int P, int H, int F, const Fp8Experts w,
    const int32_t* __restrict__ n_used, const int32_t* __restrict__ used_expert,
    const int32_t* __restrict__ used_first, const int32_t* __restrict__ pair_list,
    float* __restrict__ y) {
    extern __shared__ __align__(16) float as[];
    const int lane = threadIdx.x & 31, hw = lane >> 4, hl = lane & 15;
    const int gw = (blockIdx.x * F8_THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * F8_THREADS) >> 5;
    const int per = H >> 2;
    // The routing was written two kernels back: the gate/up kernel lets this one
    // launch only after its own wait on the routing kernel, so the lists are
    // complete here and are read through L2.  The first item's weights are
    // loaded before the wait on the gate/up kernel (they are never written).
    const int items = __ldcg(n_used) * per;
    lowbit::F8Down<NC> d;
    if (gw < items) {
        const int u = gw / per;
        lowbit::f8_down_load<NC>(d, w, __ldcg(used_expert + u), 4 * (gw - u * per) + hw, H, F, hl);
    }
    pdl_wait();                 // act of this call
    pdl_launch_dependents();
    if (STAGE) {
        lowbit::vstage(as, act, P, F);
        __syncthreads();
    }
    for (int i = gw; i < items; i += nw) {
        const int u = i / per, h = 4 * (i - u * per) + hw;
        const int e = used_expert[u];
        if (i != gw) lowbit::f8_down_load<NC>(d, w, e, h, H, F, hl);
        if (STAGE)
            lowbit::f8_down_rows<NC, lowbit::SRC_SMEM>(d, w, e, h, H, F, hl, pair_list, used_first[u],
                                                       used_first[u + 1], as, lowbit::vpad_ld(F), y);
        else
            lowbit::f8_down_rows<NC, lowbit::SRC_NC>(d, w, e, h, H, F, hl, pair_list, used_first[u],
                                                     used_first[u + 1], act, F, y);
    }
}

// x / act rows are staged in shared memory when they fit in this much
constexpr size_t LB_STAGE_MAX = 72 * 1024;

template <int NC>
cudaError_t gateup_nc(const MoeShape& s, const float* x, const Fp8Experts& w, const Route& r,
                      float* act, int items, int num_sms, cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)s.T * lowbit::vpad_ld(s.H);
    if (smem <= LB_STAGE_MAX) {
        static int resident = 0;   // per instantiation, at the largest staging
        const int grid = strided_grid(fp8_gateup_kernel<NC, true>, F8_THREADS, &resident, items, num_sms,
                                      LB_STAGE_MAX);
        return launch_pdl(fp8_gateup_kernel<NC, true>, dim3(grid), dim3(F8_THREADS), smem, st, x, s.T, s.H,
                          s.F, s.K, w, r.n_used, r.used_expert, r.used_first, r.pair_list, act);
    }
    static int resident = 0;
    const int grid = strided_grid(fp8_gateup_kernel<NC, false>, F8_THREADS, &resident, items, num_sms, 0);
    return launch_pdl(fp8_gateup_kernel<NC, false>, dim3(grid), dim3(F8_THREADS), 0, st, x, s.T, s.H, s.F,
                      s.K, w, r.n_used, r.used_expert, r.used_first, r.pair_list, act);
}

template <int NC>
cudaError_t down_nc(const MoeShape& s, const float* act, const Fp8Experts& w, const Route& r,
                    float* y, int items, int num_sms, cudaStream_t st) {
    const int P = s.T * s.K;
    const size_t smem = sizeof(float) * (size_t)P * lowbit::vpad_ld(s.F);
    if (smem <= LB_STAGE_MAX) {
        static int resident = 0;
        const int grid = strided_grid(fp8_down_kernel<NC, true>, F8_THREADS, &resident, items, num_sms,
                                      LB_STAGE_MAX);
        return launch_pdl(fp8_down_kernel<NC, true>, dim3(grid), dim3(F8_THREADS), smem, st, act, P, s.H,
                          s.F, w, r.n_used, r.used_expert, r.used_first, r.pair_list, y);
    }
    static int resident = 0;
    const int grid = strided_grid(fp8_down_kernel<NC, false>, F8_THREADS, &resident, items, num_sms, 0);
    return launch_pdl(fp8_down_kernel<NC, false>, dim3(grid), dim3(F8_THREADS), 0, st, act, P, s.H, s.F, w,
                      r.n_used, r.used_expert, r.used_first, r.pair_list, y);
}

}  // namespace

bool fp8_supported(int H, int F) {
    const int nh = H / 256, nf = F / 256;
    return H % 256 == 0 && F % 256 == 0 && (nh == 2 || nh == 4 || nh == 8 || nh == 16) &&
           (nf >= 1 && nf <= 6);
}

cudaError_t launch_fp8_experts(const MoeShape& s, const float* x, const Fp8Experts& w,
                               const Route& r, float* act, float* y, int num_sms, cudaStream_t st) {
    if (!fp8_supported(s.H, s.F)) return cudaErrorInvalidValue;
    const int maxu = s.T * s.K < s.E ? s.T * s.K : s.E;   // used experts, an upper bound
    const int i1 = maxu * (s.F / 2), i2 = maxu * (s.H / 4);
    cudaError_t e;
    switch (s.H / 256) {
        case 2: e = gateup_nc<2>(s, x, w, r, act, i1, num_sms, st); break;
        case 4: e = gateup_nc<4>(s, x, w, r, act, i1, num_sms, st); break;
        case 8: e = gateup_nc<8>(s, x, w, r, act, i1, num_sms, st); break;
        default: e = gateup_nc<16>(s, x, w, r, act, i1, num_sms, st); break;
    }
    if (e != cudaSuccess) return e;
    switch (s.F / 256) {
        case 1: return down_nc<1>(s, act, w, r, y, i2, num_sms, st);
        case 2: return down_nc<2>(s, act, w, r, y, i2, num_sms, st);
        case 3: return down_nc<3>(s, act, w, r, y, i2, num_sms, st);
        case 4: return down_nc<4>(s, act, w, r, y, i2, num_sms, st);
        case 5: return down_nc<5>(s, act, w, r, y, i2, num_sms, st);
        default: return down_nc<6>(s, act, w, r, y, i2, num_sms, st);
    }
}

}  // namespace qmoe
