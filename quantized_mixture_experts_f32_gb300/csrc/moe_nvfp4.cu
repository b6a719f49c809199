// moe_nvfp4.cu -- NVFP4 weights: the BF16 -> NVFP4 runtime quantiser and the
// expert GEMVs of the MoE FFN over NVFP4 experts.
//
// atlasinference source page "spark_model/weight_loader/qwen3.rs", load_layers:
// dense weights are quantised from BF16 to NVFP4 when the model is loaded, by a
// global-absmax kernel and a quantisation kernel.  NVFP4 (the public format):
// FP4 E2M1 elements, two per byte (the even element in the low nibble), one
// E4M3 scale per 16 consecutive elements of a row and one fp32 scale per
// matrix; W[r][c] = e2m1(code) * e4m3(bscale[r][c/16]) * global.
//
// Quantiser (every decision in fp32, in this order): amax = max |x|,
// global = amax / 2688 (448 * 6), per 16-element block s = e4m3_rn(bmax /
// (6 * global)) saturating at 448, d = e4m3(s) * global, code = e2m1_rn(x / d)
// saturating at 6 (ties to the even code; zero where d = 0).
//
// Expert GEMVs: as the FP8 ones (moe_fp8.cu); a 16-byte chunk is 32 weights, so
// a gate/up row of H = 2048 (1 KB) is 4 chunks per lane of a half-warp (items:
// two rows of gate and up) and a down row of F = 768 (384 B) 3 chunks per lane
// of a quarter-warp (items: four rows).  Each chunk's two 16-element halves are
// summed apart and scaled by their block scales; the matrix's global scale
// multiplies the row sum.
#include <math.h>

#include "lowbit_items.cuh"
#include "pdl.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

constexpr int NV_THREADS = 256;

// --------------------------------------------------------------------------- quantiser

__device__ __forceinline__ float bf16_f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// amax of matrix m (blockIdx.y) into amax_bits[m] (non-negative floats order as
// unsigned integers); amax_bits zeroed before the launch
__global__ void __launch_bounds__(256) nvfp4_absmax(const uint16_t* __restrict__ x, size_t n_per,
                                                   unsigned* __restrict__ amax_bits) {
    const uint16_t* xm = x + (size_t)blockIdx.y * n_per;
    float m = 0.f;
    for (size_t i = 8 * ((size_t)blockIdx.x * blockDim.x + threadIdx.x); i < n_per;
         i += 8 * (size_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(xm + i));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m = fmaxf(m, fabsf(bf16_f(w[k] & 0xffffu)));
            m = fmaxf(m, fabsf(bf16_f(w[k] >> 16)));
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits + blockIdx.y, __float_as_uint(m));
}

// nearest E2M1 magnitude code of a >= 0 (ties to the even code), saturating at 6
__device__ __forceinline__ uint32_t e2m1_code(float v) {
    const float a = fabsf(v);
    const uint32_t m = a <= 0.25f ? 0u : a < 0.75f ? 1u : a <= 1.25f ? 2u : a < 1.75f ? 3u
                     : a <= 2.5f ? 4u : a < 3.5f ? 5u : a <= 5.0f ? 6u : 7u;
    return m | (signbit(v) ? 8u : 0u);
}

// one thread per 16-element block of matrix blockIdx.y
__global__ void __launch_bounds__(256) nvfp4_quantize(const uint16_t* __restrict__ x, size_t n_per,
                                                     const unsigned* __restrict__ amax_bits,
                                                     uint8_t* __restrict__ codes,
                                                     uint8_t* __restrict__ bscale) {
    const size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (16 * b >= n_per) return;
    const int m = blockIdx.y;
    const float g = __uint_as_float(amax_bits[m]) / 2688.0f;
    const uint16_t* xb = x + (size_t)m * n_per + 16 * b;
    const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(xb));
    const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(xb + 8));
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    float xf[16];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        xf[2 * k] = bf16_f(w[k] & 0xffffu);
        xf[2 * k + 1] = bf16_f(w[k] >> 16);
    }
    float bmax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) bmax = fmaxf(bmax, fabsf(xf[k]));
    uint32_t s = 0;
    if (g > 0.f) {
        const float den = 6.0f * g;
        s = __nv_cvt_float_to_fp8(bmax / den, __NV_SATFINITE, __NV_E4M3);
    }
    const float d = e4m3_f(s) * g;
    uint32_t out[2] = {0u, 0u};
    if (d > 0.f) {
#pragma unroll
        for (int k = 0; k < 16; ++k) out[k >> 3] |= e2m1_code(xf[k] / d) << (4 * (k & 7));
    }
    *reinterpret_cast<uint2*>(codes + (size_t)m * (n_per / 2) + 8 * b) = make_uint2(out[0], out[1]);
    bscale[(size_t)m * (n_per / 16) + b] = (uint8_t)s;
}

__global__ void nvfp4_global(const unsigned* __restrict__ amax_bits, int n_mats, float* __restrict__ global) {
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m < n_mats) global[m] = __uint_as_float(amax_bits[m]) / 2688.0f;
}

// --------------------------------------------------------------------------- expert GEMVs

// Gate/up + SwiGLU.  Item i -> used expert u = i / (F/2), rows f0 = 2 (i % (F/2))
// and f0 + 1 (half-warp hw takes row f0 + hw of gate and up); NC = H / 512.
// STAGE: the T x rows are first staged in shared memory (padded; few tokens).
template <int NC, bool STAGE>
__global__ void __launch_bounds__(NV_THREADS) nvfp4_gateup_kernel(
    const float* __restrict__ x, int T, int H, int F, int K, const NvExperts w,
    const int32_t* __restrict__ n_used, const int32_t* __restrict__ used_expert,
    const int32_t* __restrict__ used_first, const int32_t* __restrict__ pair_list,
    float* __restrict__ act) {
    extern __shared__ __align__(16) float xs[];
    pdl_wait();
    pdl_launch_dependents();
    if (STAGE) {
        lowbit::vstage(xs, x, T, H);
        __syncthreads();
    }
    const int lane = threadIdx.x & 31, hw = lane >> 4, hl = lane & 15;
    const int gw = (blockIdx.x * NV_THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * NV_THREADS) >> 5;
    const int per = F >> 1;
    const int items = *n_used * per;
    for (int i = gw; i < items; i += nw) {
        const int u = i / per, f = 2 * (i - u * per) + hw;
        if (STAGE)
            lowbit::nv_gateup_rows<NC, lowbit::SRC_SMEM>(xs, lowbit::vpad_ld(H), H, F, K, w, used_expert[u],
                                                         f, hl, pair_list, used_first[u], used_first[u + 1],
                                                         act);
        else
            lowbit::nv_gateup_rows<NC, lowbit::SRC_NC>(x, H, H, F, K, w, used_expert[u], f, hl, pair_list,
                                                       used_first[u], used_first[u + 1], act);
    }
}

// Down projection.  Item i -> used expert u = i / (H/4), rows h0 = 4 (i % (H/4))
// .. h0 + 3 (quarter-warp q takes row h0 + q); NC = F / 256.  STAGE: the P act
// rows are first staged in shared memory (padded).
template <int NC, bool STAGE>
__global__ void __launch_bounds__(NV_THREADS) nvfp4_down_kernel(
    const float* __restrict__ act, int P, int H, int F, const NvExperts w,
    const int32_t* __restrict__ n_used, const int32_t* __restrict__ used_expert,
    const int32_t* __restrict__ used_first, const int32_t* __restrict__ pair_list,
    float* __restrict__ y) {
    extern __shared__ __align__(16) float as[];
    const int lane = threadIdx.x & 31, q = lane >> 3, ql = lane & 7;
    const int gw = (blockIdx.x * NV_THREADS + threadIdx.x) >> 5;
    const int nw = (gridDim.x * NV_THREADS) >> 5;
    const int per = H >> 2;
    // the routing is complete here (see the FP8 down kernel); the first item's
    // weights are loaded before the wait on the gate/up kernel
    const int items = __ldcg(n_used) * per;
    lowbit::NvDown<NC> d;
    if (gw < items) {
        const int u = gw / per;
        lowbit::nv_down_load<NC>(d, w, __ldcg(used_expert + u), 4 * (gw - u * per) + q, H, F, ql);
    }
    pdl_wait();
    pdl_launch_dependents();
    if (STAGE) {
        lowbit::vstage(as, act, P, F);
        __syncthreads();
    }
    for (int i = gw; i < items; i += nw) {
        const int u = i / per, h = 4 * (i - u * per) + q;
        const int e = used_expert[u];
        if (i != gw) lowbit::nv_down_load<NC>(d, w, e, h, H, F, ql);
        if (STAGE)
            lowbit::nv_down_rows<NC, lowbit::SRC_SMEM>(d, w, e, h, H, F, ql, pair_list, used_first[u],
                                                       used_first[u + 1], as, lowbit::vpad_ld(F), y);
        else
            lowbit::nv_down_rows<NC, lowbit::SRC_NC>(d, w, e, h, H, F, ql, pair_list, used_first[u],
                                                     used_first[u + 1], act, F, y);
    }
}

// x / act rows are staged in shared memory when they fit in this much
constexpr size_t NV_STAGE_MAX = 72 * 1024;

template <int NC>
cudaError_t nv_gateup(const MoeShape& s, const float* x, const NvExperts& w, const Route& r,
                      float* act, int items, int num_sms, cudaStream_t st) {
    const size_t smem = sizeof(float) * (size_t)s.T * lowbit::vpad_ld(s.H);
    if (smem <= NV_STAGE_MAX) {
        static int resident = 0;   // per instantiation, at the largest staging
        const int grid = strided_grid(nvfp4_gateup_kernel<NC, true>, NV_THREADS, &resident, items, num_sms,
                                      NV_STAGE_MAX);
        return launch_pdl(nvfp4_gateup_kernel<NC, true>, dim3(grid), dim3(NV_THREADS), smem, st, x, s.T,
                          s.H, s.F, s.K, w, r.n_used, r.used_expert, r.used_first, r.pair_list, act);
    }
    static int resident = 0;
    const int grid = strided_grid(nvfp4_gateup_kernel<NC, false>, NV_THREADS, &resident, items, num_sms, 0);
    return launch_pdl(nvfp4_gateup_kernel<NC, false>, dim3(grid), dim3(NV_THREADS), 0, st, x, s.T, s.H,
                      s.F, s.K, w, r.n_used, r.used_expert, r.used_first, r.pair_list, act);
}

template <int NC>
cudaError_t nv_down(const MoeShape& s, const float* act, const NvExperts& w, const Route& r,
                    float* y, int items, int num_sms, cudaStream_t st) {
    const int P = s.T * s.K;
    const size_t smem = sizeof(float) * (size_t)P * lowbit::vpad_ld(s.F);
    if (smem <= NV_STAGE_MAX) {
        static int resident = 0;
        const int grid = strided_grid(nvfp4_down_kernel<NC, true>, NV_THREADS, &resident, items, num_sms,
                                      NV_STAGE_MAX);
        return launch_pdl(nvfp4_down_kernel<NC, true>, dim3(grid), dim3(NV_THREADS), smem, st, act, P, s.H,
                          s.F, w, r.n_used, r.used_expert, r.used_first, r.pair_list, y);
    }
    static int resident = 0;
    const int grid = strided_grid(nvfp4_down_kernel<NC, false>, NV_THREADS, &resident, items, num_sms, 0);
    return launch_pdl(nvfp4_down_kernel<NC, false>, dim3(grid), dim3(NV_THREADS), 0, st, act, P, s.H, s.F,
                      w, r.n_used, r.used_expert, r.used_first, r.pair_list, y);
}

}  // namespace

bool nvfp4_supported(int H, int F) {
    const int nh = H / 512, nf = F / 256;
    return H % 512 == 0 && F % 256 == 0 && (nh == 1 || nh == 2 || nh == 4 || nh == 8) && nf >= 1 &&
           nf <= 6;
}

cudaError_t launch_nvfp4_experts(const MoeShape& s, const float* x, const NvExperts& w,
                                 const Route& r, float* act, float* y, int num_sms, cudaStream_t st) {
    if (!nvfp4_supported(s.H, s.F)) return cudaErrorInvalidValue;
    const int maxu = s.T * s.K < s.E ? s.T * s.K : s.E;   // used experts, an upper bound
    const int i1 = maxu * (s.F / 2), i2 = maxu * (s.H / 4);
    cudaError_t e;
    switch (s.H / 512) {
        case 1: e = nv_gateup<1>(s, x, w, r, act, i1, num_sms, st); break;
        case 2: e = nv_gateup<2>(s, x, w, r, act, i1, num_sms, st); break;
        case 4: e = nv_gateup<4>(s, x, w, r, act, i1, num_sms, st); break;
        default: e = nv_gateup<8>(s, x, w, r, act, i1, num_sms, st); break;
    }
    if (e != cudaSuccess) return e;
    switch (s.F / 256) {
        case 1: return nv_down<1>(s, act, w, r, y, i2, num_sms, st);
        case 2: return nv_down<2>(s, act, w, r, y, i2, num_sms, st);
        case 3: return nv_down<3>(s, act, w, r, y, i2, num_sms, st);
        case 4: return nv_down<4>(s, act, w, r, y, i2, num_sms, st);
        case 5: return nv_down<5>(s, act, w, r, y, i2, num_sms, st);
        default: return nv_down<6>(s, act, w, r, y, i2, num_sms, st);
    }
}

cudaError_t launch_nvfp4_quantize(const uint16_t* x, int n_mats, int rows, int cols, uint8_t* codes,
                                  uint8_t* bscale, float* global, unsigned* amax_bits, int num_sms,
                                  cudaStream_t st) {
    const size_t n_per = (size_t)rows * cols;
    cudaError_t e = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned) * n_mats, st);
    if (e != cudaSuccess) return e;
    const size_t want = (n_per / 8 + 255) / 256;
    const int gx = (int)(want < (size_t)(4 * num_sms) ? (want > 0 ? want : 1) : (size_t)(4 * num_sms));
    nvfp4_absmax<<<dim3(gx, n_mats), 256, 0, st>>>(x, n_per, amax_bits);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t nb = n_per / 16;
    nvfp4_quantize<<<dim3((unsigned)((nb + 255) / 256), n_mats), 256, 0, st>>>(x, n_per, amax_bits, codes,
                                                                              bscale);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    nvfp4_global<<<(n_mats + 255) / 256, 256, 0, st>>>(amax_bits, n_mats, global);
    return cudaGetLastError();
}

}  // namespace qmoe
