// lowbit.cuh -- helpers shared by the expert GEMVs over FP8 and NVFP4 weights:
// hardware widening of E4M3 / E2M1 pairs, streaming 16-byte loads, lane-group
// sums and the grid of a grid-strided launch.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmoe {

// two E4M3 codes (low byte first) -> two floats (exact: every E4M3 value is an fp16 value)
__device__ __forceinline__ float2 e4m3x2_f2(uint32_t two) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    return __half22float2(__half2(r));
}

__device__ __forceinline__ float e4m3_f(uint32_t one) {
    const __half_raw r = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(one & 0xffu), __NV_E4M3);
    return __half2float(__half(r));
}

// two E2M1 codes of one byte (low nibble first) -> two floats (exact)
__device__ __forceinline__ float2 e2m1x2_f2(uint32_t byte) {
    const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(static_cast<__nv_fp4x2_storage_t>(byte & 0xffu), __NV_E2M1);
    return __half22float2(__half2(r));
}

__device__ __forceinline__ uint4 ld_stream(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// An opaque identity on a register-held weight chunk: applied at the top of a
// loop over tokens, it keeps the compiler from widening every weight once
// before the loop (loop-invariant hoisting that needs several times the
// registers the raw bytes do) and makes it widen them per use instead.
__device__ __forceinline__ void opaque(uint4& w) {
    asm volatile("" : "+r"(w.x), "+r"(w.y), "+r"(w.z), "+r"(w.w));
}

// sum over aligned groups of W lanes (every lane gets its group's sum)
template <int W>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
    for (int o = W / 2; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// CTAs of a grid-strided launch: enough for every warp item, at most the CTAs
// resident at once (resident: per-kernel cache, filled on first use)
template <typename Kern>
int strided_grid(Kern kern, int threads, int* resident, int items, int num_sms, size_t smem = 0) {
    if (!*resident) {
        int n = 0;
        if (smem && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                        cudaSuccess)
            cudaGetLastError();
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess || n < 1)
            n = 1;
        *resident = n;
    }
    const int warps = threads / 32;
    const int need = (items + warps - 1) / warps;
    const int cap = num_sms * *resident;
    return need < cap ? (need > 0 ? need : 1) : cap;
}

}  // namespace qmoe
