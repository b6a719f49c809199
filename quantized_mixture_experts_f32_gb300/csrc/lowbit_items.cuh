// lowbit_items.cuh -- the per-item work of the FP8 and NVFP4 expert GEMVs of the
// grid-strided kernels (moe_fp8.cu, moe_nvfp4.cu).
//
// FP8 (atlasinference source page "spark_model/weight_loader/qwen3.rs",
// load_layers: FP8 weights with one scale per 128 x 128 block): a 16-byte chunk
// is 16 weights inside one scale block.  NVFP4 (same page: BF16 -> NVFP4 at
// load): a 16-byte chunk is 32 weights, two 16-element scale blocks.
//
// Gate/up items: rows f of gate and up of one expert, one half-warp per row (lane
// chunk k of a row at byte 16 ((lane & 15) + 16 k)).  Down items: FP8 rows h and
// h + 2 per half-warp, NVFP4 row h per quarter-warp (an F = 768 row of 384 B is
// 3 chunks a lane of 8).  Every item handles all pairs plist[p0 .. p1) routed to
// its expert; weights are widened per use (the opaque identity at the top of the
// pair loop keeps the compiler from widening them all once before it).
#pragma once
#include <math.h>

#include "lowbit.cuh"
#include "qmoe_internal.h"

namespace qmoe {
namespace lowbit {

// Where a dot's fp32 values come from (x rows by token, act rows by pair):
//   SRC_NC    global memory, read-only for the kernel (the non-coherent path)
//   SRC_CG    global memory written earlier in the same kernel (through L2)
//   SRC_SMEM  staged in shared memory with 4 floats of padding after every 64
//             (column c at c + 4 (c / 64)): a lane's 16- or 32-float run then
//             sits 64 or 128 bytes + 16 from its neighbour's, so one 16-byte
//             load instruction of a half-warp touches every bank about twice
//             instead of one 128-byte line per lane through L1
constexpr int SRC_NC = 0, SRC_CG = 1, SRC_SMEM = 2;

template <int SRC>
__device__ __forceinline__ float4 ldv(const float4* p) {
    if (SRC == SRC_CG) return __ldcg(p);
    if (SRC == SRC_SMEM) return *p;
    return __ldg(p);
}

// padded row length and column position of the shared-memory staging
__host__ __device__ __forceinline__ int vpad_ld(int n) { return n + n / 16; }
__device__ __forceinline__ int vpad(int c) { return c + 4 * (c >> 6); }

// the 16 or 32 consecutive values at column c of row r of a source
template <int SRC>
__device__ __forceinline__ const float* vrow(const float* base, int ld, int r, int c) {
    return base + (size_t)r * ld + (SRC == SRC_SMEM ? vpad(c) : c);
}

// stage rows [0, n) of a global [n][cols] matrix into shared memory, padded
__device__ __forceinline__ void vstage(float* dst, const float* __restrict__ src, int n, int cols) {
    const int ld = vpad_ld(cols), q = cols / 4;
    for (int i = threadIdx.x; i < n * q; i += blockDim.x) {
        const int r = i / q, c = 4 * (i - r * q);
        *reinterpret_cast<float4*>(dst + (size_t)r * ld + vpad(c)) =
            __ldcg(reinterpret_cast<const float4*>(src + (size_t)r * cols + c));
    }
}

// ---------------------------------------------------------------------------- FP8

// 16 E4M3 weights (one chunk) . 16 consecutive fp32 values
template <int SRC>
__device__ __forceinline__ float f8_dot(uint4 w, const float* __restrict__ v) {
    const float4* v4 = reinterpret_cast<const float4*>(v);
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 x = ldv<SRC>(v4 + i);
        const float2 lo = e4m3x2_f2(q[i] & 0xffffu), hi = e4m3x2_f2(q[i] >> 16);
        a0 = fmaf(lo.x, x.x, a0);
        a1 = fmaf(lo.y, x.y, a1);
        a0 = fmaf(hi.x, x.z, a0);
        a1 = fmaf(hi.y, x.w, a1);
    }
    return a0 + a1;
}

// act[p][f] = silu(g) * u for every pair of the item (NC = H / 256 chunks a
// lane); x: token rows of xld floats from the source SRC
template <int NC, int SRC>
__device__ __forceinline__ void f8_gateup_rows(const float* __restrict__ x, int xld, int H, int F,
                                               int K, const Fp8Experts& w, int e, int f, int hl,
                                               const int32_t* plist, int p0, int p1,
                                               float* __restrict__ act) {
    const size_t row = (size_t)e * F + f;
    const uint8_t* gr = w.gate + row * H + 16 * hl;
    const uint8_t* ur = w.up + row * H + 16 * hl;
    uint4 wg[NC], wu[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        wg[k] = ld_stream(gr + 256 * k);
        wu[k] = ld_stream(ur + 256 * k);
    }
    const size_t sb = ((size_t)e * (F >> 7) + (f >> 7)) * (H >> 7);
    float sg[NC], su[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        sg[k] = __ldg(w.gate_scale + sb + 2 * k + (hl >> 3));
        su[k] = __ldg(w.up_scale + sb + 2 * k + (hl >> 3));
    }
    for (int q = p0; q < p1; ++q) {
        const int p = plist[q];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            opaque(wg[k]);
            opaque(wu[k]);
        }
        float g = 0.f, v = 0.f;
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            const float* xc = vrow<SRC>(x, xld, p / K, 16 * hl + 256 * k);
            g = fmaf(sg[k], f8_dot<SRC>(wg[k], xc), g);
            v = fmaf(su[k], f8_dot<SRC>(wu[k], xc), v);
        }
        g = group_sum<16>(g);
        v = group_sum<16>(v);
        if (hl == 0) act[(size_t)p * F + f] = g / (1.f + expf(-g)) * v;
    }
}

// down rows h and h + 2 of a half-warp (NC = F / 256 chunks a lane)
template <int NC>
struct F8Down {
    uint4 w0[NC], w1[NC];
};

template <int NC>
__device__ __forceinline__ void f8_down_load(F8Down<NC>& d, const Fp8Experts& w, int e, int h, int H,
                                             int F, int hl) {
    const uint8_t* r0 = w.down + ((size_t)e * H + h) * F + 16 * hl;
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        d.w0[k] = ld_stream(r0 + 256 * k);
        d.w1[k] = ld_stream(r0 + 2 * (size_t)F + 256 * k);
    }
}

template <int NC, int SRC>
__device__ __forceinline__ void f8_down_rows(F8Down<NC>& d, const Fp8Experts& w, int e, int h, int H,
                                             int F, int hl, const int32_t* plist, int p0, int p1,
                                             const float* act, int ald, float* __restrict__ y) {
    // rows h and h + 2 lie in one 128-row block (items start at multiples of 4)
    const size_t sb = ((size_t)e * (H >> 7) + (h >> 7)) * (F >> 7);
    float s[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) s[k] = __ldg(w.down_scale + sb + 2 * k + (hl >> 3));
    for (int q = p0; q < p1; ++q) {
        const int p = plist[q];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            opaque(d.w0[k]);
            opaque(d.w1[k]);
        }
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            const float* ac = vrow<SRC>(act, ald, p, 16 * hl + 256 * k);
            a = fmaf(s[k], f8_dot<SRC>(d.w0[k], ac), a);
            b = fmaf(s[k], f8_dot<SRC>(d.w1[k], ac), b);
        }
        a = group_sum<16>(a);
        b = group_sum<16>(b);
        if (hl == 0) {
            y[(size_t)p * H + h] = a;
            y[(size_t)p * H + h + 2] = b;
        }
    }
}

// ---------------------------------------------------------------------------- NVFP4

// 32 E2M1 weights (one chunk: elements 0..15 with block scale sa, 16..31 with sb)
// . 32 consecutive fp32 values
template <int SRC>
__device__ __forceinline__ float nv_dot(uint4 w, const float* __restrict__ v, float sa, float sb) {
    const float4* v4 = reinterpret_cast<const float4*>(v);
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
    float hsum[2];
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint32_t word = q[2 * half + i];
#pragma unroll
            for (int by = 0; by < 4; by += 2) {
                const float4 x = ldv<SRC>(v4 + 4 * half + 2 * i + by / 2);
                const float2 p0 = e2m1x2_f2(word >> (8 * by)), p1 = e2m1x2_f2(word >> (8 * by + 8));
                a0 = fmaf(p0.x, x.x, a0);
                a1 = fmaf(p0.y, x.y, a1);
                a0 = fmaf(p1.x, x.z, a0);
                a1 = fmaf(p1.y, x.w, a1);
            }
        }
        hsum[half] = a0 + a1;
    }
    return fmaf(sa, hsum[0], sb * hsum[1]);
}

// two chunks (gate and up) against the same 32 values, each value loaded once
template <int SRC>
__device__ __forceinline__ void nv_dot2(uint4 wa, uint4 wb, const float* __restrict__ v, float2 sa,
                                        float2 sb, float& ra, float& rb) {
    const float4* v4 = reinterpret_cast<const float4*>(v);
    const uint32_t qa[4] = {wa.x, wa.y, wa.z, wa.w}, qb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        float a = 0.f, b = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int by = 0; by < 4; by += 2) {
                const float4 x = ldv<SRC>(v4 + 4 * half + 2 * i + by / 2);
                const uint32_t wa_ = qa[2 * half + i] >> (8 * by), wb_ = qb[2 * half + i] >> (8 * by);
                const float2 a0 = e2m1x2_f2(wa_), a1 = e2m1x2_f2(wa_ >> 8);
                const float2 b0 = e2m1x2_f2(wb_), b1 = e2m1x2_f2(wb_ >> 8);
                a = fmaf(a0.x, x.x, a);
                b = fmaf(b0.x, x.x, b);
                a = fmaf(a0.y, x.y, a);
                b = fmaf(b0.y, x.y, b);
                a = fmaf(a1.x, x.z, a);
                b = fmaf(b1.x, x.z, b);
                a = fmaf(a1.y, x.w, a);
                b = fmaf(b1.y, x.w, b);
            }
        }
        ra = fmaf(half ? sa.y : sa.x, a, ra);
        rb = fmaf(half ? sb.y : sb.x, b, rb);
    }
}

// the two E4M3 block scales of a chunk (bytes idx and idx + 1 of the row's scales)
__device__ __forceinline__ float2 nv_scales(const uint8_t* __restrict__ row_bs, int idx) {
    const uint32_t two = __ldg(reinterpret_cast<const unsigned short*>(row_bs + idx));
    return e4m3x2_f2(two);
}

// act[p][f] = silu(g) * u for every pair of the item (NC = H / 512 chunks a
// lane); x: token rows of xld floats from the source SRC
template <int NC, int SRC>
__device__ __forceinline__ void nv_gateup_rows(const float* __restrict__ x, int xld, int H, int F,
                                               int K, const NvExperts& w, int e, int f, int hl,
                                               const int32_t* plist, int p0, int p1,
                                               float* __restrict__ act) {
    const size_t row = (size_t)e * F + f;
    const uint8_t* gr = w.gate + row * (H / 2) + 16 * hl;
    const uint8_t* ur = w.up + row * (H / 2) + 16 * hl;
    uint4 wg[NC], wu[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        wg[k] = ld_stream(gr + 256 * k);
        wu[k] = ld_stream(ur + 256 * k);
    }
    const uint8_t* gbs = w.gate_bs + row * (H / 16);
    const uint8_t* ubs = w.up_bs + row * (H / 16);
    float2 sg[NC], su[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        sg[k] = nv_scales(gbs, 2 * (hl + 16 * k));
        su[k] = nv_scales(ubs, 2 * (hl + 16 * k));
    }
    const float gg = __ldg(w.gate_gs + e), ug = __ldg(w.up_gs + e);
    for (int pq = p0; pq < p1; ++pq) {
        const int p = plist[pq];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            opaque(wg[k]);
            opaque(wu[k]);
        }
        float g = 0.f, v = 0.f;
#pragma unroll
        for (int k = 0; k < NC; ++k)
            nv_dot2<SRC>(wg[k], wu[k], vrow<SRC>(x, xld, p / K, 32 * hl + 512 * k), sg[k], su[k], g, v);
        g = group_sum<16>(g) * gg;
        v = group_sum<16>(v) * ug;
        if (hl == 0) act[(size_t)p * F + f] = g / (1.f + expf(-g)) * v;
    }
}

// down row h of a quarter-warp (NC = F / 256 chunks a lane of 8)
template <int NC>
struct NvDown {
    uint4 w[NC];
};

template <int NC>
__device__ __forceinline__ void nv_down_load(NvDown<NC>& d, const NvExperts& w, int e, int h, int H,
                                             int F, int ql) {
    const uint8_t* r = w.down + ((size_t)e * H + h) * (F / 2) + 16 * ql;
#pragma unroll
    for (int k = 0; k < NC; ++k) d.w[k] = ld_stream(r + 128 * k);
}

template <int NC, int SRC>
__device__ __forceinline__ void nv_down_rows(NvDown<NC>& d, const NvExperts& w, int e, int h, int H,
                                             int F, int ql, const int32_t* plist, int p0, int p1,
                                             const float* act, int ald, float* __restrict__ y) {
    const uint8_t* dbs = w.down_bs + ((size_t)e * H + h) * (F / 16);
    float2 s[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) s[k] = nv_scales(dbs, 2 * (ql + 8 * k));
    const float dg = __ldg(w.down_gs + e);
    for (int pq = p0; pq < p1; ++pq) {
        const int p = plist[pq];
#pragma unroll
        for (int k = 0; k < NC; ++k) opaque(d.w[k]);
        float a = 0.f;
#pragma unroll
        for (int k = 0; k < NC; ++k)
            a += nv_dot<SRC>(d.w[k], vrow<SRC>(act, ald, p, 32 * ql + 256 * k), s[k].x, s[k].y);
        a = group_sum<8>(a) * dg;
        if (ql == 0) y[(size_t)p * H + h] = a;
    }
}

}  // namespace lowbit
}  // namespace qmoe
