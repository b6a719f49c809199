// moe_experts.cu -- expert dequant-GEMVs of the qwen3moe MoE FFN (decode path):
// gate/up with fused SwiGLU, down projection, weighted combine into the residual.
//
// aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path":
// "File facts" (expert e at base + e*stride inside the 3-D tensor, no
// repacking; down is Q6_K or Q4_K per layer) and "Gaps ... G3" (per-qtype
// expert GEMVs, fused_swiglu, weighted sum + residual add).  The expert id is
// read from device memory (the page's planned K3 pointer gather), so nothing
// waits on the host.
//
// Work is expert-centric: each used expert's rows are read once and applied to
// every token routed to it.  Superblock bytes are loaded 16 B per lane and
// decoded in registers (kquant.cuh); x / act are fp32, accumulation is fp32.
#include <math.h>

#include "kquant.cuh"
#include "pdl.cuh"
#include "qmoe_internal.h"

namespace qmoe {

size_t row_bytes(int qtype, int cols) {
    return (size_t)(cols / QK) * (qtype == 1 ? Q4K_BYTES : Q6K_BYTES);
}

__device__ __forceinline__ size_t drow_bytes(int qtype, int cols) {
    return (size_t)(cols / QK) * (qtype == 1 ? Q4K_BYTES : Q6K_BYTES);
}

namespace {

constexpr int ROWS_PER_CTA = 8;   // one output row per warp

// sum_{tasks} of one Q4_K row: lane task t = lane + 32 i -> superblock t>>3,
// nibble piece t&7 (16 bytes = 32 weights).
__device__ __forceinline__ float q4_row_dot(const uint8_t* __restrict__ row, int nsb,
                                            const float* __restrict__ x, int lane) {
    float acc = 0.f;
    for (int t = lane; t < 8 * nsb; t += 32) {
        const int s = t >> 3, pc = t & 7;
        const uint8_t* sb = row + (size_t)s * Q4K_BYTES;
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(sb));
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(sb + 16 + 16 * pc));
        const float* xa = x + QK * s + 64 * (pc >> 1) + 16 * (pc & 1);
        const float4* xa4 = reinterpret_cast<const float4*>(xa);
        const float4* xb4 = reinterpret_cast<const float4*>(xa + 32);
        float PA, PB;
        q4_piece_dot(q, xa4, xb4, PA, PB);
        float XA = 0.f, XB = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 u = xa4[i], v = xb4[i];
            XA += (u.x + u.y) + (u.z + u.w);
            XB += (v.x + v.y) + (v.z + v.w);
        }
        acc += q4_piece_finish(hdr, pc, PA, PB, XA, XB);
    }
    return warp_sum(acc);
}

// sum over one Q6_K row: lane task t -> superblock t>>3, half (t>>2)&1, run t&3.
__device__ __forceinline__ float q6_row_dot(const uint8_t* __restrict__ row, int nsb,
                                            const float* __restrict__ a, int lane) {
    float acc = 0.f;
    for (int t = lane; t < 8 * nsb; t += 32) {
        const int s = t >> 3, k = t & 7;
        acc += q6_task_dot(row + (size_t)s * Q6K_BYTES, k >> 2, k & 3, a + QK * s);
    }
    return warp_sum(acc);
}

__device__ __forceinline__ float row_dot(int qtype, const uint8_t* row, int nsb, const float* x,
                                         int lane) {
    return qtype == 1 ? q4_row_dot(row, nsb, x, lane) : q6_row_dot(row, nsb, x, lane);
}

// grid (ceil(F/8), max used experts); warp -> row f of expert used_expert[blockIdx.y]
__global__ void __launch_bounds__(256) gateup_kernel(
    const float* __restrict__ x, int H, int F, int K, const uint8_t* __restrict__ gate,
    int gate_t, const uint8_t* __restrict__ up, int up_t, const int32_t* __restrict__ n_used,
    const int32_t* __restrict__ used_expert, const int32_t* __restrict__ used_first,
    const int32_t* __restrict__ pair_list, float* __restrict__ act) {
    const int u = blockIdx.y;
    if (u >= *n_used) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int f = blockIdx.x * ROWS_PER_CTA + warp;
    if (f >= F) return;
    const int e = used_expert[u];
    const int nsb = H / QK;
    const size_t rbg = drow_bytes(gate_t, H), rbu = drow_bytes(up_t, H);
    const uint8_t* grow = gate + (size_t)e * F * rbg + (size_t)f * rbg;
    const uint8_t* urow = up + (size_t)e * F * rbu + (size_t)f * rbu;
    const int p0 = used_first[u], p1 = used_first[u + 1];
    for (int i = p0; i < p1; ++i) {
        const int p = pair_list[i];
        const float* xt = x + (size_t)(p / K) * H;
        const float g = row_dot(gate_t, grow, nsb, xt, lane);
        const float v = row_dot(up_t, urow, nsb, xt, lane);
        if (lane == 0) act[(size_t)p * F + f] = g / (1.f + expf(-g)) * v;
    }
}

// grid (ceil(H/8), max used experts); warp -> row h of expert used_expert[blockIdx.y]
__global__ void __launch_bounds__(256) down_kernel(
    const float* __restrict__ act, int H, int F, const uint8_t* __restrict__ down, int down_t,
    const int32_t* __restrict__ n_used, const int32_t* __restrict__ used_expert,
    const int32_t* __restrict__ used_first, const int32_t* __restrict__ pair_list,
    float* __restrict__ y) {
    const int u = blockIdx.y;
    if (u >= *n_used) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * ROWS_PER_CTA + warp;
    if (h >= H) return;
    const int e = used_expert[u];
    const int nsb = F / QK;
    const size_t rb = drow_bytes(down_t, F);
    const uint8_t* row = down + (size_t)e * H * rb + (size_t)h * rb;
    const int p0 = used_first[u], p1 = used_first[u + 1];
    for (int i = p0; i < p1; ++i) {
        const int p = pair_list[i];
        const float v = row_dot(down_t, row, nsb, act + (size_t)p * F, lane);
        if (lane == 0) y[(size_t)p * H + h] = v;
    }
}

// out[t][h] = res[t][h] + sum_j w[t][j] * y[t*K+j][h]  (slot order j = 0..K-1)
__global__ void combine_kernel(const float* __restrict__ y, const float* __restrict__ wts,
                               const float* res, int H, int K, float* out) {
    pdl_wait();                 // y of this call (launched as a programmatic dependent)
    const int t = blockIdx.y;
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    float acc = res[(size_t)t * H + h];
    for (int j = 0; j < K; ++j) acc = fmaf(wts[t * K + j], y[((size_t)t * K + j) * H + h], acc);
    out[(size_t)t * H + h] = acc;
}

}  // namespace

cudaError_t launch_gateup(const MoeShape& s, const float* x, const uint8_t* gate, int gate_t,
                          const uint8_t* up, int up_t, const Route& r, float* act,
                          cudaStream_t st) {
    const int max_used = s.T * s.K < s.E ? s.T * s.K : s.E;
    dim3 g((s.F + ROWS_PER_CTA - 1) / ROWS_PER_CTA, max_used);
    gateup_kernel<<<g, 32 * ROWS_PER_CTA, 0, st>>>(x, s.H, s.F, s.K, gate, gate_t, up, up_t,
                                                   r.n_used, r.used_expert, r.used_first,
                                                   r.pair_list, act);
    return cudaGetLastError();
}

cudaError_t launch_down(const MoeShape& s, const float* act, const uint8_t* down, int down_t,
                        const Route& r, float* y, cudaStream_t st) {
    const int max_used = s.T * s.K < s.E ? s.T * s.K : s.E;
    dim3 g((s.H + ROWS_PER_CTA - 1) / ROWS_PER_CTA, max_used);
    down_kernel<<<g, 32 * ROWS_PER_CTA, 0, st>>>(act, s.H, s.F, down, down_t, r.n_used,
                                                 r.used_expert, r.used_first, r.pair_list, y);
    return cudaGetLastError();
}

cudaError_t launch_combine(const MoeShape& s, const float* y, const Route& r, const float* res,
                           float* out, cudaStream_t st) {
    dim3 g((s.H + 255) / 256, s.T);
    return launch_pdl(combine_kernel, g, dim3(256), 0, st, y, r.wts, res, s.H, s.K, out);
}

}  // namespace qmoe
