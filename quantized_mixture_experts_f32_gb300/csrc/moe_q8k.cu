// moe_q8k.cu -- the qwen3moe MoE FFN with 8-bit (Q8_K) activations in every
// expert GEMV: the variant the aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has
// NO working CUDA path" runs on DP4A kernels ("Gaps ... G8") and whose accuracy
// its R1 receipt measures against FP32 activations.
//
// Q8_K (the GGUF 8-bit activation block; the page names it without defining
// it): 256 values, an fp32 scale d, int8 codes q and 16 sums of 16 codes.  The
// block's value of largest magnitude v (the first, on a tie) takes code -128:
// s = -128/v, q = min(127, rint(s*x)), d = 1/s, each an IEEE fp32 operation;
// an all-zero block has d = 0.
//
//   q8k_quantize   x of every token -> Q8_K (one warp per 256 values)
//   q8k_gateup     per (used expert, gate/up row f): integer dots (dp4a) of the
//                  Q4_K (or Q6_K) rows with the token's codes, silu(g)*u -> act
//   q8k_quantize   act of every pair -> Q8_K
//   q8k_down       per (used expert, down row h): the same against the pair's
//                  codes -> y
//   combine        (moe_experts.cu) out = res + sum_j w_j y_j, slot order
// Q4_K rows: per 32-value sub-block j, d*s_j*sum(q4*q8) - dmin*m_j*sum(q8), the
// second sum from the two 16-code group sums; Q6_K rows: per 16-value group,
// d*sc*sum((q6-32)*q8); each superblock's part times the activation block's d.
// Integer sums are exact (int32); the scaling and the row sum are fp32.
#include <math.h>

#include "kquant.cuh"
#include "qmoe_internal.h"

namespace qmoe {

namespace {

constexpr int Q8_ROWS_PER_CTA = 8;   // one output row per warp

__device__ __forceinline__ size_t q8_row_bytes(int qtype, int cols) {
    return (size_t)(cols / QK) * (qtype == 1 ? Q4K_BYTES : Q6K_BYTES);
}

// Row blockIdx.y of x (n values, n % 256 == 0), 256-value block blockIdx.x: lane
// l quantises values 8l..8l+7.
__global__ void __launch_bounds__(32) q8k_quantize(const float* __restrict__ x, int n,
                                                   float* __restrict__ d, int8_t* __restrict__ q,
                                                   int16_t* __restrict__ bs) {
    const int lane = threadIdx.x;
    const size_t base = (size_t)blockIdx.y * n + (size_t)blockIdx.x * QK + 8 * lane;
    const float4 a = *reinterpret_cast<const float4*>(x + base);
    const float4 b = *reinterpret_cast<const float4*>(x + base + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float amax = 0.f, vmax = 0.f;
    int imax = 8 * lane;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (fabsf(v[i]) > amax) {
            amax = fabsf(v[i]);
            vmax = v[i];
            imax = 8 * lane + i;
        }
    // the block's largest magnitude, the lowest index on a tie: a total order,
    // so every lane ends with the same winner
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oa = __shfl_xor_sync(0xffffffffu, amax, o);
        const float ov = __shfl_xor_sync(0xffffffffu, vmax, o);
        const int oi = __shfl_xor_sync(0xffffffffu, imax, o);
        if (oa > amax || (oa == amax && oi < imax)) {
            amax = oa;
            vmax = ov;
            imax = oi;
        }
    }
    int c[8];
    float dd = 0.f;
    if (amax == 0.f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = 0;
    } else {
        const float s = __fdiv_rn(-128.f, vmax);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = min(__float2int_rn(__fmul_rn(s, v[i])), 127);
        dd = __fdiv_rn(1.f, s);
    }
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        w0 |= ((uint32_t)c[i] & 0xFFu) << (8 * i);
        w1 |= ((uint32_t)c[i + 4] & 0xFFu) << (8 * i);
    }
    *reinterpret_cast<uint2*>(q + base) = make_uint2(w0, w1);
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += c[i];
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    if ((lane & 1) == 0)
        bs[(size_t)blockIdx.y * (n / 16) + (size_t)blockIdx.x * 16 + (lane >> 1)] = (int16_t)sum;
    if (lane == 0) d[(size_t)blockIdx.y * (n / QK) + blockIdx.x] = dd;
}

// One Q4_K row (nsb superblocks) against Q8_K codes; lane task t -> superblock
// t >> 3, sub-block t & 7 (32 values: 8 dp4a).
__device__ __forceinline__ float q4_q8_row(const uint8_t* __restrict__ row, int nsb,
                                           const float* __restrict__ d8, const int8_t* __restrict__ q8,
                                           const int16_t* __restrict__ bs8, int lane) {
    float acc = 0.f;
    for (int t = lane; t < 8 * nsb; t += 32) {
        const int sb = t >> 3, j = t & 7;
        const uint8_t* blk = row + (size_t)sb * Q4K_BYTES;
        const uint4 hdr = __ldg(reinterpret_cast<const uint4*>(blk));
        const uint4* np = reinterpret_cast<const uint4*>(blk + 16 + 32 * (j >> 1));
        const uint4 n0 = __ldg(np), n1 = __ldg(np + 1);
        const int4* cp = reinterpret_cast<const int4*>(q8 + (size_t)sb * QK + 32 * j);
        const int4 c0 = cp[0], c1 = cp[1];
        const uint32_t nw[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
        const int cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const int sh = 4 * (j & 1);
        int S = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) S = __dp4a((int)((nw[w] >> sh) & 0x0F0F0F0Fu), cw[w], S);
        const int B = (int)bs8[sb * 16 + 2 * j] + (int)bs8[sb * 16 + 2 * j + 1];
        int sA, mA, sB, mB;
        q4_scales(hdr.y, hdr.z, hdr.w, j >> 1, sA, mA, sB, mB);
        const int sj = (j & 1) ? sB : sA, mj = (j & 1) ? mB : mA;
        const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
        acc += d8[sb] * (d * (float)sj * (float)S - dmin * (float)mj * (float)B);
    }
    return warp_sum(acc);
}

// One Q6_K row against Q8_K codes; lane task t -> superblock t >> 4, 16-value
// group g = t & 15 (half n = g >> 3, 32-group gg = (g & 7) >> 1, positions
// 16 (g & 1) .. + 15; one int8 scale; 4 dp4a).
__device__ __forceinline__ float q6_q8_row(const uint8_t* __restrict__ row, int nsb,
                                           const float* __restrict__ d8, const int8_t* __restrict__ q8,
                                           int lane) {
    float acc = 0.f;
    for (int t = lane; t < 16 * nsb; t += 32) {
        const int sb = t >> 4, g = t & 15;
        const int n = g >> 3, gg = (g & 7) >> 1, hf = g & 1;
        const uint8_t* blk = row + (size_t)sb * Q6K_BYTES;
        const uint8_t* lp = blk + 64 * n + 32 * (gg & 1) + 16 * hf;
        const uint8_t* hp = blk + 128 + 32 * n + 16 * hf;
        const uint2 l0 = ld8_a2(lp), l1 = ld8_a2(lp + 8);
        const uint2 h0 = ld8_a2(hp), h1 = ld8_a2(hp + 8);
        const uint32_t lw[4] = {l0.x, l0.y, l1.x, l1.y}, hw[4] = {h0.x, h0.y, h1.x, h1.y};
        const int4 cv = *reinterpret_cast<const int4*>(q8 + (size_t)sb * QK + 16 * g);
        const int cw[4] = {cv.x, cv.y, cv.z, cv.w};
        const int shl = 4 * (gg >> 1), shh = 2 * gg;
        int S = 0;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const uint32_t code = ((lw[w] >> shl) & 0x0F0F0F0Fu) | (((hw[w] >> shh) & 0x03030303u) << 4);
            S = __dp4a((int)__vsub4(code, 0x20202020u), cw[w], S);   // q6 - 32 per byte
        }
        const int sc = (int)static_cast<int8_t>(__ldg(blk + 192 + 8 * n + hf + 2 * gg));
        const float d = __half2float(__ldg(reinterpret_cast<const __half*>(blk + 208)));
        acc += d8[sb] * (d * (float)sc * (float)S);
    }
    return warp_sum(acc);
}

__device__ __forceinline__ float q8_row_dot(int qtype, const uint8_t* row, int nsb, const float* d8,
                                            const int8_t* q8, const int16_t* bs8, int lane) {
    return qtype == 1 ? q4_q8_row(row, nsb, d8, q8, bs8, lane) : q6_q8_row(row, nsb, d8, q8, lane);
}

// grid (ceil(F/8), max used experts); warp -> row f of expert used_expert[blockIdx.y]
__global__ void __launch_bounds__(256) q8k_gateup(
    const Q8Bufs b, int H, int F, int K, const uint8_t* __restrict__ gate, int gate_t,
    const uint8_t* __restrict__ up, int up_t, const int32_t* __restrict__ n_used,
    const int32_t* __restrict__ used_expert, const int32_t* __restrict__ used_first,
    const int32_t* __restrict__ pair_list, float* __restrict__ act) {
    const int u = blockIdx.y;
    if (u >= *n_used) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int f = blockIdx.x * Q8_ROWS_PER_CTA + warp;
    if (f >= F) return;
    const int e = used_expert[u];
    const int nsb = H / QK;
    const size_t rbg = q8_row_bytes(gate_t, H), rbu = q8_row_bytes(up_t, H);
    const uint8_t* grow = gate + (size_t)e * F * rbg + (size_t)f * rbg;
    const uint8_t* urow = up + (size_t)e * F * rbu + (size_t)f * rbu;
    const int p0 = used_first[u], p1 = used_first[u + 1];
    for (int i = p0; i < p1; ++i) {
        const int p = pair_list[i], t = p / K;
        const float* d8 = b.dx + (size_t)t * nsb;
        const int8_t* q8 = b.qx + (size_t)t * H;
        const int16_t* bs8 = b.bx + (size_t)t * (H / 16);
        const float g = q8_row_dot(gate_t, grow, nsb, d8, q8, bs8, lane);
        const float v = q8_row_dot(up_t, urow, nsb, d8, q8, bs8, lane);
        if (lane == 0) act[(size_t)p * F + f] = g / (1.f + expf(-g)) * v;
    }
}

// grid (ceil(H/8), max used experts); warp -> row h of expert used_expert[blockIdx.y]
__global__ void __launch_bounds__(256) q8k_down(
    const Q8Bufs b, int H, int F, const uint8_t* __restrict__ down, int down_t,
    const int32_t* __restrict__ n_used, const int32_t* __restrict__ used_expert,
    const int32_t* __restrict__ used_first, const int32_t* __restrict__ pair_list,
    float* __restrict__ y) {
    const int u = blockIdx.y;
    if (u >= *n_used) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x * Q8_ROWS_PER_CTA + warp;
    if (h >= H) return;
    const int e = used_expert[u];
    const int nsb = F / QK;
    const size_t rb = q8_row_bytes(down_t, F);
    const uint8_t* row = down + (size_t)e * H * rb + (size_t)h * rb;
    const int p0 = used_first[u], p1 = used_first[u + 1];
    for (int i = p0; i < p1; ++i) {
        const int p = pair_list[i];
        const float v = q8_row_dot(down_t, row, nsb, b.da + (size_t)p * nsb, b.qa + (size_t)p * F,
                                   b.ba + (size_t)p * (F / 16), lane);
        if (lane == 0) y[(size_t)p * H + h] = v;
    }
}

}  // namespace

size_t q8_bufs_bytes(int T, int H, int K, int F) {
    const size_t P = (size_t)T * K;
    auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
    return al((size_t)T * H) + al(sizeof(float) * (size_t)T * H / QK) + al(sizeof(int16_t) * (size_t)T * H / 16) +
           al(P * F) + al(sizeof(float) * P * F / QK) + al(sizeof(int16_t) * P * F / 16);
}

Q8Bufs q8_bufs_carve(unsigned char* base, int T, int H, int K, int F) {
    const size_t P = (size_t)T * K;
    auto al = [](size_t v) { return (v + 255) & ~size_t(255); };
    Q8Bufs b;
    size_t off = 0;
    b.qx = reinterpret_cast<int8_t*>(base + off);
    off += al((size_t)T * H);
    b.dx = reinterpret_cast<float*>(base + off);
    off += al(sizeof(float) * (size_t)T * H / QK);
    b.bx = reinterpret_cast<int16_t*>(base + off);
    off += al(sizeof(int16_t) * (size_t)T * H / 16);
    b.qa = reinterpret_cast<int8_t*>(base + off);
    off += al(P * F);
    b.da = reinterpret_cast<float*>(base + off);
    off += al(sizeof(float) * P * F / QK);
    b.ba = reinterpret_cast<int16_t*>(base + off);
    return b;
}

cudaError_t launch_moe_q8k(const MoeShape& s, const float* x, const float* res, const uint8_t* gate,
                           int gate_t, const uint8_t* up, int up_t, const uint8_t* down, int down_t,
                           const Route& r, const Q8Bufs& b, float* act, float* y, float* out,
                           cudaStream_t st) {
    const int P = s.T * s.K;
    const int max_used = P < s.E ? P : s.E;
    q8k_quantize<<<dim3(s.H / QK, s.T), 32, 0, st>>>(x, s.H, b.dx, b.qx, b.bx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    q8k_gateup<<<dim3((s.F + Q8_ROWS_PER_CTA - 1) / Q8_ROWS_PER_CTA, max_used), 32 * Q8_ROWS_PER_CTA, 0, st>>>(
        b, s.H, s.F, s.K, gate, gate_t, up, up_t, r.n_used, r.used_expert, r.used_first, r.pair_list, act);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    q8k_quantize<<<dim3(s.F / QK, P), 32, 0, st>>>(act, s.F, b.da, b.qa, b.ba);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    q8k_down<<<dim3((s.H + Q8_ROWS_PER_CTA - 1) / Q8_ROWS_PER_CTA, max_used), 32 * Q8_ROWS_PER_CTA, 0, st>>>(
        b, s.H, s.F, down, down_t, r.n_used, r.used_expert, r.used_first, r.pair_list, y);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_combine(s, y, r, res, out, st);
}

}  // namespace qmoe
