// kquant.cuh -- register-level decoding of GGUF k-quant superblocks for the
// CUDA-core dequant-GEMV kernels (sm_103a).
//
// Block formats (public GGUF k-quant layout; sizes fixed by the aprender issue
// "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path", section "File facts"):
//   Q4_K, 144 B / 256 weights: [0..1] d fp16, [2..3] dmin fp16, [4..15] 6-bit
//     scales/mins of 8 sub-blocks of 32, [16..143] nibbles: 32-byte chunk c holds
//     sub-block 2c in its low nibbles and 2c+1 in its high nibbles.
//     w = d*s_j*q - dmin*m_j.
//   Q6_K, 210 B / 256 weights: [0..127] ql, [128..191] qh, [192..207] int8
//     scales (one per 16 weights), [208..209] d fp16.  w = d*sc*(q6 - 32).
//
// Conversion trick used throughout: a 4-bit or 6-bit code q placed in bits
// 16..21 of the word 0x3F000000 is the float 0.5 + q/256 exactly, built with one
// byte permute (PRMT) and no int->float conversion.  Dot products accumulate
// sum (0.5 + q/256) * x in fp32 and the constant part is removed once per
// sub-block with the precomputed sum of x:  sum q*x = 256*P - 128*X.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace qmoe {

constexpr int QK = 256;
constexpr int Q4K_BYTES = 144;
constexpr int Q6K_BYTES = 210;

__device__ __forceinline__ float half_bits(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)(b & 0xFFFFu)));
}

// byte k (compile-time) of m, as float 0.5 + byte/256 (byte < 128)
template <int K>
__device__ __forceinline__ float mag(uint32_t m) {
    return __uint_as_float(__byte_perm(m, 0x3F000000u, 0x7044 | (K << 8)));
}

// (acc0, acc1) += (a0, a1) * (b0, b1) as one packed fp32x2 FMA
__device__ __forceinline__ void fma2(float& acc0, float& acc1, float a0, float a1, float b0,
                                     float b1) {
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%0, %1};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Integer key with the order of the float comparison (-0 folded into +0); NaN
// gets an extreme key, so ranks taken on it stay a permutation whatever the
// input (routing top-k).
__device__ __forceinline__ int order_key(float v) {
    const int b = __float_as_int(v + 0.f);
    return b ^ ((b >> 31) & 0x7fffffff);
}

// Sum over four consecutive 32-bit words of (0.5 + nibble/256) * x for the low
// nibbles (PA) and the high nibbles (PB) of 16 bytes; xa/xb point at the 16 x
// values paired with the low / high nibbles.
__device__ __forceinline__ void q4_piece_dot(uint4 q, const float4* xa, const float4* xb,
                                             float& PA, float& PB) {
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0x0F0F0F0Fu;
        const uint32_t hi = (w[i] >> 4) & 0x0F0F0F0Fu;
        const float4 u = xa[i], v = xb[i];
        fma2(a0, a1, mag<0>(lo), mag<1>(lo), u.x, u.y);
        fma2(a0, a1, mag<2>(lo), mag<3>(lo), u.z, u.w);
        fma2(b0, b1, mag<0>(hi), mag<1>(hi), v.x, v.y);
        fma2(b0, b1, mag<2>(hi), mag<3>(hi), v.z, v.w);
    }
    PA = a0 + a1;
    PB = b0 + b1;
}

// 6-bit scale and min of Q4_K sub-blocks 2c and 2c+1 from header words
// h1 = scales[0..3], h2 = scales[4..7], h3 = scales[8..11].
__device__ __forceinline__ void q4_scales(uint32_t h1, uint32_t h2, uint32_t h3, int c,
                                          int& sA, int& mA, int& sB, int& mB) {
    const int sh = 16 * (c & 1);                  // byte 2(c&1) and 2(c&1)+1
    const uint32_t b1 = h1 >> sh, b2 = h2 >> sh, b3 = h3 >> sh;
    if (c < 2) {
        sA = b1 & 63;          mA = b2 & 63;
        sB = (b1 >> 8) & 63;   mB = (b2 >> 8) & 63;
    } else {
        sA = (b3 & 15) | (((b1 >> 6) & 3) << 4);
        mA = ((b3 >> 4) & 15) | (((b2 >> 6) & 3) << 4);
        sB = ((b3 >> 8) & 15) | (((b1 >> 14) & 3) << 4);
        mB = ((b3 >> 12) & 15) | (((b2 >> 14) & 3) << 4);
    }
}

// Contribution of one 16-byte nibble piece pc (0..7) of a Q4_K superblock whose
// header is hdr, given PA/PB from q4_piece_dot and the x sums XA/XB of the 16
// columns paired with the low / high nibbles.
__device__ __forceinline__ float q4_piece_finish(uint4 hdr, int pc, float PA, float PB, float XA,
                                                 float XB) {
    int sA, mA, sB, mB;
    q4_scales(hdr.y, hdr.z, hdr.w, pc >> 1, sA, mA, sB, mB);
    const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
    const float dA = d * (float)sA, dB = d * (float)sB;
    float r = (256.f * dA) * PA - fmaf(dmin, (float)mA, 128.f * dA) * XA;
    r = fmaf(256.f * dB, PB, r) - fmaf(dmin, (float)mB, 128.f * dB) * XB;
    return r;
}

// 8 bytes at a 2-byte-aligned address, read as aligned words: two when the
// address is 4-byte aligned, three (starting 2 bytes early) when it is not.
// Never touches a byte outside [p - 2, p + 10), and only [p, p + 8) when aligned.
__device__ __forceinline__ uint2 ld8_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3) * 8u;
    const uint32_t w0 = __ldg(b), w1 = __ldg(b + 1);
    const uint32_t w2 = sh ? __ldg(b + 2) : 0u;
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// One Q6_K task: half n (0/1), position run m (0..3) -> l in [8m, 8m+8), all
// four groups g: 32 weights.  a points at the 256 activation values of this
// superblock.  Returns sum_i w_i * a_i.
__device__ __forceinline__ float q6_task_dot(const uint8_t* sb, int n, int m, const float* a) {
    const uint2 qa = ld8_a2(sb + 64 * n + 8 * m);
    const uint2 qb = ld8_a2(sb + 64 * n + 32 + 8 * m);
    const uint2 qh = ld8_a2(sb + 128 + 32 * n + 8 * m);
    const uint2 scw = ld8_a2(sb + 192 + 8 * n);
    const float d = __half2float(__ldg(reinterpret_cast<const __half*>(sb + 208)));
    const int sb0 = (m >> 1) * 8;                 // bit offset of scale (m>>1) within scw
    float total = 0.f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        // scale 8n + (m>>1) + 2g: byte (m>>1) + 2g of the 8 loaded bytes
        const int bo = sb0 + 16 * g;
        const uint32_t sw = bo < 32 ? (scw.x >> bo) : (scw.y >> (bo - 32));
        const float sc = (float)(int8_t)(sw & 0xFF);
        float p0 = 0.f, p1 = 0.f, asum = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const uint32_t A = half ? qa.y : qa.x, B = half ? qb.y : qb.x;
            const uint32_t Hh = half ? qh.y : qh.x;
            uint32_t q6;
            if (g == 0) q6 = (A & 0x0F0F0F0Fu) | ((Hh << 4) & 0x30303030u);
            else if (g == 1) q6 = (B & 0x0F0F0F0Fu) | ((Hh << 2) & 0x30303030u);
            else if (g == 2) q6 = ((A >> 4) & 0x0F0F0F0Fu) | (Hh & 0x30303030u);
            else q6 = ((B >> 4) & 0x0F0F0F0Fu) | ((Hh >> 2) & 0x30303030u);
            const float4 x = *reinterpret_cast<const float4*>(a + 128 * n + 32 * g + 8 * m + 4 * half);
            fma2(p0, p1, mag<0>(q6), mag<1>(q6), x.x, x.y);
            fma2(p0, p1, mag<2>(q6), mag<3>(q6), x.z, x.w);
            asum += (x.x + x.y) + (x.z + x.w);
        }
        // sum (q6-32)*a = 256*P - 128*A - 32*A
        total = fmaf(d * sc, fmaf(256.f, p0 + p1, -160.f * asum), total);
    }
    return total;
}

}  // namespace qmoe
