// prefill_umma.cu -- the MoE FFN for many tokens (prefill) as grouped GEMMs on
// the 5th-generation tensor cores (tcgen05), weights dequantised on the fly.
//
// The aprender issue "qwen3moe (Qwen3-30B-A3B, ...) has NO working CUDA path"
// (later gap list: prefill is token-by-token, 1,685 tokens in 21.9 s; the fix it
// names is a batched prefill with expert grouping, gather, a per-expert GEMM
// and a weighted scatter-add).  Here, after the device routing of moe_route.cu
// (pairs sorted by expert):
//   gather_x_f16    x rows of every (token, slot) pair, in expert order, as fp16
//   prefill_gateup  per (expert, 64-f tile, token tile): A = 64 gate rows + 64 up
//                   rows of Q4_K superblocks, TMA-loaded raw (3 stages) and
//                   converted to fp16 in shared memory (128B-swizzled K-major)
//                   by 16 dequant warps, a quarter of them per k-block of each
//                   superblock; B = the expert's gathered x rows via TMA; fp32
//                   accumulator in TMEM; epilogue silu(g)*u -> fp16 act rows
//   prefill_down    per (expert, 128-row tile, token tile): A = 128 down rows
//                   (Q6_K or Q4_K, one bulk copy of the whole K), B = act rows,
//                   epilogue -> fp32 y rows per pair
//   combine_pairs   out[t] = res[t] + sum_j w[t][j] y[pos(t, j)] in slot order
// Weights are on the MMA's M side ("swap-AB"): expert segments are short (32
// tokens on average), so token tiles of 16..256 are the N side.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "kquant.cuh"
#include "qmoe_internal.h"
#include "umma.cuh"

namespace qmoe {

namespace {

constexpr int KBLK = 64;                       // k per tensor-core block (128 B of fp16)
constexpr int TILE_M = 128;
constexpr int TILE_NMAX = 256;
constexpr int A_STAGE = TILE_M * KBLK * 2;     // 16 KB fp16 A block
constexpr int NDQ = 16;                        // dequant / epilogue warps (4 threads per A row)
constexpr int W_QLOAD = NDQ;                   // weight copies
constexpr int W_BLOAD = NDQ + 1;               // activation (B) tiles
constexpr int W_MMA = NDQ + 2;                 // tcgen05.mma issue
constexpr int PF_THREADS = (NDQ + 3) * 32;
constexpr uint32_t TMEM_COLS = 256;
constexpr int NA = 4;                          // A (fp16 weight) stages of the down GEMM: one per
static_assert(NA * KBLK == QK, "k-block of a superblock");
constexpr int NQ = 3;                          // raw Q4_K stages of the gate/up kernel
constexpr int QSTAGE_GU = 2 * 64 * Q4K_BYTES;  // 64 gate + 64 up rows of one superblock column
constexpr int NBMAX = 8;                       // B stages, at most
constexpr int B_BYTES_GU = 96 * 1024;
constexpr int B_BYTES_DN = 64 * 1024;

struct PfBars {
    uint64_t qfull[NQ], qempty[NQ], afull[NA], aempty[NA], bfull[NBMAX], bempty[NBMAX], acc;
    uint32_t tmem;
};

// B stages that fit the region for a token tile of nb rows
__host__ __device__ inline int b_stages(int b_bytes, int nb) {
    const int n = b_bytes / (nb * KBLK * 2);
    return n < NBMAX ? n : NBMAX;
}

// token-tile height and the matching B tensor map (64 / 128 / 256 rows)
__device__ __forceinline__ int box_rows(int n) { return n <= 64 ? 64 : n <= 128 ? 128 : 256; }

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t b) { return *reinterpret_cast<__half2*>(&b); }

// 8 code bytes (4 per word, each < 1024, k order) -> 8 fp16 weights
// (code - sub) * s + c in packed half2 arithmetic: a byte permute puts two codes
// into the mantissas of the halves 1024 + code, the subtraction of sub (1024,
// or 1024 + 32 for Q6_K) is exact, one HFMA2 applies scale and offset.
__device__ __forceinline__ uint4 codes_to_half8(uint32_t w0, uint32_t w1, __half2 sub, __half2 s,
                                                __half2 c) {
    uint4 r;
    r.x = h2_bits(__hfma2(__hsub2(bits_h2(__byte_perm(w0, 0x64646464u, 0x4140)), sub), s, c));
    r.y = h2_bits(__hfma2(__hsub2(bits_h2(__byte_perm(w0, 0x64646464u, 0x4342)), sub), s, c));
    r.z = h2_bits(__hfma2(__hsub2(bits_h2(__byte_perm(w1, 0x64646464u, 0x4140)), sub), s, c));
    r.w = h2_bits(__hfma2(__hsub2(bits_h2(__byte_perm(w1, 0x64646464u, 0x4342)), sub), s, c));
    return r;
}

// one thread: k-block c (64 k) of one A row from a Q4_K superblock at q: the
// 32-byte chunk c holds sub-block 2c in its low nibbles (k 0..31) and 2c+1 in
// its high nibbles (k 32..63) -> fp16 SW128 tile
__device__ __forceinline__ void dq_q4k_k64_regs(uint4 hdr, uint4 v0, uint4 v1, int c,
                                                uint8_t* atile, int row);

__device__ __forceinline__ void dq_q4k_k64(const uint8_t* q, int c, uint8_t* atile, int row) {
    const uint4* src = reinterpret_cast<const uint4*>(q + 16 + 32 * c);
    dq_q4k_k64_regs(*reinterpret_cast<const uint4*>(q), src[0], src[1], c, atile, row);
}

// the same from registers: header hdr, chunk c as v0 (bytes 0..15), v1 (16..31)
__device__ __forceinline__ void dq_q4k_k64_regs(uint4 hdr, uint4 v0, uint4 v1, int c,
                                                uint8_t* atile, int row) {
    int sA, mA, sB, mB;
    q4_scales(hdr.y, hdr.z, hdr.w, c, sA, mA, sB, mB);
    const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
    // w = d*s*q - dmin*m
    const __half2 sub = __float2half2_rn(1024.f);
    const __half2 sA2 = __float2half2_rn(d * (float)sA), cA2 = __float2half2_rn(-dmin * (float)mA);
    const __half2 sB2 = __float2half2_rn(d * (float)sB), cB2 = __float2half2_rn(-dmin * (float)mB);
    uint8_t* rb = atile + row * 128;
    const int sw = row & 7;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint4 v = half ? v1 : v0;
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const uint32_t a0 = w[2 * cc], a1 = w[2 * cc + 1];
            const int k8 = 2 * half + cc;                   // 8-k group of the low nibbles
            *reinterpret_cast<uint4*>(rb + ((k8 ^ sw) << 4)) =
                codes_to_half8(a0 & 0x0F0F0F0Fu, a1 & 0x0F0F0F0Fu, sub, sA2, cA2);
            *reinterpret_cast<uint4*>(rb + (((k8 + 4) ^ sw) << 4)) =
                codes_to_half8((a0 >> 4) & 0x0F0F0F0Fu, (a1 >> 4) & 0x0F0F0F0Fu, sub, sB2, cB2);
        }
    }
}

// 8 bytes at an even shared-memory address
__device__ __forceinline__ uint2 lds8(const uint8_t* p) {
    const uint32_t off = smem_u32(p) & 3u;
    const uint32_t* b = reinterpret_cast<const uint32_t*>(p - off);   // stays a shared pointer
    const uint32_t sh = off * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2];
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// one thread: k-block qb (64 k) of one A row from a Q6_K superblock at blk
// (2-byte aligned): groups g = 2(qb&1) and 2(qb&1)+1 of half n = qb>>1,
// positions l = 0..31 each
__device__ __forceinline__ void dq_q6k_k64(const uint8_t* blk, int qb, uint8_t* atile, int row) {
    const int n = qb >> 1;
    const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
    const uint8_t* qhp = blk + 128 + 32 * n;
    const __half2 sub = __float2half2_rn(1056.f), zero = __float2half2_rn(0.f);
    uint8_t* rb = atile + row * 128;
    const int sw = row & 7;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int g = 2 * (qb & 1) + h;
        const uint8_t* qlp = blk + 64 * n + 32 * (g & 1);
        const __half2 ds0 = __float2half2_rn(d * (float)static_cast<int8_t>(blk[192 + 8 * n + 2 * g]));
        const __half2 ds1 = __float2half2_rn(d * (float)static_cast<int8_t>(blk[192 + 8 * n + 2 * g + 1]));
        const int shl = 4 * (g >> 1), shh = 2 * g;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {                     // 8 positions each
            const uint2 ql = lds8(qlp + 8 * cc), qh = lds8(qhp + 8 * cc);
            const uint32_t c0 = ((ql.x >> shl) & 0x0F0F0F0Fu) | (((qh.x >> shh) & 0x03030303u) << 4);
            const uint32_t c1 = ((ql.y >> shl) & 0x0F0F0F0Fu) | (((qh.y >> shh) & 0x03030303u) << 4);
            // w = d*sc*(q6 - 32)
            *reinterpret_cast<uint4*>(rb + (((4 * h + cc) ^ sw) << 4)) =
                codes_to_half8(c0, c1, sub, cc < 2 ? ds0 : ds1, zero);
        }
    }
}

struct GuParams {
    const int32_t* n_used;
    const int32_t* used_expert;
    const int32_t* used_first;
    __half* act;          // [P][F] fp16, rows in pair-list order
    int H, F, ntiles;     // ntiles: token tiles per expert slot in grid.y
};

// grid (F/64, max_used * ntiles), PF_THREADS threads
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_gateup(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                   const __grid_constant__ CUtensorMap tm_x64, const __grid_constant__ CUtensorMap tm_x128,
                   const __grid_constant__ CUtensorMap tm_x256, const GuParams p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    // 1024-aligned base, kept a shared-space pointer (an integer round trip
    // would turn every access into a generic one)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const int u = blockIdx.y / p.ntiles, nt = blockIdx.y % p.ntiles;
    if (u >= *p.n_used) return;
    const int first = p.used_first[u], cnt = p.used_first[u + 1] - first;
    const int n0 = nt * TILE_NMAX;
    if (n0 >= cnt) return;
    const int n = min(TILE_NMAX, cnt - n0);
    const int N = (n + 15) & ~15;
    const int nb = box_rows(n);
    const CUtensorMap* tmx = nb == 64 ? &tm_x64 : nb == 128 ? &tm_x128 : &tm_x256;
    const int e = p.used_expert[u];
    const int f0 = blockIdx.x * 64;
    const int H = p.H, F = p.F;
    const int NKB = H / KBLK, NSB = H / QK;

    uint8_t* qst = sm;                                   // NQ x QSTAGE_GU
    uint8_t* ast = sm + ((NQ * QSTAGE_GU + 1023) & ~1023);  // NA x A_STAGE (1024-aligned)
    uint8_t* bst = ast + NA * A_STAGE;                   // B_BYTES_GU
    PfBars* bars = reinterpret_cast<PfBars*>(bst + B_BYTES_GU);
    const int NB = b_stages(B_BYTES_GU, nb);
    const int BSTAGE = nb * KBLK * 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < NQ; ++i) {
            mbar_init(&bars->qfull[i], 1);
            mbar_init(&bars->qempty[i], NDQ);
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(&bars->afull[i], NDQ / NA);
            mbar_init(&bars->aempty[i], 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&bars->bfull[i], 1);
            mbar_init(&bars->bempty[i], 1);
        }
        mbar_init(&bars->acc, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&bars->tmem, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem;

    if (warp == W_QLOAD) {
        // raw gate/up superblock columns, NQ ahead of the dequant warps
        if (lane == 0) {
            const int ybase = e * F + f0;
            for (int sb = 0; sb < NSB; ++sb) {
                const int st = sb % NQ;
                if (!mbar_wait(&bars->qempty[st], ((uint32_t)(sb / NQ) & 1u) ^ 1u)) break;
                uint8_t* dst = qst + st * QSTAGE_GU;
                mbar_arrive_expect_tx(&bars->qfull[st], QSTAGE_GU);
                tma_load_2d(dst, &tm_gate, sb * Q4K_BYTES, ybase, &bars->qfull[st]);
                tma_load_2d(dst + 64 * Q4K_BYTES, &tm_up, sb * Q4K_BYTES, ybase, &bars->qfull[st]);
            }
        }
    } else if (warp == W_BLOAD) {
        // the expert's gathered x rows, NB k-blocks ahead of the MMA
        if (lane == 0) {
            for (int kb = 0; kb < NKB; ++kb) {
                const int st = kb % NB;
                if (!mbar_wait(&bars->bempty[st], ((uint32_t)(kb / NB) & 1u) ^ 1u)) break;
                mbar_arrive_expect_tx(&bars->bfull[st], (uint32_t)BSTAGE);
                tma_load_2d(bst + st * BSTAGE, tmx, kb * KBLK, first + n0, &bars->bfull[st]);
            }
        }
    } else if (warp == W_MMA) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16(TILE_M, N);
            for (int kb = 0; kb < NKB; ++kb) {
                const int sa = kb % NA, sb = kb % NB;
                if (!mbar_wait(&bars->afull[sa], (uint32_t)(kb / NA) & 1u) ||
                    !mbar_wait(&bars->bfull[sb], (uint32_t)(kb / NB) & 1u))
                    break;
                tc_fence_after();
                const uint64_t ad = umma_sdesc(smem_u32(ast + sa * A_STAGE));
                const uint64_t bd = umma_sdesc(smem_u32(bst + sb * BSTAGE));
#pragma unroll
                for (int k = 0; k < KBLK / 16; ++k)
                    umma_f16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                             (kb | k) != 0);
                umma_commit(&bars->aempty[sa]);
                umma_commit(&bars->bempty[sb]);
            }
            umma_commit(&bars->acc);
        }
    } else {
        // dequant: thread -> A row (tid & 127) and k-block c = tid >> 7 of every
        // superblock (A stage c): 64 weights per visit, one scale decode
        const int row = tid & 127, c = tid >> 7;
        const int grp = row >> 5, w32 = row & 31;
        const int src = w32 < 16 ? 16 * grp + w32 : 64 + 16 * grp + (w32 - 16);
        for (int sb = 0; sb < NSB; ++sb) {
            const int sq = sb % NQ;
            mbar_wait(&bars->qfull[sq], (uint32_t)(sb / NQ) & 1u);
            mbar_wait(&bars->aempty[c], ((uint32_t)sb & 1u) ^ 1u);
            dq_q4k_k64(qst + sq * QSTAGE_GU + src * Q4K_BYTES, c, ast + c * A_STAGE, row);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars->afull[c]);
                mbar_arrive(&bars->qempty[sq]);
            }
        }
        // epilogue: TMEM lane quarter (warp % 4); column quarter (warp / 4)
        mbar_wait(&bars->acc, 0);
        tc_fence_after();
        const int lq = warp & 3, ch = warp >> 2;
        const int f = f0 + 16 * lq + (lane & 15);
        for (int c0 = ch * 64; c0 < min(N, ch * 64 + 64); c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * lq) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float up = __shfl_down_sync(0xffffffffu, v[j], 16);
                const int col = c0 + j;
                if (lane < 16 && col < n) {
                    const float g = v[j];
                    p.act[(size_t)(first + n0 + col) * F + f] = __float2half_rn(g / (1.f + expf(-g)) * up);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

struct DnParams {
    const int32_t* n_used;
    const int32_t* used_expert;
    const int32_t* used_first;
    const uint8_t* down;
    float* y;             // [P][H] fp32, rows in pair-list order
    int H, F, ntiles, down_t;
};

// grid (H/128, max_used * ntiles)
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_down(const __grid_constant__ CUtensorMap tm_a64, const __grid_constant__ CUtensorMap tm_a128,
                 const __grid_constant__ CUtensorMap tm_a256, const DnParams p) {
    extern __shared__ __align__(1024) uint8_t smraw[];
    // 1024-aligned base, kept a shared-space pointer (an integer round trip
    // would turn every access into a generic one)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const int u = blockIdx.y / p.ntiles, nt = blockIdx.y % p.ntiles;
    if (u >= *p.n_used) return;
    const int first = p.used_first[u], cnt = p.used_first[u + 1] - first;
    const int n0 = nt * TILE_NMAX;
    if (n0 >= cnt) return;
    const int n = min(TILE_NMAX, cnt - n0);
    const int N = (n + 15) & ~15;
    const int nb = box_rows(n);
    const CUtensorMap* tmb = nb == 64 ? &tm_a64 : nb == 128 ? &tm_a128 : &tm_a256;
    const int e = p.used_expert[u];
    const int h0 = blockIdx.x * TILE_M;
    const int H = p.H, F = p.F;
    const int NKB = F / KBLK;
    const int BB = p.down_t == 1 ? Q4K_BYTES : Q6K_BYTES;
    const int RB = (F / QK) * BB;
    const uint32_t qbytes = (uint32_t)(TILE_M * RB);       // whole K of 128 rows

    uint8_t* ast = sm;                                    // NA x A_STAGE
    uint8_t* bst = ast + NA * A_STAGE;                    // B_BYTES_DN
    uint8_t* qbuf = bst + B_BYTES_DN;                     // qbytes (+ slack)
    PfBars* bars = reinterpret_cast<PfBars*>(qbuf + ((qbytes + 1023) & ~1023u) + 1024);
    const int NB = b_stages(B_BYTES_DN, nb);
    const int BSTAGE = nb * KBLK * 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&bars->qfull[0], 1);
        for (int i = 0; i < NA; ++i) {
            mbar_init(&bars->afull[i], NDQ / NA);
            mbar_init(&bars->aempty[i], 1);
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(&bars->bfull[i], 1);
            mbar_init(&bars->bempty[i], 1);
        }
        mbar_init(&bars->acc, 1);
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&bars->tmem, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem;

    if (warp == W_QLOAD) {
        // the whole K of this CTA's 128 down rows: one bulk copy
        if (lane == 0) {
            const uint8_t* src = p.down + (size_t)e * H * RB + (size_t)h0 * RB;
            mbar_arrive_expect_tx(&bars->qfull[0], qbytes);
            bulk_g2s(qbuf, src, qbytes, &bars->qfull[0]);
        }
    } else if (warp == W_BLOAD) {
        if (lane == 0) {
            for (int kb = 0; kb < NKB; ++kb) {
                const int st = kb % NB;
                if (!mbar_wait(&bars->bempty[st], ((uint32_t)(kb / NB) & 1u) ^ 1u)) break;
                mbar_arrive_expect_tx(&bars->bfull[st], (uint32_t)BSTAGE);
                tma_load_2d(bst + st * BSTAGE, tmb, kb * KBLK, first + n0, &bars->bfull[st]);
            }
        }
    } else if (warp == W_MMA) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16(TILE_M, N);
            for (int kb = 0; kb < NKB; ++kb) {
                const int sa = kb % NA, sb = kb % NB;
                if (!mbar_wait(&bars->afull[sa], (uint32_t)(kb / NA) & 1u) ||
                    !mbar_wait(&bars->bfull[sb], (uint32_t)(kb / NB) & 1u))
                    break;
                tc_fence_after();
                const uint64_t ad = umma_sdesc(smem_u32(ast + sa * A_STAGE));
                const uint64_t bd = umma_sdesc(smem_u32(bst + sb * BSTAGE));
#pragma unroll
                for (int k = 0; k < KBLK / 16; ++k)
                    umma_f16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                             (kb | k) != 0);
                umma_commit(&bars->aempty[sa]);
                umma_commit(&bars->bempty[sb]);
            }
            umma_commit(&bars->acc);
        }
    } else {
        // thread -> A row (tid & 127) and k-block c = tid >> 7 of every superblock
        const int row = tid & 127, c = tid >> 7;
        mbar_wait(&bars->qfull[0], 0);
        const uint8_t* rowp = qbuf + (size_t)row * RB;
        for (int sb = 0; sb < NKB / NA; ++sb) {
            mbar_wait(&bars->aempty[c], ((uint32_t)sb & 1u) ^ 1u);
            if (p.down_t == 2)
                dq_q6k_k64(rowp + sb * Q6K_BYTES, c, ast + c * A_STAGE, row);
            else
                dq_q4k_k64(rowp + sb * Q4K_BYTES, c, ast + c * A_STAGE, row);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->afull[c]);
        }
        mbar_wait(&bars->acc, 0);
        tc_fence_after();
        const int lq = warp & 3, ch = warp >> 2;
        const int hrow = h0 + 32 * lq + lane;
        for (int c0 = ch * 64; c0 < min(N, ch * 64 + 64); c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * lq) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int col = c0 + j;
                if (col < n) p.y[(size_t)(first + n0 + col) * H + hrow] = v[j];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, TMEM_COLS);
}

// x rows of every pair, in pair-list order, as fp16; inverse pair -> position map
__global__ void gather_x_f16(const float* __restrict__ x, const int32_t* __restrict__ pair_list,
                             int K, int H, __half* __restrict__ xp, int32_t* __restrict__ inv_pos) {
    const int pos = blockIdx.x;
    const int pr = pair_list[pos];
    const int t = pr / K;
    if (threadIdx.x == 0) inv_pos[pr] = pos;
    const float4* src = reinterpret_cast<const float4*>(x + (size_t)t * H);
    uint2* dst = reinterpret_cast<uint2*>(xp + (size_t)pos * H);
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
        const float4 v = src[i];
        dst[i] = make_uint2(pack_half2(v.x, v.y), pack_half2(v.z, v.w));
    }
}

// out[t][h] = res[t][h] + sum_j w[t][j] * y[pos(t,j)][h], slot order j = 0..K-1
__global__ void combine_pairs(const float* __restrict__ y, const int32_t* __restrict__ inv_pos,
                              const float* __restrict__ wts, const float* res, int H, int K,
                              float* out) {
    const int t = blockIdx.y;
    const int h = blockIdx.x * blockDim.x + threadIdx.x;
    if (h >= H) return;
    float acc = res[(size_t)t * H + h];
    for (int j = 0; j < K; ++j)
        acc = fmaf(wts[t * K + j], y[(size_t)inv_pos[t * K + j] * H + h], acc);
    out[(size_t)t * H + h] = acc;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 2-D map over a byte matrix [rows][row_bytes] (raw superblocks), box = box_bytes x box_rows
bool map_bytes(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_bytes,
               uint32_t box_r) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_bytes, box_r};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over an fp16 matrix [rows][cols], box = 64 cols x box_r rows, 128B swizzle
bool map_half(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_r) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {KBLK, box_r};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr size_t GU_SMEM = 1024 + ((NQ * QSTAGE_GU + 1023) & ~1023) + NA * A_STAGE + B_BYTES_GU +
                           sizeof(PfBars) + 64;

size_t dn_smem(int F, int down_t) {
    const size_t rb = (size_t)(F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    const size_t q = (TILE_M * rb + 1023) & ~size_t(1023);
    return 1024 + NA * A_STAGE + B_BYTES_DN + q + 1024 + sizeof(PfBars) + 64;
}

}  // namespace

bool prefill_supported(const MoeShape& s, int gate_t, int up_t, int down_t) {
    if (gate_t != 1 || up_t != 1) return false;
    if (s.H % QK || s.F % QK || s.H % TILE_M || s.F % 64) return false;
    return dn_smem(s.F, down_t) <= 227 * 1024 && GU_SMEM <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_prefill(const MoeShape& s, const float* x, const float* res,
                           const uint8_t* gate, const uint8_t* up, const uint8_t* down, int down_t,
                           const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                           float* out, cudaStream_t st) {
    const int P = s.T * s.K;
    const int max_used = P < s.E ? P : s.E;
    const int ntiles = (s.T + TILE_NMAX - 1) / TILE_NMAX;   // an expert sees each token once at most
    gather_x_f16<<<P, 128, 0, st>>>(x, r.pair_list, s.K, s.H, xp, inv_pos);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    CUtensorMap tg, tu, tx64, tx128, tx256, ta64, ta128, ta256;
    const uint64_t rbg = (uint64_t)(s.H / QK) * Q4K_BYTES;
    if (!map_bytes(&tg, gate, rbg, (uint64_t)s.E * s.F, Q4K_BYTES, 64) ||
        !map_bytes(&tu, up, rbg, (uint64_t)s.E * s.F, Q4K_BYTES, 64) ||
        !map_half(&tx64, xp, s.H, P, 64) || !map_half(&tx128, xp, s.H, P, 128) ||
        !map_half(&tx256, xp, s.H, P, 256) || !map_half(&ta64, actp, s.F, P, 64) ||
        !map_half(&ta128, actp, s.F, P, 128) || !map_half(&ta256, actp, s.F, P, 256))
        return cudaErrorInvalidValue;

    static bool attr_set = false;
    if (!attr_set) {
        e = cudaFuncSetAttribute(prefill_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(prefill_down, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    GuParams gp{r.n_used, r.used_expert, r.used_first, actp, s.H, s.F, ntiles};
    dim3 g1(s.F / 64, max_used * ntiles);
    prefill_gateup<<<g1, PF_THREADS, GU_SMEM, st>>>(tg, tu, tx64, tx128, tx256, gp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    DnParams dp{r.n_used, r.used_expert, r.used_first, down, y, s.H, s.F, ntiles, down_t};
    dim3 g2(s.H / TILE_M, max_used * ntiles);
    prefill_down<<<g2, PF_THREADS, dn_smem(s.F, down_t), st>>>(ta64, ta128, ta256, dp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g3((s.H + 255) / 256, s.T);
    combine_pairs<<<g3, 256, 0, st>>>(y, inv_pos, r.wts, res, s.H, s.K, out);
    return cudaGetLastError();
}

}  // namespace qmoe
