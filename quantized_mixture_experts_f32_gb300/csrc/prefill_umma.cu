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
//                   rows of Q4_K superblocks, TMA-loaded raw and dequantised to
//                   fp16 in shared memory (128B-swizzled K-major); B = the
//                   expert's gathered x rows via TMA; fp32 accumulator in TMEM;
//                   epilogue silu(g)*u -> fp16 act rows
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
constexpr int B_STAGE = TILE_NMAX * KBLK * 2;  // 32 KB fp16 B block (largest box)
constexpr int NDQ = 8;                         // dequant / epilogue warps
constexpr int PF_THREADS = (NDQ + 1) * 32;     // + producer / MMA warp
constexpr uint32_t TMEM_COLS = 256;

struct PfBars {
    uint64_t qfull[2], qempty[2], afull[2], aempty[2], bfull[3], bempty[3], acc;
    uint32_t tmem;
};

// token-tile height and the matching B tensor map (64 / 128 / 256 rows)
__device__ __forceinline__ int box_rows(int n) { return n <= 64 ? 64 : n <= 128 ? 128 : 256; }

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// 8 weights w = A*f - B with f = 0.5 + q/256 from 8 code bytes (4 per word,
// codes < 128) -> 4 packed half2
__device__ __forceinline__ uint4 codes_to_half8(uint32_t w0, uint32_t w1, float A, float B) {
    uint4 r;
    r.x = pack_half2(fmaf(A, mag<0>(w0), -B), fmaf(A, mag<1>(w0), -B));
    r.y = pack_half2(fmaf(A, mag<2>(w0), -B), fmaf(A, mag<3>(w0), -B));
    r.z = pack_half2(fmaf(A, mag<0>(w1), -B), fmaf(A, mag<1>(w1), -B));
    r.w = pack_half2(fmaf(A, mag<2>(w1), -B), fmaf(A, mag<3>(w1), -B));
    return r;
}

// one thread: 32 consecutive k of one A row from a Q4_K superblock at q
// (k-block c of the superblock, half h: sub-block 2c+h) -> fp16 SW128 tile
__device__ __forceinline__ void dq_q4k_row32(const uint8_t* q, int c, int h, uint8_t* atile, int row) {
    const uint4 hdr = *reinterpret_cast<const uint4*>(q);
    int sA, mA, sB, mB;
    q4_scales(hdr.y, hdr.z, hdr.w, c, sA, mA, sB, mB);
    const int s = h ? sB : sA, m = h ? mB : mA;
    const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
    const float ds = d * (float)s;
    const float A = 256.f * ds, B = fmaf(dmin, (float)m, 128.f * ds);   // w = ds*q - dmin*m
    const uint4* src = reinterpret_cast<const uint4*>(q + 16 + 32 * c);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint4 v = src[half];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            uint32_t a0 = w[2 * cc], a1 = w[2 * cc + 1];
            if (h) { a0 >>= 4; a1 >>= 4; }
            a0 &= 0x0F0F0F0Fu;
            a1 &= 0x0F0F0F0Fu;
            const int k = 32 * h + 16 * half + 8 * cc;           // first k of these 8
            *reinterpret_cast<uint4*>(atile + sw128_offset(row, k)) = codes_to_half8(a0, a1, A, B);
        }
    }
}

// 8 bytes at an even shared-memory address
__device__ __forceinline__ uint2 lds8(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* b = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = (uint32_t)(a & 3) * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2];
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

// one thread: 32 consecutive k of one A row from a Q6_K superblock at blk
// (2-byte aligned).  k-block q of the superblock (0..3), half h: group g =
// 2(q&1)+h of half n = q>>1, positions l = 0..31.
__device__ __forceinline__ void dq_q6k_row32(const uint8_t* blk, int qb, int h, uint8_t* atile,
                                             int row) {
    const int n = qb >> 1, g = 2 * (qb & 1) + h;
    const float d = __half2float(*reinterpret_cast<const __half*>(blk + 208));
    const uint8_t* qlp = blk + 64 * n + 32 * (g & 1);
    const uint8_t* qhp = blk + 128 + 32 * n;
    const int8_t s0 = static_cast<int8_t>(blk[192 + 8 * n + 2 * g]);       // l < 16
    const int8_t s1 = static_cast<int8_t>(blk[192 + 8 * n + 2 * g + 1]);   // l >= 16
    const int kbase = 32 * h;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {                         // 8 positions each
        const uint2 ql = lds8(qlp + 8 * cc), qh = lds8(qhp + 8 * cc);
        const int shl = 4 * (g >> 1), shh = 2 * g;
        const uint32_t c0 = ((ql.x >> shl) & 0x0F0F0F0Fu) | (((qh.x >> shh) & 0x03030303u) << 4);
        const uint32_t c1 = ((ql.y >> shl) & 0x0F0F0F0Fu) | (((qh.y >> shh) & 0x03030303u) << 4);
        const float ds = d * (float)(cc < 2 ? s0 : s1);
        // w = ds*(q6 - 32) = 256 ds f - 160 ds with f = 0.5 + q6/256
        *reinterpret_cast<uint4*>(atile + sw128_offset(row, kbase + 8 * cc)) =
            codes_to_half8(c0, c1, 256.f * ds, 160.f * ds);
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
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
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

    uint8_t* qst = sm;                                   // 2 x QSTAGE_GU
    uint8_t* ast = sm + 2 * 18432;                       // 2 x A_STAGE (1024-aligned)
    uint8_t* bst = ast + 2 * A_STAGE;                    // 3 x B_STAGE
    PfBars* bars = reinterpret_cast<PfBars*>(bst + 3 * B_STAGE);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->qfull[i], 1);
            mbar_init(&bars->qempty[i], NDQ);
            mbar_init(&bars->afull[i], NDQ);
            mbar_init(&bars->aempty[i], 1);
        }
        for (int i = 0; i < 3; ++i) {
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

    if (warp == NDQ) {
        if (lane == 0) {
            const int ybase = e * F + f0;
            auto load_q = [&](int s) {
                uint8_t* dst = qst + (s & 1) * 18432;
                mbar_arrive_expect_tx(&bars->qfull[s & 1], 2 * 64 * Q4K_BYTES);
                tma_load_2d(dst, &tm_gate, s * Q4K_BYTES, ybase, &bars->qfull[s & 1]);
                tma_load_2d(dst + 64 * Q4K_BYTES, &tm_up, s * Q4K_BYTES, ybase, &bars->qfull[s & 1]);
            };
            auto load_b = [&](int kb) {
                const int st = kb % 3;
                mbar_arrive_expect_tx(&bars->bfull[st], (uint32_t)(nb * KBLK * 2));
                tma_load_2d(bst + st * B_STAGE, tmx, kb * KBLK, first + n0, &bars->bfull[st]);
            };
            bool ok = true;
            for (int s = 0; s < 2 && s < NSB; ++s) load_q(s);
            for (int kb = 0; kb < 3 && kb < NKB; ++kb) load_b(kb);
            const uint32_t idesc = umma_idesc_f16(TILE_M, N);
            for (int kb = 0; kb < NKB && ok; ++kb) {
                const int sa = kb & 1, sb = kb % 3;
                ok = mbar_wait(&bars->afull[sa], (uint32_t)(kb >> 1) & 1u) &&
                     mbar_wait(&bars->bfull[sb], (uint32_t)(kb / 3) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = umma_sdesc(smem_u32(ast + sa * A_STAGE));
                const uint64_t bd = umma_sdesc(smem_u32(bst + sb * B_STAGE));
#pragma unroll
                for (int k = 0; k < KBLK / 16; ++k)
                    umma_f16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                             (kb | k) != 0);
                umma_commit(&bars->aempty[sa]);
                umma_commit(&bars->bempty[sb]);
                if (kb + 3 < NKB) {
                    ok = mbar_wait(&bars->bempty[sb], (uint32_t)(kb / 3) & 1u);
                    if (ok) load_b(kb + 3);
                }
                if ((kb & 3) == 3 && (kb >> 2) + 2 < NSB) {
                    const int s = kb >> 2;
                    ok = ok && mbar_wait(&bars->qempty[s & 1], (uint32_t)(s >> 1) & 1u);
                    if (ok) load_q(s + 2);
                }
            }
            umma_commit(&bars->acc);
        }
    } else {
        // dequant: thread -> A row (tid & 127), k half (tid >> 7)
        const int row = tid & 127, h = tid >> 7;
        const int grp = row >> 5, w32 = row & 31;
        const int src = w32 < 16 ? 16 * grp + w32 : 64 + 16 * grp + (w32 - 16);
        for (int kb = 0; kb < NKB; ++kb) {
            const int s = kb >> 2, c = kb & 3, sa = kb & 1;
            if (c == 0) mbar_wait(&bars->qfull[s & 1], (uint32_t)(s >> 1) & 1u);
            mbar_wait(&bars->aempty[sa], ((uint32_t)(kb >> 1) & 1u) ^ 1u);
            dq_q4k_row32(qst + (s & 1) * 18432 + src * Q4K_BYTES, c, h, ast + sa * A_STAGE, row);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars->afull[sa]);
                if (c == 3) mbar_arrive(&bars->qempty[s & 1]);
            }
        }
        // epilogue: TMEM lane quarter (warp % 4); column half (warp / 4)
        mbar_wait(&bars->acc, 0);
        tc_fence_after();
        const int lq = warp & 3, ch = warp >> 2;
        const int f = f0 + 16 * lq + (lane & 15);
        for (int c0 = ch * 128; c0 < min(N, ch * 128 + 128); c0 += 16) {
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
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
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

    uint8_t* ast = sm;                                    // 2 x A_STAGE
    uint8_t* bst = ast + 2 * A_STAGE;                     // 3 x B_STAGE
    uint8_t* qbuf = bst + 3 * B_STAGE;                    // qbytes (+ slack)
    PfBars* bars = reinterpret_cast<PfBars*>(qbuf + ((qbytes + 1023) & ~1023u) + 1024);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&bars->qfull[0], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->afull[i], NDQ);
            mbar_init(&bars->aempty[i], 1);
        }
        for (int i = 0; i < 3; ++i) {
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

    if (warp == NDQ) {
        if (lane == 0) {
            const uint8_t* src = p.down + (size_t)e * H * RB + (size_t)h0 * RB;
            mbar_arrive_expect_tx(&bars->qfull[0], qbytes);
            bulk_g2s(qbuf, src, qbytes, &bars->qfull[0]);
            auto load_b = [&](int kb) {
                const int st = kb % 3;
                mbar_arrive_expect_tx(&bars->bfull[st], (uint32_t)(nb * KBLK * 2));
                tma_load_2d(bst + st * B_STAGE, tmb, kb * KBLK, first + n0, &bars->bfull[st]);
            };
            bool ok = true;
            for (int kb = 0; kb < 3 && kb < NKB; ++kb) load_b(kb);
            const uint32_t idesc = umma_idesc_f16(TILE_M, N);
            for (int kb = 0; kb < NKB && ok; ++kb) {
                const int sa = kb & 1, sb = kb % 3;
                ok = mbar_wait(&bars->afull[sa], (uint32_t)(kb >> 1) & 1u) &&
                     mbar_wait(&bars->bfull[sb], (uint32_t)(kb / 3) & 1u);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = umma_sdesc(smem_u32(ast + sa * A_STAGE));
                const uint64_t bd = umma_sdesc(smem_u32(bst + sb * B_STAGE));
#pragma unroll
                for (int k = 0; k < KBLK / 16; ++k)
                    umma_f16(tmem, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc,
                             (kb | k) != 0);
                umma_commit(&bars->aempty[sa]);
                umma_commit(&bars->bempty[sb]);
                if (kb + 3 < NKB) {
                    ok = mbar_wait(&bars->bempty[sb], (uint32_t)(kb / 3) & 1u);
                    if (ok) load_b(kb + 3);
                }
            }
            umma_commit(&bars->acc);
        }
    } else {
        const int row = tid & 127, h = tid >> 7;
        mbar_wait(&bars->qfull[0], 0);
        const uint8_t* rowp = qbuf + (size_t)row * RB;
        for (int kb = 0; kb < NKB; ++kb) {
            const int sa = kb & 1;
            mbar_wait(&bars->aempty[sa], ((uint32_t)(kb >> 1) & 1u) ^ 1u);
            const int s = kb >> 2, qb = kb & 3;
            if (p.down_t == 2)
                dq_q6k_row32(rowp + s * Q6K_BYTES, qb, h, ast + sa * A_STAGE, row);
            else
                dq_q4k_row32(rowp + s * Q4K_BYTES, qb, h, ast + sa * A_STAGE, row);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->afull[sa]);
        }
        mbar_wait(&bars->acc, 0);
        tc_fence_after();
        const int lq = warp & 3, ch = warp >> 2;
        const int hrow = h0 + 32 * lq + lane;
        for (int c0 = ch * 128; c0 < min(N, ch * 128 + 128); c0 += 16) {
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

constexpr size_t GU_SMEM = 1024 + 2 * 18432 + 2 * A_STAGE + 3 * B_STAGE + sizeof(PfBars) + 64;

size_t dn_smem(int F, int down_t) {
    const size_t rb = (size_t)(F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    const size_t q = (TILE_M * rb + 1023) & ~size_t(1023);
    return 1024 + 2 * A_STAGE + 3 * B_STAGE + q + 1024 + sizeof(PfBars) + 64;
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
