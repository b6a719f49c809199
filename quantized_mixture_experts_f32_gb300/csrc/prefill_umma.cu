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
//                   by 16 dequant warps, all of them on each k-block in turn
//                   (4 A stages ahead of the MMA); B = the expert's gathered
//                   x rows via TMA; fp32
//                   accumulator in TMEM; epilogue silu(g)*u -> fp16 act rows
//   prefill_down    per (expert, 128-row tile, token tile): A = 128 down rows
//                   (Q6_K or Q4_K, one bulk copy of the whole K), B = act rows,
//                   epilogue -> fp32 y rows per pair
//   combine_pairs   out[t] = res[t] + sum_j w[t][j] y[pos(t, j)] in slot order
// Weights are on the MMA's M side ("swap-AB"): expert segments are short (32
// tokens on average), so token tiles of 16..256 are the N side.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cudaTypedefs.h>
#include <math.h>

#include "kquant.cuh"
#include "pdl.cuh"
#include "qmoe_internal.h"
#include "umma.cuh"

namespace qmoe {

namespace {

constexpr int KBLK = 64;                       // k per tensor-core block (128 B of fp16)
constexpr int TILE_M = 128;
constexpr int A_STAGE = TILE_M * KBLK * 2;     // 16 KB fp16 A block
constexpr int NDQ = 16;                        // dequant / epilogue warps (4 threads per A row)
constexpr int RPT = 16 / NDQ;                  // A rows per dequant thread
static_assert(NDQ * RPT == 16 && NDQ % 4 == 0, "128 A rows, 8 per warp per pass");
constexpr int W_QLOAD = NDQ;                   // weight copies
constexpr int W_BLOAD = NDQ + 1;               // activation (B) tiles
constexpr int W_MMA = NDQ + 2;                 // tcgen05.mma issue
constexpr int NA = 4;                          // A (fp16 weight) stages: the 4 k-blocks of a superblock
static_assert(NA * KBLK == QK, "one A stage per k-block of a superblock");
constexpr int NQ = 3;                          // raw Q4_K stages, at most
// gate/up kernel: token-tile rows, raw and A stages, CTAs per SM it is built
// for (the stage rings and TMEM columns must fit that many CTAs), TMEM columns.
// The A (weight) and B (token) rings have the same depth and share their
// barriers, one full / empty pair per two consecutive stages: the MMA thread
// waits once and commits once per two k-blocks.  Its loop is a chain of
// dependent operations (barrier wait, tcgen05.mma issues, commit), and that
// chain, not the tensor core, sets the pace for token tiles of a few dozen
// rows; fewer barrier operations per MMA shorten it.
constexpr int GU_NMAX = 192;
constexpr int GU_NQ = 3;
constexpr int GU_NA = 4;
constexpr int GU_ACC_COLS = 256;               // TMEM columns per accumulator (two of them)
constexpr uint32_t GU_TMEM = 2 * GU_ACC_COLS;
constexpr int GU_NEPI = 8;                     // epilogue warps, two per TMEM lane quarter
constexpr int W_EPI = NDQ + 4;                 // the first of them (a multiple of 4)
constexpr int GU_THREADS = (NDQ + 4 + GU_NEPI) * 32;
static_assert(GU_NQ <= NQ && GU_NA == 4 && GU_NMAX <= GU_ACC_COLS &&
                  W_EPI % 4 == 0,
              "gate/up rings");
constexpr int QSTAGE_GU = 2 * 64 * Q4K_BYTES;  // 64 gate + 64 up rows of one superblock column
// FP8 experts: a raw stage is one 128-column scale block of the item's rows
// (64 gate + 64 up rows for gate/up, 128 rows for down): two k-blocks
constexpr int F8_COLS = 128;
constexpr int QSTAGE_F8 = 128 * F8_COLS;
constexpr int F8_NQ = 3;
// NVFP4 experts (QF 2): a raw stage is one 256-column slice of the item's rows,
// E2M1 codes (128 bytes a row) then their E4M3 block scales (16 bytes a row)
constexpr int NV_COLS = 256;
constexpr int NV_CB = NV_COLS / 2, NV_SB = NV_COLS / 16;      // code / scale bytes per row
constexpr int QSTAGE_NV = 128 * (NV_CB + NV_SB);
template <int QF> __host__ __device__ constexpr int gu_qbytes() {
    return QF == 1 ? F8_NQ * QSTAGE_F8 : QF == 2 ? F8_NQ * QSTAGE_NV : GU_NQ * QSTAGE_GU;
}
// raw bytes of the down kernel's ring (two halves, 2 KB-aligned so that the A
// stages after it stay 1 KB-aligned)
template <int QF> __host__ __device__ constexpr int dn_qring() {
    return QF == 1 ? F8_NQ * QSTAGE_F8 : QF == 2 ? ((F8_NQ * QSTAGE_NV + 2047) & ~2047) : 0;
}
// down kernel: token-tile rows, A / B stages, TMEM columns (two accumulators)
constexpr int DN_NMAX = 128;
constexpr int DN_NA = 2;
constexpr int DN_BSTAGE = DN_NMAX * KBLK * 2;
constexpr uint32_t DN_TMEM = 2 * DN_NMAX;
constexpr int GU_BSTAGE = GU_NMAX * KBLK * 2;  // B stage stride (an item loads nb <= GU_NMAX rows)
constexpr int B_BYTES_GU = GU_NA * GU_BSTAGE;

struct PfBars {
    uint64_t qfull[NQ], qempty[NQ], afull[NA], aempty[NA];
    uint64_t accfull[2], accempty[2];
    uint32_t tmem;
};

// token-tile height of the gate/up kernel and the matching B tensor map (64 /
// 128 / GU_NMAX rows)
__device__ __forceinline__ int box_rows_gu(int n) { return n <= 64 ? 64 : n <= 128 ? 128 : GU_NMAX; }

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

// 16 E4M3 codes (k order) times the block scale -> two 16-byte runs of 8 fp16
// weights, stored at the row's swizzled chunks o0 and o1 (the E4M3 -> fp16
// widening is exact; the product is rounded once, to fp16)
__device__ __forceinline__ void f8_quarter(uint4 q, float s, uint8_t* arow, int o0, int o1) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
                static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * hh)) & 0xffffu), __NV_E4M3);
            const float2 f = __half22float2(__half2(r));
            h[2 * i + hh] = pack_half2(f.x * s, f.y * s);
        }
    }
    *reinterpret_cast<uint4*>(arow + o0) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(arow + o1) = make_uint4(h[4], h[5], h[6], h[7]);
}

// 16 E2M1 codes (8 bytes, the even element in each low nibble) times the block
// scale -> two 16-byte runs of 8 fp16 weights at the row's swizzled chunks
__device__ __forceinline__ void nv_quarter(uint2 q, float s, uint8_t* arow, int o0, int o1) {
    const uint32_t w[2] = {q.x, q.y};
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const __half2_raw r = __nv_cvt_fp4x2_to_halfraw2(
                static_cast<__nv_fp4x2_storage_t>((w[i] >> (8 * b)) & 0xffu), __NV_E2M1);
            const float2 f = __half22float2(__half2(r));
            h[4 * i + b] = pack_half2(f.x * s, f.y * s);
        }
    }
    *reinterpret_cast<uint4*>(arow + o0) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(arow + o1) = make_uint4(h[4], h[5], h[6], h[7]);
}

__device__ __forceinline__ float e4m3_float(uint32_t byte) {
    const __half_raw r = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(byte & 0xffu), __NV_E4M3);
    return __half2float(__half(r));
}

// Q4_K: scale and offset of the two sub-blocks (2c, 2c + 1) of k-block c, as
// half2 bit patterns {d*s, -dmin*m} (w = d*s*q - dmin*m)
struct Q4Half {
    uint32_t sA, cA, sB, cB;
};

__device__ __forceinline__ Q4Half q4_half_scales(uint4 hdr, int c) {
    int sA, mA, sB, mB;
    q4_scales(hdr.y, hdr.z, hdr.w, c, sA, mA, sB, mB);
    const float d = half_bits(hdr.x), dmin = half_bits(hdr.x >> 16);
    return {h2_bits(__float2half2_rn(d * (float)sA)), h2_bits(__float2half2_rn(-dmin * (float)mA)),
            h2_bits(__float2half2_rn(d * (float)sB)), h2_bits(__float2half2_rn(-dmin * (float)mB))};
}

__device__ __forceinline__ Q4Half shfl_half(const Q4Half& v, int src) {
    return {__shfl_sync(0xffffffffu, v.sA, src), __shfl_sync(0xffffffffu, v.cA, src),
            __shfl_sync(0xffffffffu, v.sB, src), __shfl_sync(0xffffffffu, v.cB, src)};
}

// one 16-k quarter of a Q4_K k-block: 8 code bytes v hold 8 k of sub-block 2c
// in their low nibbles and the same 8 k of sub-block 2c + 1 in their high
// nibbles -> two 16-byte fp16 pieces of the row (offsets o_lo, o_hi in the
// 128B-swizzled tile)
__device__ __forceinline__ void q4_quarter(uint2 v, const Q4Half& s, uint8_t* rb, int o_lo, int o_hi) {
    const __half2 sub = __float2half2_rn(1024.f);
    *reinterpret_cast<uint4*>(rb + o_lo) =
        codes_to_half8(v.x & 0x0F0F0F0Fu, v.y & 0x0F0F0F0Fu, sub, bits_h2(s.sA), bits_h2(s.cA));
    *reinterpret_cast<uint4*>(rb + o_hi) = codes_to_half8((v.x >> 4) & 0x0F0F0F0Fu, (v.y >> 4) & 0x0F0F0F0Fu,
                                                          sub, bits_h2(s.sB), bits_h2(s.cB));
}

// 16 bytes at an even shared-memory address (five aligned words, funnel shift)
__device__ __forceinline__ uint4 lds16(const uint8_t* p) {
    const uint32_t off = smem_u32(p) & 3u;
    const uint32_t* b = reinterpret_cast<const uint32_t*>(p - off);   // stays a shared pointer
    const uint32_t sh = off * 8u;
    const uint32_t w0 = b[0], w1 = b[1], w2 = b[2], w3 = b[3], w4 = b[4];
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh),
                      __funnelshift_r(w2, w3, sh), __funnelshift_r(w3, w4, sh));
}

// one 16-k quarter of a Q6_K k-block: 16 ql bytes (nibble at shl) and 16 qh
// bytes (2 bits at shh) -> 6-bit codes, w = ds*(q6 - 32) -> two 16-byte pieces
__device__ __forceinline__ void q6_quarter(uint4 ql, uint4 qh, int shl, int shh, __half2 ds, uint8_t* rb,
                                           int o0, int o1) {
    const __half2 sub = __float2half2_rn(1056.f), zero = __float2half2_rn(0.f);
    const uint32_t l[4] = {ql.x, ql.y, ql.z, ql.w}, hb[4] = {qh.x, qh.y, qh.z, qh.w};
    uint32_t c[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        c[i] = ((l[i] >> shl) & 0x0F0F0F0Fu) | (((hb[i] >> shh) & 0x03030303u) << 4);
    *reinterpret_cast<uint4*>(rb + o0) = codes_to_half8(c[0], c[1], sub, ds, zero);
    *reinterpret_cast<uint4*>(rb + o1) = codes_to_half8(c[2], c[3], sub, ds, zero);
}

struct GuParams {
    const int32_t* n_used;
    const int32_t* used_expert;
    const int32_t* used_first;
    __half* act;          // [P][F] fp16, rows in pair-list order
    int H, F;             // K of the GEMM; rows per expert (MODE 0) / of all segments (MODE 1)
    // plain mode (dense Q4_K GEMMs): up to three weight matrices ("segments",
    // maps tm_gate, tm_up, tm_w2) over the same x, segment s writing
    // y[t][seg_yoff[s] + r] = sum_k W_s[r][k] x[t][k] (+ res[t][...]); with
    // ksplit = 2 each item takes half of K and writes its own plane
    // y + kh * part_stride (no res), the caller adding the two
    float* y;
    const float* res;
    int dense_T, ldy;
    int seg_rows[3], seg_yoff[3];
    int ksplit;
    size_t part_stride;
    // FP8 experts (QF 1): fp32 scales per 128 x 128 block, [E][F/128][H/128];
    // NVFP4 experts (QF 2): fp32 global scales [E] (block scales come by TMA)
    const float* gscale;
    const float* uscale;
};

// One work item of the gate/up kernel: weight rows f0 .. of expert e (MODE 1:
// of segment e) against the token rows first + n0 .. first + n0 + n - 1, over
// K half kh (MODE 1 with ksplit 2; else 0).
struct GuItem {
    int e, first, n0, n, f0, kh;
};

// Items in the order (token tile, weight-row tile), the row tile fastest, so
// that CTAs working at the same time share the token rows in L2.  MODE 0: the
// token tiles are those of every used expert in turn (tfirst: exclusive
// prefix of the tiles per used expert); MODE 1: the dense_T tokens.
template <int MODE>
__device__ __forceinline__ GuItem gu_item(const GuParams& p, const int* tfirst, int n_used, int it) {
    GuItem w;
    const int FT = MODE == 0 ? p.F / 64 : p.F / TILE_M;
    const int KS = MODE == 0 ? 1 : p.ksplit;
    const int tt = it / (FT * KS), rem = it - tt * FT * KS;
    w.kh = rem / FT;
    const int ft = rem - w.kh * FT;
    if (MODE == 0) {
        int lo = 0, hi = n_used - 1;                     // last u with tfirst[u] <= tt
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tfirst[mid] <= tt) lo = mid;
            else hi = mid - 1;
        }
        w.e = p.used_expert[lo];
        w.first = p.used_first[lo];
        w.n0 = (tt - tfirst[lo]) * GU_NMAX;
        w.n = min(GU_NMAX, p.used_first[lo + 1] - w.first - w.n0);
        w.f0 = ft * 64;
    } else {
        int seg = 0, f = ft * TILE_M;
        if (f >= p.seg_rows[0]) {
            f -= p.seg_rows[0];
            seg = 1;
            if (f >= p.seg_rows[1]) {
                f -= p.seg_rows[1];
                seg = 2;
            }
        }
        w.e = seg;
        w.first = 0;
        w.n0 = tt * GU_NMAX;
        w.n = min(GU_NMAX, p.dense_T - w.n0);
        w.f0 = f;
    }
    return w;
}

// Persistent: one CTA per SM walks the items blockIdx.x, blockIdx.x + gridDim.x,
// ...; every ring (raw superblocks, A + B k-blocks, two TMEM accumulators)
// runs on across items, so one item's loads and dequantisation overlap the
// previous item's last MMAs and its epilogue.  MODE 0: A = 64 gate + 64 up
// rows of one expert, epilogue silu(g)*u -> fp16 act.  MODE 1: A = 128
// consecutive rows of one Q4_K matrix [F][H], B = the dense_T token rows of x,
// epilogue fp32 y (+ res).  Warps: NDQ dequant, Q load, B load, MMA, one idle,
// GU_NEPI epilogue.
template <int MODE, int QF>
__global__ void __launch_bounds__(GU_THREADS, 1)
    prefill_gateup(const __grid_constant__ CUtensorMap tm_gate, const __grid_constant__ CUtensorMap tm_up,
                   const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_x64,
                   const __grid_constant__ CUtensorMap tm_x128, const __grid_constant__ CUtensorMap tm_xg,
                   const __grid_constant__ CUtensorMap tm_gsc, const __grid_constant__ CUtensorMap tm_usc,
                   const GuParams p) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(1024) uint8_t smraw[];
    // 1024-aligned base, kept a shared-space pointer (an integer round trip
    // would turn every access into a generic one)
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const int H = p.H, F = p.F;
    const int KS = MODE == 0 ? 1 : p.ksplit;
    static_assert(QF == 0 || MODE == 0, "FP8 / NVFP4 weights in the MoE mode only");
    constexpr int NQS = QF ? F8_NQ : GU_NQ;              // raw stages
    constexpr int QSB = QF == 1 ? QSTAGE_F8 : QF == 2 ? QSTAGE_NV : QSTAGE_GU;   // raw stage bytes
    constexpr int QCOL = QF == 1 ? F8_COLS : QF == 2 ? NV_CB : Q4K_BYTES;   // code bytes per row per stage
    constexpr int KPS = QF == 1 ? F8_COLS / KBLK : QK / KBLK;   // k-blocks per raw stage
    const int NKB = H / KBLK / KS, NSB = NKB / KPS;      // per item
    const int FT = MODE == 0 ? F / 64 : F / TILE_M;

    uint8_t* qst = sm;                                   // NQS x QSB
    uint8_t* ast = sm + ((gu_qbytes<QF>() + 1023) & ~1023);  // GU_NA x A_STAGE (1024-aligned)
    uint8_t* bst = ast + GU_NA * A_STAGE;                // GU_NA x GU_BSTAGE
    PfBars* bars = reinterpret_cast<PfBars*>(bst + B_BYTES_GU);
    int* tfirst = reinterpret_cast<int*>(bars + 1);      // [n_used + 1] (MODE 0)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int n_used = MODE == 0 ? *p.n_used : 0;
    if (tid == 0) {
        for (int i = 0; i < NQS; ++i) {
            mbar_init(&bars->qfull[i], 1);
            mbar_init(&bars->qempty[i], NDQ);
        }
        for (int i = 0; i < GU_NA / 2; ++i) {
            mbar_init(&bars->afull[i], 2 * (NDQ + 1));   // per k-block: dequant warps + the B copy
            mbar_init(&bars->aempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->accfull[i], 1);
            mbar_init(&bars->accempty[i], GU_NEPI);
        }
        fence_barrier_init();
    }
    if (MODE == 0 && warp == W_QLOAD) {
        // token tiles per used expert, exclusive prefix (one warp)
        int carry = 0;
        for (int u0 = 0; u0 < n_used; u0 += 32) {
            const int u = u0 + lane;
            const int t = u < n_used ? (p.used_first[u + 1] - p.used_first[u] + GU_NMAX - 1) / GU_NMAX : 0;
            int incl = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (u < n_used) tfirst[u] = carry + incl - t;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) tfirst[n_used] = carry;
    }
    if (warp == 0) tmem_alloc(&bars->tmem, GU_TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem;
    const int n_items = MODE == 0 ? FT * tfirst[n_used] : FT * KS * ((p.dense_T + GU_NMAX - 1) / GU_NMAX);

    if (warp == W_QLOAD) {
        // raw superblock columns of each item's 128 weight rows, GU_NQ ahead
        if (lane == 0) {
            int gs = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const GuItem w = gu_item<MODE>(p, tfirst, n_used, it);
                const int ybase = MODE == 0 ? w.e * F + w.f0 : w.f0;
                const CUtensorMap* tw = MODE == 0 ? &tm_gate : w.e == 0 ? &tm_gate : w.e == 1 ? &tm_up : &tm_w2;
                const int sb0 = w.kh * NSB;
                for (int sb = 0; sb < NSB; ++sb, ++gs) {
                    const int st = gs % NQS;
                    if (!mbar_wait(&bars->qempty[st], ((uint32_t)(gs / NQS) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = qst + st * QSB;
                    mbar_arrive_expect_tx(&bars->qfull[st], QSB);
                    tma_load_2d(dst, tw, (sb0 + sb) * QCOL, ybase, &bars->qfull[st]);
                    if (MODE == 0)
                        tma_load_2d(dst + 64 * QCOL, &tm_up, sb * QCOL, ybase, &bars->qfull[st]);
                    else
                        tma_load_2d(dst + 64 * QCOL, tw, (sb0 + sb) * QCOL, ybase + 64, &bars->qfull[st]);
                    if (QF == 2) {
                        tma_load_2d(dst + 128 * NV_CB, &tm_gsc, sb * NV_SB, ybase, &bars->qfull[st]);
                        tma_load_2d(dst + 128 * NV_CB + 64 * NV_SB, &tm_usc, sb * NV_SB, ybase, &bars->qfull[st]);
                    }
                }
            }
        }
    } else if (warp == W_BLOAD) {
        // each item's token rows, in step with the A stages (which share the
        // stage barriers: full = the dequant warps' arrivals plus this copy)
        if (lane == 0) {
            int gk = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                const GuItem w = gu_item<MODE>(p, tfirst, n_used, it);
                const int nb = box_rows_gu(w.n);
                const CUtensorMap* tmx = nb == 64 ? &tm_x64 : nb == 128 ? &tm_x128 : &tm_xg;
                for (int kb = 0; kb < NKB; ++kb, ++gk) {
                    const int st = gk % GU_NA, pr = (gk >> 1) & 1;
                    if (!mbar_wait(&bars->aempty[pr], ((uint32_t)(gk / GU_NA) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->afull[pr], (uint32_t)(nb * KBLK * 2));
                    tma_load_2d(bst + st * GU_BSTAGE, tmx, (w.kh * NKB + kb) * KBLK, w.first + w.n0,
                                &bars->afull[pr]);
                }
            }
        }
    } else if (warp == W_MMA) {
        if (lane == 0) {
            int gp = 0, j = 0;                           // k-block pairs, items
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++j) {
                const GuItem w = gu_item<MODE>(p, tfirst, n_used, it);
                const int buf = j & 1;
                // the epilogue has drained this accumulator (item j - 2)
                if (!mbar_wait(&bars->accempty[buf], ((uint32_t)(j >> 1) & 1u) ^ 1u)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * GU_ACC_COLS);
                const uint32_t idesc = umma_idesc_f16(TILE_M, (w.n + 15) & ~15);
                for (int kp = 0; kp < NKB / 2; ++kp, ++gp) {
                    const int pr = gp & 1;
                    if (!mbar_wait(&bars->afull[pr], (uint32_t)(gp >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int sa = 2 * pr + h, kb = 2 * kp + h;
                        const uint64_t ad = umma_sdesc(smem_u32(ast + sa * A_STAGE));
                        const uint64_t bd = umma_sdesc(smem_u32(bst + sa * GU_BSTAGE));
#pragma unroll
                        for (int k = 0; k < KBLK / 16; ++k)
                            umma_f16(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, (kb | k) != 0);
                    }
                    umma_commit(&bars->aempty[pr]);
                }
                if (ok) umma_commit(&bars->accfull[buf]);
            }
        }
    } else if (QF == 2 && warp < NDQ) {
        // NVFP4 dequant: thread -> A row 8*warp + (lane & 7) and 16-k quarter
        // qq = lane >> 3 of each k-block (one 16-element scale block: 8 code
        // bytes and one scale byte); A rows paired gate / up as for k-quants
        const int qq = lane >> 3, sw = lane & 7;
        const int row = 8 * warp + (lane & 7);
        const int grp = row >> 5, w32 = row & 31;
        const bool is_gate = w32 < 16;
        const int srow = is_gate ? 16 * grp + w32 : 64 + 16 * grp + (w32 - 16);
        const int rowb = row * 128;
        const int o0 = ((2 * qq) ^ sw) << 4, o1 = ((2 * qq + 1) ^ sw) << 4;
        const float* glob = is_gate ? p.gscale : p.uscale;
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        int gk = 0, gs = 0;
        bool ok = true;
        for (int j = 0; ok && j < my_items; ++j) {
            const GuItem w = gu_item<MODE>(p, tfirst, n_used, blockIdx.x + j * gridDim.x);
            const float gsc = __ldg(glob + w.e);
            for (int sb = 0; sb < NSB; ++sb, ++gs) {
                const int sq = gs % NQS;
                const uint8_t* stg = qst + sq * QSB;
                if (!mbar_wait(&bars->qfull[sq], (uint32_t)(gs / NQS) & 1u)) {
                    ok = false;
                    break;
                }
                uint2 v[KPS];
#pragma unroll
                for (int c = 0; c < KPS; ++c)
                    v[c] = *reinterpret_cast<const uint2*>(stg + srow * NV_CB + 32 * c + 8 * qq);
                const uint4 scw = *reinterpret_cast<const uint4*>(stg + 128 * NV_CB + srow * NV_SB);
                const uint32_t sc4[4] = {scw.x, scw.y, scw.z, scw.w};   // byte 4 c + qq: word c, byte qq
#pragma unroll
                for (int c = 0; c < KPS; ++c, ++gk) {
                    const int sa = gk % GU_NA, pr = (gk >> 1) & 1;
                    const float sc = e4m3_float(sc4[c] >> (8 * qq)) * gsc;
                    if (!mbar_wait(&bars->aempty[pr], ((uint32_t)(gk / GU_NA) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    nv_quarter(v[c], sc, ast + sa * A_STAGE + rowb, o0, o1);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->afull[pr]);
                }
                if (!ok) break;
                if (lane == 0) mbar_arrive(&bars->qempty[sq]);
            }
        }
    } else if (QF == 1 && warp < NDQ) {
        // FP8 dequant: thread -> A row 8*warp + (lane & 7) and 16-k quarter
        // qq = lane >> 3 of each k-block; A rows 32 g .. 32 g + 15 are gate rows
        // 16 g .., the next 16 the matching up rows (as for k-quants).  The
        // row's scale is the item's (row block, column block) scale of gate or up.
        const int qq = lane >> 3, sw = lane & 7;
        const int row = 8 * warp + (lane & 7);
        const int grp = row >> 5, w32 = row & 31;
        const bool is_gate = w32 < 16;
        const int srow = (is_gate ? 16 * grp + w32 : 64 + 16 * grp + (w32 - 16)) * F8_COLS;
        const int rowb = row * 128;
        const int o0 = ((2 * qq) ^ sw) << 4, o1 = ((2 * qq + 1) ^ sw) << 4;
        const float* scale = is_gate ? p.gscale : p.uscale;
        const int nbh = H / F8_COLS;
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        int gk = 0, gs = 0;
        bool ok = true;
        for (int j = 0; ok && j < my_items; ++j) {
            const GuItem w = gu_item<MODE>(p, tfirst, n_used, blockIdx.x + j * gridDim.x);
            const float* srow_scale = scale + ((size_t)w.e * (F / F8_COLS) + w.f0 / F8_COLS) * nbh;
            for (int sb = 0; sb < NSB; ++sb, ++gs) {
                const int sq = gs % NQS;
                const uint8_t* stg = qst + sq * QSB;
                if (!mbar_wait(&bars->qfull[sq], (uint32_t)(gs / NQS) & 1u)) {
                    ok = false;
                    break;
                }
                uint4 v[KPS];
#pragma unroll
                for (int c = 0; c < KPS; ++c) v[c] = *reinterpret_cast<const uint4*>(stg + srow + KBLK * c + 16 * qq);
                const float sc = __ldg(srow_scale + sb);
#pragma unroll
                for (int c = 0; c < KPS; ++c, ++gk) {
                    const int sa = gk % GU_NA, pr = (gk >> 1) & 1;
                    if (!mbar_wait(&bars->aempty[pr], ((uint32_t)(gk / GU_NA) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    f8_quarter(v[c], sc, ast + sa * A_STAGE + rowb, o0, o1);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->afull[pr]);
                }
                if (!ok) break;
                // every value loaded from the raw stage has fed a store above
                if (lane == 0) mbar_arrive(&bars->qempty[sq]);
            }
        }
    } else if (QF == 0 && warp < NDQ) {
        // dequant: thread -> A rows 8*warp + (lane & 7) (+ 8*NDQ*r) and 16-k
        // quarter qq = lane >> 3 of every k-block (each 8-lane phase of a 16-byte
        // store then covers all 32 banks).  All NDQ warps fill each A stage in turn, so
        // the GU_NA stages run ahead of the MMA.
        // A raw superblock column is read into registers at once (its stage is
        // released after the superblock's k-blocks); the scales of k-block c are
        // decoded by the row's lane with qq == c and shuffled to the other three.
        const int qq = lane >> 3;
        int src[RPT], rowb[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = 8 * warp + (lane & 7) + 8 * NDQ * r;
            const int grp = row >> 5, w32 = row & 31;
            // gate/up: A rows 32 g .. 32 g + 15 are gate rows 16 g .., the next 16
            // the matching up rows (so TMEM lanes l and l + 16 pair up in the
            // epilogue); plain: A row = stage row
            src[r] = (MODE == 1 ? row : w32 < 16 ? 16 * grp + w32 : 64 + 16 * grp + (w32 - 16)) * Q4K_BYTES;
            rowb[r] = row * 128;
        }
        const int o_lo = (qq ^ (lane & 7)) << 4, o_hi = ((qq + 4) ^ (lane & 7)) << 4;   // row % 8 == lane % 8
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        int gk = 0;
        for (int gs = 0; gs < my_items * NSB; ++gs) {
            const int sq = gs % NQS;
            const uint8_t* stg = qst + sq * QSB;
            if (!mbar_wait(&bars->qfull[sq], (uint32_t)(gs / NQS) & 1u)) break;
            uint4 hdr[RPT];
            uint2 v[RPT][4];
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                hdr[r] = *reinterpret_cast<const uint4*>(stg + src[r]);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    v[r][c] = *reinterpret_cast<const uint2*>(stg + src[r] + 16 + 32 * c + 8 * qq);
            }
            Q4Half own[RPT];
#pragma unroll
            for (int r = 0; r < RPT; ++r) own[r] = q4_half_scales(hdr[r], qq);
            bool ok = true;
#pragma unroll
            for (int c = 0; c < 4; ++c, ++gk) {
                const int sa = gk % GU_NA, pr = (gk >> 1) & 1;
                Q4Half sc[RPT];
#pragma unroll
                for (int r = 0; r < RPT; ++r) sc[r] = shfl_half(own[r], (lane & 7) + 8 * c);
                if (!mbar_wait(&bars->aempty[pr], ((uint32_t)(gk / GU_NA) & 1u) ^ 1u)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int r = 0; r < RPT; ++r) q4_quarter(v[r][c], sc[r], ast + sa * A_STAGE + rowb[r], o_lo, o_hi);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->afull[pr]);
            }
            if (!ok) break;
            // the raw stage is handed back only now: every value loaded from it
            // has fed a store above, so no load of this warp is still pending
            // when the next TMA copy may overwrite it (releasing right after the
            // loads were issued let a late load read the next superblock)
            if (lane == 0) mbar_arrive(&bars->qempty[sq]);
        }
    } else if (warp >= W_EPI) {
        // epilogue: TMEM lane quarter warp % 4; the two warps of a quarter take
        // alternate 16-column chunks
        const int lq = warp & 3, half = (warp - W_EPI) >> 2;
        int j = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
            const GuItem w = gu_item<MODE>(p, tfirst, n_used, it);
            const int buf = j & 1, N = (w.n + 15) & ~15;
            if (!mbar_wait(&bars->accfull[buf], (uint32_t)(j >> 1) & 1u)) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * GU_ACC_COLS) + ((uint32_t)(32 * lq) << 16);
            if (MODE == 0) {
                const int f = w.f0 + 16 * lq + (lane & 15);
                for (int c0 = 16 * half; c0 < N; c0 += 32) {
                    float v[16];
                    tmem_ld16(d + (uint32_t)c0, v);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const float up = __shfl_down_sync(0xffffffffu, v[jj], 16);
                        const int col = c0 + jj;
                        if (lane < 16 && col < w.n) {
                            const float g = v[jj];
                            p.act[(size_t)(w.first + w.n0 + col) * F + f] =
                                __float2half_rn(__fdividef(g, 1.f + __expf(-g)) * up);
                        }
                    }
                }
            } else {
                const int yoff = w.e == 0 ? p.seg_yoff[0] : w.e == 1 ? p.seg_yoff[1] : p.seg_yoff[2];
                const int row = yoff + w.f0 + 32 * lq + lane;
                float* yp = p.y + (size_t)w.kh * p.part_stride;
                const float* rp = KS == 1 ? p.res : nullptr;
                for (int c0 = 16 * half; c0 < N; c0 += 32) {
                    float v[16];
                    tmem_ld16(d + (uint32_t)c0, v);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int col = c0 + jj;
                        if (col < w.n) {
                            const size_t o = (size_t)(w.n0 + col) * p.ldy + row;
                            yp[o] = v[jj] + (rp ? rp[o] : 0.f);
                        }
                    }
                }
            }
            // every value of this accumulator is in registers: hand it back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->accempty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, GU_TMEM);
}

struct DnParams {
    const int32_t* n_used;
    const int32_t* used_expert;
    const int32_t* used_first;
    const uint8_t* down;
    float* y;             // [P][H] fp32, rows in pair-list order
    int H, F, down_t;
    const float* dscale;  // FP8 (QF 1): [E][H/128][F/128] block scales; NVFP4 (QF 2): globals [E]
};

// Persistent down GEMM: one CTA per SM walks the items (token tile of DN_NMAX
// rows of a used expert, 128-row tile of H), the row tile fastest.  An item's
// 128 down rows are contiguous in memory (Q6_K rows of F/256 superblocks of
// 210 bytes have no 16-byte aligned superblock columns, so they cannot be
// tiled by TMA): one bulk copy of the whole K per item into one of two raw
// buffers, so the next item's copy runs while this one is dequantised.  A and
// B k-block stages (DN_NA deep) share one full / empty barrier pair each; two
// TMEM accumulators; DN epilogue warps write fp32 y rows.  Warps as in the
// gate/up kernel.
template <int QF>
__global__ void __launch_bounds__(GU_THREADS, 1)
    prefill_down(const __grid_constant__ CUtensorMap tm_a64, const __grid_constant__ CUtensorMap tm_a128,
                 const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ws,
                 const DnParams p) {
    pdl_wait();
    pdl_launch_dependents();
    extern __shared__ __align__(1024) uint8_t smraw[];
    uint8_t* sm = smraw + ((1024u - (smem_u32(smraw) & 1023u)) & 1023u);
    const int H = p.H, F = p.F;
    const int NKB = F / KBLK, NSB = F / QK;
    const int HT = H / TILE_M;
    const int BB = p.down_t == 1 ? Q4K_BYTES : Q6K_BYTES;
    const int RB = (F / QK) * BB;
    // k-quants: one bulk copy of the whole K of 128 rows per item, two raw
    // buffers; FP8 (QF 1): a ring of F8_NQ raw stages of one 128-column scale
    // block each, loaded by TMA (tm_w: [E*H][F] bytes, box 128 x 128)
    const uint32_t qbytes = QF ? 0u : (uint32_t)(TILE_M * RB);
    const uint32_t RQ = QF ? (uint32_t)dn_qring<QF>() / 2u : (qbytes + 1023u) & ~1023u;
    constexpr int DQS = QF == 2 ? QSTAGE_NV : QSTAGE_F8;   // raw stage bytes (QF 1, 2)
    constexpr int DCOLS = QF == 2 ? NV_COLS : F8_COLS;    // columns per raw stage

    uint8_t* qbuf = sm;                                   // 2 x RQ raw bytes
    uint8_t* ast = sm + 2 * RQ;                           // DN_NA x A_STAGE
    uint8_t* bst = ast + DN_NA * A_STAGE;                 // DN_NA x DN_BSTAGE
    PfBars* bars = reinterpret_cast<PfBars*>(bst + DN_NA * DN_BSTAGE);
    int* tfirst = reinterpret_cast<int*>(bars + 1);       // [n_used + 1]
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int n_used = *p.n_used;
    if (tid == 0) {
        for (int i = 0; i < (QF ? F8_NQ : 2); ++i) {
            mbar_init(&bars->qfull[i], 1);
            mbar_init(&bars->qempty[i], NDQ);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->accfull[i], 1);
            mbar_init(&bars->accempty[i], GU_NEPI);
        }
        for (int i = 0; i < DN_NA; ++i) {
            mbar_init(&bars->afull[i], NDQ + 1);          // dequant warps + the B copy
            mbar_init(&bars->aempty[i], 1);
        }
        fence_barrier_init();
    }
    if (warp == W_QLOAD) {
        // token tiles per used expert, exclusive prefix (one warp)
        int carry = 0;
        for (int u0 = 0; u0 < n_used; u0 += 32) {
            const int u = u0 + lane;
            const int t = u < n_used ? (p.used_first[u + 1] - p.used_first[u] + DN_NMAX - 1) / DN_NMAX : 0;
            int incl = t;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            if (u < n_used) tfirst[u] = carry + incl - t;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) tfirst[n_used] = carry;
    }
    if (warp == 0) tmem_alloc(&bars->tmem, DN_TMEM);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem;
    const int n_items = HT * tfirst[n_used];
    // item -> (used expert u, token tile, row tile)
    auto item = [&](int it, int& e, int& first, int& n0, int& n, int& h0) {
        const int tt = it / HT;
        h0 = (it - tt * HT) * TILE_M;
        int lo = 0, hi = n_used - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tfirst[mid] <= tt) lo = mid;
            else hi = mid - 1;
        }
        e = p.used_expert[lo];
        first = p.used_first[lo];
        n0 = (tt - tfirst[lo]) * DN_NMAX;
        n = min(DN_NMAX, p.used_first[lo + 1] - first - n0);
    };

    if (QF != 0 && warp == W_QLOAD) {
        if (lane == 0) {
            int gs = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                int e, first, n0, n, h0;
                item(it, e, first, n0, n, h0);
                for (int sb = 0; sb < F / DCOLS; ++sb, ++gs) {
                    const int st = gs % F8_NQ;
                    if (!mbar_wait(&bars->qempty[st], ((uint32_t)(gs / F8_NQ) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    uint8_t* dst = qbuf + st * DQS;
                    mbar_arrive_expect_tx(&bars->qfull[st], DQS);
                    if (QF == 1) {
                        tma_load_2d(dst, &tm_w, sb * F8_COLS, e * H + h0, &bars->qfull[st]);
                    } else {
                        tma_load_2d(dst, &tm_w, sb * NV_CB, e * H + h0, &bars->qfull[st]);
                        tma_load_2d(dst + TILE_M * NV_CB, &tm_ws, sb * NV_SB, e * H + h0, &bars->qfull[st]);
                    }
                }
            }
        }
    } else if (QF == 0 && warp == W_QLOAD) {
        if (lane == 0) {
            int j = 0;
            for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
                int e, first, n0, n, h0;
                item(it, e, first, n0, n, h0);
                const int rb = j & 1;
                if (!mbar_wait(&bars->qempty[rb], ((uint32_t)(j >> 1) & 1u) ^ 1u)) break;
                mbar_arrive_expect_tx(&bars->qfull[rb], qbytes);
                bulk_g2s(qbuf + rb * RQ, p.down + (size_t)e * H * RB + (size_t)h0 * RB, qbytes, &bars->qfull[rb]);
            }
        }
    } else if (warp == W_BLOAD) {
        if (lane == 0) {
            int gk = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
                int e, first, n0, n, h0;
                item(it, e, first, n0, n, h0);
                const int nb = n <= 64 ? 64 : 128;
                const CUtensorMap* tmb = nb == 64 ? &tm_a64 : &tm_a128;
                for (int kb = 0; kb < NKB; ++kb, ++gk) {
                    const int st = gk % DN_NA;
                    if (!mbar_wait(&bars->aempty[st], ((uint32_t)(gk / DN_NA) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&bars->afull[st], (uint32_t)(nb * KBLK * 2));
                    tma_load_2d(bst + st * DN_BSTAGE, tmb, kb * KBLK, first + n0, &bars->afull[st]);
                }
            }
        }
    } else if (warp == W_MMA) {
        if (lane == 0) {
            int gk = 0, j = 0;
            bool ok = true;
            for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x, ++j) {
                int e, first, n0, n, h0;
                item(it, e, first, n0, n, h0);
                const int buf = j & 1;
                if (!mbar_wait(&bars->accempty[buf], ((uint32_t)(j >> 1) & 1u) ^ 1u)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * DN_NMAX);
                const uint32_t idesc = umma_idesc_f16(TILE_M, (n + 15) & ~15);
                for (int kb = 0; kb < NKB; ++kb, ++gk) {
                    const int sa = gk % DN_NA;
                    if (!mbar_wait(&bars->afull[sa], (uint32_t)(gk / DN_NA) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = umma_sdesc(smem_u32(ast + sa * A_STAGE));
                    const uint64_t bd = umma_sdesc(smem_u32(bst + sa * DN_BSTAGE));
#pragma unroll
                    for (int k = 0; k < KBLK / 16; ++k)
                        umma_f16(d, ad + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), idesc, (kb | k) != 0);
                    umma_commit(&bars->aempty[sa]);
                }
                if (ok) umma_commit(&bars->accfull[buf]);
            }
        }
    } else if (QF == 2 && warp < NDQ) {
        // NVFP4: thread -> A row 8*warp + (lane & 7), 16-k quarter qq = lane >> 3
        // (8 code bytes and one scale byte of each k-block)
        const int qq = lane >> 3, sw = lane & 7;
        const int row = 8 * warp + (lane & 7);
        const int o0 = ((2 * qq) ^ sw) << 4, o1 = ((2 * qq + 1) ^ sw) << 4;
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        int gk = 0, gs = 0;
        bool ok = true;
        for (int j = 0; ok && j < my_items; ++j) {
            int e, first, n0, n, h0;
            item(blockIdx.x + j * gridDim.x, e, first, n0, n, h0);
            const float gsc = __ldg(p.dscale + e);
            for (int sb = 0; sb < F / NV_COLS; ++sb, ++gs) {
                const int sq = gs % F8_NQ;
                const uint8_t* stg = qbuf + sq * QSTAGE_NV;
                if (!mbar_wait(&bars->qfull[sq], (uint32_t)(gs / F8_NQ) & 1u)) {
                    ok = false;
                    break;
                }
                uint2 v[NV_COLS / KBLK];
#pragma unroll
                for (int c = 0; c < NV_COLS / KBLK; ++c)
                    v[c] = *reinterpret_cast<const uint2*>(stg + row * NV_CB + 32 * c + 8 * qq);
                const uint4 scw = *reinterpret_cast<const uint4*>(stg + TILE_M * NV_CB + row * NV_SB);
                const uint32_t sc4[4] = {scw.x, scw.y, scw.z, scw.w};
#pragma unroll
                for (int c = 0; c < NV_COLS / KBLK; ++c, ++gk) {
                    const int sa = gk % DN_NA;
                    const float sc = e4m3_float(sc4[c] >> (8 * qq)) * gsc;
                    if (!mbar_wait(&bars->aempty[sa], ((uint32_t)(gk / DN_NA) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    nv_quarter(v[c], sc, ast + sa * A_STAGE + row * 128, o0, o1);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->afull[sa]);
                }
                if (!ok) break;
                if (lane == 0) mbar_arrive(&bars->qempty[sq]);
            }
        }
    } else if (QF == 1 && warp < NDQ) {
        // FP8: thread -> A row 8*warp + (lane & 7), 16-k quarter qq = lane >> 3
        const int qq = lane >> 3, sw = lane & 7;
        const int row = 8 * warp + (lane & 7);
        const int o0 = ((2 * qq) ^ sw) << 4, o1 = ((2 * qq + 1) ^ sw) << 4;
        const int nbf = F / F8_COLS;
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        int gk = 0, gs = 0;
        bool ok = true;
        for (int j = 0; ok && j < my_items; ++j) {
            int e, first, n0, n, h0;
            item(blockIdx.x + j * gridDim.x, e, first, n0, n, h0);
            const float* srow_scale = p.dscale + ((size_t)e * (H / F8_COLS) + h0 / F8_COLS) * nbf;
            for (int sb = 0; sb < nbf; ++sb, ++gs) {
                const int sq = gs % F8_NQ;
                const uint8_t* stg = qbuf + sq * QSTAGE_F8;
                if (!mbar_wait(&bars->qfull[sq], (uint32_t)(gs / F8_NQ) & 1u)) {
                    ok = false;
                    break;
                }
                uint4 v[F8_COLS / KBLK];
#pragma unroll
                for (int c = 0; c < F8_COLS / KBLK; ++c)
                    v[c] = *reinterpret_cast<const uint4*>(stg + row * F8_COLS + KBLK * c + 16 * qq);
                const float sc = __ldg(srow_scale + sb);
#pragma unroll
                for (int c = 0; c < F8_COLS / KBLK; ++c, ++gk) {
                    const int sa = gk % DN_NA;
                    if (!mbar_wait(&bars->aempty[sa], ((uint32_t)(gk / DN_NA) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    f8_quarter(v[c], sc, ast + sa * A_STAGE + row * 128, o0, o1);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->afull[sa]);
                }
                if (!ok) break;
                if (lane == 0) mbar_arrive(&bars->qempty[sq]);
            }
        }
    } else if (QF == 0 && warp < NDQ) {
        // thread -> A rows 8*warp + (lane & 7) (+ 8*NDQ*r), 16-k quarter
        // qq = lane >> 3 of every k-block; all warps fill each A stage in turn
        const int qq = lane >> 3, sw = lane & 7;                 // row % 8 == lane % 8
        const int my_items = blockIdx.x < n_items ? (n_items - 1 - blockIdx.x) / gridDim.x + 1 : 0;
        int rowo[RPT], rowb[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int row = 8 * warp + (lane & 7) + 8 * NDQ * r;
            rowo[r] = row * RB;
            rowb[r] = row * 128;
        }
        int gk = 0;
        bool ok = true;
        for (int j = 0; ok && j < my_items; ++j) {
            const int rb = j & 1;
            if (!mbar_wait(&bars->qfull[rb], (uint32_t)(j >> 1) & 1u)) break;
            const uint8_t* qb0 = qbuf + rb * RQ;
            for (int sb = 0; ok && sb < NSB; ++sb) {
                if (p.down_t == 2) {
                    // k-block 2n + par of the superblock is half n, groups g = 2 par + h
                    // (h = qq >> 1), positions 16(qq & 1) .. + 15: the same ql / qh
                    // bytes serve par 0 and 1
                    const int h = qq >> 1, hq = qq & 1;
                    const int o0 = ((2 * qq) ^ sw) << 4, o1 = ((2 * qq + 1) ^ sw) << 4;
                    float d[RPT];
                    uint32_t scv[RPT][4];
#pragma unroll
                    for (int r = 0; r < RPT; ++r) {
                        const uint8_t* blk = qb0 + rowo[r] + sb * Q6K_BYTES;
                        d[r] = __half2float(*reinterpret_cast<const __half*>(blk + 208));
                        const uint4 scw = lds16(blk + 192);
                        scv[r][0] = scw.x;
                        scv[r][1] = scw.y;
                        scv[r][2] = scw.z;
                        scv[r][3] = scw.w;
                    }
#pragma unroll
                    for (int n = 0; n < 2; ++n) {
                        uint4 ql[RPT], qh[RPT];
#pragma unroll
                        for (int r = 0; r < RPT; ++r) {
                            const uint8_t* blk = qb0 + rowo[r] + sb * Q6K_BYTES;
                            ql[r] = lds16(blk + 64 * n + 32 * h + 16 * hq);
                            qh[r] = lds16(blk + 128 + 32 * n + 16 * hq);
                        }
#pragma unroll
                        for (int par = 0; par < 2; ++par, ++gk) {
                            const int sa = gk % DN_NA;
                            if (!mbar_wait(&bars->aempty[sa], ((uint32_t)(gk / DN_NA) & 1u) ^ 1u)) {
                                ok = false;
                                break;
                            }
#pragma unroll
                            for (int r = 0; r < RPT; ++r) {
                                // scale byte 8n + 2g + hq = 8n + 4 par + qq: word 2n + par, byte qq
                                const int sc = (int)(scv[r][2 * n + par] << (24 - 8 * qq)) >> 24;
                                q6_quarter(ql[r], qh[r], 4 * par, 4 * par + 2 * h,
                                           __float2half2_rn(d[r] * (float)sc), ast + sa * A_STAGE + rowb[r], o0, o1);
                            }
                            fence_proxy_async();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars->afull[sa]);
                        }
                        if (!ok) break;
                    }
                } else {
                    const int o_lo = (qq ^ sw) << 4, o_hi = ((qq + 4) ^ sw) << 4;
                    Q4Half own[RPT];
#pragma unroll
                    for (int r = 0; r < RPT; ++r)
                        own[r] = q4_half_scales(*reinterpret_cast<const uint4*>(qb0 + rowo[r] + sb * Q4K_BYTES), qq);
#pragma unroll
                    for (int c = 0; c < 4; ++c, ++gk) {
                        const int sa = gk % DN_NA;
                        uint2 v[RPT];
                        Q4Half sc[RPT];
#pragma unroll
                        for (int r = 0; r < RPT; ++r) {
                            v[r] = *reinterpret_cast<const uint2*>(qb0 + rowo[r] + sb * Q4K_BYTES + 16 + 32 * c + 8 * qq);
                            sc[r] = shfl_half(own[r], (lane & 7) + 8 * c);
                        }
                        if (!mbar_wait(&bars->aempty[sa], ((uint32_t)(gk / DN_NA) & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int r = 0; r < RPT; ++r) q4_quarter(v[r], sc[r], ast + sa * A_STAGE + rowb[r], o_lo, o_hi);
                        fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->afull[sa]);
                    }
                }
            }
            // every value read from this raw buffer has fed a store above
            if (ok && lane == 0) mbar_arrive(&bars->qempty[rb]);
        }
    } else if (warp >= W_EPI) {
        const int lq = warp & 3, half = (warp - W_EPI) >> 2;
        int j = 0;
        for (int it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
            int e, first, n0, n, h0;
            item(it, e, first, n0, n, h0);
            const int buf = j & 1, N = (n + 15) & ~15;
            if (!mbar_wait(&bars->accfull[buf], (uint32_t)(j >> 1) & 1u)) break;
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(buf * DN_NMAX) + ((uint32_t)(32 * lq) << 16);
            const int hrow = h0 + 32 * lq + lane;
            for (int c0 = 16 * half; c0 < N; c0 += 32) {
                float v[16];
                tmem_ld16(d + (uint32_t)c0, v);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const int col = c0 + jj;
                    if (col < n) p.y[(size_t)(first + n0 + col) * H + hrow] = v[jj];
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->accempty[buf]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, DN_TMEM);
}

// x rows of every pair, in pair-list order, as fp16; inverse pair -> position map
__global__ void gather_x_f16(const float* __restrict__ x, const int32_t* __restrict__ pair_list,
                             int K, int H, __half* __restrict__ xp, int32_t* __restrict__ inv_pos) {
    pdl_wait();
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
// (four consecutive h per thread; every element is read and written by the
// same thread, so out may alias res)
__global__ void combine_pairs(const float* __restrict__ y, const int32_t* __restrict__ inv_pos,
                              const float* __restrict__ wts, const float* res, int H, int K,
                              float* out) {
    pdl_wait();
    const int t = blockIdx.y;
    const int h4 = blockIdx.x * blockDim.x + threadIdx.x;
    if (4 * h4 >= H) return;
    const int H4 = H / 4;
    float4 acc = reinterpret_cast<const float4*>(res)[(size_t)t * H4 + h4];
    for (int j = 0; j < K; ++j) {
        const float w = wts[t * K + j];
        const float4 v = reinterpret_cast<const float4*>(y)[(size_t)inv_pos[t * K + j] * H4 + h4];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    reinterpret_cast<float4*>(out)[(size_t)t * H4 + h4] = acc;
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


constexpr size_t GU_SMEM = 1024 + ((GU_NQ * QSTAGE_GU + 1023) & ~1023) + GU_NA * A_STAGE + B_BYTES_GU +
                           sizeof(PfBars) + sizeof(int) * 1025 + 64;   // + tfirst[E + 1]

// SMs of the current device: the persistent gate/up grid
int sm_count() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            n = 1;
    }
    return n;
}

size_t dn_smem(int F, int down_t, int E) {
    const size_t rb = (size_t)(F / QK) * (down_t == 1 ? Q4K_BYTES : Q6K_BYTES);
    const size_t q = down_t == 3   ? (size_t)dn_qring<1>() / 2
                     : down_t == 4 ? (size_t)dn_qring<2>() / 2
                                   : (TILE_M * rb + 1023) & ~size_t(1023);
    return 1024 + 2 * q + DN_NA * A_STAGE + DN_NA * DN_BSTAGE + sizeof(PfBars) + sizeof(int) * (E + 1) + 64;
}

// the attribute raising the dynamic shared-memory limit of every prefill GEMM
// instantiation, once per process
cudaError_t prefill_attrs() {
    static cudaError_t e = [] {
        cudaError_t r = cudaFuncSetAttribute(prefill_gateup<0, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_gateup<1, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_gateup<0, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_down<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_gateup<0, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_down<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(prefill_down<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        return r;
    }();
    return e;
}

}  // namespace

bool tensor_map_half(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    return map_half(m, base, cols, rows, box_rows);
}

bool prefill_supported(const MoeShape& s, int gate_t, int up_t, int down_t) {
    if (gate_t != 1 || up_t != 1) return false;
    if (s.H % QK || s.F % QK || s.H % TILE_M || s.F % 64) return false;
    return dn_smem(s.F, down_t, s.E) <= 227 * 1024 && GU_SMEM <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_prefill(const MoeShape& s, const float* x, const float* res,
                           const uint8_t* gate, const uint8_t* up, const uint8_t* down, int down_t,
                           const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                           float* out, cudaStream_t st) {
    const int P = s.T * s.K;
    cudaError_t e = launch_pdl(gather_x_f16, dim3(P), dim3(128), 0, st, x, r.pair_list, s.K, s.H, xp, inv_pos);
    if (e != cudaSuccess) return e;

    CUtensorMap tg, tu, tx64, tx128, txg, ta64, ta128;
    const uint64_t rbg = (uint64_t)(s.H / QK) * Q4K_BYTES;
    // B maps: boxes of 64 / 128 / 256 token rows
    if (!map_bytes(&tg, gate, rbg, (uint64_t)s.E * s.F, Q4K_BYTES, 64) ||
        !map_bytes(&tu, up, rbg, (uint64_t)s.E * s.F, Q4K_BYTES, 64) ||
        !map_half(&tx64, xp, s.H, P, 64) || !map_half(&tx128, xp, s.H, P, 128) ||
        !map_half(&txg, xp, s.H, P, GU_NMAX) || !map_half(&ta64, actp, s.F, P, 64) ||
        !map_half(&ta128, actp, s.F, P, 128))
        return cudaErrorInvalidValue;

    e = prefill_attrs();
    if (e != cudaSuccess) return e;
    GuParams gp{r.n_used, r.used_expert, r.used_first, actp, s.H, s.F, nullptr, nullptr, 0, 0,
                {0, 0, 0}, {0, 0, 0}, 1, 0, nullptr, nullptr};
    e = launch_pdl(prefill_gateup<0, 0>, dim3(sm_count()), dim3(GU_THREADS), GU_SMEM, st, tg, tu, tu, tx64,
                   tx128, txg, tg, tg, gp);
    if (e != cudaSuccess) return e;
    DnParams dp{r.n_used, r.used_expert, r.used_first, down, y, s.H, s.F, down_t, nullptr};
    e = launch_pdl(prefill_down<0>, dim3(sm_count()), dim3(GU_THREADS), dn_smem(s.F, down_t, s.E), st, ta64,
                   ta128, ta64, ta64, dp);
    if (e != cudaSuccess) return e;
    dim3 g3((s.H / 4 + 255) / 256, s.T);
    return launch_pdl(combine_pairs, g3, dim3(256), 0, st, y, inv_pos, r.wts, res, s.H, s.K, out);
}

bool prefill_fp8_supported(const MoeShape& s) {
    if (s.H % F8_COLS || s.F % F8_COLS || s.H % TILE_M || s.F % 64) return false;
    return dn_smem(s.F, 3, s.E) <= 227 * 1024 && GU_SMEM <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_prefill_fp8(const MoeShape& s, const float* x, const float* res, const Fp8Experts& w,
                               const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                               float* out, cudaStream_t st) {
    const int P = s.T * s.K;
    cudaError_t e = launch_pdl(gather_x_f16, dim3(P), dim3(128), 0, st, x, r.pair_list, s.K, s.H, xp, inv_pos);
    if (e != cudaSuccess) return e;
    CUtensorMap tg, tu, td, tx64, tx128, txg, ta64, ta128;
    if (!map_bytes(&tg, w.gate, (uint64_t)s.H, (uint64_t)s.E * s.F, F8_COLS, 64) ||
        !map_bytes(&tu, w.up, (uint64_t)s.H, (uint64_t)s.E * s.F, F8_COLS, 64) ||
        !map_bytes(&td, w.down, (uint64_t)s.F, (uint64_t)s.E * s.H, F8_COLS, TILE_M) ||
        !map_half(&tx64, xp, s.H, P, 64) || !map_half(&tx128, xp, s.H, P, 128) ||
        !map_half(&txg, xp, s.H, P, GU_NMAX) || !map_half(&ta64, actp, s.F, P, 64) ||
        !map_half(&ta128, actp, s.F, P, 128))
        return cudaErrorInvalidValue;
    e = prefill_attrs();
    if (e != cudaSuccess) return e;
    GuParams gp{r.n_used, r.used_expert, r.used_first, actp, s.H, s.F, nullptr, nullptr, 0, 0,
                {0, 0, 0}, {0, 0, 0}, 1, 0, w.gate_scale, w.up_scale};
    e = launch_pdl(prefill_gateup<0, 1>, dim3(sm_count()), dim3(GU_THREADS), GU_SMEM, st, tg, tu, tu, tx64,
                   tx128, txg, tg, tg, gp);
    if (e != cudaSuccess) return e;
    DnParams dp{r.n_used, r.used_expert, r.used_first, w.down, y, s.H, s.F, 3, w.down_scale};
    e = launch_pdl(prefill_down<1>, dim3(sm_count()), dim3(GU_THREADS), dn_smem(s.F, 3, s.E), st, ta64, ta128,
                   td, td, dp);
    if (e != cudaSuccess) return e;
    dim3 g3((s.H / 4 + 255) / 256, s.T);
    return launch_pdl(combine_pairs, g3, dim3(256), 0, st, y, inv_pos, r.wts, res, s.H, s.K, out);
}

bool prefill_nvfp4_supported(const MoeShape& s) {
    if (s.H % NV_COLS || s.F % NV_COLS || s.H % TILE_M || s.F % 64) return false;
    return dn_smem(s.F, 4, s.E) <= 227 * 1024 && GU_SMEM <= 227 * 1024 && encode_fn() != nullptr;
}

cudaError_t launch_prefill_nvfp4(const MoeShape& s, const float* x, const float* res, const NvExperts& w,
                                 const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                                 float* out, cudaStream_t st) {
    const int P = s.T * s.K;
    cudaError_t e = launch_pdl(gather_x_f16, dim3(P), dim3(128), 0, st, x, r.pair_list, s.K, s.H, xp, inv_pos);
    if (e != cudaSuccess) return e;
    CUtensorMap tg, tu, tgs, tus, td, tds, tx64, tx128, txg, ta64, ta128;
    const uint64_t gu_rows = (uint64_t)s.E * s.F, dn_rows = (uint64_t)s.E * s.H;
    if (!map_bytes(&tg, w.gate, (uint64_t)s.H / 2, gu_rows, NV_CB, 64) ||
        !map_bytes(&tu, w.up, (uint64_t)s.H / 2, gu_rows, NV_CB, 64) ||
        !map_bytes(&tgs, w.gate_bs, (uint64_t)s.H / 16, gu_rows, NV_SB, 64) ||
        !map_bytes(&tus, w.up_bs, (uint64_t)s.H / 16, gu_rows, NV_SB, 64) ||
        !map_bytes(&td, w.down, (uint64_t)s.F / 2, dn_rows, NV_CB, TILE_M) ||
        !map_bytes(&tds, w.down_bs, (uint64_t)s.F / 16, dn_rows, NV_SB, TILE_M) ||
        !map_half(&tx64, xp, s.H, P, 64) || !map_half(&tx128, xp, s.H, P, 128) ||
        !map_half(&txg, xp, s.H, P, GU_NMAX) || !map_half(&ta64, actp, s.F, P, 64) ||
        !map_half(&ta128, actp, s.F, P, 128))
        return cudaErrorInvalidValue;
    e = prefill_attrs();
    if (e != cudaSuccess) return e;
    GuParams gp{r.n_used, r.used_expert, r.used_first, actp, s.H, s.F, nullptr, nullptr, 0, 0,
                {0, 0, 0}, {0, 0, 0}, 1, 0, w.gate_gs, w.up_gs};
    e = launch_pdl(prefill_gateup<0, 2>, dim3(sm_count()), dim3(GU_THREADS), GU_SMEM, st, tg, tu, tu, tx64,
                   tx128, txg, tgs, tus, gp);
    if (e != cudaSuccess) return e;
    DnParams dp{r.n_used, r.used_expert, r.used_first, w.down, y, s.H, s.F, 4, w.down_gs};
    e = launch_pdl(prefill_down<2>, dim3(sm_count()), dim3(GU_THREADS), dn_smem(s.F, 4, s.E), st, ta64, ta128,
                   td, tds, dp);
    if (e != cudaSuccess) return e;
    dim3 g3((s.H / 4 + 255) / 256, s.T);
    return launch_pdl(combine_pairs, g3, dim3(256), 0, st, y, inv_pos, r.wts, res, s.H, s.K, out);
}

cudaError_t launch_dense_q4k_gemm_multi(const DenseSeg* seg, int nseg, int K, const __half* x, int T,
                                        float* y, int ldy, const float* res, int ksplit, size_t part_stride,
                                        cudaStream_t st) {
    if (nseg < 1 || nseg > 3 || K % QK || T < 1 || (ksplit != 1 && ksplit != 2) || (K / QK) % ksplit)
        return cudaErrorInvalidValue;
    CUtensorMap tw[3], tx64, tx128, txg;
    const uint64_t rb = (uint64_t)(K / QK) * Q4K_BYTES;
    int rows = 0;
    for (int i = 0; i < nseg; ++i) {
        if (seg[i].rows % TILE_M || !map_bytes(&tw[i], seg[i].W, rb, (uint64_t)seg[i].rows, Q4K_BYTES, 64))
            return cudaErrorInvalidValue;
        rows += seg[i].rows;
    }
    for (int i = nseg; i < 3; ++i) tw[i] = tw[0];
    if (!map_half(&tx64, x, K, T, 64) || !map_half(&tx128, x, K, T, 128) || !map_half(&txg, x, K, T, GU_NMAX))
        return cudaErrorInvalidValue;
    {
        const cudaError_t e = prefill_attrs();
        if (e != cudaSuccess) return e;
    }
    GuParams gp{nullptr, nullptr, nullptr, nullptr, K, rows, y, res, T, ldy,
                {nseg > 0 ? seg[0].rows : 0, nseg > 1 ? seg[1].rows : 0, nseg > 2 ? seg[2].rows : 0},
                {nseg > 0 ? seg[0].yoff : 0, nseg > 1 ? seg[1].yoff : 0, nseg > 2 ? seg[2].yoff : 0},
                ksplit, part_stride, nullptr, nullptr};
    const int items = (rows / TILE_M) * ksplit * ((T + GU_NMAX - 1) / GU_NMAX);
    const int grid = items < sm_count() ? items : sm_count();
    return launch_pdl(prefill_gateup<1, 0>, dim3(grid), dim3(GU_THREADS), GU_SMEM, st, tw[0], tw[1], tw[2],
                      tx64, tx128, txg, tw[0], tw[0], gp);
}

cudaError_t launch_dense_q4k_gemm(const uint8_t* W, int rows, int K, const __half* x, int T, float* y,
                                  int ldy, int yoff, const float* res, cudaStream_t st) {
    const DenseSeg seg{W, rows, yoff};
    return launch_dense_q4k_gemm_multi(&seg, 1, K, x, T, y, ldy, res, 1, 0, st);
}

int dense_q4k_items(int rows, int T) { return (rows / TILE_M) * ((T + GU_NMAX - 1) / GU_NMAX); }

int device_sm_count() { return sm_count(); }

}  // namespace qmoe
