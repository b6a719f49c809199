// qmoe_internal.h -- launchers shared between the C-ABI layer and the kernels.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qmoe {

// Routing results of one layer call, all in the context workspace (device).
// Pairs p = t*K + j (token t, slot j).  The per-expert pair lists group the
// pairs of each used expert, experts in ascending id order, pairs in ascending
// p inside an expert: pair_list[used_first[u] .. used_first[u+1]) belong to
// expert used_expert[u], for u < *n_used.
struct Route {
    float* logits;        // [T][E]
    int32_t* ids;         // [T*K]
    float* wts;           // [T*K]
    int32_t* n_used;      // [1]
    int32_t* used_expert; // [E]
    int32_t* used_first;  // [E+1]
    int32_t* pair_list;   // [T*K]
    float* logits_part;   // [H/128][T][E] split-k router partials (many-token path), or null
    uint32_t* tokmap;     // [E][ceil(T/32)] token bitmap per expert, then [E] pair counts
                          // (many-token path), or null
    uint8_t* jmap;        // [E][T] slot j of pair (t, e) where e's bitmap has t (many-token path)
    unsigned* arrive;     // [1] arrival counter of the one-launch routing (zero between launches), or null
};

struct MoeShape {
    int T, H, E, K, F;
    int norm_topk;
};

// A1 + A2 + A3: router logits, softmax / top-k / renorm, per-expert pair lists.
cudaError_t launch_route(const MoeShape& s, const float* x, const float* router_w,
                         const float* bias, const Route& r, cudaStream_t st);

// The same for many tokens (tiled router GEMM, per-token rank top-k, per-expert
// lists from token bitmaps); requires route_many_supported().
cudaError_t launch_route_many(const MoeShape& s, const float* x, const float* router_w,
                              const float* bias, const Route& r, cudaStream_t st);
bool route_many_supported(const MoeShape& s, const Route& r);
size_t route_many_part_floats(int T, int H, int E);
size_t route_many_tokmap_words(int T, int E);
cudaError_t route_prepare();

// A4 + A5: act[p][f] = silu(Wg_e x_t)[f] * (Wu_e x_t)[f] for every pair p.
cudaError_t launch_gateup(const MoeShape& s, const float* x, const uint8_t* gate, int gate_t,
                          const uint8_t* up, int up_t, const Route& r, float* act,
                          cudaStream_t st);

// A6: y[p][h] = (Wd_e act_p)[h] for every pair p.
cudaError_t launch_down(const MoeShape& s, const float* act, const uint8_t* down, int down_t,
                        const Route& r, float* y, cudaStream_t st);

// A7: out[t][h] = res[t][h] + sum_j wts[t][j] * y[t*K+j][h].
cudaError_t launch_combine(const MoeShape& s, const float* y, const Route& r, const float* res,
                           float* out, cudaStream_t st);

// Copy the routing results out (ids int32, weights f32), async.
// The MoE FFN with 8-bit (Q8_K) activations in every expert GEMV (moe_q8k.cu):
// the codes, scales and 16-value code sums of x (per token) and of act (per pair).
struct Q8Bufs {
    int8_t* qx;
    float* dx;
    int16_t* bx;
    int8_t* qa;
    float* da;
    int16_t* ba;
};
size_t q8_bufs_bytes(int T, int H, int K, int F);
Q8Bufs q8_bufs_carve(unsigned char* base, int T, int H, int K, int F);
// after launch_route: quantise x, gate/up + SwiGLU into act, quantise act, down
// into y, combine into out (= res + sum_j w_j y_j)
cudaError_t launch_moe_q8k(const MoeShape& s, const float* x, const float* res, const uint8_t* gate,
                           int gate_t, const uint8_t* up, int up_t, const uint8_t* down, int down_t,
                           const Route& r, const Q8Bufs& b, float* act, float* y, float* out,
                           cudaStream_t st);

cudaError_t copy_route_out(const MoeShape& s, const Route& r, int32_t* ids_out, float* w_out,
                           cudaStream_t st);

// FP8 block-scaled experts (moe_fp8.cu): E4M3 codes [E][rows][cols] and one fp32
// scale per 128 x 128 block [E][rows/128][cols/128]; gate/up [F][H], down [H][F].
struct Fp8Experts {
    const uint8_t* gate;
    const float* gate_scale;
    const uint8_t* up;
    const float* up_scale;
    const uint8_t* down;
    const float* down_scale;
};
bool fp8_supported(int H, int F);
// after launch_route / launch_route_many: gate/up + SwiGLU into act [P][F], down
// into y [P][H] (launch_combine finishes the layer)
cudaError_t launch_fp8_experts(const MoeShape& s, const float* x, const Fp8Experts& w,
                               const Route& r, float* act, float* y, int num_sms, cudaStream_t st);
// NVFP4 experts (moe_nvfp4.cu): E2M1 codes [E][rows][cols/2] (even element in
// the low nibble), E4M3 block scales [E][rows][cols/16], fp32 globals [E].
struct NvExperts {
    const uint8_t* gate;
    const uint8_t* gate_bs;
    const float* gate_gs;
    const uint8_t* up;
    const uint8_t* up_bs;
    const float* up_gs;
    const uint8_t* down;
    const uint8_t* down_bs;
    const float* down_gs;
};
bool nvfp4_supported(int H, int F);
cudaError_t launch_nvfp4_experts(const MoeShape& s, const float* x, const NvExperts& w,
                                 const Route& r, float* act, float* y, int num_sms, cudaStream_t st);
// One token over FP8 (fmt 1) or NVFP4 (fmt 2) experts: the whole layer in one
// launch of one CTA per SM, a programmatic dependent of the previous kernel
// (moe_lowbit_t1.cu); lg: E tagged words, ctl: 4 words, both zero at creation
// and owned by this kernel
bool lowbit_t1_supported(int fmt, int T, int H, int E, int K, int F, int num_sms);
cudaError_t launch_lowbit_t1(int fmt, const MoeShape& s, const float* x, const float* router_w,
                             const Fp8Experts* f8, const NvExperts* nv, float* act, float* out,
                             int32_t* ids_out, float* w_out, unsigned long long* lg, unsigned* ctl,
                             int* status, int num_sms, cudaStream_t st);
// BF16 -> NVFP4 of n_mats matrices [rows][cols] (consecutive); amax_bits: n_mats
// words of scratch
cudaError_t launch_nvfp4_quantize(const uint16_t* x, int n_mats, int rows, int cols, uint8_t* codes,
                                  uint8_t* bscale, float* global, unsigned* amax_bits, int num_sms,
                                  cudaStream_t st);
// many tokens over NVFP4 experts: as launch_prefill_fp8 (E2M1 widened and
// scaled by block and global scale to fp16 in shared memory)
bool prefill_nvfp4_supported(const MoeShape& s);
cudaError_t launch_prefill_nvfp4(const MoeShape& s, const float* x, const float* res, const NvExperts& w,
                                 const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                                 float* out, cudaStream_t st);
// many tokens (after launch_route_many): gather x as fp16, grouped gate/up and
// down GEMMs on the tensor cores with the FP8 weights widened to fp16 in shared
// memory, combine into out (prefill_umma.cu)
bool prefill_fp8_supported(const MoeShape& s);
cudaError_t launch_prefill_fp8(const MoeShape& s, const float* x, const float* res, const Fp8Experts& w,
                               const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                               float* out, cudaStream_t st);

size_t row_bytes(int qtype, int cols);

// Fused single-kernel decode path (T <= 8): launch plan chosen once per shape.
struct FusedPlan {
    int grid;          // CTAs (one per SM, cooperative)
    int smem;          // dynamic shared memory bytes
    const void* fn;    // kernel variant
    int slot_bytes;    // ring slot size
    int cf;            // f rows per gate/up chunk
    int ns;            // ring slots per warp
    int nloc_max;      // pairs of the experts one CTA's down rows can touch
};

// Values passed between the CTAs of the fused kernel, each tagged with its
// launch (zero-initialised once; never shared with other kernels).
struct FusedBufs {
    unsigned long long* lg;     // [T][E] router logits
    unsigned long long* act;    // [T*K][F] silu(gate)*up
    unsigned long long* y;      // [T*K][H] down outputs
    unsigned long long* xflag;  // [grid] "x staged" marks
    float* plain_act;           // [K][F] batch-1 kernel's SwiGLU output (plain fp32)
    unsigned* ctl;              // [0] exit counter, [1] tag of the last launch,
                                // [3] batch-1 kernel's act arrival count
    int* status;
};
size_t fused_bufs_bytes(int T, int H, int E, int K, int F, int grid);
FusedBufs fused_bufs_carve(unsigned char* base, int T, int H, int E, int K, int F, int grid,
                           unsigned* ctl, int* status);

bool fused_decode_plan(const MoeShape& s, int gate_t, int up_t, int down_t, int num_sms,
                       FusedPlan* plan);

// Test hook of the bounded waits: a launch with stall = 1 waits for router
// logits carrying a tag that no CTA writes, for wait_ns, then records
// QMOE_ERR_TIMEOUT and exits without computing (null: the normal 200 ms limit).
struct FusedDebug {
    unsigned long long wait_ns;
    int stall;
};

cudaError_t launch_fused_decode(const MoeShape& s, const FusedPlan& plan, const float* x,
                                const float* res, const float* bias, const float* router,
                                const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                                float* out, int32_t* ids_out, float* w_out, const FusedBufs& b,
                                const float* norm_w, float eps, cudaStream_t st,
                                const FusedDebug* dbg = nullptr);

int fused_threads();
cudaError_t fused_prepare();

// Batch-1 decode kernel (moe_decode_t1.cu): one token, every weight copy of a
// CTA issued at once, output rows owned by CTAs (no partial sums cross CTAs),
// launched as a programmatic dependent of the previous kernel.  Uses the lg
// and act buffers and the control words of FusedBufs.
struct T1Plan {
    int grid;
    int smem;
    const void* fn;
};
bool t1_decode_plan(const MoeShape& s, int gate_t, int up_t, int down_t, int num_sms, T1Plan* plan);
cudaError_t launch_t1_decode(const MoeShape& s, const T1Plan& plan, int down_t, const float* x,
                             const float* res, const float* bias, const float* router,
                             const uint8_t* gate, const uint8_t* up, const uint8_t* down, float* out,
                             int32_t* ids_out, float* w_out, const FusedBufs& b, const float* norm_w,
                             float eps, cudaStream_t st, const FusedDebug* dbg = nullptr);
cudaError_t t1_prepare();

// Attention half of a decoder layer at decode time (batch 1).
struct AttnShape {
    int H, nq, nkv, hd, max_ctx, pos;
    float eps, rope_base;
    const double* inv_freq;   // [hd/2] rope_base^(-2j/hd), device
    const float2* rope_cs;    // [hd/2] cos/sin of the angles at pos (launch_rope_table)
};
struct LayerAttn {
    const float* attn_norm;
    const uint8_t* wq;
    const uint8_t* wk;
    const uint8_t* wv;
    const uint8_t* wo;
    const float* q_norm;
    const float* k_norm;
    __half* k_cache;
    __half* v_cache;
};
// h_out = h + Wo attn(RoPE(norm(Wq x)), cache), x = RMSNorm(h); writes slot pos
cudaError_t launch_attention_block(const AttnShape& a, const LayerAttn& L, const float* h,
                                   float* xs, float* q, float* kv, float* att, float* part,
                                   float* h_out, cudaStream_t st);
cudaError_t launch_rmsnorm(const float* h, const float* w, float eps, int n, float* out,
                           cudaStream_t st);
int attn_splits(int max_ctx);
cudaError_t decode_step_prepare();
cudaError_t launch_rope_table(const double* inv_freq, int hd, int pos, float2* cs,
                              cudaStream_t st);
bool attention_supported(int nq, int nkv, int hd);

// Prefill path (T > 8): tcgen05 grouped GEMMs with on-the-fly dequantisation.
bool prefill_supported(const MoeShape& s, int gate_t, int up_t, int down_t);
cudaError_t launch_prefill(const MoeShape& s, const float* x, const float* res,
                           const uint8_t* gate, const uint8_t* up, const uint8_t* down, int down_t,
                           const Route& r, __half* xp, __half* actp, float* y, int32_t* inv_pos,
                           float* out, cudaStream_t st);

// A dense Q4_K GEMM on the tensor cores (prefill_umma.cu):
// y[t][yoff + r] = sum_k W[r][k] x[t][k] (+ res[t][yoff + r]) for t < T,
// W [rows][K] Q4_K rows (rows % 128 == 0, K % 256 == 0), x fp16 [T][K], y / res
// fp32 with row pitch ldy.  res may equal y (in place).
cudaError_t launch_dense_q4k_gemm(const uint8_t* W, int rows, int K, const __half* x, int T, float* y,
                                  int ldy, int yoff, const float* res, cudaStream_t st);
// Up to three such GEMMs over the same x in one launch (segment i: W, rows,
// output column offset yoff).  ksplit 2: each half of K writes its own plane
// y + kh * part_stride with no residual (the caller adds the two planes).
struct DenseSeg {
    const uint8_t* W;
    int rows, yoff;
};
cudaError_t launch_dense_q4k_gemm_multi(const DenseSeg* seg, int nseg, int K, const __half* x, int T,
                                        float* y, int ldy, const float* res, int ksplit, size_t part_stride,
                                        cudaStream_t st);
int dense_q4k_items(int rows, int T);   // work items of one dense GEMM of `rows` rows
int device_sm_count();

// Batched prefill of one decoder layer (prefill_layer.cu): everything up to
// the MoE input.  hidden [T][H] fp32 is updated in place to h + Wo attn, the
// KV cache slots pos0 .. pos0+T-1 are written, and the MoE input
// x2 = RMSNorm(h) * ffn_norm is left in the scratch (prefill_layer_x2).
struct PrefillLayerArgs {
    int T, H, nq, nkv, hd, max_ctx, pos0;
    float eps;
    const double* inv_freq;
    const float* attn_norm;
    const uint8_t* wq;
    const uint8_t* wk;
    const uint8_t* wv;
    const uint8_t* wo;
    const float* q_norm;
    const float* k_norm;
    const float* ffn_norm;
    __half* k_cache;
    __half* v_cache;
    float* hidden;
    void* scratch;            // prefill_layer_scratch_bytes(T, ...)
    int* status;              // device status word (a bounded wait that ran out)
};
size_t prefill_layer_scratch_bytes(int T, int H, int nq, int nkv, int hd);
bool prefill_layer_supported(int H, int nq, int nkv, int hd);
cudaError_t prefill_layer_prepare();
cudaError_t launch_prefill_layer_attn(const PrefillLayerArgs& a, cudaStream_t st);
float* prefill_layer_x2(void* scratch, int T, int H, int nq, int nkv, int hd);

}  // namespace qmoe
