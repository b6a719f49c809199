// qmoe_noalloc.cu -- qmoe_forward_noalloc: the decode-size MoE-FFN layer for
// callers that cannot allocate device memory.
//
// Some callers own every byte of device memory through their own pool (a host
// framework whose allocator must not be bypassed, a plugin loaded into such a
// process), or run latency-critical loops in which a cudaMalloc, with its
// implicit device synchronisation, is not acceptable after start-up.  For them
// this entry point needs no context and performs no allocation: the scratch of
// the fused decode kernel (the tagged router logits, SwiGLU activations and
// down outputs it passes between CTAs, its two control words and the device
// status word) lives in one file-scope device array of fixed size, which every
// GPU that loads this library keeps until the process exits.  The array starts
// zeroed with the module and the control words carry over from call to call
// (they count launches), so only the status word is cleared per call.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/qmoe.h"
#include "qmoe_internal.h"

namespace {

// Capacity of the shared scratch (bytes).
constexpr size_t NA_HEAD = 256;               // control words at 0, status word at 128
constexpr size_t NA_TAGGED = 2u << 20;        // tagged logits, act, down outputs, marks
constexpr size_t NA_BYTES = NA_HEAD + NA_TAGGED;

constexpr int NA_MAX_DEVICES = 64;

struct DeviceSetup {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_qmoe_noalloc_scratch
    int num_sms = 0;
};

DeviceSetup g_setup[NA_MAX_DEVICES];
std::mutex g_setup_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// The scratch itself.  In host code this name is only a stand-in for the
// symbol, never a device address: the address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_qmoe_noalloc_scratch[NA_BYTES];

extern "C" qmoe_status qmoe_forward_noalloc(const float* hidden_in, const float* router_w,
                                            const void* gate_exps, const void* up_exps,
                                            const void* down_exps, qmoe_qtype gate_t,
                                            qmoe_qtype up_t, qmoe_qtype down_t, int hidden,
                                            int n_experts, int top_k, int ffn,
                                            int norm_topk_prob, int n_tokens,
                                            float* hidden_out, void* stream) {
    if (!hidden_in || !router_w || !gate_exps || !up_exps || !down_exps || !hidden_out)
        return QMOE_ERR_INVALID_ARG;
    if (hidden <= 0 || hidden % 256 || ffn <= 0 || ffn % 256 || n_experts < 1 ||
        n_experts > 1024 || top_k < 1 || top_k > 16 || top_k > n_experts || n_tokens < 1)
        return QMOE_ERR_SHAPE;
    if ((gate_t != QMOE_Q4_K && gate_t != QMOE_Q6_K) || (up_t != QMOE_Q4_K && up_t != QMOE_Q6_K) ||
        (down_t != QMOE_Q4_K && down_t != QMOE_Q6_K))
        return QMOE_ERR_UNSUPPORTED_QTYPE;
    if (!aligned16(hidden_in) || !aligned16(router_w) || !aligned16(gate_exps) ||
        !aligned16(up_exps) || !aligned16(down_exps) || !aligned16(hidden_out))
        return QMOE_ERR_MISALIGNED;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES)
        return QMOE_ERR_CUDA;
    DeviceSetup* su = &g_setup[dev];
    {
        // first call on this device: look up the scratch's device address and
        // prepare the kernel (no allocation happens here either)
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!su->ready) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_qmoe_noalloc_scratch) != cudaSuccess)
                return QMOE_ERR_CUDA;
            if (qmoe::fused_prepare() != cudaSuccess || qmoe::t1_prepare() != cudaSuccess)
                return QMOE_ERR_CUDA;
            int sms = 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
                return QMOE_ERR_CUDA;
            su->scratch = static_cast<unsigned char*>(ptr);
            su->num_sms = sms;
            su->ready = true;
        }
    }

    qmoe::MoeShape s{n_tokens, hidden, n_experts, top_k, ffn, norm_topk_prob ? 1 : 0};
    qmoe::FusedPlan plan;
    qmoe::T1Plan p1;
    const bool t1 = qmoe::t1_decode_plan(s, gate_t, up_t, down_t, su->num_sms, &p1);
    if (!t1 && !qmoe::fused_decode_plan(s, gate_t, up_t, down_t, su->num_sms, &plan))
        return QMOE_ERR_SHAPE;                 // only the single-kernel decode shapes are served
    const int grid = t1 ? p1.grid : plan.grid;
    // capacity of the shared scratch
    if (qmoe::fused_bufs_bytes(n_tokens, hidden, n_experts, top_k, ffn, grid) > NA_TAGGED)
        return QMOE_ERR_SHAPE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned* ctl = reinterpret_cast<unsigned*>(su->scratch);
    int* status = reinterpret_cast<int*>(su->scratch + 128);
    const qmoe::FusedBufs fb = qmoe::fused_bufs_carve(su->scratch + NA_HEAD, n_tokens, hidden,
                                                      n_experts, top_k, ffn, grid, ctl, status);
    // the status word reports this call only
    if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return QMOE_ERR_CUDA;
    cudaError_t e =
        t1 ? qmoe::launch_t1_decode(s, p1, down_t, hidden_in, nullptr, nullptr, router_w,
                                    static_cast<const uint8_t*>(gate_exps),
                                    static_cast<const uint8_t*>(up_exps),
                                    static_cast<const uint8_t*>(down_exps), hidden_out, nullptr,
                                    nullptr, fb, nullptr, 0.f, st)
           : qmoe::launch_fused_decode(s, plan, hidden_in, nullptr, nullptr, router_w,
                                       static_cast<const uint8_t*>(gate_exps),
                                       static_cast<const uint8_t*>(up_exps),
                                       static_cast<const uint8_t*>(down_exps), hidden_out, nullptr,
                                       nullptr, fb, nullptr, 0.f, st);
    return e == cudaSuccess ? QMOE_OK : QMOE_ERR_CUDA;
}

extern "C" qmoe_status qmoe_noalloc_status(void* stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NA_MAX_DEVICES)
        return QMOE_ERR_CUDA;
    unsigned char* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mu);
        if (!g_setup[dev].ready) return QMOE_ERR_CUDA;
        scratch = g_setup[dev].scratch;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return QMOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, scratch + 128, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return QMOE_ERR_CUDA;
    if (v != 0 && cudaMemset(scratch + 128, 0, sizeof(int)) != cudaSuccess) return QMOE_ERR_CUDA;
    return static_cast<qmoe_status>(v);
}
