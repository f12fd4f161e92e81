// beam_moe_route_noalloc (include/beam_moe.h): the router of the MoE block with no
// device allocation at all.
//
// Why it exists: the regular entry points take their scratch memory from a stream-ordered
// pool, which can grow through the driver allocator. Some callers cannot let a library do
// that: a serving engine that has already claimed all free HBM for its weights and KV
// cache (an allocation would fail), or a runtime that allows no allocator call on its
// per-token path, where a new allocation may synchronise the device or add unbounded
// latency. This entry point gives them the router with its scratch (the BF16 pieces of
// the router weights and the split-K partial logits) in a fixed array that is part of the
// library's device image.
//
// The array: BEAM_MOE_NOALLOC_SCRATCH_BYTES (40 MiB). It is created when the library's
// device code is loaded on a GPU, and that GPU keeps it until the process exits, whether
// or not this entry point is ever called. It fits the router scratch of any call with
// T <= BEAM_MOE_NOALLOC_MAX_TOKENS (8192) at Beam's shape on GPUs of up to ~170 SMs. On a
// GPU where the router would pick more K splits than the array holds, fewer splits are
// used; only the summation order of the logits changes then.
//
// Host code cannot pass the array's name to a kernel (on the host it is a stand-in
// symbol, not a device address), so the first call on each device looks up the array's
// device address with cudaGetSymbolAddress while that device is current, and every later
// call on that device reuses it. Make that first call before any stream capture.
//
// Every call on a device shares the array, and it keeps what the last call wrote. Each
// call writes every element it later reads before reading it, so nothing needs clearing;
// but calls whose work overlaps on the GPU (several streams, or several host threads with
// their own streams) race on the array and must be serialised by the caller.
#include <mutex>

#include "internal.cuh"

static __device__ __align__(256) uint8_t g_route_noalloc_scratch[BEAM_MOE_NOALLOC_SCRATCH_BYTES];

namespace beam {
namespace {

struct NoAllocDevice {
    bool ready = false;
    int num_sms = 0;
    uint8_t* scratch = nullptr;  // device address of g_route_noalloc_scratch on this device
};
constexpr int kMaxNoAllocDevices = 64;
NoAllocDevice g_noalloc[kMaxNoAllocDevices];
std::mutex g_noalloc_mu;

// Once per device, with that device current: SM count and the array's device address.
int noalloc_device(NoAllocDevice** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxNoAllocDevices) return abi_fail(BEAM_MOE_ERR_ARG, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoAllocDevice& s = g_noalloc[dev];
    if (!s.ready) {
        if ((e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return abi_fail(BEAM_MOE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        void* p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_route_noalloc_scratch)) != cudaSuccess || p == nullptr)
            return abi_fail(BEAM_MOE_ERR_CUDA, "cudaGetSymbolAddress(router scratch): %s", cudaGetErrorString(e));
        s.scratch = static_cast<uint8_t*>(p);
        s.ready = true;
    }
    *out = &s;
    return BEAM_MOE_OK;
}

}  // namespace
}  // namespace beam

using namespace beam;

extern "C" int beam_moe_route_noalloc(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w,
                                      const float* expert_bias, int T, int32_t* topk_idx, float* topk_w,
                                      cudaStream_t stream) {
    int rc;
    if ((rc = abi_check_config(cfg))) return rc;
    if (T < 0 || T > BEAM_MOE_NOALLOC_MAX_TOKENS)
        return abi_fail(BEAM_MOE_ERR_ARG,
                        "T=%d is outside [0, %d], the token limit of beam_moe_route_noalloc (its fixed scratch "
                        "array holds %u bytes); use beam_moe_route_ex for larger batches",
                        T, BEAM_MOE_NOALLOC_MAX_TOKENS, static_cast<unsigned>(BEAM_MOE_NOALLOC_SCRATCH_BYTES));
    if ((rc = abi_check_ptr(x, "x")) || (rc = abi_check_ptr(router_w, "router_w")) ||
        (rc = abi_check_ptr(expert_bias, "expert_bias")) || (rc = abi_check_ptr(topk_idx, "topk_idx")) ||
        (rc = abi_check_ptr(topk_w, "topk_w")))
        return rc;
    if (T == 0) return BEAM_MOE_OK;
    if ((rc = abi_check_stream(stream))) return rc;
    NoAllocDevice* dev = nullptr;
    if ((rc = noalloc_device(&dev))) return rc;

    const Shape s{cfg->d, cfg->I, cfg->E, cfg->n_group, cfg->topk_group, cfg->top_k, cfg->scale};
    // Same plan as beam_moe_route_ex; layout: weight pieces, then the partial planes.
    RouterPlan plan = router_plan(s, T, dev->num_sms);
    const size_t w3_bytes = (plan.w3_elems * sizeof(bf16) + 255) & ~size_t(255);
    const size_t capacity = sizeof(g_route_noalloc_scratch);
    const int nk = s.d / 64;  // K chunks of the tensor-core product; its splits divide it
    while (plan.splits > 1 && w3_bytes + static_cast<size_t>(plan.splits) * T * s.E * sizeof(float) > capacity) {
        do {
            --plan.splits;
        } while (nk % plan.splits);
    }
    if (w3_bytes + static_cast<size_t>(plan.splits) * T * s.E * sizeof(float) > capacity)
        return abi_fail(BEAM_MOE_ERR_ARG, "T=%d with E=%d and d=%d needs more router scratch than the %u bytes of "
                        "beam_moe_route_noalloc", T, s.E, s.d, static_cast<unsigned>(capacity));
    bf16* w3 = plan.tensor ? reinterpret_cast<bf16*>(dev->scratch) : nullptr;
    float* partial = reinterpret_cast<float*>(dev->scratch + w3_bytes);
    cudaError_t e = cudaSuccess;
    if (plan.tensor) {
        e = launch_router_split_weights(s, router_w, w3, dev->num_sms, stream);
        if (e != cudaSuccess)
            return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router weight split failed: %s", cudaGetErrorString(e));
    }
    e = launch_router_logits(s, plan, x, router_w, T, w3, partial, nullptr, dev->num_sms, stream);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router logits failed: %s", cudaGetErrorString(e));
    e = launch_router_select(s, partial, plan.splits, expert_bias, T, topk_idx, topk_w, nullptr, stream);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router select failed: %s", cudaGetErrorString(e));
    return BEAM_MOE_OK;
}
