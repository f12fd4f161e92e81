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
// used; only the summation order of the logits changes then (noalloc_plan below; the
// exported beam_moe_route_noalloc_plan gives the same answer for any SM count).
//
// A second file-scope word holds this entry point's kernel status: the tensor-core logits
// kernel records there a pipeline wait that ran past its limit (its partial planes are then
// incomplete, and the array still holds the previous call's values), and
// beam_moe_route_noalloc_status reads and clears it without touching the library's pool.
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
static __device__ int g_route_noalloc_status;  // 0, or the first status code a kernel recorded

namespace beam {
namespace {

struct NoAllocDevice {
    bool ready = false;
    int num_sms = 0;
    uint8_t* scratch = nullptr;  // device address of g_route_noalloc_scratch on this device
    int* status = nullptr;       // device address of g_route_noalloc_status on this device
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
        p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_route_noalloc_status)) != cudaSuccess || p == nullptr)
            return abi_fail(BEAM_MOE_ERR_CUDA, "cudaGetSymbolAddress(router status): %s", cudaGetErrorString(e));
        s.status = static_cast<int*>(p);
        s.ready = true;
    }
    *out = &s;
    return BEAM_MOE_OK;
}

// The router plan of a call with T tokens on a GPU with num_sms SMs, its K split count
// lowered (to divisors of the d/64 K chunks) until the BF16 weight pieces and the FP32
// partial planes fit the array. Returns BEAM_MOE_OK, or BEAM_MOE_ERR_ARG with a message if
// T is outside [1, BEAM_MOE_NOALLOC_MAX_TOKENS] or even one split does not fit.
int noalloc_plan(const Shape& s, int T, int num_sms, RouterPlan* plan, size_t* w3_bytes) {
    if (T < 1 || T > BEAM_MOE_NOALLOC_MAX_TOKENS)
        return abi_fail(BEAM_MOE_ERR_ARG,
                        "T=%d is outside [0, %d], the token limit of beam_moe_route_noalloc (its fixed scratch "
                        "array holds %u bytes); use beam_moe_route_ex for larger batches",
                        T, BEAM_MOE_NOALLOC_MAX_TOKENS, static_cast<unsigned>(BEAM_MOE_NOALLOC_SCRATCH_BYTES));
    if (num_sms < 1) return abi_fail(BEAM_MOE_ERR_ARG, "num_sms=%d must be positive", num_sms);
    RouterPlan p = router_plan(s, T, num_sms);
    const size_t wb = (p.w3_elems * sizeof(bf16) + 255) & ~size_t(255);
    const size_t capacity = BEAM_MOE_NOALLOC_SCRATCH_BYTES;
    const size_t plane = static_cast<size_t>(T) * s.E * sizeof(float);
    const int nk = s.d / 64;  // K chunks of the tensor-core product; its splits divide it
    while (p.splits > 1 && wb + static_cast<size_t>(p.splits) * plane > capacity) {
        do {
            --p.splits;
        } while (nk % p.splits);
    }
    if (wb + static_cast<size_t>(p.splits) * plane > capacity)
        return abi_fail(BEAM_MOE_ERR_ARG, "T=%d with E=%d and d=%d needs more router scratch than the %u bytes of "
                        "beam_moe_route_noalloc", T, s.E, s.d, static_cast<unsigned>(capacity));
    *plan = p;
    *w3_bytes = wb;
    return BEAM_MOE_OK;
}

Shape shape_of_cfg(const beam_moe_config* c) {
    return Shape{c->d, c->I, c->E, c->n_group, c->topk_group, c->top_k, c->scale};
}

}  // namespace
}  // namespace beam

using namespace beam;

extern "C" int beam_moe_route_noalloc_plan(const beam_moe_config* cfg, int T, int num_sms, int* splits) {
    int rc;
    if ((rc = abi_check_config(cfg))) return rc;
    if (!splits) return abi_fail(BEAM_MOE_ERR_ARG, "splits is null");
    RouterPlan plan;
    size_t w3_bytes = 0;
    if ((rc = noalloc_plan(shape_of_cfg(cfg), T, num_sms, &plan, &w3_bytes))) return rc;
    *splits = plan.splits;
    return BEAM_MOE_OK;
}

extern "C" int beam_moe_route_noalloc_status(cudaStream_t stream) {
    int rc;
    if ((rc = abi_check_stream(stream))) return rc;
    NoAllocDevice* dev = nullptr;
    if ((rc = noalloc_device(&dev))) return rc;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    int word = 0;
    if ((e = cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return abi_fail(BEAM_MOE_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (word == kStatusOk) return BEAM_MOE_OK;
    if ((e = cudaMemset(dev->status, 0, sizeof word)) != cudaSuccess)
        return abi_fail(BEAM_MOE_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    return abi_fail(BEAM_MOE_ERR_DEVICE, "no-allocation router kernel status %d (%s)", word,
                    word == kStatusWaitTimeout ? "a GEMM pipeline wait ran past its limit" : "unknown");
}

extern "C" int beam_moe_route_noalloc_selftest(cudaStream_t stream) {
    int rc;
    if ((rc = abi_check_stream(stream))) return rc;
    NoAllocDevice* dev = nullptr;
    if ((rc = noalloc_device(&dev))) return rc;
    // One 128-expert tile of the tensor-core logits product over d = 128, 48 tokens, on
    // zeros laid out in the array: weight pieces [3][128][128], tokens [48][128], one plane.
    const Shape s{128, 128, 128, 4, 1, 1, 1.0f};
    const int T = 48;
    bf16* w3 = reinterpret_cast<bf16*>(dev->scratch);
    bf16* x = w3 + 3 * 128 * 128;
    float* partial = reinterpret_cast<float*>(x + T * 128);
    const size_t bytes = reinterpret_cast<uint8_t*>(partial + T * 128) - dev->scratch;
    cudaError_t e = cudaMemsetAsync(dev->scratch, 0, bytes, stream);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "scratch clear: %s", cudaGetErrorString(e));
    e = launch_router_tc(s, w3, x, T, 1, partial, dev->status, 1, stream, 16u);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router logits failed: %s", cudaGetErrorString(e));
    return BEAM_MOE_OK;
}

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

    const Shape s = shape_of_cfg(cfg);
    // Same plan as beam_moe_route_ex (fewer splits only if the array cannot hold them);
    // layout: weight pieces, then the partial planes.
    RouterPlan plan;
    size_t w3_bytes = 0;
    if ((rc = noalloc_plan(s, T, dev->num_sms, &plan, &w3_bytes))) return rc;
    bf16* w3 = plan.tensor ? reinterpret_cast<bf16*>(dev->scratch) : nullptr;
    float* partial = reinterpret_cast<float*>(dev->scratch + w3_bytes);
    cudaError_t e = cudaSuccess;
    if (plan.tensor) {
        e = launch_router_split_weights(s, router_w, w3, dev->num_sms, stream);
        if (e != cudaSuccess)
            return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router weight split failed: %s", cudaGetErrorString(e));
    }
    e = launch_router_logits(s, plan, x, router_w, T, w3, partial, dev->status, dev->num_sms, stream);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router logits failed: %s", cudaGetErrorString(e));
    e = launch_router_select(s, partial, plan.splits, expert_bias, T, topk_idx, topk_w, nullptr, stream);
    if (e != cudaSuccess) return abi_fail(BEAM_MOE_ERR_CUDA, "launch of router select failed: %s", cudaGetErrorString(e));
    return BEAM_MOE_OK;
}
