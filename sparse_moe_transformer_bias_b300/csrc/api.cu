// C ABI of libbeam_moe.so (declared and documented in include/beam_moe.h): argument
// checks, per-device state (scratch pool, status word), scratch layout and the launch
// sequence of the Beam MoE forward pass.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "beam_moe.h"
#include "internal.cuh"

namespace beam {
namespace {

thread_local char g_err[512] = "";
thread_local int g_launches = 0;

// Debug aid: fill every scratch allocation with 0xFF bytes (NaN in BF16 and FP32, -1 in
// int32) before the call's kernels run, so that a value read before it is written shows
// up in the output. Off unless beam_moe_debug_poison_scratch(1) or BEAM_MOE_DEBUG=1.
std::atomic<int> g_poison{-1};  // -1: not yet read from the environment

bool poison_scratch() {
    int v = g_poison.load(std::memory_order_relaxed);
    if (v < 0) {
        const char* env = getenv("BEAM_MOE_DEBUG");
        v = (env && env[0] && strcmp(env, "0") != 0) ? 1 : 0;
        int expect = -1;
        g_poison.compare_exchange_strong(expect, v);
        v = g_poison.load(std::memory_order_relaxed);
    }
    return v == 1;
}

// Fills a fresh scratch allocation when the debug aid is on.
cudaError_t maybe_poison(void* mem, size_t bytes, cudaStream_t st) {
    return poison_scratch() ? cudaMemsetAsync(mem, 0xFF, bytes, st) : cudaSuccess;
}

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

// ---------------------------------------------------------------- per-device state
struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    cudaMemPool_t pool = nullptr;
    int* status = nullptr;  // device word written by kernels
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

int device_state(DeviceState** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(BEAM_MOE_ERR_ARG, "device %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState& s = g_dev[dev];
    if (!s.ready) {
        if ((e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail(BEAM_MOE_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
        cudaMemPoolProps props;
        memset(&props, 0, sizeof props);
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if ((e = cudaMemPoolCreate(&s.pool, &props)) != cudaSuccess)
            return fail(BEAM_MOE_ERR_CUDA, "cudaMemPoolCreate: %s", cudaGetErrorString(e));
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(s.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if ((e = cudaMalloc(&s.status, 16)) != cudaSuccess)
            return fail(BEAM_MOE_ERR_CUDA, "cudaMalloc(status): %s", cudaGetErrorString(e));
        if ((e = cudaMemset(s.status, 0, 16)) != cudaSuccess)
            return fail(BEAM_MOE_ERR_CUDA, "cudaMemset(status): %s", cudaGetErrorString(e));
        s.ready = true;
    }
    *out = &s;
    return BEAM_MOE_OK;
}

int check_stream(cudaStream_t st) {
    if (st == nullptr) return BEAM_MOE_OK;
    // While the stream is being captured into a graph the device query below is not
    // allowed; the launches are recorded on the capturing stream as they are.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusActive) return BEAM_MOE_OK;
    cudaGetLastError();
    int sdev = -1, cdev = -1;
    if (cudaStreamGetDevice(st, &sdev) != cudaSuccess || cudaGetDevice(&cdev) != cudaSuccess) {
        cudaGetLastError();
        return fail(BEAM_MOE_ERR_ARG, "invalid stream");
    }
    if (sdev != cdev) return fail(BEAM_MOE_ERR_ARG, "stream belongs to device %d but device %d is current", sdev, cdev);
    return BEAM_MOE_OK;
}

// ---------------------------------------------------------------- stage timing
enum Stage {
    kPreNorm, kSplitW, kLogits, kSelect, kCount, kScan, kScatter, kGather, kExpert, kCombine, kActPrep, kNumStages
};
struct Timing {
    bool enabled = false;
    bool created = false;
    int device = -1;
    cudaEvent_t start[kNumStages], stop[kNumStages];
    bool ran[kNumStages] = {};
    cudaEvent_t last = nullptr;
};
thread_local Timing g_timing;

void timing_begin_call() {
    for (bool& r : g_timing.ran) r = false;
    g_timing.last = nullptr;
}
void stage_begin(Stage s, cudaStream_t st) {
    if (!g_timing.enabled) return;
    cudaEventRecord(g_timing.start[s], st);
}
void stage_end(Stage s, cudaStream_t st) {
    ++g_launches;
    if (!g_timing.enabled) return;
    cudaEventRecord(g_timing.stop[s], st);
    g_timing.ran[s] = true;
    g_timing.last = g_timing.stop[s];
}

// ---------------------------------------------------------------- checks and layout
int check_cfg(const beam_moe_config* c) {
    if (!c) return fail(BEAM_MOE_ERR_ARG, "config is null");
    if (c->d < 128 || c->d % 128) return fail(BEAM_MOE_ERR_ARG, "d=%d must be a positive multiple of 128", c->d);
    if (c->I < 128 || c->I % 128) return fail(BEAM_MOE_ERR_ARG, "I=%d must be a positive multiple of 128", c->I);
    if (c->n_group < 1 || c->n_group > 8) return fail(BEAM_MOE_ERR_ARG, "n_group=%d must be in [1, 8]", c->n_group);
    if (c->E != 32 * c->n_group) return fail(BEAM_MOE_ERR_ARG, "E=%d must equal 32 * n_group", c->E);
    if (c->topk_group < 1 || c->topk_group > c->n_group)
        return fail(BEAM_MOE_ERR_ARG, "topk_group=%d must be in [1, n_group]", c->topk_group);
    if (c->top_k < 1 || c->top_k > 32 || c->top_k > 32 * c->topk_group)
        return fail(BEAM_MOE_ERR_ARG, "top_k=%d must be in [1, min(32, 32 * topk_group)]", c->top_k);
    if (!std::isfinite(c->scale)) return fail(BEAM_MOE_ERR_ARG, "scale must be finite");
    return BEAM_MOE_OK;
}

int check_T(int T) {
    if (T < 0 || T > BEAM_MOE_MAX_TOKENS) return fail(BEAM_MOE_ERR_ARG, "T=%d must be in [0, %d]", T, BEAM_MOE_MAX_TOKENS);
    return BEAM_MOE_OK;
}

int check_ptr(const void* p, const char* name) {
    if (!p) return fail(BEAM_MOE_ERR_ARG, "%s is null", name);
    if (reinterpret_cast<uintptr_t>(p) % 16) return fail(BEAM_MOE_ERR_ALIGN, "%s is not 16-byte aligned", name);
    return BEAM_MOE_OK;
}

Shape shape_of(const beam_moe_config* c) { return Shape{c->d, c->I, c->E, c->n_group, c->topk_group, c->top_k, c->scale}; }

struct Scratch {
    bf16* x_norm = nullptr;
    bf16* w3 = nullptr;
    float* partial = nullptr;
    int32_t* idx = nullptr;
    float* w = nullptr;
    int* chunk = nullptr;
    int* expert_offset = nullptr;
    int4* tiles = nullptr;
    int* tile_done = nullptr;
    int* perm_src = nullptr;
    int* inv_slot = nullptr;
    bf16* x_perm = nullptr;
    bf16* h = nullptr;
    bf16* y = nullptr;
    float* xmax = nullptr;    // FP8 products: largest |x| per token
    float* amax_h = nullptr;  // FP8 products: largest |h| per permuted row
    uint8_t* x8 = nullptr;    // the pieces of every token row: FP8 [T][2][d], NVFP4 codes [T][4][d/2]
    uint8_t* xs = nullptr;    // NVFP4 products: block scales of the token rows' pieces [T][4][d/16]
    uint8_t* xs_perm = nullptr;  // the same for the dispatched rows [rows][4][d/16]
    uint8_t* hs = nullptr;    // NVFP4 products: block scales of h's pieces [rows][4][I/16]
};

struct Carver {
    char* base;
    size_t off = 0;
    template <typename T>
    T* take(size_t count) {
        off = (off + 255) & ~size_t(255);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
};

// Lays scratch out from `base` (nullptr: size only). Returns the byte count.
size_t layout(const Shape& s, int T, const RouterPlan& plan, int max_tiles, bool forward, bool route_out,
              bool pre_norm, int pieces, char* base, Scratch* sc) {
    Carver c{base};
    const size_t pairs = static_cast<size_t>(T) * s.top_k;
    sc->x_norm = pre_norm ? c.take<bf16>(static_cast<size_t>(T) * s.d) : nullptr;
    sc->w3 = plan.w3_elems ? c.take<bf16>(plan.w3_elems) : nullptr;
    sc->partial = c.take<float>(static_cast<size_t>(plan.splits) * T * s.E);
    if (route_out) {
        sc->idx = c.take<int32_t>(pairs);
        sc->w = c.take<float>(pairs);
    }
    if (forward) {
        const int nchunks = (T + kDispatchChunk - 1) / kDispatchChunk;
        sc->chunk = c.take<int>(static_cast<size_t>(nchunks) * s.E);
        sc->expert_offset = c.take<int>(s.E + 1);
        sc->tiles = c.take<int4>(1 + static_cast<size_t>(max_tiles));
        sc->tile_done = c.take<int>(static_cast<size_t>(max_tiles));
        sc->perm_src = c.take<int>(pairs);
        sc->inv_slot = c.take<int>(pairs);
        sc->x_perm = c.take<bf16>(pairs * s.d);
        sc->h = c.take<bf16>(pairs * s.I);
        sc->y = c.take<bf16>(pairs * s.d);
        if (pieces == 2) {
            sc->xmax = c.take<float>(static_cast<size_t>(T));
            sc->amax_h = c.take<float>(pairs);
            sc->x8 = c.take<uint8_t>(static_cast<size_t>(T) * 2 * s.d);
        } else if (pieces == 4) {
            sc->x8 = c.take<uint8_t>(static_cast<size_t>(T) * 2 * s.d);
            sc->xs = c.take<uint8_t>(static_cast<size_t>(T) * s.d / 4);
            sc->xs_perm = c.take<uint8_t>(pairs * s.d / 4);
            sc->hs = c.take<uint8_t>(pairs * s.I / 4);
        }
    }
    return c.off + 256;
}

#define LAUNCH(stage, expr)                                                                         \
    do {                                                                                            \
        stage_begin(stage, st);                                                                     \
        cudaError_t e_ = (expr);                                                                    \
        stage_end(stage, st);                                                                       \
        if (e_ != cudaSuccess) {                                                                    \
            rc = fail(BEAM_MOE_ERR_CUDA, "launch of %s failed: %s", #stage, cudaGetErrorString(e_)); \
            goto done;                                                                              \
        }                                                                                           \
    } while (0)

// The MoE sublayer's extra inputs (mode 3).
struct SublayerArgs {
    const bf16* pre_gamma;
    const bf16* post_gamma;
    float eps;
    int k;
};

// An expert-parallel shard's extra inputs (mode 4): its experts and its FP32 output.
struct ShardArgs {
    int e_begin, e_end;
    float* out_partial;
};

// mode 0: route (outputs topk_idx/topk_w); 1: logits only; 2: forward; 3: sublayer (x is
// the residual stream: pre-norm, forward, then combine fused with the post-norm and the
// residual update into out); 4: forward of one expert-parallel shard (wg/wu/wd hold only
// experts [e_begin, e_end); FP32 partial output over the slots routed there); 5: forward
// with FP8 expert weights (q8; wg/wu/wd unused); 6: forward with NVFP4 expert weights (q4;
// wg/wu/wd unused).
int run(const beam_moe_config* cfg, const bf16* x, const float* wr, const float* bias, const bf16* wg,
        const bf16* wu, const bf16* wd, int T, int32_t* topk_idx, float* topk_w, float* logits, bf16* out, int mode,
        cudaStream_t st, const SublayerArgs* sub = nullptr, const ShardArgs* shard = nullptr,
        const Fp8Experts* q8 = nullptr, const Nvfp4Experts* q4 = nullptr) {
    g_launches = 0;
    timing_begin_call();
    int rc;
    if ((rc = check_cfg(cfg)) || (rc = check_T(T)) || (rc = check_ptr(x, mode == 3 ? "stream_in" : "x")) ||
        (rc = check_ptr(wr, "router_w")))
        return rc;
    if (mode == 3) {
        if ((rc = check_ptr(sub->pre_gamma, "pre_gamma")) || (rc = check_ptr(sub->post_gamma, "post_gamma"))) return rc;
        if (!(sub->eps >= 0.f) || !std::isfinite(sub->eps)) return fail(BEAM_MOE_ERR_ARG, "eps must be finite and >= 0");
        if (sub->k < 2) return fail(BEAM_MOE_ERR_ARG, "k=%d must be >= 2 (the embedding is contribution 1)", sub->k);
        if (cfg->d > kNormMaxD) return fail(BEAM_MOE_ERR_ARG, "d=%d exceeds the sublayer limit %d", cfg->d, kNormMaxD);
    }
    if (mode != 1 && (rc = check_ptr(bias, "expert_bias"))) return rc;
    if (mode == 0 && ((rc = check_ptr(topk_idx, "topk_idx")) || (rc = check_ptr(topk_w, "topk_w")))) return rc;
    if (mode == 1 && (rc = check_ptr(logits, "logits"))) return rc;
    if (mode == 6) {
        if ((rc = check_ptr(q4->wg, "w_gate_q")) || (rc = check_ptr(q4->gbs, "gate_block_scale")) ||
            (rc = check_ptr(q4->gts, "gate_tensor_scale")) || (rc = check_ptr(q4->wu, "w_up_q")) ||
            (rc = check_ptr(q4->ubs, "up_block_scale")) || (rc = check_ptr(q4->uts, "up_tensor_scale")) ||
            (rc = check_ptr(q4->wd, "w_down_q")) || (rc = check_ptr(q4->dbs, "down_block_scale")) ||
            (rc = check_ptr(q4->dts, "down_tensor_scale")))
            return rc;
        if (cfg->d % 256 || cfg->I % 256)
            return fail(BEAM_MOE_ERR_ARG, "NVFP4 experts need d and I to be multiples of 256 (d=%d, I=%d)", cfg->d,
                        cfg->I);
    } else if (mode == 5) {
        if ((rc = check_ptr(q8->wg, "w_gate_q")) || (rc = check_ptr(q8->gs, "gate_scale")) ||
            (rc = check_ptr(q8->wu, "w_up_q")) || (rc = check_ptr(q8->us, "up_scale")) ||
            (rc = check_ptr(q8->wd, "w_down_q")) || (rc = check_ptr(q8->ds, "down_scale")))
            return rc;
    } else if (mode >= 2 &&
               ((rc = check_ptr(wg, "w_gate")) || (rc = check_ptr(wu, "w_up")) || (rc = check_ptr(wd, "w_down")))) {
        return rc;
    }
    if (mode == 4) {
        if ((rc = check_ptr(shard->out_partial, "out_partial"))) return rc;
        if (shard->e_begin < 0 || shard->e_begin >= shard->e_end || shard->e_end > cfg->E)
            return fail(BEAM_MOE_ERR_ARG, "expert range [%d, %d) must be a non-empty part of [0, %d)", shard->e_begin,
                        shard->e_end, cfg->E);
    } else if (mode >= 2 && (rc = check_ptr(out, mode == 3 ? "stream_out" : "out"))) {
        return rc;
    }
    if (T == 0) return BEAM_MOE_OK;
    if ((rc = check_stream(st))) return rc;
    DeviceState* dev = nullptr;
    if ((rc = device_state(&dev))) return rc;

    if (g_timing.enabled) {
        int d = -1;
        cudaGetDevice(&d);
        if (g_timing.created && g_timing.device != d) {
            for (int i = 0; i < kNumStages; ++i) {
                cudaEventDestroy(g_timing.start[i]);
                cudaEventDestroy(g_timing.stop[i]);
            }
            g_timing.created = false;
        }
        if (!g_timing.created) {
            for (int i = 0; i < kNumStages; ++i) {
                cudaEventCreate(&g_timing.start[i]);
                cudaEventCreate(&g_timing.stop[i]);
            }
            g_timing.created = true;
            g_timing.device = d;
        }
    }

    const Shape s = shape_of(cfg);
    // The experts this call runs: all of them, or the shard's (local ids from 0).
    const int e_lo = mode == 4 ? shard->e_begin : 0;
    Shape se = s;
    se.E = mode == 4 ? shard->e_end - shard->e_begin : s.E;
    const RouterPlan plan = router_plan(s, T, dev->num_sms);
    const int bn_max = mode == 5 ? gemm_bn_max_f8(s, T) : mode == 6 ? gemm_bn_max_nvf4(s, T) : gemm_bn_max(s, T);
    const int pieces = mode == 5 ? 2 : mode == 6 ? 4 : 0;  // activation pieces of the low-precision products
    const int max_tiles = dispatch_max_tiles(se, T, bn_max);
    const int rows = T * s.top_k;
    Scratch sc;
    const bool fwd = mode >= 2;
    const size_t bytes = layout(s, T, plan, max_tiles, fwd, mode != 0, mode == 3, pieces, nullptr, &sc);
    void* mem = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&mem, bytes, dev->pool, st);
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "scratch allocation of %zu bytes: %s", bytes, cudaGetErrorString(e));
    layout(s, T, plan, max_tiles, fwd, mode != 0, mode == 3, pieces, static_cast<char*>(mem), &sc);
    if ((e = maybe_poison(mem, bytes, st)) != cudaSuccess) {
        rc = fail(BEAM_MOE_ERR_CUDA, "scratch poison: %s", cudaGetErrorString(e));
        goto done;
    }
    {
        int32_t* idx = mode == 0 ? topk_idx : sc.idx;
        float* w = mode == 0 ? topk_w : sc.w;
        const bf16* stream_in = x;
        if (mode == 3) {
            LAUNCH(kPreNorm, launch_rmsnorm(s.d, stream_in, sub->pre_gamma, sub->eps, T, sc.x_norm, st));
            x = sc.x_norm;
        }
        if (plan.tensor) LAUNCH(kSplitW, launch_router_split_weights(s, wr, sc.w3, dev->num_sms, st));
        LAUNCH(kLogits, launch_router_logits(s, plan, x, wr, T, sc.w3, sc.partial, dev->status, dev->num_sms, st));
        LAUNCH(kSelect, launch_router_select(s, sc.partial, plan.splits, mode == 1 ? nullptr : bias, T, idx, w,
                                             mode == 1 ? logits : nullptr, st));
        if (fwd) {
            // FP8 / NVFP4 products: each token row is split into its two E4M3 or four NVFP4
            // pieces first; the dispatch then moves those rows (2d bytes each, as a BF16 row)
            // instead of x, and for NVFP4 the pieces' block scales beside them.
            const bf16* rows_src = x;
            if (mode == 5) {
                LAUNCH(kActPrep, launch_fp8_prep(x, s.d, T, sc.xmax, sc.x8, sc.amax_h, rows, dev->num_sms, st));
                rows_src = reinterpret_cast<const bf16*>(sc.x8);
            } else if (mode == 6) {
                LAUNCH(kActPrep, launch_act4_prep(x, s.d, T, sc.x8, sc.xs, dev->status, dev->num_sms, st));
                rows_src = reinterpret_cast<const bf16*>(sc.x8);
            }
            const int side_bytes = mode == 6 ? s.d / 4 : 0;
            if (T <= kSmallDispatchT) {
                // one launch for the whole dispatch (timed as the count stage)
                LAUNCH(kCount, launch_dispatch_small(s, e_lo, se.E, idx, T, bn_max, rows_src, sc.expert_offset, sc.tiles,
                                                     sc.tile_done, sc.perm_src, sc.inv_slot, sc.x_perm, dev->status,
                                                     dev->num_sms, st, sc.xs, side_bytes, sc.xs_perm));
            } else {
                LAUNCH(kCount, launch_dispatch_count(s, e_lo, se.E, idx, T, sc.chunk, dev->status, st));
                LAUNCH(kScan,
                       launch_dispatch_scan(se.E, T, bn_max, sc.chunk, sc.expert_offset, sc.tiles, sc.tile_done, st));
                LAUNCH(kScatter, launch_dispatch_scatter(s, e_lo, se.E, idx, T, sc.chunk, sc.perm_src, sc.inv_slot,
                                                         dev->status, st));
                LAUNCH(kGather, launch_gather_rows(rows_src, s.d, T, sc.perm_src, sc.expert_offset + se.E, rows, sc.x_perm,
                                                   dev->status, dev->num_sms, st, sc.xs, side_bytes, sc.xs_perm));
            }
            if (mode == 5) {
                LAUNCH(kExpert, launch_expert_mlp_f8(se, *q8, reinterpret_cast<const uint8_t*>(sc.x_perm), rows, T,
                                                     sc.perm_src, sc.xmax, sc.amax_h,
                                                     sc.tiles, sc.tile_done, max_tiles, bn_max, sc.h, sc.y,
                                                     dev->status, dev->num_sms, st));
            } else if (mode == 6) {
                LAUNCH(kExpert, launch_expert_mlp_nvf4(se, *q4, reinterpret_cast<const uint8_t*>(sc.x_perm), sc.xs_perm,
                                                       rows, sc.tiles, sc.tile_done, max_tiles, bn_max,
                                                       reinterpret_cast<uint8_t*>(sc.h), sc.hs, sc.y, dev->status,
                                                       dev->num_sms, st));
            } else
                LAUNCH(kExpert, launch_expert_mlp(se, wg, wu, wd, sc.x_perm, rows, sc.tiles, sc.tile_done,
                                                  max_tiles, bn_max, sc.h, sc.y, dev->status, dev->num_sms, st));
            if (mode == 4)
                LAUNCH(kCombine, launch_combine_partial(s, sc.y, sc.inv_slot, w, T, shard->out_partial, dev->status,
                                                        st));
            else if (mode == 3)
                LAUNCH(kCombine, launch_combine_residual(s, sc.y, sc.inv_slot, w, T, stream_in, sub->post_gamma,
                                                         sub->eps, sub->k, out, dev->status, st));
            else
                LAUNCH(kCombine, launch_combine(s, sc.y, sc.inv_slot, w, T, out, dev->status, st));
        }
    }
    rc = BEAM_MOE_OK;
done:
    e = cudaFreeAsync(mem, st);
    if (rc == BEAM_MOE_OK && e != cudaSuccess)
        rc = fail(BEAM_MOE_ERR_CUDA, "scratch release: %s", cudaGetErrorString(e));
    return rc;
}

}  // namespace

int abi_fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}
int abi_check_config(const beam_moe_config* cfg) { return check_cfg(cfg); }
int abi_check_ptr(const void* p, const char* name) { return check_ptr(p, name); }
int abi_check_stream(cudaStream_t st) { return check_stream(st); }

}  // namespace beam

using namespace beam;

extern "C" {

beam_moe_config beam_moe_default_config(void) {
    beam_moe_config c;
    c.d = 5120;
    c.I = 2560;
    c.E = 256;
    c.n_group = 8;
    c.topk_group = 4;
    c.top_k = 8;
    c.scale = 2.5f;
    return c;
}

int beam_moe_route_ex(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w,
                      const float* expert_bias, int T, int32_t* topk_idx, float* topk_w, cudaStream_t stream) {
    return run(cfg, x, router_w, expert_bias, nullptr, nullptr, nullptr, T, topk_idx, topk_w, nullptr, nullptr, 0,
               stream);
}

int beam_moe_route(const __nv_bfloat16* x, const float* router_w, const float* expert_bias, int T, int32_t* topk_idx,
                   float* topk_w, cudaStream_t stream) {
    const beam_moe_config c = beam_moe_default_config();
    return beam_moe_route_ex(&c, x, router_w, expert_bias, T, topk_idx, topk_w, stream);
}

int beam_moe_forward_ex(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w,
                        const float* expert_bias, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                        const __nv_bfloat16* w_down, int T, __nv_bfloat16* out, cudaStream_t stream) {
    return run(cfg, x, router_w, expert_bias, w_gate, w_up, w_down, T, nullptr, nullptr, nullptr, out, 2, stream);
}

int beam_moe_forward(const __nv_bfloat16* x, const float* router_w, const float* expert_bias,
                     const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up, const __nv_bfloat16* w_down, int T,
                     __nv_bfloat16* out, cudaStream_t stream) {
    const beam_moe_config c = beam_moe_default_config();
    return beam_moe_forward_ex(&c, x, router_w, expert_bias, w_gate, w_up, w_down, T, out, stream);
}

int beam_moe_forward_host(const beam_moe_config* cfg, const __nv_bfloat16* x_host, const float* router_w,
                          const float* expert_bias, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                          const __nv_bfloat16* w_down, int T, __nv_bfloat16* out_host, cudaStream_t stream) {
    int rc;
    if ((rc = check_cfg(cfg)) || (rc = check_T(T))) return rc;
    if (!x_host) return fail(BEAM_MOE_ERR_ARG, "x_host is null");
    if (!out_host) return fail(BEAM_MOE_ERR_ARG, "out_host is null");
    if (T == 0) return BEAM_MOE_OK;
    if ((rc = check_stream(stream))) return rc;
    DeviceState* dev = nullptr;
    if ((rc = device_state(&dev))) return rc;
    const size_t row_bytes = static_cast<size_t>(cfg->d) * sizeof(bf16);
    const size_t bytes = ((static_cast<size_t>(T) * row_bytes + 255) & ~size_t(255)) * 2;
    void* mem = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&mem, bytes, dev->pool, stream);
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "device buffers of %zu bytes: %s", bytes, cudaGetErrorString(e));
    bf16* x_dev = static_cast<bf16*>(mem);
    bf16* out_dev = reinterpret_cast<bf16*>(static_cast<char*>(mem) + bytes / 2);
    rc = BEAM_MOE_OK;
    if ((e = cudaMemcpyAsync(x_dev, x_host, T * row_bytes, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
        rc = fail(BEAM_MOE_ERR_CUDA, "copy of x to the device: %s", cudaGetErrorString(e));
    if (rc == BEAM_MOE_OK)
        rc = run(cfg, x_dev, router_w, expert_bias, w_gate, w_up, w_down, T, nullptr, nullptr, nullptr, out_dev, 2,
                 stream);
    const int launches = g_launches;
    if (rc == BEAM_MOE_OK &&
        (e = cudaMemcpyAsync(out_host, out_dev, T * row_bytes, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
        rc = fail(BEAM_MOE_ERR_CUDA, "copy of out to the host: %s", cudaGetErrorString(e));
    e = cudaFreeAsync(mem, stream);
    if (rc == BEAM_MOE_OK && e != cudaSuccess) rc = fail(BEAM_MOE_ERR_CUDA, "buffer release: %s", cudaGetErrorString(e));
    e = cudaStreamSynchronize(stream);
    if (rc == BEAM_MOE_OK && e != cudaSuccess)
        rc = fail(BEAM_MOE_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    g_launches = launches;
    return rc;
}

int beam_moe_sublayer_forward(const beam_moe_config* cfg, const __nv_bfloat16* stream_in,
                              const __nv_bfloat16* pre_gamma, const __nv_bfloat16* post_gamma, float eps, int k,
                              const float* router_w, const float* expert_bias, const __nv_bfloat16* w_gate,
                              const __nv_bfloat16* w_up, const __nv_bfloat16* w_down, int T, __nv_bfloat16* stream_out,
                              cudaStream_t stream) {
    const SublayerArgs sub{pre_gamma, post_gamma, eps, k};
    return run(cfg, stream_in, router_w, expert_bias, w_gate, w_up, w_down, T, nullptr, nullptr, nullptr, stream_out, 3,
               stream, &sub);
}

int beam_moe_forward_shard(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w,
                           const float* expert_bias, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                           const __nv_bfloat16* w_down, int e_begin, int e_end, int T, float* out_partial,
                           cudaStream_t stream) {
    const ShardArgs sh{e_begin, e_end, out_partial};
    return run(cfg, x, router_w, expert_bias, w_gate, w_up, w_down, T, nullptr, nullptr, nullptr, nullptr, 4, stream,
               nullptr, &sh);
}

int beam_moe_forward_fp8(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w,
                         const float* expert_bias, const uint8_t* w_gate_q, const float* gate_scale,
                         const uint8_t* w_up_q, const float* up_scale, const uint8_t* w_down_q,
                         const float* down_scale, int T, __nv_bfloat16* out, cudaStream_t stream) {
    const Fp8Experts q{w_gate_q, gate_scale, w_up_q, up_scale, w_down_q, down_scale};
    return run(cfg, x, router_w, expert_bias, nullptr, nullptr, nullptr, T, nullptr, nullptr, nullptr, out, 5, stream,
               nullptr, nullptr, &q);
}

int beam_moe_forward_nvfp4(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w,
                           const float* expert_bias, const uint8_t* w_gate_q, const uint8_t* gate_block_scale,
                           const float* gate_tensor_scale, const uint8_t* w_up_q, const uint8_t* up_block_scale,
                           const float* up_tensor_scale, const uint8_t* w_down_q, const uint8_t* down_block_scale,
                           const float* down_tensor_scale, int T, __nv_bfloat16* out, cudaStream_t stream) {
    const Nvfp4Experts q{w_gate_q,       gate_block_scale, gate_tensor_scale, w_up_q,           up_block_scale,
                         up_tensor_scale, w_down_q,        down_block_scale,  down_tensor_scale};
    return run(cfg, x, router_w, expert_bias, nullptr, nullptr, nullptr, T, nullptr, nullptr, nullptr, out, 6, stream,
               nullptr, nullptr, nullptr, &q);
}

int beam_moe_dense_mlp(int d, int I, const __nv_bfloat16* x, const __nv_bfloat16* w_gate, const __nv_bfloat16* w_up,
                       const __nv_bfloat16* w_down, int T, __nv_bfloat16* out, cudaStream_t stream) {
    g_launches = 0;
    timing_begin_call();
    int rc;
    if (d < 128 || d % 128) return fail(BEAM_MOE_ERR_ARG, "d=%d must be a positive multiple of 128", d);
    if (I < 128 || I % 128) return fail(BEAM_MOE_ERR_ARG, "I=%d must be a positive multiple of 128", I);
    if ((rc = check_T(T)) || (rc = check_ptr(x, "x")) || (rc = check_ptr(w_gate, "w_gate")) ||
        (rc = check_ptr(w_up, "w_up")) || (rc = check_ptr(w_down, "w_down")) || (rc = check_ptr(out, "out")))
        return rc;
    if (T == 0) return BEAM_MOE_OK;
    if ((rc = check_stream(stream))) return rc;
    DeviceState* dev = nullptr;
    if ((rc = device_state(&dev))) return rc;
    const Shape s{d, I, 1, 1, 1, 1, 1.0f};
    const int bn_max = gemm_bn_max(s, T);
    const int max_tiles = dense_max_tiles(T, bn_max);
    Carver c{nullptr};
    c.take<int4>(1 + static_cast<size_t>(max_tiles));
    c.take<int>(static_cast<size_t>(max_tiles));
    c.take<bf16>(static_cast<size_t>(T) * I);
    const size_t bytes = c.off + 256;
    void* mem = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&mem, bytes, dev->pool, stream);
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "scratch allocation of %zu bytes: %s", bytes, cudaGetErrorString(e));
    Carver cc{static_cast<char*>(mem)};
    int4* tiles = cc.take<int4>(1 + static_cast<size_t>(max_tiles));
    int* tile_done = cc.take<int>(static_cast<size_t>(max_tiles));
    bf16* h = cc.take<bf16>(static_cast<size_t>(T) * I);
    const cudaStream_t st = stream;
    rc = BEAM_MOE_OK;
    if ((e = maybe_poison(mem, bytes, st)) != cudaSuccess) {
        rc = fail(BEAM_MOE_ERR_CUDA, "scratch poison: %s", cudaGetErrorString(e));
        goto done;
    }
    LAUNCH(kCount, launch_dense_tiles(T, bn_max, tiles, tile_done, st));
    LAUNCH(kExpert, launch_expert_mlp(s, w_gate, w_up, w_down, x, T, tiles, tile_done, max_tiles, bn_max, h, out,
                                      dev->status, dev->num_sms, st));
done:
    e = cudaFreeAsync(mem, stream);
    if (rc == BEAM_MOE_OK && e != cudaSuccess)
        rc = fail(BEAM_MOE_ERR_CUDA, "scratch release: %s", cudaGetErrorString(e));
    return rc;
}

int beam_moe_selftest_wait_timeout(cudaStream_t stream) {
    g_launches = 0;
    timing_begin_call();
    int rc;
    if ((rc = check_stream(stream))) return rc;
    DeviceState* dev = nullptr;
    if ((rc = device_state(&dev))) return rc;
    // One expert of d = I = 128, one N-tile of 16 of 32 rows: one gate/up item, one down item.
    const Shape s{128, 128, 1, 1, 1, 1, 1.0f};
    const int rows = 32, T = 16, bn_max = 32;
    const int max_tiles = dense_max_tiles(T, bn_max);
    Carver c{nullptr};
    c.take<bf16>(3 * 128 * 128);
    c.take<bf16>(3 * static_cast<size_t>(rows) * 128);
    c.take<int4>(1 + static_cast<size_t>(max_tiles));
    c.take<int>(static_cast<size_t>(max_tiles));
    const size_t bytes = c.off + 256;
    void* mem = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&mem, bytes, dev->pool, stream);
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "scratch allocation of %zu bytes: %s", bytes, cudaGetErrorString(e));
    Carver cc{static_cast<char*>(mem)};
    bf16* w = cc.take<bf16>(3 * 128 * 128);
    bf16* act = cc.take<bf16>(3 * static_cast<size_t>(rows) * 128);
    int4* tiles = cc.take<int4>(1 + static_cast<size_t>(max_tiles));
    int* tile_done = cc.take<int>(static_cast<size_t>(max_tiles));
    const cudaStream_t st = stream;
    rc = BEAM_MOE_OK;
    if ((e = cudaMemsetAsync(mem, 0, bytes, st)) != cudaSuccess) {
        rc = fail(BEAM_MOE_ERR_CUDA, "scratch clear: %s", cudaGetErrorString(e));
        goto done;
    }
    LAUNCH(kCount, launch_dense_tiles(T, bn_max, tiles, tile_done, st));
    // The tile's completion counter starts far below zero, so the gate/up epilogue can never
    // raise it to the count the down item waits for.
    if ((e = cudaMemsetAsync(tile_done, 0x80, sizeof(int), st)) != cudaSuccess) {
        rc = fail(BEAM_MOE_ERR_CUDA, "counter poison: %s", cudaGetErrorString(e));
        goto done;
    }
    LAUNCH(kExpert, launch_expert_mlp(s, w, w + 128 * 128, w + 2 * 128 * 128, act, rows, tiles, tile_done, max_tiles,
                                      bn_max, act + rows * 128, act + 2 * rows * 128, dev->status, dev->num_sms, st));
done:
    e = cudaFreeAsync(mem, stream);
    if (rc == BEAM_MOE_OK && e != cudaSuccess)
        rc = fail(BEAM_MOE_ERR_CUDA, "scratch release: %s", cudaGetErrorString(e));
    return rc;
}

int beam_moe_rmsnorm(int d, const __nv_bfloat16* v, const __nv_bfloat16* gamma, float eps, int T,
                     __nv_bfloat16* out, cudaStream_t stream) {
    g_launches = 0;
    timing_begin_call();
    int rc;
    if (d < 4 || d % 4 || d > kNormMaxD) return fail(BEAM_MOE_ERR_ARG, "d=%d must be a multiple of 4 in [4, %d]", d, kNormMaxD);
    if ((rc = check_T(T)) || (rc = check_ptr(v, "v")) || (rc = check_ptr(gamma, "gamma")) ||
        (rc = check_ptr(out, "out")))
        return rc;
    if (!(eps >= 0.f) || !std::isfinite(eps)) return fail(BEAM_MOE_ERR_ARG, "eps must be finite and >= 0");
    if (T == 0) return BEAM_MOE_OK;
    if ((rc = check_stream(stream))) return rc;
    const cudaError_t e = launch_rmsnorm(d, v, gamma, eps, T, out, stream);
    ++g_launches;
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "launch of rmsnorm failed: %s", cudaGetErrorString(e));
    return BEAM_MOE_OK;
}

int beam_moe_router_logits(const beam_moe_config* cfg, const __nv_bfloat16* x, const float* router_w, int T,
                           float* logits, cudaStream_t stream) {
    return run(cfg, x, router_w, nullptr, nullptr, nullptr, nullptr, T, nullptr, nullptr, logits, nullptr, 1, stream);
}

const char* beam_moe_last_error(void) { return g_err; }

int beam_moe_device_status(cudaStream_t stream) {
    int rc;
    if ((rc = check_stream(stream))) return rc;
    DeviceState* dev = nullptr;
    if ((rc = device_state(&dev))) return rc;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    int word = 0;
    if ((e = cudaMemcpy(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail(BEAM_MOE_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
    if (word == kStatusOk) return BEAM_MOE_OK;
    cudaMemset(dev->status, 0, sizeof word);
    return fail(BEAM_MOE_ERR_DEVICE, "kernel status %d (%s)", word,
                word == kStatusBadExpert    ? "expert index out of range in dispatch"
                : word == kStatusWaitTimeout ? "a GEMM pipeline wait ran past its limit"
                : word == kStatusBadIndex    ? "a permuted row or work-list index out of range (access skipped)"
                : word == kStatusRange       ? "an NVFP4 activation block above 2688 in magnitude (clamped)"
                                             : "unknown");
}

int beam_moe_timing_enable(int enable) {
    g_timing.enabled = enable != 0;
    return BEAM_MOE_OK;
}

int beam_moe_timing_read(float* ms, int max_stages) {
    if (!ms || max_stages < 0) return fail(BEAM_MOE_ERR_ARG, "bad timing buffer");
    if (g_timing.last) {
        cudaError_t e = cudaEventSynchronize(g_timing.last);
        if (e != cudaSuccess) return fail(BEAM_MOE_ERR_CUDA, "event synchronize: %s", cudaGetErrorString(e));
    }
    for (int i = 0; i < max_stages && i < kNumStages; ++i) {
        float v = 0.f;
        if (g_timing.ran[i] && cudaEventElapsedTime(&v, g_timing.start[i], g_timing.stop[i]) != cudaSuccess) v = 0.f;
        ms[i] = v;
    }
    return kNumStages;
}

int beam_moe_last_launch_count(void) { return g_launches; }

int beam_moe_debug_poison_scratch(int enable) {
    g_poison.store(enable ? 1 : 0, std::memory_order_relaxed);
    return BEAM_MOE_OK;
}

}  // extern "C"
