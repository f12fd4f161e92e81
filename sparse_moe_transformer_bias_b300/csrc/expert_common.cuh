// Pieces shared by the persistent expert kernels (expert_mlp.cu: BF16 weights;
// expert_mlp_fp8.cu: FP8 tensor-core products; expert_mlp_nvf4.cu: block-scaled FP4
// tensor-core products): the kernel arguments, the work-item
// decoding of the dispatch work list, the bounded cross-CTA wait and the host-side
// argument and grid helpers.
#pragma once
#include "internal.cuh"
#include "ptx.cuh"

namespace beam {
namespace mlp {

constexpr int kEpiWarps = 8;
constexpr int kRing = 4;  // item ids in flight between the scheduler and the other roles
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

struct MlpArgs {
    const int4* tiles;   // header int4 {tile count, next item id, 0, 0}, then per N-tile
                         // {e, row0, rows, index among the expert's tiles | their count << 16}
    int* next_item;      // = &tiles[0].y, zeroed by dispatch for every call
    int* tile_done;      // [max_tiles] gate/up items finished per tile, zeroed by dispatch
    int max_tiles;
    int n_experts;
    int rows;            // permuted rows (x_perm, h, y)
    int m_gu, m_dn;      // items per tile: I / 128 gate/up items, ceil(d / 256) down items
    int kc_gu, kc_dn;    // K chunks: d / 64, I / 64
    int I, d;
    bf16* h;
    bf16* y;             // [rows, d] expert outputs (the dense MLP: its output)
    const float* gs;     // FP8 weights: per-row scales of Wg, Wu [E, I] and Wd [E, d];
                         // NVFP4 weights: the tensor scales of Wg, Wu and Wd [E]
    const float* us;
    const float* ds;
    // FP8 tensor-core products only (null otherwise): token of each permuted row, the
    // largest |x| of each token, and the largest |h| of each permuted row (zeroed before
    // the launch, raised by the gate/up epilogues)
    const int* perm_src;
    const float* xmax;
    float* amax_h;
    int n_tokens;        // T (bounds the tokens perm_src names)
    int* status;
};

struct MItem {
    int4 tl;     // {expert, first row, rows, 0}
    int tile;
    int m;
    int n_t;     // N-tiles of the item's expert
    bool down;
    bool ok;
};

// Item id -> (N-tile, weight tile m). The ids of one expert's n_t consecutive N-tiles
// (first .. first + n_t - 1) are [first * mt, (first + n_t) * mt), taken m-major.
__device__ __forceinline__ MItem decode(const MlpArgs& a, int id, int n_gu, int n_tiles) {
    MItem it;
    it.down = id >= n_gu;
    const int j = it.down ? id - n_gu : id;
    const int mt = it.down ? a.m_dn : a.m_gu;
    const int tg = j / mt;  // a tile of the right expert
    const int w = a.tiles[1 + tg].w;
    const int t_in = w & 0xffff, n_t = (w >> 16) & 0xffff;
    const int first = tg - t_in;
    bool ok = n_t >= 1 && t_in < n_t && first >= 0 && first + n_t <= n_tiles;
    it.n_t = n_t;
    if (ok) {
        const int local = j - first * mt;
        it.m = local / n_t;
        it.tile = first + local % n_t;
    } else {
        it.m = 0;
        it.tile = tg;
    }
    const int4 tl = a.tiles[1 + it.tile];
    it.tl = tl;
    it.ok = ok && !(tl.x < 0 || tl.x >= a.n_experts || tl.z <= 0 || tl.z > 256 || tl.y < 0 || tl.y > a.rows - tl.z);
    return it;
}

__device__ __forceinline__ void flag_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *counter >= need (another CTA's gate/up epilogues raise it).
__device__ __forceinline__ bool wait_counter(const int* counter, int need, const volatile int* abort_flag) {
    if (ld_acquire_gpu(counter) >= need) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        __nanosleep(128);
        if (ld_acquire_gpu(counter) >= need) return true;
        if (*abort_flag) return false;
        if (ptx::globaltimer() - t0 > kWaitLimitNs) return false;
    }
}

inline MlpArgs mlp_args(const Shape& s, int rows, const int4* tiles, int* tile_done, int max_tiles, bf16* h, bf16* y,
                 int* status, int k_stage) {
    MlpArgs a;
    a.tiles = tiles;
    a.next_item = const_cast<int*>(reinterpret_cast<const int*>(tiles)) + 1;
    a.tile_done = tile_done;
    a.max_tiles = max_tiles;
    a.n_experts = s.E;
    a.rows = rows;
    a.m_gu = s.I / kTileM;
    a.m_dn = (s.d / kTileM + 1) / 2;
    a.kc_gu = s.d / k_stage;
    a.kc_dn = s.I / k_stage;
    a.I = s.I;
    a.d = s.d;
    a.h = h;
    a.y = y;
    a.gs = a.us = a.ds = nullptr;
    a.perm_src = nullptr;
    a.xmax = nullptr;
    a.amax_h = nullptr;
    a.n_tokens = 0;
    a.status = status;
    return a;
}

inline int mlp_grid(const MlpArgs& a, int max_tiles, int num_sms) {
    const long long items = static_cast<long long>(max_tiles) * (a.m_gu + a.m_dn);
    return static_cast<int>(items < num_sms ? (items < 1 ? 1 : items) : num_sms);
}


}  // namespace mlp
}  // namespace beam
