// The routed experts of the Beam MoE block as ONE persistent tcgen05 kernel (Glonce
// "Reflection releases Beam ...", Architecture paragraph: each expert a SwiGLU MLP of
// intermediate size 2,560 on hidden size 5,120; transformers "Beam" doc: SwiGLU activation
// in FP32):
//     h[rows, I] = silu(x_perm . Wg[e]^T) * (x_perm . Wu[e]^T)      gate/up items
//     y[rows, d] = h . Wd[e]^T                                       down items
// per N-tile of the dispatch work list (rows of one expert, at most kBNMax).
//
// Work items, all "weights as M" (128 weight rows x the tile's token rows):
//   gate/up item (tile, m), m < I/128: two accumulators (gate, up) share the token rows;
//          the epilogue computes silu(g) * u in FP32 and stores BF16 h;
//   down item (tile, p), p < d/256: two accumulators for the weight tiles 2p and 2p+1
//          (two adjacent 128-row tiles of Wd) sharing the h rows; the epilogue rounds the
//          FP32 accumulators to BF16 y (the expert output, in the model's dtype).
// So every item streams two 128-row weight tiles against one set of token rows per K
// step and fills the same stage layout.
// Item ids run over every gate/up item, then every down item; CTAs take the next id from
// an atomic counter (dynamic scheduling), so no SM idles while work is left and the down
// items start on SMs that finish gate/up work early, with no kernel boundary between the
// two products. Within one expert the ids run m-major over the expert's N-tiles (the items
// of weight tile m for every N-tile of the expert, then m + 1, ...): an expert with more
// rows than one N-tile holds has its N-tiles' items of the same weight tile handed out
// together, so the CTAs running them stream those weights at the same time and the
// repeats are served by L2 instead of HBM (those weight loads carry the normal L2
// priority; weights read once carry evict-first).
// A down item of tile n reads h rows that the gate/up items of tile n write: each
// epilogue warp of a gate/up item increments tile_done[n] after its stores, and the
// producer of a down item waits (bounded) until tile_done[n] counts every warp of every
// gate/up item of the tile. All gate/up ids are handed out before any down id, and a
// producer only waits after it has issued every copy of its earlier items, so the MMAs
// and epilogues that raise the counts never wait on it: the waits always end.
// Every item writes its own output tile and sums its whole K range in a fixed order, so
// the result does not depend on which CTA runs which item.
//
// Roles (one CTA per SM):
//   warp 0 lane 0: scheduler + TMA producer: takes item ids, publishes them to the other
//                  roles through a shared-memory ring, and streams per 64-wide K chunk the
//                  weight tile(s) [128 x 64] and the tile's token rows (in the fewest
//                  power-of-two boxes) into a ring of stages;
//   warp 1:        allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=rows rounded up
//                  to 16, K=16) and tcgen05.commit;
//   warps 2..9:    epilogue - tcgen05.ld of their TMEM lane quarter, two warps per quarter
//                  taking alternate 16-column granules.
// TMEM is a ring of accumulator slots of kBNMax columns; every item takes two, so with
// four slots (kBNMax <= 128) the epilogue of one item overlaps the MMAs of the next (two
// slots at 192 and 256 rows).
// Every wait is bounded (2 s); on expiry the CTA records kStatusWaitTimeout, the roles
// leave their loops, copies and MMAs already issued are drained (bounded), and TMEM is
// freed before the CTA exits.

#include "expert_common.cuh"

namespace beam {
namespace {

using namespace mlp;

constexpr int kThreads = 64 + 32 * kEpiWarps;
template <int kBNMax>
struct MlpCfg {
    static constexpr int kKStage = kTileK;                     // K per stage
    static constexpr int kA = kTileM * kKStage * 2;            // one weight tile: 16 KB
    static constexpr int kBHalf = kBNMax * kTileK * 2;         // token rows x 64 of K (one swizzle row)
    static constexpr int kB = kBHalf;
    static constexpr int kStage = 2 * kA + kB;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int kStages = (kBudget / kStage) > 10 ? 10 : (kBudget / kStage);
    static constexpr int kSlots = ((512 / kBNMax) < 4 ? (512 / kBNMax) : 4) & ~1;  // items take pairs
    static constexpr int kColsNeeded = kSlots * kBNMax;
    static constexpr int kTmemCols = kColsNeeded <= 32    ? 32
                                     : kColsNeeded <= 64  ? 64
                                     : kColsNeeded <= 128 ? 128
                                     : kColsNeeded <= 256 ? 256
                                                          : 512;
    // FULL, EMPTY per stage; TFULL, TEMPTY per slot; RFULL, REMPTY per ring entry; DRAIN.
    static constexpr int kNumBars = 2 * kStages + 2 * kSlots + 2 * kRing + 1;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kNumBars * 8 + kRing * 4 + 16;
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kSlots >= 2 && kSlots % 2 == 0, "an item takes two accumulator slots");
    static_assert(kColsNeeded <= 512, "TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
};

template <int kBNMax>
__global__ void __launch_bounds__(kThreads, 1)
    expert_mlp_kernel(const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
                      const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ BMaps tmX,
                      const __grid_constant__ BMaps tmH, const __grid_constant__ MlpArgs args) {
    using C = MlpCfg<kBNMax>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
    volatile int* ring = reinterpret_cast<volatile int*>(bars + C::kNumBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    constexpr int FULL0 = 0, EMPTY0 = C::kStages, TFULL0 = 2 * C::kStages, TEMPTY0 = TFULL0 + C::kSlots,
                  RFULL0 = TEMPTY0 + C::kSlots, REMPTY0 = RFULL0 + kRing, DRAIN = REMPTY0 + kRing;
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };
    int* status = args.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(bar(FULL0 + s), 1);
            ptx::mbar_init(bar(EMPTY0 + s), 1);
        }
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(bar(TFULL0 + s), 1);
            ptx::mbar_init(bar(TEMPTY0 + s), 32 * kEpiWarps);
        }
        for (int r = 0; r < kRing; ++r) {
            ptx::mbar_init(bar(RFULL0 + r), 1);
            ptx::mbar_init(bar(REMPTY0 + r), 1 + kEpiWarps);
        }
        ptx::mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmWg);
        ptx::prefetch_tmap(&tmWu);
        ptx::prefetch_tmap(&tmWd);
        for (int i = 0; i < kBoxKinds && (kBoxRows << i) <= kBNMax; ++i) {
            ptx::prefetch_tmap(&tmX.m[i]);
            ptx::prefetch_tmap(&tmH.m[i]);
        }
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    pdl_wait();  // the prologue above touches no global memory
    pdl_trigger();
    int n_tiles = args.tiles[0].x;
    if (n_tiles < 0 || n_tiles > args.max_tiles) {
        if (threadIdx.x == 0) flag_status(status, kStatusBadIndex);
        n_tiles = 0;
    }
    const int n_gu = n_tiles * args.m_gu;
    const int n_total = n_gu + n_tiles * args.m_dn;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ scheduler + TMA producer
            // Weights of an expert with one N-tile are read once: evict first. An expert
            // with several N-tiles has its weight tiles streamed by several CTAs at about
            // the same time (m-major ids): normal priority, so that the others hit L2.
            const uint64_t pol_w_once = ptx::policy_evict_first();
            const uint64_t pol_w_shared = ptx::policy_evict_normal();
            const uint64_t pol_x = ptx::policy_evict_last();
            int stage = 0, rslot = 0;
            uint32_t phase = 0, rphase = 0;
            uint32_t issued = 0, parity = 0;  // per stage: ever loaded / parity of the last load
            bool ok = true;
            int next = atomicAdd(args.next_item, 1);
            while (ok) {
                const int id = next < n_total ? next : -1;
                if (id >= 0) next = atomicAdd(args.next_item, 1);  // used at the next iteration
                if (!ptx::mbar_wait(bar(REMPTY0 + rslot), rphase ^ 1, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ring[rslot] = id;
                ptx::mbar_arrive(bar(RFULL0 + rslot));  // release: the id is visible to the waiters
                if (++rslot == kRing) {
                    rslot = 0;
                    rphase ^= 1;
                }
                if (id < 0) break;
                const MItem it = decode(args, id, n_gu, n_tiles);
                if (!it.ok || it.tl.z > kBNMax) {
                    flag_status(status, kStatusBadIndex);
                    continue;
                }
                if (it.down) {
                    // the h rows of this tile come from the tile's gate/up items
                    if (!wait_counter(args.tile_done + it.tile, args.m_gu * kEpiWarps, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();  // order the copies below after that observation
                }
                const int b_rows = ((it.tl.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t bytes = 2 * C::kA + b_rows * C::kKStage * 2;
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                const int a_row = it.down ? it.tl.x * args.d + it.m * 2 * kTileM : it.tl.x * args.I + it.m * kTileM;
                const BMaps& bm = it.down ? tmH : tmX;
                const uint64_t pol_w = it.n_t > 1 ? pol_w_shared : pol_w_once;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    const int kx = kc * C::kKStage;  // K of the stage, in elements
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes);
                    if (it.down) {
                        // rows past the expert's last tile (d not a multiple of 256) belong to
                        // the next expert or lie past the end (zero fill); never stored
                        ptx::tma_load_2d(sa, &tmWd, kx, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWd, kx, a_row + kTileM, bar(FULL0 + stage), pol_w);
                    } else {
                        ptx::tma_load_2d(sa, &tmWg, kx, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWu, kx, a_row, bar(FULL0 + stage), pol_w);
                    }
                    const uint32_t sb = sa + 2 * C::kA;
#pragma unroll
                    for (int half = 0; half < C::kKStage / kTileK; ++half) {
                        for (int i = kBoxKinds - 1, r = 0; i >= 0; --i) {
                            const int hh = kBoxRows << i;
                            if (hh > kBNMax || b_rows - r < hh) continue;
                            ptx::tma_load_2d(sb + half * C::kBHalf + r * kTileK * 2, &bm.m[i], kx + half * kTileK,
                                             it.tl.y + r, bar(FULL0 + stage), pol_x);
                            r += hh;
                        }
                    }
                    issued |= 1u << stage;
                    parity = (parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                flag_status(status, kStatusWaitTimeout);
                const int never = 0;
                for (int s = 0; s < C::kStages; ++s)
                    if ((issued >> s) & 1u) ptx::mbar_wait(bar(FULL0 + s), (parity >> s) & 1u, &never, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            int stage = 0, rslot = 0, slot = 0;
            uint32_t phase = 0, rphase = 0, tph = 0;  // tph bit s: parity of slot s's current use
            bool ok = true;
            while (ok) {
                if (!ptx::mbar_wait(bar(RFULL0 + rslot), rphase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const int id = ring[rslot];
                ptx::mbar_arrive(bar(REMPTY0 + rslot));
                if (++rslot == kRing) {
                    rslot = 0;
                    rphase ^= 1;
                }
                if (id < 0) break;
                const MItem it = decode(args, id, n_gu, n_tiles);
                if (!it.ok || it.tl.z > kBNMax) continue;
                const int s0 = slot, s1 = (slot + 1) % C::kSlots;
                if (!ptx::mbar_wait(bar(TEMPTY0 + s0), ((tph >> s0) & 1u) ^ 1u, abort_flag, kWaitLimitNs) ||
                    !ptx::mbar_wait(bar(TEMPTY0 + s1), ((tph >> s1) & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t idesc = ptx::idesc_bf16_f32(kTileM, ((it.tl.z + 15) / 16) * 16);
                const uint32_t d0 = tmem_base + s0 * kBNMax, d1 = tmem_base + s1 * kBNMax;
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    const uint32_t sb = sa + 2 * C::kA;
                    constexpr int kPerRow = kTileK / kMmaK;  // K steps per 128-byte swizzle row
#pragma unroll
                    for (int kk = 0; kk < C::kKStage / kMmaK; ++kk) {
                        const uint64_t bdesc =
                            ptx::sw128_kmajor_desc(sb + (kk / kPerRow) * C::kBHalf + (kk % kPerRow) * kMmaK * 2);
                        const uint32_t accum = (kc | kk) ? 1u : 0u;
                        ptx::mma_bf16(d0, ptx::sw128_kmajor_desc(sa + kk * kMmaK * 2), bdesc, idesc, accum);
                        ptx::mma_bf16(d1, ptx::sw128_kmajor_desc(sa + C::kA + kk * kMmaK * 2), bdesc, idesc, accum);
                    }
                    ptx::mma_commit(bar(EMPTY0 + stage));
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bar(TFULL0 + s0));
                ptx::mma_commit(bar(TFULL0 + s1));
                tph ^= (1u << s0) | (1u << s1);
                slot = (slot + 2) % C::kSlots;
            }
            if (!ok) {
                *abort_flag = 1;
                flag_status(status, kStatusWaitTimeout);
                const int never = 0;
                ptx::mma_commit(bar(DRAIN));
                ptx::mbar_wait(bar(DRAIN), 0, &never, kDrainLimitNs);
            }
        }
    } else if (warp >= 2) {
        // ---------------------------------------------------------------- epilogue    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;                      // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;               // weight row within the M-tile
        const int col_part = (warp - 2) >> 2;        // which 16-column granules this warp takes
        constexpr int kColStep = 16 * (kEpiWarps / 4);
        int rslot = 0, slot = 0;
        uint32_t rphase = 0, tph = 0;
        while (true) {
            if (!ptx::mbar_wait(bar(RFULL0 + rslot), rphase, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                flag_status(status, kStatusWaitTimeout);
                break;
            }
            const int id = ring[rslot];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(REMPTY0 + rslot));
            if (++rslot == kRing) {
                rslot = 0;
                rphase ^= 1;
            }
            if (id < 0) break;
            const MItem it = decode(args, id, n_gu, n_tiles);
            if (!it.ok || it.tl.z > kBNMax) continue;
            const int s0 = slot, s1 = (slot + 1) % C::kSlots;
            if (!ptx::mbar_wait(bar(TFULL0 + s0), (tph >> s0) & 1u, abort_flag, kWaitLimitNs) ||
                !ptx::mbar_wait(bar(TFULL0 + s1), (tph >> s1) & 1u, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                flag_status(status, kStatusWaitTimeout);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
            const uint32_t t0 = tmem_base + lane_off + s0 * kBNMax, t1 = tmem_base + lane_off + s1 * kBNMax;
            const int col = (it.down ? it.m * 2 * kTileM : it.m * kTileM) + row;
            const bool col1_ok = col + kTileM < args.d;  // down: the pair's second tile exists
            for (int c0 = col_part * 16; c0 < it.tl.z; c0 += kColStep) {
                uint32_t g[16];
                ptx::tmem_ld16(t0 + c0, g);
                if (!it.down) {
                    uint32_t u[16];
                    ptx::tmem_ld16(t1 + c0, u);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < it.tl.z) {
                            const float gv = __uint_as_float(g[j]);
                            const float uv = __uint_as_float(u[j]);
                            // silu(g) * u in FP32 with the fast exponential and division
                            // (a few ulp; the result is rounded to BF16 next)
                            const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                            args.h[static_cast<size_t>(it.tl.y + c0 + j) * args.I + col] = __float2bfloat16_rn(hv);
                        }
                    }
                } else {
                    uint32_t g1[16];
                    ptx::tmem_ld16(t1 + c0, g1);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < it.tl.z) {
                            const size_t r0 = static_cast<size_t>(it.tl.y + c0 + j) * args.d;
                            const float y0 = __uint_as_float(g[j]), y1 = __uint_as_float(g1[j]);
                            args.y[r0 + col] = __float2bfloat16_rn(y0);
                            if (col1_ok) args.y[r0 + col + kTileM] = __float2bfloat16_rn(y1);
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(TEMPTY0 + s0));
            ptx::mbar_arrive(bar(TEMPTY0 + s1));
            tph ^= (1u << s0) | (1u << s1);
            if (!it.down) {
                // Publish this warp's h stores to the down items of the tile (other CTAs
                // read them with TMA): each writer orders its stores for the async proxy,
                // the warp meets, and lane 0 releases one count (kEpiWarps per item).
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(args.tile_done + it.tile, 1);
                }
            }
            slot = (slot + 2) % C::kSlots;
        }
    }

    __syncwarp();
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

template <int kBNMax>
cudaError_t launch_mlp(const CUtensorMap& wg, const CUtensorMap& wu, const CUtensorMap& wd, const BMaps& x,
                       const BMaps& h, const MlpArgs& args, int grid, cudaStream_t st) {
    using C = MlpCfg<kBNMax>;
    cudaError_t e = set_smem_limit_once<expert_mlp_kernel<kBNMax>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const cudaError_t le_ =
        launch_pdl(expert_mlp_kernel<kBNMax>, dim3(grid), dim3(kThreads), C::kSmemBytes, st, wg, wu, wd, x, h, args);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

}  // namespace

// N-tile capacity for a batch of T tokens: 32 for decode-sized batches; 128 while the
// average expert gets at most 32 rows (one tile holds nearly every expert's rows, and the
// smaller B stage leaves room for more stages and four accumulator slots); 192 while it
// gets at most 160 (stages of 56 KB: four in flight instead of three of 64 KB, which more
// than pays for the experts split over two tiles); else 256, so that a weight tile is
// streamed once for up to 256 of its expert's rows.
int gemm_bn_max(const Shape& s, int T) {
    if (T <= 32) return 32;
    const long long avg_rows = static_cast<long long>(T) * s.top_k / s.E;
    return avg_rows <= 32 ? 128 : avg_rows <= 160 ? 192 : 256;
}

namespace {

// Work list of one "expert" holding every token in order (the dense MLP): N-tiles of at
// most bn_max rows, split evenly like dispatch does; counters zeroed.
__global__ void __launch_bounds__(256) dense_tiles_kernel(int T, int bn_max, int4* __restrict__ tiles,
                                                          int* __restrict__ tile_done) {
    pdl_wait();
    pdl_trigger();
    const int q = (T + bn_max - 1) / bn_max;
    const int per = min(bn_max, (((T + q - 1) / q + 15) / 16) * 16);
    const int nt = (T + per - 1) / per;
    for (int i = threadIdx.x; i < nt; i += blockDim.x) {
        tiles[1 + i] = make_int4(0, i * per, min(per, T - i * per), i | (nt << 16));
        tile_done[i] = 0;
    }
    if (threadIdx.x == 0) tiles[0] = make_int4(nt, 0, 0, 0);
}

}  // namespace

int dense_max_tiles(int T, int bn_max) { return T / bn_max + 2; }

cudaError_t launch_dense_tiles(int T, int bn_max, int4* tiles, int* tile_done, cudaStream_t st) {
    const cudaError_t le_ = launch_pdl(dense_tiles_kernel, dim3(1), dim3(256), 0, st, T, bn_max, tiles, tile_done);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

using mlp::mlp_args;
using mlp::mlp_grid;

cudaError_t launch_expert_mlp(const Shape& s, const bf16* w_gate, const bf16* w_up, const bf16* w_down,
                              const bf16* x_perm, int rows, const int4* tiles, int* tile_done, int max_tiles,
                              int bn_max, bf16* h, bf16* y, int* status, int num_sms,
                              cudaStream_t st) {
    CUtensorMap wg, wu, wd;
    BMaps bx, bh;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&wg, w_gate, static_cast<uint64_t>(s.E) * s.I, s.d, kTileM, kTileK, &why) ||
        !encode_tmap_bf16_2d(&wu, w_up, static_cast<uint64_t>(s.E) * s.I, s.d, kTileM, kTileK, &why) ||
        !encode_tmap_bf16_2d(&wd, w_down, static_cast<uint64_t>(s.E) * s.d, s.I, kTileM, kTileK, &why) ||
        !encode_bmaps(&bx, x_perm, rows, s.d, bn_max, &why) || !encode_bmaps(&bh, h, rows, s.I, bn_max, &why))
        return cudaErrorInvalidValue;
    const MlpArgs a = mlp_args(s, rows, tiles, tile_done, max_tiles, h, y, status, kTileK);
    const int grid = mlp_grid(a, max_tiles, num_sms);
    if (bn_max <= 32) return launch_mlp<32>(wg, wu, wd, bx, bh, a, grid, st);
    if (bn_max <= 128) return launch_mlp<128>(wg, wu, wd, bx, bh, a, grid, st);
    if (bn_max <= 192) return launch_mlp<192>(wg, wu, wd, bx, bh, a, grid, st);
    return launch_mlp<256>(wg, wu, wd, bx, bh, a, grid, st);
}

}  // namespace beam
