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
//
// NVFP4 weights (kFP4): E2M1 codes packed two per byte, one E4M3 scale per 16 elements of
// a row, one FP32 scale per expert matrix. No tensor-core product takes E2M1 weights with
// E4M3 block scales against 16-bit activations, so the weights are widened on chip: a stage
// covers K = 256: TMA streams the code tiles [128 rows x 128 bytes] (128-byte swizzle), the
// block-scale tiles [128 rows x 16 bytes] and the token rows as four 64-wide BF16 quarters;
// eight converter warps (two per TMEM lane quarter, one per weight tile of the stage) turn
// each row's codes into BF16 and store them with tcgen05.st into a ring of A buffers in
// TMEM (K = 128 per buffer), and the MMA reads A from TMEM (B, the token rows, from shared
// memory). The widening is exact: a code pair -> F16 pair by cvt, times its block scale as
// an F16 pair (E2M1 has 2 significant bits and E4M3 4, so the product has at most 6 and
// lies in [2^-10, 2688]: an exact F16 normal or zero), then F16 -> BF16 by moving the
// exponent and mantissa bits down three places, which keeps every bit and multiplies the
// value by 2^-112. The epilogue multiplies each accumulator by 2^112 and by the matrix's
// tensor scale, so the products are those of W[r][c] = t * e4m3(bs[r][c/16]) * e2m1(q[r][c])
// with FP32 accumulation.
#include <cstring>

#include "expert_common.cuh"

namespace beam {
namespace {

using namespace mlp;

constexpr int kConvWarps = 8;  // NVFP4 weights: two converter warps per TMEM lane quarter
constexpr int kThreadsFor(bool fp4) { return 64 + 32 * kEpiWarps + (fp4 ? 32 * kConvWarps : 0); }
template <int kBNMax, bool kFP4>
struct MlpCfg {
    static constexpr int kThreads = kThreadsFor(kFP4);
    static constexpr int kKStage = kFP4 ? 4 * kTileK : kTileK;  // K per stage
    static constexpr int kA = kTileM * (kFP4 ? kKStage / 2 : kKStage * 2);  // one weight tile: 16 KB
    static constexpr int kS = kFP4 ? kTileM * (kKStage / 16) : 0;         // its block scales: 2 KB
    static constexpr int kBHalf = kBNMax * kTileK * 2;          // token rows x 64 of K (one swizzle row)
    static constexpr int kB = kBHalf * (kKStage / kTileK);
    static constexpr int kStage = 2 * kA + 2 * kS + kB;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int kStages = (kBudget / kStage) > 10 ? 10 : (kBudget / kStage);
    // NVFP4: a ring of converted A buffers in TMEM after the accumulator slots. A buffer
    // holds K = 128 of the stage's two weight tiles as BF16 (2 x 64 columns); two per stage.
    static constexpr int kAParts = kFP4 ? 2 : 1;
    static constexpr int kAK = kKStage / kAParts;
    static constexpr int kACols = kFP4 ? kAK : 0;
    static constexpr int kABufs = kFP4 ? (kBNMax <= 32 ? 3 : 2) : 0;
    static constexpr int kAccCols = 512 - kABufs * kACols;
    static constexpr int kSlots = ((kAccCols / kBNMax) < 4 ? (kAccCols / kBNMax) : 4) & ~1;  // items take pairs
    static constexpr int kABase = kSlots * kBNMax;  // first TMEM column of the A buffers
    static constexpr int kColsNeeded = kSlots * kBNMax + kABufs * kACols;
    static constexpr int kTmemCols = kColsNeeded <= 32    ? 32
                                     : kColsNeeded <= 64  ? 64
                                     : kColsNeeded <= 128 ? 128
                                     : kColsNeeded <= 256 ? 256
                                                          : 512;
    // FULL, EMPTY per stage; TFULL, TEMPTY per slot; RFULL, REMPTY per ring entry; DRAIN;
    // AFULL, AEMPTY per A buffer.
    static constexpr int kNumBars = 2 * kStages + 2 * kSlots + 2 * kRing + 1 + 2 * kABufs;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kNumBars * 8 + kRing * 4 + 16;
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kSlots >= 2 && kSlots % 2 == 0, "an item takes two accumulator slots");
    static_assert(kColsNeeded <= 512 && kABase + kABufs * kACols <= 512, "TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
};

// NVFP4 block-scale tiles (E4M3 codes [rows, cols / 16], boxes of 128 rows x 16 bytes) of
// the gate, up and down matrices (unused for BF16 weights).
struct ScaleMaps {
    CUtensorMap g, u, d;
};

// Four NVFP4 code bytes (8 E2M1 codes, element 2k in the low half of byte k) of one block
// with block scale `scale2` (the E4M3 scale as an F16 pair (s, s)) -> four words of two
// BF16 each (the lower element in the lower half), every value times 2^-112 exactly.
__device__ __forceinline__ void e2m1x8_to_bf16x8_scaled(uint32_t w, uint32_t scale2, uint32_t (&o)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t f;
        asm("{\n .reg .b8 c;\n .reg .b32 t;\n"
            " shr.u32 t, %1, %2;\n"
            " cvt.u8.u32 c, t;\n"
            " cvt.rn.f16x2.e2m1x2 %0, c;\n}\n"
            : "=r"(f)
            : "r"(w), "r"(8 * i));
        const __half2 p = __hmul2(*reinterpret_cast<const __half2*>(&f), *reinterpret_cast<const __half2*>(&scale2));
        const uint32_t v = *reinterpret_cast<const uint32_t*>(&p);
        o[i] = ((v & 0x7fff7fffu) >> 3) | (v & 0x80008000u);
    }
}

// An E4M3 block scale (one byte) as the F16 pair (s, s).
__device__ __forceinline__ uint32_t e4m3_scale_pair(uint32_t byte) {
    uint32_t f;
    const uint32_t two = byte | (byte << 8);
    asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}\n" : "=r"(f) : "r"(two));
    return f;
}

template <int kBNMax, bool kFP4>
__global__ void __launch_bounds__(kThreadsFor(kFP4), 1)
    expert_mlp_kernel(const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
                      const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ BMaps tmX,
                      const __grid_constant__ BMaps tmH, const __grid_constant__ ScaleMaps tmS,
                      const __grid_constant__ MlpArgs args) {
    using C = MlpCfg<kBNMax, kFP4>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
    volatile int* ring = reinterpret_cast<volatile int*>(bars + C::kNumBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    constexpr int FULL0 = 0, EMPTY0 = C::kStages, TFULL0 = 2 * C::kStages, TEMPTY0 = TFULL0 + C::kSlots,
                  RFULL0 = TEMPTY0 + C::kSlots, REMPTY0 = RFULL0 + kRing, DRAIN = REMPTY0 + kRing,
                  AFULL0 = DRAIN + 1, AEMPTY0 = AFULL0 + C::kABufs;
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };
    int* status = args.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(bar(FULL0 + s), 1);
            ptx::mbar_init(bar(EMPTY0 + s), kFP4 ? 1 + kConvWarps : 1);  // NVFP4: converters read it too
        }
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(bar(TFULL0 + s), 1);
            ptx::mbar_init(bar(TEMPTY0 + s), 32 * kEpiWarps);
        }
        for (int r = 0; r < kRing; ++r) {
            ptx::mbar_init(bar(RFULL0 + r), 1);
            ptx::mbar_init(bar(REMPTY0 + r), 1 + kEpiWarps + (kFP4 ? kConvWarps : 0));
        }
        ptx::mbar_init(bar(DRAIN), 1);
        for (int b = 0; b < C::kABufs; ++b) {
            ptx::mbar_init(bar(AFULL0 + b), kConvWarps);
            ptx::mbar_init(bar(AEMPTY0 + b), 1);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmWg);
        ptx::prefetch_tmap(&tmWu);
        ptx::prefetch_tmap(&tmWd);
        if constexpr (kFP4) {
            ptx::prefetch_tmap(&tmS.g);
            ptx::prefetch_tmap(&tmS.u);
            ptx::prefetch_tmap(&tmS.d);
        }
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
                const uint32_t bytes = 2 * C::kA + 2 * C::kS + b_rows * C::kKStage * 2;
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                const int a_row = it.down ? it.tl.x * args.d + it.m * 2 * kTileM : it.tl.x * args.I + it.m * kTileM;
                const BMaps& bm = it.down ? tmH : tmX;
                const uint64_t pol_w = it.n_t > 1 ? pol_w_shared : pol_w_once;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    const int kx = kc * C::kKStage;                // K of the stage, in elements
                    const int ax = kFP4 ? kx / 2 : kx;               // ... in units of the weight map
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes);
                    if (it.down) {
                        // rows past the expert's last tile (d not a multiple of 256) belong to
                        // the next expert or lie past the end (zero fill); never stored
                        ptx::tma_load_2d(sa, &tmWd, ax, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWd, ax, a_row + kTileM, bar(FULL0 + stage), pol_w);
                        if constexpr (kFP4) {
                            ptx::tma_load_2d(sa + 2 * C::kA, &tmS.d, kx / 16, a_row, bar(FULL0 + stage), pol_w);
                            ptx::tma_load_2d(sa + 2 * C::kA + C::kS, &tmS.d, kx / 16, a_row + kTileM, bar(FULL0 + stage),
                                             pol_w);
                        }
                    } else {
                        ptx::tma_load_2d(sa, &tmWg, ax, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWu, ax, a_row, bar(FULL0 + stage), pol_w);
                        if constexpr (kFP4) {
                            ptx::tma_load_2d(sa + 2 * C::kA, &tmS.g, kx / 16, a_row, bar(FULL0 + stage), pol_w);
                            ptx::tma_load_2d(sa + 2 * C::kA + C::kS, &tmS.u, kx / 16, a_row, bar(FULL0 + stage), pol_w);
                        }
                    }
                    const uint32_t sb = sa + 2 * C::kA + 2 * C::kS;
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
            int stage = 0, rslot = 0, slot = 0, abuf = 0;
            uint32_t phase = 0, rphase = 0, tph = 0, aphase = 0;  // tph bit s: parity of slot s's current use
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
                    const uint32_t sb = sa + 2 * C::kA + 2 * C::kS;
                    constexpr int kPerRow = kTileK / kMmaK;  // K steps per 128-byte swizzle row
                    if constexpr (kFP4) {
                        // kAParts A buffers per stage, each kAK of K
                        for (int part = 0; part < C::kAParts && ok; ++part) {
                            if (!ptx::mbar_wait(bar(AFULL0 + abuf), aphase, abort_flag, kWaitLimitNs)) {
                                ok = false;
                                break;
                            }
                            ptx::tc_fence_after();
                            const uint32_t ta0 = tmem_base + C::kABase + abuf * C::kACols;
#pragma unroll
                            for (int kk = 0; kk < C::kAK / kMmaK; ++kk) {
                                const int g = part * (C::kAK / kMmaK) + kk;  // K step within the stage
                                const uint64_t bdesc =
                                    ptx::sw128_kmajor_desc(sb + (g / kPerRow) * C::kBHalf + (g % kPerRow) * kMmaK * 2);
                                const uint32_t accum = (kc | g) ? 1u : 0u;
                                const uint32_t ta = ta0 + kk * (kMmaK / 2);
                                ptx::mma_bf16_ta(d0, ta, bdesc, idesc, accum);
                                ptx::mma_bf16_ta(d1, ta + C::kAK / 2, bdesc, idesc, accum);
                            }
                            ptx::mma_commit(bar(AEMPTY0 + abuf));
                            if (++abuf == C::kABufs) {
                                abuf = 0;
                                aphase ^= 1;
                            }
                        }
                        if (!ok) break;
                    } else {
#pragma unroll
                        for (int kk = 0; kk < C::kKStage / kMmaK; ++kk) {
                            const uint64_t bdesc =
                                ptx::sw128_kmajor_desc(sb + (kk / kPerRow) * C::kBHalf + (kk % kPerRow) * kMmaK * 2);
                            const uint32_t accum = (kc | kk) ? 1u : 0u;
                            ptx::mma_bf16(d0, ptx::sw128_kmajor_desc(sa + kk * kMmaK * 2), bdesc, idesc, accum);
                            ptx::mma_bf16(d1, ptx::sw128_kmajor_desc(sa + C::kA + kk * kMmaK * 2), bdesc, idesc,
                                          accum);
                        }
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
    } else if (warp >= 2 + kEpiWarps) {
        if constexpr (kFP4) {
            // ------------------------------------------------------------ NVFP4 -> BF16 converters
            // Warp pair per lane quarter: weight tile t (gate or the even Wd tile: 0; up or
            // the odd Wd tile: 1) of every stage, one weight row per thread.
            const int q = warp & 3;
            const int t = (warp - 2 - kEpiWarps) >> 2;
            const int r = q * 32 + lane;
            const int swz = r & 7;  // the 128-byte swizzle of the byte tile
            const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
            int stage = 0, rslot = 0, abuf = 0;
            uint32_t phase = 0, rphase = 0, aphase = 0;
            bool ok = true;
            while (ok) {
                if (!ptx::mbar_wait(bar(RFULL0 + rslot), rphase, abort_flag, kWaitLimitNs)) {
                    ok = false;
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
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    // this row's 256 codes (128 bytes, 128-byte swizzle) and 16 block scales
                    const uint8_t* src = smem + stage * C::kStage + t * C::kA + r * 128;
                    const uint4 sc16 = *reinterpret_cast<const uint4*>(smem + stage * C::kStage + 2 * C::kA + t * C::kS + r * 16);
                    const uint32_t scw[4] = {sc16.x, sc16.y, sc16.z, sc16.w};
                    for (int part = 0; part < C::kAParts; ++part) {  // one A buffer: K = 128 of the row
                        if (!ptx::mbar_wait(bar(AEMPTY0 + abuf), aphase ^ 1, abort_flag, kWaitLimitNs)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t dst = tmem_base + lane_off + C::kABase + abuf * C::kACols + t * (C::kAK / 2);
#pragma unroll
                        for (int sub = 0; sub < 2; ++sub) {  // 64 codes (two 16-byte chunks) -> 32 columns
                            uint32_t o[32];
#pragma unroll
                            for (int j = 0; j < 2; ++j) {
                                const int cc = 4 * part + 2 * sub + j;  // 16-byte chunk: blocks 2cc, 2cc + 1
                                const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * (cc ^ swz));
                                const uint32_t s0 = e4m3_scale_pair((scw[(2 * cc) >> 2] >> (8 * ((2 * cc) & 3))) & 0xffu);
                                const uint32_t s1 =
                                    e4m3_scale_pair((scw[(2 * cc + 1) >> 2] >> (8 * ((2 * cc + 1) & 3))) & 0xffu);
                                uint32_t w4[4];
                                e2m1x8_to_bf16x8_scaled(v.x, s0, w4);
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[16 * j + i] = w4[i];
                                e2m1x8_to_bf16x8_scaled(v.y, s0, w4);
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[16 * j + 4 + i] = w4[i];
                                e2m1x8_to_bf16x8_scaled(v.z, s1, w4);
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[16 * j + 8 + i] = w4[i];
                                e2m1x8_to_bf16x8_scaled(v.w, s1, w4);
#pragma unroll
                                for (int i = 0; i < 4; ++i) o[16 * j + 12 + i] = w4[i];
                            }
                            ptx::tmem_st32(dst + 32 * sub, o);
                        }
                        ptx::tmem_wait_st();
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(AFULL0 + abuf));
                        if (++abuf == C::kABufs) {
                            abuf = 0;
                            aphase ^= 1;
                        }
                    }
                    if (!ok) break;
                    if (lane == 0) ptx::mbar_arrive(bar(EMPTY0 + stage));  // this tile's codes are read
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok) {
                *abort_flag = 1;
                flag_status(status, kStatusWaitTimeout);
            }
        }
    } else {
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
            // NVFP4: the tensor scales of the expert's matrices, the 2^112 of the widening
            // applied first (exact)
            float sc0 = 1.0f, sc1 = 1.0f;
            if constexpr (kFP4) {
                if (!it.down) {
                    sc0 = args.gs[it.tl.x];
                    sc1 = args.us[it.tl.x];
                } else {
                    sc0 = args.ds[it.tl.x];
                    sc1 = col1_ok ? sc0 : 0.0f;
                }
            }
            constexpr float kP112 = 5.192296858534828e33f;  // 2^112
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
                            float gv = __uint_as_float(g[j]);
                            float uv = __uint_as_float(u[j]);
                            if constexpr (kFP4) {
                                gv = (gv * kP112) * sc0;
                                uv = (uv * kP112) * sc1;
                            }
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
                            float y0 = __uint_as_float(g[j]), y1 = __uint_as_float(g1[j]);
                            if constexpr (kFP4) {
                                y0 = (y0 * kP112) * sc0;
                                y1 = (y1 * kP112) * sc1;
                            }
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

template <int kBNMax, bool kFP4>
cudaError_t launch_mlp(const CUtensorMap& wg, const CUtensorMap& wu, const CUtensorMap& wd, const ScaleMaps& sm,
                       const BMaps& x, const BMaps& h, const MlpArgs& args, int grid, cudaStream_t st) {
    using C = MlpCfg<kBNMax, kFP4>;
    auto kern = expert_mlp_kernel<kBNMax, kFP4>;
    cudaError_t e = set_smem_limit_once<expert_mlp_kernel<kBNMax, kFP4>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const cudaError_t le_ =
        launch_pdl(kern, dim3(grid), dim3(C::kThreads), C::kSmemBytes, st, wg, wu, wd, x, h, sm, args);
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

int gemm_bn_max_fp4(const Shape& s, int T) {
    const int b = gemm_bn_max(s, T);
    return b < 128 ? b : 128;
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
    ScaleMaps none;
    memset(&none, 0, sizeof none);
    if (bn_max <= 32) return launch_mlp<32, false>(wg, wu, wd, none, bx, bh, a, grid, st);
    if (bn_max <= 128) return launch_mlp<128, false>(wg, wu, wd, none, bx, bh, a, grid, st);
    if (bn_max <= 192) return launch_mlp<192, false>(wg, wu, wd, none, bx, bh, a, grid, st);
    return launch_mlp<256, false>(wg, wu, wd, none, bx, bh, a, grid, st);
}

cudaError_t launch_expert_mlp_nvfp4(const Shape& s, const Nvfp4Experts& q, const bf16* x_perm, int rows,
                                    const int4* tiles, int* tile_done, int max_tiles, int bn_max, bf16* h, bf16* y,
                                    int* status, int num_sms, cudaStream_t st) {
    if (bn_max > 128 || s.d % 256 || s.I % 256) return cudaErrorInvalidValue;
    CUtensorMap wg, wu, wd;
    ScaleMaps sm;
    BMaps bx, bh;
    const char* why = nullptr;
    const uint64_t gu_rows = static_cast<uint64_t>(s.E) * s.I, dn_rows = static_cast<uint64_t>(s.E) * s.d;
    // codes: 128-byte boxes (256 elements of K); block scales: 16-byte boxes (16 blocks)
    if (!encode_tmap_u8_2d(&wg, q.wg, gu_rows, s.d / 2, kTileM, 128, &why) ||
        !encode_tmap_u8_2d(&wu, q.wu, gu_rows, s.d / 2, kTileM, 128, &why) ||
        !encode_tmap_u8_2d(&wd, q.wd, dn_rows, s.I / 2, kTileM, 128, &why) ||
        !encode_tmap_u8_2d_plain(&sm.g, q.gbs, gu_rows, s.d / 16, kTileM, 16, &why) ||
        !encode_tmap_u8_2d_plain(&sm.u, q.ubs, gu_rows, s.d / 16, kTileM, 16, &why) ||
        !encode_tmap_u8_2d_plain(&sm.d, q.dbs, dn_rows, s.I / 16, kTileM, 16, &why) ||
        !encode_bmaps(&bx, x_perm, rows, s.d, bn_max, &why) || !encode_bmaps(&bh, h, rows, s.I, bn_max, &why))
        return cudaErrorInvalidValue;
    MlpArgs a = mlp_args(s, rows, tiles, tile_done, max_tiles, h, y, status, 4 * kTileK);
    a.gs = q.gts;
    a.us = q.uts;
    a.ds = q.dts;
    const int grid = mlp_grid(a, max_tiles, num_sms);
    if (bn_max <= 32) return launch_mlp<32, true>(wg, wu, wd, sm, bx, bh, a, grid, st);
    return launch_mlp<128, true>(wg, wu, wd, sm, bx, bh, a, grid, st);
}

}  // namespace beam
