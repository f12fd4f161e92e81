// Grouped GEMMs on the 5th-generation tensor cores (tcgen05, TMEM accumulators, TMA-fed
// shared-memory pipeline) for the Beam MoE block: the SwiGLU experts (Glonce "Reflection
// releases Beam ...", Architecture paragraph: each expert a SwiGLU MLP of intermediate size
// 2,560; transformers "Beam" doc: SwiGLU activation in FP32) and the FP32 router product
// (same doc: routing computed in FP32 with FP32 router weights).
//
// Every mode is written "weights as M": for an N-tile of `rows` token rows and an M-tile of
// 128 weight rows,
//     D[128 weight rows, N tokens] = W[m-tile, :] . X[tile rows, :]^T      (FP32, TMEM)
// so the weights are the 128-row A operand and the tile's tokens (up to kBNMax) sit in the
// N dimension of one MMA: each weight tile is read once per N-tile.
//   gate/up: per expert; two accumulators (gate rows, up rows) share the B tile; the
//            epilogue computes h = silu(g) * u in FP32 and stores BF16 h[row, I].
//   down:    per expert; one accumulator; the epilogue stores FP32 y[row, d].
//   router:  logits = x . Wr^T with FP32 Wr given as three BF16 pieces hi + mid + lo whose
//            sum is exactly Wr (x is exactly BF16): three MMAs per K step accumulate
//            x.hi + x.mid + x.lo into one FP32 accumulator, i.e. the FP32 product with
//            exact BF16 x BF16 partial products. K is split into `splits` ranges; each
//            split stores its FP32 plane partial[split][token][expert], added in split
//            order by the selection kernel.
//
// Roles (one CTA per SM, persistent over a static round-robin of work items):
//   warp 0 lane 0: TMA producer - per 64-wide K chunk, the weight tile(s) [128 x 64] and
//                  the tile's activation rows (rounded up to 16) in the fewest boxes of
//                  16..256 rows, 128-byte swizzle, into a ring of shared-memory stages
//                  (full/empty mbarriers). Every TMA copy costs the single issuing thread
//                  tens of cycles, so fewer, larger boxes keep it ahead of the MMAs;
//   warp 1:        allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=rows rounded up to
//                  16, K=16 per instruction) and tcgen05.commit to release stages and to
//                  publish a finished accumulator;
//   warps 2..:     epilogue - tcgen05.ld of their 32-lane TMEM quarter (warp % 4), the
//                  warps of one quarter taking alternate 16-column granules; activation,
//                  stores.
// Accumulators are double-buffered in TMEM when two fit (512 columns), so the epilogue of
// one tile overlaps the MMAs of the next.
// Every mbarrier wait is bounded (2 s of wall time); on expiry the CTA records
// kStatusWaitTimeout, the other roles leave their loops, the producer waits (bounded) for
// its issued copies to land, the MMA warp waits (bounded) for its issued MMAs, and TMEM is
// freed before the CTA exits.
#include <mutex>

#include "internal.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

constexpr int BM = 128;        // weight rows per tile (MMA M)
constexpr int BK = 64;         // K per stage: one 128-byte swizzle row of BF16
constexpr int UK = 16;         // K per tcgen05.mma (kind::f16)
constexpr int kBoxRows = 16;   // granule of activation rows (MMA N step, smallest TMA box)
constexpr int kBoxKinds = 5;   // activation tensor maps with boxes of 16, 32, 64, 128, 256 rows
#ifndef BEAM_GEMM_EPI_WARPS
#define BEAM_GEMM_EPI_WARPS 8
#endif
constexpr int kEpiWarps = BEAM_GEMM_EPI_WARPS;   // warps per TMEM lane quarter = kEpiWarps / 4
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

enum : int { kModeDown = 0, kModeGateUp = 1, kModeRouter = 2 };

template <int kMode, int kBNMax>
struct Cfg {
    static constexpr int kNumA = kMode == kModeGateUp ? 2 : kMode == kModeRouter ? 3 : 1;
    static constexpr int kNumAcc = kMode == kModeGateUp ? 2 : 1;
    static constexpr int kA = BM * BK * 2;
    static constexpr int kB = kBNMax * BK * 2;
    static constexpr int kStage = kA * kNumA + kB;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int kStages = (kBudget / kStage) > 10 ? 10 : (kBudget / kStage);
    static constexpr int kAccCols = kBNMax * kNumAcc;
    static constexpr int kAccBufs = (2 * kAccCols <= 512) ? 2 : 1;
    static constexpr int kColsNeeded = kAccCols * kAccBufs;
    static constexpr int kTmemCols = kColsNeeded <= 32    ? 32
                                     : kColsNeeded <= 64  ? 64
                                     : kColsNeeded <= 128 ? 128
                                     : kColsNeeded <= 256 ? 256
                                                          : 512;
    static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kNumBars * 8 + 16;
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kColsNeeded <= 512, "accumulators exceed TMEM");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Everything the kernel needs besides the tensor maps.
struct GemmArgs {
    const int4* tiles;      // expert modes: header int4 (.x = tile count), then {e, row0, rows, 0}
    int max_tiles;          // expert modes: capacity of the work list
    int n_experts;          // expert modes: valid expert ids are [0, n_experts)
    int total_rows;         // rows of the B operand (permuted rows, or tokens for the router)
    int m_tiles;            // 128-row weight tiles per item column
    int rows_per_expert;    // expert modes: A rows of one expert
    int k_chunks;           // 64-wide K chunks per item
    int splits;             // router: K ranges per (token tile, weight tile); else 1
    int piece_rows;         // router: A rows between the hi, mid and lo weight pieces (E)
    int out_cols;           // columns of the output actually stored (router: E)
    void* out;
    int ldo;                // output row pitch in elements
    long long split_stride; // router: elements between the output planes of two splits
    int* status;            // may be null
};

// The B operand (token rows) as tensor maps that differ only in box height:
// m[i] has boxes of (16 << i) rows x 64 columns.
struct BMaps {
    CUtensorMap m[kBoxKinds];
};

struct Item {
    int4 tl;    // {expert, first B row, rows, 0}
    int m;      // weight tile
    int split;  // K range
    bool ok;
};

// Decodes work item `item` the same way in every role.
template <int kMode, int kBNMax>
__device__ __forceinline__ Item item_of(const GemmArgs& a, int item) {
    Item it;
    if constexpr (kMode == kModeRouter) {
        it.split = item % a.splits;
        const int r = item / a.splits;
        it.m = r % a.m_tiles;
        const int row0 = (r / a.m_tiles) * kBNMax;
        it.tl = make_int4(0, row0, min(kBNMax, a.total_rows - row0), 0);
        it.ok = true;
    } else {
        const int4 tl = a.tiles[1 + item / a.m_tiles];
        it.tl = tl;
        it.m = item % a.m_tiles;
        it.split = 0;
        it.ok = !(tl.x < 0 || tl.x >= a.n_experts || tl.z <= 0 || tl.z > kBNMax || tl.y < 0 ||
                  tl.y > a.total_rows - tl.z);
    }
    return it;
}

// Records `code` in the status word unless one is already recorded (status may be null:
// callers without a status word only get the abort behaviour).
__device__ __forceinline__ void flag_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ void record_failure(volatile int* abort_flag, int* status) {
    *abort_flag = 1;
    flag_status(status, kStatusWaitTimeout);
}

template <int kMode, int kBNMax>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ BMaps tmB, const __grid_constant__ GemmArgs args) {
    using C = Cfg<kMode, kBNMax>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    constexpr int FULL0 = 0, EMPTY0 = C::kStages, TFULL0 = 2 * C::kStages, TEMPTY0 = TFULL0 + C::kAccBufs,
                  DRAIN = TEMPTY0 + C::kAccBufs;
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };
    int* status = args.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(bar(FULL0 + s), 1);
            ptx::mbar_init(bar(EMPTY0 + s), 1);
        }
        for (int b = 0; b < C::kAccBufs; ++b) {
            ptx::mbar_init(bar(TFULL0 + b), 1);
            ptx::mbar_init(bar(TEMPTY0 + b), 32 * kEpiWarps);
        }
        ptx::mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA0);
        if (kMode == kModeGateUp) ptx::prefetch_tmap(&tmA1);
        for (int i = 0; i < kBoxKinds && (kBoxRows << i) <= kBNMax; ++i) ptx::prefetch_tmap(&tmB.m[i]);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    int n_items;
    if constexpr (kMode == kModeRouter) {
        n_items = ((args.total_rows + kBNMax - 1) / kBNMax) * args.m_tiles * args.splits;
    } else {
        int n_tiles = args.tiles[0].x;
        if (n_tiles < 0 || n_tiles > args.max_tiles) {
            if (threadIdx.x == 0) flag_status(status, kStatusBadIndex);
            n_tiles = 0;
        }
        n_items = n_tiles * args.m_tiles;
    }
    const int k_chunks = args.k_chunks;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            // Expert weights stream once (evict first); the router's weight pieces are
            // re-read by every token tile (keep them).
            const uint64_t pol_w = kMode == kModeRouter ? ptx::policy_evict_last() : ptx::policy_evict_first();
            const uint64_t pol_x = ptx::policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, parity = 0;  // per stage: ever loaded / parity of the last load
            bool ok = true;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const Item it = item_of<kMode, kBNMax>(args, item);
                if (!it.ok) {
                    flag_status(status, kStatusBadIndex);
                    continue;
                }
                const int b_rows = ((it.tl.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t bytes = C::kA * C::kNumA + b_rows * BK * 2;
                const int a_row = (kMode == kModeRouter ? 0 : it.tl.x * args.rows_per_expert) + it.m * BM;
                const int kc0 = it.split * k_chunks;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    const int kx = (kc0 + kc) * BK;
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes);
#pragma unroll
                    for (int j = 0; j < C::kNumA; ++j) {
                        const CUtensorMap* map = (kMode == kModeGateUp && j == 1) ? &tmA1 : &tmA0;
                        const int row = a_row + (kMode == kModeRouter ? j * args.piece_rows : 0);
                        ptx::tma_load_2d(sa + j * C::kA, map, kx, row, bar(FULL0 + stage), pol_w);
                    }
                    const uint32_t sb = sa + C::kA * C::kNumA;
                    // The tile's rows (rounded up to 16) in the fewest boxes: greedy powers
                    // of two, largest first (at most 4 copies for up to 256 rows).
                    for (int i = kBoxKinds - 1, r = 0; i >= 0; --i) {
                        const int h = kBoxRows << i;
                        if (h > kBNMax || b_rows - r < h) continue;
                        ptx::tma_load_2d(sb + r * BK * 2, &tmB.m[i], kx, it.tl.y + r, bar(FULL0 + stage), pol_x);
                        r += h;
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
                record_failure(abort_flag, status);
                const int never = 0;
                for (int s = 0; s < C::kStages; ++s)
                    if ((issued >> s) & 1u) ptx::mbar_wait(bar(FULL0 + s), (parity >> s) & 1u, &never, kDrainLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const Item it = item_of<kMode, kBNMax>(args, item);
                if (!it.ok) continue;
                const int n_mma = ((it.tl.z + 15) / 16) * 16;
                const uint32_t idesc = ptx::idesc_bf16_f32(BM, n_mma);
                if (!ptx::mbar_wait(bar(TEMPTY0 + acc), acc_phase ^ 1, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d0 = tmem_base + acc * C::kAccCols;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    const uint32_t sb = sa + C::kA * C::kNumA;
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk) {
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(sb + kk * UK * 2);
                        if constexpr (kMode == kModeRouter) {
#pragma unroll
                            for (int j = 0; j < C::kNumA; ++j)
                                ptx::mma_bf16(d0, ptx::sw128_kmajor_desc(sa + j * C::kA + kk * UK * 2), bdesc, idesc,
                                              (kc | kk | j) ? 1u : 0u);
                        } else {
                            const uint32_t accum = (kc | kk) ? 1u : 0u;
                            ptx::mma_bf16(d0, ptx::sw128_kmajor_desc(sa + kk * UK * 2), bdesc, idesc, accum);
                            if (kMode == kModeGateUp)
                                ptx::mma_bf16(d0 + kBNMax, ptx::sw128_kmajor_desc(sa + C::kA + kk * UK * 2), bdesc,
                                              idesc, accum);
                        }
                    }
                    ptx::mma_commit(bar(EMPTY0 + stage));
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(bar(TFULL0 + acc));
                if (++acc == C::kAccBufs) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (!ok) {
                record_failure(abort_flag, status);
                const int never = 0;
                ptx::mma_commit(bar(DRAIN));
                ptx::mbar_wait(bar(DRAIN), 0, &never, kDrainLimitNs);
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;                          // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;                   // weight row within the M-tile
        const int col_part = (warp - 2) >> 2;            // which 16-column granules this warp takes
        constexpr int kColStep = 16 * (kEpiWarps / 4);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const Item it = item_of<kMode, kBNMax>(args, item);
            if (!it.ok) continue;
            if (!ptx::mbar_wait(bar(TFULL0 + acc), acc_phase, abort_flag, kWaitLimitNs)) {
                record_failure(abort_flag, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
            const int col = it.m * BM + row;
            const bool col_ok = col < args.out_cols;
            for (int c0 = col_part * 16; c0 < it.tl.z; c0 += kColStep) {
                uint32_t g[16];
                ptx::tmem_ld16(taddr + c0, g);
                if constexpr (kMode == kModeGateUp) {
                    uint32_t u[16];
                    ptx::tmem_ld16(taddr + kBNMax + c0, u);
                    ptx::tmem_wait_ld();
                    bf16* h = static_cast<bf16*>(args.out);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < it.tl.z && col_ok) {
                            const float gv = __uint_as_float(g[j]);
                            const float uv = __uint_as_float(u[j]);
                            const float hv = gv / (1.0f + expf(-gv)) * uv;
                            h[static_cast<size_t>(it.tl.y + c0 + j) * args.ldo + col] = __float2bfloat16_rn(hv);
                        }
                    }
                } else {
                    ptx::tmem_wait_ld();
                    float* y = static_cast<float*>(args.out) + it.split * args.split_stride;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < it.tl.z && col_ok)
                            y[static_cast<size_t>(it.tl.y + c0 + j) * args.ldo + col] = __uint_as_float(g[j]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(TEMPTY0 + acc));
            if (++acc == C::kAccBufs) {
                acc = 0;
                acc_phase ^= 1;
            }
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

template <int kMode, int kBNMax>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const BMaps& b, const GemmArgs& args,
                        int grid, cudaStream_t st) {
    using C = Cfg<kMode, kBNMax>;
    auto kern = grouped_gemm_kernel<kMode, kBNMax>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::kSmemBytes, st>>>(a0, a1, b, args);
    return cudaGetLastError();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

int grid_for(long long max_items, int num_sms) {
    long long g = max_items < num_sms ? max_items : num_sms;
    return g < 1 ? 1 : static_cast<int>(g);
}

GemmArgs expert_args(const int4* tiles, int max_tiles, int n_experts, int rows, int m_tiles, int rows_per_expert,
                     int k_chunks, void* out, int ldo, int* status) {
    GemmArgs a;
    a.tiles = tiles;
    a.max_tiles = max_tiles;
    a.n_experts = n_experts;
    a.total_rows = rows;
    a.m_tiles = m_tiles;
    a.rows_per_expert = rows_per_expert;
    a.k_chunks = k_chunks;
    a.splits = 1;
    a.piece_rows = 0;
    a.out_cols = m_tiles * BM;
    a.out = out;
    a.ldo = ldo;
    a.split_stride = 0;
    a.status = status;
    return a;
}

constexpr int kRouterBN = 128;  // tokens per router N-tile

}  // namespace

namespace {
// Tensor maps of a [rows, cols] BF16 B operand for every box height up to bn_max.
bool encode_bmaps(BMaps* b, const void* base, uint64_t rows, uint64_t cols, int bn_max, const char** why) {
    for (int i = 0; i < kBoxKinds; ++i) {
        const uint32_t h = kBoxRows << i;
        if (static_cast<int>(h) > bn_max) {
            b->m[i] = b->m[0];
            continue;
        }
        if (!encode_tmap_bf16_2d(&b->m[i], base, rows, cols, h, BK, why)) return false;
    }
    return true;
}
}  // namespace

bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                         uint32_t box_cols, const char** why) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        *why = "driver entry point cuTensorMapEncodeTiled is not available";
        return false;
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        *why = "cuTensorMapEncodeTiled rejected a tensor map";
        return false;
    }
    return true;
}

// N-tile capacity for a batch of T tokens: 32 for decode-sized batches; 128 while the
// average expert gets at most 32 rows (one tile holds nearly every expert's rows, and the
// smaller B stage leaves room for a fourth stage); else 256, so that a weight tile is
// streamed once for up to 256 of its expert's rows.
int gemm_bn_max(const Shape& s, int T) {
    if (T <= 32) return 32;
    const long long avg_rows = static_cast<long long>(T) * s.top_k / s.E;
    return avg_rows <= 32 ? 128 : 256;
}

cudaError_t launch_gateup(const Shape& s, const bf16* w_gate, const bf16* w_up, const bf16* x_perm, int rows,
                          const int4* tiles, int max_tiles, int bn_max, bf16* h, int* status, int num_sms,
                          cudaStream_t st) {
    CUtensorMap a0, a1;
    BMaps b;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&a0, w_gate, static_cast<uint64_t>(s.E) * s.I, s.d, BM, BK, &why) ||
        !encode_tmap_bf16_2d(&a1, w_up, static_cast<uint64_t>(s.E) * s.I, s.d, BM, BK, &why) ||
        !encode_bmaps(&b, x_perm, rows, s.d, bn_max, &why))
        return cudaErrorInvalidValue;
    const int m_tiles = s.I / BM;
    const GemmArgs args = expert_args(tiles, max_tiles, s.E, rows, m_tiles, s.I, s.d / BK, h, s.I, status);
    const int grid = grid_for(static_cast<long long>(max_tiles) * m_tiles, num_sms);
    if (bn_max <= 32) return launch_gemm<kModeGateUp, 32>(a0, a1, b, args, grid, st);
    if (bn_max <= 128) return launch_gemm<kModeGateUp, 128>(a0, a1, b, args, grid, st);
    return launch_gemm<kModeGateUp, 256>(a0, a1, b, args, grid, st);
}

cudaError_t launch_down(const Shape& s, const bf16* w_down, const bf16* h, int rows, const int4* tiles, int max_tiles,
                        int bn_max, float* y, int* status, int num_sms, cudaStream_t st) {
    CUtensorMap a0;
    BMaps b;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&a0, w_down, static_cast<uint64_t>(s.E) * s.d, s.I, BM, BK, &why) ||
        !encode_bmaps(&b, h, rows, s.I, bn_max, &why))
        return cudaErrorInvalidValue;
    const int m_tiles = s.d / BM;
    const GemmArgs args = expert_args(tiles, max_tiles, s.E, rows, m_tiles, s.d, s.I / BK, y, s.d, status);
    const int grid = grid_for(static_cast<long long>(max_tiles) * m_tiles, num_sms);
    if (bn_max <= 32) return launch_gemm<kModeDown, 32>(a0, a0, b, args, grid, st);
    if (bn_max <= 128) return launch_gemm<kModeDown, 128>(a0, a0, b, args, grid, st);
    return launch_gemm<kModeDown, 256>(a0, a0, b, args, grid, st);
}

int router_tc_splits(const Shape& s, int T, int num_sms) {
    // Estimated time on the busiest SM, in ns: ~550 per K chunk of an item and ~1500 per
    // item (pipeline fill, epilogue), plus the partial planes written here and read back by
    // the selection kernel at ~6 TB/s. Ties go to fewer splits.
    const int kc_total = s.d / BK;
    const long long tiles = static_cast<long long>((T + kRouterBN - 1) / kRouterBN) * ((s.E + BM - 1) / BM);
    int best = 1;
    long long best_cost = -1;
    for (int sp = 1; sp <= 16 && sp <= kc_total; ++sp) {
        if (kc_total % sp) continue;
        const long long items = tiles * sp;
        const long long waves = (items + num_sms - 1) / num_sms;
        const long long cost = waves * ((kc_total / sp) * 550ll + 1500ll) +
                               static_cast<long long>(sp) * T * s.E * 8 / 6000;
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = sp;
        }
    }
    return best;
}

cudaError_t launch_router_tc(const Shape& s, const bf16* w3, const bf16* x, int T, int splits, float* partial,
                             int* status, int num_sms, cudaStream_t st) {
    CUtensorMap a0;
    BMaps b;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&a0, w3, 3ull * s.E, s.d, BM, BK, &why) ||
        !encode_bmaps(&b, x, T, s.d, kRouterBN, &why))
        return cudaErrorInvalidValue;
    const int kc_total = s.d / BK;
    if (splits < 1 || kc_total % splits) return cudaErrorInvalidValue;
    GemmArgs a = expert_args(nullptr, 0, 1, T, (s.E + BM - 1) / BM, 0, kc_total / splits, partial, s.E, status);
    a.splits = splits;
    a.piece_rows = s.E;
    a.out_cols = s.E;
    a.split_stride = static_cast<long long>(T) * s.E;
    const long long items = static_cast<long long>((T + kRouterBN - 1) / kRouterBN) * a.m_tiles * splits;
    return launch_gemm<kModeRouter, kRouterBN>(a0, a0, b, a, grid_for(items, num_sms), st);
}

}  // namespace beam
