// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, TMEM accumulators,
// TMA-fed shared-memory pipeline) for the SwiGLU experts of the Beam MoE block (Glonce
// "Reflection releases Beam ...", Architecture paragraph: each expert a SwiGLU MLP of
// intermediate size 2,560; transformers "Beam" doc: SwiGLU activation in FP32).
//
// Both GEMMs are written "weights as M": for an N-tile of `rows` permuted token rows of
// expert e and an M-tile of 128 weight rows,
//     D[128 weight rows, N tokens] = W_e[m-tile, :] . X[tile rows, :]^T      (FP32, TMEM)
// so the streamed weights are the 128-row A operand, and all of an expert's tokens (up to
// 256) sit in the N dimension of one MMA: each weight tile is read from HBM once per
// N-tile, which is what bounds decode and prefill.
//   gate/up: two accumulators (gate rows, up rows) share the B tile; the epilogue computes
//            h = silu(g) * u in FP32 and stores BF16 h[row, I].
//   down:    one accumulator; the epilogue stores FP32 y[row, d].
//
// Roles (192 threads, one CTA per SM, persistent over a static round-robin of work items
// item = n_tile * m_tiles + m_tile):
//   warp 0 lane 0: TMA producer - per 64-wide K chunk, the weight tile(s) [128 x 64] and
//                  the activation rows in boxes of 16 [16 x 64], 128-byte swizzle, into a
//                  ring of shared-memory stages (full/empty mbarriers);
//   warp 1:        allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=rows rounded up to
//                  16, K=16 per instruction) and tcgen05.commit to release stages and to
//                  publish a finished accumulator;
//   warps 2-5:     epilogue - tcgen05.ld of their 32-lane TMEM quarter, activation, stores.
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
constexpr int kBoxRows = 16;   // activation rows per TMA box
constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

template <bool kGateUp, int kBNMax>
struct Cfg {
    static constexpr int kA = BM * BK * 2;
    static constexpr int kB = kBNMax * BK * 2;
    static constexpr int kStage = kA * (kGateUp ? 2 : 1) + kB;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int kStages = (kBudget / kStage) > 10 ? 10 : (kBudget / kStage);
    static constexpr int kAccCols = kBNMax * (kGateUp ? 2 : 1);
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

__device__ __forceinline__ void record_failure(volatile int* abort_flag, int* status) {
    *abort_flag = 1;
    atomicCAS(status, 0, kStatusWaitTimeout);
}

template <bool kGateUp, int kBNMax>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB, const int4* __restrict__ tiles, int max_tiles,
                        int n_experts, int total_rows, int m_tiles, int rows_per_expert, int k_chunks,
                        void* __restrict__ out, int ldo, int* status) {
    using C = Cfg<kGateUp, kBNMax>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    constexpr int FULL0 = 0, EMPTY0 = C::kStages, TFULL0 = 2 * C::kStages, TEMPTY0 = TFULL0 + C::kAccBufs,
                  DRAIN = TEMPTY0 + C::kAccBufs;
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(bar(FULL0 + s), 1);
            ptx::mbar_init(bar(EMPTY0 + s), 1);
        }
        for (int b = 0; b < C::kAccBufs; ++b) {
            ptx::mbar_init(bar(TFULL0 + b), 1);
            ptx::mbar_init(bar(TEMPTY0 + b), 128);
        }
        ptx::mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA0);
        if (kGateUp) ptx::prefetch_tmap(&tmA1);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    int n_tiles = tiles[0].x;
    if (n_tiles < 0 || n_tiles > max_tiles) {
        if (threadIdx.x == 0) atomicCAS(status, 0, kStatusBadIndex);
        n_tiles = 0;
    }
    const int n_items = n_tiles * m_tiles;
    // A work-list entry every role checks the same way; a bad one is skipped by all roles.
    auto bad_tile = [&](const int4& tl) {
        return tl.x < 0 || tl.x >= n_experts || tl.z <= 0 || tl.z > kBNMax || tl.y < 0 || tl.y > total_rows - tl.z;
    };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const uint64_t pol_w = ptx::policy_evict_first();
            const uint64_t pol_x = ptx::policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, parity = 0;  // per stage: ever loaded / parity of the last load
            bool ok = true;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const int4 tl = tiles[1 + item / m_tiles];
                const int m = item % m_tiles;
                if (bad_tile(tl)) {
                    atomicCAS(status, 0, kStatusBadIndex);
                    continue;
                }
                const int nbox = (tl.z + kBoxRows - 1) / kBoxRows;
                const uint32_t bytes = C::kA * (kGateUp ? 2 : 1) + nbox * kBoxRows * BK * 2;
                const int a_row = tl.x * rows_per_expert + m * BM;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes);
                    ptx::tma_load_2d(sa, &tmA0, kc * BK, a_row, bar(FULL0 + stage), pol_w);
                    if (kGateUp) ptx::tma_load_2d(sa + C::kA, &tmA1, kc * BK, a_row, bar(FULL0 + stage), pol_w);
                    const uint32_t sb = sa + C::kA * (kGateUp ? 2 : 1);
                    for (int j = 0; j < nbox; ++j)
                        ptx::tma_load_2d(sb + j * kBoxRows * BK * 2, &tmB, kc * BK, tl.y + j * kBoxRows,
                                         bar(FULL0 + stage), pol_x);
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
                const int4 tl = tiles[1 + item / m_tiles];
                if (bad_tile(tl)) continue;
                const int n_mma = ((tl.z + 15) / 16) * 16;
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
                    const uint32_t sb = sa + C::kA * (kGateUp ? 2 : 1);
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk) {
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(sb + kk * UK * 2);
                        const uint32_t accum = (kc | kk) ? 1u : 0u;
                        ptx::mma_bf16(d0, ptx::sw128_kmajor_desc(sa + kk * UK * 2), bdesc, idesc, accum);
                        if (kGateUp)
                            ptx::mma_bf16(d0 + kBNMax, ptx::sw128_kmajor_desc(sa + C::kA + kk * UK * 2), bdesc, idesc,
                                          accum);
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
        const int q = warp & 3;           // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;    // weight row within the M-tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const int4 tl = tiles[1 + item / m_tiles];
            const int m = item % m_tiles;
            if (bad_tile(tl)) continue;
            if (!ptx::mbar_wait(bar(TFULL0 + acc), acc_phase, abort_flag, kWaitLimitNs)) {
                record_failure(abort_flag, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * C::kAccCols;
            const size_t col = static_cast<size_t>(m) * BM + row;
            for (int c0 = 0; c0 < tl.z; c0 += 16) {
                uint32_t g[16];
                ptx::tmem_ld16(taddr + c0, g);
                if constexpr (kGateUp) {
                    uint32_t u[16];
                    ptx::tmem_ld16(taddr + kBNMax + c0, u);
                    ptx::tmem_wait_ld();
                    bf16* h = static_cast<bf16*>(out);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < tl.z) {
                            const float gv = __uint_as_float(g[j]);
                            const float uv = __uint_as_float(u[j]);
                            const float hv = gv / (1.0f + expf(-gv)) * uv;
                            h[static_cast<size_t>(tl.y + c0 + j) * ldo + col] = __float2bfloat16_rn(hv);
                        }
                    }
                } else {
                    ptx::tmem_wait_ld();
                    float* y = static_cast<float*>(out);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < tl.z) y[static_cast<size_t>(tl.y + c0 + j) * ldo + col] = __uint_as_float(g[j]);
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

template <bool kGateUp, int kBNMax>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b, const int4* tiles,
                        int max_tiles, int n_experts, int total_rows, int m_tiles, int rows_per_expert, int k_chunks,
                        void* out, int ldo, int* status, int grid, cudaStream_t st) {
    using C = Cfg<kGateUp, kBNMax>;
    auto kern = grouped_gemm_kernel<kGateUp, kBNMax>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, C::kSmemBytes, st>>>(a0, a1, b, tiles, max_tiles, n_experts, total_rows, m_tiles,
                                                rows_per_expert, k_chunks, out, ldo, status);
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

int grid_for(int max_items, int num_sms) {
    int g = max_items < num_sms ? max_items : num_sms;
    return g < 1 ? 1 : g;
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

int gemm_bn_max(int T) { return T <= 32 ? 32 : 256; }

cudaError_t launch_gateup(const Shape& s, const bf16* w_gate, const bf16* w_up, const bf16* x_perm, int rows,
                          const int4* tiles, int max_tiles, int bn_max, bf16* h, int* status, int num_sms,
                          cudaStream_t st) {
    CUtensorMap a0, a1, b;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&a0, w_gate, static_cast<uint64_t>(s.E) * s.I, s.d, BM, BK, &why) ||
        !encode_tmap_bf16_2d(&a1, w_up, static_cast<uint64_t>(s.E) * s.I, s.d, BM, BK, &why) ||
        !encode_tmap_bf16_2d(&b, x_perm, rows, s.d, kBoxRows, BK, &why))
        return cudaErrorInvalidValue;
    const int m_tiles = s.I / BM;
    const int grid = grid_for(max_tiles * m_tiles, num_sms);
    if (bn_max <= 32)
        return launch_gemm<true, 32>(a0, a1, b, tiles, max_tiles, s.E, rows, m_tiles, s.I, s.d / BK, h, s.I, status,
                                     grid, st);
    return launch_gemm<true, 256>(a0, a1, b, tiles, max_tiles, s.E, rows, m_tiles, s.I, s.d / BK, h, s.I, status,
                                  grid, st);
}

cudaError_t launch_down(const Shape& s, const bf16* w_down, const bf16* h, int rows, const int4* tiles, int max_tiles,
                        int bn_max, float* y, int* status, int num_sms, cudaStream_t st) {
    CUtensorMap a0, b;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&a0, w_down, static_cast<uint64_t>(s.E) * s.d, s.I, BM, BK, &why) ||
        !encode_tmap_bf16_2d(&b, h, rows, s.I, kBoxRows, BK, &why))
        return cudaErrorInvalidValue;
    const int m_tiles = s.d / BM;
    const int grid = grid_for(max_tiles * m_tiles, num_sms);
    if (bn_max <= 32)
        return launch_gemm<false, 32>(a0, a0, b, tiles, max_tiles, s.E, rows, m_tiles, s.d, s.I / BK, y, s.d, status,
                                      grid, st);
    return launch_gemm<false, 256>(a0, a0, b, tiles, max_tiles, s.E, rows, m_tiles, s.d, s.I / BK, y, s.d, status,
                                   grid, st);
}

}  // namespace beam
