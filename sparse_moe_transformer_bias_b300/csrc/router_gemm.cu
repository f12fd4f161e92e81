// The router's FP32 product on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators, TMA-fed shared-memory pipeline). transformers "Beam" doc, paragraph after
// the Overview bullets: routing is computed in FP32 with FP32 router weights.
//
// logits = x . Wr^T with the FP32 Wr given as three BF16 pieces hi + mid + lo whose sum is
// exactly Wr (router.cu writes them) and x exactly BF16: three MMAs per K step accumulate
// x.hi + x.mid + x.lo into one FP32 accumulator, i.e. the FP32 product with exact
// BF16 x BF16 partial products. Written "weights as M": D[128 experts, N tokens] per work
// item (an N-tile of up to 128 tokens, an M-tile of 128 experts and a K range). K is split
// into `splits` ranges; each split stores its FP32 plane partial[split][token][expert],
// added in split order by the selection kernel, so the result is deterministic.
//
// Roles (one CTA per SM, persistent over a static round-robin of work items):
//   warp 0 lane 0: TMA producer - per 64-wide K chunk, the three weight-piece tiles
//                  [128 x 64] and the tile's tokens (rounded up to 16) in the fewest
//                  power-of-two boxes, 128-byte swizzle, into a ring of stages;
//   warp 1:        allocates TMEM; lane 0 issues tcgen05.mma (M=128, N=tokens rounded up
//                  to 16, K=16) and tcgen05.commit;
//   warps 2-9:     epilogue - tcgen05.ld of their TMEM lane quarter (two warps per
//                  quarter, alternate 16-column granules), FP32 stores.
// Accumulators are double-buffered in TMEM. Every mbarrier wait is bounded (2 s); on expiry
// the CTA records kStatusWaitTimeout (when given a status word), the roles leave their
// loops, issued copies and MMAs are drained (bounded), and TMEM is freed before exit.
#include "internal.cuh"
#include "ptx.cuh"

namespace beam {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kBN = 128;     // tokens per N-tile
constexpr int kPieces = 3;   // hi, mid, lo
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint64_t kDrainLimitNs = 200000000ull;

struct Cfg {
    static constexpr int kA = kTileM * kTileK * 2;
    static constexpr int kB = kBN * kTileK * 2;
    static constexpr int kStage = kA * kPieces + kB;
    static constexpr int kStages = (227 * 1024 - 2048) / kStage;
    static constexpr int kAccBufs = 2;
    static constexpr int kTmemCols = kBN * kAccBufs;
    static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kNumBars * 8 + 16;
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

struct RouterArgs {
    int T;               // tokens (rows of x)
    int E;               // experts: rows of one weight piece, columns of the output
    int m_tiles;         // ceil(E / 128)
    int splits;          // K ranges
    int k_chunks;        // 64-wide K chunks per range
    float* partial;      // [splits][T][E]
    int* status;         // may be null
    uint32_t extra_tx;   // self-test only (0 otherwise): bytes the first stage of CTA 0 expects
                         // beyond what its copies deliver, so that stage never completes
};

struct Item {
    int row0, rows, m, split;
};

__device__ __forceinline__ Item item_of(const RouterArgs& a, int item) {
    Item it;
    it.split = item % a.splits;
    const int r = item / a.splits;
    it.m = r % a.m_tiles;
    it.row0 = (r / a.m_tiles) * kBN;
    it.rows = min(kBN, a.T - it.row0);
    return it;
}

__device__ __forceinline__ void flag_status(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ void record_failure(volatile int* abort_flag, int* status) {
    *abort_flag = 1;
    flag_status(status, kStatusWaitTimeout);
}

__global__ void __launch_bounds__(kThreads, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ BMaps tmX,
                       const __grid_constant__ RouterArgs args) {
    using C = Cfg;
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
        ptx::prefetch_tmap(&tmW);
        for (int i = 0; i < kBoxKinds && (kBoxRows << i) <= kBN; ++i) ptx::prefetch_tmap(&tmX.m[i]);
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
    const int n_items = ((args.T + kBN - 1) / kBN) * args.m_tiles * args.splits;
    const int k_chunks = args.k_chunks;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const uint64_t pol_w = ptx::policy_evict_last();  // the pieces are re-read by every token tile
            const uint64_t pol_x = ptx::policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, parity = 0;  // per stage: ever loaded / parity of the last load
            bool ok = true;
            uint32_t extra = blockIdx.x == 0 ? args.extra_tx : 0u;
            for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
                const Item it = item_of(args, item);
                const int b_rows = ((it.rows + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t bytes = C::kA * kPieces + b_rows * kTileK * 2;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    const int kx = (it.split * k_chunks + kc) * kTileK;
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes + extra);
                    extra = 0u;
#pragma unroll
                    for (int j = 0; j < kPieces; ++j)
                        ptx::tma_load_2d(sa + j * C::kA, &tmW, kx, j * args.E + it.m * kTileM, bar(FULL0 + stage),
                                         pol_w);
                    const uint32_t sb = sa + C::kA * kPieces;
                    for (int i = kBoxKinds - 1, r = 0; i >= 0; --i) {
                        const int h = kBoxRows << i;
                        if (h > kBN || b_rows - r < h) continue;
                        ptx::tma_load_2d(sb + r * kTileK * 2, &tmX.m[i], kx, it.row0 + r, bar(FULL0 + stage), pol_x);
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
                const Item it = item_of(args, item);
                const uint32_t idesc = ptx::idesc_bf16_f32(kTileM, ((it.rows + 15) / 16) * 16);
                if (!ptx::mbar_wait(bar(TEMPTY0 + acc), acc_phase ^ 1, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d0 = tmem_base + acc * kBN;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    const uint32_t sb = sa + C::kA * kPieces;
#pragma unroll
                    for (int kk = 0; kk < kTileK / kMmaK; ++kk) {
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(sb + kk * kMmaK * 2);
#pragma unroll
                        for (int j = 0; j < kPieces; ++j)
                            ptx::mma_bf16(d0, ptx::sw128_kmajor_desc(sa + j * C::kA + kk * kMmaK * 2), bdesc, idesc,
                                          (kc | kk | j) ? 1u : 0u);
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
        const int q = warp & 3;
        const int row = q * 32 + lane;                  // expert within the M-tile
        const int col_part = (warp - 2) >> 2;
        constexpr int kColStep = 16 * (kEpiWarps / 4);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
            const Item it = item_of(args, item);
            if (!ptx::mbar_wait(bar(TFULL0 + acc), acc_phase, abort_flag, kWaitLimitNs)) {
                record_failure(abort_flag, status);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBN;
            const int e = it.m * kTileM + row;
            float* out = args.partial + static_cast<size_t>(it.split) * args.T * args.E;
            for (int c0 = col_part * 16; c0 < it.rows; c0 += kColStep) {
                uint32_t v[16];
                ptx::tmem_ld16(taddr + c0, v);
                ptx::tmem_wait_ld();
                if (e < args.E) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < it.rows)
                            out[static_cast<size_t>(it.row0 + c0 + j) * args.E + e] = __uint_as_float(v[j]);
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

}  // namespace

int router_tc_splits(const Shape& s, int T, int num_sms) {
    // Estimated time on the busiest SM, in ns: ~550 per K chunk of an item and ~1500 per
    // item (pipeline fill, epilogue), plus the partial planes written here and read back by
    // the selection kernel at ~6 TB/s. Ties go to fewer splits.
    const int kc_total = s.d / kTileK;
    const long long tiles = static_cast<long long>((T + kBN - 1) / kBN) * ((s.E + kTileM - 1) / kTileM);
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
                             int* status, int num_sms, cudaStream_t st, uint32_t selftest_extra_tx) {
    CUtensorMap w;
    BMaps b;
    const char* why = nullptr;
    if (!encode_tmap_bf16_2d(&w, w3, 3ull * s.E, s.d, kTileM, kTileK, &why) || !encode_bmaps(&b, x, T, s.d, kBN, &why))
        return cudaErrorInvalidValue;
    const int kc_total = s.d / kTileK;
    if (splits < 1 || kc_total % splits) return cudaErrorInvalidValue;
    RouterArgs a;
    a.T = T;
    a.E = s.E;
    a.m_tiles = (s.E + kTileM - 1) / kTileM;
    a.splits = splits;
    a.k_chunks = kc_total / splits;
    a.partial = partial;
    a.status = status;
    a.extra_tx = selftest_extra_tx;
    const long long items = static_cast<long long>((T + kBN - 1) / kBN) * a.m_tiles * splits;
    const int grid = static_cast<int>(items < num_sms ? (items < 1 ? 1 : items) : num_sms);
    cudaError_t e = set_smem_limit_once<router_gemm_kernel>(Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    const cudaError_t le_ = launch_pdl(router_gemm_kernel, dim3(grid), dim3(kThreads), Cfg::kSmemBytes, st, w, b, a);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

}  // namespace beam
