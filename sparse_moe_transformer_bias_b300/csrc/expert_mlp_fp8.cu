// The routed experts on FP8 E4M3 weights with FP8 tensor-core products (tcgen05.mma
// kind::f8f6f4): the block of beam_moe_forward_fp8 (Glonce "Reflection releases Beam ...",
// Hardware paragraph: FP8 checkpoints; the weight-only reading W[r][c] = scale[r] *
// e4m3(q[r][c]) with one FP32 scale per output row).
//
// Why: a tcgen05.mma of M = 128 costs about the same time whatever its N up to 128 (about
// 100 cycles measured on B300, for kind::f16 and kind::f8f6f4 alike), and kind::f8f6f4 takes
// K = 32 per instruction against 16 for
// BF16. Weights read as FP8 codes straight from shared memory therefore need half the MMA
// instructions per weight byte of codes widened to BF16, which is what lets the decode
// kernel run at the HBM rate of one byte per weight.
//
// The activations (x for the gate/up product, h for the down product) enter the products as
// two E4M3 pieces per token row, with one power-of-two scale s per row chosen from the
// row's largest magnitude a (s = the least power of two with a <= 448 s):
//     v = s * p1 + (s / 16) * p2,   p1 = e4m3(v / s),   p2 = e4m3((v - s * p1) * 16 / s).
// A BF16 value has 8 significant bits; p1 keeps the top 4 and the remainder has at most 4,
// so both pieces are exact for every value within 2^-10 of the row's largest (smaller ones
// land in the E4M3 subnormal range: an absolute error of at most 2^-14 s < 2.8e-7 a). The pieces of token
// row j of a tile are the B operand's rows 2j and 2j + 1, so one MMA of N = 2b (b = the
// tile's rows rounded up to 16) gives both partial products, and the epilogue takes
// acc = s * (D[:, 2c] + D[:, 2c + 1] / 16)  per token column c, then the weight row's scale,
// SwiGLU (gate/up) or the BF16 expert output (down), as the BF16 kernel does.
//
// x is split once per token by a preparatory kernel before dispatch (which then moves the
// pieces, 2d bytes per row like a BF16 row), so gate/up items load their B operand with TMA
// as it is. h is known only once every gate/up item of its tile has run: its per-row
// maximum is raised with atomicMax by the gate/up epilogues over the BF16-rounded h they
// store, final once the tile's completion counter is complete (which a down item waits for
// anyway), and the down items' BF16 h rows are split on chip by converter warps.
//
// Items, ids, scheduling, completion counters and bounded waits are those of the BF16
// kernel (expert_mlp.cu). Roles (one CTA per SM):
//   warp 0 lane 0: scheduler + TMA producer: per stage (K = 128) the two FP8 weight tiles
//                  [128 x 128] (128-byte rows, 128-byte swizzle), then the tile's x pieces
//                  (2b rows of 128 bytes; gate/up) or its BF16 h rows as two 64-wide halves
//                  (down);
//   warp 1:        TMEM; lane 0 issues the MMAs (M = 128, N = 2b, K = 32, A and B from
//                  shared memory) once the stage's pieces are in place;
//   warps 2..9:    epilogue (two warps per TMEM lane quarter, alternate 16-column granules);
//   warps 10..17:  converters (down items): each thread turns 16-element chunks of h rows
//                  into the two pieces, written in place over the BF16 rows (same size) in
//                  the 128-byte-swizzled K-major layout the MMA reads; on gate/up items they
//                  only pass the stage on.
#include "expert_common.cuh"

namespace beam {
namespace {

using namespace mlp;

constexpr int kCvtWarps = 8;
constexpr int kCvtThreads = 32 * kCvtWarps;
constexpr int kF8Threads = 64 + 32 * kEpiWarps + kCvtThreads;
constexpr int kF8KStage = 128;  // K per stage: one 128-byte row of codes

template <int kBNMax>
struct F8Cfg {
    static constexpr int kA = kTileM * kF8KStage;     // one FP8 weight tile: 16 KB
    static constexpr int kBHalf = kBNMax * kTileK * 2;  // BF16 token rows x 64 of K
    // BF16 token rows x 128 of K, overwritten in place by their two E4M3 pieces per row
    // (2 x rows x 128 bytes: the same size)
    static constexpr int kB = 2 * kBHalf;
    static constexpr int kStage = 2 * kA + kB;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int kStages = (kBudget / kStage) > 6 ? 6 : (kBudget / kStage);
    static constexpr int kSlotCols = 2 * kBNMax;  // an accumulator: both pieces of every token
    static constexpr int kSlots = ((512 / kSlotCols) < 4 ? (512 / kSlotCols) : 4) & ~1;
    static constexpr int kCols = kSlots * kSlotCols;
    static constexpr int kTmemCols = kCols <= 32 ? 32 : kCols <= 64 ? 64 : kCols <= 128 ? 128 : kCols <= 256 ? 256 : 512;
    // FULL (TMA), CONV (pieces written), EMPTY (MMAs done) per stage; TFULL, TEMPTY per slot;
    // RFULL, REMPTY per ring entry; DRAIN.
    static constexpr int kNumBars = 3 * kStages + 2 * kSlots + 2 * kRing + 1;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kNumBars * 8 + kRing * 4 + 16;
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kSlots >= 2, "an item takes two accumulator slots");
    static_assert(kStage % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Instruction descriptor, kind::f8f6f4: D F32 (bits 4-5 = 1), A and B E4M3 (bits 7-9 = 0,
// bits 10-12 = 0), both K-major, N >> 3 in bits 17-22, M >> 4 in bits 24-28.
__device__ __forceinline__ uint32_t idesc_e4m3_f32(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, E4M3 inputs, FP32 accumulate, K = 32.
__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The row scale s (a power of two) for a row whose largest magnitude is `amax`: the least
// power of two with amax <= 448 s, i.e. 2^(e - 8) when amax = m 2^e with m <= 1.75, else
// 2^(e - 7); 1 for an all-zero (or vanishingly small) row. Returns s and 1/s, both exact.
__device__ __forceinline__ void row_scale(float amax, float& s, float& inv) {
    const uint32_t b = __float_as_uint(amax) & 0x7fffffffu;
    const int e = static_cast<int>(b >> 23);          // biased exponent of amax
    const int es = e - 8 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);  // biased exponent of s
    if (e == 0 || es < 2 || es > 252) {
        s = 1.0f;
        inv = 1.0f;
        return;
    }
    s = __uint_as_float(static_cast<uint32_t>(es) << 23);
    inv = __uint_as_float(static_cast<uint32_t>(254 - es) << 23);
}

// Eight BF16 values (one 16-byte chunk) -> eight p1 codes and eight p2 codes (element 0 in
// the lowest byte), for a row with 1/s = inv. a = v / s is exact in FP32 and in FP16 (8
// significant bits, |a| <= 448; FP16 subnormals only round values below 2^-17 of the row's
// largest), and so is the remainder a - e4m3(a) and its product with 16, so the
// remainder's arithmetic runs on packed FP16 pairs.
__device__ __forceinline__ void split8(uint4 v, float inv, uint2& p1, uint2& p2) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c1[4], c2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
        const __half2 a = __floats2half2_rn(f.x * inv, f.y * inv);  // element 2i in the low half
        const uint32_t ab = *reinterpret_cast<const uint32_t*>(&a);
        uint32_t q, back;
        asm("{\n .reg .b16 c;\n"
            " cvt.rn.satfinite.e4m3x2.f16x2 c, %2;\n"   // p1 codes (low byte: low half)
            " cvt.u32.u16 %0, c;\n"
            " cvt.rn.f16x2.e4m3x2 %1, c;\n}\n"         // their values
            : "=r"(q), "=r"(back)
            : "r"(ab));
        const __half2 r = __hmul2(__hsub2(a, *reinterpret_cast<const __half2*>(&back)), __float2half2_rn(16.0f));
        const uint32_t rb = *reinterpret_cast<const uint32_t*>(&r);
        uint32_t q2;
        asm("{\n .reg .b16 c;\n cvt.rn.satfinite.e4m3x2.f16x2 c, %1;\n cvt.u32.u16 %0, c;\n}\n" : "=r"(q2) : "r"(rb));
        c1[i] = q;
        c2[i] = q2;
    }
    p1 = make_uint2(c1[0] | (c1[1] << 16), c1[2] | (c1[3] << 16));
    p2 = make_uint2(c2[0] | (c2[1] << 16), c2[2] | (c2[3] << 16));
}

template <int kBNMax>
__global__ void __launch_bounds__(kF8Threads, 1)
    expert_mlp_f8_kernel(const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
                         const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ BMaps tmX,
                         const __grid_constant__ BMaps tmH, const __grid_constant__ MlpArgs args) {
    using C = F8Cfg<kBNMax>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
    volatile int* ring = reinterpret_cast<volatile int*>(bars + C::kNumBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(ring) + kRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    constexpr int FULL0 = 0, CONV0 = C::kStages, EMPTY0 = 2 * C::kStages, TFULL0 = 3 * C::kStages,
                  TEMPTY0 = TFULL0 + C::kSlots, RFULL0 = TEMPTY0 + C::kSlots, REMPTY0 = RFULL0 + kRing,
                  DRAIN = REMPTY0 + kRing;
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };
    int* status = args.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(bar(FULL0 + s), 1);
            ptx::mbar_init(bar(CONV0 + s), kCvtWarps);
            ptx::mbar_init(bar(EMPTY0 + s), 1);
        }
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(bar(TFULL0 + s), 1);
            ptx::mbar_init(bar(TEMPTY0 + s), 32 * kEpiWarps);
        }
        for (int r = 0; r < kRing; ++r) {
            ptx::mbar_init(bar(RFULL0 + r), 1);
            ptx::mbar_init(bar(REMPTY0 + r), 1 + kEpiWarps + kCvtWarps);
        }
        ptx::mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmWg);
        ptx::prefetch_tmap(&tmWu);
        ptx::prefetch_tmap(&tmWd);
        for (int i = 0; i < kBoxKinds && (kBoxRows << i) <= 2 * kBNMax; ++i) {
            ptx::prefetch_tmap(&tmX.m[i]);
            if ((kBoxRows << i) <= kBNMax) ptx::prefetch_tmap(&tmH.m[i]);
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
                if (id >= 0) next = atomicAdd(args.next_item, 1);
                if (!ptx::mbar_wait(bar(REMPTY0 + rslot), rphase ^ 1, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ring[rslot] = id;
                ptx::mbar_arrive(bar(RFULL0 + rslot));
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
                    if (!wait_counter(args.tile_done + it.tile, args.m_gu * kEpiWarps, abort_flag)) {
                        ok = false;
                        break;
                    }
                    fence_proxy_async_global();  // order the copies of h below after that observation
                }
                const int b_rows = ((it.tl.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t bytes = 2 * C::kA + b_rows * kF8KStage * 2;  // 2b rows of pieces or b BF16 rows
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                const int a_row = it.down ? it.tl.x * args.d + it.m * 2 * kTileM : it.tl.x * args.I + it.m * kTileM;
                const uint64_t pol_w = it.n_t > 1 ? pol_w_shared : pol_w_once;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    const int kx = kc * kF8KStage;
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes);
                    if (it.down) {
                        ptx::tma_load_2d(sa, &tmWd, kx, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWd, kx, a_row + kTileM, bar(FULL0 + stage), pol_w);
                    } else {
                        ptx::tma_load_2d(sa, &tmWg, kx, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWu, kx, a_row, bar(FULL0 + stage), pol_w);
                    }
                    const uint32_t sb = sa + 2 * C::kA;
                    if (it.down) {
                        // BF16 h rows, two 64-wide halves (split by the converters)
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            for (int i = kBoxKinds - 1, r = 0; i >= 0; --i) {
                                const int hh = kBoxRows << i;
                                if (hh > kBNMax || b_rows - r < hh) continue;
                                ptx::tma_load_2d(sb + half * C::kBHalf + r * kTileK * 2, &tmH.m[i], kx + half * kTileK,
                                                 it.tl.y + r, bar(FULL0 + stage), pol_x);
                                r += hh;
                            }
                        }
                    } else {
                        // the x pieces: rows 2j (p1) and 2j + 1 (p2) of token row j, 128 bytes each
                        for (int i = kBoxKinds - 1, r = 0; i >= 0; --i) {
                            const int hh = kBoxRows << i;
                            if (hh > 2 * kBNMax || 2 * b_rows - r < hh) continue;
                            ptx::tma_load_2d(sb + r * kF8KStage, &tmX.m[i], kx, 2 * it.tl.y + r, bar(FULL0 + stage),
                                             pol_x);
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
                const int b_rows = ((it.tl.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
                const uint32_t idesc = idesc_e4m3_f32(kTileM, 2 * b_rows);
                const uint32_t d0 = tmem_base + s0 * C::kSlotCols, d1 = tmem_base + s1 * C::kSlotCols;
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs) ||
                        !ptx::mbar_wait(bar(CONV0 + stage), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    const uint32_t s8 = sa + 2 * C::kA;
#pragma unroll
                    for (int kk = 0; kk < kF8KStage / 32; ++kk) {
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(s8 + kk * 32);
                        const uint32_t accum = (kc | kk) ? 1u : 0u;
                        mma_e4m3(d0, ptx::sw128_kmajor_desc(sa + kk * 32), bdesc, idesc, accum);
                        mma_e4m3(d1, ptx::sw128_kmajor_desc(sa + C::kA + kk * 32), bdesc, idesc, accum);
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
        // ---------------------------------------------------------------- converters
        const int ct = threadIdx.x - (64 + 32 * kEpiWarps);  // 0 .. kCvtThreads - 1
        constexpr int kMaxTasks = (kBNMax * 8 + kCvtThreads - 1) / kCvtThreads;  // (row, chunk) per thread
        int stage = 0, rslot = 0;
        uint32_t phase = 0, rphase = 0;
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
            // h's row maxima are final once the tile's gate/up epilogues are all counted
            if (it.down && !wait_counter(args.tile_done + it.tile, args.m_gu * kEpiWarps, abort_flag)) {
                ok = false;
                break;
            }
            const int b_rows = ((it.tl.z + kBoxRows - 1) / kBoxRows) * kBoxRows;
            float inv[kMaxTasks];
#pragma unroll
            for (int q = 0; q < kMaxTasks; ++q) {
                const int task = ct + q * kCvtThreads;
                const int j = task >> 3;
                inv[q] = 0.0f;  // padding rows (j >= rows) get zero pieces
                if (it.down && task < b_rows * 8 && j < it.tl.z) {
                    float sc;
                    row_scale(args.amax_h[it.tl.y + j], sc, inv[q]);
                }
            }
            const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
            for (int kc = 0; kc < k_chunks; ++kc) {
                if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                if (it.down) {
                    // The pieces overwrite the BF16 rows they come from: every converter
                    // thread first computes its tasks' pieces in registers, then all of them
                    // meet at a named barrier, then they store.
                    uint8_t* buf = smem + stage * C::kStage + 2 * C::kA;
                    uint4 o1[kMaxTasks], o2[kMaxTasks];
#pragma unroll
                    for (int q = 0; q < kMaxTasks; ++q) {
                        const int task = ct + q * kCvtThreads;
                        o1[q] = make_uint4(0, 0, 0, 0);
                        o2[q] = make_uint4(0, 0, 0, 0);
                        if (task < b_rows * 8 && inv[q] != 0.0f) {
                            // elements 16c .. 16c+15 of token row j: half c/4 of the BF16 rows,
                            // 16-byte chunks 2(c%4) and 2(c%4)+1 of row j (128-byte swizzle)
                            const int j = task >> 3, c = task & 7, sw = j & 7;
                            const uint8_t* row_src = buf + (c >> 2) * C::kBHalf + j * 128;
                            const int q0 = 2 * (c & 3);
                            const uint4 v0 = *reinterpret_cast<const uint4*>(row_src + ((q0 ^ sw) << 4));
                            const uint4 v1 = *reinterpret_cast<const uint4*>(row_src + (((q0 + 1) ^ sw) << 4));
                            uint2 a1, a2, b1, b2;
                            split8(v0, inv[q], a1, a2);
                            split8(v1, inv[q], b1, b2);
                            o1[q] = make_uint4(a1.x, a1.y, b1.x, b1.y);
                            o2[q] = make_uint4(a2.x, a2.y, b2.x, b2.y);
                        }
                    }
                    asm volatile("bar.sync 1, %0;" ::"n"(kCvtThreads) : "memory");  // converters only
#pragma unroll
                    for (int q = 0; q < kMaxTasks; ++q) {
                        const int task = ct + q * kCvtThreads;
                        if (task < b_rows * 8) {
                            // p1 of token row j is piece row 2j, p2 piece row 2j + 1; chunk c
                            const int j = task >> 3, c = task & 7;
                            *reinterpret_cast<uint4*>(buf + (2 * j) * 128 + ((c ^ ((2 * j) & 7)) << 4)) = o1[q];
                            *reinterpret_cast<uint4*>(buf + (2 * j + 1) * 128 + ((c ^ ((2 * j + 1) & 7)) << 4)) =
                                o2[q];
                        }
                    }
                    fence_proxy_async_smem();  // the MMA (async proxy) reads the pieces
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(CONV0 + stage));
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
            const uint32_t t0 = tmem_base + lane_off + s0 * C::kSlotCols, t1 = tmem_base + lane_off + s1 * C::kSlotCols;
            const int col = (it.down ? it.m * 2 * kTileM : it.m * kTileM) + row;
            const bool col1_ok = col + kTileM < args.d;  // down: the pair's second tile exists
            float sc0, sc1;
            if (!it.down) {
                sc0 = args.gs[static_cast<size_t>(it.tl.x) * args.I + col];
                sc1 = args.us[static_cast<size_t>(it.tl.x) * args.I + col];
            } else {
                sc0 = args.ds[static_cast<size_t>(it.tl.x) * args.d + col];
                sc1 = col1_ok ? args.ds[static_cast<size_t>(it.tl.x) * args.d + col + kTileM] : 0.0f;
            }
            for (int c0 = col_part * 16; c0 < it.tl.z; c0 += kColStep) {
                // the row scale of token column c0 + lane (lanes 0..15), shared below
                float s_lane = 1.0f;
                if (lane < 16 && c0 + lane < it.tl.z) {
                    const int prow = it.tl.y + c0 + lane;
                    float amax = 0.0f;
                    if (it.down) {
                        amax = args.amax_h[prow];
                    } else {
                        const int src = args.perm_src[prow];
                        if (static_cast<unsigned>(src) < static_cast<unsigned>(args.n_tokens)) amax = args.xmax[src];
                    }
                    float inv;
                    row_scale(amax, s_lane, inv);
                }
                // token column c0 + j: its p1 product in accumulator column 2(c0 + j), its p2
                // product in the next one
                uint32_t a[32], b[32];
                ptx::tmem_ld16(t0 + 2 * c0, *reinterpret_cast<uint32_t(*)[16]>(a));
                ptx::tmem_ld16(t0 + 2 * c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(a + 16));
                ptx::tmem_ld16(t1 + 2 * c0, *reinterpret_cast<uint32_t(*)[16]>(b));
                ptx::tmem_ld16(t1 + 2 * c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(b + 16));
                ptx::tmem_wait_ld();
                if (!it.down) {
                    float hmax[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float s = __shfl_sync(0xffffffffu, s_lane, j);
                        hmax[j] = 0.0f;
                        if (c0 + j < it.tl.z) {
                            const float gv = sc0 * (s * (__uint_as_float(a[2 * j]) + __uint_as_float(a[2 * j + 1]) * 0.0625f));
                            const float uv = sc1 * (s * (__uint_as_float(b[2 * j]) + __uint_as_float(b[2 * j + 1]) * 0.0625f));
                            const bf16 hb = __float2bfloat16_rn(__fdividef(gv, 1.0f + __expf(-gv)) * uv);
                            args.h[static_cast<size_t>(it.tl.y + c0 + j) * args.I + col] = hb;
                            hmax[j] = fabsf(__bfloat162float(hb));
                        }
                    }
                    // largest |h| of each token column over this warp's 32 rows, then over
                    // every CTA writing the row (atomicMax on the bits of a non-negative float)
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) hmax[j] = fmaxf(hmax[j], __shfl_xor_sync(0xffffffffu, hmax[j], o));
                    }
                    float mine = 0.0f;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (lane == j) mine = hmax[j];
                    if (lane < 16 && c0 + lane < it.tl.z)
                        atomicMax(reinterpret_cast<int*>(args.amax_h) + it.tl.y + c0 + lane, __float_as_int(mine));
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float s = __shfl_sync(0xffffffffu, s_lane, j);
                        if (c0 + j < it.tl.z) {
                            const size_t r0 = static_cast<size_t>(it.tl.y + c0 + j) * args.d;
                            const float y0 = sc0 * (s * (__uint_as_float(a[2 * j]) + __uint_as_float(a[2 * j + 1]) * 0.0625f));
                            const float y1 = sc1 * (s * (__uint_as_float(b[2 * j]) + __uint_as_float(b[2 * j + 1]) * 0.0625f));
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
                // publish this warp's h stores (read by TMA in other CTAs) and its row maxima
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
cudaError_t launch_f8(const CUtensorMap& wg, const CUtensorMap& wu, const CUtensorMap& wd, const BMaps& x,
                      const BMaps& h, const MlpArgs& args, int grid, cudaStream_t st) {
    using C = F8Cfg<kBNMax>;
    cudaError_t e = set_smem_limit_once<expert_mlp_f8_kernel<kBNMax>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const cudaError_t le_ =
        launch_pdl(expert_mlp_f8_kernel<kBNMax>, dim3(grid), dim3(kF8Threads), C::kSmemBytes, st, wg, wu, wd, x, h,
                   args);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

// Per BF16 token row t (one warp): xmax[t] = max_j |x[t][j]|, then the row's two E4M3
// pieces under its power-of-two scale, x8[t] = p1 [d] then p2 [d]; amax_h[0, rows) = 0.
__global__ void __launch_bounds__(256) fp8_prep_kernel(const uint4* __restrict__ x, int T, int row_vecs,
                                                       float* __restrict__ xmax, uint2* __restrict__ x8,
                                                       float* __restrict__ amax_h, int rows) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const uint4* row = x + static_cast<size_t>(t) * row_vecs;
        float m = 0.0f;
        for (int v = lane; v < row_vecs; v += 32) {
            const uint4 w = row[v];
            const uint32_t p[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&p[i]));
                m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) xmax[t] = m;
        float sc, inv;
        row_scale(m, sc, inv);
        uint2* out = x8 + static_cast<size_t>(t) * 2 * row_vecs;  // 8 codes per uint2
        for (int v = lane; v < row_vecs; v += 32) {
            uint2 p1, p2;
            split8(row[v], inv, p1, p2);
            out[v] = p1;
            out[row_vecs + v] = p2;
        }
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < rows; i += gridDim.x * blockDim.x) amax_h[i] = 0.0f;
}

}  // namespace

int gemm_bn_max_f8(const Shape& s, int T) {
    if (T <= 32) return 32;
    const long long avg_rows = static_cast<long long>(T) * s.top_k / s.E;
    return avg_rows <= 24 ? 64 : 128;
}

cudaError_t launch_fp8_prep(const bf16* x, int d, int T, float* xmax, uint8_t* x8, float* amax_h, int rows,
                            int num_sms, cudaStream_t st) {
    long long blocks = (T + 7) / 8;
    const long long cap = static_cast<long long>(num_sms) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const cudaError_t le_ = launch_pdl(fp8_prep_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                                       reinterpret_cast<const uint4*>(x), T, d / 8, xmax, reinterpret_cast<uint2*>(x8),
                                       amax_h, rows);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_expert_mlp_f8(const Shape& s, const Fp8Experts& q, const uint8_t* x8_perm, int rows, int T,
                                 const int* perm_src, const float* xmax, float* amax_h, const int4* tiles,
                                 int* tile_done, int max_tiles, int bn_max, bf16* h, bf16* y, int* status,
                                 int num_sms, cudaStream_t st) {
    if (bn_max > 128) return cudaErrorInvalidValue;
    CUtensorMap wg, wu, wd;
    BMaps bx, bh;
    const char* why = nullptr;
    if (!encode_tmap_u8_2d(&wg, q.wg, static_cast<uint64_t>(s.E) * s.I, s.d, kTileM, kF8KStage, &why) ||
        !encode_tmap_u8_2d(&wu, q.wu, static_cast<uint64_t>(s.E) * s.I, s.d, kTileM, kF8KStage, &why) ||
        !encode_tmap_u8_2d(&wd, q.wd, static_cast<uint64_t>(s.E) * s.d, s.I, kTileM, kF8KStage, &why) ||
        !encode_bmaps_u8(&bx, x8_perm, 2ull * rows, s.d, 2 * bn_max, &why) ||
        !encode_bmaps(&bh, h, rows, s.I, bn_max, &why))
        return cudaErrorInvalidValue;
    MlpArgs a = mlp_args(s, rows, tiles, tile_done, max_tiles, h, y, status, kF8KStage);
    a.gs = q.gs;
    a.us = q.us;
    a.ds = q.ds;
    a.perm_src = perm_src;
    a.xmax = xmax;
    a.amax_h = amax_h;
    a.n_tokens = T;
    const int grid = mlp_grid(a, max_tiles, num_sms);
    if (bn_max <= 32) return launch_f8<32>(wg, wu, wd, bx, bh, a, grid, st);
    if (bn_max <= 64) return launch_f8<64>(wg, wu, wd, bx, bh, a, grid, st);
    return launch_f8<128>(wg, wu, wd, bx, bh, a, grid, st);
}

}  // namespace beam
