// The routed experts on NVFP4 weights with NVFP4 tensor-core products (tcgen05.mma
// kind::mxf4nvf4 with 16-element block scales): the block of beam_moe_forward_nvfp4 (Glonce
// "Reflection releases Beam ...", Hardware paragraph: the NVFP4 checkpoint runs natively on
// Blackwell; the reading W[r][c] = t * e4m3(bs[r][c/16]) * e2m1(q[r][c])).
//
// Why: the block-scaled FP4 product takes K = 64 per instruction, four times the 16 of a
// BF16 product, and applies the E4M3 block scales of both operands itself, so the codes and
// block scales of the weights go to the tensor cores as they are stored: one instruction per
// 8,192 weights of 4.5 bits, where widening them to BF16 took one per 2,048 plus the
// converter work (which made that path ALU-bound at a third of the HBM rate).
//
// Both operands of this product are NVFP4, so the activations (x for the gate/up product, h
// for the down product) enter as four NVFP4 pieces per row. For each block of 16 consecutive
// elements, with r_0 = v and g_p = 4^(-p):
//     u_p = the least E4M3 value >= max|r_p| * 4^p / 6,   s_p = g_p * u_p,
//     q_p = e2m1(r_p / s_p),   r_(p+1) = r_p - s_p * q_p        (p = 0 .. 3)
// so v = sum_p g_p * u_p * q_p + r_4 with every step exact in FP32. Each piece leaves at most
// s_p of its block (the largest E2M1 gap is 2) and s_p <= 1.125 max|r_p| / 6, so
// |r_4| <= (1.125 / 6)^4 max|v| = 1.2e-3 of the block's largest magnitude (usually far less),
// above the floor of the smallest scales (2^-9 * 4^-3). The factor 4 per piece keeps every
// later scale below the first one (max|r_p| * 4^p / 6 <= 0.75^p max|v| / 6), so no piece
// after the first runs into the E4M3 maximum; with 8 the worst case grows by 1.5 per piece
// and blocks above about 1,100 can lose precision in the last pieces.
// The pieces of token row j of a tile are the B operand's rows 4j .. 4j+3 and u_p their
// UE4M3 block scales; one MMA over the tile's piece rows (4 per token, rounded up to 16)
// gives all four partial products of every token, and the epilogue
// takes acc = sum_p g_p * D[:, 4c + p] per token column c, then the weight matrix's tensor
// scale, SwiGLU (gate/up, which splits h into its pieces at once) or the BF16 expert output
// (down). The first piece covers block maxima up to 6 * 448 = 2688; a larger one is clamped
// and recorded in the status word (kStatusRange).
//
// x is split by a preparatory kernel before dispatch (the pieces take 2d bytes per row, as a
// BF16 row; their block scales d/4 more bytes, moved by the dispatch beside them); h is split
// by the gate/up epilogues, which write its pieces and scales in the layout the down items
// load. Items, ids, scheduling, completion counters and bounded waits are those of the BF16
// kernel (expert_mlp.cu). Roles (one CTA per SM):
//   warp 0 lane 0: scheduler + TMA producer: per stage (K = 256) the two weight code tiles
//                  [128 rows x 128 bytes] (128-byte swizzle) and their block-scale tiles
//                  [128 x 16 bytes], the tile's activation piece rows [128 bytes each] and
//                  their block scales [16 bytes each];
//   warp 1:        TMEM; lane 0 issues the MMAs (M = 128, N = the piece rows, K = 64, A and
//                  B from shared memory, scale factors from TMEM) once the stage's scales
//                  are there;
//   warps 2..9:    epilogue (two warps per TMEM lane quarter, alternate 8-token granules);
//                  each reads all its accumulator columns into registers and hands the
//                  accumulators back before its arithmetic;
//   warps 10..13:  scale-factor writers, one per TMEM lane quarter: each copies the stage's
//                  block scales from shared memory into TMEM in the layout the MMA reads
//                  (matrix row r at column r / 32 and lane r % 32 of a lane quarter, the four
//                  16-element blocks of a K = 64 step in the four bytes of the word). Each of
//                  the tensor core's four sub-partitions reads its own lane quarter: the
//                  weights' scales only for its 32 rows, the activation pieces' scales for
//                  every row (measured with a probe: scales left out of the other quarters
//                  change no result).
#include <type_traits>

#include "expert_common.cuh"

namespace beam {
namespace {

using namespace mlp;

constexpr int kSfWarps = 4;
constexpr int kQ4Threads = 64 + 32 * kEpiWarps + 32 * kSfWarps;
constexpr int kQStage = 256;  // K per stage: one 128-byte row of FP4 codes
constexpr int kPieces = 4;
constexpr int kPieceShift = 2;  // piece p is weighted 2^(-kPieceShift * p)

template <int kBNMax>
struct Q4Cfg {
    static constexpr int kA = kTileM * (kQStage / 2);   // one weight code tile: 16 KB
    static constexpr int kS = kTileM * (kQStage / 16);  // its block scales: 2 KB
    static constexpr int kBRows = kPieces * kBNMax;     // activation piece rows of a tile
    static constexpr int kB = kBRows * (kQStage / 2);   // their codes
    static constexpr int kBS = kBRows * (kQStage / 16); // their block scales
    static constexpr int kOffS = 2 * kA, kOffB = 2 * kA + 2 * kS, kOffBS = kOffB + kB;
    static constexpr int kStage = (kOffBS + kBS + 1023) / 1024 * 1024;
    static constexpr int kBudget = 227 * 1024 - 2048;
    static constexpr int kStages = (kBudget / kStage) > 5 ? 5 : (kBudget / kStage);
    static constexpr int kSlotCols = kBRows;  // an accumulator: all pieces of every token
    // scale factors per stage: A (2 tiles x 4 K steps x 4 row groups of 32) then B (4 K
    // steps x 4 columns, of which the ceil(kBRows / 32) row groups use the first)
    static constexpr int kSfB = (kBRows + 31) / 32;
    static constexpr int kSfCols = 32 + 16;
    // four accumulators (two items in flight) when they fit beside the scale factors
    static constexpr int kSlots = 4 * kSlotCols + kStages * kSfCols <= 512 ? 4 : 2;
    static constexpr int kSfBase = kSlots * kSlotCols;
    static constexpr int kTmemCols = 512;
    // FULL (TMA), SFREADY (scales in TMEM), EMPTY (MMAs done) per stage; TFULL, TEMPTY per
    // slot; RFULL, REMPTY per ring entry; DRAIN.
    static constexpr int kNumBars = 3 * kStages + 2 * kSlots + 2 * kRing + 1;
    static constexpr int kSmemBytes = 1024 + kStages * kStage + kNumBars * 8 + kRing * 4 + 16 + kRing * 32 + 16;
    static_assert(kBRows % kBoxRows == 0 && kSfB <= 4, "piece rows in whole boxes, at most 128");
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kOffB % 1024 == 0, "swizzled tiles stay 1024-byte aligned");
    static_assert(kSfBase + kStages * kSfCols <= kTmemCols, "TMEM columns");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Instruction descriptor, kind::mxf4nvf4 (the accumulator is always F32): A and B E2M1
// (bits 7-9 = 1, bits 10-11 = 1), both K-major, N >> 3 in bits 17-22, UE4M3 scale factors
// (bit 23 = 0), M >> 4 in bits 24-28; the scale-factor ids (bits 4-5 for B, 29-30 for A)
// stay 0, as the four scales of a K = 64 step fill the whole 32-bit word.
__device__ __forceinline__ uint32_t idesc_nvf4(int M, int N) {
    return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// D[tmem] (+)= (A scaled per 16 by SFA) * (B scaled per 16 by SFB)^T, E2M1 operands, K = 64.
__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// The least E4M3 value u >= x for 0 <= x <= 448, and its code (codes 0 .. 0x7E are ordered
// like their values). From 2^-6 up, E4M3 values are the FP32 values with 3 fraction bits:
// round the FP32 significand up to them (a carry moves into the exponent); below 2^-6 they
// are the multiples of 2^-9, whose codes are those multiples (code 8 is 2^-6 either way).
// Larger x give 448 and set `over`.
__device__ __forceinline__ uint32_t e4m3_ceil(float x, float& u, bool& over) {
    if (x >= 0.015625f) {
        uint32_t b = (__float_as_uint(x) + 0xFFFFFu) & ~0xFFFFFu;
        if (b > 0x43E00000u) {  // above 448
            b = 0x43E00000u;
            over = true;
        }
        u = __uint_as_float(b);
        return (((b >> 23) - 120u) << 3) | ((b >> 20) & 7u);
    }
    const float k = ceilf(x * 512.0f);
    u = k * 0.001953125f;
    return static_cast<uint32_t>(k);
}

// The E2M1 codes nearest to y0 and y1 (saturated at +-6) in one byte, y0's in the low half,
// and their values. (The paired conversion puts its first operand in the high half.)
__device__ __forceinline__ uint32_t e2m1_pair(float y0, float y1, float& v0, float& v1) {
    uint32_t c, f;
    asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n" : "=r"(c) : "f"(y1), "f"(y0));
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(f) : "r"(c));
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&f));
    v0 = v.x;
    v1 = v.y;
    return c & 0xffu;
}

// Piece p of a block whose remainder has largest magnitude amax: the E4M3 scale u (its code
// returned), the piece's step s = 4^-p u and 1 / s (0 for an all-zero remainder). `over`
// is set when the first piece needs a scale above 448.
template <int p>
__device__ __forceinline__ uint32_t piece_scale(float amax, float& s, float& inv, bool& over) {
    constexpr float kUp = static_cast<float>(1 << (kPieceShift * p)) / 6.0f;
    constexpr float kDown = 1.0f / static_cast<float>(1 << (kPieceShift * p));
    float u;
    bool o = false;
    const uint32_t code = e4m3_ceil(amax * kUp, u, o);
    if (p == 0 && o) over = true;
    s = u * kDown;
    inv = u > 0.0f ? static_cast<float>(1 << (kPieceShift * p)) * __frcp_rn(u) : 0.0f;
    return code;
}

// A work item as the scheduler decoded it, handed to the other roles with its id (so they
// do not read the work list from global memory again).
struct RingItem {
    int4 tl;   // {expert, first row, rows, 0}
    int tile;
    int m;
    int flags;  // bit 0: down item; bit 1: valid
    int pad;
};

__device__ __forceinline__ MItem item_of(const RingItem& r) {
    MItem it;
    it.tl = r.tl;
    it.tile = r.tile;
    it.m = r.m;
    it.n_t = 0;
    it.down = (r.flags & 1) != 0;
    it.ok = (r.flags & 2) != 0;
    return it;
}

template <int kBNMax>
__global__ void __launch_bounds__(kQ4Threads, 1)
    expert_mlp_nvf4_kernel(const __grid_constant__ CUtensorMap tmWg, const __grid_constant__ CUtensorMap tmWu,
                           const __grid_constant__ CUtensorMap tmWd, const __grid_constant__ CUtensorMap tmSg,
                           const __grid_constant__ CUtensorMap tmSu, const __grid_constant__ CUtensorMap tmSd,
                           const __grid_constant__ BMaps tmX, const __grid_constant__ BMaps tmXs,
                           const __grid_constant__ BMaps tmH, const __grid_constant__ BMaps tmHs,
                           const __grid_constant__ MlpArgs args, uint8_t* __restrict__ h4,
                           uint8_t* __restrict__ hs) {
    using C = Q4Cfg<kBNMax>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStage);
    volatile int* ring = reinterpret_cast<volatile int*>(bars + C::kNumBars);
    RingItem* items = reinterpret_cast<RingItem*>((reinterpret_cast<uintptr_t>(ring + kRing) + 15) & ~uintptr_t(15));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(items + kRing);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    constexpr int FULL0 = 0, SFR0 = C::kStages, EMPTY0 = 2 * C::kStages, TFULL0 = 3 * C::kStages,
                  TEMPTY0 = TFULL0 + C::kSlots, RFULL0 = TEMPTY0 + C::kSlots, REMPTY0 = RFULL0 + kRing,
                  DRAIN = REMPTY0 + kRing;
    auto bar = [&](int i) { return ptx::smem_u32(bars + i); };
    int* status = args.status;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(bar(FULL0 + s), 1);
            ptx::mbar_init(bar(SFR0 + s), kSfWarps);
            ptx::mbar_init(bar(EMPTY0 + s), 1);
        }
        for (int s = 0; s < C::kSlots; ++s) {
            ptx::mbar_init(bar(TFULL0 + s), 1);
            ptx::mbar_init(bar(TEMPTY0 + s), 32 * kEpiWarps);
        }
        for (int r = 0; r < kRing; ++r) {
            ptx::mbar_init(bar(RFULL0 + r), 1);
            ptx::mbar_init(bar(REMPTY0 + r), 1 + kEpiWarps + kSfWarps);
        }
        ptx::mbar_init(bar(DRAIN), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmWg);
        ptx::prefetch_tmap(&tmWu);
        ptx::prefetch_tmap(&tmWd);
        ptx::prefetch_tmap(&tmSg);
        ptx::prefetch_tmap(&tmSu);
        ptx::prefetch_tmap(&tmSd);
        for (int i = 0; i < kBoxKinds && (kBoxRows << i) <= C::kBRows; ++i) {
            ptx::prefetch_tmap(&tmX.m[i]);
            ptx::prefetch_tmap(&tmXs.m[i]);
            ptx::prefetch_tmap(&tmH.m[i]);
            ptx::prefetch_tmap(&tmHs.m[i]);
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
                MItem it;
                it.ok = false;
                if (id >= 0) it = decode(args, id, n_gu, n_tiles);
                if (!ptx::mbar_wait(bar(REMPTY0 + rslot), rphase ^ 1, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ring[rslot] = id;
                if (id >= 0) {
                    RingItem r;
                    r.tl = it.tl;
                    r.tile = it.tile;
                    r.m = it.m;
                    r.flags = (it.down ? 1 : 0) | (it.ok ? 2 : 0);
                    r.pad = 0;
                    items[rslot] = r;
                }
                ptx::mbar_arrive(bar(RFULL0 + rslot));  // release: the id and item are visible to the waiters
                if (++rslot == kRing) {
                    rslot = 0;
                    rphase ^= 1;
                }
                if (id < 0) break;
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
                const int p_rows = (kPieces * it.tl.z + kBoxRows - 1) / kBoxRows * kBoxRows;  // piece rows loaded
                const uint32_t bytes = 2 * C::kA + 2 * C::kS + p_rows * (kQStage / 2 + kQStage / 16);
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                const int a_row = it.down ? it.tl.x * args.d + it.m * 2 * kTileM : it.tl.x * args.I + it.m * kTileM;
                const BMaps& bm = it.down ? tmH : tmX;
                const BMaps& bsm = it.down ? tmHs : tmXs;
                const uint64_t pol_w = it.n_t > 1 ? pol_w_shared : pol_w_once;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    const int kb = kc * (kQStage / 2);   // byte column of the codes
                    const int ks = kc * (kQStage / 16);  // byte column of the block scales
                    if (!ptx::mbar_wait(bar(EMPTY0 + stage), phase ^ 1, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    ptx::mbar_arrive_expect_tx(bar(FULL0 + stage), bytes);
                    if (it.down) {
                        ptx::tma_load_2d(sa, &tmWd, kb, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWd, kb, a_row + kTileM, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kOffS, &tmSd, ks, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kOffS + C::kS, &tmSd, ks, a_row + kTileM, bar(FULL0 + stage), pol_w);
                    } else {
                        ptx::tma_load_2d(sa, &tmWg, kb, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kA, &tmWu, kb, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kOffS, &tmSg, ks, a_row, bar(FULL0 + stage), pol_w);
                        ptx::tma_load_2d(sa + C::kOffS + C::kS, &tmSu, ks, a_row, bar(FULL0 + stage), pol_w);
                    }
                    // piece rows 4j .. 4j+3 of token row j: codes (128 bytes) and block scales (16)
                    for (int i = kBoxKinds - 1, r = 0; i >= 0; --i) {
                        const int hh = kBoxRows << i;
                        if (hh > C::kBRows || p_rows - r < hh) continue;
                        ptx::tma_load_2d(sa + C::kOffB + r * (kQStage / 2), &bm.m[i], kb, kPieces * it.tl.y + r,
                                         bar(FULL0 + stage), pol_x);
                        ptx::tma_load_2d(sa + C::kOffBS + r * (kQStage / 16), &bsm.m[i], ks, kPieces * it.tl.y + r,
                                         bar(FULL0 + stage), pol_x);
                        r += hh;
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
                const MItem it = item_of(items[rslot]);
                ptx::mbar_arrive(bar(REMPTY0 + rslot));
                if (++rslot == kRing) {
                    rslot = 0;
                    rphase ^= 1;
                }
                if (id < 0) break;
                if (!it.ok || it.tl.z > kBNMax) continue;
                const int s0 = slot, s1 = (slot + 1) % C::kSlots;
                if (!ptx::mbar_wait(bar(TEMPTY0 + s0), ((tph >> s0) & 1u) ^ 1u, abort_flag, kWaitLimitNs) ||
                    !ptx::mbar_wait(bar(TEMPTY0 + s1), ((tph >> s1) & 1u) ^ 1u, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const int p_rows = (kPieces * it.tl.z + kBoxRows - 1) / kBoxRows * kBoxRows;
                const uint32_t idesc = idesc_nvf4(kTileM, p_rows);  // N: the piece rows loaded
                const uint32_t d0 = tmem_base + s0 * C::kSlotCols, d1 = tmem_base + s1 * C::kSlotCols;
                const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
                for (int kc = 0; kc < k_chunks; ++kc) {
                    if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs) ||
                        !ptx::mbar_wait(bar(SFR0 + stage), phase, abort_flag, kWaitLimitNs)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStage);
                    const uint32_t sb = sa + C::kOffB;
                    const uint32_t sf = tmem_base + C::kSfBase + stage * C::kSfCols;
#pragma unroll
                    for (int kk = 0; kk < kQStage / 64; ++kk) {
                        const uint64_t bdesc = ptx::sw128_kmajor_desc(sb + kk * 32);
                        const uint32_t accum = (kc | kk) ? 1u : 0u;
                        const uint32_t sfb = sf + 32 + kk * 4;
                        mma_nvf4(d0, ptx::sw128_kmajor_desc(sa + kk * 32), bdesc, idesc, sf + kk * 4, sfb, accum);
                        mma_nvf4(d1, ptx::sw128_kmajor_desc(sa + C::kA + kk * 32), bdesc, idesc, sf + 16 + kk * 4, sfb,
                                 accum);
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
        // ---------------------------------------------------------------- scale-factor writers
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        int stage = 0, rslot = 0;
        uint32_t phase = 0, rphase = 0;
        bool ok = true;
        while (ok) {
            if (!ptx::mbar_wait(bar(RFULL0 + rslot), rphase, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
            }
            const int id = ring[rslot];
            const MItem it = item_of(items[rslot]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(REMPTY0 + rslot));
            if (++rslot == kRing) {
                rslot = 0;
                rphase ^= 1;
            }
            if (id < 0) break;
            if (!it.ok || it.tl.z > kBNMax) continue;
            const int k_chunks = it.down ? args.kc_dn : args.kc_gu;
            for (int kc = 0; kc < k_chunks; ++kc) {
                if (!ptx::mbar_wait(bar(FULL0 + stage), phase, abort_flag, kWaitLimitNs)) {
                    ok = false;
                    break;
                }
                const uint8_t* st_base = smem + stage * C::kStage;
                const uint32_t sf = tmem_base + lane_off + C::kSfBase + stage * C::kSfCols;
                // The tensor core's four sub-partitions each read scale factors from their own
                // TMEM lane quarter: the weights' scales of row r (K step kk) only by the
                // sub-partition of rows 32q .. 32q+31 (lane r, column kk*4 + r/32 of the
                // tile's group), the activation pieces' scales of row r by every one (lane
                // 32q + r % 32, column kk*4 + r/32). So this warp loads only its quarter's
                // weight rows (one 16-byte row per lane and tile) but every piece row.
                const int q = warp & 3;
                uint32_t a[32];
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const uint4 w = *reinterpret_cast<const uint4*>(st_base + C::kOffS + t * C::kS + (32 * q + lane) * 16);
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        a[t * 16 + 0 * 4 + g] = w.x;
                        a[t * 16 + 1 * 4 + g] = w.y;
                        a[t * 16 + 2 * 4 + g] = w.z;
                        a[t * 16 + 3 * 4 + g] = w.w;
                    }
                }
                ptx::tmem_st32(sf, a);
                // column 32 + kk*4 + g holds piece row 32g + lane (zero past the tile's rows)
                uint32_t b[16];
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint4 w = make_uint4(0u, 0u, 0u, 0u);
                    if (g < C::kSfB && 32 * g + lane < C::kBRows)
                        w = *reinterpret_cast<const uint4*>(st_base + C::kOffBS + (32 * g + lane) * 16);
                    b[0 * 4 + g] = w.x;
                    b[1 * 4 + g] = w.y;
                    b[2 * 4 + g] = w.z;
                    b[3 * 4 + g] = w.w;
                }
                tmem_st16(sf + 32, b);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(SFR0 + stage));
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
        const int col_part = (warp - 2) >> 2;        // which 8-token granules this warp takes
        constexpr int kTokStep = 8 * (kEpiWarps / 4);
        const int I2 = args.I / 2, I16 = args.I / 16;
        int rslot = 0, slot = 0;
        uint32_t rphase = 0, tph = 0;
        bool over = false;  // an h block beyond the first piece's range
        while (true) {
            if (!ptx::mbar_wait(bar(RFULL0 + rslot), rphase, abort_flag, kWaitLimitNs)) {
                *abort_flag = 1;
                flag_status(status, kStatusWaitTimeout);
                break;
            }
            const int id = ring[rslot];
            const MItem it = item_of(items[rslot]);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(REMPTY0 + rslot));
            if (++rslot == kRing) {
                rslot = 0;
                rphase ^= 1;
            }
            if (id < 0) break;
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
                sc0 = args.gs[it.tl.x];
                sc1 = args.us[it.tl.x];
            } else {
                sc0 = args.ds[it.tl.x];
                sc1 = col1_ok ? sc0 : 0.0f;
            }
            // Every accumulator value this warp needs goes to registers first (at most kGran
            // granules of 8 tokens, each reduced over its pieces at once); the accumulators then
            // go back to the MMAs while the arithmetic below runs.
            constexpr int kGran = (kBNMax + kTokStep - 1) / kTokStep;
            constexpr float kG1 = 1.0f / (1 << kPieceShift), kG2 = kG1 * kG1, kG3 = kG2 * kG1;  // piece weights
            float vag[kGran][8], vbg[kGran][8];
#pragma unroll
            for (int g = 0; g < kGran; ++g) {
                const int c0 = col_part * 8 + g * kTokStep;
                if (c0 >= it.tl.z) break;  // warp-uniform
                // token column c0 + j: its piece p product in accumulator column 4(c0 + j) + p
                uint32_t a[32], b[32];
                ptx::tmem_ld16(t0 + 4 * c0, *reinterpret_cast<uint32_t(*)[16]>(a));
                ptx::tmem_ld16(t0 + 4 * c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(a + 16));
                ptx::tmem_ld16(t1 + 4 * c0, *reinterpret_cast<uint32_t(*)[16]>(b));
                ptx::tmem_ld16(t1 + 4 * c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(b + 16));
                ptx::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    vag[g][j] = __uint_as_float(a[4 * j]) + kG1 * __uint_as_float(a[4 * j + 1]) +
                                kG2 * __uint_as_float(a[4 * j + 2]) + kG3 * __uint_as_float(a[4 * j + 3]);
                    vbg[g][j] = __uint_as_float(b[4 * j]) + kG1 * __uint_as_float(b[4 * j + 1]) +
                                kG2 * __uint_as_float(b[4 * j + 2]) + kG3 * __uint_as_float(b[4 * j + 3]);
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(TEMPTY0 + s0));
            ptx::mbar_arrive(bar(TEMPTY0 + s1));
            tph ^= (1u << s0) | (1u << s1);
#pragma unroll
            for (int g = 0; g < kGran; ++g) {
                const int c0 = col_part * 8 + g * kTokStep;
                if (c0 >= it.tl.z) break;  // warp-uniform
                const float (&va)[8] = vag[g];
                const float (&vb)[8] = vbg[g];
                const int n_live = it.tl.z - c0;  // tokens j < n_live are rows of the tile
                const size_t prow0 = static_cast<size_t>(it.tl.y) + c0;
                if (!it.down) {
                    // SwiGLU in FP32, then h's four pieces over the 16-row block of each lane;
                    // the eight tokens run side by side
                    float r[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float gv = sc0 * va[j], uv = sc1 * vb[j];
                        r[j] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                    }
                    uint8_t* hrow = h4 + prow0 * kPieces * I2 + (col >> 1);
                    uint8_t* srow = hs + prow0 * kPieces * I16 + (col >> 4);
                    auto piece = [&](auto pc) {
                        constexpr int p = decltype(pc)::value;
                        float amax[8], sp[8], inv[8];
                        uint32_t ucode[8], word[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) amax[j] = fabsf(r[j]);
#pragma unroll
                        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
                            for (int j = 0; j < 8; ++j) amax[j] = fmaxf(amax[j], __shfl_xor_sync(0xffffffffu, amax[j], o));
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // columns past the tile's tokens hold whatever TMEM held: never flagged
                            bool o = false;
                            ucode[j] = piece_scale<p>(amax[j], sp[j], inv[j], o);
                            if (o && j < n_live) over = true;
                        }
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {
                            float q0, q1;
                            const uint32_t c = e2m1_pair(r[j] * inv[j], r[j + 1] * inv[j + 1], q0, q1);
                            r[j] -= sp[j] * q0;
                            r[j + 1] -= sp[j + 1] * q1;
                            // eight codes per word: lanes 8i .. 8i+7 -> nibbles 0 .. 7
                            word[j] = (c & 0xfu) << (4 * (lane & 7));
                            word[j + 1] = (c >> 4) << (4 * (lane & 7));
                        }
#pragma unroll
                        for (int o = 1; o < 8; o <<= 1)
#pragma unroll
                            for (int j = 0; j < 8; ++j) word[j] |= __shfl_xor_sync(0xffffffffu, word[j], o);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if (j >= n_live) break;  // warp-uniform
                            const size_t off = static_cast<size_t>(kPieces * j + p);
                            if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(hrow + off * I2) = word[j];
                            if ((lane & 15) == 0) srow[off * I16] = static_cast<uint8_t>(ucode[j]);
                        }
                    };
                    piece(std::integral_constant<int, 0>{});
                    piece(std::integral_constant<int, 1>{});
                    piece(std::integral_constant<int, 2>{});
                    piece(std::integral_constant<int, 3>{});
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j >= n_live) break;  // warp-uniform
                        const size_t r0 = (prow0 + j) * args.d;
                        args.y[r0 + col] = __float2bfloat16_rn(sc0 * va[j]);
                        if (col1_ok) args.y[r0 + col + kTileM] = __float2bfloat16_rn(sc1 * vb[j]);
                    }
                }
            }
            if (!it.down) {
                // publish this warp's h pieces (read by TMA in other CTAs)
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    atomicAdd(args.tile_done + it.tile, 1);
                }
            }
            slot = (slot + 2) % C::kSlots;
        }
        if (over) flag_status(status, kStatusRange);
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
cudaError_t launch_q4(const CUtensorMap (&w)[6], const BMaps& x, const BMaps& xs, const BMaps& h, const BMaps& hsm,
                      const MlpArgs& args, uint8_t* h4, uint8_t* hs, int grid, cudaStream_t st) {
    using C = Q4Cfg<kBNMax>;
    cudaError_t e = set_smem_limit_once<expert_mlp_nvf4_kernel<kBNMax>>(C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const cudaError_t le_ = launch_pdl(expert_mlp_nvf4_kernel<kBNMax>, dim3(grid), dim3(kQ4Threads), C::kSmemBytes,
                                       st, w[0], w[1], w[2], w[3], w[4], w[5], x, xs, h, hsm, args, h4, hs);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

// The four NVFP4 pieces of each 16-element block of the T BF16 token rows (one thread per
// block): codes x4[t][p][d/2] (element 2k in the low half of byte k), E4M3 block scales
// xs[t][p][d/16].
__global__ void __launch_bounds__(256) act4_prep_kernel(const uint4* __restrict__ x, int T, int d,
                                                        uint8_t* __restrict__ x4, uint8_t* __restrict__ xs,
                                                        int* status) {
    pdl_wait();
    pdl_trigger();
    const int nb = d / 16;
    const long long total = static_cast<long long>(T) * nb;
    bool over = false;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / nb), blk = static_cast<int>(i - static_cast<long long>(t) * nb);
        float r[16];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 w = x[(static_cast<size_t>(t) * d + blk * 16) / 8 + h];
            const uint32_t p[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&p[k]));
                r[8 * h + 2 * k] = f.x;
                r[8 * h + 2 * k + 1] = f.y;
            }
        }
        auto piece = [&](auto pc) {
            constexpr int p = decltype(pc)::value;
            float amax = 0.0f;
#pragma unroll
            for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(r[k]));
            float sp, inv;
            const uint32_t ucode = piece_scale<p>(amax, sp, inv, over);
            uint32_t packed[2] = {0u, 0u};
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                float q0, q1;
                const uint32_t c = e2m1_pair(r[k] * inv, r[k + 1] * inv, q0, q1);
                r[k] -= sp * q0;
                r[k + 1] -= sp * q1;
                packed[k >> 3] |= c << (4 * (k & 7));  // byte k/2: element k low, k+1 high
            }
            const size_t prow = static_cast<size_t>(kPieces) * t + p;
            *reinterpret_cast<uint2*>(x4 + prow * (d / 2) + blk * 8) = make_uint2(packed[0], packed[1]);
            xs[prow * nb + blk] = static_cast<uint8_t>(ucode);
        };
        piece(std::integral_constant<int, 0>{});
        piece(std::integral_constant<int, 1>{});
        piece(std::integral_constant<int, 2>{});
        piece(std::integral_constant<int, 3>{});
    }
    if (over) atomicCAS(status, 0, kStatusRange);
}

bool encode_bmaps_u8_plain(BMaps* b, const void* base, uint64_t rows, uint64_t cols, int box_max,
                           const char** why) {
    for (int i = 0; i < kBoxKinds; ++i) {
        const uint32_t hh = kBoxRows << i;
        if (static_cast<int>(hh) > box_max) {
            b->m[i] = b->m[0];
            continue;
        }
        if (!encode_tmap_u8_2d_plain(&b->m[i], base, rows, cols, hh, 16, why)) return false;
    }
    return true;
}

}  // namespace

// N-tiles of 16 token rows (64 piece rows, four accumulators) while experts average at most
// 8 rows, else 32 (128 piece rows: the two accumulators of one item fill TMEM beside the
// scale factors; faster at 4096 tokens than 20-row tiles with four accumulators).
int gemm_bn_max_nvf4(const Shape& s, int T) {
    const long long avg_rows = static_cast<long long>(T) * s.top_k / s.E;
    return avg_rows <= 8 ? 16 : 32;
}

cudaError_t launch_act4_prep(const bf16* x, int d, int T, uint8_t* x4, uint8_t* xs, int* status, int num_sms,
                             cudaStream_t st) {
    const long long total = static_cast<long long>(T) * (d / 16);
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const cudaError_t le_ = launch_pdl(act4_prep_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st,
                                       reinterpret_cast<const uint4*>(x), T, d, x4, xs, status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_expert_mlp_nvf4(const Shape& s, const Nvfp4Experts& q, const uint8_t* x4_perm,
                                   const uint8_t* xs_perm, int rows, const int4* tiles, int* tile_done, int max_tiles,
                                   int bn_max, uint8_t* h4, uint8_t* hs, bf16* y, int* status, int num_sms,
                                   cudaStream_t st) {
    if (bn_max > 32 || s.d % 256 || s.I % 256) return cudaErrorInvalidValue;
    CUtensorMap w[6];
    BMaps bx, bxs, bh, bhs;
    const char* why = nullptr;
    const uint64_t gu_rows = static_cast<uint64_t>(s.E) * s.I, dn_rows = static_cast<uint64_t>(s.E) * s.d;
    const uint64_t prows = static_cast<uint64_t>(kPieces) * rows;
    const int box_max = kPieces * bn_max;
    if (!encode_tmap_u8_2d(&w[0], q.wg, gu_rows, s.d / 2, kTileM, 128, &why) ||
        !encode_tmap_u8_2d(&w[1], q.wu, gu_rows, s.d / 2, kTileM, 128, &why) ||
        !encode_tmap_u8_2d(&w[2], q.wd, dn_rows, s.I / 2, kTileM, 128, &why) ||
        !encode_tmap_u8_2d_plain(&w[3], q.gbs, gu_rows, s.d / 16, kTileM, 16, &why) ||
        !encode_tmap_u8_2d_plain(&w[4], q.ubs, gu_rows, s.d / 16, kTileM, 16, &why) ||
        !encode_tmap_u8_2d_plain(&w[5], q.dbs, dn_rows, s.I / 16, kTileM, 16, &why) ||
        !encode_bmaps_u8(&bx, x4_perm, prows, s.d / 2, box_max, &why) ||
        !encode_bmaps_u8_plain(&bxs, xs_perm, prows, s.d / 16, box_max, &why) ||
        !encode_bmaps_u8(&bh, h4, prows, s.I / 2, box_max, &why) ||
        !encode_bmaps_u8_plain(&bhs, hs, prows, s.I / 16, box_max, &why))
        return cudaErrorInvalidValue;
    MlpArgs a = mlp_args(s, rows, tiles, tile_done, max_tiles, nullptr, y, status, kQStage);
    a.gs = q.gts;
    a.us = q.uts;
    a.ds = q.dts;
    const int grid = mlp_grid(a, max_tiles, num_sms);
    if (bn_max <= 16) return launch_q4<16>(w, bx, bxs, bh, bhs, a, h4, hs, grid, st);
    return launch_q4<32>(w, bx, bxs, bh, bhs, a, h4, hs, grid, st);
}

}  // namespace beam
