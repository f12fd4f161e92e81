// Router of the Beam MoE block (release pages: Glonce "Reflection releases Beam ...",
// Architecture paragraph; transformers "Beam" doc, Overview, "Sparse MoE" bullet and the
// FP32-numerics paragraph after the bullets).
//
// Stage 1: FP32 logits l = x . Wr^T (x is exactly BF16).
//   T <= 32 (decode): router_logits_small_kernel on CUDA cores, FP32 fused multiply-adds,
//   one CTA per expert over the whole K, reduced in a fixed order.
//   T > 32: the tensor-core product of router_gemm.cu, after
//   router_split_weights_kernel has written Wr as three BF16 pieces hi + mid + lo == Wr
//   (exactly); the products x.piece are exact and accumulate in FP32. Split-K partial
//   planes are added in split order by stage 2, so the result is deterministic.
// Stage 2 (router_select_kernel): one warp per token. Lane j holds expert 32g + j of every
// group g in registers: sigmoid, bias add, group top-2 sums by butterfly shuffles, group
// top-k and expert top-k by warp argmax rounds, weights normalised to `scale`.
#include <cfloat>
#include <climits>

#include "internal.cuh"

namespace beam {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Small batches (T <= kSmallT, decode): one CTA per kSmallEPB experts computes their logits
// for every token over the whole K, so no split-K partials are written. Warp w sums the
// K range [w*d/8, (w+1)*d/8): each lane first loads its 4-wide slices of the experts'
// weights for the whole range (all loads in flight at once), then streams the tokens,
// FMA-ing in ascending K. The 32 lanes are combined by a fixed butterfly and the 8 warps
// in warp order, so the result is deterministic.
constexpr int kSmallT = 32;
constexpr int kSmallEPB = 1;  // one CTA per expert: 256 CTAs, shorter per-lane token chains
constexpr int kSmallWarps = 8;
constexpr int kSmallMaxIt = 8;  // 128-wide K steps per warp: d <= 8 * 128 * 8

__global__ void __launch_bounds__(kSmallWarps * 32) router_logits_small_kernel(const bf16* __restrict__ x,
                                                                              const float* __restrict__ wr, int T,
                                                                              int d, int E,
                                                                              float* __restrict__ logits) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kSmallWarps][kSmallT * kSmallEPB];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e0 = blockIdx.x * kSmallEPB;
    const int kw = d / kSmallWarps;
    const int kbeg = warp * kw + 4 * lane, kend = (warp + 1) * kw;
    float4 w[kSmallMaxIt][kSmallEPB];
#pragma unroll
    for (int it = 0; it < kSmallMaxIt; ++it) {
        const int k = kbeg + 128 * it;
#pragma unroll
        for (int j = 0; j < kSmallEPB; ++j)
            w[it][j] = (k < kend && e0 + j < E) ? *reinterpret_cast<const float4*>(wr + static_cast<size_t>(e0 + j) * d + k)
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float acc[kSmallT][kSmallEPB];
#pragma unroll
    for (int t = 0; t < kSmallT; ++t) {
#pragma unroll
        for (int j = 0; j < kSmallEPB; ++j) acc[t][j] = 0.f;
        if (t < T) {
#pragma unroll
            for (int it = 0; it < kSmallMaxIt; ++it) {
                const int k = kbeg + 128 * it;
                if (k < kend) {
                    const uint2 raw = *reinterpret_cast<const uint2*>(x + static_cast<size_t>(t) * d + k);
                    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
                    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
                    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
#pragma unroll
                    for (int j = 0; j < kSmallEPB; ++j) {
                        float v = acc[t][j];
                        v = fmaf(a.x, w[it][j].x, v);
                        v = fmaf(a.y, w[it][j].y, v);
                        v = fmaf(b.x, w[it][j].z, v);
                        v = fmaf(b.y, w[it][j].w, v);
                        acc[t][j] = v;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kSmallT; ++t) {
#pragma unroll
        for (int j = 0; j < kSmallEPB; ++j) {
            float v = acc[t][j];
#pragma unroll
            for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
            if (lane == 0) red[warp][t * kSmallEPB + j] = v;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < T * kSmallEPB; i += blockDim.x) {
        const int t = i / kSmallEPB, j = i % kSmallEPB;
        if (e0 + j >= E) continue;
        float v = red[0][i];
#pragma unroll
        for (int w8 = 1; w8 < kSmallWarps; ++w8) v += red[w8][i];
        logits[static_cast<size_t>(t) * E + e0 + j] = v;
    }
}

// One warp per token. Experts per group are 32 (one per lane); up to 8 groups. `bias` may
// be null (logits-only calls), in which case the biased score is the sigmoid score.
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ partial, int splits,
                                                            const float* __restrict__ bias, int T, int E, int G,
                                                            int TG, int K, float scale,
                                                            int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ topk_w,
                                                            float* __restrict__ logits_out) {
    pdl_wait();
    pdl_trigger();
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;

    float s[8], c[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        s[g] = 0.f;
        c[g] = -FLT_MAX;
        if (g < G) {
            const int e = g * 32 + lane;
            float l = partial[static_cast<size_t>(t) * E + e];
            for (int sp = 1; sp < splits; ++sp) l += partial[(static_cast<size_t>(sp) * T + t) * E + e];
            if (logits_out) logits_out[static_cast<size_t>(t) * E + e] = l;
            s[g] = 1.0f / (1.0f + expf(-l));
            c[g] = bias ? s[g] + bias[e] : s[g];
        }
    }

    // Group score: sum of the two largest biased scores of the group (butterfly merge of
    // sorted pairs: the top two of {a1>=a2} U {b1>=b2} are max(a1,b1) and
    // max(min(a1,b1), max(a2,b2))).
    float gs[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        float a1 = c[g], a2 = -FLT_MAX;
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float b1 = __shfl_xor_sync(kFull, a1, off);
            const float b2 = __shfl_xor_sync(kFull, a2, off);
            a2 = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
            a1 = fmaxf(a1, b1);
        }
        gs[g] = a1 + a2;
    }

    // Keep the TG best groups; strict '>' while scanning g upwards sends ties to the lower g.
    unsigned kept = 0;
    for (int r = 0; r < TG; ++r) {
        int best = -1;
        float bv = 0.f;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const bool avail = g < G && !((kept >> g) & 1u);
            if (avail && (best < 0 || gs[g] > bv)) {
                best = g;
                bv = gs[g];
            }
        }
        kept |= 1u << best;
    }

    // Top-K experts of the kept groups: K rounds of a warp argmax over (c desc, e asc).
    unsigned taken = 0;  // this lane's picked groups
    int my_e = 0;
    float my_s = 0.f;
    for (int k = 0; k < K; ++k) {
        float bv = 0.f, bs = 0.f;
        int be = INT_MAX;
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const bool avail = g < G && ((kept >> g) & 1u) && !((taken >> g) & 1u);
            if (avail && (be == INT_MAX || c[g] > bv)) {
                bv = c[g];
                be = g * 32 + lane;
                bs = s[g];
            }
        }
#pragma unroll
        for (int off = 16; off; off >>= 1) {
            const float ov = __shfl_xor_sync(kFull, bv, off);
            const int oe = __shfl_xor_sync(kFull, be, off);
            const float os = __shfl_xor_sync(kFull, bs, off);
            const bool take = oe != INT_MAX && (be == INT_MAX || ov > bv || (ov == bv && oe < be));
            if (take) {
                bv = ov;
                be = oe;
                bs = os;
            }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        if (lane == k) {
            my_e = be;
            my_s = bs;
        }
    }
    float sum = 0.f;
    for (int k = 0; k < K; ++k) sum += __shfl_sync(kFull, my_s, k);
    if (lane < K) {
        topk_idx[static_cast<size_t>(t) * K + lane] = my_e;
        topk_w[static_cast<size_t>(t) * K + lane] = scale * my_s / sum;
    }
}

// FP32 router weights as three BF16 pieces with hi + mid + lo == w exactly: hi is w
// rounded to BF16, mid the rounded remainder, lo the rest. Each remainder is exact in FP32
// (the difference of two numbers within a factor of two), and the last one has at most 8
// significant bits, so it is a BF16 value (for |w| above the BF16 normal range's bottom
// plus 16 binades, far below any router weight).
__global__ void __launch_bounds__(256) router_split_weights_kernel(const float4* __restrict__ w, size_t n4,
                                                                  size_t n, bf16* __restrict__ w3) {
    pdl_wait();
    pdl_trigger();
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const float4 v = w[i];
        const float vs[4] = {v.x, v.y, v.z, v.w};
        bf16 hi[4], mid[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            hi[j] = __float2bfloat16_rn(vs[j]);
            const float r1 = vs[j] - __bfloat162float(hi[j]);
            mid[j] = __float2bfloat16_rn(r1);
            const float r2 = r1 - __bfloat162float(mid[j]);
            lo[j] = __float2bfloat16_rn(r2);
        }
        *reinterpret_cast<uint2*>(w3 + 4 * i) = *reinterpret_cast<const uint2*>(hi);
        *reinterpret_cast<uint2*>(w3 + n + 4 * i) = *reinterpret_cast<const uint2*>(mid);
        *reinterpret_cast<uint2*>(w3 + 2 * n + 4 * i) = *reinterpret_cast<const uint2*>(lo);
    }
}

}  // namespace

RouterPlan router_plan(const Shape& s, int T, int num_sms) {
    RouterPlan p;
    if (T <= kSmallT && s.d <= kSmallWarps * 128 * kSmallMaxIt) {
        p.tensor = false;
        p.splits = 1;
        p.w3_elems = 0;
    } else {
        p.tensor = true;
        p.splits = router_tc_splits(s, T, num_sms);
        p.w3_elems = 3ull * s.E * s.d;
    }
    return p;
}

cudaError_t launch_router_split_weights(const Shape& s, const float* wr, bf16* w3, int num_sms, cudaStream_t st) {
    const size_t n = static_cast<size_t>(s.E) * s.d;
    const size_t n4 = n / 4;
    long long blocks = static_cast<long long>((n4 + 255) / 256);
    const long long cap = static_cast<long long>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    const cudaError_t le_ = launch_pdl(router_split_weights_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, reinterpret_cast<const float4*>(wr),
                                                                               n4, n, w3);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_router_logits(const Shape& s, const RouterPlan& p, const bf16* x, const float* wr, int T,
                                 const bf16* w3, float* partial, int* status, int num_sms, cudaStream_t st) {
    if (!p.tensor) {
        if (p.splits != 1 || T > kSmallT) return cudaErrorInvalidValue;
        const cudaError_t le_ = launch_pdl(router_logits_small_kernel, dim3((s.E + kSmallEPB - 1) / kSmallEPB), dim3(kSmallWarps * 32), 0, st, x, wr, T, s.d, s.E,
                                                                                                partial);
    if (le_ != cudaSuccess) return le_;
        return cudaGetLastError();
    }
    return launch_router_tc(s, w3, x, T, p.splits, partial, status, num_sms, st);
}

cudaError_t launch_router_select(const Shape& s, const float* partial, int splits, const float* bias, int T,
                                 int32_t* topk_idx, float* topk_w, float* logits_out, cudaStream_t st) {
    const int warps_per_block = 8;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
    const cudaError_t le_ = launch_pdl(router_select_kernel, dim3(blocks), dim3(warps_per_block * 32), 0, st, partial, splits, bias, T, s.E, s.n_group,
                                                                  s.topk_group, s.top_k, s.scale, topk_idx, topk_w,
                                                                  logits_out);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

}  // namespace beam
