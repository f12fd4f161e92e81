// Router of the Beam MoE block (release pages: Glonce "Reflection releases Beam ...",
// Architecture paragraph; transformers "Beam" doc, Overview, "Sparse MoE" bullet and the
// FP32-numerics paragraph after the bullets).
//
// Stage 1 (router_logits_kernel): FP32 logits l = x . Wr^T on CUDA cores, x widened
// exactly from BF16, FP32 fused multiply-adds in ascending K order. Split-K partial sums
// (for small T) are written per split and added in split order by stage 2, so the result
// is deterministic.
// Stage 2 (router_select_kernel): one warp per token. Lane j holds expert 32g + j of every
// group g in registers: sigmoid, bias add, group top-2 sums by butterfly shuffles, group
// top-k and expert top-k by warp argmax rounds, weights normalised to `scale`.
#include <cfloat>
#include <climits>

#include "internal.cuh"

namespace beam {
namespace {

constexpr int RT = 64;    // tokens per CTA
constexpr int RE = 64;    // experts per CTA
constexpr int RK = 32;    // K per shared-memory stage
constexpr int RTHREADS = 256;

__global__ void __launch_bounds__(RTHREADS) router_logits_kernel(const bf16* __restrict__ x,
                                                                 const float* __restrict__ wr, int T, int d, int E,
                                                                 int k_per_split, float* __restrict__ partial) {
    __shared__ __align__(16) float xs[2][RK][RT + 4];
    __shared__ __align__(16) float ws[2][RK][RE + 4];
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * RT, e0 = blockIdx.y * RE, split = blockIdx.z;
    const int kbeg = split * k_per_split, kend = kbeg + k_per_split;

    // Global->shared mapping: x row xt, 8 bf16 at xk; W rows we and we+32, 4 floats at wk.
    const int xt = tid >> 2, xk = (tid & 3) * 8;
    const int we = tid >> 3, wk = (tid & 7) * 4;
    const bool x_ok = (t0 + xt) < T;
    const bool w0_ok = (e0 + we) < E, w1_ok = (e0 + we + 32) < E;
    const bf16* xp = x + static_cast<size_t>(x_ok ? t0 + xt : 0) * d + xk;
    const float* wp0 = wr + static_cast<size_t>(w0_ok ? e0 + we : 0) * d + wk;
    const float* wp1 = wr + static_cast<size_t>(w1_ok ? e0 + we + 32 : 0) * d + wk;

    // Compute mapping: tokens ty*4..ty*4+3, experts tx*4..tx*4+3.
    const int tx = tid & 15, ty = tid >> 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    uint4 xr;
    float4 w0r, w1r;
    auto gload = [&](int k) {
        xr = x_ok ? *reinterpret_cast<const uint4*>(xp + k) : make_uint4(0, 0, 0, 0);
        w0r = w0_ok ? *reinterpret_cast<const float4*>(wp0 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        w1r = w1_ok ? *reinterpret_cast<const float4*>(wp1 + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    auto sstore = [&](int b) {
        const bf16* xv = reinterpret_cast<const bf16*>(&xr);
#pragma unroll
        for (int i = 0; i < 8; ++i) xs[b][xk + i][xt] = __bfloat162float(xv[i]);
        ws[b][wk + 0][we] = w0r.x;
        ws[b][wk + 1][we] = w0r.y;
        ws[b][wk + 2][we] = w0r.z;
        ws[b][wk + 3][we] = w0r.w;
        ws[b][wk + 0][we + 32] = w1r.x;
        ws[b][wk + 1][we + 32] = w1r.y;
        ws[b][wk + 2][we + 32] = w1r.z;
        ws[b][wk + 3][we + 32] = w1r.w;
    };

    gload(kbeg);
    sstore(0);
    __syncthreads();
    int b = 0;
    for (int k = kbeg; k < kend; k += RK) {
        const bool more = k + RK < kend;
        if (more) gload(k + RK);
#pragma unroll
        for (int kk = 0; kk < RK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&xs[b][kk][ty * 4]);
            const float4 w = *reinterpret_cast<const float4*>(&ws[b][kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
        }
        if (more) sstore(b ^ 1);
        __syncthreads();
        b ^= 1;
    }
    const int e = e0 + tx * 4;
    if (e < E) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + ty * 4 + i;
            if (t < T)
                *reinterpret_cast<float4*>(partial + (static_cast<size_t>(split) * T + t) * E + e) =
                    make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        }
    }
}

constexpr unsigned kFull = 0xffffffffu;

// One warp per token. Experts per group are 32 (one per lane); up to 8 groups. `bias` may
// be null (logits-only calls), in which case the biased score is the sigmoid score.
__global__ void __launch_bounds__(256) router_select_kernel(const float* __restrict__ partial, int splits,
                                                            const float* __restrict__ bias, int T, int E, int G,
                                                            int TG, int K, float scale,
                                                            int32_t* __restrict__ topk_idx,
                                                            float* __restrict__ topk_w,
                                                            float* __restrict__ logits_out) {
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

}  // namespace

int router_splits(const Shape& s, int T, int num_sms) {
    const int nk = s.d / RK;
    const int base = ((T + RT - 1) / RT) * ((s.E + RE - 1) / RE);
    int best = 1;
    for (int sp = 1; sp <= 32 && sp <= nk; ++sp) {
        if (nk % sp) continue;
        best = sp;
        if (base * sp >= 2 * num_sms) break;
    }
    return best;
}

cudaError_t launch_router_logits(const Shape& s, const bf16* x, const float* wr, int T, int splits, float* partial,
                                 cudaStream_t st) {
    const dim3 grid((T + RT - 1) / RT, (s.E + RE - 1) / RE, splits);
    router_logits_kernel<<<grid, RTHREADS, 0, st>>>(x, wr, T, s.d, s.E, s.d / splits, partial);
    return cudaGetLastError();
}

cudaError_t launch_router_select(const Shape& s, const float* partial, int splits, const float* bias, int T,
                                 int32_t* topk_idx, float* topk_w, float* logits_out, cudaStream_t st) {
    const int warps_per_block = 8;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
    router_select_kernel<<<blocks, warps_per_block * 32, 0, st>>>(partial, splits, bias, T, s.E, s.n_group,
                                                                  s.topk_group, s.top_k, s.scale, topk_idx, topk_w,
                                                                  logits_out);
    return cudaGetLastError();
}

}  // namespace beam
