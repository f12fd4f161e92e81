// Sandwich norm and depth-scaled residual of the MoE sublayer (transformers "Beam" doc,
// Overview, "Sandwich norms with depth-scaled residuals" bullet: each block is wrapped in
// an RMSNorm before and after; residual additions are rescaled so that after k
// contributions, counting the embeddings as the first, the stream is their sum divided by
// sqrt(k); the paragraph after the bullets: RMSNorm scaling is computed in FP32. Glonce
// "Reflection releases Beam ...", paragraph on the residual connections: at step k the
// sublayer output is added with weight 1/sqrt(k) and the stream kept with weight
// sqrt((k-1)/k)).
//
// rmsnorm_kernel:           out[t] = gamma * v[t] / sqrt(mean(v[t]^2) + eps)     (pre-norm)
// combine_residual_kernel:  m = sum_k w[t,k] y[slot(t,k)]  (FP32, slot order, as combine.cu)
//                           out[t] = sqrt((k-1)/k) stream[t] + gamma * m / sqrt(mean(m^2) + eps) / sqrt(k)
// One block of 256 threads per token row; each thread keeps its share of the row in
// registers (d <= 8192); the sum of squares is reduced in a fixed order (per-thread
// components in order, warp butterfly, warps in order), so results are deterministic.
#include "internal.cuh"

namespace beam {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormMaxVec = kNormMaxD / (4 * kNormThreads);  // 4-wide vectors per thread

__device__ __forceinline__ float4 bf16x4_to_float4(uint2 v) {
    const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    const float2 a = __bfloat1622float2(lo), b = __bfloat1622float2(hi);
    return make_float4(a.x, a.y, b.x, b.y);
}

__device__ __forceinline__ uint2 float4_to_bf16x4(float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    return o;
}

// Sum of `v` over the block, the same order on every run; every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) total += red[w];
    return total;
}

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const uint2* __restrict__ v,
                                                               const uint2* __restrict__ gamma, float eps, int d4,
                                                               uint2* __restrict__ out) {
    pdl_wait();
    pdl_trigger();
    __shared__ float red[kNormThreads / 32];
    const size_t row = static_cast<size_t>(blockIdx.x) * d4;
    float4 x[kNormMaxVec];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNormMaxVec; ++i) {
        const int c = threadIdx.x + i * kNormThreads;
        x[i] = c < d4 ? bf16x4_to_float4(v[row + c]) : make_float4(0.f, 0.f, 0.f, 0.f);
        ss = fmaf(x[i].x, x[i].x, ss);
        ss = fmaf(x[i].y, x[i].y, ss);
        ss = fmaf(x[i].z, x[i].z, ss);
        ss = fmaf(x[i].w, x[i].w, ss);
    }
    const float r = 1.0f / sqrtf(block_sum(ss, red) / static_cast<float>(4 * d4) + eps);
#pragma unroll
    for (int i = 0; i < kNormMaxVec; ++i) {
        const int c = threadIdx.x + i * kNormThreads;
        if (c < d4) {
            const float4 g = bf16x4_to_float4(gamma[c]);
            out[row + c] = float4_to_bf16x4(make_float4(g.x * (x[i].x * r), g.y * (x[i].y * r), g.z * (x[i].z * r),
                                                        g.w * (x[i].w * r)));
        }
    }
}

__global__ void __launch_bounds__(kNormThreads) combine_residual_kernel(
    const uint2* __restrict__ y, const int* __restrict__ inv_slot, const float* __restrict__ topk_w, int K, int d4,
    int n_rows, const uint2* stream_in, const uint2* __restrict__ gamma, float eps, float a, float b,
    uint2* stream_out, int* status) {
    pdl_wait();
    pdl_trigger();
    __shared__ int rows[32];
    __shared__ float ws[32];
    __shared__ float red[kNormThreads / 32];
    const int t = blockIdx.x;
    if (threadIdx.x < K) {
        int r = inv_slot[static_cast<size_t>(t) * K + threadIdx.x];
        float w = topk_w[static_cast<size_t>(t) * K + threadIdx.x];
        if (static_cast<unsigned>(r) >= static_cast<unsigned>(n_rows)) {
            atomicCAS(status, 0, kStatusBadIndex);
            r = 0;
            w = 0.f;
        }
        rows[threadIdx.x] = r;
        ws[threadIdx.x] = w;
    }
    __syncthreads();
    float4 m[kNormMaxVec];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < kNormMaxVec; ++i) {
        const int c = threadIdx.x + i * kNormThreads;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < d4) {
            for (int k = 0; k < K; ++k) {
                const float4 v = bf16x4_to_float4(y[static_cast<size_t>(rows[k]) * d4 + c]);
                const float w = ws[k];
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        m[i] = acc;
        ss = fmaf(acc.x, acc.x, ss);
        ss = fmaf(acc.y, acc.y, ss);
        ss = fmaf(acc.z, acc.z, ss);
        ss = fmaf(acc.w, acc.w, ss);
    }
    const float r = 1.0f / sqrtf(block_sum(ss, red) / static_cast<float>(4 * d4) + eps);
    const size_t row = static_cast<size_t>(t) * d4;
#pragma unroll
    for (int i = 0; i < kNormMaxVec; ++i) {
        const int c = threadIdx.x + i * kNormThreads;
        if (c < d4) {
            const float4 s = bf16x4_to_float4(stream_in[row + c]);
            const float4 g = bf16x4_to_float4(gamma[c]);
            float4 o;
            o.x = fmaf(a, s.x, b * (g.x * (m[i].x * r)));
            o.y = fmaf(a, s.y, b * (g.y * (m[i].y * r)));
            o.z = fmaf(a, s.z, b * (g.z * (m[i].z * r)));
            o.w = fmaf(a, s.w, b * (g.w * (m[i].w * r)));
            stream_out[row + c] = float4_to_bf16x4(o);
        }
    }
}

}  // namespace

cudaError_t launch_rmsnorm(int d, const bf16* v, const bf16* gamma, float eps, int T, bf16* out, cudaStream_t st) {
    if (d % 4 || d > kNormMaxD) return cudaErrorInvalidValue;
    const cudaError_t le_ = launch_pdl(rmsnorm_kernel, dim3(T), dim3(kNormThreads), 0, st, reinterpret_cast<const uint2*>(v), reinterpret_cast<const uint2*>(gamma),
                                               eps, d / 4, reinterpret_cast<uint2*>(out));
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_combine_residual(const Shape& s, const bf16* y, const int* inv_slot, const float* topk_w, int T,
                                    const bf16* stream_in, const bf16* gamma, float eps, int k_contrib,
                                    bf16* stream_out, int* status, cudaStream_t st) {
    if (s.d % 4 || s.d > kNormMaxD || k_contrib < 2) return cudaErrorInvalidValue;
    const float a = static_cast<float>(sqrt(static_cast<double>(k_contrib - 1) / k_contrib));
    const float b = static_cast<float>(1.0 / sqrt(static_cast<double>(k_contrib)));
    const cudaError_t le_ = launch_pdl(combine_residual_kernel, dim3(T), dim3(kNormThreads), 0, st, 
        reinterpret_cast<const uint2*>(y), inv_slot, topk_w, s.top_k, s.d / 4, T * s.top_k,
        reinterpret_cast<const uint2*>(stream_in), reinterpret_cast<const uint2*>(gamma), eps, a, b,
        reinterpret_cast<uint2*>(stream_out), status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

}  // namespace beam
