// Weighted combine (Glonce "Reflection releases Beam ...", Architecture paragraph: expert
// outputs are combined with normalized router weights, scaled by 2.5 - the scale is
// already inside the weights): out[t] = sum_k w[t,k] * y[inv_slot[t,k]], FP32 fused
// multiply-adds in slot order k = 0..top_k-1 (a gather, so the order is fixed and the
// result deterministic), rounded once to BF16. y (the experts' BF16 outputs) is read in
// 8-byte loads of four values, out stored in 8-byte stores.
// Shard mode (expert parallelism): slots routed to another shard (inv_slot = -1) are left
// out and the FP32 partial sum is stored unrounded, for the sum over shards.
#include "internal.cuh"

namespace beam {
namespace {

template <bool kPartial>
__global__ void __launch_bounds__(256) combine_kernel(const uint2* __restrict__ y, const int* __restrict__ inv_slot,
                                                      const float* __restrict__ topk_w, int K, int d4, int n_rows,
                                                      void* __restrict__ out, int* status) {
    pdl_wait();
    pdl_trigger();
    const int t = blockIdx.x;
    __shared__ int rows[32];
    __shared__ float ws[32];
    if (threadIdx.x < K) {
        int r = inv_slot[static_cast<size_t>(t) * K + threadIdx.x];
        float w = topk_w[static_cast<size_t>(t) * K + threadIdx.x];
        if (kPartial && r < 0) {  // another shard's expert
            r = 0;
            w = 0.f;
        } else if (static_cast<unsigned>(r) >= static_cast<unsigned>(n_rows)) {
            atomicCAS(status, 0, kStatusBadIndex);
            r = 0;
            w = 0.f;
        }
        rows[threadIdx.x] = r;
        ws[threadIdx.x] = w;
    }
    __syncthreads();
    for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < d4; c += gridDim.y * blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int k = 0; k < K; ++k) {
            const float w = ws[k];
            if (kPartial && w == 0.f) continue;
            const uint2 raw = y[static_cast<size_t>(rows[k]) * d4 + c];
            const float2 v01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
            const float2 v23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
            const float4 v = make_float4(v01.x, v01.y, v23.x, v23.y);
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        if constexpr (kPartial) {
            static_cast<float4*>(out)[static_cast<size_t>(t) * d4 + c] = acc;
        } else {
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t*>(&lo);
            o.y = *reinterpret_cast<uint32_t*>(&hi);
            static_cast<uint2*>(out)[static_cast<size_t>(t) * d4 + c] = o;
        }
    }
}

}  // namespace

cudaError_t launch_combine(const Shape& s, const bf16* y, const int* inv_slot, const float* topk_w, int T, bf16* out,
                           int* status, cudaStream_t st) {
    const int d4 = s.d / 4;
    // Split the row across a few blocks when there are few tokens.
    int ysplit = 1;
    while (T * ysplit < 296 && ysplit * 256 * 2 <= d4) ysplit *= 2;
    const dim3 grid(T, ysplit);
    const cudaError_t le_ = launch_pdl(combine_kernel<false>, dim3(grid), dim3(256), 0, st, reinterpret_cast<const uint2*>(y), inv_slot, topk_w, s.top_k, d4,
                                                T * s.top_k, out, status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_combine_partial(const Shape& s, const bf16* y, const int* inv_slot, const float* topk_w, int T,
                                   float* out, int* status, cudaStream_t st) {
    const int d4 = s.d / 4;
    int ysplit = 1;
    while (T * ysplit < 296 && ysplit * 256 * 2 <= d4) ysplit *= 2;
    const dim3 grid(T, ysplit);
    const cudaError_t le_ = launch_pdl(combine_kernel<true>, dim3(grid), dim3(256), 0, st, reinterpret_cast<const uint2*>(y), inv_slot, topk_w, s.top_k, d4,
                                               T * s.top_k, out, status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

}  // namespace beam
