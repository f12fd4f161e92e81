// Dispatch: group the T*top_k (token, slot) pairs by expert, in token order within each
// expert, without order-dependent atomics, so the permutation is the same on every run.
//
// Tokens are taken in chunks of 256. For each chunk, a shared-memory bitmap holds one bit
// per (expert, token of the chunk); it is built with atomicOr, whose result does not
// depend on the order of the ORs. The rank of token t among the chunk's tokens routed to
// expert e is the popcount of e's bits below t.
//   count:   per-chunk expert histogram from the bitmap;
//   scan:    per expert, exclusive scan over chunks; then an exclusive scan over experts
//            gives each expert's first permuted row; also emits the GEMM work list of
//            N-tiles (at most bn_max rows each, split evenly), with the header's item
//            counter and every tile's completion counter set to zero;
//   scatter: permuted row of (t, k) = chunk base of e + rank; writes perm_src[row] = t
//            and inv_slot[t, k] = row;
//   gather:  x_perm[row] = x[perm_src[row]] with 16-byte loads and stores.
// Small batches (T <= kSmallDispatchT, decode) run all four steps in one launch: every
// block builds the same permutation in shared memory (per-expert token bitmaps of at most
// four words), block 0 writes the work list, offsets, perm_src and inv_slot, and all
// blocks copy their share of the rows. The result is the one the four kernels give.
#include "internal.cuh"

namespace beam {
namespace {

constexpr int kChunk = kDispatchChunk;
constexpr int kWords = kChunk / 32;

// Experts [e_lo, e_lo + E) are this call's (all of them, or one expert-parallel shard);
// pairs routed elsewhere are left out. Bitmap rows are local expert ids.
__device__ __forceinline__ void build_bitmap(uint32_t* bm, const int32_t* __restrict__ idx, int T, int E_all,
                                             int e_lo, int E, int K, int t0, int* status) {
    for (int i = threadIdx.x; i < E * kWords; i += blockDim.x) bm[i] = 0u;
    __syncthreads();
    const int tl = threadIdx.x;
    const int t = t0 + tl;
    if (t < T) {
        for (int k = 0; k < K; ++k) {
            const int e = idx[static_cast<size_t>(t) * K + k];
            if (e < 0 || e >= E_all) {
                atomicCAS(status, 0, kStatusBadExpert);
                continue;
            }
            const int el = e - e_lo;
            if (el < 0 || el >= E) continue;
            atomicOr(&bm[el * kWords + (tl >> 5)], 1u << (tl & 31));
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kChunk) dispatch_count_kernel(const int32_t* __restrict__ idx, int T, int E_all,
                                                                int e_lo, int E, int K,
                                                                int* __restrict__ chunk_count, int* status) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint32_t bm[];
    build_bitmap(bm, idx, T, E_all, e_lo, E, K, blockIdx.x * kChunk, status);
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int n = 0;
#pragma unroll
        for (int w = 0; w < kWords; ++w) n += __popc(bm[e * kWords + w]);
        chunk_count[static_cast<size_t>(blockIdx.x) * E + e] = n;
    }
}

// One block of 1024 threads; thread e < E owns expert e.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int nchunks, int E, int bn_max,
                                                             int* __restrict__ chunk_count,
                                                             int* __restrict__ expert_offset,
                                                             int4* __restrict__ tiles,
                                                             int* __restrict__ tile_done) {
    pdl_wait();
    pdl_trigger();
    __shared__ int tot[1024];
    __shared__ int ntl[1024];
    const int e = threadIdx.x;
    int n = 0;
    if (e < E) {
        for (int c = 0; c < nchunks; ++c) {
            const int v = chunk_count[static_cast<size_t>(c) * E + e];
            chunk_count[static_cast<size_t>(c) * E + e] = n;
            n += v;
        }
    }
    // N-tiles of expert e: an even split into pieces of `per` rows (a multiple of 16,
    // at most bn_max); the last piece takes the remainder.
    int per = 0, nt = 0;
    if (n > 0) {
        const int q = (n + bn_max - 1) / bn_max;
        per = min(bn_max, (((n + q - 1) / q + 15) / 16) * 16);
        nt = (n + per - 1) / per;
    }
    tot[e] = n;
    ntl[e] = nt;
    __syncthreads();
    // Inclusive Hillis-Steele scans of expert totals and tile counts.
    for (int off = 1; off < 1024; off <<= 1) {
        const int a = e >= off ? tot[e - off] : 0;
        const int b = e >= off ? ntl[e - off] : 0;
        __syncthreads();
        tot[e] += a;
        ntl[e] += b;
        __syncthreads();
    }
    if (e < E) {
        const int base = tot[e] - n;   // first permuted row of expert e
        expert_offset[e] = base;
        if (e == E - 1) {
            expert_offset[E] = tot[e];
            tiles[0] = make_int4(ntl[e], 0, 0, 0);
        }
        for (int c = 0; c < nchunks; ++c) chunk_count[static_cast<size_t>(c) * E + e] += base;
        if (nt > 0) {
            const int first = ntl[e] - nt;
            for (int r = 0, tile = first; r < n; r += per, ++tile) {
                const int rows = min(per, n - r);
                if (tile_done) tile_done[tile] = 0;
                // .w: the tile's index among its expert's tiles and their count (the
                // expert kernel orders its items m-major within an expert)
                tiles[1 + tile] = make_int4(e, base + r, rows, (tile - first) | (nt << 16));
            }
        }
    }
}

__global__ void __launch_bounds__(kChunk) dispatch_scatter_kernel(const int32_t* __restrict__ idx, int T, int E_all,
                                                                  int e_lo, int E, int K,
                                                                  const int* __restrict__ chunk_base,
                                                                  int* __restrict__ perm_src,
                                                                  int* __restrict__ inv_slot, int* status) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint32_t bm[];
    const int t0 = blockIdx.x * kChunk;
    build_bitmap(bm, idx, T, E_all, e_lo, E, K, t0, status);
    const int tl = threadIdx.x;
    const int t = t0 + tl;
    if (t >= T) return;
    const int w = tl >> 5;
    const uint32_t below = (1u << (tl & 31)) - 1u;
    for (int k = 0; k < K; ++k) {
        const int el = idx[static_cast<size_t>(t) * K + k] - e_lo;
        if (el < 0 || el >= E) {  // routed to another shard (or invalid, already flagged)
            inv_slot[static_cast<size_t>(t) * K + k] = -1;
            continue;
        }
        int rank = __popc(bm[el * kWords + w] & below);
        for (int j = 0; j < w; ++j) rank += __popc(bm[el * kWords + j]);
        const int row = chunk_base[static_cast<size_t>(blockIdx.x) * E + el] + rank;
        if (row < 0 || row >= T * K) {
            atomicCAS(status, 0, kStatusBadIndex);
            continue;
        }
        inv_slot[static_cast<size_t>(t) * K + k] = row;
        perm_src[row] = t;
    }
}

// x_perm[row] = x[perm_src[row]] for the dispatched rows, 16 bytes at a time; with a side
// array (side_vecs > 0) also side_dst[row] = side_src[perm_src[row]] (rows of side_vecs
// 16-byte pieces: the block scales of the NVFP4 activation pieces).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, int row_vecs, int T,
                                                          const int* __restrict__ perm_src,
                                                          const int* __restrict__ n_rows,
                                                          uint4* __restrict__ x_perm, const uint4* __restrict__ side_src,
                                                          int side_vecs, uint4* __restrict__ side_dst, int* status) {
    pdl_wait();
    pdl_trigger();
    const size_t n = static_cast<size_t>(*n_rows);  // rows this call dispatched
    const size_t main_total = n * row_vecs;
    const size_t total = main_total + n * side_vecs;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const bool side = i >= main_total;
        const size_t j = side ? i - main_total : i;
        const int w = side ? side_vecs : row_vecs;
        const size_t r = j / w;
        const size_t v = j - r * w;
        const int src = perm_src[r];
        if (static_cast<unsigned>(src) >= static_cast<unsigned>(T)) {
            atomicCAS(status, 0, kStatusBadIndex);
            continue;
        }
        if (side) side_dst[j] = side_src[static_cast<size_t>(src) * w + v];
        else x_perm[j] = x[static_cast<size_t>(src) * w + v];
    }
}

constexpr int kSmallWords = kSmallDispatchT / 32;
constexpr int kSmallThreads = 256;  // >= the largest expert count (256)

__global__ void __launch_bounds__(kSmallThreads) dispatch_small_kernel(
    const int32_t* __restrict__ idx, int T, int E_all, int e_lo, int E, int K, int bn_max, const uint4* __restrict__ x,
    int row_vecs, int* __restrict__ expert_offset, int4* __restrict__ tiles, int* __restrict__ tile_done,
    int* __restrict__ perm_src, int* __restrict__ inv_slot, uint4* __restrict__ x_perm,
    const uint4* __restrict__ side_src, int side_vecs, uint4* __restrict__ side_dst, int* status) {
    pdl_wait();
    pdl_trigger();
    __shared__ uint32_t bm[kSmallThreads * kSmallWords];
    __shared__ int base_s[kSmallThreads + 1];  // exclusive scan of rows per expert
    __shared__ int tile_s[kSmallThreads + 1];  // exclusive scan of N-tiles per expert
    __shared__ int src_s[kSmallDispatchT * 32];  // permuted row -> token
    const int tid = threadIdx.x;
    for (int i = tid; i < E * kSmallWords; i += blockDim.x) bm[i] = 0u;
    __syncthreads();
    const bool lead = blockIdx.x == 0;
    for (int p = tid; p < T * K; p += blockDim.x) {
        const int e = idx[p];
        const int t = p / K;
        if (e < 0 || e >= E_all) {
            if (lead) atomicCAS(status, 0, kStatusBadExpert);
            continue;
        }
        const int el = e - e_lo;
        if (el >= 0 && el < E) atomicOr(&bm[el * kSmallWords + (t >> 5)], 1u << (t & 31));
    }
    __syncthreads();
    // rows and N-tiles of expert tid (same split as dispatch_scan_kernel)
    int n = 0, per = 0, nt = 0;
    if (tid < E) {
#pragma unroll
        for (int w = 0; w < kSmallWords; ++w) n += __popc(bm[tid * kSmallWords + w]);
        if (n > 0) {
            const int q = (n + bn_max - 1) / bn_max;
            per = min(bn_max, (((n + q - 1) / q + 15) / 16) * 16);
            nt = (n + per - 1) / per;
        }
    }
    base_s[tid + 1] = n;
    tile_s[tid + 1] = nt;
    if (tid == 0) base_s[0] = tile_s[0] = 0;
    __syncthreads();
    for (int off = 1; off < kSmallThreads; off <<= 1) {  // inclusive scans of entries 1..256
        const int a = tid >= off ? base_s[tid + 1 - off] : 0;
        const int b = tid >= off ? tile_s[tid + 1 - off] : 0;
        __syncthreads();
        base_s[tid + 1] += a;
        tile_s[tid + 1] += b;
        __syncthreads();
    }
    const int total_rows = base_s[E], total_tiles = tile_s[E];
    if (lead && tid < E) {
        const int base = base_s[tid], first = tile_s[tid];
        expert_offset[tid] = base;
        for (int r = 0, tile = first; r < n; r += per, ++tile) {
            tile_done[tile] = 0;
            tiles[1 + tile] = make_int4(tid, base + r, min(per, n - r), (tile - first) | (nt << 16));
        }
        if (tid == E - 1) {
            expert_offset[E] = total_rows;
            tiles[0] = make_int4(total_tiles, 0, 0, 0);
        }
    }
    // row of every pair: expert base + the token's rank among the expert's tokens
    for (int p = tid; p < T * K; p += blockDim.x) {
        const int t = p / K;
        const int el = idx[p] - e_lo;
        if (el < 0 || el >= E || idx[p] < 0 || idx[p] >= E_all) {
            if (lead) inv_slot[p] = -1;
            continue;
        }
        int rank = __popc(bm[el * kSmallWords + (t >> 5)] & ((1u << (t & 31)) - 1u));
        for (int w = 0; w < (t >> 5); ++w) rank += __popc(bm[el * kSmallWords + w]);
        const int row = base_s[el] + rank;
        src_s[row] = t;
        if (lead) {
            inv_slot[p] = row;
            perm_src[row] = t;
        }
    }
    __syncthreads();
    // gather: this block's share of the 16-byte pieces of the dispatched rows (and of the
    // side rows, if any)
    const long long main_total = static_cast<long long>(total_rows) * row_vecs;
    const long long total = main_total + static_cast<long long>(total_rows) * side_vecs;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + tid; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const bool side = i >= main_total;
        const long long j = side ? i - main_total : i;
        const int w = side ? side_vecs : row_vecs;
        const int r = static_cast<int>(j / w);
        const int v = static_cast<int>(j - static_cast<long long>(r) * w);
        if (side) side_dst[j] = side_src[static_cast<size_t>(src_s[r]) * w + v];
        else x_perm[j] = x[static_cast<size_t>(src_s[r]) * w + v];
    }
}

}  // namespace

int dispatch_max_tiles(const Shape& s, int T, int bn_max) {
    const long long pairs = static_cast<long long>(T) * s.top_k;
    const long long used = pairs < s.E ? pairs : s.E;
    return static_cast<int>(pairs / bn_max + used + 1);
}

cudaError_t launch_dispatch_count(const Shape& s, int e_lo, int E_loc, const int32_t* topk_idx, int T, int* chunk_count,
                                  int* status, cudaStream_t st) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    const size_t smem = static_cast<size_t>(E_loc) * kWords * sizeof(uint32_t);
    const cudaError_t le_ = launch_pdl(dispatch_count_kernel, dim3(nchunks), dim3(kChunk), smem, st, topk_idx, T, s.E, e_lo, E_loc, s.top_k, chunk_count, status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_dispatch_scan(int E_loc, int T, int bn_max, int* chunk_count, int* expert_offset, int4* tiles,
                                 int* tile_done, cudaStream_t st) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    const cudaError_t le_ = launch_pdl(dispatch_scan_kernel, dim3(1), dim3(1024), 0, st, nchunks, E_loc, bn_max, chunk_count, expert_offset, tiles, tile_done);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_dispatch_scatter(const Shape& s, int e_lo, int E_loc, const int32_t* topk_idx, int T,
                                    const int* chunk_base, int* perm_src, int* inv_slot, int* status, cudaStream_t st) {
    const int nchunks = (T + kChunk - 1) / kChunk;
    const size_t smem = static_cast<size_t>(E_loc) * kWords * sizeof(uint32_t);
    const cudaError_t le_ = launch_pdl(dispatch_scatter_kernel, dim3(nchunks), dim3(kChunk), smem, st, topk_idx, T, s.E, e_lo, E_loc, s.top_k, chunk_base, perm_src,
                                                           inv_slot, status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_dispatch_small(const Shape& s, int e_lo, int E_loc, const int32_t* topk_idx, int T, int bn_max,
                                  const bf16* x, int* expert_offset, int4* tiles, int* tile_done, int* perm_src,
                                  int* inv_slot, bf16* x_perm, int* status, int num_sms, cudaStream_t st,
                                  const void* side_src, int side_bytes, void* side_dst) {
    if (T > kSmallDispatchT || E_loc > kSmallThreads || s.top_k > 32) return cudaErrorInvalidValue;
    const int row_vecs = s.d / 8;
    const int side_vecs = side_src ? side_bytes / 16 : 0;
    const long long total = static_cast<long long>(T) * s.top_k * (row_vecs + side_vecs);
    long long blocks = (total + 4 * kSmallThreads - 1) / (4 * kSmallThreads);
    if (blocks > num_sms) blocks = num_sms;
    if (blocks < 1) blocks = 1;
    const cudaError_t le_ = launch_pdl(dispatch_small_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kSmallThreads),
                                       0, st, topk_idx, T, s.E, e_lo, E_loc, s.top_k, bn_max,
                                       reinterpret_cast<const uint4*>(x), row_vecs, expert_offset, tiles, tile_done,
                                       perm_src, inv_slot, reinterpret_cast<uint4*>(x_perm),
                                       reinterpret_cast<const uint4*>(side_src), side_vecs,
                                       reinterpret_cast<uint4*>(side_dst), status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const bf16* x, int d, int T, const int* perm_src, const int* n_rows, int rows,
                               bf16* x_perm, int* status, int num_sms, cudaStream_t st, const void* side_src,
                               int side_bytes, void* side_dst) {
    const int row_vecs = d / 8;
    const int side_vecs = side_src ? side_bytes / 16 : 0;
    const long long total = static_cast<long long>(rows) * (row_vecs + side_vecs);
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const cudaError_t le_ = launch_pdl(gather_rows_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, st, reinterpret_cast<const uint4*>(x), row_vecs, T,
                                                                      perm_src, n_rows,
                                                                      reinterpret_cast<uint4*>(x_perm),
                                                                      reinterpret_cast<const uint4*>(side_src), side_vecs,
                                                                      reinterpret_cast<uint4*>(side_dst), status);
    if (le_ != cudaSuccess) return le_;
    return cudaGetLastError();
}

}  // namespace beam
