// Declarations shared by the kernels' host launchers and the C-ABI layer.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "beam_moe.h"

namespace beam {

using bf16 = __nv_bfloat16;

// Programmatic dependent launch. Every kernel of the library is launched with
// launch_pdl, so it may start while its predecessor in the stream finishes; each kernel
// calls pdl_wait() before its first global-memory access (read or write), which returns
// once every earlier kernel has completed and its memory is visible, so memory effects
// keep stream order (scratch reuse through the stream-ordered pool included).
// pdl_trigger() lets the next kernel start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
#ifdef BEAM_NO_PDL
    cfg.numAttrs = 0;
#else
    cfg.numAttrs = 1;
#endif
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Raises kernel Kern's dynamic shared-memory limit to `bytes` once per device (the setting
// lasts for the device's context), so steady-state launches make no attribute call. One
// instantiation per kernel: the flag word belongs to that kernel alone.
template <auto Kern>
cudaError_t set_smem_limit_once(int bytes) {
    static std::atomic<uint64_t> done{0};  // bit d: set on device d (devices 0..63)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

struct Shape {
    int d, I, E, n_group, topk_group, top_k;
    float scale;
};

// Device status codes written to the status word (first error wins).
enum : int {
    kStatusOk = 0,
    kStatusBadExpert = 1,
    kStatusWaitTimeout = 2,
    kStatusBadIndex = 3,
    kStatusRange = 4  // an NVFP4 activation block beyond its first piece's range (clamped)
};

// One N-tile of the grouped GEMMs: `rows` consecutive permuted rows starting at `row0`,
// all routed to expert `e`. The work list is int4 {e, row0, rows, 0} after an int4 header
// whose .x is the tile count.
constexpr int kDispatchChunk = 256;  // tokens per dispatch block

// ---------------------------------------------------------------- router (router.cu)
// How the router's logits stage runs for T tokens: the small-batch CUDA-core kernel
// (T <= 32, one partial plane) or the tensor-core product over BF16 pieces of the FP32
// router weights (split-K partial planes).
struct RouterPlan {
    bool tensor;      // tensor-core path (needs the weight pieces)
    int splits;       // partial planes of [T, E] the logits stage writes
    size_t w3_elems;  // BF16 elements of the three weight pieces (0 on the CUDA-core path)
};
RouterPlan router_plan(const Shape& s, int T, int num_sms);
// Writes the pieces hi, mid, lo of router_w ([3][E][d] BF16) for the tensor-core path.
cudaError_t launch_router_split_weights(const Shape& s, const float* wr, bf16* w3, int num_sms, cudaStream_t st);
cudaError_t launch_router_logits(const Shape& s, const RouterPlan& p, const bf16* x, const float* wr, int T,
                                 const bf16* w3, float* partial, int* status, int num_sms, cudaStream_t st);
cudaError_t launch_router_select(const Shape& s, const float* partial, int splits, const float* bias, int T,
                                 int32_t* topk_idx, float* topk_w, float* logits_out, cudaStream_t st);

// ---------------------------------------------------------------- dispatch (dispatch.cu)
int dispatch_max_tiles(const Shape& s, int T, int bn_max);
// Dispatch of the (token, slot) pairs routed to experts [e_lo, e_lo + E_loc) (all experts,
// or one expert-parallel shard; other pairs get inv_slot = -1). Work-list expert ids are
// local (e - e_lo).
cudaError_t launch_dispatch_count(const Shape& s, int e_lo, int E_loc, const int32_t* topk_idx, int T, int* chunk_count,
                                  int* status, cudaStream_t st);
cudaError_t launch_dispatch_scan(int E_loc, int T, int bn_max, int* chunk_count, int* expert_offset, int4* tiles,
                                 int* tile_done, cudaStream_t st);
cudaError_t launch_dispatch_scatter(const Shape& s, int e_lo, int E_loc, const int32_t* topk_idx, int T,
                                    const int* chunk_base, int* perm_src, int* inv_slot, int* status, cudaStream_t st);
// Count, scan, scatter and gather in one launch for small batches (T <= kSmallDispatchT,
// E_loc <= 256, top_k <= 32): the same outputs as the four launches.
constexpr int kSmallDispatchT = 128;
// A side array (side_src rows of side_bytes, a multiple of 16, per token) is gathered into
// side_dst beside the token rows when given.
cudaError_t launch_dispatch_small(const Shape& s, int e_lo, int E_loc, const int32_t* topk_idx, int T, int bn_max,
                                  const bf16* x, int* expert_offset, int4* tiles, int* tile_done, int* perm_src,
                                  int* inv_slot, bf16* x_perm, int* status, int num_sms, cudaStream_t st,
                                  const void* side_src = nullptr, int side_bytes = 0, void* side_dst = nullptr);
// x_perm[row] = x[perm_src[row]] for the *n_rows rows dispatched (rows: an upper bound), and
// likewise for the side array when given.
cudaError_t launch_gather_rows(const bf16* x, int d, int T, const int* perm_src, const int* n_rows, int rows,
                               bf16* x_perm, int* status, int num_sms, cudaStream_t st, const void* side_src = nullptr,
                               int side_bytes = 0, void* side_dst = nullptr);

// ---------------------------------------------------------------- expert MLP (expert_mlp.cu)
// Largest N-tile (token rows per tile) the expert kernel uses for a batch of T tokens.
int gemm_bn_max(const Shape& s, int T);
// Both expert products in one persistent kernel (expert_mlp.cu): h = SwiGLU(x_perm) and
// y = h . Wd^T (BF16) per N-tile of the work list, scheduled dynamically; tile_done[max_tiles]
// and the work list's item counter must be zero (dispatch_scan sets them).
cudaError_t launch_expert_mlp(const Shape& s, const bf16* w_gate, const bf16* w_up, const bf16* w_down,
                              const bf16* x_perm, int rows, const int4* tiles, int* tile_done, int max_tiles,
                              int bn_max, bf16* h, bf16* y, int* status, int num_sms,
                              cudaStream_t st);
// FP8 E4M3 expert weights, one FP32 scale per output row: W[r][c] = scale[r] * e4m3(q[r][c]).
// wg, wu [E, I, d] with gs, us [E, I]; wd [E, d, I] with ds [E, d].
struct Fp8Experts {
    const uint8_t* wg;
    const float* gs;
    const uint8_t* wu;
    const float* us;
    const uint8_t* wd;
    const float* ds;
};
// NVFP4 expert weights: E2M1 codes packed two per byte (element 2k in the low half of byte
// k), one E4M3 block scale per 16 elements of a row, one FP32 tensor scale per expert
// matrix: W[r][c] = ts * e4m3(bs[r][c / 16]) * e2m1(code c of row r).
// wg, wu [E, I, d/2] with gbs, ubs [E, I, d/16] and gts, uts [E]; wd [E, d, I/2] with dbs
// [E, d, I/16] and dts [E].
struct Nvfp4Experts {
    const uint8_t* wg;
    const uint8_t* gbs;
    const float* gts;
    const uint8_t* wu;
    const uint8_t* ubs;
    const float* uts;
    const uint8_t* wd;
    const uint8_t* dbs;
    const float* dts;
};
// NVFP4 expert weights on the block-scaled FP4 tensor cores (expert_mlp_nvf4.cu): the same
// items and outputs as launch_expert_mlp. Activations enter the products as four NVFP4
// pieces per row (E2M1 codes, E4M3 scale per 16 elements, piece p weighted 2^-3p): x4_perm
// [rows][4][d/2] codes and xs_perm [rows][4][d/16] scales of the dispatched rows; the gate/up
// epilogues write h's pieces to h4 [rows][4][I/2] and hs [rows][4][I/16]. N-tiles of at most
// 32 token rows; d and I multiples of 256.
int gemm_bn_max_nvf4(const Shape& s, int T);
cudaError_t launch_expert_mlp_nvf4(const Shape& s, const Nvfp4Experts& q, const uint8_t* x4_perm,
                                   const uint8_t* xs_perm, int rows, const int4* tiles, int* tile_done, int max_tiles,
                                   int bn_max, uint8_t* h4, uint8_t* hs, bf16* y, int* status, int num_sms,
                                   cudaStream_t st);
// The four NVFP4 pieces of the T BF16 token rows of width d: x4 [T][4][d/2], xs [T][4][d/16].
cudaError_t launch_act4_prep(const bf16* x, int d, int T, uint8_t* x4, uint8_t* xs, int* status, int num_sms,
                             cudaStream_t st);
// FP8 E4M3 expert weights on the FP8 tensor cores (expert_mlp_fp8.cu): the same items and
// outputs as launch_expert_mlp. Activations enter the products as two E4M3 pieces per row
// under a power-of-two row scale: x8_perm holds the dispatched pieces of x (per permuted
// row: p1 [d] then p2 [d], bytes), scaled by xmax[perm_src[row]]; h is split on chip with
// amax_h[row] (raised by the gate/up epilogues; zero on entry). N-tiles of at most 128 rows.
int gemm_bn_max_f8(const Shape& s, int T);
cudaError_t launch_expert_mlp_f8(const Shape& s, const Fp8Experts& q, const uint8_t* x8_perm, int rows, int T,
                                 const int* perm_src, const float* xmax, float* amax_h, const int4* tiles,
                                 int* tile_done, int max_tiles, int bn_max, bf16* h, bf16* y, int* status,
                                 int num_sms, cudaStream_t st);
// For the T BF16 token rows of width d: xmax[t] = max_j |x[t][j]| and x8[t] = the row's two
// E4M3 pieces (p1 [d] then p2 [d]) under the row's power-of-two scale; amax_h[0, rows) = 0.
cudaError_t launch_fp8_prep(const bf16* x, int d, int T, float* xmax, uint8_t* x8, float* amax_h, int rows,
                            int num_sms, cudaStream_t st);
// Dense MLP (one "expert", every token in order): the work list and its capacity.
int dense_max_tiles(int T, int bn_max);
cudaError_t launch_dense_tiles(int T, int bn_max, int4* tiles, int* tile_done, cudaStream_t st);

// ---------------------------------------------------------------- router product (router_gemm.cu)
// Split-K count of the tensor-core router product for T tokens.
int router_tc_splits(const Shape& s, int T, int num_sms);
// partial[split][t][e] = sum over the split's K range of x[t] . (hi + mid + lo)[e].
// selftest_extra_tx > 0 (failure-detection self-test only): the first pipeline stage of CTA
// 0 expects that many bytes more than its copies bring, so the MMA thread's bounded wait on
// it runs out and the kernel records kStatusWaitTimeout in `status`.
cudaError_t launch_router_tc(const Shape& s, const bf16* w3, const bf16* x, int T, int splits, float* partial,
                             int* status, int num_sms, cudaStream_t st, uint32_t selftest_extra_tx = 0);

// ---------------------------------------------------------------- combine (combine.cu)
cudaError_t launch_combine(const Shape& s, const bf16* y, const int* inv_slot, const float* topk_w, int T, bf16* out,
                           int* status, cudaStream_t st);
// Shard combine: FP32 partial sums over the slots of this shard (inv_slot >= 0).
cudaError_t launch_combine_partial(const Shape& s, const bf16* y, const int* inv_slot, const float* topk_w, int T,
                                   float* out, int* status, cudaStream_t st);

// ---------------------------------------------------------------- C-ABI helpers (api.cu)
// The calling thread's error message (what beam_moe_last_error returns) and the argument
// checks every entry point applies; each returns BEAM_MOE_OK or the failing code.
int abi_fail(int code, const char* fmt, ...);
int abi_check_config(const beam_moe_config* cfg);
int abi_check_ptr(const void* p, const char* name);
int abi_check_stream(cudaStream_t st);

// ---------------------------------------------------------------- sandwich norm (norm.cu)
// Largest row width the norm kernels take.
constexpr int kNormMaxD = 8192;
// out[t] = gamma * v[t] / sqrt(mean(v[t]^2) + eps), FP32, BF16 rows of width d (d % 4 == 0).
cudaError_t launch_rmsnorm(int d, const bf16* v, const bf16* gamma, float eps, int T, bf16* out, cudaStream_t st);
// Combine fused with the post-norm and the depth-scaled residual of contribution k:
// stream_out[t] = sqrt((k-1)/k) stream_in[t] + gamma * m / sqrt(mean(m^2) + eps) / sqrt(k),
// m = sum_k w[t,k] y[slot(t,k)] in FP32.
cudaError_t launch_combine_residual(const Shape& s, const bf16* y, const int* inv_slot, const float* topk_w, int T,
                                    const bf16* stream_in, const bf16* gamma, float eps, int k_contrib,
                                    bf16* stream_out, int* status, cudaStream_t st);

// ---------------------------------------------------------------- tcgen05 GEMM tiling (shared)
constexpr int kTileM = 128;    // weight rows per tile (MMA M)
constexpr int kTileK = 64;     // K per pipeline stage: one 128-byte swizzle row of BF16
constexpr int kMmaK = 16;      // K per tcgen05.mma (kind::f16)
constexpr int kBoxRows = 16;   // granule of token rows (MMA N step, smallest TMA box)
constexpr int kBoxKinds = 5;   // token-row tensor maps with boxes of 16, 32, 64, 128, 256 rows

// A BF16 [rows, cols] token-row operand as tensor maps that differ only in box height:
// m[i] has boxes of (16 << i) rows x 64 columns (128-byte swizzle).
struct BMaps {
    CUtensorMap m[kBoxKinds];
};
// Encodes the maps for every box height up to bn_max (larger ones repeat m[0]).
bool encode_bmaps(BMaps* b, const void* base, uint64_t rows, uint64_t cols, int bn_max, const char** why);
// As encode_bmaps for a byte matrix (E4M3 pieces): boxes of (16 << i) rows x 128 bytes.
bool encode_bmaps_u8(BMaps* b, const void* base, uint64_t rows, uint64_t cols, int box_max, const char** why);

// Host helper: encode a 2-D BF16 tensor map (rows x cols, row-major) with the 128-byte
// swizzle and a box of box_cols x box_rows. Returns false if the driver refuses it.
bool encode_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                         uint32_t box_cols, const char** why);

// Host helper: encode a 2-D byte tensor map (FP8 codes, rows x cols, row-major) with the
// 128-byte swizzle (box_cols <= 128): in shared memory the 16-byte chunk c of row r of a
// 128-byte-wide box sits at chunk c ^ (r & 7).
bool encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                       uint32_t box_cols, const char** why);
// The same without swizzle (rows of box_cols bytes one after another in shared memory).
bool encode_tmap_u8_2d_plain(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                             uint32_t box_cols, const char** why);

}  // namespace beam
