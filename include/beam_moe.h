/*
 * beam_moe.h - C ABI of the B300 (sm_103a) routed-MoE forward library, libbeam_moe.so.
 *
 * The operation is the forward pass of one routed Mixture-of-Experts block of Reflection's
 * Beam model, as the release pages describe it:
 *   - "Reflection releases Beam, a 501B open MoE model with 1M context" (Glonce),
 *     Architecture paragraph: 256 experts scored with a sigmoid, split into 8 groups of 32;
 *     the 4 best groups are kept and the top 8 experts picked from them; no shared expert;
 *     expert outputs combined with normalized router weights and scaled by 2.5; each
 *     expert a SwiGLU MLP with intermediate size 2,560 on hidden size 5,120.
 *   - transformers "Beam" model doc, Overview, "Sparse MoE" bullet: a learned per-expert
 *     bias balances load (selection); best topk_group of n_group groups; weights
 *     normalized; output scaled by routed_scaling_factor.
 *   - same page, paragraph after the bullets: routing and the SwiGLU activation run in
 *     FP32; router weights and expert bias are FP32; returned router logits are FP32.
 * Readings where the pages are silent: a group scores the sum of its two largest biased
 * scores (the DeepSeek-V3 convention the pages name); the bias is used for selection only;
 * ties go to the lower group, then the lower expert index; experts of dropped groups are
 * excluded; slots are ordered by descending biased score; the scale is folded into the
 * weights (they sum to `scale`); experts have no linear biases.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers on the current CUDA device, row-major and contiguous,
 *     16-byte aligned. The caller owns every buffer; the library keeps no pointer after
 *     a call returns. Outputs must not alias inputs.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream): results are valid
 *     once the stream has synchronised. No entry point synchronises the host except
 *     beam_moe_forward_host, beam_moe_device_status, beam_moe_route_noalloc_status and
 *     beam_moe_timing_read.
 *   - Scratch memory is taken from a library-owned stream-ordered pool on the current
 *     device and returned before the call's work completes (cudaMallocFromPoolAsync /
 *     cudaFreeAsync on `stream`); the pool keeps freed memory cached for the next call.
 *   - Return value: BEAM_MOE_OK (0) or a negative code; beam_moe_last_error() returns a
 *     message for the calling thread's last failure. T == 0 returns BEAM_MOE_OK and
 *     launches nothing. Device kernels never trap: a kernel that detects a bad index or a
 *     wait that ran past its limit records a code that beam_moe_device_status() returns.
 *   - Results are deterministic run to run for identical inputs.
 *   - Inputs must be finite.
 *
 * Supported shapes: d and I multiples of 128; E = 32 * n_group with 1 <= n_group <= 8;
 * 1 <= topk_group <= n_group; 1 <= top_k <= min(32, 32 * topk_group);
 * 0 <= T <= BEAM_MOE_MAX_TOKENS.
 */
#ifndef BEAM_MOE_H
#define BEAM_MOE_H

#include <stdint.h>
#include <cuda_runtime_api.h>
#include <cuda_bf16.h>

#if defined(__GNUC__)
#define BEAM_MOE_API __attribute__((visibility("default")))
#else
#define BEAM_MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define BEAM_MOE_OK 0
#define BEAM_MOE_ERR_ARG (-1)        /* null pointer, negative T, T too large, bad config */
#define BEAM_MOE_ERR_ALIGN (-2)      /* a pointer is not 16-byte aligned */
#define BEAM_MOE_ERR_CUDA (-3)       /* a CUDA runtime/driver call failed (message says which) */
#define BEAM_MOE_ERR_DEVICE (-4)     /* a kernel recorded a device-side error (beam_moe_device_status) */

#define BEAM_MOE_MAX_TOKENS 262144

/* Layer shape. Field names d, I, E are ours; n_group, topk_group and scale
 * (routed_scaling_factor) follow the transformers BeamConfig. */
typedef struct {
    int d;            /* hidden size (Beam: 5120) */
    int I;            /* expert intermediate size (Beam: 2560) */
    int E;            /* routed experts (Beam: 256) */
    int n_group;      /* expert groups (Beam: 8) */
    int topk_group;   /* groups kept per token (Beam: 4) */
    int top_k;        /* experts per token (Beam: 8) */
    float scale;      /* routed_scaling_factor (Beam: 2.5) */
} beam_moe_config;

/* Beam's layer: d=5120, I=2560, E=256, n_group=8, topk_group=4, top_k=8, scale=2.5. */
BEAM_MOE_API beam_moe_config beam_moe_default_config(void);

/* Router: FP32 logits l = x . router_w^T, s = sigmoid(l), c = s + expert_bias (selection
 * only), group score = top-2 sum of c, keep topk_group groups, pick top_k experts among
 * them by c, weights w_k = scale * s_k / sum_k s_k.
 *   x            bf16 [T, d]
 *   router_w     fp32 [E, d]
 *   expert_bias  fp32 [E]
 *   topk_idx     int32 [T, top_k]  out: expert ids, descending c, ties -> lower id
 *   topk_w       fp32  [T, top_k]  out: weights, sum = scale per token
 * beam_moe_route uses Beam's shape (beam_moe_default_config()). */
BEAM_MOE_API int beam_moe_route(const __nv_bfloat16 *x, const float *router_w, const float *expert_bias, int T,
                   int32_t *topk_idx, float *topk_w, cudaStream_t stream);
BEAM_MOE_API int beam_moe_route_ex(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w,
                      const float *expert_bias, int T, int32_t *topk_idx, float *topk_w, cudaStream_t stream);

/* Whole MoE block: route as above, then out[t] = sum_k w_k * SwiGLU_{e_k}(x[t]) with
 * SwiGLU_e(v) = w_down[e] . ( silu(w_gate[e] . v) * (w_up[e] . v) ), silu(z) = z sigmoid(z).
 *   w_gate, w_up  bf16 [E, I, d]   (nn.Linear [out, in] per expert)
 *   w_down        bf16 [E, d, I]
 *   out           bf16 [T, d]
 * Numerics: FP32 router; BF16 tensor-core products with FP32 accumulation; SwiGLU in FP32,
 * its result rounded to BF16 for the down product; each expert's output rounded to BF16 (the
 * model's dtype), the weighted combine summed in FP32 in slot order and rounded once to BF16.
 * beam_moe_forward uses Beam's shape. */
BEAM_MOE_API int beam_moe_forward(const __nv_bfloat16 *x, const float *router_w, const float *expert_bias,
                     const __nv_bfloat16 *w_gate, const __nv_bfloat16 *w_up, const __nv_bfloat16 *w_down, int T,
                     __nv_bfloat16 *out, cudaStream_t stream);
BEAM_MOE_API int beam_moe_forward_ex(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w,
                        const float *expert_bias, const __nv_bfloat16 *w_gate, const __nv_bfloat16 *w_up,
                        const __nv_bfloat16 *w_down, int T, __nv_bfloat16 *out, cudaStream_t stream);

/* The block of beam_moe_forward_ex with the tokens and the output in HOST memory: copies
 * x_host [T, d] BF16 to the device, runs the block, copies the output back to out_host
 * [T, d] BF16, all on `stream`, and returns once the stream has finished (this call
 * synchronises the host). The device copies of x and out come from the library's pool.
 * Page-locked (pinned) host buffers let the copies run asynchronously; pageable ones work,
 * with copies the driver stages. The weights, router and bias are device pointers as for
 * beam_moe_forward_ex; errors as there. */
BEAM_MOE_API int beam_moe_forward_host(const beam_moe_config *cfg, const __nv_bfloat16 *x_host, const float *router_w,
                          const float *expert_bias, const __nv_bfloat16 *w_gate, const __nv_bfloat16 *w_up,
                          const __nv_bfloat16 *w_down, int T, __nv_bfloat16 *out_host, cudaStream_t stream);

/* Whole MoE block with FP8 expert weights. The pages ship FP8 (and NVFP4) checkpoints of the
 * model (Glonce "Reflection releases Beam ...", Hardware paragraph; transformers "Beam" doc,
 * checkpoint formats) but give no quantisation recipe; this call takes the plainest
 * weight-only reading: FP8 E4M3 codes (bit 7 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; 0x7F/0xFF are NaN and must not occur) with one FP32 scale per output row,
 *   Wg[e][i][j] = gate_scale[e][i] * e4m3(w_gate_q[e][i][j])      w_gate_q, w_up_q u8 [E, I, d]
 *   Wu[e][i][j] = up_scale[e][i]   * e4m3(w_up_q[e][i][j])        gate_scale, up_scale f32 [E, I]
 *   Wd[e][j][i] = down_scale[e][j] * e4m3(w_down_q[e][j][i])      w_down_q u8 [E, d, I], down_scale f32 [E, d]
 * and otherwise the block of beam_moe_forward_ex: same routing, activations and output in
 * BF16. Numerics: the products run on the FP8 tensor cores with the codes as they are and
 * FP32 accumulation; each BF16 activation row (x, and h after its BF16 rounding) enters
 * them as two E4M3 pieces under one power-of-two row scale s, v = s p1 + (s/16) p2, which is
 * exact for every value within 2^-10 of the row's largest magnitude (smaller ones carry an
 * absolute error of at most 2^-14 s, below 2.8e-7 of it); each accumulator is multiplied by its row's scale in
 * FP32 before SwiGLU (gate/up) or before rounding the expert output (down). All pointers are
 * device memory, 16-byte aligned, owned by the caller and only read (out is written); errors
 * as for beam_moe_forward_ex. */
BEAM_MOE_API int beam_moe_forward_fp8(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w,
                         const float *expert_bias, const uint8_t *w_gate_q, const float *gate_scale,
                         const uint8_t *w_up_q, const float *up_scale, const uint8_t *w_down_q,
                         const float *down_scale, int T, __nv_bfloat16 *out, cudaStream_t stream);

/* Whole MoE block with NVFP4 expert weights. The pages ship an NVFP4 checkpoint of about 4.5
 * bits per weight for Blackwell GPUs (Glonce "Reflection releases Beam ...", Hardware
 * paragraph; Atech "Reflection ... Beam ...", checkpoint sizes) but give no layout; this call
 * takes the public NVFP4 layout as the reading: E2M1 codes (bit 3 sign, 2 exponent bits with
 * bias 1, 1 mantissa bit) packed two per byte, element 2k in the low half of byte k; one E4M3
 * scale per block of 16 consecutive elements of a row; one FP32 scale per expert matrix:
 *   Wg[e][i][j] = gate_tensor_scale[e] * e4m3(gate_block_scale[e][i][j/16]) * e2m1(code j of row i)
 *   w_gate_q, w_up_q u8 [E, I, d/2]; gate_block_scale, up_block_scale u8 [E, I, d/16]
 *   w_down_q u8 [E, d, I/2]; down_block_scale u8 [E, d, I/16]; *_tensor_scale f32 [E]
 * and otherwise the block of beam_moe_forward_ex (same routing, BF16 activations and
 * output). Numerics: the products run on the block-scaled FP4 tensor cores with the codes
 * and block scales as they are and FP32 accumulation. Each activation row (x, and h in FP32
 * straight from SwiGLU) enters them as four NVFP4 pieces: per block of 16 elements, piece p
 * has the E4M3 scale u_p = the least E4M3 value >= 4^p max|r_p| / 6 and the E2M1 codes of
 * r_p / (4^-p u_p) rounded to nearest, r_0 = v, r_(p+1) = r_p - 4^-p u_p e2m1(code); what
 * is left after four pieces is at most 1.2e-3 of the block's largest magnitude (above an
 * absolute floor of 2^-15 from the smallest scales). The tensor
 * scale is applied to each accumulator. A block whose largest magnitude exceeds 2688 is
 * clamped and recorded in the device status word (code 4). d and I must be multiples of 256.
 * Pointers as for beam_moe_forward_fp8. */
BEAM_MOE_API int beam_moe_forward_nvfp4(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w,
                           const float *expert_bias, const uint8_t *w_gate_q, const uint8_t *gate_block_scale,
                           const float *gate_tensor_scale, const uint8_t *w_up_q, const uint8_t *up_block_scale,
                           const float *up_tensor_scale, const uint8_t *w_down_q, const uint8_t *down_block_scale,
                           const float *down_tensor_scale, int T, __nv_bfloat16 *out, cudaStream_t stream);

/* One expert-parallel shard of the MoE block. The pages' multi-GPU plan puts each expert on
 * one device and replicates the rest, with a device count that divides 256 (Glonce "Reflection
 * releases Beam ...", Running it paragraph; transformers "Beam" doc, Usage examples: expert
 * parallelism with torchrun). The calling device holds experts [e_begin, e_end) only:
 *   w_gate, w_up  bf16 [e_end - e_begin, I, d];  w_down  bf16 [e_end - e_begin, d, I]
 * Routing runs over all E experts (router_w and expert_bias are the full, replicated ones);
 * the call runs the (token, slot) pairs routed to its experts and writes
 *   out_partial[t] = sum over slots k with e_k in [e_begin, e_end) of w_k * SwiGLU_{e_k}(x[t])
 * FP32 [T, d], not rounded (slots in order). The sum of out_partial over shards that cover
 * [0, E) is the block's output before its rounding to BF16: the combine of expert
 * parallelism is a sum over devices (an all-reduce). Tokens with no slot on this shard get 0. */
BEAM_MOE_API int beam_moe_forward_shard(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w,
                           const float *expert_bias, const __nv_bfloat16 *w_gate, const __nv_bfloat16 *w_up,
                           const __nv_bfloat16 *w_down, int e_begin, int e_end, int T, float *out_partial,
                           cudaStream_t stream);

/* Dense SwiGLU MLP of the first decoder layers (Glonce "Reflection releases Beam ...",
 * Architecture paragraph: the first 3 layers are dense SwiGLU MLPs; transformers "Beam" doc:
 * mlp_layer_types sets the pattern, SwiGLU activation in FP32). The pages give no width for
 * it, so I is the caller's:
 *   out[t] = w_down . ( silu(w_gate . x[t]) * (w_up . x[t]) ),  silu(z) = z sigmoid(z)
 *   x, out bf16 [T, d]; w_gate, w_up bf16 [I, d]; w_down bf16 [d, I]; d, I multiples of 128.
 * Same kernel and numerics as the experts (BF16 products, FP32 accumulation and activation,
 * the activation rounded to BF16 for the down product), output rounded once to BF16. */
BEAM_MOE_API int beam_moe_dense_mlp(int d, int I, const __nv_bfloat16 *x, const __nv_bfloat16 *w_gate,
                       const __nv_bfloat16 *w_up, const __nv_bfloat16 *w_down, int T, __nv_bfloat16 *out,
                       cudaStream_t stream);

/* Pre-norm of the MoE sublayer (transformers "Beam" doc, Overview, "Sandwich norms with
 * depth-scaled residuals" bullet: each block is wrapped in an RMSNorm before and after;
 * the paragraph after the bullets: RMSNorm scaling is computed in FP32):
 *   out[t][j] = gamma[j] * v[t][j] / sqrt( (1/d) sum_i v[t][i]^2 + eps ),  FP32, rounded to BF16.
 * Readings: the gain multiplies the normalised row directly; eps is the caller's (the
 * pages give no value).
 *   v, out  bf16 [T, d], rows contiguous; gamma bf16 [d]; d a multiple of 4, at most 8192.
 * out may equal v (in place). Deterministic (fixed reduction order). */
BEAM_MOE_API int beam_moe_rmsnorm(int d, const __nv_bfloat16 *v, const __nv_bfloat16 *gamma, float eps, int T,
                     __nv_bfloat16 *out, cudaStream_t stream);

/* The whole MoE sublayer of a decoder layer on the residual stream: sandwich norms around
 * the MoE block and the depth-scaled residual (same bullet; Glonce "Reflection releases
 * Beam ...", paragraph on the residual connections: counting the input embedding as step
 * 1, step k adds the sublayer output with weight 1/sqrt(k) and keeps the stream with
 * weight sqrt((k-1)/k)):
 *   x   = RMSNorm(stream_in; pre_gamma, eps)                       (BF16, as beam_moe_rmsnorm)
 *   m   = MoE block of beam_moe_forward_ex on x, kept in FP32 (not rounded to BF16)
 *   stream_out = sqrt((k-1)/k) stream_in + RMSNorm(m; post_gamma, eps) / sqrt(k)   (FP32 -> BF16)
 * The post-norm and the residual update run fused into the combine kernel.
 *   stream_in, stream_out  bf16 [T, d]; pre_gamma, post_gamma bf16 [d]; k >= 2 is this
 *   sublayer's contribution index (the MoE sublayer of decoder layer l, 0-based, is
 *   k = 2l + 3 when every layer has an attention and an MLP sublayer); d <= 8192.
 * stream_out may equal stream_in (in-place update); other outputs must not alias inputs. */
BEAM_MOE_API int beam_moe_sublayer_forward(const beam_moe_config *cfg, const __nv_bfloat16 *stream_in,
                              const __nv_bfloat16 *pre_gamma, const __nv_bfloat16 *post_gamma, float eps, int k,
                              const float *router_w, const float *expert_bias, const __nv_bfloat16 *w_gate,
                              const __nv_bfloat16 *w_up, const __nv_bfloat16 *w_down, int T,
                              __nv_bfloat16 *stream_out, cudaStream_t stream);

/* Router with no device allocation. The release pages have no counterpart: this is a
 * deployment variant of beam_moe_route_ex for callers that must not have a library
 * allocate device memory (an engine that has claimed all free HBM for weights and KV
 * cache, or a per-token path where an allocator call could synchronise the device or
 * stall). Same arguments, layouts and outputs as beam_moe_route_ex; calls no cudaMalloc,
 * cudaFree or pool allocation.
 *   - Scratch: one fixed array of BEAM_MOE_NOALLOC_SCRATCH_BYTES in the library's device
 *     image; every GPU that loads the library holds it until the process exits.
 *   - Limit: T <= BEAM_MOE_NOALLOC_MAX_TOKENS, else BEAM_MOE_ERR_ARG with a message.
 *   - Results equal beam_moe_route_ex's bit for bit while the array holds the K split
 *     count beam_moe_route_ex picks, which is the case for every T <= 8192 on a 148-SM
 *     B300 at Beam's shape. On a GPU where it cannot (more SMs, hence more splits), fewer
 *     splits are used: only the summation order of the FP32 logits differs then, which can
 *     change a pick only between near-tied experts. beam_moe_route_noalloc_plan tells.
 *   - The first call on each device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents (every value a call
 *     reads is written earlier in the same call). Calls that overlap on the GPU race on
 *     it: serialise them (one stream, or events between streams).
 *   - Kernel errors (a pipeline wait that ran past its limit) go to this entry point's own
 *     status word, read with beam_moe_route_noalloc_status, not beam_moe_device_status.
 *   - Not counted by beam_moe_last_launch_count or timed by beam_moe_timing_*. */
#define BEAM_MOE_NOALLOC_MAX_TOKENS 8192
#define BEAM_MOE_NOALLOC_SCRATCH_BYTES (40u << 20)
BEAM_MOE_API int beam_moe_route_noalloc(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w,
                           const float *expert_bias, int T, int32_t *topk_idx, float *topk_w, cudaStream_t stream);

/* Host-only planning query of beam_moe_route_noalloc (no GPU work, no allocation): writes to
 * *splits the number of K split planes a call with T tokens makes on a GPU with num_sms SMs,
 * or returns BEAM_MOE_ERR_ARG if T is outside [1, BEAM_MOE_NOALLOC_MAX_TOKENS] or the array
 * cannot hold even one plane. The split count of beam_moe_route_ex is the same unless the
 * array forced fewer. */
BEAM_MOE_API int beam_moe_route_noalloc_plan(const beam_moe_config *cfg, int T, int num_sms, int *splits);

/* Synchronises `stream`, then returns and clears the no-allocation router's kernel status
 * word on the current device: BEAM_MOE_OK, or BEAM_MOE_ERR_DEVICE if one of its kernels
 * recorded an error since the last read (its outputs are then not valid). Allocates
 * nothing. */
BEAM_MOE_API int beam_moe_route_noalloc_status(cudaStream_t stream);

/* Self-test of the no-allocation router's failure detection (no counterpart on the pages):
 * runs its tensor-core logits kernel on one tile of zeros laid out in the fixed array, with
 * the first pipeline stage expecting 16 bytes more than its copies deliver, so the MMA
 * thread's bounded wait (2 s) runs out and the kernel records it in the status word that
 * beam_moe_route_noalloc_status reads; the CTA frees its tensor memory and exits, and the
 * context stays usable. Overwrites the start of the array; allocates nothing. */
BEAM_MOE_API int beam_moe_route_noalloc_selftest(cudaStream_t stream);

/* Router logits only (output_router_logits in the transformers doc, Notes): the same
 * kernels as the router's first stage; logits fp32 [T, E]. */
BEAM_MOE_API int beam_moe_router_logits(const beam_moe_config *cfg, const __nv_bfloat16 *x, const float *router_w, int T,
                           float *logits, cudaStream_t stream);

/* Message for the calling thread's last non-zero return (empty string if none). */
BEAM_MOE_API const char *beam_moe_last_error(void);

/* Synchronises `stream`, then returns and clears the current device's kernel status word:
 * 0 if no kernel recorded an error since the last call, else BEAM_MOE_ERR_DEVICE (the
 * message names the recorded code: 1 = an expert index out of range reached dispatch,
 * 2 = a pipeline wait in a GEMM ran past its limit, 3 = a permuted row or work-list index
 * out of range, 4 = an activation block of the NVFP4 block above 2688 in magnitude). */
BEAM_MOE_API int beam_moe_device_status(cudaStream_t stream);

/* Self-test of failure detection (no counterpart on the pages). Runs the expert kernel on a
 * library-built one-tile work list (one expert, d = I = 128, zero weights) whose completion
 * counter is set far below zero, so the down item's producer waits out its bounded wait
 * (2 s), records "a GEMM pipeline wait ran past its limit" in the device status word, and
 * its CTA drains its copies and MMAs and frees its tensor memory before exiting. Returns
 * BEAM_MOE_OK once the work is queued on `stream`; a following beam_moe_device_status()
 * then returns BEAM_MOE_ERR_DEVICE (and clears the word), and the context stays usable.
 * Takes about two seconds of GPU time. */
BEAM_MOE_API int beam_moe_selftest_wait_timeout(cudaStream_t stream);

/* Per-stage timing for profiling. While enabled (per thread), each forward/route call
 * records CUDA events on its stream around each stage; beam_moe_timing_read synchronises
 * on the last call's final event and writes up to max_stages durations in milliseconds
 * (stage order: pre-norm, router weight split, router logits, router select, dispatch count,
 * dispatch scan, dispatch scatter, gather, expert MLP (gate/up, SwiGLU and down in one
 * kernel), combine (fused with the post-norm and residual in beam_moe_sublayer_forward),
 * activation split (the FP8 and NVFP4 blocks' pieces of the token rows); for T <= 128 the whole dispatch and gather is one launch, timed as dispatch count; unrun
 * stages read 0). Returns the number of stages, or a negative error. */
BEAM_MOE_API int beam_moe_timing_enable(int enable);
BEAM_MOE_API int beam_moe_timing_read(float *ms, int max_stages);

/* Number of kernel launches the last forward/route call on this thread made. */
BEAM_MOE_API int beam_moe_last_launch_count(void);

/* Debug aid (process-wide): while enabled, every scratch allocation of the pool-backed
 * entry points is filled with 0xFF bytes (NaN in BF16 and FP32, -1 in int32) on `stream`
 * before the call's kernels run, so that any scratch value read before it is written
 * reaches the output as a NaN or an out-of-range index (recorded in the status word). The
 * results of a correct build do not change. Off by default; the environment variable
 * BEAM_MOE_DEBUG=1 turns it on at the library's first call. Costs one memset per call. */
BEAM_MOE_API int beam_moe_debug_poison_scratch(int enable);

#ifdef __cplusplus
}
#endif
#endif /* BEAM_MOE_H */
