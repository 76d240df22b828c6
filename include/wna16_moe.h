/*
 * wna16_moe.h - C ABI of a fused Mixture-of-Experts layer with weight-only,
 * group-quantized experts (int4 "W4A16" GPTQ/AWQ style and int8 "W8A16"), for
 * one NVIDIA GB300 (sm_103a).
 *
 * The operation. Pages on which this is based:
 *   - vLLM PR #12185 "[Kernel] add triton fused moe kernel for gptq/awq": one
 *     fused MoE launch over gptq/awq int4 expert weights instead of one GEMM per
 *     expert; note 1 of that PR: a shared-memory, CUDA-graph-safe
 *     moe_align_block_size that scales to DeepSeek-V3's 256 experts.
 *   - vLLM PR #6502 "[Model] Add Support for GPTQ Fused MOE": the K tile of the
 *     GEMM must respect the quantization group (bug report on BLOCK_SIZE_K).
 *   - vLLM fused_moe/oracle/int8.py: int8 W8A16 experts, symmetric, one scale
 *     per output channel; weights shaped [experts, ..., N, K].
 *   - vLLM PR #14138 "optimize performance of gptq marlin kernel when n is
 *     small": uint4 codes, group_size 128, integer zero points; reducing split
 *     partial results without a grid barrier.
 *
 * For M tokens x[t] (hidden size H), top-k expert ids e = ids[t, j] and weights
 * w[t, j], each expert holding a gate/up matrix W13[e] (2I x H) and a down
 * matrix W2[e] (H x I):
 *     g = W13[e][0:I] x_t,  u = W13[e][I:2I] x_t,  a = silu(g) * u,
 *     y_{t,j} = W2[e] a,    out_t = sum_j w[t, j] * y_{t,j}   (slot order).
 * Dequantized weight: W[n, k] = (code[n, k] - zero[k / G, n]) * scale[k / G, n].
 *
 * Memory layout of the quantized weights (all row-major, little-endian):
 *   pf = 32 / bits codes per int32 word.
 *   q      [E, N, K/pf] int32   code of k in bits [bits*(k%pf), +bits) of word k/pf
 *   scales [E, K/G, N]  fp16 or bf16 (scale_dtype), group-major
 *   zeros  [E, K/G, N/pf] int32 zero point of row n in bits [bits*(n%pf), +bits)
 *                       of word n/pf; NULL = symmetric, zero point 2^(bits-1)
 *   with (N, K) = (2I, H) for w13 (rows [0,I) gate, [I,2I) up) and (H, I) for w2.
 *   group_size G: 64 or a multiple of 128 that divides K (a 128-wide K stage
 *   of the kernels never straddles two groups), or -1 for one group per output
 *   channel (G = K).
 *
 * Ownership and threading. Every pointer is a non-owning DEVICE pointer on the
 * current CUDA device unless stated otherwise, 16-byte aligned. The library
 * never allocates, frees or synchronizes device memory (except
 * wna16_read_device_status, which synchronizes the given stream). All compute
 * calls are asynchronous on `stream` (a cudaStream_t; NULL = default stream),
 * issue no host synchronization and, with fixed arguments, can be captured in a
 * CUDA graph and replayed.
 *
 * Errors. Argument errors are detected on the host and returned before
 * anything is launched. Launch failures return WNA16_ERR_CUDA. Errors found on
 * the device (an expert id outside [0, E), a pipeline wait that gave up) do not
 * trap: the offending pair is dropped or the kernel returns early, and a bit is
 * set in the status word at the start of the workspace (read it with
 * wna16_read_device_status).
 */
#ifndef WNA16_MOE_H_
#define WNA16_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  WNA16_OK = 0,
  WNA16_ERR_INVALID_ARG = 1,          /* null pointer, bad size or alignment */
  WNA16_ERR_UNSUPPORTED = 2,          /* valid but not supported (shape, bits, G) */
  WNA16_ERR_WORKSPACE_TOO_SMALL = 3,
  WNA16_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed */
  WNA16_ERR_DEVICE_BAD_EXPERT_ID = 5, /* device: an id outside [0, E) was dropped */
  WNA16_ERR_DEVICE_TIMEOUT = 6,       /* device: a pipeline wait gave up */
  WNA16_ERR_DEVICE_BAD_GROUPS = 7     /* device: act-order g_idx is not a split into groups of G */
} wna16_status;

/* Element types. Activations, outputs and scales: F16 or BF16; F32 only for
 * router logits (wna16_topk_routing). */
typedef enum { WNA16_F16 = 0, WNA16_BF16 = 1, WNA16_F32 = 2 } wna16_dtype;

/* Router score functions of wna16_topk_routing. */
typedef enum { WNA16_SCORE_SOFTMAX = 0, WNA16_SCORE_SIGMOID = 1 } wna16_scoring;

/* Device status bits (the int32 at offset 0 of the fused-call workspace). */
#define WNA16_DEV_BAD_EXPERT_ID 0x1
#define WNA16_DEV_TIMEOUT 0x2
#define WNA16_DEV_BAD_GROUPS 0x4

/*
 * Capacity of the align outputs: an upper bound on padded slots for
 * num_pairs = M * topk pairs over E experts and GEMM block size `block`:
 * roundup(num_pairs + min(num_pairs, E) * (block - 1), block).
 * (Every non-empty expert pads fewer than `block` slots.) Returns -1 on bad
 * arguments.
 */
int64_t wna16_align_capacity(int64_t num_pairs, int E, int block);

/*
 * moe_align_block_size (vLLM PR #12185, note 1; one CTA, shared-memory
 * histogram, warp-level ranking, block scan; graph-safe).
 *   topk_ids   [M, topk] int32 expert id per (token, slot); pair p = t*topk + j.
 *   sorted_ids [cap] int32 out: pairs grouped by expert in ascending expert
 *              order, ascending pair index within an expert, each expert padded
 *              to a multiple of `block` with the sentinel M*topk; slots past the
 *              padded total hold the sentinel. cap = wna16_align_capacity(...).
 *   expert_ids [cap / block] int32 out: expert of each block, -1 past the end.
 *   num_tokens_post_padded [1] int32 out: padded total (a multiple of block).
 *   expert_counts [E] int32 out, optional (NULL): pairs per expert.
 *   device_status [1] int32, optional (NULL): reset to 0 by this call, then
 *              WNA16_DEV_BAD_EXPERT_ID is or-ed in if an id is outside [0, E)
 *              (that pair is dropped).
 *   block: a power of two in [16, 256]. E in [1, 256]. M*topk < 2^31.
 */
wna16_status wna16_moe_align_block_size(const int32_t* topk_ids, int64_t M, int topk, int E,
                                        int block, int32_t* sorted_ids, int32_t* expert_ids,
                                        int32_t* num_tokens_post_padded, int32_t* expert_counts,
                                        int32_t* device_status, void* stream);

/*
 * Block size the fused call uses when given block = 0, from the average routed
 * pairs per active expert, avg = M * topk / min(M * topk, E) (the routing
 * itself is not seen on the host):
 *   E <= 16 and avg > 48: 128 (one block per expert; the MMA width and the
 *     epilogue cover only the block's routed pairs, rounded up to 16);
 *   avg <= 64 (weight streaming dominates): the tile of 16, 32 or 64 tokens
 *     with the least estimated streaming cost, ceil(1.3 * avg / tile) passes
 *     over the expert's weights times the measured cost of one pass with that
 *     tile (1.0, 1.28, 1.34);
 *   avg > 64 (tensor-bound): the smallest power of two >= avg, from 64 up to
 *     128.
 * Returns 16 when M * topk <= 0.
 */
int wna16_choose_block(int64_t M, int topk, int E);

/*
 * Top-k routing: router logits -> the topk_ids / topk_weights the align and
 * fused calls take. The pages name top-k routing ids and weights as the
 * layer's first stage (vLLM PR #12185; the Mixtral, Qwen2-MoE and DeepSeek-V3
 * models of PR #12185 and PR #6502) and give no formulas; these are the
 * readings implemented:
 *   scores: softmax over the row's E logits, or sigmoid 1 / (1 + exp(-l));
 *   ranking: larger logit first, ties to the lower expert index, NaN ranked as
 *     -inf (both score functions increase with the logit, so this is the
 *     ranking by score, taken on the exact input values);
 *   n_groups > 1 (DeepSeek-V3 style): experts [g*E/n_groups, (g+1)*E/n_groups)
 *     form group g; a group's score is the sum of the scores of its two
 *     best-ranked experts (fp32); the topk_groups best groups are kept (larger
 *     score first, ties to the lower group, NaN as -inf) and the top-k experts
 *     are ranked among them only;
 *   weights: the selected scores; with renormalize != 0 divided by their sum
 *     (for softmax: the softmax over the selected logits). Computed in fp32.
 *   logits       [M, E] fp32, fp16 or bf16 (logits_dtype), row-major, aligned
 *                to its element size.
 *   topk_ids     [M, topk] int32 out: slot j = the j-th best selected expert.
 *   topk_weights [M, topk] fp32 out.
 *   E in [1, 256], topk in [1, min(E, 32)], n_groups in [1, 32] dividing E;
 *   with n_groups > 1: E / n_groups >= 2, topk_groups in [1, n_groups] and
 *   topk <= topk_groups * E / n_groups (topk_groups is ignored otherwise).
 * One warp per row, one launch, no workspace, graph-safe. M = 0 launches
 * nothing. Non-finite logits give valid, distinct ids; their weights follow
 * IEEE arithmetic (NaN may appear).
 */
wna16_status wna16_topk_routing(const void* logits, wna16_dtype logits_dtype, int64_t M, int E, int topk,
                                wna16_scoring scoring, int renormalize, int n_groups, int topk_groups,
                                int32_t* topk_ids, float* topk_weights, void* stream);

/*
 * Bytes of workspace wna16_fused_moe needs for these sizes on the current
 * device (block = 0: the automatic choice, split_k = 0: automatic). Returns 0
 * on bad arguments.
 */
size_t wna16_fused_moe_workspace_bytes(int64_t M, int64_t H, int64_t I, int E, int topk,
                                       int bits, int group_size, int block, int split_k);

/*
 * The fused layer: align -> gather of the routed token rows into expert order
 * -> gate/up GEMM with in-kernel dequant and silu(gate)*up -> down GEMM with
 * in-kernel dequant and the top-k weight -> ordered top-k combine. One launch
 * per stage (5 launches), none per expert.
 *   hidden       [M, H] act_dtype.
 *   w13_q/w13_scales/w13_zeros, w2_q/w2_scales/w2_zeros: layout above
 *                (zeros may be NULL; both NULL or both non-NULL).
 *   scale_dtype  dtype of both scale tensors.
 *   bits         4 or 8. group_size: 64 or a multiple of 128 dividing H and I,
 *                or -1.
 *   topk_ids     [M, topk] int32; topk_weights [M, topk] fp32.
 *   out          [M, H] act_dtype, written (never read).
 *   workspace    device memory of at least wna16_fused_moe_workspace_bytes();
 *                its first int32 is the device status word (reset by the call).
 *   block        align block size (0 = automatic), as in
 *                wna16_moe_align_block_size; it is also the GEMM token tile.
 *                With more than 16 experts, blocks of 128 and 256 are refused
 *                (WNA16_ERR_UNSUPPORTED; the automatic choice never takes them
 *                there): forced 128-token blocks on such layers ended in an
 *                unexplained launch failure (256 experts at M = 256, 64 experts
 *                at M = 128), although wna16_check_launch_plan finds every
 *                index of those launch plans in bounds. Forced 32 and 64 are
 *                accepted on any layer.
 *   split_k      K-splits of the down GEMM (0 = automatic, else 1..8).
 * Shapes: H a multiple of 64, I a multiple of 64, 1 <= topk <= E <= 256,
 * M*topk < 2^31. M = 0 returns WNA16_OK and launches nothing.
 * Numerics: fp32 accumulation, one rounding of the output; the act cache
 * silu(g)*u is stored in act_dtype. Token tiles of 32+ rows dequantize each
 * weight to act_dtype, (code - zero) * scale rounded once. 16-row tiles with
 * G >= 128 or per-channel scales (int4, or int8 with fp16) never round the
 * weights: the MMA multiplies exact integer codes and the zero point and scale
 * are applied in fp32. With fp16 activations the sum of one 128-wide K
 * stage's activations (of one token) must stay below about 2.1e6 there.
 */
wna16_status wna16_fused_moe(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                             int64_t I, int E, int topk, const int32_t* w13_q,
                             const void* w13_scales, const int32_t* w13_zeros,
                             const int32_t* w2_q, const void* w2_scales,
                             const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits,
                             int group_size, const int32_t* topk_ids,
                             const float* topk_weights, void* out, void* workspace,
                             size_t workspace_bytes, int block, int split_k, void* stream);

/*
 * wna16_fused_moe with per-launch timing: identical launches, and if
 * `events` is non-NULL, events[i] (a cudaEvent_t, NULL entries skipped) is
 * recorded on `stream` right before launch i (0 align, 1 token gather,
 * 2 gate/up GEMM, 3 down GEMM, 4 combine) and events[5] after the last launch.
 * For benchmarks.
 */
wna16_status wna16_fused_moe_timed(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                   int64_t I, int E, int topk, const int32_t* w13_q,
                                   const void* w13_scales, const int32_t* w13_zeros,
                                   const int32_t* w2_q, const void* w2_scales,
                                   const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits,
                                   int group_size, const int32_t* topk_ids,
                                   const float* topk_weights, void* out, void* workspace,
                                   size_t workspace_bytes, int block, int split_k, void* stream,
                                   void* const* events);

/*
 * Plans: the fused layer for a fixed set of weights, called many times (a
 * serving loop that does not capture CUDA graphs). wna16_plan_create checks
 * the weight arguments once and encodes the weights' TMA descriptors once, in
 * host memory; wna16_fused_moe_plan then runs the layer on a batch with only
 * the batch-dependent work left on the host (the batch's checks, its launch
 * plan, the two token-tile descriptors and the launches).
 *   wna16_plan_create: arguments as wna16_fused_moe (weights: device pointers
 *     that must stay valid and unchanged while the plan is used). Writes a
 *     new plan to *plan (NULL on error). Makes no CUDA allocation, launch or
 *     synchronization.
 *   wna16_plan_destroy: frees a plan (NULL is ignored). Calls still running on
 *     the GPU are not affected (they hold copies of the descriptors).
 *   wna16_fused_moe_plan: wna16_fused_moe with the plan's weights; same
 *     workspace size (wna16_fused_moe_workspace_bytes), errors and semantics.
 * A plan may be used from several host threads at once (it is only read).
 */
typedef struct wna16_plan_t wna16_plan_t;

wna16_status wna16_plan_create(wna16_dtype act_dtype, int64_t H, int64_t I, int E, int topk, const int32_t* w13_q,
                               const void* w13_scales, const int32_t* w13_zeros, const int32_t* w2_q,
                               const void* w2_scales, const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits,
                               int group_size, wna16_plan_t** plan);
void wna16_plan_destroy(wna16_plan_t* plan);
wna16_status wna16_fused_moe_plan(const wna16_plan_t* plan, const void* hidden, int64_t M, const int32_t* topk_ids,
                                  const float* topk_weights, void* out, void* workspace, size_t workspace_bytes,
                                  int block, int split_k, void* stream);

/*
 * Size of the library-owned scratch area used by wna16_fused_moe_noalloc:
 * 64 MiB, reserved on every GPU that loads the library, for as long as the
 * library stays loaded.
 */
#define WNA16_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * wna16_fused_moe for callers that cannot hand the library a workspace. The
 * pages this library follows have no counterpart of this entry point; it exists
 * for host code that has no allocator to draw from: a plain C program or a
 * plugin living inside a process whose memory manager owns the device memory
 * (where an extra cudaMalloc would fail against a fixed budget or break that
 * manager's bookkeeping). It takes the same arguments as wna16_fused_moe minus
 * the workspace, and allocates nothing: the workspace is a fixed area of
 * WNA16_NOALLOC_SCRATCH_BYTES inside the library's own device data.
 *   - Sizes whose wna16_fused_moe_workspace_bytes() exceeds
 *     WNA16_NOALLOC_SCRATCH_BYTES are rejected with
 *     WNA16_ERR_WORKSPACE_TOO_SMALL before anything is launched (decode-sized
 *     batches of the supported layers fit; large prefill batches do not: use
 *     wna16_fused_moe with a workspace for those).
 *   - The first call on a device looks up the area's device address on the
 *     current device (a one-time set-up per device, repeated only if the
 *     device's CUDA context was replaced, e.g. after cudaDeviceReset); make
 *     that first call before any stream capture.
 *   - Every call on a device shares the one area, which keeps whatever the
 *     last call left in it. Each call rewrites everything it later reads (the
 *     device status word at its start is reset by the call), so nothing has
 *     to be cleared between calls. wna16_noalloc_read_status reads that
 *     status word (the errors found on the device by the last call).
 *   - Calls whose GPU execution overlaps (issued on different streams, or
 *     from different host threads without ordering) race on the area and
 *     corrupt each other's results: serialize them.
 */
wna16_status wna16_fused_moe_noalloc(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                     int64_t I, int E, int topk, const int32_t* w13_q,
                                     const void* w13_scales, const int32_t* w13_zeros,
                                     const int32_t* w2_q, const void* w2_scales,
                                     const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits,
                                     int group_size, const int32_t* topk_ids,
                                     const float* topk_weights, void* out, int block, int split_k,
                                     void* stream);

/*
 * The device status word of the last wna16_fused_moe_noalloc call on the
 * current device (the pages have no counterpart either): the
 * wna16_read_device_status of the library-owned area. Synchronizes `stream`
 * (issue it on the stream of that call, or after it completed), writes the
 * raw WNA16_DEV_* bits to *bits_out (may be NULL) and returns as
 * wna16_read_device_status does.
 */
wna16_status wna16_noalloc_read_status(int32_t* bits_out, void* stream);

/*
 * Prepacked weights (optional, a one-time conversion at load time).
 *
 * The GPTQ-Marlin kernels of vLLM PR #14138 run on weights repacked offline
 * into the kernel's own tile order; this is the same idea for this library.
 * wna16_prepack rewrites one projection (w13 or w2) from the plain layout above
 * into stage images: for every (expert, 128-row tile, 128-wide K stage), one
 * contiguous block that is byte-identical to the shared-memory stage the GEMM
 * kernels assemble from the plain layout (codes in their swizzled order, then
 * the stage's scales, then its zero points). The fused call then moves each
 * stage with one contiguous bulk copy instead of three strided tiled copies;
 * the arithmetic, and so the output, is unchanged (bit-identical).
 *
 *   wna16_prepack_bytes: size of the packed form of one projection with
 *     (N, K) = (2I, H), gate_up = 1 for w13, or (H, I), gate_up = 0 for w2;
 *     0 for unsupported shapes (same rules as wna16_fused_moe).
 *   wna16_prepack: q / scales / zeros (zeros may be NULL) in the plain layout
 *     -> dst (device, 16-byte aligned, wna16_prepack_bytes() bytes). One launch
 *     on `stream`; the inputs may be freed once it completed.
 *   wna16_fused_moe_prepacked: wna16_fused_moe on packed w13 and w2 (both made
 *     with the same bits, group_size and zero-point presence, has_zeros = 1 if
 *     they carry zero points). Same workspace size, errors and semantics;
 *     `events` as in wna16_fused_moe_timed (may be NULL).
 */
size_t wna16_prepack_bytes(int E, int64_t N, int64_t K, int bits, int group_size, int has_zeros, int gate_up);
wna16_status wna16_prepack(const int32_t* q, const void* scales, const int32_t* zeros, int E, int64_t N,
                           int64_t K, int bits, int group_size, int gate_up, void* dst, void* stream);
wna16_status wna16_fused_moe_prepacked(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                       int64_t I, int E, int topk, const void* w13_packed,
                                       const void* w2_packed, int has_zeros, wna16_dtype scale_dtype,
                                       int bits, int group_size, const int32_t* topk_ids,
                                       const float* topk_weights, void* out, void* workspace,
                                       size_t workspace_bytes, int block, int split_k, void* stream,
                                       void* const* events);

/*
 * Checkpoint conversion (vLLM PR #12185: the fused kernel's weight format "is
 * just compatible with gptq/awq" and accepts their weights after a one-off
 * conversion). The layouts are those of the public packers:
 *   WNA16_CKPT_GPTQ / _GPTQ_V2: qweight [E, K/pf, N] int32, the codes of
 *     column n packed along K (LSB first); qzeros [E, K/G, N/pf] packed along
 *     N, storing z - 1 (GPTQ) or z (GPTQ_V2); bits 4 or 8.
 *   WNA16_CKPT_AWQ: qweight [E, K, N/8] and qzeros [E, K/G, N/8], 4-bit, packed
 *     along N with field i of a word holding column 8c + (0 2 4 6 1 3 5 7)[i];
 *     zero points stored as they are.
 *   Scales [E, K/G, N] are the library's layout already (no conversion).
 * Outputs: q_out [E, N, K/pf] and zeros_out [E, K/G, N/pf] in the layout of
 * this header (qzeros and zeros_out both NULL for symmetric weights). For the
 * gate/up projection, N = 2I with the gate columns first (concatenate the
 * checkpoint's gate and up tensors along N before converting). group_size: as
 * in the layer calls, or -1. Argument errors return before any launch; the
 * conversion itself cannot fail on the device.
 */
typedef enum { WNA16_CKPT_GPTQ = 0, WNA16_CKPT_GPTQ_V2 = 1, WNA16_CKPT_AWQ = 2 } wna16_checkpoint;

wna16_status wna16_convert_checkpoint(wna16_checkpoint format, const int32_t* qweight, const int32_t* qzeros,
                                      int E, int64_t N, int64_t K, int bits, int group_size, int32_t* q_out,
                                      int32_t* zeros_out, void* stream);

/*
 * Model variants (vLLM fused_moe/oracle/int8.py: the int8 MoE quant config
 * carries w1_bias / w2_bias, and passes swiglu_alpha / swiglu_beta /
 * swiglu_limit to its clamped-SwiGLU backend; the pages give no formulas, these
 * are the readings implemented).
 *   w13_bias  [E, 2I] act_dtype (gate rows, then up rows) or NULL: added in
 *             fp32 to the gate/up GEMM output before the activation.
 *   w2_bias   [E, H] act_dtype or NULL: added in fp32 to the down GEMM output
 *             before the top-k weight (once per (token, slot), whatever the
 *             K split).
 *   activation WNA16_ACT_SILU: silu(g) * u (the default layer).
 *             WNA16_ACT_SWIGLU_CLAMP: g' * sigmoid(alpha * g') * (u' + beta)
 *             with g' = min(g, limit), u' = clamp(u, -limit, limit) when
 *             limit > 0 (no clamp otherwise); alpha and beta finite.
 *   w13_perm  [E, H] int32 or NULL: act-order gate/up weights, repacked by
 *             wna16_act_order_prepare; entry i is the original hidden index
 *             of repacked column i (its `perm`). The layer reads each routed
 *             token row in this order.
 *   w2_inv_perm [E, I] int32 or NULL: act-order down weights, repacked;
 *             entry f is the repacked column of intermediate feature f (the
 *             prepare call's `inv_perm`).
 *             With either permutation the layer runs the general GEMM kernel
 *             (the 16-token deferred-scale kernel needs contiguous feature
 *             runs). Out-of-range entries are skipped, never dereferenced.
 *   router_logits [M, E] (logits_dtype) or NULL: route on the device first.
 *             The call runs wna16_topk_routing (scoring, renormalize,
 *             n_groups, topk_groups as there) into routed_ids [M, topk] int32
 *             and routed_weights [M, topk] fp32 (both required, written), then
 *             the layer on them; the topk_ids / topk_weights arguments are then
 *             ignored and may be NULL. Routing argument errors return before
 *             any launch. Batches of up to 128 tokens are routed and aligned by
 *             one launch (five launches in all); larger ones run the routing
 *             launch before the layer's five. The timed variant's first event
 *             is recorded before the align launch (routing included when fused).
 *   atomic_reduce (vLLM PR #14138's use_atomic_add, for comparison): != 0
 *             makes the down GEMM add each (token, slot) row, already scaled
 *             by its top-k weight, into an fp32 [M, H] accumulator with
 *             atomicAdd (all slots and K splits of a token into one row; the
 *             addition order, and so the last bits, varies from run to run),
 *             and the last launch only rounds it. The default (0) writes each
 *             row once to its own place and adds them in slot order (the
 *             result is reproducible). Not combined with act-order weights.
 * A zero-initialized struct (or a NULL pointer) is the default layer. Both
 * bias pointers must be aligned to their 2-byte elements, the permutations to
 * 4 bytes.
 */
typedef enum { WNA16_ACT_SILU = 0, WNA16_ACT_SWIGLU_CLAMP = 1 } wna16_activation;

typedef struct {
  const void* w13_bias;
  const void* w2_bias;
  wna16_activation activation;
  float swiglu_alpha;
  float swiglu_beta;
  float swiglu_limit;
  const int32_t* w13_perm;
  const int32_t* w2_inv_perm;
  const void* router_logits;
  wna16_dtype logits_dtype;
  wna16_scoring scoring;
  int renormalize;
  int n_groups;
  int topk_groups;
  int32_t* routed_ids;
  float* routed_weights;
  int atomic_reduce;
} wna16_moe_options;

/*
 * Act-order (GPTQ desc_act) weights: column k of expert e belongs to group
 * g_idx[e, k] (vLLM PR #14138 passes `g_idx` and `sort_indices` to the marlin
 * GEMM; empty in its benchmark). This call lists each expert's columns by
 * ascending group, ascending k within a group:
 *   perm     [E, K] int32 out: perm[e, i] = original column of column i;
 *   inv_perm [E, K] int32 out or NULL: inv_perm[e, perm[e, i]] = i;
 *   q_out    [E, N, K/pf] int32 out or NULL (then q must be NULL too): the codes
 *            of q [E, N, K/pf] (layout as in the header) with column i taken
 *            from column perm[e, i]. With group_size G, repacked column i is in
 *            group i / G, so q_out with the unchanged scales and zero points
 *            [E, K/G, ...] is a plain grouped matrix for the layer calls (and
 *            for wna16_prepack).
 *   g_idx    [E, K] int32. Every group must hold exactly G columns (as GPTQ
 *            writes them); otherwise WNA16_DEV_BAD_GROUPS is or-ed into
 *            *device_status (not reset by this call) and the outputs, though
 *            in range, are meaningless.
 * Pass perm as the gate/up GEMM's w13_perm (K = H) and inv_perm of the down
 * weights as w2_inv_perm (K = I) in wna16_moe_options. One-off conversion
 * (a CTA per expert scans its g_idx once per group): not a per-call step.
 */
wna16_status wna16_act_order_prepare(const int32_t* q, const int32_t* g_idx, int E, int64_t N, int64_t K,
                                     int bits, int group_size, int32_t* q_out, int32_t* perm, int32_t* inv_perm,
                                     int32_t* device_status, void* stream);

/*
 * wna16_fused_moe_timed / wna16_fused_moe_prepacked with model-variant
 * options (may be NULL). Same workspace size, errors and semantics; a bad
 * `options` field returns WNA16_ERR_INVALID_ARG before any launch.
 */
wna16_status wna16_fused_moe_ex(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I,
                                int E, int topk, const int32_t* w13_q, const void* w13_scales,
                                const int32_t* w13_zeros, const int32_t* w2_q, const void* w2_scales,
                                const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits, int group_size,
                                const int32_t* topk_ids, const float* topk_weights, void* out, void* workspace,
                                size_t workspace_bytes, int block, int split_k, void* stream,
                                void* const* events, const wna16_moe_options* options);
wna16_status wna16_fused_moe_prepacked_ex(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                          int64_t I, int E, int topk, const void* w13_packed,
                                          const void* w2_packed, int has_zeros, wna16_dtype scale_dtype, int bits,
                                          int group_size, const int32_t* topk_ids, const float* topk_weights,
                                          void* out, void* workspace, size_t workspace_bytes, int block,
                                          int split_k, void* stream, void* const* events,
                                          const wna16_moe_options* options);

/*
 * Synchronizes `stream`, then reads the device status word at the start of a
 * fused-call workspace (or any int32 status word the caller passed to the
 * align call, or wna16_act_order_prepare). Writes the raw bits to *bits_out
 * (may be NULL) and returns WNA16_OK, WNA16_ERR_DEVICE_TIMEOUT,
 * WNA16_ERR_DEVICE_BAD_EXPERT_ID or WNA16_ERR_DEVICE_BAD_GROUPS (in that order
 * of precedence), or WNA16_ERR_CUDA if the copy fails. For tests and debugging.
 */
wna16_status wna16_read_device_status(const void* status_word, int32_t* bits_out, void* stream);

/*
 * Failure-path self-check (diagnostics and tests): launches one CTA whose warps
 * wait, with the pipelines' own bounded wait, on barriers that nothing
 * completes. After the bound (about 2 s) the wait gives up, or-s
 * WNA16_DEV_TIMEOUT into *device_status (not reset here), and the CTA's other
 * waiting warp leaves through the abort flag; each waiting warp that left adds
 * 1 to *roles_left (optional, 2 when both did). Tensor memory the CTA held is
 * freed and the context stays usable. Asynchronous on `stream`.
 */
wna16_status wna16_check_wait_timeout(int32_t* device_status, int32_t* roles_left, void* stream);

/*
 * Host-only check of one fused call's launch plan (no GPU, no CUDA call):
 * builds the plan wna16_fused_moe would launch for these sizes on a device
 * with `sms` SMs (plain weight layout, default options), and replays every
 * role of every CTA of both GEMM launches, plus the gather and the combine,
 * through the kernels' own index expressions, on the given align output
 * (host arrays: topk_ids [M, topk], sorted_ids [cap], expert_ids [cap/block]
 * and num_tokens_post_padded, e.g. from a reference implementation of
 * moe_align_block_size with the same block). It checks that every TMA box lies
 * inside its tensor map with a 16-byte-aligned innermost coordinate, that a
 * stage's boxes add up to the bytes its barrier expects, that the work units
 * cover every (block, weight tile, K split) once, that tensor-memory and
 * shared-memory layouts fit and do not overlap, and that every global write
 * lands inside its workspace region, each routed pair's fp32 rows written once.
 * Returns the number of violations (0: all in bounds), or minus a
 * wna16_status for arguments the fused call would reject. The first few
 * violations are written, one per line, to `report` (may be NULL).
 */
int64_t wna16_check_launch_plan(int64_t M, int64_t H, int64_t I, int E, int topk, int bits, int group_size,
                                int has_zeros, wna16_dtype act_dtype, wna16_dtype scale_dtype, int block,
                                int split_k, int sms, const int32_t* topk_ids, const int32_t* sorted_ids,
                                const int32_t* expert_ids, int32_t num_tokens_post_padded, char* report,
                                size_t report_bytes);

/* Static, human-readable name of a status code. */
const char* wna16_status_string(wna16_status status);

#ifdef __cplusplus
}
#endif

#endif /* WNA16_MOE_H_ */
