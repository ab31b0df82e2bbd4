/*
 * moe_lora.h -- C ABI of the GB300 (sm_103a) multi-adapter LoRA MoE expert layer.
 *
 * The layer (sglang PR #14105 page, "LoRA on MoE expert layers", section
 * 实现拆解, FusedMoEWithLoRA formula), per token t with adapter l = mapping[t]:
 *
 *   y_t = sum_k w[t,k] * (W_down,e + s_l B_d A_d) [ SiLU((W_gate,e + s_l B_g A_g) x_t)
 *                                                   (.) ((W_up,e + s_l B_u A_u) x_t) ]
 *
 * with e = topk_ids[t,k], s_l = alpha_l / r_l, and the adapter used iff l >= 0
 * and r_l > 0.  The per-batch adapter metadata follows the sglang PR #24160
 * page ("shared MoE LoRA batch info", sections 实现拆解 and 关键源码片段:
 * MoELoRABatchInfo and test_moe_lora_info.py).
 *
 * Conventions for every call:
 *   - Array pointers are DEVICE memory owned by the caller unless a comment
 *     says otherwise.  The library never allocates device memory: scratch is the
 *     caller's `workspace` of at least the size the matching *_workspace_bytes()
 *     query returns, 256-byte aligned.
 *   - `stream` is a cudaStream_t passed as void*.  Every call only enqueues work
 *     on it and never synchronises the device or the stream.
 *   - The return value is a host-detected status (MLR_OK or a negative
 *     MLR_ERR_*).  On an error return nothing was enqueued.
 *   - `d_status` (nullable, device int32) receives device-detected errors as
 *     OR-ed MLR_STATUS_* bits; the library never clears it (the caller zeroes it).
 *     Kernels never trap: on bad input they set a bit, skip the offending
 *     element and keep every write inside the caller's buffers.
 *   - bf16 operands are passed as their 16-bit patterns (mlr_bf16).
 *   - All int32 ids; pair index p = t*topk + k for token t and slot k.
 */
#ifndef MOE_LORA_H_
#define MOE_LORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host return codes */
#define MLR_OK 0
#define MLR_ERR_INVALID (-1)      /* bad scalar argument or null pointer          */
#define MLR_ERR_UNDERCOVERED (-2) /* bs * max_len < num_tokens ("under-covers")   */
#define MLR_ERR_INDEX (-3)        /* an id outside its range (host-visible cases)  */
#define MLR_ERR_CAPACITY (-4)     /* output capacity or workspace too small        */
#define MLR_ERR_CUDA (-5)         /* a CUDA launch or driver call failed           */
#define MLR_ERR_TIMEOUT (-6)      /* reserved: device wait timed out (see status)  */
#define MLR_ERR_UNSUPPORTED (-8)  /* shape outside what the kernels implement      */

/* device status bits, OR-ed into *d_status */
#define MLR_STATUS_BAD_INDPTR 0x01   /* seg_indptr not 0..num_tokens non-decreasing    */
#define MLR_STATUS_UNDERCOVERED 0x02 /* a segment is longer than max_len               */
#define MLR_STATUS_INDEX 0x04        /* adapter or expert id out of range (skipped)     */
#define MLR_STATUS_CAPACITY 0x08     /* padded length exceeded capacity (truncated)     */
#define MLR_STATUS_TIMEOUT 0x10      /* a pipeline wait gave up; results are invalid    */
#define MLR_STATUS_RANK 0x20         /* lora_ranks[l] outside [0, max_rank]             */

typedef uint16_t mlr_bf16; /* bfloat16 bit pattern */

/* Library version string (static storage). */
const char* moe_lora_version(void);

/* Human-readable text for an MLR_OK / MLR_ERR_* code (static storage). */
const char* moe_lora_status_string(int code);

/*
 * moe_lora_batch_info -- once per batch, expand request segments into the
 * per-token adapter map and the per-slot enabled mask.
 * Source: sglang PR #24160 page, 实现拆解 items 1-3 (MoELoRABatchInfo fields,
 * _compute_moe_lora_info computed once per batch) and 关键源码片段
 * (test_compute_moe_lora_info_expands_segments / ..._rejects_undercovered_launch).
 *
 *   seg_indptr[bs+1]      request segment offsets, 0 = seg_indptr[0] <= ... <= seg_indptr[bs] = num_tokens
 *   weight_indices[bs]    adapter slot of each request, in [-1, num_loras); -1 = no adapter
 *   lora_ranks[num_loras] rank of each slot (0 = slot holds no adapter)
 *   max_len               0: no hint.  > 0: the longest segment the caller promises;
 *                         bs * max_len < num_tokens returns MLR_ERR_UNDERCOVERED (host),
 *                         a longer segment sets MLR_STATUS_UNDERCOVERED (device)
 *   token_lora_mapping    out [>= num_tokens]: weight_indices of the token's request.
 *                         Entries at and beyond num_tokens are never written.
 *   adapter_enabled       out [num_loras]: 1 iff some request uses the slot and its rank
 *                         is > 0, else 0 (every entry written; -1 requests are skipped)
 * Limits: 0 <= bs, num_tokens < 2^31; 0 <= num_loras <= 65536.
 */
int moe_lora_batch_info(const int32_t* seg_indptr, const int32_t* weight_indices,
                        const int32_t* lora_ranks, int32_t bs, int32_t num_loras,
                        int32_t num_tokens, int32_t max_len, int32_t* token_lora_mapping,
                        int32_t* adapter_enabled, int32_t* d_status, void* stream);

/*
 * moe_lora_align_capacity -- length the sorted_token_ids buffer must have:
 * roundup(P + min(P, E*(L+1)) * (block_size-1), block_size) with P = num_tokens*topk.
 * The block arrays need capacity / block_size entries.  Returns -1 on bad sizes.
 */
int64_t moe_lora_align_capacity(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                int32_t num_loras, int32_t block_size);

/* Scratch bytes moe_lora_align needs for these sizes (0 on bad sizes). */
size_t moe_lora_align_workspace_bytes(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                      int32_t num_loras, int32_t block_size);

/*
 * moe_lora_align -- per layer, bucket the (token, slot) pairs by (expert, adapter).
 * Source: sglang PR #14105 page, 实现拆解 (moe_lora_align_block_size: sorts tokens by
 * LoRA adapter and expert id; padded to block_size).
 *
 * Order: key(p) = e*(L+1) + (lora(t)+1) with e = topk_ids[p], lora(t) =
 * token_lora_mapping[t] in [-1, L): expert-major, "no adapter" first inside an
 * expert, then adapters by id; inside a bucket pairs keep ascending p (stable).
 * Each non-empty bucket is padded to a multiple of block_size with the sentinel P.
 *
 *   topk_ids[T*K], token_lora_mapping[T]        inputs
 *   sorted_token_ids[capacity]                  out: pair ids, pads = P; valid prefix
 *                                               [0, *num_tokens_post_pad)
 *   block_expert_ids, block_lora_ids[capacity/block_size]
 *                                               out: expert and adapter (-1 = none) of
 *                                               each block of the valid prefix
 *   num_tokens_post_pad[1]                      out (device)
 * Ids out of range set MLR_STATUS_INDEX and the pair is dropped; a padded length
 * above capacity sets MLR_STATUS_CAPACITY and writes stop at capacity.
 * Limits: T*K < 2^31, E*(L+1) <= 40960, 1 <= block_size <= 4096.
 */
int moe_lora_align(const int32_t* topk_ids, const int32_t* token_lora_mapping,
                   int32_t num_tokens, int32_t topk, int32_t num_experts, int32_t num_loras,
                   int32_t block_size, int32_t* sorted_token_ids, int32_t* block_expert_ids,
                   int32_t* block_lora_ids, int32_t* num_tokens_post_pad, int64_t capacity,
                   void* workspace, size_t ws_bytes, int32_t* d_status, void* stream);

/*
 * moe_lora_align_noalloc -- moe_lora_align for callers that cannot allocate
 * device memory (an engine that owns all GPU memory through its own pools and
 * forbids later allocations, a latency-critical path where cudaMalloc/cudaFree
 * may synchronise the device, a layer given no allocator).  The pages have no
 * counterpart: this is an addition of this library.
 *
 * Same arguments, results and device status bits as moe_lora_align, minus the
 * workspace.  The scratch is one fixed 4 MiB array inside the library's device
 * image (held on every GPU that loads the library until the process exits);
 * sizes whose align scratch exceeds it (moe_lora_align_workspace_bytes(...) >
 * 4 MiB, e.g. 1,048,576 tokens x top-8 over 256 experts x 65 adapter classes)
 * return MLR_ERR_CAPACITY before anything is enqueued -- use moe_lora_align with
 * a workspace there.  The call allocates nothing.
 * The first call on a device looks up the array's address on that device (the
 * current device, which must be the stream's); make that first call before
 * any stream capture.  The address is cached per device ordinal for the life of
 * the process: it assumes the device's primary context, so do not use this
 * call after cudaDeviceReset or under another driver-API context.  All calls share the one array, so calls whose work may
 * overlap on the GPU (different streams, or different host threads) race and
 * corrupt each other's results; calls ordered on one stream are safe, and no
 * clearing is needed between them.
 */
int moe_lora_align_noalloc(const int32_t* topk_ids, const int32_t* token_lora_mapping,
                           int32_t num_tokens, int32_t topk, int32_t num_experts, int32_t num_loras,
                           int32_t block_size, int32_t* sorted_token_ids, int32_t* block_expert_ids,
                           int32_t* block_lora_ids, int32_t* num_tokens_post_pad, int64_t capacity,
                           int32_t* d_status, void* stream);

/* Scratch bytes fused_moe_lora_forward needs for these sizes (0 on bad sizes). */
size_t fused_moe_lora_workspace_bytes(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                      int32_t hidden, int32_t intermediate, int32_t num_loras,
                                      int32_t max_rank);

/*
 * fused_moe_lora_forward -- the LoRA MoE expert layer (formula at the top).
 * Source: sglang PR #14105 page, 实现拆解 (FusedMoEWithLoRA: LoRA after gate_up and
 * before down; align kernel; fused LoRA A/B kernel; 4-D stacks
 * [num_loras, num_experts, rank, dim]); the top-k weighted sum over experts.
 *
 *   x             bf16 [T, H]
 *   topk_ids      int32 [T, K] in [0, E);  topk_weights float [T, K]
 *   token_lora_mapping int32 [T] in [-1, L) (from moe_lora_batch_info)
 *   lora_ranks    int32 [L] in [0, R];  scalings float [L] = alpha_l / r_l
 *   w_gate_up     bf16 [E, 2I, H]   rows 0..I-1 gate, rows I..2I-1 up
 *   w_down        bf16 [E, H, I]
 *   lora_a_gu     bf16 [L, E, 2, R, H]   [.., 0, ..] gate, [.., 1, ..] up
 *   lora_b_gu     bf16 [L, E, 2, I, R]
 *   lora_a_down   bf16 [L, E, R, I]
 *   lora_b_down   bf16 [L, E, H, R]
 *   y             bf16 [T, H] out
 * Stacks hold slot l's factors in the first r_l rank rows/columns; the rank
 * padding must be finite (the adapter pool keeps it zero).  Accumulation is
 * fp32; the gate/up activation and the LoRA intermediates are rounded to bf16.
 * Runs the align internally (block 16).  Requirements: H, I multiples of 8,
 * H >= 128, I >= 64, R a multiple of 16 in [16, 256] when L > 0,
 * E * (L + 1) <= 16384, every base pointer 16-byte aligned.  Sizes outside
 * these return MLR_ERR_UNSUPPORTED (and fused_moe_lora_workspace_bytes 0).
 * The top-k combine is set process-wide by moe_lora_set_deterministic (below):
 * fp32 atomic reductions, whose order (and so y's last bits) may differ
 * between runs, or per-pair rows summed in increasing k, bit-identical between
 * runs.
 */
int fused_moe_lora_forward(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                           const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                           const float* scalings, const mlr_bf16* w_gate_up,
                           const mlr_bf16* w_down, const mlr_bf16* lora_a_gu,
                           const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                           const mlr_bf16* lora_b_down, int32_t num_tokens, int32_t topk,
                           int32_t num_experts, int32_t hidden, int32_t intermediate,
                           int32_t num_loras, int32_t max_rank, mlr_bf16* y, void* workspace,
                           size_t ws_bytes, int32_t* d_status, void* stream);

/*
 * fused_moe_lora_forward_fp8 -- the same layer with FP8 base experts (sglang
 * PR #22323 page, 功能与动机 and 实现拆解 item 1: quantised MoE methods hand
 * their scales to the LoRA MoE layer, which then runs on quantised experts).
 *
 * The pages name the methods, not a format.  Here: w_gate_up_q [E, 2I, H]
 * and w_down_q [E, H, I] hold FP8 E4M3 codes (one byte each, same row order as
 * the bf16 weights).  w_gate_up_scale [E, ceil(2I/128), ceil(H/128)] and
 * w_down_scale [E, ceil(H/128), ceil(I/128)] are float32 scales.  Weight
 * (e, row, col) = value of its code x scale[e][row / 128][col / 128]: the
 * DeepSeek-V3 block-FP8 layout (128 x 128 blocks, inverse scales).  x, the
 * LoRA stacks and y stay bf16; only the base weights are quantised.  All
 * other arguments, the workspace (fused_moe_lora_workspace_bytes) and the
 * status behaviour are those of fused_moe_lora_forward.  Additional limits:
 * hidden and intermediate multiples of 16; the scale arrays non-null and
 * 4-byte aligned (else MLR_ERR_INVALID; sizes MLR_ERR_UNSUPPORTED).  Each
 * weight is dequantised to bf16 on chip (one rounding of code x scale), so
 * y matches the exact dequantised layer within the bf16 forward's tolerance.
 */
int fused_moe_lora_forward_fp8(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                               const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                               const float* scalings, const uint8_t* w_gate_up_q,
                               const float* w_gate_up_scale, const uint8_t* w_down_q,
                               const float* w_down_scale, const mlr_bf16* lora_a_gu,
                               const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                               const mlr_bf16* lora_b_down, int32_t num_tokens, int32_t topk,
                               int32_t num_experts, int32_t hidden, int32_t intermediate,
                               int32_t num_loras, int32_t max_rank, mlr_bf16* y, void* workspace,
                               size_t ws_bytes, int32_t* d_status, void* stream);

/*
 * fused_moe_lora_forward_int8 -- the same layer with block-wise INT8 base
 * experts (sglang PR #22323 page, 功能与动机 and 实现拆解 item 1: the INT8
 * method, blockwise_int8, among those that hand their scales to the LoRA MoE
 * layer).  w_gate_up_q [E, 2I, H] and w_down_q [E, H, I] hold two's-complement
 * int8 codes; the scale arrays and their 128 x 128 blocks are laid out as for
 * fused_moe_lora_forward_fp8; weight = code x scale.  Everything else, the
 * workspace and the limits are those of fused_moe_lora_forward_fp8.
 */
int fused_moe_lora_forward_int8(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                                const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                                const float* scalings, const int8_t* w_gate_up_q,
                                const float* w_gate_up_scale, const int8_t* w_down_q,
                                const float* w_down_scale, const mlr_bf16* lora_a_gu,
                                const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                                const mlr_bf16* lora_b_down, int32_t num_tokens, int32_t topk,
                                int32_t num_experts, int32_t hidden, int32_t intermediate,
                                int32_t num_loras, int32_t max_rank, mlr_bf16* y, void* workspace,
                                size_t ws_bytes, int32_t* d_status, void* stream);

/*
 * fused_moe_lora_forward_w4a16 -- the same layer with 4-bit base experts and
 * bf16 activations (the page's WNA16 method).  The pages name the method only;
 * the format here: w_gate_up_q [E, 2I, H/2] and w_down_q [E, H, I/2] hold two
 * UINT4 codes per byte along a row (the even column in the low nibble);
 * w_gate_up_scale (float) and w_gate_up_zero (uint8, 0..15) are
 * [E, 2I, ceil(H/128)], w_down_scale and w_down_zero [E, H, ceil(I/128)]: one
 * scale and zero point per row and group of 128 input columns;
 * weight = (code - zero) x scale.  Additional limits: hidden and intermediate
 * multiples of 32 (else MLR_ERR_UNSUPPORTED); scale arrays 4-byte aligned and
 * every quantisation array non-null (else MLR_ERR_INVALID).  Everything else
 * as fused_moe_lora_forward_fp8.
 */
int fused_moe_lora_forward_w4a16(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                                 const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                                 const float* scalings, const uint8_t* w_gate_up_q,
                                 const float* w_gate_up_scale, const uint8_t* w_gate_up_zero,
                                 const uint8_t* w_down_q, const float* w_down_scale,
                                 const uint8_t* w_down_zero, const mlr_bf16* lora_a_gu,
                                 const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                                 const mlr_bf16* lora_b_down, int32_t num_tokens, int32_t topk,
                                 int32_t num_experts, int32_t hidden, int32_t intermediate,
                                 int32_t num_loras, int32_t max_rank, mlr_bf16* y, void* workspace,
                                 size_t ws_bytes, int32_t* d_status, void* stream);

/* Scratch bytes fused_moe_lora_forward_fp8_w8a8 needs for these sizes (0 on bad
 * sizes): fused_moe_lora_workspace_bytes plus the quantised activations. */
size_t fused_moe_lora_workspace_bytes_fp8_w8a8(int32_t num_tokens, int32_t topk, int32_t num_experts,
                                              int32_t hidden, int32_t intermediate, int32_t num_loras,
                                              int32_t max_rank);

/*
 * fused_moe_lora_forward_fp8_w8a8 -- the layer on the FP8 tensor cores (sglang
 * PR #22323 page, 功能与动机 and 实现拆解 item 1 name the FP8 method; the
 * format is a reading): both base GEMMs multiply E4M3 weights by E4M3
 * activations with power-of-two block scales, accumulating in fp32.
 *
 *   w_gate_up_q   uint8 [E, 2I, H]  E4M3 codes;  w_down_q uint8 [E, H, I]
 *   w_gate_up_exp uint8 [E, ceil(2I/128), ceil(H/128)]  biased exponent e of
 *                 each 128 x 128 block: weight = code value x 2^(e - 127)
 *   w_down_exp    uint8 [E, ceil(H/128), ceil(I/128)]
 * Exponent bytes must be below 255.  The activations that feed the base GEMMs
 * are quantised on the way, per token (pair) and group of 128 channels: scale
 * 2^s with s the smallest integer such that max|group| x 2^-s <= 448
 * (clamped to [-127, 127]; 0 for an all-zero group), each value rounded to
 * the nearest E4M3 value, ties to even.  x is quantised from its bf16 value,
 * the gate_up output SiLU(g) * u after its rounding to bf16.  The LoRA
 * shrinks read the unquantised bf16 x and gate_up output; LoRA stacks, y and
 * every other argument are those of fused_moe_lora_forward, except the
 * workspace size (fused_moe_lora_workspace_bytes_fp8_w8a8).  Additional
 * limits: hidden and intermediate multiples of 16; both exponent arrays
 * non-null (else MLR_ERR_INVALID).
 */
int fused_moe_lora_forward_fp8_w8a8(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                                    const int32_t* token_lora_mapping, const int32_t* lora_ranks,
                                    const float* scalings, const uint8_t* w_gate_up_q,
                                    const uint8_t* w_gate_up_exp, const uint8_t* w_down_q,
                                    const uint8_t* w_down_exp, const mlr_bf16* lora_a_gu,
                                    const mlr_bf16* lora_b_gu, const mlr_bf16* lora_a_down,
                                    const mlr_bf16* lora_b_down, int32_t num_tokens, int32_t topk,
                                    int32_t num_experts, int32_t hidden, int32_t intermediate,
                                    int32_t num_loras, int32_t max_rank, mlr_bf16* y, void* workspace,
                                    size_t ws_bytes, int32_t* d_status, void* stream);

/* Scratch bytes lora_linear_forward needs for these sizes (0 on bad sizes). */
size_t lora_linear_workspace_bytes(int32_t num_tokens, int32_t in_features, int32_t out_features,
                                   int32_t num_loras, int32_t max_rank, int32_t num_slices);

/*
 * lora_linear_forward -- a dense projection with per-segment LoRA and a split B.
 * Source: sglang PR #22323 page (LoRA quantisation info and the DeepSeek-V3 MLA
 * fused projection), section 实现拆解 items 2-3: ReplicatedLinearWithLoRA applies
 * LoRA to the fused q_a_proj + kv_a_proj_with_mqa projection, whose output rows
 * hold two parts of unequal width; the LoRA B is split into the two parts and
 * each part is applied by its own segment GEMM to its own LoRA A's shrink.
 *
 * The output rows are split into S parts at slice_offsets; for token t with
 * adapter l = token_lora_mapping[t] (used iff l >= 0 and r_l > 0) and row o in
 * part s:
 *   y[t][o] = sum_i w[o][i] x[t][i] + s_l * sum_{q < r_l} lora_b[l][o][q] * z_s[q],
 *   z_s[q]  = sum_i lora_a[l][s][q][i] x[t][i].
 *
 *   x             bf16 [T, D_in]
 *   w             bf16 [D_out, D_in]
 *   token_lora_mapping int32 [T] in [-1, L) (from moe_lora_batch_info)
 *   lora_ranks    int32 [L] in [0, R];  scalings float [L] = alpha_l / r_l
 *   lora_a        bf16 [L, S, R, D_in]   part s's A
 *   lora_b        bf16 [L, D_out, R]     rows of part s multiply part s's z
 *   slice_offsets HOST int32 [S + 1]: 0 = offsets[0] < ... < offsets[S] = D_out
 *   y             bf16 [T, D_out] out
 * Requirements: S = 1 or 2; with S = 2 the second part starts on a multiple of
 * 256 rows (the MLA projection: 1536 + 576); D_in, D_out multiples of 8 and
 * >= 128; R a multiple of 16 in [16, 256] when L > 0; L + 1 <= 16384; every base
 * pointer 16-byte aligned.  Bad offsets return MLR_ERR_INVALID, other sizes
 * outside these MLR_ERR_UNSUPPORTED (and lora_linear_workspace_bytes 0).
 * Accumulation is fp32 and the LoRA intermediate z is rounded to bf16.  The
 * profile stages (see below) of this call are "align_plan", "gather",
 * "shrink_gate_up" (the shrink), "down" (the projection) and "convert".
 */
int lora_linear_forward(const mlr_bf16* x, const mlr_bf16* w, const int32_t* token_lora_mapping,
                        const int32_t* lora_ranks, const float* scalings, const mlr_bf16* lora_a,
                        const mlr_bf16* lora_b, const int32_t* slice_offsets, int32_t num_tokens,
                        int32_t in_features, int32_t out_features, int32_t num_loras, int32_t max_rank,
                        int32_t num_slices, mlr_bf16* y, void* workspace, size_t ws_bytes,
                        int32_t* d_status, void* stream);

/*
 * lora_tp_qkv_b_rows -- the rows of a fused q/k/v projection's LoRA B (and of
 * its base weight) that tensor-parallel rank tp_rank holds (sglang PR #24420
 * page, 关键源码片段: mem_pool.py _column_parallel_lora_b_per_rank_dim and
 * layers.py slice_lora_b_weights).  B is stacked along its output rows as q
 * (num_heads * head_dim rows), then k and v (num_kv_heads * head_dim rows
 * each).  While tp_size <= num_kv_heads a rank takes an even 1/tp_size of each
 * block.  Beyond that, each KV head is replicated over tp_size / num_kv_heads
 * ranks, and a rank takes its 1/tp_size of q plus one whole head of k and of v
 * (the head of index tp_rank / replicas).
 *
 * Host only: no device memory, no stream.  ranges (host int32[6]) receives
 * [q_begin, q_end, k_begin, k_end, v_begin, v_end) as rows of the full B;
 * *per_rank_rows (nullable) = (q_end - q_begin) + (k_end - k_begin) +
 * (v_end - v_begin).  The rank's projection is lora_linear_forward on those
 * rows of W and B (one part).  Returns MLR_ERR_INVALID on a null ranges,
 * non-positive sizes, a rank outside [0, tp_size), num_heads not divisible by
 * tp_size, or tp_size and num_kv_heads neither dividing the other.
 */
int lora_tp_qkv_b_rows(int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t tp_size,
                       int32_t tp_rank, int32_t* ranges, int32_t* per_rank_rows);

/*
 * Observability.  The pages describe no tracing; these calls exist so that a
 * caller can attribute the forward's GPU time to its stages without a profiler.
 *
 * moe_lora_profile_begin(max_calls): the next max_calls (<= 4096) forward calls
 *   record a CUDA event on their stream between consecutive stages.  Returns
 *   MLR_ERR_CUDA if the events cannot be created.
 * moe_lora_profile_end(stage_ms, max_stages, n_stages, n_calls): blocks until the
 *   recorded events complete, writes the summed milliseconds of each stage over
 *   the recorded calls into stage_ms[0..min(max_stages, *n_stages)), the number of
 *   recorded calls into *n_calls (host pointers), and stops recording.
 * moe_lora_profile_stages(mask): stages that later moe_lora_profile_begin
 *   calls time (bit i = stage i; all stages by default).  Only the events that
 *   bound a selected stage are recorded, so timing one stage adds two events
 *   per call instead of eight; unselected stages report 0 ms.  Returns
 *   MLR_ERR_INVALID for an empty mask or bits past the last stage.
 * moe_lora_profile_stage_name(i): "align_plan" (the (expert, adapter) align in
 *   dense order and the tile plan), "gather" (x copied into sorted row order; zeroes the fp32
 *   accumulator), "shrink_gate_up", "gate_up", "shrink_down", "down", "convert"
 *   (static storage; NULL past the last stage).
 * moe_lora_launch_count(): kernels this library has launched in this process.
 */
/*
 * Expert parallelism (the multi-GPU form of the layer that the pages point to
 * in other PRs: the DeepEP dispatch among the sglang PR #22323 page's related
 * PRs, 关联脉络, and the TP/EP question of the sglang PR #14105 page's review,
 * 评论区精华).  The E experts are split over n_ranks ranks in equal contiguous
 * ranges: rank d owns experts [d*E/n_ranks, (d+1)*E/n_ranks).  One step on
 * every rank:
 *   1. moe_lora_ep_dispatch packs this rank's (token, slot) pairs by owner;
 *   2. the caller exchanges the packed rows with an all-to-all (send_counts
 *      rows to each rank; NCCL, or any transport: the library moves no data
 *      between GPUs);
 *   3. each owner runs fused_moe_lora_forward on the rows it received with
 *      top-1 routing (topk_ids = the received expert ids, topk_weights = the
 *      received weights, token_lora_mapping = the received adapters) over its
 *      own experts' weights and LoRA stacks [L, E/n_ranks, ...]: each output
 *      row is w * (expert output);
 *   4. the caller returns those rows with the reverse all-to-all, so this rank
 *      holds them in its send order;
 *   5. moe_lora_ep_combine sums each token's rows.
 *
 * moe_lora_ep_workspace_bytes(T, K, n_ranks): scratch of the dispatch (0 on
 *   bad sizes).  Limits: 1 <= n_ranks <= 64, T*K < 2^31.
 *
 * moe_lora_ep_dispatch: pair p = t*K + k with expert e in [0, E) goes to rank
 *   e / (E/n_ranks); the send order lists rank 0's pairs first, each rank's in
 *   increasing p.  Outputs (device, caller-owned, T*K rows of capacity):
 *     send_x      bf16 [T*K, H]: x row of the pair's token
 *     send_expert int32 [T*K]:   e - (first expert of the destination)
 *     send_weight float [T*K]:   topk_weights[p]
 *     send_lora   int32 [T*K]:   token_lora_mapping[t]
 *     send_counts int32 [n_ranks]: rows for each rank (rows [sum of earlier
 *                 counts, + count) of the send buffers)
 *     pair_pos    int32 [T*K]:   row of pair p in the send order, -1 if dropped
 *   A pair whose expert id is outside [0, E) is dropped and sets
 *   MLR_STATUS_INDEX.  Requirements: E a multiple of n_ranks, H a multiple of
 *   8, x and send_x 16-byte aligned; else MLR_ERR_INVALID (n_ranks above 64:
 *   MLR_ERR_UNSUPPORTED).
 *
 * moe_lora_ep_combine: y[t] = sum over k in increasing order of
 *   rows[pair_pos[t*K + k]] (skipping -1), in fp32, rounded to bf16: y is
 *   bit-identical between runs.  rows: bf16 [>= valid pairs, H], 16-byte
 *   aligned; y: bf16 [T, H].
 */
size_t moe_lora_ep_workspace_bytes(int32_t num_tokens, int32_t topk, int32_t n_ranks);
int moe_lora_ep_dispatch(const mlr_bf16* x, const int32_t* topk_ids, const float* topk_weights,
                         const int32_t* token_lora_mapping, int32_t num_tokens, int32_t topk, int32_t hidden,
                         int32_t num_experts, int32_t n_ranks, mlr_bf16* send_x, int32_t* send_expert,
                         float* send_weight, int32_t* send_lora, int32_t* send_counts, int32_t* pair_pos,
                         void* workspace, size_t ws_bytes, int32_t* d_status, void* stream);
int moe_lora_ep_combine(const mlr_bf16* rows, const int32_t* pair_pos, int32_t num_tokens, int32_t topk,
                        int32_t hidden, mlr_bf16* y, void* stream);

/*
 * Failure detection.  The pages describe none; every pipeline wait of the GEMM
 * kernels (a stage of operands to land, an accumulator to fill or drain) gives
 * up after a limit instead of spinning forever, sets MLR_STATUS_TIMEOUT in
 * d_status, and every role of the kernel then leaves, frees its TMEM and
 * returns, so the CUDA context stays usable.  Results of that call are invalid.
 *
 * moe_lora_set_wait_limit_ns(ns): the limit for launches enqueued from now on,
 *   process-wide (default 2 s; 0 is taken as 1 ns, so a wait that is not
 *   already satisfied gives up at once).  Returns MLR_ERR_INVALID above 60 s.
 *   Teardown waits (in-flight copies and MMAs before TMEM is freed) keep their
 *   own fixed 2 s limit.
 * moe_lora_wait_limit_ns(): the current limit.
 */
int moe_lora_set_wait_limit_ns(uint64_t ns);
uint64_t moe_lora_wait_limit_ns(void);

/*
 * The top-k combine of fused_moe_lora_forward(_fp8) (the weighted sum over a
 * token's K experts, named by the layer formula's sum over top-k; the pages
 * leave its order open).  Process-wide, for calls enqueued from now on;
 * deterministic (1) by default.
 *   on = 0: the down GEMM adds w * d into an fp32 accumulator with atomic
 *           reductions, in whatever order the pairs finish; y may differ in
 *           its last bits between runs.
 *   on = 1: the down GEMM writes w * d of each pair, rounded to bf16, into a
 *           row of its own (inside the workspace, no extra bytes), and a
 *           combine kernel sums a token's K rows in increasing k in fp32:
 *           y is bit-identical between runs.
 * Returns MLR_ERR_INVALID for other values.  moe_lora_deterministic() reads it.
 */
int moe_lora_set_deterministic(int32_t on);
int32_t moe_lora_deterministic(void);

int moe_lora_profile_stages(uint32_t mask);
int moe_lora_profile_begin(int32_t max_calls);
int moe_lora_profile_end(double* stage_ms, int32_t max_stages, int32_t* n_stages, int32_t* n_calls);
const char* moe_lora_profile_stage_name(int32_t stage);
uint64_t moe_lora_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LORA_H_ */
