/*
 * qmoe.h -- C ABI of the GB300 (sm_103a) weight-only FP4 mixture-of-experts
 * layer (QMoE, W4A16): top-k softmax routing, permute-by-expert, FC1 with
 * SwiGLU, FC2, weighted un-permute, and the FP4 -> bf16 weight dequantisation
 * used at prefill.
 *
 * The operation follows the pages' operator statement:
 *   "MoE and QMoE - CUDA Operator Documentation" §1 (pipeline: router top-k
 *   softmax -> permute by expert -> GEMM1 -> activation -> GEMM2 -> un-permute
 *   -> weighted sum), §2 (inputs: router probabilities, fc1/fc2 weights, block
 *   scales, global scales; attributes k, swiglu_fusion, activation_alpha/beta,
 *   swiglu_limit, normalize_routing_weights), §6.5 (packed [E, K, N/2] e2m1
 *   storage and W = fp4(W) * block_scale * global_scale), §8 (SwiGLU), §9b
 *   (NVFP4: E4M3 scale per 16 k and a per-expert fp32 global scale);
 *   "[CUDA] Coalesce QMoE MXFP4/NVFP4 weight dequantization" (the [E, K, N/2]
 *   -> [E, N, K] dequantisation);
 *   "[CUDA] Cut the MoE routing prologue/epilogue cost for small-batch decode"
 *   (stable top-k, renormalised weights, stable expert ranking).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never allocates, frees or keeps them.  bf16 tensors are passed as their
 *    16-bit patterns (uint16_t).
 *  - Packed FP4 weights: uint8 [E, K, N/2]; byte (e, k, j) holds logical
 *    element (n = 2j) in its low nibble and (n = 2j + 1) in its high nibble.
 *    E2M1 code: bit 3 sign, bits 2:0 select 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *  - Block scales: uint8 [E, N, K/bs]: E4M3FN with bs = 16 (QMOE_NVFP4) or
 *    E8M0 (bias 127, 0xFF = NaN) with bs = 32 (QMOE_MXFP4).  The forward
 *    entry points also take the k-major layout [E, K/bs, N] (the same bytes
 *    transposed per expert, written once by qmoe_fp4_scales_kmajor) when
 *    QMOE_SCALES_KMAJOR is OR'd into their format argument.
 *  - Global scales: fp32 [E]; NULL means 1.0 for every expert.
 *  - Weights, scales and activations must be 16-byte aligned
 *    (QMOE_ERR_MISALIGNED otherwise).
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream) and
 *    never synchronise.  Every argument is validated on the host before any
 *    launch; an invalid call launches nothing and returns a status != 0.
 *    A launch failure is reported as QMOE_ERR_CUDA (cudaGetLastError).
 *    qmoe_last_error() gives a one-line reason for the last failure on the
 *    calling host thread.
 *  - Scratch memory is a caller-provided device workspace.  Calling with
 *    workspace == NULL stores the required size in *workspace_bytes and
 *    returns QMOE_OK without launching.  The workspace needs no
 *    initialisation; its contents on return are unspecified.  Two calls that
 *    share one workspace must not run concurrently on the GPU.
 */
#ifndef QMOE_H_
#define QMOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMOE_OK = 0,
    QMOE_ERR_INVALID_ARG = 1,  /* NULL pointer, non-positive size, k > E, k > 8, ... */
    QMOE_ERR_MISALIGNED = 2,   /* a tensor pointer is not 16-byte aligned */
    QMOE_ERR_UNSUPPORTED = 3,  /* shape outside what the kernels cover */
    QMOE_ERR_WORKSPACE = 4,    /* *workspace_bytes smaller than required */
    QMOE_ERR_CUDA = 5,         /* a CUDA call or kernel launch failed */
    QMOE_ERR_DEVICE = 6        /* a bounded wait inside a kernel gave up (qmoe_check_device_error) */
} qmoe_status;

typedef enum {
    QMOE_NVFP4 = 0, /* E2M1 + E4M3FN scale per 16 k + fp32 global scale per expert */
    QMOE_MXFP4 = 1, /* E2M1 + E8M0 scale per 32 k (+ optional fp32 global scale) */
    /* Flag, OR'd into QMOE_NVFP4 or QMOE_MXFP4 for the forward entry points:
     * the block scales are k-major, [E, K/bs, N].  One scale window of the
     * decode kernel (16 or fewer consecutive blocks of a column tile) is then
     * one contiguous run of bytes per block row instead of N runs of <= 16
     * bytes, which is what lets it stream at full bandwidth. */
    QMOE_SCALES_KMAJOR = 0x100,
    /* Flag, OR'd into the format of qmoe_fp4_moe_forward: the workspace's
     * header (its first QMOE_WORKSPACE_HEADER_BYTES bytes) is already zero.
     * The caller zeroes it once (cudaMemsetAsync) when it sets the workspace
     * aside; after that the library keeps it zero: a decode call leaves it so
     * when its kernel returns (the last CTA out clears the counters) and the
     * prefill path never writes it.  With the flag a decode call launches its
     * kernel alone, without the per-call header reset, and with programmatic
     * dependent launch: the kernel may start on an SM while the previous
     * kernel of the stream is still finishing elsewhere, and waits until that
     * kernel's results are visible before it touches global memory.  Back-to-
     * back layers then pay no memset node and no full launch gap.  Header
     * word 1 (int32) is the device error flag (see qmoe_check_device_error):
     * any kernel of a forward call sets it to 1 when one of its bounded waits
     * gave up.  Only that word can become nonzero; it stays set until
     * qmoe_check_device_error reads and clears it. */
    QMOE_WORKSPACE_PRIMED = 0x200,
    /* Flag, OR'd with QMOE_SCALES_KMAJOR into the format of
     * qmoe_fp4_moe_forward: a decode call (T * k <= QMOE_GEMV_MAX_ROWS) runs
     * on the multi-row decode kernel whatever its size.  Without the flag the
     * kernel is chosen by the length of the weight stream: when one SM's share
     * of FC1 is under 16 units of 32 KB (e.g. 4 tokens, 256 experts, top-8,
     * hidden 2048, intermediate 512) the one-row-per-pass kernel runs, whose
     * stream starts sooner; longer streams run on the multi-row kernel, which
     * decodes every row of an expert in one pass over its weights and copies
     * column tiles as 2-D tensor copies.  Both give the layer within the same
     * tolerance; the flag exists so that either can be run on any shape. */
    QMOE_DECODE_MULTIROW = 0x400
} qmoe_fp4_format;

/* Bytes at the start of every forward workspace reserved for the decode
 * kernel's error flag and grid-barrier counters (see QMOE_WORKSPACE_PRIMED). */
#define QMOE_WORKSPACE_HEADER_BYTES 64

/* Largest number of expanded rows (T * k) the decode GEMV path takes; more rows
 * take the prefill path (tensor-core grouped GEMMs over the packed weights).
 * The window is the one PR #31159 sets for MTP verification
 * ("kMaxProfiledExpandedRows 8 -> 64"). */
#define QMOE_GEMV_MAX_ROWS 64

/*
 * qmoe_route_topk -- top-k softmax routing and permute-by-expert maps.
 * Operator doc §1 ("router (top-k softmax) -> permute by expert"); PR #31156
 * (warp top-k with a stable tie-break, renormalised weights, stable ranking of
 * the T*k assignments by expert).
 *
 *   logits           fp32 [T, E] router logits (router_probs): they select.
 *   router_weights   fp32 [T, E] mixing weights, or NULL (operator doc §2.3,
 *                    input 14: "DeepSeek-style routing", router_probs select
 *                    and router_weights, gathered at the selected experts,
 *                    mix).  NULL: the softmax of the logits mixes.  4-byte
 *                    aligned.
 *   T, E, k          tokens (>= 1), experts (1..256), experts per token (1..min(8, E)).
 *   normalize        0: weight = softmax over all E at the selected expert
 *                    (with router_weights: router_weights[t][expert]);
 *                    != 0: those k weights divided by their sum.
 *   topk_ids         int32 [T, k] out: selected experts per token, ordered by
 *                    (logit descending, expert index ascending).
 *   topk_weights     fp32 [T, k] out: routing weights in the same order.
 *   expert_offsets   int32 [E + 1] out: first permuted row of each expert;
 *                    expert_offsets[E] = T * k.
 *   perm_to_expanded int32 [T * k] out: expanded index (t * k + j) of each
 *                    permuted row; rows of one expert keep ascending expanded
 *                    index (stable).
 *   expanded_to_perm int32 [T * k] out: the inverse permutation.
 *   workspace, workspace_bytes: see the conventions above.
 * Selection is exact (made on the fp32 logits; -0.0 and +0.0 compare equal).
 * NaN logits are outside the contract.
 */
qmoe_status qmoe_route_topk(const float *logits, const float *router_weights, int T, int E, int k, int normalize,
                            int32_t *topk_ids, float *topk_weights,
                            int32_t *expert_offsets, int32_t *perm_to_expanded,
                            int32_t *expanded_to_perm,
                            void *workspace, size_t *workspace_bytes,
                            cudaStream_t stream);

/*
 * qmoe_fp4_moe_forward -- the whole MoE layer:
 *   out[t] = bf16( sum_j w[t][j] * FFN_{id[t][j]}(x[t]) ),
 *   FFN_e(x) = Wd2_e * bf16( SwiGLU( Wd1_e * x ) ),
 * with Wd the dequantised weights, fp32 accumulation, the SwiGLU of operator
 * doc §8 on the FC1 columns' (gate, linear) pairs:
 *   G = min(gate, limit); L = clamp(linear, -limit, limit);
 *   SwiGLU = G * sigmoid(alpha * G) * (L + beta)
 * (alpha = 1, beta = 0, limit = +inf is SiLU(gate) * linear).
 *
 *   x            bf16 [T, H] activations.
 *   logits       fp32 [T, E] router logits (routed as in qmoe_route_topk).
 *   router_weights fp32 [T, E] mixing weights gathered at the selected
 *                experts, or NULL (as in qmoe_route_topk).
 *   fc1_w        uint8 [E, H, I]  packed e2m1, K = H, N = 2I.
 *   fc1_s        uint8 [E, 2I, H/bs] block scales ([E, H/bs, 2I] with
 *                QMOE_SCALES_KMAJOR).
 *   fc1_g        fp32 [E] global scales, or NULL.
 *   fc2_w        uint8 [E, I, H/2] packed e2m1, K = I, N = H.
 *   fc2_s        uint8 [E, H, I/bs] block scales ([E, I/bs, H] with
 *                QMOE_SCALES_KMAJOR).
 *   fc2_g        fp32 [E] global scales, or NULL.
 *   fc1_wd       bf16 [E, 2I, H] already-dequantised FC1 weights, or NULL;
 *   fc2_wd       bf16 [E, H, I] already-dequantised FC2 weights, or NULL.
 *                (Used only when T * k > QMOE_GEMV_MAX_ROWS: an FC whose
 *                fc*_wd is given runs a bf16 grouped GEMM over it; one
 *                without runs the fused W4A16 GEMM over fc*_w / fc*_s, and
 *                with block scales as stored ([E, N, K/bs]) its scales are
 *                first rewritten k-major into the workspace, E * N * K / bs
 *                bytes more.  The fused FC1 also keeps x in expert order in
 *                the workspace, T * k * H bf16 values.)
 *   fmt          QMOE_NVFP4 or QMOE_MXFP4, optionally | QMOE_SCALES_KMAJOR
 *                (both FCs' block scales in the k-major layout).  The result
 *                does not depend on the layout beyond the order of the fp32
 *                partial sums (the two layouts may tile N differently).
 *   T, H, I, E, k  sizes: T >= 1; H, I multiples of 64; 1 <= E <= 256;
 *                1 <= k <= min(8, E).
 *   normalize    as in qmoe_route_topk.
 *   swiglu_fusion  where FC1's 2I columns hold the pairs (operator doc §8):
 *                1 interleaved, 2m = gate and 2m + 1 = linear; 2
 *                concatenated, m = gate and I + m = linear (fc1 (gate) and
 *                fc3 (value) fused offline); 0 is read as 1, the operator's
 *                backward-compatibility remap for QMoE.  Other values:
 *                QMOE_ERR_UNSUPPORTED.
 *   alpha, beta, limit  SwiGLU parameters (limit may be +inf).
 *   out          bf16 [T, H] result.
 *   topk_ids_out int32 [T, k] selected experts, or NULL.
 *   workspace, workspace_bytes: see the conventions above.
 * T * k <= QMOE_GEMV_MAX_ROWS runs the decode path: one persistent kernel for
 * routing, FC1, SwiGLU, FC2 and the un-permute, dequantising in registers
 * (after a memset of the workspace header, unless fmt carries
 * QMOE_WORKSPACE_PRIMED).  Its top-k is the code of qmoe_route_topk, so the
 * selected experts are identical.
 * The decode kernel is a cooperative launch of one CTA per SM:
 * it needs the whole GPU's residency and returns QMOE_ERR_CUDA if another
 * context keeps it from launching.  Larger T * k runs the prefill path
 * (operator doc §1 pipeline, §4.3, §9b): routing, then per FC a grouped GEMM
 * on the tensor cores with fp32 accumulation -- over the packed weights,
 * decoded to bf16 (e2m1 * block scale, exact) inside the GEMM with the global
 * scale applied to the accumulator, or over the caller's fc*_wd -- with the
 * gather folded into the first GEMM and the SwiGLU into its epilogue (the
 * activation rounded to bf16), and the weighted un-permute.  Numerically the
 * paths agree within the tolerance of fp32 accumulation, not bit for bit.
 */
qmoe_status qmoe_fp4_moe_forward(const uint16_t *x, const float *logits, const float *router_weights,
                                 const uint8_t *fc1_w, const uint8_t *fc1_s, const float *fc1_g,
                                 const uint8_t *fc2_w, const uint8_t *fc2_s, const float *fc2_g,
                                 const uint16_t *fc1_wd, const uint16_t *fc2_wd,
                                 qmoe_fp4_format fmt, int T, int H, int I, int E, int k,
                                 int normalize, int swiglu_fusion,
                                 float alpha, float beta, float limit,
                                 uint16_t *out, int32_t *topk_ids_out,
                                 void *workspace, size_t *workspace_bytes,
                                 cudaStream_t stream);

/*
 * qmoe_fp4_dequant -- FP4 -> bf16 weight dequantisation (PR #31349; operator
 * doc §4.3, §6.5, §9b):
 *   out[e][n][k] = bf16_rne( e2m1(nibble(packed[e][k][n/2], n % 2))
 *                            * scale(block_scales[e][n][k/bs]) * global_scale[e] )
 * with the product taken exactly and rounded once (round to nearest even);
 * a NaN scale gives the bf16 NaN 0x7FC0.
 *
 *   packed        uint8 [E, K, N/2].
 *   block_scales  uint8 [E, N, K/bs].
 *   global_scale  fp32 [E], or NULL (1.0).
 *   E, N, K       E >= 1; N a multiple of 64; K a multiple of 64.
 *   fmt           QMOE_NVFP4 or QMOE_MXFP4 (block scales in the [E, N, K/bs]
 *                 layout; QMOE_SCALES_KMAJOR is QMOE_ERR_UNSUPPORTED here).
 *   out           bf16 [E, N, K].
 * Needs no workspace.
 */
qmoe_status qmoe_fp4_dequant(const uint8_t *packed, const uint8_t *block_scales,
                             const float *global_scale, int E, int N, int K,
                             qmoe_fp4_format fmt, uint16_t *out, cudaStream_t stream);

/*
 * qmoe_fp4_scales_kmajor -- block scales [E, N, K/bs] -> k-major [E, K/bs, N]:
 *   out[e][b][n] = block_scales[e][n][b]   (bytes copied unchanged).
 * A weight-load-time preparation step for the forward entry points
 * (QMOE_SCALES_KMAJOR); the pages store scales row-major per output column
 * (operator doc §6.5, §9b), and this is the same data transposed per expert.
 *
 *   block_scales  uint8 [E, N, K/bs], 16-byte aligned.
 *   E, N, K       E >= 1; N a multiple of 64; K a multiple of 64.
 *   fmt           QMOE_NVFP4 (bs = 16) or QMOE_MXFP4 (bs = 32).
 *   out           uint8 [E, K/bs, N], 16-byte aligned; must not overlap the
 *                 input.
 * Needs no workspace.  Asynchronous on `stream`.
 */
qmoe_status qmoe_fp4_scales_kmajor(const uint8_t *block_scales, int E, int N, int K,
                                   qmoe_fp4_format fmt, uint8_t *out, cudaStream_t stream);

/*
 * qmoe_fp4_moe_forward_no_alloc -- the same layer as qmoe_fp4_moe_forward for
 * callers that cannot allocate device memory.  The pages have no counterpart
 * to this entry point; it exists for callers such as a plug-in that runs inside
 * another engine's memory pool and only receives its input and output buffers,
 * or a latency-critical loop in which a cudaMalloc (it can stall the whole
 * device) is not allowed.
 *
 * Scratch comes from a device array inside the library of
 * QMOE_NO_ALLOC_SCRATCH_BYTES bytes, which every GPU that loads the library
 * holds until the process exits.  The caller still passes all inputs and
 * outputs; arguments, results and errors are those of qmoe_fp4_moe_forward
 * (without fc*_wd, workspace and workspace_bytes).  Sizes whose scratch need
 * exceeds QMOE_NO_ALLOC_SCRATCH_BYTES are rejected with QMOE_ERR_WORKSPACE
 * before anything is launched.  No cudaMalloc, cudaFree or other allocating
 * routine is called.
 *  - The first call on a device looks up the array's device address there
 *    (cudaGetSymbolAddress); make that first call before any stream capture.
 *  - Every call, on any stream or host thread, uses the same array, which keeps
 *    the last call's contents: calls that overlap on the GPU race and corrupt
 *    each other's results.  Order them (one stream, or events).
 *  - The array starts at zero.  The counters in its header
 *    (QMOE_WORKSPACE_HEADER_BYTES) are back at zero whenever a call returns
 *    (see QMOE_WORKSPACE_PRIMED), so every call runs as a primed one: no
 *    per-call reset, programmatic dependent launch.  The header's error flag
 *    is the one exception: qmoe_check_device_error(NULL, stream) reads and
 *    clears it.
 */
#define QMOE_NO_ALLOC_SCRATCH_BYTES ((size_t)32 << 20)

qmoe_status qmoe_fp4_moe_forward_no_alloc(const uint16_t *x, const float *logits,
                                          const uint8_t *fc1_w, const uint8_t *fc1_s,
                                          const float *fc1_g, const uint8_t *fc2_w,
                                          const uint8_t *fc2_s, const float *fc2_g,
                                          qmoe_fp4_format fmt, int T, int H, int I, int E, int k,
                                          int normalize, int swiglu_fusion,
                                          float alpha, float beta, float limit,
                                          uint16_t *out, int32_t *topk_ids_out,
                                          cudaStream_t stream);

/*
 * qmoe_check_device_error -- read and clear the device error flag of a
 * forward workspace.  Every wait inside the library's kernels is bounded (a
 * kernel never hangs the GPU): a wait that gives up sets word 1 of the
 * workspace header to 1 and the kernel returns early, so the outputs of that
 * call (and of later calls on the same workspace until the flag is cleared)
 * are not to be trusted.  The flag is never set by a call that ran normally.
 *
 *   workspace  the workspace passed to qmoe_fp4_moe_forward, or NULL for the
 *              static scratch of qmoe_fp4_moe_forward_no_alloc on the
 *              current device.
 *   stream     the stream of the calls to check.
 * Synchronises `stream`, reads the flag (a 4-byte device-to-host copy) and,
 * when it is set, resets it to 0 (a 4-byte memset on `stream`, then a
 * synchronisation) and returns QMOE_ERR_DEVICE; otherwise returns QMOE_OK.
 * A call without QMOE_WORKSPACE_PRIMED resets the flag with the rest of the
 * header before it launches, so check before the next such call on the same
 * workspace.  Allocates nothing.
 */
qmoe_status qmoe_check_device_error(void *workspace, cudaStream_t stream);

/* Diagnostics: the binary version (compute capability x 10 + minor, 103 for
 * sm_103a) of the decode kernel as the CUDA runtime reports it on the current
 * device (cudaFuncGetAttributes), or -1 when the query fails (no device, or
 * no image for it). */
int qmoe_binary_version(void);

/* One-line description of the last failed call on this host thread ("" if none). */
const char *qmoe_last_error(void);

/*
 * Instrumentation (benchmarks): when `events` is non-NULL, every later
 * qmoe_fp4_moe_forward call records events[0] on its stream before its first
 * kernel and events[i] after its i-th kernel, for i < n_events.  The events
 * are created by the caller (cudaEventCreate) and must outlive the calls.
 * Pass NULL to switch it off.  Process-wide setting; not thread-safe.
 * Returns the number of kernels one forward call launches for decode shapes
 * (one: the fused routing + FC1 + FC2 + un-permute kernel, after a memset of
 * the workspace header unless QMOE_WORKSPACE_PRIMED), i.e. how many events
 * after the first are used.  Prefill shapes record six points: events[0]
 * before routing, [1] after routing, [2] after the block-scale rewrites (if
 * any), [3] after the FC1 GEMM, [4] after the FC2 GEMM, [5] after the
 * un-permute.
 */
int qmoe_set_stage_events(cudaEvent_t *events, int n_events);

#ifdef __cplusplus
}
#endif
#endif /* QMOE_H_ */
