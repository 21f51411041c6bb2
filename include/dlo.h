/*
 * dlo.h -- layerwise weight offload of a DiT block stack through two device
 * slots, for one GB300 (sm_103a).  C ABI of libdlo.so.
 *
 * Every block's weights live flattened in host memory (pinned, or registered
 * by this library).  Two device slots hold streamed blocks.  While streamed
 * block i computes on the caller's compute stream, the next block (block i+1,
 * or the first streamed block again after the last one) is copied into the
 * other slot on the caller's copy stream; CUDA events order slot reuse.  The
 * first k blocks may stay resident in caller-provided device buffers.
 *
 * Sources (vLLM-Omni documentation pages):
 *  [LW]  "CPU Offloading for Diffusion Models", section "Layerwise (Blockwise)
 *        Offloading": How It Works and the Execution Flow table.
 *  [DLO] "Distributed Layerwise Offload": Feature compatibility table,
 *        "Startup and runtime sequence", "Host backing and transfer
 *        composition", "Failure and lifecycle boundaries", "Registered
 *        runtime-cache transfer", "Rank-local path without DLO AllGather".
 *  [OFF] "CPU Offloading" (offloader design README): "Shared lifecycle",
 *        "Cross-strategy invariants".
 * The DiT block math is not on those pages; it is the standard DiT adaLN-zero
 * block and a video-DiT block (self-attention, cross-attention to text, FFN),
 * stated in full at dlo_forward.
 *
 * Conventions for every call:
 *  - Pointers named d_* (or documented as device) are device pointers of the
 *    context's device; host pointers are plain process addresses.
 *  - Streams are cudaStream_t passed as void*.
 *  - The caller owns every buffer it passes and keeps it alive until
 *    dlo_destroy returns.  The library owns only its events, the host ranges
 *    it registered itself, the two pinned host staging slots of
 *    DLO_HOST_PAGEABLE and the context object.
 *  - Calls are not thread-safe on one context.  Different contexts are
 *    independent.
 *  - Errors return a negative dlo_status; dlo_last_error() gives the message.
 *    Argument errors are detected before any state changes.
 */
#ifndef DLO_H
#define DLO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DLO_ABI_VERSION 3
#define DLO_MAX_CONTAINERS 64   /* block containers of one stack (dlo_create_multi) */

typedef int dlo_status;
#define DLO_OK            0
#define DLO_EINVAL       -1  /* bad argument; nothing changed                    */
#define DLO_ESTATE       -2  /* call out of lifecycle order; nothing changed     */
#define DLO_ENOMEM       -3  /* a caller buffer is too small                     */
#define DLO_ECUDA        -4  /* a CUDA runtime call failed (message has the code) */
#define DLO_EREGISTER    -5  /* host registration failed and was rolled back     */
#define DLO_ETIMEDOUT    -6  /* a bounded wait ran out (host or device side)     */
#define DLO_EUNSUPPORTED -7  /* valid but not implemented combination            */
#define DLO_EMISMATCH    -8  /* dlo_verify_slot: slot bytes differ from the host */

/* block kinds */
#define DLO_BLOCK_DIT    0   /* DiT adaLN-zero block, self-attention only        */
#define DLO_BLOCK_VIDEO  1   /* video-DiT block: self-attn, cross-attn, FFN      */
#define DLO_BLOCK_BYTES  2   /* opaque bytes; compute = checksum of the slot     */

/* weight storage of the linears in a block */
#define DLO_W_BF16       0
/* W8A16: e4m3 weights + one fp32 scale per linear tensor, streamed as codes
 * (half the bytes of bf16) and dequantised inside the GEMM kernel: widened
 * to exact bf16 values per weight tile in the mainloop, or, for linears with
 * at least DLO_WIDEN_ROWS rows (default 4096), once per launch by the
 * kernel's own CTAs before its mainloop; activations stay bf16 and the scale
 * multiplies the fp32 accumulator (y = s * (x q^T) + b). */
#define DLO_W_E4M3       1
/* W8A8: the DLO_W_E4M3 weights (same layout and bytes), and every linear's
 * input activation quantised to E4M3 on the fly with one dynamic per-tensor
 * scale (dlo_op_quantize_act); the product runs on the 8-bit tensor cores:
 * y = s_x * s_w * (q_x q_w^T) + b, fp32 accumulation. */
#define DLO_W_E4M3_A8    2

/* slot staging engine */
#define DLO_STAGE_MEMCPY 0   /* cudaMemcpyAsync on the copy stream (copy engine) */
#define DLO_STAGE_GATHER 1   /* SM kernel reading mapped host memory, 16-B loads */
/* one cudaMemcpyAsync per layout tensor, host offset -> the same slot offset
 * ("Distributed Layerwise Offload", Registered runtime-cache transfer: each
 * immutable tensor view is copied directly into its offset of the flattened
 * rotating device buffer; more copy operations than one packed block copy) */
#define DLO_STAGE_PER_TENSOR 2

/* host block flags for dlo_register_host_blocks */
#define DLO_HOST_PINNED   1u /* caller's memory is already page-locked           */
#define DLO_HOST_REGISTER 2u /* library page-locks it (all-or-nothing)           */
#define DLO_HOST_PAGEABLE 4u /* pageable; packed through two pinned host slots    */

/* number of kernel classes counted in dlo_stats (DLO_K_* below) */
#define DLO_K_COUNT 16

/* tensor dtypes in the flat block layout */
#define DLO_DT_BF16 0
#define DLO_DT_E4M3 1
#define DLO_DT_F32  2
#define DLO_DT_U8   3   /* opaque bytes (DLO_BLOCK_BYTES)                     */

/* Stack description.  Constraints (else DLO_EINVAL): abi_version ==
 * DLO_ABI_VERSION; n_blocks >= 1; hidden == heads * head_dim; hidden % 16 == 0;
 * head_dim % 8 == 0 and head_dim <= 128; ffn % 16 == 0; max_batch >= 1;
 * max_tokens >= 1; DiT: cond_dim % 8 == 0; video: text_dim % 16 == 0 and
 * max_text_tokens >= 1; eps > 0.  DLO_W_E4M3 and DLO_W_E4M3_A8 require
 * DLO_BLOCK_VIDEO (else DLO_EUNSUPPORTED).
 * DLO_BLOCK_BYTES streams opaque blocks of bytes_block bytes (a multiple of
 * 256) through the same slots and schedule; only n_blocks, staging,
 * register_budget_bytes and bytes_block are read.  Its "compute" reads the
 * whole slot and adds its 64-bit little-endian words (mod 2^64) into a
 * per-block checksum, so a slot reused too early shows up as a wrong sum. */
typedef struct dlo_desc {
    int abi_version;
    int block_kind;      /* DLO_BLOCK_*                                          */
    int wdtype;          /* DLO_W_*                                              */
    int n_blocks;        /* blocks in the stack                                  */
    int hidden;          /* D                                                    */
    int heads;           /* H                                                    */
    int head_dim;        /* hd = D / H                                           */
    int ffn;             /* F, MLP width                                         */
    int cond_dim;        /* DiT: width of the conditioning vector c              */
    int text_dim;        /* video: width Dt of the text context                  */
    int max_batch;       /* largest B passed to dlo_forward                      */
    int max_tokens;      /* largest N                                            */
    int max_text_tokens; /* video: largest L                                     */
    float eps;           /* LayerNorm / RMSNorm epsilon                          */
    int staging;         /* DLO_STAGE_*                                          */
    /* [DLO] "Registered runtime-cache transfer": the complete registration byte
     * count is checked against this budget before any registration; 0 = none. */
    unsigned long long register_budget_bytes;
    unsigned long long bytes_block;  /* DLO_BLOCK_BYTES: bytes per block          */
} dlo_desc;

typedef struct dlo_tensor_info {
    char name[40];              /* e.g. "attn.qkv.weight"                       */
    unsigned long long offset;  /* byte offset in the flat block, 256-B aligned
                                   for the first tensor of each group            */
    unsigned long long bytes;
    int dtype;                  /* DLO_DT_*                                     */
    int ndim;                   /* 1 or 2                                       */
    long long shape[2];         /* [out, in] for linear weights                 */
    int source;                 /* 1: supplied by the caller to dlo_pack_block;
                                   0: derived by dlo_pack_block (FP8 scales)    */
} dlo_tensor_info;

typedef struct dlo_ctx dlo_ctx;

/* ---------------------------------------------------------------- layout */

/* Bytes of one flattened block (K0 layout table), identical for all blocks.
 * [LW] How It Works: block parameters are kept as flattened tensors in pinned
 * host memory and re-materialised from them.  Returns 0 for an invalid desc. */
size_t dlo_block_bytes(const dlo_desc* desc);

/* Layout table of one flat block, in storage order.  out may be NULL to query
 * the count.  cap = entries available in out.  DLO_EINVAL on a bad desc,
 * DLO_ENOMEM when cap is too small (count is still set). */
dlo_status dlo_block_layout(const dlo_desc* desc, dlo_tensor_info* out, int cap, int* count);

/* Device workspace bytes dlo_create needs for this desc (activations of
 * max_batch x max_tokens, scratch for the block kernels, the kernels' error
 * word; with W8A16 weights also a bf16 copy of the block's largest linear,
 * into which each linear of a forward with at least DLO_WIDEN_ROWS rows --
 * default 4096 -- is widened before its GEMM).  Returns 0 for an invalid
 * desc. */
size_t dlo_workspace_bytes(const dlo_desc* desc);

/* Workspace bytes of a multi-container stack (dlo_create_multi): one carve-up
 * that serves every container.  Returns 0 when the descriptions are invalid
 * as a stack (see dlo_create_multi). */
size_t dlo_workspace_bytes_multi(const dlo_desc* descs, int n_containers);

/* Fill one flat host block from fp32 source tensors.
 * tensors[i] points at the fp32 values of layout entry i (row-major, the
 * entry's shape) for every entry with source == 1, and is ignored (may be
 * NULL) for derived entries.  bf16 entries are rounded to nearest even; with
 * DLO_W_E4M3 each linear weight is quantised per tensor (dlo_quantize_e4m3)
 * and its scale written into the "linear_scales" entry.  flat must hold
 * dlo_block_bytes(desc) bytes; padding bytes are zeroed.  Host only. */
dlo_status dlo_pack_block(const dlo_desc* desc, const float* const* tensors, int n_tensors,
                          void* flat, size_t flat_bytes);

/* Per-tensor FP8 quantiser ([DLO] Feature compatibility, row "Per-tensor online
 * FP8 linears"): s = amax|w| / 448 in fp32 (1 when amax == 0); codes[i] =
 * E4M3(w[i] / s) with w[i] / s in fp32, round to nearest even, saturating at
 * +-448 (OCP 8-bit floating point, E4M3).  Host only; n may be 0. */
dlo_status dlo_quantize_e4m3(const float* w, size_t n, uint8_t* codes, float* scale);

/* ---------------------------------------------------------------- lifecycle */

/* Create a context ([OFF] Shared lifecycle "enable"; [DLO] Startup and runtime
 * sequence "allocate device slots").
 *  device:        CUDA ordinal; made current by every call on the context.
 *  slot0, slot1:  device buffers of slot_bytes >= dlo_block_bytes(desc) each,
 *                 256-B aligned, not overlapping (the two device slots).
 *  workspace:     device buffer of ws_bytes >= dlo_workspace_bytes(desc),
 *                 256-B aligned, owned by the context until destroy.
 *  compute_stream, copy_stream: distinct caller streams; blocks compute on the
 *                 first, slot copies run on the second ([LW] copy_stream).
 * On error *out is NULL and nothing is retained. */
dlo_status dlo_create(const dlo_desc* desc, int device, void* slot0, void* slot1,
                      size_t slot_bytes, void* workspace, size_t ws_bytes,
                      void* compute_stream, void* copy_stream, dlo_ctx** out);

/* A stack of several ordered block containers ([LW] "For models with multiple
 * block types": a model lists more than one attribute holding transformer
 * blocks, e.g. double-stream then single-stream blocks).  descs[c] describes
 * container c (its own block_kind, wdtype, heads, head_dim, ffn, cond_dim and
 * n_blocks); the stack runs container 0's blocks, then container 1's, ..., as
 * one list of sum(n_blocks) blocks, numbered in that order by every other
 * call (registration, residency, the schedule, logs, dlo_verify_slot).  The
 * prefetch crosses container boundaries and, after the last block, wraps to
 * the first streamed block as for one container.  Both slots are shared by
 * all containers: slot_bytes >= the largest dlo_block_bytes(&descs[c])
 * ([DLO] Startup and runtime sequence: "two shared device slots sized for the
 * largest streamed block"); ws_bytes >= dlo_workspace_bytes_multi.
 * 1 <= n_containers <= DLO_MAX_CONTAINERS.  The containers must agree on
 * hidden, max_batch, max_tokens, eps, staging and register_budget_bytes;
 * video containers also on text_dim and max_text_tokens; DLO_BLOCK_BYTES
 * stacks have a single container.  Else DLO_EINVAL.  Host blocks for such a
 * stack are registered with block_bytes = 0 (each block holds its own
 * container's dlo_block_bytes); resident buffer i holds block i's bytes. */
dlo_status dlo_create_multi(const dlo_desc* descs, int n_containers, int device, void* slot0,
                            void* slot1, size_t slot_bytes, void* workspace, size_t ws_bytes,
                            void* compute_stream, void* copy_stream, dlo_ctx** out);

/* Attach the n = desc->n_blocks flat host blocks (host_blocks[i], block_bytes
 * = dlo_block_bytes(desc) each, or 0 meaning each block's own layout size --
 * the only value for multi-container stacks; immutable while attached: [OFF]
 * "a parameter has one authoritative host representation").
 *  DLO_HOST_PINNED:   memory is already page-locked (cudaHostAlloc or
 *                     registered); verified with cudaPointerGetAttributes.
 *  DLO_HOST_REGISTER: the library page-aligns the block ranges, merges
 *                     overlapping or adjacent ones, checks the total against
 *                     register_budget_bytes before any mutation, then
 *                     registers each range (read-only where the platform
 *                     supports it) and verifies every block reads as pinned
 *                     ([DLO] Registered runtime-cache transfer).  Any failure
 *                     unregisters the ranges already registered and returns
 *                     DLO_EREGISTER with the context unchanged, so the call can
 *                     be retried ([DLO] Failure and lifecycle boundaries).
 *  DLO_HOST_PAGEABLE: memory stays pageable (e.g. views of a file mapping);
 *                     the library allocates two pinned host staging slots of
 *                     block_bytes each (cudaHostAlloc; freed by dlo_destroy)
 *                     and, for every staging, packs the block into the next
 *                     host slot with a stream-ordered host function on the
 *                     copy stream (a synchronous host copy spread over a few
 *                     library threads) before the pinned host-to-device copy
 *                     ([DLO] Host backing and transfer composition: "mmap views
 *                     -> pinned staging slot -> device slot"; the user guide's
 *                     mmap weight storage: packing into the host slot is
 *                     synchronous, the pinned copy overlaps computation).
 *                     Needs DLO_STAGE_MEMCPY.  Allocation failure: DLO_ENOMEM.
 * Exactly one of the flags.  With DLO_STAGE_GATHER the blocks must be
 * device-accessible (mapped); checked here.  Allowed once, before forward. */
dlo_status dlo_register_host_blocks(dlo_ctx* ctx, int n, const void* const* host_blocks,
                                    size_t block_bytes, unsigned flags);

/* Keep blocks 0..k-1 resident ([DLO] Feature compatibility, row "Resident
 * leading layers").  device_blocks[i] (i < k) are caller device buffers of
 * block_bytes, 256-B aligned; the library copies host block i into each on
 * the copy stream.  Then the first streamed block k is staged into slot 0
 * (priming, [DLO] Startup and runtime sequence).  0 <= k <= n.  Allowed once,
 * after registration and before the first forward; without it the first
 * forward primes block 0 itself (k = 0). */
dlo_status dlo_set_resident(dlo_ctx* ctx, int k, void* const* device_blocks);

/* One forward of the block stack (one denoising step), enqueued on the compute
 * stream; returns after enqueue ([LW] Execution Flow; [DLO] "each streamed
 * block during pipeline.forward").
 *  x_in, x_out:  device bf16 [batch, tokens, hidden]; x_out may equal x_in.
 *  cond:         DiT: device bf16 c [batch, cond_dim];
 *                video: device fp32 e [batch, 6, hidden].
 *  ctx_tokens:   video: device bf16 text context [batch, text_tokens,
 *                text_dim]; DiT: NULL.
 * 1 <= batch <= max_batch, 1 <= tokens <= max_tokens, video: 1 <= text_tokens
 * <= max_text_tokens.
 * Per streamed execution j (over all forwards) of block i: the copy stream
 * waits until the compute that last read slot (j+1)%2 is done, stages block
 * i+1 (or the first streamed block after the last) into it and records
 * copy_done; the compute stream waits on copy_done of slot j%2, runs block i
 * from that slot and records compute_done.
 * DiT block (eps = desc->eps; LN has no affine and biased variance):
 *   m = SiLU(c) W_ada^T + b_ada -> shift1, scale1, gate1, shift2, scale2, gate2
 *   x += gate1 * (Attn(LN(x)(1+scale1)+shift1) W_o^T + b_o)
 *   x += gate2 * (GELU_tanh((LN(x)(1+scale2)+shift2) W_1^T + b_1) W_2^T + b_2)
 *   Attn: qkv = h W_qkv^T + b_qkv, q|k|v each [H, hd] per token,
 *         softmax(q k^T / sqrt(hd)) v per head, non-causal.
 * Bytes block (DLO_BLOCK_BYTES): batch = tokens = 1; x_in, cond, ctx_tokens
 *   are ignored (may be NULL); x_out is a device uint64 array [n_blocks] that
 *   receives, for every block executed by this call, the sum of its 64-bit
 *   words as read from the slot (or resident buffer) it ran from.
 * Video block: m = e + T_mod; self-attention as above with separate q,k,v
 *   linears and RMSNorm (gain, over hidden) on q and k, x += gate1 * o;
 *   cross-attention with q = RMSNorm(LN_affine(x) W_q^T + b_q), k = RMSNorm(
 *   ctx W_k^T + b_k), v = ctx W_v^T + b_v, x += o; FFN as DiT with gate2.
 * The hidden state is carried in fp32 between kernels; x_out is its bf16
 * rounding.  Device-side bounded waits that run out are reported by the next
 * dlo_wait / dlo_forward_host as DLO_ETIMEDOUT (dlo_stats.device_error keeps
 * the word read). */
dlo_status dlo_forward(dlo_ctx* ctx, const void* x_in, const void* cond, const void* ctx_tokens,
                       int batch, int tokens, int text_tokens, void* x_out);

/* dlo_forward of a multi-container stack: conds[c] (device, layout of that
 * container's block_kind as for dlo_forward) conditions the blocks of
 * container c; ctx_tokens serves every video container.  dlo_forward itself
 * accepts a multi-container stack only when all containers share block_kind
 * and cond_dim (one cond for all); else DLO_EINVAL.  dlo_forward_host takes
 * single-container stacks only (DLO_EUNSUPPORTED otherwise). */
dlo_status dlo_forward_multi(dlo_ctx* ctx, const void* x_in, const void* const* conds,
                             const void* ctx_tokens, int batch, int tokens, int text_tokens,
                             void* x_out);

/* dlo_forward with HOST inputs and output: copies x_in, cond and ctx_tokens
 * (same layouts as dlo_forward) into the workspace on the compute stream,
 * runs the stack, copies the bf16 result back into x_out and waits for it
 * (bounded by timeout_ms; <= 0 means 60000).  Pinned host buffers give
 * asynchronous copies; pageable ones work too. */
dlo_status dlo_forward_host(dlo_ctx* ctx, const void* x_in, const void* cond,
                            const void* ctx_tokens, int batch, int tokens, int text_tokens,
                            void* x_out, int timeout_ms);

/* Host wait for all work of the context on both streams, polling with a time
 * limit; DLO_ETIMEDOUT when it runs out or when a kernel reported a timed-out
 * device wait.  timeout_ms <= 0 means 60000. */
dlo_status dlo_wait(dlo_ctx* ctx, int timeout_ms);

/* Tear down ([DLO] Failure and lifecycle boundaries, shutdown order):
 * synchronise both streams, unregister the ranges this library registered,
 * destroy events, free the context.  NULL is accepted.  Returns the first
 * error met but always frees the context. */
dlo_status dlo_destroy(dlo_ctx* ctx);

/* Message of the last error on ctx, or of the last failed dlo_create in this
 * thread when ctx is NULL.  Never NULL. */
const char* dlo_last_error(const dlo_ctx* ctx);

/* ---------------------------------------------------------------- introspection */

typedef struct dlo_stats {
    unsigned long long forwards;         /* dlo_forward calls completed enqueue  */
    unsigned long long stagings;         /* block copies into slots (incl. prime) */
    unsigned long long staged_bytes;
    unsigned long long streamed_execs;   /* streamed block executions            */
    unsigned long long kernel_launches;  /* kernels this library launched        */
    int resident;                        /* k                                    */
    int slot_block[2];                   /* block last staged into each slot, -1 */
    int registered_ranges;               /* host ranges this library registered  */
    int registered_read_only;            /* 1 if they were registered read-only  */
    int device_error;                    /* kernels' error word (0 = none)       */
    /* With dlo_set_timing(ctx, 1 or 2): sums over timed streamed executions, ms. */
    int timed_execs;
    double copy_ms;                      /* slot copy durations                  */
    double compute_ms;                   /* block compute durations              */
    double exposed_wait_ms;              /* compute stream idle waiting on copies */
    /* With dlo_set_timing(ctx, 2 or 3): per kernel class (DLO_K_*), CUDA-event time
     * of each launch on its own stream, launches, and the algorithmic work of
     * those launches: 2*M*N*K per GEMM, 4*B*H*nq*nk*hd per attention, bytes
     * read + written once per element for the bandwidth-bound kernels. */
    double kclass_ms[DLO_K_COUNT];
    double kclass_flops[DLO_K_COUNT];
    double kclass_bytes[DLO_K_COUNT];
    unsigned long long kclass_launches[DLO_K_COUNT];
    unsigned long long h2d_copies;       /* host-to-device copy calls issued     */
    unsigned long long graph_captures;   /* forwards captured as CUDA graphs     */
    unsigned long long graph_launches;   /* forwards run as a CUDA graph launch  */
} dlo_stats;

/* kernel classes of dlo_stats.kclass_* */
#define DLO_K_GEMM_BF16  0
#define DLO_K_GEMM_E4M3  1
#define DLO_K_ATTENTION  2
#define DLO_K_LAYERNORM  3
#define DLO_K_RMSNORM    4
#define DLO_K_MODULATION 5   /* adaLN GEMV or modulation-table add            */
#define DLO_K_CONVERT    6   /* bf16 <-> fp32 of the hidden state; bytes-block
                                checksum                                       */
#define DLO_K_GATHER     7   /* zero-copy slot staging kernel                  */
#define DLO_K_GEMM_FP8   8   /* W8A8 GEMM (kind::f8f6f4, both operands E4M3)   */
#define DLO_K_QUANT      9   /* dynamic per-tensor E4M3 activation quantiser  */

/* Counters and timing.  Timing sums need the timed work finished (call
 * dlo_wait first); they are read from CUDA events. */
dlo_status dlo_get_stats(dlo_ctx* ctx, dlo_stats* out);

/* Ordered log of enqueued staging and execution events since create or the
 * last dlo_reset_log: kind[i] 0 = stage, 1 = execute; block[i]; slot[i] (-1
 * for a resident execution).  Up to cap entries are written; *count gets the
 * total logged (the log keeps the first 65536). */
dlo_status dlo_get_log(dlo_ctx* ctx, int* kind, int* block, int* slot, int cap, int* count);
dlo_status dlo_reset_log(dlo_ctx* ctx);

/* CUDA-event timing: 0 off (default); 1 five events per streamed execution
 * (copy, wait and compute intervals); 2 also an event pair around every
 * kernel launch (per-class stats); 3 the per-kernel pairs alone, and these
 * also inside CUDA graphs (dlo_set_graphs): a forward captured at level 3
 * holds its pairs as event-record nodes, read back after each launch of the
 * graph (a graph launched again before its last launch was read first waits
 * for that launch).  Timing adds event records to the streams; between two
 * kernels an event record also takes the place of their programmatic-launch
 * edge, so a kernel's time includes its own launch and prologue. */
dlo_status dlo_set_timing(dlo_ctx* ctx, int on);

/* Whole-forward CUDA graphs: 0 off (default), 1 on.  With graphs on and
 * timing 0 or 3, dlo_forward / dlo_forward_multi / dlo_forward_host capture the
 * forward's work on both streams (staging copies, event dependencies and
 * every kernel, with their programmatic-launch edges) into a CUDA graph the
 * first time they see a set of arguments (pointers, batch, tokens, text
 * tokens) at a slot parity (which slot holds the first streamed block: the
 * parity of the streamed executions so far), and launch that graph on later
 * calls with the same arguments and parity -- up to four graphs per context
 * (e.g. ping-pong input/output buffers at both parities), the least recently
 * used one replaced by a new capture.  A context's first forward is always
 * enqueued directly (kernels' one-time set-up stays outside captures).  Results, staging order, slot contents,
 * log and counters are the same as without graphs; the graph's launch waits
 * for all earlier work of both streams.  The pageable host mode and timing
 * levels 1 and 2 enqueue directly; a graph is reused only at the timing
 * level it was captured at.  If a capture fails, nothing of it has run:
 * graphs are turned off for the context, the forward is enqueued directly
 * and dlo_last_error keeps the reason.  Turning graphs off frees the
 * captured graphs.  Not thread-safe with concurrent calls on one context. */
dlo_status dlo_set_graphs(dlo_ctx* ctx, int on);

/* Debug: wait for the copy that last wrote `slot`, copy the slot back and
 * compare it byte for byte with host block `block` (-1: the block the library
 * staged there last).  DLO_OK if identical, DLO_EMISMATCH if not.  Blocks the
 * host (bounded, 60 s). */
dlo_status dlo_verify_slot(dlo_ctx* ctx, int slot, int block);

/* Test hook (process-wide): make the nth cudaHostRegister call issued by
 * dlo_register_host_blocks from now on report failure (n >= 1), or disable
 * with n <= 0.  Exercises the rollback path without a platform fault. */
void dlo_debug_fail_register(int nth);

/* ---------------------------------------------------------------- unit ops
 * The kernels one block is made of, callable on their own (device pointers,
 * enqueued on `stream`).  They check arguments and return DLO_EINVAL before
 * launching.  `err` is a device int (0 on entry) that a kernel sets when one
 * of its bounded waits runs out; it may be NULL for kernels without waits. */

/* GEMM epilogues */
#define DLO_EPI_BIAS      0  /* out bf16 [M, ldo] = acc*s + bias                 */
#define DLO_EPI_GELU      1  /* out bf16 = GELU_tanh(acc*s + bias)               */
#define DLO_EPI_RESIDUAL  2  /* out fp32 [M, ldo] += gate * (acc*s + bias)       */

/* Y = A W^T on the tensor cores (tcgen05, TMA), fp32 accumulate, fused
 * epilogue.  A: bf16 [M, K] row-major (lda = K).  W: [N, K] row-major, bf16
 * or e4m3 (w_dtype DLO_DT_*).  scales: NULL (s = 1) or fp32 per column
 * segment, s = scales[col / scale_seg] (e4m3 per-tensor scales of the
 * concatenated tensors).  bias: bf16 [N] or NULL.  gate (RESIDUAL only): NULL
 * (1) or fp32 with gate[(row / rows_per_batch) * gate_ld + col].
 * M >= 1, N % 16 == 0, K % 16 == 0, K >= 16; pointers 16-B aligned, ldo % 8 == 0. */
dlo_status dlo_op_gemm(const void* A, const void* W, int w_dtype, const float* scales,
                       int scale_seg, const void* bias, int M, int N, int K, int epilogue,
                       void* out, int ldo, const float* gate, int gate_ld, int rows_per_batch,
                       int* err, void* stream);

/* Time-out path of the kernels' bounded waits, without a fault ([DLO]
 * Failure and lifecycle boundaries: a failure is reported, not hidden, and
 * leaves the process usable).  One thread waits on an mbarrier that nothing
 * completes; after the library's wait limit (2 s) it writes 1 to *err (a
 * device int) and the kernel exits normally, as every kernel of this library
 * does when one of its waits runs out.  For tests. */
dlo_status dlo_op_wait_selftest(int* err, void* stream);

/* Enqueue the same waiting kernel on ctx's compute stream with ctx's error
 * word, so the next dlo_wait / dlo_forward_host reports DLO_ETIMEDOUT (and
 * clears the word; the context stays usable).  For tests. */
dlo_status dlo_debug_device_timeout(dlo_ctx* ctx);

/* Dynamic per-tensor E4M3 quantisation of an activation (DLO_W_E4M3_A8):
 * x bf16 [rows, cols] with row stride ld (elements); q receives E4M3 codes
 * [rows, cols], contiguous; *scale (device fp32) receives s = amax|x| / 448
 * (1 when amax = 0) -- the weights' scale rule (dlo_quantize_e4m3) -- and
 * q = E4M3(x * r) with r = 1 / s rounded to fp32 and the product rounded to
 * fp32, then round to nearest even, saturating at +-448 (the inverted-scale
 * form of dynamic FP8 activation quantisers: one multiply per element).  scratch: device
 * buffer of DLO_QUANT_SCRATCH floats (partial maxima; no allocation here).
 * cols % 8 == 0, ld % 8 == 0, x and q 16-B aligned.  Two kernel launches. */
#define DLO_QUANT_SCRATCH 1024
dlo_status dlo_op_quantize_act(const void* x, int rows, int cols, int ld, void* q, float* scale,
                               float* scratch, void* stream);

/* Y = s_x s_w (A W^T) + bias with A E4M3 codes [M, K] (lda = K) and its scale
 * *a_scale (device fp32, e.g. from dlo_op_quantize_act), W E4M3 codes [N, K]
 * with per-tensor scales as dlo_op_gemm (scales required); kind::f8f6f4 on
 * the tensor cores, fp32 accumulation, then the epilogues of dlo_op_gemm.
 * M >= 1, N % 16 == 0, K % 16 == 0; pointers 16-B aligned, ldo % 8 == 0. */
dlo_status dlo_op_gemm_w8a8(const void* A, const float* a_scale, const void* W, const float* scales,
                            int scale_seg, const void* bias, int M, int N, int K, int epilogue,
                            void* out, int ldo, const float* gate, int gate_ld, int rows_per_batch,
                            int* err, void* stream);

/* dlo_op_gemm for callers that cannot allocate device memory.  Some code may
 * not call cudaMalloc at all: a plugin running inside another framework whose
 * caching allocator owns the device's memory (a direct allocation would
 * bypass its accounting, or find no memory left), or a serving process whose
 * memory plan is fixed at start-up.  Such a caller still owns its inputs and
 * outputs; it has no buffer to hand over for the kernel's scratch.
 * The pages have no counterpart; this is an addition of this library.
 * Same arguments, checks and results as dlo_op_gemm minus `err`: the kernel's
 * scratch (its device error word) lives in a static device array of at most
 * 256 bytes that every GPU which loads this library holds until the process
 * exits; this entry uses 4 bytes of it and clears them before each launch.
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array, so calls that
 * overlap on the GPU race on the error word; a bounded wait that runs out
 * leaves `out` incomplete and is not reported (use dlo_op_gemm with your own
 * error word when you need that report).  Argument errors return DLO_EINVAL
 * before anything is enqueued, launch errors DLO_ECUDA; the message is in
 * dlo_last_error(NULL). */
dlo_status dlo_op_gemm_noalloc(const void* A, const void* W, int w_dtype, const float* scales,
                               int scale_seg, const void* bias, int M, int N, int K,
                               int epilogue, void* out, int ldo, const float* gate, int gate_ld,
                               int rows_per_batch, void* stream);

/* Multi-head softmax attention, non-causal: O = softmax(Q K^T / sqrt(hd)) V per
 * (batch, head).  Q, K, V, O bf16; row r of batch b of Q starts at
 * Q + (b * nq + r) * ldq, head h at column h * head_dim (same for K, V with nk
 * and ldk / ldv, O with nq and ldo).  head_dim % 8 == 0, <= 128; ld* % 8 == 0. */
dlo_status dlo_op_attention(const void* Q, const void* K, const void* V, void* O, int batch,
                            int heads, int head_dim, int nq, int nk, int ldq, int ldk, int ldv,
                            int ldo, void* stream);

/* out bf16 [rows, D] = LN(x) * (1 + scale) + shift   (shift/scale non-NULL), or
 *                    = LN(x) * w + b                  (w/b non-NULL), or LN(x).
 * x fp32 [rows, D]; shift/scale fp32 indexed [(row / rows_per_batch) * mod_ld + d];
 * w, b bf16 [D]. */
dlo_status dlo_op_layernorm(const float* x, int rows, int D, int rows_per_batch,
                            const float* shift, const float* scale, int mod_ld,
                            const void* w, const void* b, float eps, void* out, void* stream);

/* In place on bf16 x: row r, columns col0 .. col0+D-1 of a row stride ld:
 * x = x / sqrt(mean(x^2) + eps) * w, w bf16 [D]. */
dlo_status dlo_op_rmsnorm(void* x, int rows, int D, int ld, int col0, const void* w, float eps,
                          void* stream);

/* m fp32 [B, N] = SiLU(c) W^T + bias; c bf16 [B, C], W bf16 [N, C], bias bf16 [N]. */
dlo_status dlo_op_adaln(const void* c, int B, int C, const void* W, const void* bias, int N,
                        float* m, void* stream);

/* Copy `bytes` (% 16 == 0, both pointers 16-B aligned) from device-accessible
 * src (device memory or mapped host memory) to device dst with the gather
 * kernel (mode DLO_STAGE_GATHER) or cudaMemcpyAsync (DLO_STAGE_MEMCPY). */
dlo_status dlo_op_stage(void* dst, const void* src, size_t bytes, int mode, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DLO_H */
