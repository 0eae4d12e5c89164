/*
 * moe_lora.h -- C ABI of libmoelora.so, the multi-LoRA fused MoE layer forward
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation (AWS machine-learning blog "Efficiently serve dozens of
 * fine-tuned models with vLLM on Amazon SageMaker AI and Amazon Bedrock",
 * section "Implementing multi-LoRA inference for MoE models in vLLM",
 * Figure 1): a router has sent every token t to k experts e = topk_ids[t][j]
 * with weights w = topk_weights[t][j]; the token carries one adapter id
 * l = token_lora_ids[t] (-1: base model only).  For every (token, slot) pair
 *
 *     g    = W1[e] x[t]   + B1[l][e] (A1[l][e] x[t])       (gate_up, 2I rows)
 *     act  = SiLU(g[0:I]) * g[I:2I]                        (SiLU(u) = u/(1+e^-u))
 *     d    = W2[e] act    + B2[l][e] (A2[l][e] act)        (down, H rows)
 *
 * and out[t] = bf16( sum_j w[t][j] * d[t*k+j] ).  Each LoRA term is the
 * blog's shrink (z = x A, h_in -> r) followed by its expand (z B, r -> h_out),
 * with no extra scale; it is left out when l = -1.
 *
 * Conventions for every entry point:
 *   - Tensor pointers are DEVICE pointers owned by the caller.  The library
 *     never allocates or frees device memory; scratch lives in the caller's
 *     workspace (size from moe_lora_workspace_bytes).
 *   - bf16 tensors are raw IEEE bfloat16 bits.  All layouts are row-major
 *     "[out][in]" (the reduction dimension is contiguous), i.e. the transposes
 *     of the blog's h_in x h_out matrices:
 *         x [T][H], W1 [E][2I][H] (gate rows 0..I-1, up rows I..2I-1),
 *         W2 [E][H][I], A1 [L][E][r][H], B1 [L][E][2I][r],
 *         A2 [L][E][r][I], B2 [L][E][H][r], out [T][H],
 *         topk_ids [T][k] int32, topk_weights [T][k] float32,
 *         token_lora_ids [T] int32.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Nothing synchronises the host except
 *     moe_lora_get_status.  Inputs are never modified; `out` is fully
 *     overwritten.
 *   - Errors that the host can see (null pointers, bad sizes, misalignment,
 *     a workspace that is too small) return a negative status before anything
 *     is launched.  Errors only the device can see (an expert id outside
 *     [0, E), an adapter id outside [-1, L)) leave the affected pairs out of
 *     the result and set a status word in the workspace, read back by
 *     moe_lora_get_status; no kernel traps.
 *   - Alignment: every tensor pointer and the workspace must be 16-byte
 *     aligned; H and I must be multiples of 8; r a multiple of 8 in [8, 64]
 *     when L > 0.  Otherwise MOELORA_EUNSUPPORTED.
 *   - The library keeps no state between calls beyond a per-device cache of
 *     kernel attributes; calls on different workspaces may run concurrently.
 */
#ifndef MOE_LORA_H
#define MOE_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOELORA_API __attribute__((visibility("default")))

/* Problem sizes.  block_m is the bucket padding granularity (the tile height
 * shared by every kernel of one forward, as the blog's section "Tuning kernel
 * configurations" shares one BLOCK_SIZE_M across the four LoRA ops); 0 lets
 * the library choose (16). */
typedef struct moe_lora_dims {
    int32_t T;       /* tokens, >= 0 */
    int32_t H;       /* hidden size, > 0, multiple of 8 */
    int32_t I;       /* intermediate size per expert, > 0, multiple of 8 */
    int32_t E;       /* experts, > 0 */
    int32_t k;       /* experts per token, > 0 */
    int32_t L;       /* adapters, >= 0 (0: no LoRA; A and B pointers may be NULL) */
    int32_t r;       /* LoRA rank: multiple of 8 in [8, 64] if L > 0, ignored if L == 0 */
    int32_t block_m; /* 0 = default 16; otherwise a power of two in [1, 256] */
    int32_t options; /* 0, or MOELORA_OPT_SINGLE_CTA */
    int32_t sm_count; /* SMs the work is planned for (K-split and shrink-split choice, and
                         with them the workspace size): 0 = the current device's
                         multiprocessor count (152 on GB300; 152 when no device is
                         visible), else a count in [1, 4096].  A workspace sized for one
                         count serves any forward planned with the same count; the
                         results do not depend on it. */
} moe_lora_dims;

/* Batches with wide expert chunks (more than 48 pairs per expert on average)
 * run their two GEMMs on CTA pairs by default: tcgen05.mma.cta_group::2 with
 * 256 pair rows on M (128 per CTA) and two chains of up to 256 weight rows on
 * N, when that kernel covers the layer (at most 64 adapters, the tensor-core
 * LoRA expand, its per-chunk adapter masks and zexp buffers within bounds).
 * MOELORA_OPT_SINGLE_CTA keeps them on the one-CTA kernel (one tile of 128
 * weight rows per task), the path every other batch takes: same results
 * within rounding, for comparison and testing. */
#define MOELORA_OPT_SINGLE_CTA 1

/* Status codes (return values; moe_lora_strerror gives a message). */
#define MOELORA_OK 0
#define MOELORA_EINVAL (-1)        /* null pointer or impossible size */
#define MOELORA_ENOSPC (-2)        /* workspace smaller than moe_lora_workspace_bytes */
#define MOELORA_EUNSUPPORTED (-3)  /* valid but outside what the kernels handle (alignment, r > 64, ...) */
#define MOELORA_ECUDA (-4)         /* a CUDA runtime call failed (e.g. no device) */
#define MOELORA_EDEVICE_ID (-5)    /* the device met an out-of-range expert or adapter id */
#define MOELORA_ETIMEOUT (-6)      /* a kernel gave up a bounded wait (its output is incomplete) */

/* Human-readable message for a status code; never NULL. Host only. */
MOELORA_API const char *moe_lora_strerror(int code);

/* ABI version (major * 10000 + minor * 100 + patch). Host only. */
MOELORA_API int moe_lora_version(void);

/* Entries that moe_lora_align may write into sorted_ids:
 * P + min(E*(L+1), P) * (block_m - 1) with P = T*k; tile_expert and tile_lora
 * need capacity / block_m entries.  Returns < 0 (a status) on bad dims.
 * Host only, pure. */
MOELORA_API int64_t moe_lora_align_capacity(const moe_lora_dims *d);

/* Bytes of device workspace that moe_lora_forward, moe_lora_forward_w8 and
 * moe_lora_align need for these dims (0 if the dims are invalid).  Host only; with
 * d->sm_count == 0 it reads the current device's multiprocessor count (no
 * launch, no allocation), else it is pure. */
MOELORA_API size_t moe_lora_workspace_bytes(const moe_lora_dims *d);

/*
 * Expert x adapter bucketing of the T*k (token, slot) pairs: the extra
 * adapter grid dimension the blog adds to fused_moe, and the compound
 * sparsity (expert routing times adapter choice) it describes, both in the
 * section "Implementing multi-LoRA inference for MoE models in vLLM".
 *
 * Pair p = t*k + j goes to bucket b = e*(L+1) + (l+1) with e = topk_ids[p],
 * l = token_lora_ids[t]; buckets are laid out in ascending b, pairs keep
 * ascending p inside a bucket, and each non-empty bucket is padded up to a
 * multiple of block_m with the sentinel value P = T*k (empty buckets take no
 * room).  Outputs (device pointers, int32):
 *   sorted_ids      [moe_lora_align_capacity] -- entries past num_post_padded untouched
 *   tile_expert     [capacity / block_m]      -- expert of each block_m-row tile
 *   tile_lora       [capacity / block_m]      -- adapter of each tile (-1: base)
 *   num_post_padded [1]                       -- total padded length
 *   bucket_count    [E*(L+1)]                 -- valid pairs per bucket
 *   bucket_offset   [E*(L+1) + 1]             -- padded start of each bucket
 * Pairs with an out-of-range id are left out and flagged in the workspace
 * status word (see moe_lora_get_status).  The result is unique and
 * deterministic.  Returns a status; asynchronous on `stream`.
 */
MOELORA_API int moe_lora_align(const moe_lora_dims *d, const int32_t *topk_ids,
                               const int32_t *token_lora_ids, int32_t *sorted_ids,
                               int32_t *tile_expert, int32_t *tile_lora,
                               int32_t *num_post_padded, int32_t *bucket_count,
                               int32_t *bucket_offset, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * The layer forward described at the top of this header, computed by the
 * library's kernels in bf16 inputs / fp32 accumulation, the sum over the k
 * slots in fp32 and rounded once to bf16 (round to nearest even).
 * Intermediates: the LoRA shrink outputs in fp32, the activation in bf16, and
 * each pair's weighted down output in bf16 (fp32 partial sums when the down
 * GEMM splits K; see moe_lora_ws_layout).
 * A1, B1, A2, B2 may be NULL only when L == 0.  `out` [T][H] bf16 is fully
 * overwritten.  The workspace must hold moe_lora_workspace_bytes(d) bytes;
 * its contents on entry do not matter.  Results are deterministic (no
 * floating-point atomics): the same inputs give the same bits.
 * Returns a status; asynchronous on `stream`; capturable in a CUDA graph.
 */
MOELORA_API int moe_lora_forward(const moe_lora_dims *d, const void *x,
                                 const int32_t *topk_ids, const float *topk_weights,
                                 const int32_t *token_lora_ids, const void *W1,
                                 const void *W2, const void *A1, const void *B1,
                                 const void *A2, const void *B2, void *out,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * The forward with FP8 base expert weights and bf16 LoRA (the fused-MoE news
 * item's second optimisation: FP8 MoE weights, dequantised inside the fused
 * GEMM).  Instead of W1 and W2:
 *   W1q [E][2I][H], W2q [E][H][I]: 8-bit E4M3 codes (the finite "fn" form:
 *     sign, 4-bit exponent with bias 7, 3-bit mantissa; largest value 448);
 *   W1s [E][2I], W2s [E][H]: one fp32 scale per output row; the weight is
 *     scale * value(code).
 * Every other argument, the workspace and the result are those of
 * moe_lora_forward.  The GEMMs run on the CTA-pair kernels for every batch
 * size: the codes stream from HBM by TMA, and each code is turned into a
 * bf16 weight in shared memory right before the bf16 MMAs read it: the
 * row's scale is rounded to bf16 precision once (8 significant bits), and
 * each weight is value(code) times that, rounded to bf16 (activations stay
 * bf16, fp32 accumulation).  H and I must be multiples of 16 and the layer within the
 * CTA-pair kernels' bounds (at most 64 adapters, zexp within bounds), else
 * MOELORA_EUNSUPPORTED.  Pointers 16-byte aligned.  Asynchronous on
 * `stream`; same status codes as moe_lora_forward.
 */
MOELORA_API int moe_lora_forward_w8(const moe_lora_dims *d, const void *x,
                                    const int32_t *topk_ids, const float *topk_weights,
                                    const int32_t *token_lora_ids, const void *W1q,
                                    const float *W1s, const void *W2q, const float *W2s,
                                    const void *A1, const void *B1, const void *A2,
                                    const void *B2, void *out, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * moe_lora_forward with timing marks, for profiling the kernels one by one on
 * the stream they run on.  kernel_events holds MOELORA_TRACE_EVENTS
 * cudaEvent_t handles created by the caller (cudaEventCreate); event i is
 * recorded on `stream` just before kernel slot i and the last one after the
 * final kernel.  Kernel slots: 0 align, 1 gather of x into bucket order,
 * 2 gate_up tcgen05 kernel (LoRA shrink items, grouped GEMM, expand,
 * SiLU*up), 3 down tcgen05 kernel (LoRA shrink items, grouped GEMM, expand,
 * x weight), 4 top-k reduce.  The recorded events replace the programmatic
 * launch overlap between consecutive kernels with plain stream order.  Same
 * results and status codes as moe_lora_forward, plus MOELORA_EINVAL if
 * kernel_events is NULL or n_events < MOELORA_TRACE_EVENTS.
 */
#define MOELORA_TRACE_EVENTS 6
MOELORA_API int moe_lora_forward_traced(const moe_lora_dims *d, const void *x,
                                        const int32_t *topk_ids, const float *topk_weights,
                                        const int32_t *token_lora_ids, const void *W1,
                                        const void *W2, const void *A1, const void *B1,
                                        const void *A2, const void *B2, void *out,
                                        void *workspace, size_t workspace_bytes, void *stream,
                                        void *const *kernel_events, int32_t n_events);

/*
 * moe_lora_forward_w8 with the timing marks of moe_lora_forward_traced (same
 * events, kernel slots and extra status codes).
 */
MOELORA_API int moe_lora_forward_w8_traced(const moe_lora_dims *d, const void *x,
                                           const int32_t *topk_ids, const float *topk_weights,
                                           const int32_t *token_lora_ids, const void *W1q,
                                           const float *W1s, const void *W2q, const float *W2s,
                                           const void *A1, const void *B1, const void *A2,
                                           const void *B2, void *out, void *workspace,
                                           size_t workspace_bytes, void *stream,
                                           void *const *kernel_events, int32_t n_events);

/*
 * Self-test of the device-side wait bounds (the pages have no counterpart).
 * Launches one small kernel on `stream` whose wait nothing will satisfy --
 * kind 0: an mbarrier phase that expects an arrival nobody makes; kind 1: a
 * global counter (in the workspace header) nobody increments.  The wait gives
 * up under the same bounds as the forward's waits (2^20 rounds or one second
 * of the GPU's global timer) and records the timeout in the workspace status
 * word, so a following moe_lora_get_status returns MOELORA_ETIMEOUT; the
 * context stays usable.  workspace: device pointer to at least 256 bytes, 16-byte aligned,
 * overwritten (header only).  Returns MOELORA_EINVAL for another kind or a NULL
 * workspace, MOELORA_ECUDA if the launch fails.  Asynchronous.
 */
MOELORA_API int moe_lora_selftest_wait(int32_t kind, void *workspace, void *stream);

/*
 * Waits for `stream`, then returns MOELORA_OK if the last align/forward that
 * used this workspace met no out-of-range id, MOELORA_EDEVICE_ID if it did,
 * MOELORA_ETIMEOUT if one of its kernels abandoned a bounded wait inside its
 * copy pipeline (every wait in the library is bounded, so no kernel can spin
 * forever; the output is then incomplete), or MOELORA_ECUDA if a CUDA call
 * failed.  The only synchronising entry point.
 */
MOELORA_API int moe_lora_get_status(const void *workspace, void *stream);

/*
 * moe_lora_forward for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it serves code that may not call
 * cudaMalloc (which can wait for the whole device to go idle, so
 * latency-bound loops avoid it), plugins whose host framework owns every
 * device allocation and offers them none, or callers with no allocator at all.
 *
 * Same arguments, results and host-side status codes as moe_lora_forward,
 * minus the workspace: the scratch is a buffer of
 * MOELORA_NOALLOC_SCRATCH_BYTES (16 MiB) inside the library's device image,
 * held by every GPU that loads the library until the process exits.  Nothing
 * is allocated or freed by this call.
 *   - Problems whose moe_lora_workspace_bytes(d) exceeds that size return
 *     MOELORA_ENOSPC before anything is launched (e.g. the decode layer
 *     T=16, H=I=2880, E=32, top-4, r=32 needs about 1.3 MiB).
 *   - The first call on each device looks the buffer's device address up
 *     (cudaGetSymbolAddress, with that device current).
 *   - All calls in the process share the one buffer per device, and each call
 *     leaves its intermediates in it.  Calls whose work overlaps on the GPU
 *     (two streams, or two host threads, of the same device) race on it:
 *     order them on one stream or serialise them.  No part of the buffer has
 *     to start at zero; every call rewrites what it reads.
 *   - The status word lives in the shared buffer and is not reported:
 *     out-of-range expert or adapter ids are still left out of the result, and
 *     a kernel that gives up a bounded wait (MOELORA_ETIMEOUT with a
 *     workspace) still leaves an incomplete output, but this call returns
 *     MOELORA_OK for both.  Use moe_lora_forward with a workspace where that
 *     status matters.
 */
#define MOELORA_NOALLOC_SCRATCH_BYTES (16u << 20)
MOELORA_API int moe_lora_forward_noalloc(const moe_lora_dims *d, const void *x,
                                         const int32_t *topk_ids, const float *topk_weights,
                                         const int32_t *token_lora_ids, const void *W1,
                                         const void *W2, const void *A1, const void *B1,
                                         const void *A2, const void *B2, void *out,
                                         void *stream);

/*
 * Where the forward keeps its intermediates inside the workspace, for
 * diagnostics and per-kernel tests (byte offsets from the workspace start;
 * 0 bytes means absent).  Rows are the valid pairs in bucket order (the
 * unpadded order of moe_lora_align).
 */
typedef struct moe_lora_ws_layout {
    size_t compact_ids;      /* int32 [P]: pair id of each row */
    size_t compact_offset;   /* int32 [E*(L+1)+1]: first row of each bucket */
    size_t z1;               /* float [P][r]: gate_up LoRA shrink A1 x per row (rows of
                                adapter pairs only; other rows are left undefined) */
    size_t act;              /* bf16 [P][I]: SiLU(gate)*up per row */
    size_t z2;               /* float [P][r]: down LoRA shrink A2 act per row (same rows) */
    size_t pair_out;         /* w * d per pair id p: bf16 [P][H] when pair_out_bf16 (the down
                                GEMM does not split K: the activation type, rounded to nearest
                                even once), else float [down_splits][P][H], one slab per
                                K-split of the down GEMM (their sum is the pair's output) */
    int32_t s1, s2;          /* K-split counts the two shrinks used */
    int32_t down_splits;     /* K-splits of the down GEMM (>= 1) */
    int32_t launches;        /* kernels one forward launches for these dims (T > 0) */
    int32_t gemm_ctas;       /* CTAs per GEMM task: 2 on the CTA-pair kernel (wide chunks), else 1 */
    int32_t tc_expand;       /* 1: the LoRA expand runs as tensor-core K blocks of the base GEMMs;
                                0: on CUDA cores in the epilogue (or no adapters) */
    int32_t pair_out_bf16;   /* 1: pair_out holds bf16 (down_splits == 1); 0: fp32 slabs */
    size_t total;            /* == moe_lora_workspace_bytes */
} moe_lora_ws_layout;

/* Fills *out for dims d; returns a status.  Host only (reads the current
 * device's multiprocessor count when d->sm_count == 0, like
 * moe_lora_workspace_bytes). */
MOELORA_API int moe_lora_workspace_layout(const moe_lora_dims *d, moe_lora_ws_layout *out);

#ifdef __cplusplus
}
#endif

#endif /* MOE_LORA_H */
