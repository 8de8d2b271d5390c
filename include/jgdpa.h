/*
 * jgdpa.h - C ABI of libjgdpa.so: jagged Generalized Dot-Product Attention
 * (GDPA) forward and backward on one GB300 GPU (sm_103a).
 *
 * What is computed.  For every segment b and head h, with segment-local query
 * rows i < Lq_b and key/value rows j < Lkv_b, and valid(i,j) = (not causal or
 * j <= i):
 *
 *     x_ij = scale * <q_i, k_j> + bias[h][clamp(i - j, -R, R) + R]
 *     GELU / SiLU mode:  O_i = sum_{valid j} act(x_ij) * v_j   (no normalisation)
 *     SOFTMAX mode:      O_i = sum_{valid j} softmax_j(x_ij) * v_j,
 *                        LSE_i = log sum_{valid j} exp(x_ij)
 *
 * Sources: "GEM Training: How Meta Doubled the Efficiency of Its ..."
 * (globalainews.in), section "What to watch" -- self-attention, PMA and
 * cross-attention are two matrix multiplications with an element-wise
 * activation (GELU or SiLU) in place of softmax, unified in one GDPA kernel;
 * section "What happened" -- Jagged Flash Attention works directly on jagged
 * tensors with custom attention biases, asymmetric query/key-value lengths and
 * a backward pass.  "Meta redesigns AI training infrastructure to solve
 * trillion-parameter ad recommendation bottlenecks" (aiuniverse.news),
 * sections "Eliminating Compute Waste in Asymmetric Workloads" and "Custom
 * Kernels and 5D Parallelism for Trillion-Parameter Scale" -- the jagged
 * masking, the software tile scheduler and the split-dQ backward.
 *
 * The pages print no formula; where they are silent this library reads them
 * as follows: no normalisation in GELU/SiLU mode; GELU means x*Phi(x) (the
 * device evaluates an approximation of it); the bias is a per-head table of
 * bias_len = 2R+1 entries indexed by clamp(i-j, -R, R)+R with segment-local
 * i, j and is added after scaling; causal masking is top-left aligned
 * (j <= i); a query row with no valid key gets O_i = 0 (and LSE_i = -inf).
 *
 * Conventions shared by every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates and frees nothing and keeps no per-call state.
 *  - Calls are asynchronous and ordered on `stream`; they return before the
 *    kernels run.  The stream must belong to the current device.
 *  - Q, K, V, O and their gradients are bf16, packed "THD": [total][H][d],
 *    row-major, with no padding between segments.  The base pointers must be
 *    16-byte aligned.  Segment b owns query rows q_offsets[b] ..
 *    q_offsets[b+1]-1 and key/value rows kv_offsets[b] .. kv_offsets[b+1]-1.
 *  - Offsets are int32 [batch+1] device arrays with offsets[0] = 0,
 *    non-decreasing, and offsets[batch] equal to total_q (total_kv).
 *  - Outputs are overwritten, never accumulated; rows of segments with no keys
 *    (or no queries, for dK/dV) are written as zeros.
 *  - head_dim is 32, 64 or 128; heads >= 1; bias_len is 0 or odd (<= 4095).
 *  - Errors that the host can see are returned before anything is launched.
 *    Errors that only the device can see (bad offsets, an internal wait that
 *    timed out) are recorded in the workspace status word, turn the remaining
 *    kernels into no-ops, and are read back with jgdpa_read_device_status().
 *  - `workspace` is caller-owned device scratch of at least
 *    jgdpa_workspace_bytes(...) bytes, 256-byte aligned; its contents need no
 *    initialisation and are clobbered by every call.  Two calls that overlap
 *    in time must not share a workspace.
 */
#ifndef JGDPA_H
#define JGDPA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define JGDPA_API __attribute__((visibility("default")))
#else
#define JGDPA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* jgdpa_stream_t;  /* a cudaStream_t (NULL = legacy default stream) */

typedef enum {
    JGDPA_ACT_GELU = 0,     /* act(x) = x * Phi(x) */
    JGDPA_ACT_SILU = 1,     /* act(x) = x * sigmoid(x) */
    JGDPA_ACT_SOFTMAX = 2   /* Jagged Flash Attention: softmax over the valid keys */
} jgdpa_act;

typedef enum {
    JGDPA_OK = 0,
    JGDPA_ERR_INVALID_ARGUMENT = 1,   /* null pointer, negative size, bad enum, even bias_len */
    JGDPA_ERR_UNSUPPORTED = 2,        /* head_dim not in {32, 64, 128}, sizes beyond int32 rows */
    JGDPA_ERR_MISALIGNED = 3,         /* a tensor or the workspace is not suitably aligned */
    JGDPA_ERR_WORKSPACE_TOO_SMALL = 4,  /* workspace (or the no-alloc array) too small for the sizes */
    JGDPA_ERR_CUDA = 5,               /* a CUDA runtime call or launch failed */
    JGDPA_ERR_BAD_OFFSETS = 6,        /* device-detected: offsets not monotone / wrong ends */
    JGDPA_ERR_DEVICE_TIMEOUT = 7      /* device-detected: an internal wait gave up */
} jgdpa_status;

/*
 * Bytes of device workspace that jgdpa_fwd (for_backward = 0) or jgdpa_bwd
 * (for_backward = 1) needs for these sizes.  Depends only on the arguments
 * and on the number of SMs of the current device.  Returns 0 if the arguments
 * are invalid.
 */
JGDPA_API size_t jgdpa_workspace_bytes(int32_t batch, int64_t total_q, int64_t total_kv,
                             int32_t heads, int32_t head_dim, jgdpa_act act,
                             int32_t bias_len, int32_t for_backward);

/*
 * Forward pass.
 *   q        bf16 [total_q][heads][head_dim]
 *   k, v     bf16 [total_kv][heads][head_dim]
 *   scale    the factor s on <q_i, k_j> (typically 1/sqrt(head_dim))
 *   bias_table  fp32 [heads][bias_len], or NULL with bias_len = 0
 *   causal   0 or 1 (top-left aligned: key j is visible to query i iff j <= i)
 *   out      bf16 [total_q][heads][head_dim], written
 *   lse      fp32 [heads][total_q], natural-log log-sum-exp of each row;
 *            required in SOFTMAX mode (needed by jgdpa_bwd), must be NULL
 *            otherwise
 * Work runs in a persistent kernel over (segment, head, pair of 128-row query
 * tiles) units ordered longest first by a scheduling kernel (the software tile
 * scheduler of the GDPA kernel redesign, "Custom Kernels and 5D Parallelism
 * ...", aiuniverse.news).
 */
JGDPA_API jgdpa_status jgdpa_fwd(const void* q, const void* k, const void* v,
                       const int32_t* q_offsets, const int32_t* kv_offsets,
                       int32_t batch, int64_t total_q, int64_t total_kv,
                       int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                       const float* bias_table, int32_t bias_len, int32_t causal,
                       void* out, float* lse,
                       void* workspace, size_t workspace_bytes, jgdpa_stream_t stream);

/*
 * Forward pass with a sliding window: the same computation, arguments and
 * errors as jgdpa_fwd, plus
 *   window   0 (no window, exactly jgdpa_fwd) or w >= 1: only pairs with
 *            |i - j| < w (segment-local) are attended, on top of the
 *            length and causal conditions; negative -> INVALID_ARGUMENT.
 * Sliding window attention is named for long sequences in "Meta redesigns AI
 * training infrastructure ..." (aiuniverse.news), section "Custom Kernels
 * and 5D Parallelism ...", without a definition; this symmetric band, with
 * the same segment-local indices as the bias and causal rules, is the reading
 * taken.  Key/value tiles wholly outside the band are neither loaded nor
 * computed, and the scheduler costs units by the tiles they visit.  A query
 * row that meets no key gets O = 0 (and LSE = -inf in SOFTMAX mode).
 */
JGDPA_API jgdpa_status jgdpa_fwd_ex(const void* q, const void* k, const void* v,
                       const int32_t* q_offsets, const int32_t* kv_offsets,
                       int32_t batch, int64_t total_q, int64_t total_kv,
                       int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                       const float* bias_table, int32_t bias_len, int32_t causal, int32_t window,
                       void* out, float* lse,
                       void* workspace, size_t workspace_bytes, jgdpa_stream_t stream);

/*
 * Backward pass: gradients of L = sum(O * dout) with respect to q, k, v and
 * the bias table.
 *   out, lse   the forward's O and LSE; read in SOFTMAX mode only (may be NULL
 *              otherwise)
 *   dout       bf16 [total_q][heads][head_dim]
 *   dq         bf16 [total_q][heads][head_dim], written
 *   dk, dv     bf16 [total_kv][heads][head_dim], written
 *   dbias      fp32 [heads][bias_len], written; NULL to skip (must be NULL
 *              when bias_table is NULL)
 * dK/dV come from a KV-major pass and dQ from a separate Q-major pass, so
 * every output tile has exactly one writer and no atomics touch dQ, dK or dV
 * (the split-dQ, atomics-free backward of "Eliminating Compute Waste in
 * Asymmetric Workloads", aiuniverse.news).
 */
JGDPA_API jgdpa_status jgdpa_bwd(const void* q, const void* k, const void* v,
                       const void* out, const float* lse, const void* dout,
                       const int32_t* q_offsets, const int32_t* kv_offsets,
                       int32_t batch, int64_t total_q, int64_t total_kv,
                       int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                       const float* bias_table, int32_t bias_len, int32_t causal,
                       void* dq, void* dk, void* dv, float* dbias,
                       void* workspace, size_t workspace_bytes, jgdpa_stream_t stream);

/*
 * Bytes of stored-dS scratch that jgdpa_bwd_ex needs for these segment
 * lengths and window: heads * sum_b nk_b * span_b tiles of 32 KB, with
 * nq_b = ceil(Lq_b/128), nk_b = ceil(Lkv_b/128), and span_b = nq_b, or under
 * a window w > 0 the 2e + 1 query tiles one key tile can meet
 * (e = ceil((w - 1)/128)) when that is fewer.  q_offsets_host /
 * kv_offsets_host are HOST copies of the offsets ([batch + 1] each); window
 * as in jgdpa_bwd_ex.  Returns 0 for invalid arguments (and for batch 0).
 */
JGDPA_API size_t jgdpa_ds_scratch_bytes(const int32_t* q_offsets_host, const int32_t* kv_offsets_host,
                                        int32_t batch, int32_t heads, int32_t window);

/*
 * Backward pass, extended.  The same computation, arguments and errors as
 * jgdpa_bwd, plus:
 *   window
 *       0 (no window) or w >= 1: the sliding window of jgdpa_fwd_ex; pass
 *       the forward's window (and its out / lse in SOFTMAX mode).
 *   ds_scratch, ds_scratch_bytes
 *       optional caller-owned device scratch (256-byte aligned) for the
 *       stored-dS backward; NULL selects the recompute backward of
 *       jgdpa_bwd.  With scratch the dK/dV pass writes every bf16 dS tile it
 *       forms to the scratch and the dQ pass is one streaming matmul
 *       dQ = s * dS K over the stored tiles, instead of recomputing S, dP and
 *       the activation derivative.  jgdpa_ds_scratch_bytes(...) bytes hold
 *       every segment's tiles; a smaller scratch is used as far as it goes:
 *       the tiles are laid out segment by segment, the segments whose tiles
 *       end within the scratch get the stored-dS dQ and the others (a suffix
 *       of the batch) get their dQ by recomputation, so the results are the
 *       same up to rounding whatever the scratch size.  A scratch smaller
 *       than one tile (32 KB) is not used.  The scratch contents need no
 *       initialisation and are clobbered.
 *   pass_events
 *       optional three CUDA events (cudaEvent_t, created by the caller on the
 *       current device; any entry, or pass_events itself, may be NULL),
 *       recorded on `stream` right before the dK/dV pass kernel, between the
 *       dK/dV and dQ pass kernels, and right after the dQ pass kernel, so
 *       that cudaEventElapsedTime gives each pass's duration.
 */
JGDPA_API jgdpa_status jgdpa_bwd_ex(const void* q, const void* k, const void* v,
                       const void* out, const float* lse, const void* dout,
                       const int32_t* q_offsets, const int32_t* kv_offsets,
                       int32_t batch, int64_t total_q, int64_t total_kv,
                       int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                       const float* bias_table, int32_t bias_len, int32_t causal, int32_t window,
                       void* dq, void* dk, void* dv, float* dbias,
                       void* workspace, size_t workspace_bytes,
                       void* ds_scratch, size_t ds_scratch_bytes, jgdpa_stream_t stream,
                       void* const* pass_events);

/*
 * Shared query rows (PMA-style pooling): every segment attends with the same
 * n_shared = S query rows, e.g. learned seed queries shared across the batch
 * ("GEM Training: How Meta Doubled the Efficiency of Its ..."
 * (globalainews.in), section "What to watch": PMA is one of the modules GDPA
 * serves).  Segment b's query row i (0 <= i < S) is row i of q; its output,
 * upstream gradient and LSE rows are b S + i.  The computation is otherwise
 * that of jgdpa_fwd_ex / jgdpa_bwd_ex with Lq_b = S for every segment, and
 * the gradient of the shared rows is the sum over segments of each
 * segment's dQ.
 *   q          bf16 [S][heads][head_dim], read by every segment (not expanded)
 *   out, dout  bf16 [batch S][heads][head_dim]
 *   lse        fp32 [heads][batch S] (SOFTMAX mode only, else NULL)
 *   dq         bf16 [S][heads][head_dim], written: sum over b of dQ_b,
 *              accumulated in fp32 in a fixed order (the same bits on every
 *              run) and rounded once
 *   kv_offsets, k, v, dk, dv, bias_table, dbias, causal, window, ds_scratch,
 *   pass_events
 *              as in jgdpa_bwd_ex (there are no query offsets: they are S b,
 *              formed in the workspace; the stored-dS scratch size is
 *              jgdpa_ds_scratch_bytes with query offsets S b)
 * The workspace must hold jgdpa_shared_q_workspace_bytes(...) bytes; what
 * the backward keeps there depends on S:
 *   S <= 64 with GELU / SiLU: the short-query kernels (the keys take the
 *     MMA's 128 rows, the S queries are its N).  The backward writes one
 *     fp32 [S][head_dim] dQ contribution per (segment, head, chunk of up to
 *     16 key tiles) and sums them in a fixed order; ds_scratch is not used.
 *   S <= 128 and head_dim <= 64 otherwise: the key-major pass writes one such
 *     contribution per (segment, head, key tile); ds_scratch is not used.
 *   otherwise: each segment's dQ rows in fp32 ([batch S][heads][head_dim]),
 *     summed in segment order; ds_scratch as in jgdpa_bwd_ex.
 * Errors as in
 * jgdpa_fwd / jgdpa_bwd; n_shared < 1 is INVALID_ARGUMENT, batch S beyond
 * int32 is UNSUPPORTED.
 */
JGDPA_API size_t jgdpa_shared_q_workspace_bytes(int32_t batch, int32_t n_shared, int64_t total_kv,
                                                int32_t heads, int32_t head_dim, jgdpa_act act,
                                                int32_t bias_len, int32_t for_backward);
JGDPA_API jgdpa_status jgdpa_fwd_shared_q(const void* q, int32_t n_shared, const void* k, const void* v,
                                          const int32_t* kv_offsets, int32_t batch, int64_t total_kv,
                                          int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                                          const float* bias_table, int32_t bias_len, int32_t causal,
                                          int32_t window, void* out, float* lse,
                                          void* workspace, size_t workspace_bytes, jgdpa_stream_t stream);
JGDPA_API jgdpa_status jgdpa_bwd_shared_q(const void* q, int32_t n_shared, const void* k, const void* v,
                                          const void* out, const float* lse, const void* dout,
                                          const int32_t* kv_offsets, int32_t batch, int64_t total_kv,
                                          int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                                          const float* bias_table, int32_t bias_len, int32_t causal,
                                          int32_t window, void* dq, void* dk, void* dv, float* dbias,
                                          void* workspace, size_t workspace_bytes,
                                          void* ds_scratch, size_t ds_scratch_bytes, jgdpa_stream_t stream,
                                          void* const* pass_events);

/*
 * Forward pass without a caller-provided workspace: the same computation and
 * arguments as jgdpa_fwd minus (workspace, workspace_bytes).  There is no
 * counterpart on the pages; this entry point exists for callers that cannot
 * allocate device memory at call time -- for example a plugin interface that
 * hands over only input and output buffers, or a process whose device memory
 * is already fully reserved by another allocator, so that a cudaMalloc would
 * fail or force a synchronising reclaim.  The caller still owns and passes
 * every input and output.
 *
 * Scratch comes from a fixed array of JGDPA_NOALLOC_SCRATCH_BYTES (4 MiB)
 * compiled into the library; every GPU that loads the library holds that
 * array until the process exits.  Sizes whose scratch would not fit (about
 * 87,000 to 130,000 units of (segment, head, pair of 128-row query tiles),
 * depending on the segment lengths) are rejected with
 * JGDPA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  The address is kept for the life of the
 * process, so a device reset (cudaDeviceReset) after the first call on that
 * device is not supported: later calls would launch on the old address.  No call allocates or frees memory.  All calls
 * on a device share the one array and it keeps the previous call's contents
 * (the parts that must start at zero are cleared on the stream by each call):
 * calls that overlap in time on the GPU -- on different streams, or from
 * different host threads -- race on it and must be serialised by the caller.
 * Device-detected errors (bad offsets) leave the outputs unwritten and are not
 * reported by this entry point; use jgdpa_fwd to read them back.
 */
#define JGDPA_NOALLOC_SCRATCH_BYTES (4u << 20)
JGDPA_API jgdpa_status jgdpa_fwd_noalloc(const void* q, const void* k, const void* v,
                       const int32_t* q_offsets, const int32_t* kv_offsets,
                       int32_t batch, int64_t total_q, int64_t total_kv,
                       int32_t heads, int32_t head_dim, jgdpa_act act, float scale,
                       const float* bias_table, int32_t bias_len, int32_t causal,
                       void* out, float* lse, jgdpa_stream_t stream);

/*
 * Reads the device status word of `workspace` (synchronises `stream`) and
 * returns JGDPA_OK, a device-detected error, or JGDPA_ERR_CUDA.
 */
JGDPA_API jgdpa_status jgdpa_read_device_status(const void* workspace, jgdpa_stream_t stream);

/* Static, human-readable name of a status code. */
JGDPA_API const char* jgdpa_status_string(jgdpa_status s);

/*
 * Test hook: evaluates the device's own activation functions, exactly as the
 * forward and backward kernels use them, on n fp32 inputs.  act is GELU or
 * SiLU; y[i] = act(x[i]) and dy[i] = act'(x[i]) (dy may be NULL).  `path`
 * selects the evaluation route: 0 = the special-function-unit route (hardware
 * tanh), 1 = the ALU-only polynomial route, 2 = the exponential route
 * (hardware ex2, reciprocal on the FMA pipe; forward only, so its dy is the
 * route-0 derivative).  x, y, dy are device pointers.
 */
JGDPA_API jgdpa_status jgdpa_eval_activation(jgdpa_act act, int32_t path, const float* x, int64_t n,
                                   float* y, float* dy, jgdpa_stream_t stream);

/*
 * Test hook: sets how long one internal device wait of the kernels may take
 * before it gives up, for every kernel launched after this call in this
 * process (any device, any stream); 0 restores the default of 2 s.  A wait
 * that gives up records JGDPA_ERR_DEVICE_TIMEOUT in the workspace status word;
 * the CTA then waits (at most 200 ms each) for its copies and tensor-core
 * operations in flight, releases its Tensor Memory and exits, and the later
 * kernels of the call do nothing.  A limit of a few nanoseconds makes the
 * waits of any multi-tile call run out, which is how the timeout path is
 * tested without faulting or hanging a GPU.  Not thread-safe with respect to
 * calls in flight on other host threads (they may see either value).
 */
JGDPA_API void jgdpa_set_wait_limit_ns(uint64_t limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* JGDPA_H */
