/*
 * lwm_attn.h - C ABI for exact causal, segment-masked (packed) softmax attention on
 * NVIDIA B300 (sm_103a).
 *
 * What is computed. The operation is the attention primitive of "World Model on
 * Million-Length Video And Language With Blockwise RingAttention" (LWM), as the
 * charles2530.github.io deep-dive page describes it:
 *   - section "RingAttention 为什么必要": exact full attention (no window, no sparse
 *     approximation), computed block by block so that memory stays linear in S;
 *   - section "模型结构": next-token prediction, hence causal attention;
 *   - section "Masked sequence packing": several documents share one packed row and
 *     an attention mask lets each attend only to itself.
 * For batch row b, head h and query i (0-based), with seg = seg_ids[b, :]:
 *     visible(i)  = { j : seg[j] == seg[i] >= 0 and j <= i }
 *     s_ij        = (q_i . k_j) / sqrt(D)
 *     lse_i       = ln sum_{j in visible(i)} exp(s_ij)
 *     out_i       = sum_{j in visible(i)} exp(s_ij - lse_i) v_j
 * and the backward pass returns dq, dk, dv of L = sum(dout * out). The softmax scale
 * is fixed at 1/sqrt(D). Rows whose segment id is negative (padding) see nothing:
 * out = 0, lse = -inf, and they receive and contribute zero gradient.
 *
 * Layouts (all dense, row-major, device memory):
 *   q, k, v, out, dout, dq, dk, dv : bf16  [B, S, H, D]  (D fastest)
 *   lse                            : fp32  [B, H, S]     (natural log)
 *   seg_ids, pos                   : int32 [B, S]
 * Preconditions on seg_ids / pos, per batch row:
 *   - documents are contiguous runs with non-decreasing ids >= 0, optionally followed
 *     by one trailing run of negative ids (padding);
 *   - pos[b, i] is the offset of token i inside its document (0, 1, 2, ... restarting
 *     at each document). Position entries of padding tokens are ignored.
 *   seg_ids == NULL means one document per row; pos == NULL means pos is derived
 *   from seg_ids. Violations are detected on the device and reported by
 *   lwm_attn_check() as LWM_ERR_SEGMENTS; the outputs of such a call are undefined.
 *
 * Ownership and synchronisation. The caller owns every buffer, including the
 * workspace (size from lwm_attn_workspace_size()). The library never allocates or
 * frees device memory and never synchronises, except in lwm_attn_check(). Every
 * call only enqueues work on `stream`; calls that share one workspace must be
 * ordered (same stream, or synchronised by the caller).
 *
 * Errors. Host-side argument errors return a status and enqueue nothing. Device-side
 * conditions (inconsistent seg/pos, an internal wait that timed out) set an error
 * word in the workspace that lwm_attn_check() returns and clears.
 *
 * Supported: D == 128 only; all pointers 16-byte aligned; 1 <= S, B, H; B*S*H*D
 * below 2^31 elements per tensor dimension product as TMA coordinates allow.
 */
#ifndef LWM_ATTN_H
#define LWM_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* bfloat16 storage (the raw 16-bit pattern). */
typedef uint16_t lwm_bf16;
/* A CUDA stream; the same type as cudaStream_t (NULL = legacy default stream). */
typedef struct CUstream_st *lwm_stream;

typedef enum {
  LWM_OK = 0,
  LWM_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, too-small workspace */
  LWM_ERR_UNSUPPORTED = 2,  /* D != 128, or no sm_100-family device */
  LWM_ERR_ALIGNMENT = 3,    /* a pointer is not 16-byte aligned */
  LWM_ERR_SEGMENTS = 4,     /* device: seg_ids / pos break the preconditions above */
  LWM_ERR_WORKSPACE = 5,    /* workspace not 256-byte aligned */
  LWM_ERR_CUDA = 6,         /* a CUDA runtime or driver call failed */
  LWM_ERR_TIMEOUT = 7,      /* device: an internal pipeline wait exceeded its bound */
  LWM_ERR_LENGTHS = 8,      /* device: a decode kv_len outside [T, S_max] */
  LWM_ERR_TARGETS = 9       /* device: a packed-loss target outside [0, V) on a weighted token */
} lwm_status;

/* Bytes of device workspace needed for problems of this shape (0 on bad sizes).
 * The workspace holds the per-token segment starts, per-tile ranges, the schedule's
 * work lists and tickets, the error word, the backward row dots (fp32 [B,H,S]) and,
 * at its end, the fp32 dQ accumulator of the single-kernel backward pass
 * (4 * B * H * S * D bytes, S rounded up to a multiple of 128). */
size_t lwm_attn_workspace_size(int B, int S, int H, int D);

/* The leading part of that workspace which every call except the single-kernel
 * backward stage LWM_BWD_FUSED uses (no dQ accumulator): enough for lwm_attn_prepare,
 * the forward entry points, lwm_attn_bwd, lwm_attn_bwd_prepared and the LWM_BWD_DELTA /
 * LWM_BWD_DKDV / LWM_BWD_DQ stages. */
size_t lwm_attn_workspace_size_fwd(int B, int S, int H, int D);

/* Metadata pre-pass alone: validates seg_ids/pos and writes segment starts, per-tile
 * key/query ranges and longest-first work lists into `workspace`. The *_prepared
 * calls below reuse it, so one prepare serves every layer that shares a packing.
 * kv_chunks >= 1 sets the ring order of the forward pass (see lwm_attn_fwd_ring). */
lwm_status lwm_attn_prepare(const int32_t *seg_ids, const int32_t *pos, int B, int S, int H, int D,
                            int kv_chunks, void *workspace, size_t workspace_bytes, lwm_stream stream);

/* Forward pass: metadata pre-pass, then the persistent tensor-core kernel.
 * Writes out [B,S,H,D] bf16 and lse [B,H,S] fp32. */
lwm_status lwm_attn_fwd(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                        const int32_t *seg_ids, const int32_t *pos, lwm_bf16 *out, float *lse,
                        int B, int S, int H, int D, void *workspace, size_t workspace_bytes,
                        lwm_stream stream);

/* Forward pass with the key/value blocks visited in ring order: the sequence is cut
 * into kv_chunks equal chunks (the blocks that the devices of a ring would hold,
 * LWM deep-dive page, section "RingAttention 为什么必要"), and a query block in chunk
 * r visits chunks r, r-1, ..., 0, all inside one launch on one GPU. The result equals
 * lwm_attn_fwd's up to floating-point rounding order. */
lwm_status lwm_attn_fwd_ring(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                             const int32_t *seg_ids, const int32_t *pos, lwm_bf16 *out, float *lse,
                             int B, int S, int H, int D, int kv_chunks, void *workspace,
                             size_t workspace_bytes, lwm_stream stream);

/* Forward pass reusing the metadata of a previous lwm_attn_prepare (same B, S and
 * segments) held in `workspace`. */
lwm_status lwm_attn_fwd_prepared(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                                 lwm_bf16 *out, float *lse, int B, int S, int H, int D,
                                 void *workspace, size_t workspace_bytes, lwm_stream stream);

/* Backward pass: metadata pre-pass, the row-dot pre-pass delta_i = dout_i . out_i,
 * then the dK/dV kernel and the dQ kernel (LWM_BWD_ALL below). `out` and `lse` are the
 * forward outputs. dq, dk, dv are fully overwritten (no accumulation into existing
 * values) and bitwise reproducible. */
lwm_status lwm_attn_bwd(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                        const lwm_bf16 *out, const lwm_bf16 *dout, const float *lse,
                        const int32_t *seg_ids, const int32_t *pos,
                        lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv,
                        int B, int S, int H, int D, void *workspace, size_t workspace_bytes,
                        lwm_stream stream);

/* Backward pass reusing the metadata of a previous lwm_attn_prepare in `workspace`
 * (same stages as lwm_attn_bwd: LWM_BWD_ALL). */
lwm_status lwm_attn_bwd_prepared(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                                 const lwm_bf16 *out, const lwm_bf16 *dout, const float *lse,
                                 lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv,
                                 int B, int S, int H, int D, void *workspace, size_t workspace_bytes,
                                 lwm_stream stream);

/* Stages of the backward pass, for lwm_attn_bwd_stages (a bit mask). */
typedef enum {
  LWM_BWD_DELTA = 1,  /* row dots delta = rowsum(dout * out) and lse rows, into the workspace */
  LWM_BWD_DKDV = 2,   /* dk, dv (needs LWM_BWD_DELTA's results in the workspace) */
  LWM_BWD_DQ = 4,     /* dq (needs LWM_BWD_DELTA's results in the workspace) */
  LWM_BWD_ALL = 7,    /* the three stages above: every gradient bitwise reproducible */
  LWM_BWD_FUSED = 8   /* dk, dv and dq in one kernel from one recomputation of the
                         probabilities (5 tensor-core products per tile pair instead of
                         7): dq is accumulated in fp32 in the workspace's dQ accumulator
                         (zeroed by the stage itself) and then converted to bf16, in an
                         order that depends on scheduling (dq is not bitwise reproducible;
                         dk, dv are). Needs LWM_BWD_DELTA's results and the whole
                         lwm_attn_workspace_size() workspace; cannot be combined with DKDV
                         or DQ. On B300 it is slower than DKDV + DQ: moving dQ out through
                         shared memory competes with the tensor core for bandwidth */
} lwm_bwd_stage;

/* Runs the selected backward stages in the order delta, fused, dK/dV, dQ, reusing the
 * metadata of a previous lwm_attn_prepare. After the delta stage has completed, the
 * dK/dV and dQ stages only read the workspace (each has its own scheduler ticket), so
 * a caller may run them on two streams. Pointers that no selected stage touches may
 * be NULL (delta: out, dout, lse; dK/dV: q, k, v, dout, dk, dv; dQ: q, k, v, dout,
 * dq; fused: q, k, v, dout, dq, dk, dv). The workspace needs lwm_attn_workspace_size()
 * bytes when LWM_BWD_FUSED is selected, lwm_attn_workspace_size_fwd() bytes otherwise. */
lwm_status lwm_attn_bwd_stages(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                               const lwm_bf16 *out, const lwm_bf16 *dout, const float *lse,
                               lwm_bf16 *dq, lwm_bf16 *dk, lwm_bf16 *dv,
                               int B, int S, int H, int D, unsigned stages, void *workspace,
                               size_t workspace_bytes, lwm_stream stream);

/* Rotary position embedding (RoPE) of q and k: the positional encoding whose base theta
 * LWM raises with the context length (deep-dive page, section "Stage I：长上下文语言模型";
 * Tables 11 and 13: theta = 1M at 32K tokens, 10M at 128K/256K, 25M at 512K, 50M at 1M
 * and in the vision-language stages). The pages name RoPE without a formula; this is
 * RoPE's published definition: for the token at position p = pos[b, i] and each
 * adjacent pair (2m, 2m+1) of every head vector, m = 0 .. D/2 - 1,
 *     angle     = p * theta^(-2m/D)
 *     y[2m]     = x[2m] cos(angle) - x[2m+1] sin(angle)
 *     y[2m+1]   = x[2m] sin(angle) + x[2m+1] cos(angle)
 * With inverse = 1 the pairs are rotated by -angle (the transpose): applied to the
 * gradients with respect to the rotated q and k, it gives the gradients with respect
 * to the unrotated ones. Attention with RoPE is therefore: rotate q and k, run
 * lwm_attn_fwd / lwm_attn_bwd on the rotated tensors (keep them for the backward
 * pass), then rotate dq and dk back with inverse = 1.
 *   q, k, q_out, k_out : bf16 [B, S, H, D]; either tensor may be skipped (q and q_out
 *                        both NULL, or k and k_out both NULL), not both; q_out == q
 *                        (in place) is allowed, other overlaps are not.
 *   pos                : int32 [B, S] positions (for packed rows: the offset inside the
 *                        document, as for lwm_attn_fwd); NULL means pos = i, the index
 *                        in the row.
 *   theta              : the base, > 0 and finite.
 * Angles are reduced in double precision, sin/cos and the rotation run in fp32, and the
 * result is rounded to bf16. Errors: LWM_ERR_INVALID_ARG (sizes, theta, inverse not
 * 0/1, pointer pairs), LWM_ERR_UNSUPPORTED (D != 128), LWM_ERR_ALIGNMENT (tensors not
 * 16-byte or pos not 4-byte aligned). Memory-bound: reads and writes each element
 * once. */
lwm_status lwm_attn_rope(const lwm_bf16 *q, const lwm_bf16 *k, const int32_t *pos, double theta,
                         lwm_bf16 *q_out, lwm_bf16 *k_out, int B, int S, int H, int D, int inverse,
                         lwm_stream stream);

/* Attention of a few new tokens against a long key/value cache (decoding): the
 * inference side of the 1M-token context (deep-dive page, section "RingAttention
 * 为什么必要": 1M-token inference needs at least a v4-128 with 32-way tensor and 4-way
 * sequence parallelism). Exactly the same attention as lwm_attn_fwd, for the last T
 * positions of each row only:
 *   q       : bf16 [B, T, H, D], the queries of the T newest tokens of each row;
 *   k_cache, v_cache : bf16 [B, S_max, H, D] (the layout of lwm_attn_fwd's k, v); row b
 *             holds kv_len[b] valid tokens, the T new ones last (positions
 *             kv_len[b] - T .. kv_len[b] - 1);
 *   kv_len  : int32 [B] on the device, T <= kv_len[b] <= S_max (NULL: all S_max);
 *   out     : bf16 [B, T, H, D];  lse : fp32 [B, H, T] (natural log).
 * Query t of row b (at position P = kv_len[b] - T + t) attends causally to keys
 * 0 .. P of its row: one document per row (no segments).
 * The cache is cut into splits of equal length; each split's partial softmax
 * (running max, sum and unnormalised output) is computed by its own CTA, which stages
 * the cache through shared memory with bulk copies, and a second kernel merges the
 * partials by their log-sum-exp: out = sum_s exp(lse_s - lse) out_s. Memory-bound: the
 * cache is read once. 1 <= T <= 4. The workspace (caller-owned, zero-filled once like
 * every workspace of this library) holds the partials and an error word:
 * lwm_attn_decode_workspace_size bytes. A kv_len outside [T, S_max] is reported by
 * lwm_attn_check as LWM_ERR_LENGTHS (that row's outputs are zero). */
size_t lwm_attn_decode_workspace_size(int B, int T, int S_max, int H, int D);

lwm_status lwm_attn_decode(const lwm_bf16 *q, const lwm_bf16 *k_cache, const lwm_bf16 *v_cache,
                           const int32_t *kv_len, lwm_bf16 *out, float *lse, int B, int T, int S_max, int H,
                           int D, void *workspace, size_t workspace_bytes, lwm_stream stream);

/* Re-weighted cross-entropy of a packed batch: the loss of masked sequence packing
 * (deep-dive page, section "Masked sequence packing": besides the attention mask, LWM
 * re-weights the loss so that packed training equals non-packed + padding training;
 * otherwise the token count of long video samples drowns short answers). The pages
 * give no formula; the reading here: non-packed, each document is its own row whose
 * loss is the weighted mean of its token losses, and the batch loss is the mean over
 * those rows. With documents d (the contiguous runs of equal seg_ids >= 0, as for the
 * attention), token weights w_t >= 0 and token losses l_t:
 *     loss = (1/N) sum_d ( sum_{t in d} w_t l_t ) / n_d,    n_d = sum_{t in d} w_t,
 *     N = number of documents with n_d > 0,  l_t = log sum_v exp(z_t[v]) - z_t[y_t],
 *     dlogits_t = w_t / (N n_d) (softmax(z_t) - onehot(y_t)).
 *   logits  : bf16 [B, S, V] (V a multiple of 8), z_t = logits[b, i, :];
 *   targets : int32 [B, S], y_t (only read where w_t > 0; must lie in [0, V));
 *   weight  : fp32 [B, S] or NULL (1 everywhere); 0 = no loss on that token (e.g. the
 *             last token of each document, whose next token belongs to another one);
 *             negative or non-finite weights count as 0. Padding tokens (seg < 0)
 *             carry no loss;
 *   seg_ids : int32 [B, S] or NULL (one document per row);
 *   loss    : one double on the device (the loss);
 *   dlogits : bf16 [B, S, V] or NULL (loss only); fully written (zeros where w_t = 0).
 * Memory-bound: the logits are read once from HBM (a second pass for the gradient
 * hits L2) and the gradient written once. The loss is summed in a fixed order
 * (reproducible); the per-document weight sums add fp64 terms atomically, exact for
 * integer weights such as 0/1 masks. Workspace: lwm_packed_loss_workspace_size bytes,
 * caller-owned. Device-side errors (seg_ids breaking the packing preconditions, a
 * target outside [0, V)) are returned by lwm_attn_check(workspace) as LWM_ERR_SEGMENTS
 * / LWM_ERR_TARGETS. Host-side: LWM_ERR_INVALID_ARG (sizes, NULLs, small workspace),
 * LWM_ERR_UNSUPPORTED (V not a multiple of 8), LWM_ERR_ALIGNMENT (logits / dlogits not
 * 16-byte, targets / weight / seg_ids not 4-byte, loss not 8-byte aligned),
 * LWM_ERR_WORKSPACE (not 256-byte aligned). */
size_t lwm_packed_loss_workspace_size(int B, int S);

lwm_status lwm_packed_loss(const lwm_bf16 *logits, const int32_t *targets, const float *weight,
                           const int32_t *seg_ids, double *loss, lwm_bf16 *dlogits, int B, int S, int V,
                           void *workspace, size_t workspace_bytes, lwm_stream stream);

/* Bytes of the library's own device scratch array used by lwm_attn_fwd_noalloc. */
#define LWM_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Forward pass for callers that cannot allocate device memory. This entry point has
 * no counterpart in the LWM pages; it exists for callers with no way to obtain a
 * workspace: a plug-in inside a host framework that owns all device memory and hands
 * its plug-ins only their tensors, or a latency-critical caller that must not call
 * cudaMalloc because cudaMalloc may synchronise the whole device.
 *
 * It computes exactly what lwm_attn_fwd computes (same kernels), with the workspace
 * replaced by a 16 MiB device array (LWM_NOALLOC_SCRATCH_BYTES) that the library
 * declares at file scope: every GPU on which the library is loaded holds that array
 * until the process exits. The caller still passes inputs and outputs. Nothing is
 * allocated or freed: no cudaMalloc, cudaFree or allocating library routine.
 *   - Limit: the forward part of the workspace for (B, S) must fit the array, which
 *     holds about 12 bytes per token: B * S up to about 1.3 million tokens (S rounded
 *     up per row to a multiple of 128). Larger problems return LWM_ERR_INVALID_ARG
 *     before anything is enqueued.
 *   - Set-up: the first call on a device looks up the array's device address with
 *     cudaGetSymbolAddress (with that device current) and caches it; make that first
 *     call before any stream capture.
 *   - Sharing: all calls on a device share the one array and it keeps the last call's
 *     contents; each call clears the words that must start at zero. Calls that overlap
 *     on the GPU (different streams, or several host threads) race on the array and
 *     must be serialised by the caller.
 *   - Errors: argument errors are returned as by lwm_attn_fwd. Device-side conditions
 *     (seg_ids / pos that break the preconditions, and a bounded pipeline wait that ran
 *     out) are not reported, because the error word lives in the shared array and no
 *     call returns it; the outputs of such a call are undefined.
 *   - Context: the cached address belongs to the device's primary runtime context; it
 *     assumes that context lives as long as the process (no cudaDeviceReset). */
lwm_status lwm_attn_fwd_noalloc(const lwm_bf16 *q, const lwm_bf16 *k, const lwm_bf16 *v,
                                const int32_t *seg_ids, const int32_t *pos, lwm_bf16 *out, float *lse,
                                int B, int S, int H, int D, lwm_stream stream);

/* Synchronises `stream`, then returns and clears the device error word held in
 * `workspace` (LWM_OK, LWM_ERR_SEGMENTS, LWM_ERR_LENGTHS, LWM_ERR_TARGETS or
 * LWM_ERR_TIMEOUT), or LWM_ERR_CUDA if the stream reported a CUDA error. */
lwm_status lwm_attn_check(void *workspace, lwm_stream stream);

/* Bound of the kernels' pipeline waits, for tests of the failure path. Every wait of a
 * kernel role on another (an mbarrier phase, a counter) gives up after a bound of wall
 * time, sets LWM_ERR_TIMEOUT in the workspace's error word, and the kernel lets copies
 * and products in flight land, frees its tensor memory and returns, so the CUDA
 * context stays usable. The default bound is 2 s, far above any legitimate wait. This
 * call sets the bound for every kernel this process launches afterwards, on any
 * device and stream (0 restores the default; it is read when a call launches its
 * kernels). A bound below 1 ms is a test setting: each kernel's producer then also
 * waits once, with its first copies in flight, for a phase that never completes, so a
 * bound of a few nanoseconds makes that wait run out for certain; a test can then check
 * that lwm_attn_check() returns LWM_ERR_TIMEOUT and that the next call with the default
 * bound still computes correct results. The waits that let in-flight work land keep the
 * default bound. Source: none on the LWM pages (failure handling of this library).
 * Always returns LWM_OK. */
lwm_status lwm_attn_set_wait_limit(uint64_t limit_ns);

/* Description of the most recent LWM_ERR_CUDA raised on the calling host thread: the
 * failing call and the CUDA error text ("" if none). The string is owned by the
 * library and stays valid until the thread's next failing call. */
const char *lwm_last_error(void);

/* Static, human-readable name of a status code. */
const char *lwm_status_string(lwm_status status);

#ifdef __cplusplus
}
#endif

#endif /* LWM_ATTN_H */
