/* Exact tiled attention for GB300 (sm_103a): the C ABI.
 *
 * What the library computes, for every batch b and head h (all tensors
 * contiguous, layout (B, H, N, d), d innermost):
 *
 *     O = softmax(scale * Q K^T  [+ causal mask]) V,   LSE_i = ln sum_j exp(scale * q_i . k_j)
 *
 * the definition of wiki.ai-engineering.at "Flash Attention" (section "Das
 * Grundproblem") and johe.ru "Flash Attention: ускорить attention в 6 раз без
 * потери точности" (section "Введение").  It is evaluated tile by tile with the
 * online-softmax recurrence of the first page (section "Lösung: Online
 * Softmax"), so the N x N score matrix never exists in device memory.  The
 * result equals standard attention up to floating-point rounding; only the
 * order of operations differs (second page, "Почему это точно?").
 *
 * Conventions shared by every entry point:
 *  - q, k, v, o, dO, dq, dk, dv, caches: bf16 (__nv_bfloat16) device pointers,
 *    16-byte aligned, contiguous (B, H, N, d); d is 64 or 128.
 *  - lse, D and every workspace: fp32 device pointers, 16-byte aligned.
 *  - scale is passed explicitly (1/sqrt(d) is the usual choice); it must be
 *    finite and > 0.
 *  - causal: 0 or 1.  The mask is aligned bottom-right: query i sees key j iff
 *    j <= i + (Nk - Nq).  A query that sees no key gets O = 0, LSE = -inf and
 *    zero gradients.
 *  - stream: a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every call is asynchronous on it; nothing is synchronised.  Kernels are
 *    launched as programmatic dependents of the work before them on the stream
 *    (their setup may overlap its end), but each waits for that work to
 *    complete before it reads or writes any buffer, so stream order holds as
 *    for ordinary launches.
 *  - Ownership: the caller allocates and owns every buffer, workspaces
 *    included.  The library allocates no device memory and keeps no state
 *    besides a device-side error word and host-side caches (the tensor-map
 *    encoder's entry point, each device's SM count, and which kernels'
 *    shared-memory limits have been raised on which device).
 *  - Errors: return codes only (fa_status); arguments are validated before
 *    anything is launched, and an invalid call launches nothing.  No fallback
 *    implementation exists: an unsupported shape is an error, never a slower
 *    path.  Device-side waits are bounded; a wait that runs out records
 *    FA_ERR_TIMEOUT in the error word, the kernel releases what it holds and
 *    returns, and fa_get_last_device_error() reports it.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, bad scale or flag */
    FA_ERR_UNSUPPORTED = -2, /* d not in {64, 128}, sizes beyond 32-bit tile indexing */
    FA_ERR_ALIGNMENT = -3,   /* a pointer not 16-byte aligned */
    FA_ERR_WORKSPACE = -4,   /* workspace null or smaller than the *_workspace_bytes query */
    FA_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed (launch, tensor map) */
    FA_ERR_TIMEOUT = -6      /* a device-side bounded wait ran out (see fa_get_last_device_error) */
} fa_status;

/* Forward pass (tiled attention with online softmax, one fused kernel).
 * q [B,H,Nq,d], k/v [B,H,Nk,d] bf16 in; o [B,H,Nq,d] bf16 and lse [B,H,Nq]
 * fp32 out (natural log of the row's sum of exp(scale * q.k)).  Source: the
 * "Tiling Algorithm" and "Lösung: Online Softmax" sections of
 * wiki.ai-engineering.at "Flash Attention"; each output row leaves the chip
 * exactly once (johe.ru, section "Проблема 2: DRAM bottleneck", the count of
 * memory round trips).  Requires B, H, Nq, Nk >= 1. */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int H, int Nq, int Nk, int d, float scale, int causal, void *stream);

/* Query rows per work tile fa_fwd takes for these sizes on the current device:
 * 256 (two 128-row query tiles share every key/value block) or 128 (split-KV
 * tiles: the key blocks of one 128-row tile alternate between two softmax
 * groups, merged at the end with the log-sum-exp weights, the combine of
 * wiki.ai-engineering.at "Flash Attention", section "Lösung: Online
 * Softmax").  The choice minimises the busiest SM's share of a static
 * persistent schedule; it only changes the rounding order.  Returns a negative
 * fa_status for invalid sizes or no usable device.  Host-only; launches
 * nothing. */
int fa_fwd_tile_rows(int B, int H, int Nq, int Nk, int d, int causal);

/* The static schedule of the persistent grids (the forward's work tiles, the
 * backward's key and query tiles): n_items work items listed in chunks of
 * chunk_items (heads whose streamed operands fit in L2 together), taken by
 * `grid` CTAs.  per_chunk != 0 (causal lists, heaviest item first in each
 * chunk): each chunk in its own rounds of alternating direction, odd chunks
 * starting reversed; otherwise, or when a chunk is smaller than the grid,
 * rounds of alternating direction over the whole list.  Writes owner[i] = the
 * CTA that takes item i (owner: n_items ints, host memory).  Returns FA_OK,
 * FA_ERR_INVALID_ARG for bad sizes or a null owner, or FA_ERR_INVALID_ARG if
 * an item would be taken twice (never: the schedule is a partition).
 * Host-only; launches nothing. */
int fa_work_schedule(int n_items, int chunk_items, int grid, int per_chunk, int *owner);

/* Causal sliding-window forward: like fa_fwd with causal = 1, except that
 * query i sees only the `window` (>= 1) keys ending at its diagonal, keys j
 * with i + Nk - Nq - window < j <= i + Nk - Nq (the fixed-window local
 * attention of johe.ru "Flash Attention: ...", section "Альтернативы").  Only
 * the key blocks inside a tile's window are loaded and multiplied. */
int fa_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                  int B, int H, int Nq, int Nk, int d, float scale, int window, void *stream);

/* Forward over a padded batch of sequences of different lengths (a mask
 * variant of fa_fwd: zimaspace.com "Wie reduziert Flash Attention ...",
 * masking is applied to the tile scores before the softmax).  seqlens_q and
 * seqlens_k are device int32 [B]: sequence b has seqlens_q[b] <= Nq query
 * rows and seqlens_k[b] <= Nk keys, stored in the first rows of its
 * [H, Nq, d] / [H, Nk, d] slices.  Row i < seqlens_q[b] attends to keys
 * j < seqlens_k[b] (causal: also j <= i + seqlens_k[b] - seqlens_q[b]).  Rows
 * past seqlens_q[b] get O = 0 and LSE = -inf.  Query and key tiles wholly past a
 * sequence are skipped.  Padding positions of q, k and v must hold finite
 * values (their contents do not change the result).  A length outside
 * [0, Nq] / [0, Nk] is clamped and recorded as FA_ERR_INVALID_ARG in the
 * device error word.  Other conventions as fa_fwd; both length pointers are
 * required (FA_ERR_INVALID_ARG if null) and 4-byte aligned. */
int fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                  const int *seqlens_q, const int *seqlens_k,
                  int B, int H, int Nq, int Nk, int d, float scale, int causal, void *stream);

/* Bytes of workspace fa_fwd_fp8 needs: a transposed copy of V,
 * [B*H, 128, Nk rounded up to 16] bytes.  Returns 0 for invalid sizes. */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int Nk, int d);

/* FP8 forward with block scales (johe.ru "Flash Attention: ...", sections
 * "Flash Attention 3": block-scaled attention, and "Flash Attention 4": FP8).
 * q [B,H,Nq,128], k and v [B,H,Nk,128] as e4m3 bytes (OCP FP8, no infinities).
 * The value an element stands for is its e4m3 value times its scale:
 *  q_scale fp32 [B*H, ceil(Nq/128)]: one per 128-row block of q;
 *  k_scale fp32 [B*H, ceil(Nk/128)]: one per 128-row block of k;
 *  v_scale fp32 [B*H]: one per head of v.
 * Computes the forward of fa_fwd on those values: o [B,H,Nq,128] bf16 and lse
 * [B,H,Nq] fp32.  Scores accumulate in fp32.  P = exp(S - m) is rounded to
 * e4m3 (relative error <= 2^-4, or 2^-10 absolute below 2^-6) for the value
 * product, and the result is multiplied by v_scale / l.  d must be 128
 * (FA_ERR_UNSUPPORTED otherwise).  workspace: at least
 * fa_fwd_fp8_workspace_bytes(B,H,Nk,d) bytes, 16-byte aligned; it receives V^T
 * (one extra pass over V) so that both products take K-major operands. */
int fa_fwd_fp8(const void *q, const void *k, const void *v, const float *q_scale, const float *k_scale,
               const float *v_scale, void *o, float *lse, int B, int H, int Nq, int Nk, int d, float scale,
               int causal, void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of fp32 workspace fa_bwd needs: the row terms D [B,H,Nq] (dQ is
 * accumulated on chip, in a pass of its own).  Returns 0 for invalid sizes. */
size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/* Backward pass (johe.ru, section "Стадии вычисления", pass 2: gradients are
 * recomputed from the same tiles, P is rebuilt from the saved LSE instead of
 * being stored).  Inputs: q, k, v, o (the forward output), lse (the forward's
 * LSE), dO [B,H,Nq,d] the upstream gradient.  Outputs dq [B,H,Nq,d],
 * dk/dv [B,H,Nk,d] bf16.  Steps: D_i = sum_c dO_ic O_ic (fp32); per key tile,
 * S = scale QK^T recomputed, P = exp(S - LSE), dV += P^T dO, dP = dO V^T,
 * dS = P (dP - D), dK += scale dS^T Q; per query tile, dQ += scale dS K.  All
 * accumulation is fp32 on chip; each gradient is rounded to bf16 once.  The
 * result is deterministic (no atomics).  workspace must hold at least
 * fa_bwd_workspace_bytes(B,H,Nq,Nk,d) bytes; its contents on entry do not
 * matter. */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dO, void *dq, void *dk, void *dv,
           int B, int H, int Nq, int Nk, int d, float scale, int causal,
           void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace fa_bwd_fused needs: D [B,H,Nq] as for fa_bwd, then an
 * fp32 dQ accumulator [B,H,Nq,d].  Returns 0 for invalid sizes and for
 * d != 128. */
size_t fa_bwd_fused_workspace_bytes(int B, int H, int Nq, int Nk, int d);

/* The same backward as fa_bwd (same arguments, outputs and tolerance) in one
 * pass over the key tiles instead of two: besides dK and dV, each 128-key
 * CTA computes its share of dQ = scale dS K as dQ^T = K^T dS^T on the tensor
 * cores and adds it to the fp32 accumulator in the workspace with reduce-adds,
 * so S and dP are rebuilt once per tile pair instead of twice (johe.ru, section
 * "Стадии вычисления", pass 2; the dQ product is one of the five).  The order
 * of those fp32 additions varies from run to run, so dq is not bit-for-bit
 * reproducible (dk and dv are).  Launches: the preprocess (which also zeroes
 * the accumulator), the pass, and a conversion of the accumulator to bf16 dq.
 * d = 128 only (FA_ERR_UNSUPPORTED otherwise).  workspace must hold at least
 * fa_bwd_fused_workspace_bytes(B,H,Nq,Nk,d) bytes, 16-byte aligned; its
 * contents on entry do not matter. */
int fa_bwd_fused(const void *q, const void *k, const void *v, const void *o, const float *lse,
                 const void *dO, void *dq, void *dk, void *dv,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Backward of fa_fwd_window (same window, same conventions as fa_bwd). */
int fa_bwd_window(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dO, void *dq, void *dk, void *dv,
                  int B, int H, int Nq, int Nk, int d, float scale, int window,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Backward of fa_fwd_varlen (same lengths, same conventions as fa_bwd).
 * Gradient rows past a sequence's length (dq past seqlens_q[b], dk and dv
 * past seqlens_k[b]) are written as zeros.  dO must be finite in padding rows
 * too; lse is fa_fwd_varlen's (-inf in padding rows). */
int fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o, const float *lse,
                  const void *dO, void *dq, void *dk, void *dv,
                  const int *seqlens_q, const int *seqlens_k,
                  int B, int H, int Nq, int Nk, int d, float scale, int causal,
                  void *workspace, size_t workspace_bytes, void *stream);

/* The three steps of fa_bwd, for callers that schedule them (or time them)
 * separately; fa_bwd is exactly these three launches in this order, except
 * that it launches each as a programmatic dependent of the one before: the
 * dK/dV pass sets up and loads K/V while the preprocess ends, and the dQ pass
 * may start on SMs that the last dK/dV CTAs leave free.  Every read of D still
 * follows the preprocess, and the dQ grid completes only after the dK/dV grid.
 *  fa_bwd_preprocess: delta [B,H,Nq] fp32 = rowsum(dO o O).
 *  fa_bwd_dkdv: dk, dv [B,H,Nk,d] from q, k, v, lse, delta, dO; each
 *    128-key tile is one work item of a persistent grid (at most one CTA per
 *    SM), P and dS rebuilt on chip for every query tile it sees.
 *  fa_bwd_dq: dq [B,H,Nq,d] from q, k, v, lse, delta, dO; each 128-query
 *    tile is one work item.  dkdv and dq only read delta, so they may run in any
 *    order (or concurrently) after the preprocess.
 * Same conventions and errors as fa_bwd. */
int fa_bwd_preprocess(const void *o, const void *dO, float *delta, int B, int H, int Nq, int d,
                      void *stream);
int fa_bwd_dkdv(const void *q, const void *k, const void *v, const float *lse, const float *delta,
                const void *dO, void *dk, void *dv, int B, int H, int Nq, int Nk, int d, float scale,
                int causal, void *stream);
int fa_bwd_dq(const void *q, const void *k, const void *v, const float *lse, const float *delta,
              const void *dO, void *dq, int B, int H, int Nq, int Nk, int d, float scale, int causal,
              void *stream);

/* fa_bwd_dkdv on CTA pairs (d = 128 only; FA_ERR_UNSUPPORTED for d = 64):
 * the two CTAs of a cluster take key tiles 2t and 2t + 1 of a head and issue
 * every product once for both as a tcgen05.mma with cta_group::2 (M = 256
 * keys), each CTA loading only the half of the B operand that it contributes.
 * Same arguments, outputs and tolerance as fa_bwd_dkdv (the same sums, split
 * differently across the tensor cores).  It needs more synchronisation
 * between the two CTAs than it saves in shared-memory reads, so it is slower
 * than fa_bwd_dkdv, which fa_bwd uses (johe.ru "Flash Attention: ...",
 * section "Flash Attention 4": kernels for the newest tensor cores).  The
 * caller's stream must allow cluster launches (every CUDA stream does). */
int fa_bwd_dkdv_pair(const void *q, const void *k, const void *v, const float *lse, const float *delta,
                     const void *dO, void *dk, void *dv, int B, int H, int Nq, int Nk, int d, float scale,
                     int causal, void *stream);

/* Bytes of fp32 workspace fa_decode needs for num_splits partials (<= 0:
 * for min(16, ceil(Nk / 256)) splits, the most the automatic count takes).
 * Host only, no device call.  Returns 0 for invalid sizes. */
size_t fa_decode_workspace_bytes(int B, int H, int Nk, int d, int num_splits);

/* Split-KV decode: one query token per (b, h) against a KV cache.  The key
 * cache is streamed, not shrunk (zimaspace.com "Wie reduziert Flash Attention
 * den Speicherverkehr ...", section "Weniger IO bedeutet nicht, dass der
 * KV-Cache entfällt").  The Nk keys are cut into num_splits contiguous chunks of
 * ceil(Nk / num_splits) keys; each chunk yields a partial output and partial
 * LSE, and the partials are merged with the max-shifted rescaling of the
 * online-softmax recurrence (wiki.ai-engineering.at "Flash Attention",
 * "Lösung: Online Softmax").  With d = 128 and Nk a multiple of 128 the
 * chunks are read by the tensor-core kernel of
 * fa_decode_paged (the cache as one page per sequence), whose chunks are
 * rounded up to whole 128-key stages, so trailing chunks may be empty; every
 * other shape takes a kernel of 16-byte loads.  The result is the same up to
 * rounding either way.  q [B,H,d], kcache/vcache [B,H,Nk,d] bf16 in;
 * o [B,H,d] bf16 out; lse [B,H] fp32 out, may be NULL.  num_splits <= 0 lets
 * the library choose: min(16, ceil(Nk / 256)) on the tensor-core kernel; on
 * the other kernel the count in 1 .. min(16, ceil(Nk / 256)) whose
 * (b, h, split) grid costs the fewest waves of resident CTAs times keys per
 * split (ties: fewer splits).  Otherwise 1 <= num_splits <= 256.  workspace:
 * at least fa_decode_workspace_bytes(B,H,Nk,d,num_splits) bytes. */
int fa_decode(const void *q, const void *kcache, const void *vcache, void *o, float *lse,
              int B, int H, int Nk, int d, float scale, int num_splits,
              void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of fp32 workspace fa_decode_paged needs (partials of B*Hq heads);
 * num_splits <= 0 (automatic) returns the size for 16 splits, the most the
 * automatic choice takes. */
size_t fa_decode_paged_workspace_bytes(int B, int Hq, int d, int num_splits);

/* Decode against a paged KV cache with grouped-query heads (the serving
 * layout: johe.ru "Flash Attention: ...", section "Альтернативы",
 * PagedAttention keeps the cache in fixed-size pages; grouped-query heads
 * share one kv head).  For every sequence b and query head h it computes the
 * same result as fa_decode against the sequence's first seq_lens[b] tokens
 * in logical order, with query head h reading kv head h / (Hq / Hkv).
 *  q [B, Hq, d] bf16; k_pages, v_pages [num_pages, Hkv, page_size, d] bf16
 *  (a page holds page_size consecutive tokens of one kv head);
 *  block_table [B, max_pages] int32: physical page of each logical page;
 *  seq_lens [B] int32, 1 <= seq_lens[b] <= max_pages * page_size;
 *  o [B, Hq, d] bf16; lse [B, Hq] fp32 or NULL.
 * num_splits <= 0 lets the library choose (from B, the heads, the longest
 * possible sequence max_pages * page_size and the SM count; at most 16).
 * Each sequence is cut into num_splits (1..256) contiguous chunks of
 * ceil(seq_lens[b] / num_splits) tokens (rounded up to whole 128-token stages
 * on the tensor-core path: page_size a multiple of 8), merged as in
 * fa_decode.  Every K/V
 * row is read once per group of up to 16 query heads on that path (4 on the
 * general one).  Tokens past seq_lens[b] in a page are never used, whatever
 * they hold.  Host checks: Hq % Hkv
 * == 0, d in {64, 128}, alignment, workspace.  The table and lengths live in
 * device memory and are checked by the kernel: a page index outside
 * [0, num_pages) or a length out of range is never dereferenced; it is read
 * as zeros and recorded as FA_ERR_INVALID_ARG in the device error word
 * (fa_get_last_device_error). */
int fa_decode_paged(const void *q, const void *k_pages, const void *v_pages, const int *block_table,
                    const int *seq_lens, void *o, float *lse, int B, int Hq, int Hkv, int page_size,
                    int max_pages, int num_pages, int d, float scale, int num_splits, void *workspace,
                    size_t workspace_bytes, void *stream);

/* Size of the scratch array that fa_decode_noalloc uses instead of a workspace. */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* Split-KV decode exactly like fa_decode, for callers that cannot allocate
 * device memory when they need a decode step.  Examples: a serving loop or
 * plugin host that hands this library only its input and output buffers and
 * owns every other byte of device memory; a real-time path that must never
 * call the allocator, because cudaMalloc/cudaFree may synchronise the whole
 * device and may fail once memory is fragmented; C callers with no access to
 * the framework allocator that owns the tensors.
 * Not a step of the method: the pages have no counterpart; it only changes
 * where the split partials live.  Instead of a caller workspace, the partials
 * go to one fixed array of FA_DECODE_NOALLOC_SCRATCH_BYTES compiled into the
 * library (every GPU that loads the library holds it until the process exits).
 * Arguments mean what they mean for fa_decode; the caller still passes q, the
 * caches, o and (optionally) lse.  A problem whose partials would need more
 * than the array (fa_decode_workspace_bytes(B,H,Nk,d,num_splits) >
 * FA_DECODE_NOALLOC_SCRATCH_BYTES) is rejected with FA_ERR_WORKSPACE before
 * anything is launched.  The call allocates nothing.  The first call on each
 * device looks up the array's device address (with that device current) and
 * caches it; make that first call before any stream capture.  All calls share
 * the one array: calls that may overlap on the GPU (different streams, no
 * ordering between them) race on it, so order them.  Nothing in the array has
 * to start at zero (every partial is written before it is read), and it keeps
 * the last call's partials. */
int fa_decode_noalloc(const void *q, const void *kcache, const void *vcache, void *o, float *lse,
                      int B, int H, int Nk, int d, float scale, int num_splits, void *stream);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device.  Returns FA_OK, the first code a kernel recorded
 * (FA_ERR_TIMEOUT: a bounded wait ran out; FA_ERR_INVALID_ARG: a device-side
 * argument check failed, e.g. a page index), or FA_ERR_CUDA if synchronising
 * or reading failed.  If `detail` is not NULL it
 * receives 4 ints: code, site (which wait), block index, and an auxiliary
 * value (the wait's phase), all 0 when no error was recorded. */
int fa_get_last_device_error(void *stream, int *detail);

/* Watchdog self-test (failure detection without a GPU fault): launches one
 * thread that waits on a barrier nothing ever arrives on, with a limit of
 * timeout_ns (1e3 .. 1e9).  The wait runs out, the kernel records
 * FA_ERR_TIMEOUT (site 19, the self-test site) in the error word and returns;
 * fa_get_last_device_error(stream, ...) then reports it and clears the word.
 * The device stays usable.  Returns the launch status. */
int fa_selftest_wait_timeout(uint64_t timeout_ns, void *stream);

/* Sets the limit of every device-side wait, in nanoseconds, for kernels
 * launched after the call (default 2e9; values below 1e6 are raised to 1e6).
 * Returns the previous value. */
uint64_t fa_set_wait_timeout_ns(uint64_t ns);

/* Static description of a status code. */
const char *fa_status_string(int status);

/* Library version, as major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
