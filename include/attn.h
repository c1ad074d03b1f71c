/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library.
 *
 * Operation (prefill): for every batch b, query head h and query row i,
 *
 *     O[b,i,h,:] = softmax_j( scale * q[b,i,h,:] . k[b,j,g,:] ) v[b,j,g,:]
 *     lse[b,h,i] = ln sum_j exp( scale * q[b,i,h,:] . k[b,j,g,:] )
 *
 * with g = h / (Hq / Hkv), j over the keys the row may see.  This is the fused
 * softmax(Q K^T / sqrt(d)) V of the MoonMath HIP attention page (opening
 * section and its feature list: bf16, BSHD or BHSD with no transpose,
 * head dim 128, any sequence lengths including cross-attention), computed
 * with the IO-aware tiling and online softmax of "FlashAttention-4 中的 IO
 * 感知块分块策略" (running max m, running sum l, m' = max(m, m_new),
 * l' = l exp(m - m') + l_new; only m and l are kept as row statistics), with
 * the causal upper-triangle skip and the grouped-query sharing of the
 * reverse-engineering page (观点一 tiling strategy and multi-query settings)
 * and the paged KV cache of the ROCm port page ("Vendor-Agnostic 多查询推理
 * 优化": 16-token pages, int32 block_table).
 *
 * Readings taken where the pages are silent:
 *   - causal alignment is bottom-right: key j is visible to row i iff
 *     j <= i + Sk - Sq;
 *   - a row that sees no key gets O = 0 and lse = -inf;
 *   - lse is the natural log of the sum of exp of the *scaled* scores;
 *   - O is rounded to bf16 round-to-nearest-even, unless a call selects one of
 *     the other two output rounding modes (attn_fwd_rounded).
 *
 * Conventions for every entry point:
 *   - Pointers named q, k, v, out, lse, k_pages, v_pages, block_table, seqlens,
 *     workspace, o_parts, lse_parts are DEVICE pointers owned by the caller
 *     (except attn_fwd_host, whose q, k, v, out and lse are host pointers);
 *     the library never frees them and keeps none past the call, except the
 *     workspace registered with attn_set_workspace.  The library allocates no
 *     device memory on any call.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously; only attn_get_device_status synchronises.
 *   - bf16 tensors are dense and contiguous; every device pointer must be
 *     16-byte aligned.
 *   - attn_fwd_host creates three streams and a few events per device on its
 *     first call and keeps them; no other entry point creates CUDA objects.
 *   - Arguments are validated before anything is launched; a rejected call
 *     returns ATTN_ERR_INVALID_ARG or ATTN_ERR_UNSUPPORTED and enqueues nothing.
 *   - A kernel that gives up on a bounded wait (see attn_set_wait_budget_ns)
 *     records ATTN_ERR_TIMEOUT in the device status word and exits cleanly;
 *     read it with attn_get_device_status.
 *   - No entry point throws or aborts; all report through attn_status_t.
 */
#ifndef ATTN_H
#define ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,   /* NULL/misaligned pointer, bad shape, bad enum, non-finite scale */
    ATTN_ERR_UNSUPPORTED = 2,   /* d != 128, page_size != 16, or not an sm_103 / sm_100 family GPU */
    ATTN_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (launch error etc.) */
    ATTN_ERR_TIMEOUT = 4,       /* a kernel's bounded wait expired (device status only) */
    ATTN_ERR_WORKSPACE = 5,     /* workspace NULL, misaligned or smaller than required */
    ATTN_ERR_DEVICE_BOUNDS = 6  /* a kernel met an out-of-range block_table entry (device status only) */
} attn_status_t;

typedef enum {
    ATTN_LAYOUT_BSHD = 0,       /* [B][S][H][d] */
    ATTN_LAYOUT_BHSD = 1        /* [B][H][S][d] */
} attn_layout_t;

/* Rounding of the fp32 result to the bf16 output (the three modes of the
 * MoonMath HIP kernel page's benchmark section). */
typedef enum {
    ATTN_ROUND_RTNE = 0,        /* to nearest, ties to even (the default) */
    ATTN_ROUND_RTNA = 1,        /* to nearest, ties away from zero */
    ATTN_ROUND_RTZ = 2          /* toward zero; never overflows to infinity */
} attn_round_t;

/*
 * attn_fwd -- fused exact attention forward (prefill), tcgen05 + TMA kernel.
 *
 * q:   bf16, layout `layout`, shape [B,Sq,Hq,d] (BSHD) or [B,Hq,Sq,d] (BHSD).
 * k,v: bf16, same layout, shape [B,Sk,Hkv,d] or [B,Hkv,Sk,d].
 * out: bf16, same layout and shape as q (written).
 * lse: fp32 [B][Hq][Sq] (written), or NULL to skip it.
 * d must be 128.  Hq must be a multiple of Hkv (MQA: Hkv = 1).  Sq and Sk are
 * any lengths >= 1 and may differ.  causal != 0 applies the bottom-right
 * causal mask.  scale is the softmax scale (usually 1/sqrt(d)); any finite
 * value >= 0 is accepted.
 * Results are deterministic: the same call on the same device returns
 * bitwise-identical out and lse.
 *
 * Scheduling.  The work is cut into units of two 128-row Q tiles.  When there
 * are more units than SMs the kernel runs one CTA per SM, and each CTA takes
 * the next free unit from a counter in device memory as it finishes one
 * (which unit a CTA gets changes nothing in the result).  The library owns a
 * pool of 256 such counters per device and gives each launch the next one in
 * turn, and a launch's last CTA sets its counter back to zero: so at most 256
 * of these launches (attn_fwd, attn_fwd_rounded, attn_fwd_varlen,
 * attn_fwd_paged, attn_fwd_host) may be in flight on one device at the same
 * time.  Launches on one stream, and graph replays, are always fine.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse,
                       int B, int Hq, int Hkv, int Sq, int Sk, int d,
                       int layout, int causal, float scale, void *stream);

/*
 * attn_fwd_rounded -- attn_fwd with a selectable rounding of the output.
 *
 * The MoonMath HIP kernel page (benchmark and limitations sections) runs its
 * bf16 forward kernel in three rounding modes, RTNE, RTNA and RTZ, each with
 * its own rule for the bf16 output.  round_mode (an attn_round_t) selects
 * how each element of O, computed in fp32, is rounded to bf16; attn_fwd is
 * this call with ATTN_ROUND_RTNE.  The mode changes nothing but that last
 * conversion (in the kernel's epilogue and in the tail-split merge): the
 * fp32 value before it, lse, and the internal bf16 rounding of the
 * probabilities before the P V product (always to nearest even) are the same
 * in every mode.  Other arguments, errors and determinism as attn_fwd; a
 * round_mode outside the enum returns ATTN_ERR_INVALID_ARG.
 */
attn_status_t attn_fwd_rounded(const void *q, const void *k, const void *v, void *out, float *lse,
                               int B, int Hq, int Hkv, int Sq, int Sk, int d,
                               int layout, int causal, float scale, int round_mode, void *stream);

/*
 * attn_fwd_varlen -- attn_fwd over a packed batch of variable-length
 * sequences (the "variable-length batches" the MoonMath HIP kernel page lists
 * among its kernel's limitations; here they are supported).
 *
 * q:   bf16 [total_q][Hq][d], the B sequences' query rows back to back.
 * k,v: bf16 [total_k][Hkv][d], the sequences' key/value rows back to back.
 * cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B+1]; sequence b owns rows
 *      cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of q and out, and rows
 *      cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1 of k and v.  Offsets must be
 *      non-decreasing and within [0, total]; lengths may be 0.
 * max_seqlen_q, max_seqlen_k: upper bounds of the sequences' lengths (the
 *      grid is sized by max_seqlen_q); 1 <= max_seqlen <= total.
 * out: bf16 [total_q][Hq][d] (written for the rows of every sequence; rows
 *      that belong to no sequence are not touched).
 * lse: fp32 [Hq][total_q] (same rows written), or NULL.
 * Each sequence is exactly attn_fwd with B = 1, Sq and Sk its own lengths:
 * its rows see only its own keys, and causal != 0 applies the bottom-right
 * causal mask within the sequence.  A sequence with queries and no keys gets
 * O = 0 and lse = -inf.  d must be 128; Hq a multiple of Hkv; round_mode as
 * in attn_fwd_rounded.  The offsets live on the device and are not read on
 * the host: a kernel that finds them out of order, out of range or past the
 * stated maxima records ATTN_ERR_DEVICE_BOUNDS in the device status word and
 * leaves that sequence's rows untouched.  No tail split; deterministic.
 */
attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse,
                              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                              int B, int Hq, int Hkv, int total_q, int total_k,
                              int max_seqlen_q, int max_seqlen_k, int d,
                              int causal, float scale, int round_mode, void *stream);

/*
 * attn_fwd_paged -- prefill of packed query chunks against a paged KV cache
 * (chunked prefill): the 16-token pages and int32 block_table of the ROCm port
 * page ("Vendor-Agnostic 多查询推理优化") combined with the causal tiling of
 * the reverse-engineering page (观点一 tiling strategy).
 *
 * q:   bf16 [total_q][Hq][d]; sequence b's query chunk is rows
 *      cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 (DEVICE int32 [B+1]).
 * k_pages, v_pages: bf16 [num_pages][16][Hkv][d] page pools.
 * block_table: DEVICE int32 [B][max_blocks_per_seq]; entry p of row b is the
 *      pool page holding keys 16p .. 16p+15 of sequence b; entries past the
 *      sequence's last page are never read.
 * seqlens_k: DEVICE int32 [B], the keys in each sequence's cache, the chunk's
 *      own keys included (the chunk is the cache's last Lq tokens).
 * out: bf16 [total_q][Hq][d]; lse: fp32 [Hq][total_q] or NULL (rows of every
 *      chunk written, others untouched).
 * Sequence b computes attn_fwd with B = 1 over its chunk and its gathered
 * keys; causal != 0 applies the bottom-right mask (query i of a chunk of Lq
 * sees keys j <= i + Lk - Lq).  Slots past a sequence's length in its last
 * page may hold anything, NaN included: they never reach the result.
 * page_size must be 16 and d 128; max_seqlen_q bounds the chunk lengths.
 * Out-of-order query offsets, lengths past max_seqlen_q or the table, and
 * table entries outside [0, num_pages) are recorded as ATTN_ERR_DEVICE_BOUNDS
 * in the device status word (a bad page reads as zeros; a bad sequence is
 * skipped).  Deterministic.
 */
attn_status_t attn_fwd_paged(const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *block_table, const int32_t *seqlens_k,
                             const int32_t *cu_seqlens_q, void *out, float *lse,
                             int B, int Hq, int Hkv, int total_q, int max_seqlen_q, int d,
                             int page_size, int num_pages, int max_blocks_per_seq,
                             int causal, float scale, int round_mode, void *stream);

/*
 * attn_fwd_host -- attn_fwd_rounded from and to HOST memory.
 *
 * q, k, v: host bf16 in `layout`, shapes as attn_fwd (read).
 * out: host bf16, q's shape (written); lse: host fp32 [B][Hq][Sq] or NULL.
 * Host buffers should be page-locked (cudaHostAlloc / pinned): the copies
 * are asynchronous only then.
 * workspace: DEVICE buffer of at least attn_fwd_host_workspace_bytes(...)
 *      bytes, 256-byte aligned, owned by the caller; it stages q, k, v, out
 *      and lse on the device (contents undefined afterwards).
 * The copies in, the forward kernel and the copies out run in batch chunks
 * on three library-owned helper streams (created once per device), so the
 * copies of one chunk overlap the compute of another; the call is ordered
 * after earlier work on `stream`, and later work on `stream` waits for it
 * (event dependencies both ways).  The result is the same as copying in,
 * calling attn_fwd_rounded on the whole batch and copying out, except that
 * each chunk of batches is its own launch (so a tail split, if a workspace is
 * registered, may differ).  Errors: those of attn_fwd (checked before any
 * copy), ATTN_ERR_WORKSPACE for a missing, misaligned or small workspace.
 */
attn_status_t attn_fwd_host(const void *q, const void *k, const void *v, void *out, float *lse,
                            int B, int Hq, int Hkv, int Sq, int Sk, int d,
                            int layout, int causal, float scale, int round_mode,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Device workspace attn_fwd_host needs for this shape (0 if invalid). */
size_t attn_fwd_host_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int d);

/*
 * attn_fwd_workspace_bytes -- device workspace that lets attn_fwd split the
 * key ranges of its last wave of work units (the Flash-Decoding style tail
 * split of the MoonMath page: the partial results are merged by log-sum-exp)
 * for this shape on the CURRENT device (the plan depends on its SM count).
 * Returns 0 when the shape gets no split (causal shapes, shapes whose units
 * fill the last wave, short key ranges) or the arguments are invalid.
 */
size_t attn_fwd_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal);

/*
 * attn_set_workspace -- register a caller-owned device buffer as the current
 * device's workspace for attn_fwd's tail split (NULL clears it).  ptr must be
 * 256-byte aligned; the library keeps the pointer until it is replaced or
 * cleared and never frees it.  attn_fwd splits only when a registered buffer
 * is at least attn_fwd_workspace_bytes(...) large; otherwise it runs every
 * unit whole, with the same result to within rounding.  The buffer is used by
 * every attn_fwd, attn_fwd_rounded and attn_fwd_host on the device (a single
 * registration per device): calls that may overlap on the GPU must not both
 * split, so order their streams, or clear the registration while they run.
 */
attn_status_t attn_set_workspace(void *ptr, size_t bytes);

/*
 * attn_fwd_simple -- the same operation and contract as attn_fwd, computed by
 * a plain SIMT CUDA kernel (one warp per query row, no tensor cores).  It is
 * a debugging cross-check for attn_fwd, not a fallback: nothing routes to it
 * automatically.  Slow; meant for small shapes.
 */
attn_status_t attn_fwd_simple(const void *q, const void *k, const void *v, void *out, float *lse,
                              int B, int Hq, int Hkv, int Sq, int Sk, int d,
                              int layout, int causal, float scale, void *stream);

/*
 * attn_decode_workspace_bytes -- bytes of device workspace attn_decode_paged
 * needs for this shape.  A pure function of the arguments (the key-split plan
 * depends only on the shape, never on device data).
 * Returns 0 for invalid arguments.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int d, int max_blocks_per_seq);

/*
 * attn_decode_paged -- one decode step over a paged KV cache, split over the
 * keys (Flash-Decoding style, as in the MoonMath page's tail split) and
 * merged by log-sum-exp.
 *
 * q:           bf16 [B][Hq][d], one query per sequence and head.
 * k_pages,
 * v_pages:     bf16 [num_pages][page_size][Hkv][d], the page pool.
 * block_table: int32 [B][max_blocks_per_seq]; entry p of row b is the
 *              physical page of keys 16p .. 16p+15 of sequence b.  Entries at
 *              or past ceil(seqlens[b]/16) are never read (may hold -1).
 * seqlens:     int32 [B] on the device, each in [0, 16 * max_blocks_per_seq].
 *              A length outside that range is not clamped: it is recorded as
 *              ATTN_ERR_DEVICE_BOUNDS in the device status word and that
 *              sequence is skipped (its rows get zeros and lse = -inf); the
 *              other sequences are unaffected.
 * out:         bf16 [B][Hq][d] (written); a sequence of length 0 gets zeros.
 * lse:         fp32 [B][Hq] (written, -inf for length 0), or NULL.
 * page_size must be 16; d must be 128; Hq % Hkv == 0.
 * workspace:   device buffer of at least attn_decode_workspace_bytes(...)
 *              bytes, 256-byte aligned, owned by the caller; its contents on
 *              entry do not matter and are overwritten.
 * A block_table entry outside [0, num_pages) that is needed is not read: the
 * keys of that page count as absent and ATTN_ERR_DEVICE_BOUNDS is recorded
 * in the device status word.
 */
attn_status_t attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *block_table, const int32_t *seqlens,
                                void *out, float *lse,
                                int B, int Hq, int Hkv, int d, int page_size,
                                int num_pages, int max_blocks_per_seq, float scale,
                                void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_decode_paged_append -- append one token per sequence to the paged
 * cache and decode over it, in the same launch (the new token's K/V written
 * into its page while the step's attention runs, as in the reverse-
 * engineering page's 观点二 decode discussion).
 *
 * k_new, v_new: bf16 [B][Hkv][d], the new token's key and value rows.
 * seqlens: the cache lengths BEFORE the append (read only; the caller
 *      advances them afterwards).  The token goes to slot seqlens[b] % 16 of
 *      page block_table[b][seqlens[b] / 16], which must be a valid page (a
 *      new page for a sequence whose length is a multiple of 16).
 * k_pages, v_pages: written at exactly those slots (B x Hkv rows each), read
 *      elsewhere.
 * Every query attends over its sequence's seqlens[b] + 1 keys, the new one
 * included; out, lse, the other arguments, the workspace and the errors are
 * those of attn_decode_paged.  A slot outside the table or the pool is
 * recorded as ATTN_ERR_DEVICE_BOUNDS and that token is not written (it is
 * still attended to).  A length outside [0, 16 * max_blocks_per_seq] skips
 * the sequence as in attn_decode_paged: nothing is appended for it.
 * k_new, v_new must not overlap the pools.
 */
attn_status_t attn_decode_paged_append(const void *q, const void *k_new, const void *v_new,
                                       void *k_pages, void *v_pages,
                                       const int32_t *block_table, const int32_t *seqlens,
                                       void *out, float *lse,
                                       int B, int Hq, int Hkv, int d, int page_size,
                                       int num_pages, int max_blocks_per_seq, float scale,
                                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES -- capacity of the device array that
 * attn_decode_paged_noalloc keeps its split partials in: 16 MiB, held on every
 * GPU that loads the library until the process exits.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * attn_decode_paged_noalloc -- attn_decode_paged for callers that cannot
 * allocate device memory.  (The pages have no counterpart of this entry point;
 * it exists for such callers, not for the method.)
 *
 * Some callers cannot hand the decode step a workspace: an operator interface
 * of a host framework that passes a kernel only its inputs and outputs and has
 * no allocator or workspace hook, or an engine that reserved all of HBM for its
 * own pools and forbids further cudaMalloc calls (which would also synchronise
 * the device inside a latency-critical loop).  This entry point takes the same
 * arguments as attn_decode_paged minus the workspace and keeps the split
 * partials in a library-owned device array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES
 * instead.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The caller still passes every input and output buffer.  Arguments are
 * checked as in attn_decode_paged first (ATTN_ERR_INVALID_ARG,
 * ATTN_ERR_UNSUPPORTED); a call that passes them but whose
 * attn_decode_workspace_bytes(B, Hq, d, max_blocks_per_seq) exceeds the array
 * is then rejected with ATTN_ERR_WORKSPACE, before anything is launched.  The
 * first call in each CUDA context looks up the array's device address
 * (cudaGetSymbolAddress) with that context current and remembers it under the
 * context's unique id; make that first call before any stream capture.  A
 * context created later (after cudaDeviceReset, for instance) gets a lookup of
 * its own, so no address outlives its context.  All calls
 * share the one array, which keeps the last call's contents (nothing in it
 * needs to start at zero): calls that overlap on the GPU, e.g. on two streams
 * with no ordering between them, race on it and must not be issued.
 */
attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                        const int32_t *block_table, const int32_t *seqlens,
                                        void *out, float *lse,
                                        int B, int Hq, int Hkv, int d, int page_size,
                                        int num_pages, int max_blocks_per_seq, float scale, void *stream);

/*
 * attn_lse_merge -- merge key-range partial results by log-sum-exp (the merge
 * step of the Flash-Decoding style split).  For each row r:
 *     M = max_s lse_parts[r][s];  lse = M + ln sum_s exp(lse_parts[r][s] - M)
 *     out[r][:] = sum_s exp(lse_parts[r][s] - lse) * o_parts[r][s][:]
 * in a fixed split order (deterministic).  Rows whose partials are all -inf
 * get out = 0 and lse = -inf.
 * o_parts: fp32 [rows][nsplit][d], each partial normalised within its range.
 * lse_parts: fp32 [rows][nsplit].  out: bf16 [rows][d], rounded from fp32 in
 * round_mode (an attn_round_t; anything else is ATTN_ERR_INVALID_ARG).
 * lse: fp32 [rows] or NULL.  d must be 128; nsplit >= 1.
 */
attn_status_t attn_lse_merge(const float *o_parts, const float *lse_parts, void *out, float *lse,
                             int rows, int nsplit, int d, int round_mode, void *stream);

/*
 * attn_get_device_status -- synchronise `stream`, then read and clear the
 * current device's status word.  Returns ATTN_OK, ATTN_ERR_TIMEOUT or
 * ATTN_ERR_DEVICE_BOUNDS as recorded by kernels since the last call (or
 * ATTN_ERR_CUDA if the synchronisation itself failed).  *site (may be NULL)
 * receives the id of the wait or check that recorded it.
 */
attn_status_t attn_get_device_status(void *stream, int *site);

/*
 * attn_set_wait_budget_ns -- time budget of every bounded wait inside the
 * kernels (mbarrier waits), in nanoseconds of the GPU's global timer.
 * Default 2e9 (2 s); 0 restores the default.  Applies to later launches.
 */
attn_status_t attn_set_wait_budget_ns(uint64_t ns);

/*
 * attn_debug_inject -- host-side fault injection for the failure-detection
 * tests.  mode 0: off (default).  mode 1: the next attn_fwd launches its
 * kernel with the load-issuing warp told to issue nothing, so the other warps'
 * bounded waits expire, they record ATTN_ERR_TIMEOUT and the kernel exits
 * cleanly (no fault, no hang, nothing left in flight).  The flag clears
 * itself after one launch.
 */
attn_status_t attn_debug_inject(int mode);

/*
 * attn_selftest_umma -- checks the tensor-core operand layouts this library
 * uses, on one 128x128x128 tile: c[i][j] = sum_k a[i][k] * b[j][k] (mode 0:
 * both operands from shared memory, K-major) or c[i][j] = sum_k a[i][k] *
 * b[k][j] (mode 1: a from tensor memory, b from shared memory N-major, the
 * form the P*V product uses).  a, b: bf16 [128][128] row-major device
 * buffers; c: fp32 [128][128] (written).
 */
attn_status_t attn_selftest_umma(const void *a, const void *b, float *c, int mode, void *stream);

/* attn_status_string -- static, human-readable name of a status code. */
const char *attn_status_string(attn_status_t status);

/* attn_version -- library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H */
