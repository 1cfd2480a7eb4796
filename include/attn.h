/*
 * attn.h -- C ABI of libattn: exact IO-aware attention on GB300, forward and
 * backward.
 *
 * What it computes (per batch element b and head h):
 *
 *     S = scale * Q K^T            (T_q x T_kv, never written to memory)
 *     P = softmax(S) row by row    (T_q x T_kv, never written to memory)
 *     O = P V                      (T_q x d)
 *     lse[i] = ln sum_j exp(S[i][j])
 *
 * following "FlashAttention IO-aware tiling lab" (the definition
 * S = QK^T/sqrt(d), P = softmax(S), O = PV and the kernel phases) and
 * "IO-Aware Attention: Tiling the Score Matrix Without Materializing It",
 * section "Softmax over blocks, exactly" (running maximum m, running sum l,
 * rescaled accumulator o, result o/l). The problem statement -- Q is T_q x d,
 * K and V are T_kv x d per head, over B sequences and h heads, with an
 * optional causal mask -- is that of "Attention and Its Computational Cost",
 * section "What is being computed". lse is the per-row normalisation
 * constant kept for a backward pass ("IO-Aware Attention ...", section
 * "What has to stay in fast memory").
 *
 * Causal mask: key j is visible to query row i iff j <= i + (T_kv - T_q)
 * (bottom-right alignment; for T_q == T_kv row i sees keys 0..i, and a single
 * query sees the whole cache). A masked row never has zero visible keys
 * because T_q <= T_kv is required.
 *
 * Dispatch: T_q == 1 runs the split-KV decode path (a split kernel over key
 * partitions, then an exact merge kernel: "IO-Aware Attention ...", section
 * "Parallelism and the cost of the split"); T_q > 1 runs the tensor-core
 * prefill kernel -- attn_fwd also cuts its key range into partitions when
 * B*h*ceil(T_q/256) units would fill less than half the SMs (see
 * attn_fwd_splitkv).
 *
 * Conventions for every entry point:
 *   - Tensors are dense, row-major, contiguous [B][h][T][d] in device memory,
 *     all four of q, k, v, o in the same 16-bit type (dtype), each base
 *     16-byte aligned. lse is fp32 [B][h][T_q], 4-byte aligned.
 *   - The caller owns every buffer; the library keeps no pointer after the
 *     work it enqueued has finished. o and lse must not overlap q, k or v
 *     or each other.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls are asynchronous: ATTN_OK means "validated and
 *     enqueued". Arguments are checked before anything is enqueued; an
 *     invalid call enqueues nothing and touches no buffer.
 *   - Supported set: d in {64, 128}; dtype ATTN_F16 or ATTN_BF16;
 *     scale finite and > 0; B, h, T_q >= 0 (a zero makes the call an empty
 *     no-op returning ATTN_OK); T_kv >= 1 whenever the output is non-empty;
 *     causal requires T_q <= T_kv; B*h < 2^31 and T_q, T_kv < 2^31.
 *   - Accumulation and rescaling are fp32; O is rounded once to the 16-bit
 *     type (round to nearest even).
 *   - Errors are return codes; nothing aborts or prints. A device-side wait
 *     that exceeds its time limit does not hang: the kernel records
 *     ATTN_ERR_TIMEOUT in a device status word, leaves its outputs undefined
 *     and returns; read it with attn_get_device_error.
 */
#ifndef EXACT_IO_AWARE_ATTN_H
#define EXACT_IO_AWARE_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_ABI_VERSION 4

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned/overlapping pointer, bad size, bad scale */
  ATTN_ERR_UNSUPPORTED = 2, /* valid request outside the supported set (e.g. d = 96) */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
  ATTN_ERR_TIMEOUT = 4,     /* a device-side bounded wait gave up (see attn_get_device_error) */
  ATTN_ERR_WORKSPACE = 5    /* workspace missing, too small or misaligned */
} attn_status_t;

typedef enum { ATTN_F16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/*
 * attn_fwd -- the whole forward: O and lse from Q, K, V.
 *   q     [B][h][T_q][d]   16-bit, read only
 *   k, v  [B][h][T_kv][d]  16-bit, read only
 *   o     [B][h][T_q][d]   16-bit, written
 *   lse   [B][h][T_q]      fp32, written (natural log, scaled-score units)
 *   scale multiplies Q K^T (1/sqrt(d) for standard attention)
 *   causal 0 or 1
 * The decode path (T_q == 1) needs a workspace of attn_workspace_bytes(...,
 * 0) bytes; attn_fwd takes it from the stream-ordered allocator
 * (cudaMallocAsync/cudaFreeAsync on `stream`, no host synchronisation). The
 * prefill path needs no workspace.
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                       int B, int h, int T_q, int T_kv, int d, float scale, int causal,
                       int dtype, void* stream);

/*
 * attn_fwd_ex -- attn_fwd with caller-chosen decode split count and
 * caller-owned workspace. The split count is the number of key partitions
 * whose partial (max, sum, output) are merged exactly ("IO-Aware
 * Attention: Tiling the Score Matrix Without Materializing It", section
 * "Parallelism and the cost of the split").
 *   num_splits  key partitions per (b, h) for the decode path: 0 = the
 *               library's choice by shape, else 1..1024 (a partition that
 *               gets no key contributes weight 0). Ignored for T_q > 1.
 *   workspace   device memory, 16-byte aligned, at least
 *               attn_workspace_bytes(B, h, T_q, T_kv, d, num_splits) bytes;
 *               may be NULL when that size is 0. Contents on entry are
 *               ignored; it must stay allocated until the work completes.
 * Returns ATTN_ERR_WORKSPACE if the workspace is needed and missing, too
 * small or misaligned.
 */
attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int h, int T_q, int T_kv, int d, float scale, int causal,
                          int dtype, int num_splits, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * attn_fwd_gqa -- grouped-query attention: q and o have h_q heads, k and v
 * have h_kv heads, h_q a multiple of h_kv; query head i attends with
 * key/value head i / (h_q / h_kv) ("Attention and Its Computational Cost",
 * section "The other shape": fewer key and value heads shrink the cache and
 * its read per step). Layouts: q, o [B][h_q][T_q][d]; k, v [B][h_kv][T_kv][d];
 * lse [B][h_q][T_q]. Other arguments as in attn_fwd_ex; with workspace NULL
 * and workspace_bytes 0 the decode path takes its workspace from the
 * stream-ordered allocator as attn_fwd does. The decode path reads each
 * cached key/value row once for up to 8 query heads of its group.
 * h_kv == h_q is plain attention (same kernels as attn_fwd_ex).
 * Groups of 4 or more query heads per key/value head decode on the tensor
 * cores with 1..64 partitions: num_splits 65..1024 then returns
 * ATTN_ERR_UNSUPPORTED (0, the library's choice, always stays in range).
 * Returns ATTN_ERR_INVALID_ARG if h_kv < 1 or h_q is not a multiple of h_kv.
 */
attn_status_t attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                           int causal, int dtype, int num_splits, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * attn_gqa_workspace_bytes -- workspace attn_fwd_gqa needs (0 for the
 * prefill path or invalid sizes): B*h_q*S*(d+4)*4 bytes, S the partition
 * count (num_splits, or the library's choice for this grouping when 0).
 * Returns 0 for a split count attn_fwd_gqa would reject (above 64 for groups
 * of 4 or more).
 */
size_t attn_gqa_workspace_bytes(int B, int h_q, int h_kv, int T_q, int T_kv, int d,
                                int num_splits);

/*
 * attn_workspace_bytes -- bytes of workspace attn_fwd_ex needs for this
 * shape (0 for the prefill path). num_splits as in attn_fwd_ex (0 = the
 * library's choice). Returns 0 for invalid sizes. The decode workspace holds
 * one partial (running max, running sum, unnormalised output of d floats)
 * per (b, h, split): B*h*S*(d+4)*4 bytes -- the per-partition state of
 * "IO-Aware Attention ...", section "Parallelism and the cost of the split".
 */
size_t attn_workspace_bytes(int B, int h, int T_q, int T_kv, int d, int num_splits);

/*
 * attn_decode_num_splits -- the split count the library chooses for a
 * decode call of this shape on the current device (0 if the shape is
 * invalid). Deterministic for a given device.
 */
int attn_decode_num_splits(int B, int h, int T_kv, int d);

/*
 * attn_fwd_host -- the forward with q, k, v, o and lse in HOST memory. The
 * path the pages describe starts and ends in HBM ("FlashAttention IO-aware
 * tiling lab", "Attention memory path": HBM to on-chip memory to the tensor
 * cores and back to HBM); this entry adds the level below it, the host, as a
 * convenience for callers whose tensors live there: the kernels are the
 * same. Shapes, dtype, scale, causal and the grouped-query heads as in
 * attn_fwd_gqa (h_kv == h_q: plain attention). In stream order on `stream`
 * the library copies q, k and v to device memory (one cudaMemcpyAsync each),
 * runs the same kernels as attn_fwd, and copies o and lse back. It returns
 * once the work is enqueued: o and lse hold the result after `stream` is
 * synchronised. Host buffers should be page-locked (cudaHostAlloc or
 * cudaHostRegister) for the copies to run asynchronously; with pageable
 * buffers the driver may stage the copies and block the calling thread.
 *   device_buffer  device memory for the device copies, 16-byte aligned, at
 *                  least attn_host_buffer_bytes(...) bytes, owned by the caller
 *                  and kept allocated until the work completes; NULL with
 *                  device_buffer_bytes 0: taken from and returned to the
 *                  stream-ordered allocator (cudaMallocAsync/cudaFreeAsync).
 * The decode path's workspace is taken from the stream-ordered allocator.
 * Returns ATTN_ERR_WORKSPACE if a caller buffer is too small or misaligned,
 * otherwise the errors of attn_fwd_gqa (host pointers are checked for NULL,
 * alignment and overlap like device pointers).
 */
attn_status_t attn_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                            int causal, int dtype, void* device_buffer,
                            size_t device_buffer_bytes, void* stream);

/*
 * attn_host_buffer_bytes -- device bytes attn_fwd_host needs for the copies
 * of q, k, v, o and lse (each at a 256-byte offset); 0 for an invalid or
 * empty shape.
 */
size_t attn_host_buffer_bytes(int B, int h_q, int h_kv, int T_q, int T_kv, int d);

/*
 * attn_get_device_error -- synchronises `stream`, then reads and clears the
 * current device's status word. Returns ATTN_OK if no kernel recorded an
 * error since the last read, ATTN_ERR_TIMEOUT if a bounded wait gave up,
 * ATTN_ERR_INVALID_ARG if a kernel found an invalid input in device memory
 * (a paged-decode block-table entry outside the page pool), or ATTN_ERR_CUDA
 * if the synchronisation itself failed. If `site` is not NULL
 * it receives the recorded word (0 if none): bits 0-7 the status code,
 * bits 8-15 the kernel, bits 16-23 the wait site.
 */
attn_status_t attn_get_device_error(void* stream, unsigned int* site);

/*
 * attn_selftest_wait_timeout -- tests the failure-detection path without
 * faulting the GPU. Enqueues on `stream` a one-thread kernel that waits on a
 * device barrier nothing will complete, using the same bounded wait as the
 * attention kernels but with a limit of `limit_us` microseconds (1 ..
 * 2,000,000). The wait gives up, the kernel records ATTN_ERR_TIMEOUT (kernel
 * id 4, site 1) in the device status word unless an error is already
 * recorded, and returns; a following attn_get_device_error reports and
 * clears it, and the context stays usable. Returns ATTN_ERR_INVALID_ARG for
 * a limit out of range, ATTN_OK once enqueued.
 */
attn_status_t attn_selftest_wait_timeout(unsigned int limit_us, void* stream);

/* attn_status_string -- static, NUL-terminated name of a status code. */
const char* attn_status_string(int status);

/* attn_abi_version -- ATTN_ABI_VERSION of the library actually loaded. */
int attn_abi_version(void);

/*
 * attn_last_kernel_name -- static name of the kernel family that the last
 * successful call on this host thread enqueued ("prefill_tcgen05_d64_bf16",
 * "decode_split_d64_bf16+decode_combine", ... or "none" for an empty call),
 * so a benchmark can record which kernel ran. Set by attn_fwd, attn_fwd_ex,
 * attn_fwd_gqa, attn_fwd_splitkv, attn_fwd_paged_decode, attn_fwd_host,
 * attn_fwd_naive, attn_bwd and attn_bwd_gqa; attn_fwd_decode_noalloc leaves
 * it unchanged.
 */
const char* attn_last_kernel_name(void);

/*
 * attn_bwd -- gradients of attn_fwd: dq, dk, dv from q, k, v, the forward's
 * o and lse, and dout = dL/dO.
 *
 * The backward pass recomputes the probabilities tile by tile from q, k and
 * the saved lse instead of reading a stored probability matrix ("IO-Aware
 * Attention: Tiling the Score Matrix Without Materializing It", section
 * "What has to stay in fast memory": the saved state is O(n d) per head plus
 * the O(n) row constants). The pages print no gradient formulas; these are
 * the derivative of the forward definition above. With P_ij =
 * exp(scale * q_i . k_j - lse_i) on visible pairs (0 elsewhere):
 *     dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D),  D_i = dO_i . o_i,
 *     dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 * Arguments: q, o, dout: [B][h][T_q][d]; k, v: [B][h][T_kv][d]; lse: fp32
 * [B][h][T_q] as written by attn_fwd for the same q, k, v, scale and causal
 * flag; dq: [B][h][T_q][d], dk, dv: [B][h][T_kv][d], written (not
 * accumulated into), in the 16-bit dtype, rounded once from fp32 sums.
 * scale, causal, dtype and the supported set as for attn_fwd (T_q == 1 is
 * allowed). Pointer rules as for attn_fwd; dq, dk, dv must not overlap each
 * other or any input. workspace: device memory of at least
 * attn_bwd_workspace_bytes(B, h, T_q, T_kv, d) bytes, 16-byte aligned, not
 * overlapping any argument; pass NULL with workspace_bytes 0 to have the
 * library take it stream-ordered (cudaMallocAsync/cudaFreeAsync on stream).
 * Deterministic: no atomics, the same inputs give the same bits.
 * Returns ATTN_ERR_WORKSPACE for a missing, short, misaligned or
 * overlapping workspace; otherwise as attn_fwd.
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const void* dout, const float* lse, void* dq, void* dk, void* dv, int B,
                       int h, int T_q, int T_kv, int d, float scale, int causal, int dtype,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_bwd_gqa -- attn_bwd for grouped-query attention (attn_fwd_gqa):
 * q, o, dout, dq: [B][h_q][T_q][d]; k, v, dk, dv: [B][h_kv][T_kv][d]. The
 * gradient of a key/value head is the sum over the h_q/h_kv query heads that
 * read it, formed in one pass (no atomics). h_kv == h_q is attn_bwd.
 */
attn_status_t attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o,
                           const void* dout, const float* lse, void* dq, void* dk, void* dv,
                           int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                           int causal, int dtype, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * attn_bwd_workspace_bytes -- workspace attn_bwd / attn_bwd_gqa need: two
 * fp32 row terms per query row, rows padded to 128 per head:
 * 8 * B * h_q * roundup(T_q, 128) bytes (0 for invalid or empty sizes).
 */
size_t attn_bwd_workspace_bytes(int B, int h, int T_q, int T_kv, int d);

/*
 * attn_fwd_paged_decode -- decode (one query row per sequence and head)
 * against a paged, variable-length KV cache, for batched serving.
 *
 * The cache lives in a pool of fixed-size pages: k_pages and v_pages are
 * [num_pages][h_kv][page_size][d] in the 16-bit dtype (a page holds
 * page_size consecutive cache rows of every key/value head, so one head's
 * rows in a page are contiguous). Sequence b's keys are rows
 * 0 .. seq_lens[b]-1 of the concatenation of pages block_table[b][0],
 * block_table[b][1], ...; block_table is int32 [B][max_pages_per_seq] and
 * seq_lens int32 [B], both in device memory (read by the kernel, never by
 * the host). q and o are [B][h_q][d] (T_q = 1), lse fp32 [B][h_q]; query
 * head i reads key/value head i / (h_q / h_kv). The pages name paging
 * among the ways serving systems manage the cache ("Attention and Its
 * Computational Cost", section "The other shape: one query, many keys");
 * the layout is this library's.
 *
 * Groups of 4 or more query heads per key/value head with pages of at least
 * 8 rows run on the tensor cores (each cached row read once for its whole
 * group); otherwise the CUDA-core kernel reads the cache once per query head.
 *
 * page_size: a power of two, 1..65536. A length above
 * max_pages_per_seq * page_size is clamped to it; a length <= 0 gives
 * o = 0 and lse = -inf for that sequence. A table entry outside
 * [0, num_pages) is never dereferenced (the CUDA-core kernel skips those
 * keys, the tensor-core path reads page 0 in their place, so that
 * sequence's outputs are unspecified) and the kernel records
 * ATTN_ERR_INVALID_ARG in the device status word (read it with
 * attn_get_device_error). Each sequence's keys are cut into num_splits
 * partitions (0 = the library's choice from max_pages_per_seq * page_size)
 * merged exactly as in attn_fwd's decode path. workspace: at least
 * attn_paged_workspace_bytes(...) bytes, 16-byte aligned, or NULL with
 * workspace_bytes 0 to have the library take it stream-ordered. Pointer
 * rules: q, o and the page pools 16-byte aligned, block_table, seq_lens and
 * lse 4-byte aligned; o and lse must not overlap any input or each other.
 */
attn_status_t attn_fwd_paged_decode(const void* q, const void* k_pages, const void* v_pages,
                                    const int* block_table, const int* seq_lens, void* o,
                                    float* lse, int B, int h_q, int h_kv, int d, int page_size,
                                    int max_pages_per_seq, int num_pages, float scale, int dtype,
                                    int num_splits, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * attn_paged_workspace_bytes -- workspace attn_fwd_paged_decode needs:
 * B*h_q*S*(d+4)*4 bytes, S = num_splits or the library's choice (which
 * depends on the grouping h_q / h_kv), 0 when the call needs none (the
 * tensor-core path with one partition) or for invalid sizes.
 */
size_t attn_paged_workspace_bytes(int B, int h_q, int h_kv, int d, int page_size,
                                  int max_pages_per_seq, int num_splits);

/*
 * attn_fwd_splitkv -- the prefill path (T_q > 1) with the key range of every
 * pair of 128-row query tiles cut into num_splits partitions: for short
 * queries against a long context, or a small batch x heads, where one CTA
 * per query-tile pair would leave most SMs idle. Each partition writes an
 * fp32 partial (unnormalised o, running max, running sum) per query row and
 * an exact merge combines them ("IO-Aware Attention: Tiling the Score Matrix
 * Without Materializing It", section "Parallelism and the cost of the
 * split": partitions over keys, merged with the same rescaling).
 *
 * Arguments as attn_fwd_gqa (h_kv == h_q for plain attention); T_q >= 2
 * (ATTN_ERR_INVALID_ARG otherwise: one row is the decode path).
 * num_splits: 0 = the library's choice (1 when the units already fill half
 * the SMs), else 1..64 (1 = the plain prefill kernel). workspace: at least
 * attn_splitkv_workspace_bytes(...) bytes (B*h_q*T_q*S*(d+4)*4; 0 when
 * S = 1), 16-byte aligned, not overlapping any argument, or NULL with
 * workspace_bytes 0 to have the library take it stream-ordered. attn_fwd
 * makes the same choice by itself; attn_fwd_ex and attn_fwd_gqa with a
 * caller workspace never split the prefill.
 */
attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               int B, int h_q, int h_kv, int T_q, int T_kv, int d, float scale,
                               int causal, int dtype, int num_splits, void* workspace,
                               size_t workspace_bytes, void* stream);

/* attn_splitkv_workspace_bytes -- workspace attn_fwd_splitkv needs (0 for
 * invalid sizes or one partition). */
size_t attn_splitkv_workspace_bytes(int B, int h_q, int T_q, int T_kv, int d, int num_splits);

/*
 * attn_fwd_naive -- the materialising forward, for comparison with the
 * IO-aware kernels: the standard attention of "Attention and Its
 * Computational Cost", section "The cost of writing down the scores" (one
 * T_q x T_kv score tensor per head, then a softmax, then P V) and of "E8.1
 * IO-aware attention" Part 2 (standard_attention). Three kernels write the
 * whole score matrix S = scale * Q K^T (masked entries -inf) and the whole
 * probability matrix P = softmax(S) to `workspace` as 16-bit
 * [B][h][T_q][T_kv] matrices, then form O = P V; lse comes from the softmax
 * pass. S and P are rounded to the 16-bit dtype (as a 16-bit framework
 * stores them), so results differ from attn_fwd by that rounding.
 * Arguments as attn_fwd (plain heads, h_kv == h); B*h <= 65535.
 *   workspace  device memory of at least attn_naive_workspace_bytes(B, h,
 *              T_q, T_kv) bytes (2 x B*h*T_q*T_kv x 2 bytes: S then P),
 *              16-byte aligned, not overlapping any argument; NULL with
 *              workspace_bytes 0: taken from and returned to the
 *              stream-ordered allocator.
 * Returns ATTN_ERR_WORKSPACE for a missing, short, misaligned or
 * overlapping workspace, ATTN_ERR_UNSUPPORTED for B*h > 65535, otherwise as
 * attn_fwd.
 */
attn_status_t attn_fwd_naive(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int h, int T_q, int T_kv, int d, float scale, int causal,
                             int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_naive_workspace_bytes -- bytes of the two materialised matrices of
 * attn_fwd_naive: 4 * B * h * T_q * T_kv (0 for negative sizes).
 */
size_t attn_naive_workspace_bytes(int B, int h, int T_q, int T_kv);

/*
 * attn_fwd_decode_noalloc -- the decode path (T_q == 1) without any
 * allocation, for callers that cannot allocate device memory at call time
 * (their memory is owned by another allocator, such as a serving engine that
 * reserves all of HBM up front, or they cannot accept the synchronisation a
 * cudaMalloc/cudaFree may bring). The pages have no counterpart: this is a
 * deployment variant of attn_fwd for one query row per (b, h).
 *
 * Same arguments and layout as attn_fwd with T_q = 1 (q, o: [B][h][1][d],
 * k, v: [B][h][T_kv][d]; a single query sees every key, so there is no
 * causal flag), plus num_splits as in attn_fwd_ex (0 = the library's
 * choice). It makes no cudaMalloc/cudaFree or other allocating call: the
 * split partials (B*h*S*(d+4)*4 bytes) live in a fixed device array owned by
 * the library, ATTN_NOALLOC_SCRATCH_BYTES on every device that loads it,
 * held until the library is unloaded. A shape whose partials do not fit
 * returns ATTN_ERR_WORKSPACE before anything is enqueued (fewer splits may
 * fit). Every call looks up the array's device address on the current
 * device (cudaGetSymbolAddress, which enqueues nothing, so a device reset
 * between calls is safe); the first call on a device may also load the
 * library's device code there, so make that first call before any stream
 * capture.
 * All calls on a device share the array: calls whose kernels overlap on the
 * GPU (e.g. on two streams without ordering) race and give wrong results.
 * The array keeps the last call's partials; nothing in it needs clearing.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
attn_status_t attn_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                      float* lse, int B, int h, int T_kv, int d, float scale,
                                      int dtype, int num_splits, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EXACT_IO_AWARE_ATTN_H */
