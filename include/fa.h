/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention forward library.
 *
 * What is computed (all entry points): for every query row i and query head h,
 *     O[i,h,:] = softmax_j( scale * q_i . k_j  over the keys j that row i may attend to ) . V
 *     LSE[i,h] = ln sum_j exp(scale * q_i . k_j)      (same key set)
 * This is the naive pipeline of "I/O-Aware Kernels" (datasystem.school, Module 5), section
 * "Naive attention: materializing the k x k score matrix", computed instead the way its section
 * "FlashAttention: tiling + online softmax" describes: one query tile stays on chip while key and
 * value tiles stream past it, with a running row maximum m and sum l and a rescaled output
 * accumulator, so the score matrix never reaches device memory. The paged entry point is the
 * serving form of its section "FlashInfer: I/O-aware attention for serving": keys and values are
 * gathered from a paged cache through a page table, over a ragged batch, with grouped-query heads.
 *
 * Conventions shared by every entry point
 *  - Tensors are bf16 (IEEE binary16-brain, passed as void*), contiguous, innermost dimension
 *    last. LSE is fp32. Accumulation is fp32; P is rounded to bf16 before P.V.
 *  - Grouped-query heads: query head h reads key/value head h / (Hq / Hkv); Hq % Hkv must be 0.
 *  - causal != 0 masks bottom-right aligned: row i of a sequence with q_len query rows and kv_len
 *    keys attends to key j iff j <= i + (kv_len - q_len). A row with no key gets O = 0 and
 *    LSE = -inf.
 *  - Supported head dims: d = 64 and d = 128. Every pointer must be 16-byte aligned.
 *  - Memory: the caller owns all device memory (inputs, outputs, workspace). The library never
 *    allocates or frees device memory. Its only global state is one device status word per GPU
 *    (see fa_get_device_status), a cached driver entry point, and for fa_cascade_fwd one stream
 *    and two events per calling host thread and GPU (created on first use, never freed).
 *  - Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *    FA_OK means validated and enqueued. Calls on different streams may run concurrently as
 *    long as they do not share an output or a workspace.
 *  - Threads: calls may be made from several host threads at once (with the exception noted at
 *    fa_paged_decode_noalloc); the library's host-side caches are atomic or behind a mutex.
 *  - Errors: arguments are checked on the host before anything is enqueued; no exception ever
 *    crosses this boundary. Kernels never trap: a device-side wait that runs past its time limit
 *    sets the device status word, which fa_get_device_status reports.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fa_stream_t; /* identical to cudaStream_t */

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, Hq % Hkv != 0, bad lengths */
  FA_ERR_UNSUPPORTED = 2,     /* head dim not 64/128, page size not in {16,32,64,128}, too large */
  FA_ERR_ALIGNMENT = 3,       /* a pointer is not 16-byte aligned */
  FA_ERR_WORKSPACE = 4,       /* workspace missing or smaller than fa_paged_workspace_bytes() */
  FA_ERR_CUDA = 5,            /* a CUDA runtime/driver call or a launch failed */
  FA_ERR_NO_DEVICE = 6,       /* current device is not an sm_103 GPU */
  FA_ERR_DEVICE_TIMEOUT = 7,  /* a kernel gave up waiting on a pipeline barrier (device status) */
  FA_ERR_DEVICE_BAD_PAGE = 8  /* a kernel met a page id outside [0, num_pages) (device status) */
} fa_status;

/* Human-readable name of a status code (static storage, never NULL). The pages define no error
 * handling; this boundary reports every failure as a returned code (never an exception or a trap),
 * and this call names the codes. */
const char* fa_status_string(fa_status s);

/*
 * Dense attention forward ("FlashAttention: tiling + online softmax").
 *   q, o: [B, S, Hq, d] bf16;  k, v: [B, S, Hkv, d] bf16;  lse: [B, S, Hq] fp32 or NULL (skip).
 *   scale multiplies q.k before the softmax (usually 1/sqrt(d)).
 * Returns FA_OK when enqueued. B, S, Hq, Hkv >= 1.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int S, int d, int causal, float scale, fa_stream_t stream);

/*
 * Paged, ragged attention forward ("FlashInfer: I/O-aware attention for serving").
 *   q, o:          [total_q, Hq, d] bf16, sequences packed back to back;
 *   k_pages, v_pages: [num_pages, page_size, Hkv, d] bf16 (a shared page pool);
 *   page_table:    [num_seqs, max_pages_per_seq] int32 physical page ids; entries past a
 *                  sequence's last page are never read (may be -1);
 *   cu_seqlens_q:  [num_seqs + 1] int32 prefix sums of query lengths (cu[0] = 0,
 *                  cu[num_seqs] = total_q);
 *   kv_lens:       [num_seqs] int32 key/value lengths, 0 <= kv_len <= max_pages_per_seq*page_size;
 *   lse:           [total_q, Hq] fp32 or NULL.
 *   max_q_len:     the largest query length (a host-side bound, used for planning).
 *                  Batches run on the tiled tensor-core kernel; when the GQA group (Hq / Hkv) is
 *                  a power of two from 2 to 128 (MQA included) the group's query heads share
 *                  each tile (rows = token x head), so decode and multi-token verify rows fill
 *                  the tensor core too (decode included: it stays bound by reading K/V).
 *   num_splits:    key splits: each sequence's keys are cut into num_splits contiguous ranges,
 *                  attended in parallel as fp32 partial states and merged by their LSE. 0 chooses
 *                  from the SM count (splits only when there is too little other parallelism).
 *   workspace:     device scratch of at least fa_paged_workspace_bytes(...) bytes (may be NULL
 *                  when that function returns 0). Its contents need no initialisation; calls that
 *                  share a workspace must be ordered on one stream.
 * Device arrays (page_table, cu_seqlens_q, kv_lens) are read on the device only.
 */
fa_status fa_paged_fwd(const void* q, const void* k_pages, const void* v_pages,
                       const int32_t* page_table, const int32_t* cu_seqlens_q,
                       const int32_t* kv_lens, int num_seqs, int total_q, int max_q_len,
                       int page_size, int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d,
                       int causal, float scale, void* o, float* lse, void* workspace,
                       size_t workspace_bytes, int num_splits, fa_stream_t stream);

/* Workspace bytes fa_paged_fwd needs for these sizes (same num_splits argument, 0 = auto). The
 * pages name no workspace: it exists because the caller owns all device memory (the library never
 * allocates), so the caller must learn how much scratch a call needs -- the planned work list and,
 * when keys are split, the fp32 partial states the LSE merge combines. It takes the same shape
 * arguments as the call it sizes because the plan (GQA packing, key splits) depends on them. */
size_t fa_paged_workspace_bytes(int num_seqs, int total_q, int max_q_len, int page_size,
                                int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d,
                                int num_splits);

/* The key-split count fa_paged_fwd plans for a batch with these sizes (num_splits = 0): 1 means
 * no split. Host-side only. */
int fa_paged_num_splits(int num_seqs, int total_q, int max_q_len, int page_size,
                        int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d);

/* The split count the split-KV CUDA-core decode kernel uses for a decode batch with these sizes
 * (num_splits = 0). That kernel serves fa_paged_decode_noalloc, and fa_paged_fwd's decode batches
 * when the environment variable FA_DECODE_TC is 0. */
int fa_decode_num_splits(int num_seqs, int page_size, int max_pages_per_seq, int num_pages,
                         int Hkv);

/*
 * Merge partial attention states (the LSE-weighted combine of split-KV decode).
 *   o_parts:   [num_parts, n_rows, H, d] fp32, each part normalised over its own keys;
 *   lse_parts: [num_parts, n_rows, H] fp32 (natural log; -inf marks a part with no keys);
 *   o:         [n_rows, H, d] bf16;  lse: [n_rows, H] fp32 or NULL.
 * Result: lse = ln sum_p exp(lse_p);  O = sum_p exp(lse_p - lse) * O_p  (O = 0 if all parts
 * are empty). Equivalent to attending over the union of the parts' keys.
 */
fa_status fa_merge_states(const float* o_parts, const float* lse_parts, int num_parts, int n_rows,
                          int H, int d, void* o, float* lse, fa_stream_t stream);

/*
 * Shared-prefix (cascade) attention over a paged cache.
 * "I/O-Aware Kernels" (datasystem.school, Module 5), section "FlashInfer: I/O-aware attention
 * for serving": serving batches reuse long shared prefixes (the prefix sharing of RadixAttention);
 * keys and values of a prefix that many sequences share are attended once for all of their query
 * rows, and the result is combined with each sequence's own keys by the LSE merge above.
 *   Sequences are split into num_groups consecutive groups. Group g owns the query rows
 *   [cu_q_groups[g], cu_q_groups[g+1]) of q -- the rows of all its sequences, so cu_q_groups[g]
 *   equals cu_seqlens_q at the group's first sequence; cu_q_groups[0] = 0 and
 *   cu_q_groups[num_groups] = total_q -- and a shared prefix of prefix_lens[g] keys in the pages
 *   prefix_page_table[g][0 .. max_prefix_pages).
 *   Sequence s owns kv_lens[s] further keys (its suffix) in page_table[s][0 .. max_pages_per_seq);
 *   its query rows [cu_seqlens_q[s], cu_seqlens_q[s+1]) are the last tokens of that suffix.
 * Result (o bf16 [total_q, Hq, d], lse fp32 [total_q, Hq] or NULL): exactly fa_paged_fwd over the
 * concatenated keys prefix(g) ++ suffix(s) of every sequence. Every query row sees the whole
 * prefix; with causal != 0 the suffix is masked bottom-right, which needs q_len(s) <= kv_lens[s]
 * (the query tokens lie in the suffix). Both passes run the same kernels as fa_paged_fwd with
 * fp32 outputs, then one merge. The suffix pass runs on a second stream of the library's (one per
 * calling host thread and GPU, created on first use), forked from `stream` with an event after
 * the prefix pass's planning kernel and joined back into it before the merge, so the two passes
 * share the GPU, the prefix pass starting on its SMs first: the
 * call is ordered on `stream` like any other (and can be captured in a CUDA graph from it).
 *   max_group_q_len / max_q_len: host-side bounds of the query rows per group / per sequence.
 *   workspace: at least fa_cascade_workspace_bytes(...) bytes, 256-byte aligned.
 * Errors as for fa_paged_fwd; also FA_ERR_INVALID_ARG when num_groups > num_seqs.
 */
size_t fa_cascade_workspace_bytes(int num_groups, int num_seqs, int total_q, int max_group_q_len,
                                  int max_q_len, int page_size, int max_prefix_pages,
                                  int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d);
fa_status fa_cascade_fwd(const void* q, const void* k_pages, const void* v_pages, int page_size,
                         int num_pages, int Hq, int Hkv, int d, float scale, int num_groups,
                         const int32_t* cu_q_groups, const int32_t* prefix_page_table,
                         const int32_t* prefix_lens, int max_prefix_pages, int max_group_q_len,
                         int num_seqs, const int32_t* cu_seqlens_q, const int32_t* page_table,
                         const int32_t* kv_lens, int max_pages_per_seq, int max_q_len, int causal,
                         int total_q, void* o, float* lse, void* workspace, size_t workspace_bytes,
                         fa_stream_t stream);

/*
 * Paged KV append: write the key/value rows of new tokens into their page slots.
 * "I/O-Aware Kernels" (datasystem.school, Module 5), section "FlashInfer: I/O-aware attention
 * for serving": the cache is a pool of fixed-size pages reached through a per-sequence page
 * table; a sequence grows by filling the slot after its current length.
 *   k_new, v_new:    [total_new, Hkv, d] bf16, the new tokens packed sequence after sequence
 *                    (may be NULL when total_new == 0);
 *   cu_seqlens_new:  [num_seqs + 1] int32 (device), row offsets of each sequence's new tokens,
 *                    cu_seqlens_new[0] == 0 and cu_seqlens_new[num_seqs] == total_new;
 *   kv_lens_before:  [num_seqs] int32 (device), cached tokens of each sequence before the call;
 *   page_table:      [num_seqs, max_pages_per_seq] int32 (device), physical page ids;
 *   k_pages, v_pages: [num_pages, page_size, Hkv, d] bf16, written in place.
 * New row r of sequence s lands at logical position p = kv_lens_before[s] + r, i.e. in page
 * page_table[s][p / page_size], slot p % page_size. Nothing else in the pool is touched and
 * kv_lens_before is not updated (the caller's new length is kv_lens_before + the row count).
 * The caller must have mapped every page the new rows reach. A row whose position falls outside
 * the table or whose page id is outside [0, num_pages) is skipped and FA_ERR_DEVICE_BAD_PAGE is
 * recorded in the device status word. Two rows mapped to one slot race (the caller's error).
 * Errors: FA_ERR_INVALID_ARG (null pointer, non-positive size), FA_ERR_UNSUPPORTED (d not 64 or
 * 128; page_size not 16, 32, 64 or 128), FA_ERR_ALIGNMENT (bf16 buffers not 16-byte aligned,
 * int32 arrays not 4-byte aligned), FA_ERR_CUDA. Asynchronous on `stream`; allocates nothing.
 */
fa_status fa_paged_append(const void* k_new, const void* v_new, const int32_t* cu_seqlens_new,
                          const int32_t* kv_lens_before, const int32_t* page_table, int num_seqs,
                          int total_new, int page_size, int max_pages_per_seq, int num_pages,
                          int Hkv, int d, void* k_pages, void* v_pages, fa_stream_t stream);

/*
 * Split-KV paged decode for callers that cannot allocate device memory. The pages have no
 * counterpart of this entry point; it exists for callers that may not call cudaMalloc (for
 * example an engine whose device memory is all handed to a fixed arena, or a plugin inside a
 * host that owns every allocation) and so cannot lend fa_paged_fwd a workspace.
 *   Arguments and results are those of fa_paged_fwd for a decode batch (every query length is
 *   0 or 1, i.e. max_q_len == 1); inputs and outputs are still the caller's. total_q must be at
 *   most num_seqs (FA_ERR_INVALID_ARG otherwise) and num_seqs at most 65535 (FA_ERR_UNSUPPORTED
 *   otherwise), both checked before anything is enqueued. It always runs the split-KV CUDA-core
 *   decode kernel, which takes GQA groups (Hq / Hkv) of 1, 2, 4 and 8; other groups return
 *   FA_ERR_UNSUPPORTED.
 *   Scratch: the per-split partials live in a fixed device array of FA_NOALLOC_SCRATCH_BYTES
 *   (16 MiB) inside this library, which every GPU that loads the library holds until the process
 *   exits. The function itself allocates and frees nothing.
 *   A split count is first capped at max_pages_per_seq. num_splits > 0 whose scratch after that
 *   cap (splits * num_seqs * Hq * (d + 1) floats of partials plus one int per sequence and block
 *   of up to 8 kv heads, each part 256-byte aligned) exceeds the array is rejected with
 *   FA_ERR_WORKSPACE before anything is enqueued; num_splits == 0 lowers the automatic count
 *   (fa_decode_num_splits) until it fits.
 *   Sharing: every call on a device uses the same scratch, which keeps the last call's contents;
 *   the merge counters in it are cleared by each call (an asynchronous memset on `stream`). Calls
 *   whose kernels overlap on the GPU -- on two streams, or from two threads -- race on it; order
 *   them on one stream.
 *   Set-up: the first call on each device looks up the scratch's device address with that device
 *   current (a host-side symbol lookup). Make that first call before any stream capture.
 */
#define FA_NOALLOC_SCRATCH_BYTES (16u << 20)
fa_status fa_paged_decode_noalloc(const void* q, const void* k_pages, const void* v_pages,
                                  const int32_t* page_table, const int32_t* cu_seqlens_q,
                                  const int32_t* kv_lens, int num_seqs, int total_q, int page_size,
                                  int max_pages_per_seq, int num_pages, int Hq, int Hkv, int d,
                                  float scale, void* o, float* lse, int num_splits,
                                  fa_stream_t stream);

/*
 * Read and clear this GPU's device status word. Synchronises `stream` first. The pages define no
 * failure reporting; kernels here never trap, so a device-side failure (a bounded wait that gave
 * up, a page id outside the pool) is recorded in this word and read back through this call.
 * *code receives FA_OK, FA_ERR_DEVICE_TIMEOUT or FA_ERR_DEVICE_BAD_PAGE; *site (may be NULL) a
 * small id of the place in the kernels that recorded it. Returns FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_get_device_status(fa_stream_t stream, int* code, int* site);

/*
 * Diagnostic of the device-side failure path: launches one warp that waits on a barrier phase
 * nothing completes, with a wait limit of limit_ms (1..2000). The wait must give up, record
 * FA_ERR_DEVICE_TIMEOUT in the device status word and let the kernel exit; nothing traps or
 * hangs. Synchronises `stream`, then returns in *code (and *site, may be NULL) what the status
 * word held, and clears it. Returns FA_OK when the check ran (inspect *code for its result).
 */
fa_status fa_selftest_wait_timeout(int limit_ms, int* code, int* site, fa_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FA_GB300_H */
