/*
 * pcp.h — C ABI of libpcp: Prefill Context Parallel (PCP) attention for GQA/MHA
 * layers on NVIDIA GB300 (sm_103a).
 *
 * The method, as the three pull-request pages on PCP for vLLM describe it:
 *  - "Feat/pcp qwen36 hybrid", section "Changes": each PCP rank takes a
 *    contiguous slice of the prompt; full-attention layers all-gather K/V and
 *    run end-aligned (bottom-right) causal attention of the slice against it.
 *  - "[MRv2] FlashAttention PCP support for GQA on MRv2", "Pull request
 *    overview": an optional cached-prefix (context) pass returning
 *    (ctx_out, ctx_lse) merged with the new-token pass by log-sum-exp; mixed
 *    prefill + decode batches; a PCP-aware KV-cache update. Review: callers
 *    pass the output and a workspace so nothing is allocated per step.
 *  - "[MRv2][PCP] Carry the row plan in attention metadata; fix mixed
 *    prefill+decode crash": a rank-local batch holds up to two rows per
 *    prefilling request (section 2); the gathered slot mapping masks every
 *    entry a rank must not write with a negative PAD slot and the cache writer
 *    skips negative slots, decode rows being written by rank 0 only (commit
 *    "drop pcp_has_prefill"); a row's seq_len is its end position, so
 *    seq_len - query_len is the row start ("What made it removable").
 *
 * On one GPU the PCP ranks are emulated as query shards of one batch and the
 * all-gathered K/V is the resident paged cache, so no call here communicates.
 *
 * Conventions for every function:
 *  - The return value is a status: PCP_OK (0) or a negative PCP_ERR_* code.
 *    No function aborts, throws or prints.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call launches nothing and leaves every buffer untouched.
 *  - Device functions are asynchronous on `stream` (0 = the legacy default
 *    stream). The caller owns every buffer and the stream; the library
 *    allocates no device memory in any call.
 *  - `status` (where present) is a device int32 that the kernels set with the
 *    first error they meet (PCP_ERR_RANGE for an out-of-range block id or
 *    slot, PCP_ERR_TIMEOUT for a bounded wait that ran out). It is never reset
 *    by the library: zero it before the call, read it after synchronising.
 *  - bf16 tensors are raw 16-bit IEEE bfloat16; pointers named *_cache and the
 *    q/k/v/out tensors must be 16-byte aligned (PCP_ERR_ALIGN otherwise).
 *
 * Layouts (T = total new tokens, packed request-major, positions ascending):
 *  q, out        [T][Hq][D]                 bf16
 *  k, v (new)    [T][Hkv][D]                bf16
 *  key_cache,
 *  value_cache   [num_blocks][block_size][Hkv][D]  bf16 (the paged cache)
 *  block_table   [num_reqs][max_blocks_per_req]    int32 page ids, row-major
 *  lse           [Hq][T]                    fp32, natural log
 *  slot_mapping  [T]                        int64, slot = page * block_size + offset
 * q head h reads kv head h / (Hq / Hkv).
 */
#ifndef PCP_H_
#define PCP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pcp_stream_t; /* == cudaStream_t */

/* status codes */
#define PCP_OK 0
#define PCP_ERR_ARG (-1)         /* null pointer, negative or inconsistent size */
#define PCP_ERR_RANGE (-2)       /* page id, slot or row range out of range */
#define PCP_ERR_UNSUPPORTED (-3) /* head_dim, block_size or head ratio not supported */
#define PCP_ERR_ALIGN (-4)       /* pointer not 16-byte aligned */
#define PCP_ERR_CUDA (-5)        /* a CUDA call failed; see pcp_last_cuda_error() */
#define PCP_ERR_TIMEOUT (-6)     /* a bounded device wait ran out (reported via status) */
#define PCP_ERR_WORKSPACE (-7)   /* workspace missing or too small */

/* split modes of pcp_build_row_plan */
#define PCP_SPLIT_CONTIGUOUS 0
#define PCP_SPLIT_DUAL_CHUNK 1

/* flags of pcp_attn_varlen */
#define PCP_ATTN_SEPARATE_CONTEXT 1  /* compute the context and new-token parts as two
                                        partials in the workspace and merge them by LSE */
#define PCP_ATTN_SPLIT_AT_ROW_START 2 /* with SEPARATE_CONTEXT: split each row at its own
                                        start instead of at the cached prefix */
/* Decode-context-parallel emulation: each prefill row is computed as n partials over n
 * contiguous shards of its keys [0, kv_end) — what n DCP ranks holding those key shards
 * would each compute — and the partials are merged by LSE in the same call
 * (2 <= n <= 64; not combinable with PCP_ATTN_SEPARATE_CONTEXT). */
#define PCP_ATTN_KV_SHARDS(n) (((n) & 0xFF) << 8)
/* Decode rows beside the prefill: the decode rows run on n SMs on a stream of the
 * library's own while the prefill rows take the other SMs, instead of one after
 * the other on every SM (1 <= n < the SM count; pcp_decode_sms picks n). Used
 * where the tensor-core decode applies (head_dim 128, up to 16 q heads per kv head
 * with a bf16 cache and 8 with an FP8 one, at most 1024 rows); with n = 0, n at or
 * above the SM count, or another shape the rows run in sequence. The prefill rows' results are the same bits
 * either way; the decode rows' agree up to the rounding of their fp32 sums (the key
 * tiles of a decode item are shared between two softmax warpgroups by a count that
 * runs on across a CTA's items, so another split adds the same terms in another
 * order). A given split gives the same bits on every run. */
#define PCP_ATTN_DECODE_SMS(n) (((n) & 0xFF) << 16)

/* One row of the plan: a contiguous run of one request's new tokens that one
 * shard evaluates. All fields are int32.
 *  req        request index
 *  shard      emulated PCP rank that owns the row
 *  q_start    packed index of the row's first token in q / out / k / v
 *  q_len      number of query tokens (> 0)
 *  ctx_len    cached prefix length of the request (keys [0, ctx_len) are the context)
 *  kv_end     end position of the row = ctx_len + (row end within the request's new tokens);
 *             the row's query j sits at position kv_end - q_len + j and sees keys
 *             [0, kv_end - q_len + j] (end-aligned causal)
 *  causal_off kv_end - ctx_len - q_len: the row start among the request's new tokens
 *  is_decode  1 for a single new token after a non-empty prefix */
typedef struct pcp_row_t {
    int32_t req, shard, q_start, q_len, ctx_len, kv_end, causal_off, is_decode;
} pcp_row_t;

/*
 * pcp_build_row_plan — host function, pure and deterministic.
 * ("Feat/pcp qwen36 hybrid", "Changes"; "Carry the row plan ...", section 2 and
 * "What made it removable"; "drop pcp_has_prefill".)
 *
 * Request r has query_len[r] >= 0 new tokens after num_computed[r] >= 0 cached
 * ones. Its new tokens are cut into shard rows:
 *   PCP_SPLIT_CONTIGUOUS  shard i gets [floor(i N / S), floor((i+1) N / S));
 *   PCP_SPLIT_DUAL_CHUNK  2S chunks [floor(k N / 2S), floor((k+1) N / 2S)); shard i
 *                         gets chunk i and chunk 2S-1-i (head and tail);
 * a request with one new token is a single row on shard 0; empty chunks give no
 * row. Rows are written shard-major: shard, then request, then chunk order.
 *
 * Inputs (host memory): query_len[num_reqs], num_computed[num_reqs],
 *   block_table[num_reqs][max_blocks_per_req] (only the pages holding new tokens are read).
 * Outputs (host memory, caller-allocated):
 *   rows[rows_capacity]     rows_capacity >= 2 * num_shards * num_reqs always suffices
 *   *num_rows
 *   cu_q[*num_rows + 1]     running sum of q_len over rows (size it rows_capacity + 1)
 *   slot_mapping[T]         slot of every new token: block_table[r][pos / bs] * bs + pos % bs
 *   owner_shard[T]          shard of the row holding each token; may be NULL
 * Errors: PCP_ERR_ARG (null pointer, negative length, num_shards < 1 or > 127,
 *   bad split mode, block_size < 1); PCP_ERR_RANGE (a needed page is negative or
 *   beyond max_blocks_per_req, or the rows do not fit rows_capacity). Outputs are
 *   unspecified after an error.
 */
int pcp_build_row_plan(int32_t num_reqs, const int32_t* query_len, const int32_t* num_computed,
                       const int32_t* block_table, int32_t max_blocks_per_req, int32_t block_size,
                       int32_t num_shards, int32_t split_mode, pcp_row_t* rows,
                       int32_t rows_capacity, int32_t* num_rows, int32_t* cu_q,
                       int64_t* slot_mapping, int8_t* owner_shard);

/*
 * pcp_mask_slots_for_shard — host function. The PAD-masked slot mapping one
 * rank hands to its cache writer ("drop pcp_has_prefill"): out[t] = slot[t]
 * where owner_shard[t] == shard, else -1. slot/owner/out are host arrays of
 * num_tokens entries; out may alias slot. Errors: PCP_ERR_ARG.
 */
int pcp_mask_slots_for_shard(const int64_t* slot_mapping, const int8_t* owner_shard,
                             int32_t num_tokens, int32_t shard, int64_t* out);

/*
 * pcp_decode_sms — host function, pure. The SMs to give the decode rows of a
 * row plan (rows, num_rows in host memory, as pcp_build_row_plan wrote them)
 * when they run beside its prefill rows (PCP_ATTN_DECODE_SMS), or 0 to run them
 * one after the other. Mixed prefill + decode batches are the pages' case
 * ("[MRv2] FlashAttention PCP support for GQA on MRv2", overview); the split is
 * this library's. On a few SMs the decode rows are no longer held to the
 * SMs' share of HBM bandwidth, so they take less SM time than on all of them.
 * The function balances that time (K and V bytes of the decode rows at a
 * per-SM rate) against the prefill rows' (per work item and per 128-key tile
 * at the measured rates of this library's kernels), rounding towards the
 * decode side. It returns 0 when either side is empty, when the decode rows
 * would need half the SMs or more, when the tensor-core decode does not apply
 * (head_dim != 128, Hq / Hkv > 16, more than 1024 rows), and for an FP8 cache
 * (kv_cache_fp8 != 0: its decode is bound by widening V on few SMs; measured no
 * gain). num_sms: the SM count of the device (>= 2). Errors: none (bad
 * arguments return 0).
 */
int32_t pcp_decode_sms(const pcp_row_t* rows, int32_t num_rows, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t kv_cache_fp8, int32_t num_sms);

/*
 * pcp_kv_cache_write — device. Scatter the new tokens' K and V into the paged
 * cache: key_cache[slot / bs][slot % bs][h][:] = k[t][h][:] (same for V) for every
 * t with slot_mapping[t] >= 0; negative slots are skipped ("drop
 * pcp_has_prefill"). The write must precede the attention of the same step
 * ("What made it removable": the cache update is ordered before attention);
 * issuing both on one stream does that.
 * k, v, slot_mapping, key_cache, value_cache, status: device pointers;
 * key_cache and value_cache overlap neither each other nor k, v or
 * slot_mapping (PCP_ERR_ARG).
 * A slot >= num_blocks * block_size is skipped and sets *status = PCP_ERR_RANGE.
 * Supported: a token row of Hkv * head_dim * 2 bytes a multiple of 16. Errors:
 * PCP_ERR_ARG, PCP_ERR_ALIGN, PCP_ERR_UNSUPPORTED, PCP_ERR_CUDA (launch failure).
 */
int pcp_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                       int32_t num_tokens, void* key_cache, void* value_cache, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t* status,
                       pcp_stream_t stream);

/*
 * pcp_attn_workspace_size — bytes of device workspace pcp_attn_varlen needs.
 * max_kv_len is the key capacity of a block-table row
 * (max_blocks_per_req * block_size). Never fails; returns 0 for invalid sizes.
 */
size_t pcp_attn_workspace_size(int32_t num_rows, int32_t total_q, int32_t num_q_heads,
                               int32_t head_dim, int32_t max_kv_len, int32_t flags);

/*
 * pcp_attn_varlen — device. Attention of every planned row in one call:
 * prefill rows (end-aligned causal over the new tokens, plus the non-causal
 * context over the cached prefix) on the tensor cores, decode rows on a
 * split-KV bandwidth path (tensor cores for head_dim 128 with up to 16 q heads
 * per kv head, 8 over an FP8 cache, and at most 1024 rows, P carried as bf16
 * hi + lo; CUDA cores in fp32 otherwise). ("Feat/pcp qwen36 hybrid", "Changes"; "[MRv2]
 * FlashAttention PCP support ...", overview and the context-pass call returning
 * (ctx_out, ctx_lse); "Carry the row plan ...", "What made it removable".)
 *
 * For query j of a row (position p = kv_end - q_len + j) and q head h:
 *   s_k   = scale * q[t][h] . K[req][k][h / G]           for keys k in [0, p]
 *   out   = sum_k softmax(s)_k V[req][k][h / G]          (bf16, rounded from fp32)
 *   lse   = log sum_k exp(s_k)                            (fp32, natural log)
 * K/V are read from the paged cache through block_table[req].
 *
 * q, key_cache, value_cache, block_table ([num_reqs][max_blocks_per_req]), rows,
 * out, lse, workspace, status: device pointers. rows[num_rows] is the plan (any
 * row order; the q ranges must be disjoint). The kernels check every row
 * (0 <= req < num_reqs, q_len >= 1, [q_start, q_start + q_len) inside
 * [0, total_q), q_len <= kv_end <= max_blocks_per_req * block_size,
 * 0 <= ctx_len <= kv_end, a decode row has q_len == 1) and skip a bad row with
 * *status = PCP_ERR_RANGE. Tokens not covered by any row are
 * not written (padding is never computed). workspace: at least
 * pcp_attn_workspace_size(num_rows, total_q, Hq, D, max_blocks_per_req * block_size, flags)
 * bytes, 256-byte aligned; its contents on entry do not matter.
 * flags: 0 computes every row in one online softmax; PCP_ATTN_SEPARATE_CONTEXT
 * computes the context part and the new-token part as two partial results in
 * the workspace and merges them by LSE (a part with no keys has lse = -inf and
 * out = 0); PCP_ATTN_SPLIT_AT_ROW_START moves the split point to the row start;
 * PCP_ATTN_KV_SHARDS(n) computes n partials over n contiguous key shards and
 * merges them (decode rows are always split-KV internally; flags do not change
 * their result). Every mode gives the same attention up to rounding.
 * PCP_ATTN_DECODE_SMS(n) runs the decode rows on n SMs beside the prefill rows,
 * on an internal stream forked from `stream` after the row checks and joined
 * back into `stream` before the call returns (a capture of `stream` takes both;
 * the first such call in a CUDA context creates the internal stream and its two
 * events, so make it before any stream capture). Calls from several host
 * threads take turns on that stream.
 * Numerics: scores, softmax and sums in fp32, P rounded to bf16 for the
 * P V product; the result is finite whenever every scale * q . k is finite in
 * fp32 and ceil(keys / 128) * max |v| < 2^64, e.g. |v| < 2^54 at 131072 keys
 * (a 128-key tile's exponentials may sum to 2^64 against a stale row maximum
 * before the exact rescaling path takes over).
 * scale: any finite float (PCP_ERR_ARG otherwise). out and lse overlap
 * neither each other nor any input buffer (q, the caches, block_table, rows,
 * the used workspace; PCP_ERR_ARG).
 * Supported: head_dim 64 or 128, block_size in {8, 16, 32, 64, 128},
 * Hq % Hkv == 0 with Hq / Hkv <= 16.
 * Rows with an out-of-range page id are skipped in part and set *status =
 * PCP_ERR_RANGE; a device wait that runs out sets PCP_ERR_TIMEOUT.
 * Errors (nothing launched): PCP_ERR_ARG, PCP_ERR_ALIGN, PCP_ERR_UNSUPPORTED,
 * PCP_ERR_WORKSPACE; PCP_ERR_CUDA for a failed launch.
 */
int pcp_attn_varlen(const void* q, const void* key_cache, const void* value_cache,
                    const int32_t* block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                    int64_t num_blocks,
                    int32_t block_size, const pcp_row_t* rows, int32_t num_rows, int32_t total_q,
                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                    void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t flags,
                    int32_t* status, pcp_stream_t stream);

/*
 * pcp_attn_varlen_noalloc — device. No counterpart on the pages: an addition
 * for callers that cannot allocate device memory (a host framework that owns
 * all device memory through its own allocator, or a serving loop that must
 * not call cudaMalloc after start-up because the call can synchronise the
 * device and has no latency bound). It is pcp_attn_varlen without the
 * workspace arguments: the library supplies a fixed 64 MiB scratch array that
 * every GPU loading the library reserves until the process exits, and the
 * call allocates nothing.
 * Same arguments, semantics, checks (in the same order) and errors as
 * pcp_attn_varlen; where that call would check the workspace size, this one
 * returns PCP_ERR_WORKSPACE (nothing launched) when
 * pcp_attn_workspace_size(num_rows, total_q, Hq, D, max_blocks_per_req *
 * block_size, flags) exceeds 64 MiB, and PCP_ERR_CUDA when the array's device
 * address cannot be looked up.
 * The first call in a CUDA context looks up the array's device address with
 * that context current (cudaGetSymbolAddress) and keeps it for that context;
 * make that first call before any stream capture. A device reset ends the
 * context, and the first call in the next one looks the address up again.
 * All calls on a device share the array: calls whose kernels may overlap on
 * the GPU (other streams or threads) race on it — serialise them on one
 * stream.
 */
int pcp_attn_varlen_noalloc(const void* q, const void* key_cache, const void* value_cache,
                            const int32_t* block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                            int64_t num_blocks, int32_t block_size, const pcp_row_t* rows,
                            int32_t num_rows, int32_t total_q, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim, float scale, void* out, float* lse,
                            int32_t flags, int32_t* status, pcp_stream_t stream);

/*
 * pcp_kv_cache_write_fp8 — device. pcp_kv_cache_write into an FP8 cache: one
 * byte per element, the e4m3 code (OCP 8-bit floating point, no infinities,
 * largest finite 448) of x / k_scale for keys and x / v_scale for values, the
 * division correctly rounded in fp32, then rounded to nearest even and
 * saturated at +-448. k_scale and v_scale are the layer's scales ("[MRv2]
 * FlashAttention PCP support ...", the context-pass call: layer._k_scale,
 * layer._v_scale), host floats, finite and > 0 (else PCP_ERR_ARG).
 * key_cache, value_cache: [num_blocks][block_size][Hkv][D] bytes. Same slot, overlap,
 * PAD and status rules as pcp_kv_cache_write. Supported: Hkv * D a multiple of
 * 16. Errors: PCP_ERR_ARG, PCP_ERR_ALIGN, PCP_ERR_UNSUPPORTED, PCP_ERR_CUDA.
 */
int pcp_kv_cache_write_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                           int32_t num_tokens, void* key_cache, void* value_cache, int64_t num_blocks,
                           int32_t block_size, int32_t num_kv_heads, int32_t head_dim, float k_scale,
                           float v_scale, int32_t* status, pcp_stream_t stream);

/*
 * pcp_attn_varlen_fp8kv — device. pcp_attn_varlen over an FP8 (e4m3) paged
 * cache with per-(request, kv head) descales ("[MRv2] FlashAttention PCP
 * support ...", the context-pass call: descales of shape (num_seqs,
 * num_kv_heads)). Key k of request r and kv head g is code_K[r][k][g][:] *
 * k_descale[r][g], its value code_V[...] * v_descale[r][g]; the result is the
 * same attention as pcp_attn_varlen over those keys and values. head_dim 128:
 * the scores take the K codes as e4m3 MMA operands against q written as two
 * e4m3 terms per element after a power-of-two scale per query row (prefill)
 * or per q head (decode rows); the terms sum to the bf16 q exactly for every
 * element of at least 2^-9 of the row's largest magnitude; a smaller element
 * can lose bits, at most 2^-17 of that largest. V is widened to f16 (exact) and the softmax weights P are f16 (decode
 * rows with up to 8 q heads per kv head: two f16 parts; more: fp32). head_dim
 * 64: the prefill rows' products run in f16 (codes widened, q converted to f16,
 * P f16) and decode rows in fp32. An
 * element of q beyond +-65504 sets *status = PCP_ERR_RANGE (with head_dim 64
 * it is saturated to +-65504). The descales multiply the fp32 scores and
 * outputs.
 * key_cache, value_cache: [num_blocks][block_size][Hkv][D] bytes (as written
 * by pcp_kv_cache_write_fp8); k_descale, v_descale: device fp32
 * [num_reqs][Hkv] (inputs: out and lse must not overlap them). Every other
 * argument, check, flag and error is that of pcp_attn_varlen, with the same
 * workspace size.
 */
int pcp_attn_varlen_fp8kv(const void* q, const void* key_cache, const void* value_cache,
                          const float* k_descale, const float* v_descale, const int32_t* block_table,
                          int32_t num_reqs, int32_t max_blocks_per_req, int64_t num_blocks,
                          int32_t block_size, const pcp_row_t* rows, int32_t num_rows, int32_t total_q,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                          void* out, float* lse, void* workspace, size_t workspace_bytes, int32_t flags,
                          int32_t* status, pcp_stream_t stream);

/*
 * pcp_lse_merge — device. Merge two partial results of the same queries by
 * log-sum-exp ("[MRv2] FlashAttention PCP support ...": (ctx_out, ctx_lse)
 * combined with the new-token pass; the per-step LSE-combine of the DCP
 * benchmark):
 *   m = max(lse_a, lse_b), w_x = exp(lse_x - m),
 *   out = (w_a out_a + w_b out_b) / (w_a + w_b), lse = m + log(w_a + w_b);
 * a part with lse = -inf contributes nothing; both -inf give out = 0, lse = -inf.
 * out_a, out_b: [total_q][Hq][D] fp32; lse_a, lse_b, lse: [Hq][total_q] fp32;
 * out: [total_q][Hq][D] bf16. All device pointers; out and lse overlap neither
 * each other nor any of the four inputs (no in-place merge: PCP_ERR_ARG).
 * Errors: PCP_ERR_ARG, PCP_ERR_ALIGN, PCP_ERR_UNSUPPORTED (head_dim % 8 != 0),
 * PCP_ERR_CUDA.
 */
int pcp_lse_merge(const float* out_a, const float* lse_a, const float* out_b, const float* lse_b,
                  void* out, float* lse, int32_t total_q, int32_t num_q_heads, int32_t head_dim,
                  pcp_stream_t stream);

/*
 * pcp_set_profile_events — host. A tracing hook with no counterpart in the
 * pages: while set, every pcp_attn_varlen call made by this thread records
 * prefill_begin / prefill_end (cudaEvent_t) on its stream right before and
 * after the prefill kernel, and decode_begin / decode_end around the decode
 * kernels, so a caller can time them with cudaEventElapsedTime. Pass NULLs to
 * stop. The events stay owned by the caller. Never fails (returns PCP_OK).
 */
int pcp_set_profile_events(void* prefill_begin, void* prefill_end, void* decode_begin,
                           void* decode_end);

/*
 * pcp_selftest_bounded_wait — device. A failure-detection self-test with no
 * counterpart in the pages: one warp waits on an mbarrier phase that nothing
 * completes, using the same bounded wait as the attention kernels, gives up
 * after timeout_us microseconds and sets *status = PCP_ERR_TIMEOUT. It checks
 * that a stuck pipeline ends with an error status and a usable context instead
 * of a hang. status: device int32 (zero it first). timeout_us in [1, 1e6].
 * Errors: PCP_ERR_ARG, PCP_ERR_CUDA.
 */
int pcp_selftest_bounded_wait(int32_t* status, uint32_t timeout_us, pcp_stream_t stream);

/* The cudaError_t value of the last failed CUDA call in this thread (0 if none). */
int pcp_last_cuda_error(void);

/* A short static description of a status code. */
const char* pcp_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* PCP_H_ */
