// Internal declarations shared by libpcp's translation units (not installed).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pcp.h"

namespace pcp {

// Query tokens per tile and keys per tile of the prefill kernel.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// Keys per split of the decode kernel.
#ifndef PCP_DECODE_CHUNK
#define PCP_DECODE_CHUNK 2048  // measured: 2048 >= 1024 > 512 > 256 keys per split on the mixed workload
#endif
constexpr int kDecodeChunk = PCP_DECODE_CHUNK;

// A unit of prefill work: one 128-token tile of one row, one pass
// (0 = the whole key range, 1 = first partial, 2 = second partial), and the
// key range [k_lo, k_hi) it attends. Items are units x head slots.
struct Unit {
    int32_t row;
    int32_t mt_pass;  // mt | pass << 24
    int32_t k_lo;
    int32_t k_hi;
};

// Workspace layout of pcp_attn_varlen (all offsets 256-byte aligned).
struct WorkspaceLayout {
    size_t header;        // int32[64]: [0] = number of units
    size_t row_ok;        // int32[num_rows]: 1 for a row that passed the checks
    size_t dec_pre;       // int32[2 num_rows + 1]: full-split decode items of the rows before each
                          // row ([num_rows]: all of them), then the rows with a partial last
                          // split, longest partial first
    size_t units;         // Unit[max_units], unsorted
    size_t units_sorted;  // Unit[max_units], longest first
    size_t part_out;      // nparts x fp32 [T][Hq][D] (separate-context / KV-shard modes)
    size_t part_lse;      // nparts x fp32 [Hq][T]
    int32_t nparts;
    size_t dec_out;       // fp32 [num_rows][Hq][2 x max_splits][D]: decode partials
    size_t dec_lse;       // fp32 [num_rows][Hq][2 x max_splits]
    size_t total;
    int64_t max_units;
    int32_t max_splits;
};

// Number of partial passes a flags word asks for (0: fused), or -1 if invalid.
inline int32_t attn_partials(int32_t flags) {
    const int32_t shards = (flags >> 8) & 0xFF;
    const bool separate = (flags & PCP_ATTN_SEPARATE_CONTEXT) != 0;
    if (flags & ~(PCP_ATTN_SEPARATE_CONTEXT | PCP_ATTN_SPLIT_AT_ROW_START | 0xFF00 | 0xFF0000)) return -1;
    if (shards == 1 || shards > 64 || (shards && separate)) return -1;
    return separate ? 2 : shards;
}

WorkspaceLayout workspace_layout(int32_t num_rows, int32_t total_q, int32_t num_q_heads,
                                 int32_t head_dim, int32_t max_kv_len, int32_t flags);

// SMs for the decode rows beside the prefill (PCP_ATTN_DECODE_SMS), 0: in sequence.
inline int32_t attn_decode_sms(int32_t flags) { return (flags >> 16) & 0xFF; }

void set_last_cuda_error(cudaError_t e);
// ID of the current CUDA context (process-unique, never reused); false when no
// context is current or the driver lacks the query.
bool current_ctx_id(uint64_t* id);
int num_sms();

struct PrefillArgs {
    const void* q;
    const void* key_cache;
    const void* value_cache;
    const int32_t* block_table;
    int32_t num_reqs;
    int32_t max_blocks;
    int64_t num_blocks;
    int32_t block_size;
    const pcp_row_t* rows;
    int32_t num_rows;
    int32_t total_q;
    int32_t hq, hkv, d;
    float scale;
    void* out;
    float* lse;
    float* part_out;   // partial p (1-based pass p) at part_out + (p - 1) * total_q * hq * d
    float* part_lse;   // ... at part_lse + (p - 1) * hq * total_q
    int32_t nparts;    // 0: one fused pass straight into out / lse
    const int32_t* row_ok;
    const Unit* units;
    const int32_t* num_units;   // header: [0] prefill units, [1] decode work items
    // decode work items (kv head x kDecodeChunk-key split of a decode row): full-split
    // items of the rows before row i, for i = 0..num_rows (the last entry: all full
    // splits), then from [num_rows + 1] the rows with a partial last split, longest first
    const int32_t* dec_pre;
    int32_t* status;
    // FP8 (e4m3) cache: per-(request, kv head) descales [num_reqs][hkv]; both
    // null for a bf16 cache
    const float* k_descale;
    const float* v_descale;
};

// TMA map of a cache viewed as [outer][mid][D] elements of esize bytes (1: FP8
// codes, 2: bf16) with a box of D x 1 x rows, no swizzle.
bool make_kv_row_map(CUtensorMap* m, const void* base, int D, int esize, int64_t mid, int64_t outer, int rows);
// TMA map of [outer][mid][D] elements of esize bytes (1: uint8, 2: bf16) with a
// box of box_x x box_mid x box_outer elements, 128-byte swizzled or not.
bool make_box_map(CUtensorMap* m, const void* base, int D, int esize, int64_t mid, int64_t outer, int box_x,
                  int box_mid, int box_outer, bool swizzle128);

// Supplies the workspace of an attention call that has passed every argument
// check: at least `need` bytes, 256-byte aligned. Returns PCP_OK after setting
// *ws and *bytes, or the status the call returns.
using WorkspaceProvider = int (*)(size_t need, void** ws, size_t* bytes);

// The body of pcp_attn_varlen (k_descale = v_descale = nullptr) and
// pcp_attn_varlen_fp8kv: host checks, then the launches on stream s. With a
// provider the workspace arguments are ignored and the provider's workspace is
// used (pcp_attn_varlen_noalloc).
int attn_call(const void* q, const void* key_cache, const void* value_cache, const float* k_descale,
              const float* v_descale, const int32_t* block_table, int32_t num_reqs,
              int32_t max_blocks_per_req, int64_t num_blocks, int32_t block_size, const pcp_row_t* rows,
              int32_t num_rows, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
              int32_t head_dim, float scale, void* out, float* lse, void* workspace,
              size_t workspace_bytes, int32_t flags, int32_t* status, cudaStream_t s,
              WorkspaceProvider provide);

int launch_schedule(const PrefillArgs& a, int32_t flags, Unit* units, Unit* units_sorted,
                    int32_t* header, int32_t* row_ok, int32_t* dec_pre, int64_t max_units,
                    cudaStream_t stream);
// grid: CTAs of the persistent kernel (0: one per SM).
int launch_prefill(const PrefillArgs& a, cudaStream_t stream, int grid = 0);
// grid: CTAs of the tensor-core decode kernel (0: one per SM); the CUDA-core
// decode sizes its own grid.
int launch_decode(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                  cudaStream_t stream, int grid = 0);
// The tensor-core decode (head_dim 128, up to 16 q heads per kv head with a
// bf16 cache and 8 with an FP8 one, at most kDecTcMaxRows rows);
// PCP_ERR_UNSUPPORTED for any other shape. Over an FP8 cache and with more
// than 8 q heads per kv head it writes two partials per split (slots 2 split
// and 2 split + 1 of the row's 2 x max_splits), else one (slot split).
constexpr int kDecTcMaxRows = 1024;
bool decode_tc_applies(const PrefillArgs& a);
int launch_decode_tc(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                     cudaStream_t stream, int grid = 0);
// True when launch_decode takes the tensor-core kernel for these arguments (the
// persistent kernel that PCP_ATTN_DECODE_SMS confines to a few SMs).
bool decode_side_applies(const PrefillArgs& a);
int launch_separate_merge(const PrefillArgs& a, cudaStream_t stream);
int launch_cache_write(const void* k, const void* v, const int64_t* slot, int32_t num_tokens,
                       int32_t vec_per_tok, void* key_cache, void* value_cache, int64_t num_slots,
                       int32_t* status, cudaStream_t stream);
// FP8 cache write: vec_per_tok = 16-element groups per token row.
int launch_cache_write_fp8(const void* k, const void* v, const int64_t* slot, int32_t num_tokens,
                           int32_t vec_per_tok, void* key_cache, void* value_cache, int64_t num_slots,
                           float k_scale, float v_scale, int32_t* status, cudaStream_t stream);
int launch_lse_merge(const float* out_a, const float* lse_a, const float* out_b, const float* lse_b,
                     void* out, float* lse, int32_t total_q, int32_t hq, int32_t d,
                     cudaStream_t stream);

}  // namespace pcp
