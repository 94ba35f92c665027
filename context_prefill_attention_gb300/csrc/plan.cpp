// Host side of the PCP step: the row plan and the PAD-masked slot mapping.
//
// Row plan: "[MRv2][PCP] Carry the row plan in attention metadata; fix mixed
// prefill+decode crash", sections 1-2 (rows per prefilling request, per-row
// context lengths) and "What made it removable" (DualChunkSwap head/tail rows;
// a row's seq_len is its end position). Contiguous per-rank slices:
// "Feat/pcp qwen36 hybrid", "Changes". Slot mapping and PAD masking: commit
// "drop pcp_has_prefill" on the row-plan page.
#include <cmath>
#include <cstdint>
#include <vector>

#include "pcp.h"

namespace {

struct Span {
    int64_t lo, hi;  // [lo, hi) among the request's new tokens
};

// The spans a shard owns of a request with n new tokens, in emission order.
inline int shard_spans(int64_t n, int32_t shard, int32_t shards, int32_t mode, Span out[2]) {
    if (n <= 0) return 0;
    if (n == 1) {  // one new token: a single row, on shard 0 only
        if (shard != 0) return 0;
        out[0] = {0, 1};
        return 1;
    }
    int k = 0;
    if (mode == PCP_SPLIT_CONTIGUOUS) {
        Span s{n * shard / shards, n * (shard + 1) / shards};
        if (s.hi > s.lo) out[k++] = s;
    } else {
        const int64_t parts = 2 * (int64_t)shards;
        const int64_t idx[2] = {shard, parts - 1 - shard};
        for (int c = 0; c < 2; ++c) {
            Span s{n * idx[c] / parts, n * (idx[c] + 1) / parts};
            if (s.hi > s.lo) out[k++] = s;
        }
    }
    return k;
}

}  // namespace

extern "C" int pcp_build_row_plan(int32_t num_reqs, const int32_t* query_len,
                                  const int32_t* num_computed, const int32_t* block_table,
                                  int32_t max_blocks_per_req, int32_t block_size,
                                  int32_t num_shards, int32_t split_mode, pcp_row_t* rows,
                                  int32_t rows_capacity, int32_t* num_rows, int32_t* cu_q,
                                  int64_t* slot_mapping, int8_t* owner_shard) {
    if (num_reqs < 0 || num_shards < 1 || num_shards > 127 || block_size < 1 ||
        max_blocks_per_req < 0 || rows_capacity < 0)
        return PCP_ERR_ARG;
    if (split_mode != PCP_SPLIT_CONTIGUOUS && split_mode != PCP_SPLIT_DUAL_CHUNK) return PCP_ERR_ARG;
    if (!num_rows || !cu_q) return PCP_ERR_ARG;
    if (num_reqs > 0 && (!query_len || !num_computed)) return PCP_ERR_ARG;

    std::vector<int64_t> first(num_reqs + 1, 0);  // packed offset of each request
    for (int32_t r = 0; r < num_reqs; ++r) {
        if (query_len[r] < 0 || num_computed[r] < 0) return PCP_ERR_ARG;
        first[r + 1] = first[r] + query_len[r];
    }
    const int64_t total = first[num_reqs];
    if (total > INT32_MAX) return PCP_ERR_ARG;
    if (total > 0 && (!slot_mapping || !block_table || !rows)) return PCP_ERR_ARG;

    // Slot mapping: every new token of every request, independent of sharding.
    for (int32_t r = 0; r < num_reqs; ++r) {
        const int32_t* table = block_table + (size_t)r * max_blocks_per_req;
        const int64_t base = num_computed[r];
        for (int64_t j = 0; j < query_len[r]; ++j) {
            const int64_t pos = base + j;
            const int64_t page = pos / block_size;
            if (page >= max_blocks_per_req) return PCP_ERR_RANGE;
            const int64_t id = table[page];
            if (id < 0) return PCP_ERR_RANGE;
            slot_mapping[first[r] + j] = id * block_size + (pos - page * block_size);
        }
    }

    int32_t n = 0;
    int64_t running = 0;
    cu_q[0] = 0;
    for (int32_t s = 0; s < num_shards; ++s) {
        for (int32_t r = 0; r < num_reqs; ++r) {
            Span spans[2];
            const int k = shard_spans(query_len[r], s, num_shards, split_mode, spans);
            for (int c = 0; c < k; ++c) {
                if (n >= rows_capacity) return PCP_ERR_RANGE;
                const int64_t qlen = spans[c].hi - spans[c].lo;
                const int64_t end = (int64_t)num_computed[r] + spans[c].hi;
                if (end > INT32_MAX) return PCP_ERR_ARG;
                pcp_row_t& row = rows[n];
                row.req = r;
                row.shard = s;
                row.q_start = (int32_t)(first[r] + spans[c].lo);
                row.q_len = (int32_t)qlen;
                row.ctx_len = num_computed[r];
                row.kv_end = (int32_t)end;
                row.causal_off = (int32_t)spans[c].lo;
                row.is_decode = (query_len[r] == 1 && num_computed[r] > 0) ? 1 : 0;
                running += qlen;
                cu_q[++n] = (int32_t)running;
                if (owner_shard)
                    for (int64_t t = row.q_start; t < row.q_start + qlen; ++t) owner_shard[t] = (int8_t)s;
            }
        }
    }
    *num_rows = n;
    return PCP_OK;
}

extern "C" int pcp_mask_slots_for_shard(const int64_t* slot_mapping, const int8_t* owner_shard,
                                        int32_t num_tokens, int32_t shard, int64_t* out) {
    if (num_tokens < 0) return PCP_ERR_ARG;
    if (num_tokens > 0 && (!slot_mapping || !owner_shard || !out)) return PCP_ERR_ARG;
    for (int32_t t = 0; t < num_tokens; ++t) out[t] = owner_shard[t] == shard ? slot_mapping[t] : -1;
    return PCP_OK;
}

// SMs for the decode rows beside the prefill rows (PCP_ATTN_DECODE_SMS), from
// the host row plan. Each side's SM time, at rates measured with this library's
// kernels on GB300 (the ratio is what matters, so the clock cancels):
//  * decode rows: their K and V bytes at what one SM of the tensor-core decode
//    streams once HBM is not shared by every SM, plus a cost per work item
//    (2048-key split x kv head);
//  * prefill rows: per work item (128-token tile x head pair, or x head for an
//    odd group) plus per 128-key tile it visits (end-aligned causal).
// The SMs are split in proportion, rounding towards the decode side: a decode
// that ends last costs the whole difference, a prefill that ends last only its
// share of one SM.
extern "C" int32_t pcp_decode_sms(const pcp_row_t* rows, int32_t num_rows, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t kv_cache_fp8, int32_t num_sms) {
    if (!rows || num_rows <= 0 || num_rows > 1024 || num_sms < 2 || num_q_heads < 1 || num_kv_heads < 1 ||
        num_q_heads % num_kv_heads != 0)
        return 0;
    const int32_t G = num_q_heads / num_kv_heads;
    if (head_dim != 128 || G > 16 || kv_cache_fp8) return 0;
    constexpr double kDecodeBytesPerSmS = 78.6e9;  // K/V bytes per second and SM
    constexpr double kDecodeItemS = 1.0e-6;        // per split and kv head
    constexpr double kPrefillItemS = 3.65e-6;      // per work item
    constexpr double kPrefillTileS = 1.68e-6;      // per 128-key tile of a two-head item
    constexpr double kPrefillTileOneHeadS = 1.0e-6;
    constexpr int32_t kSplit = 2048, kTile = 128;
    const bool dual = G % 2 == 0;
    const double items_per_tile = dual ? num_q_heads / 2 : num_q_heads;
    const double tile_s = dual ? kPrefillTileS : kPrefillTileOneHeadS;
    double dec = 0.0, pre = 0.0;
    for (int32_t i = 0; i < num_rows; ++i) {
        const pcp_row_t& r = rows[i];
        if (r.q_len < 1 || r.kv_end < r.q_len) continue;
        if (r.is_decode) {
            const double bytes = (double)r.kv_end * num_kv_heads * head_dim * 2.0 * 2.0;
            const double items = (double)((r.kv_end + kSplit - 1) / kSplit) * num_kv_heads;
            dec += bytes / kDecodeBytesPerSmS + items * kDecodeItemS;
            continue;
        }
        for (int32_t t = 0; t * kTile < r.q_len; ++t) {
            const int64_t last = (int64_t)r.kv_end - r.q_len + (r.q_len < (t + 1) * kTile ? r.q_len : (t + 1) * kTile);
            const double key_tiles = (double)((last + kTile - 1) / kTile);
            pre += items_per_tile * (kPrefillItemS + key_tiles * tile_s);
        }
    }
    if (dec <= 0.0 || pre <= 0.0) return 0;
    const double d = 1.05 * dec;
    int32_t k = (int32_t)std::ceil(num_sms * d / (d + pre));
    if (k < 1) k = 1;
    if (2 * k >= num_sms) return 0;  // decode-heavy: HBM, not the SM count, bounds it
    return k;
}
