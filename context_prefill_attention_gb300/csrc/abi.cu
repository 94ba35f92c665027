// The C ABI of libpcp (declared in include/pcp.h): argument validation on the
// host, workspace layout and the launch sequence of one attention call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "ctx_table.h"
#include "pcp.h"
#include "pcp_internal.h"

namespace pcp {

namespace {
thread_local int g_last_cuda_error = 0;
// Events recorded around the prefill and decode launches when set (profiling hook).
thread_local cudaEvent_t g_profile[4] = {nullptr, nullptr, nullptr, nullptr};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A device buffer as a byte range.
struct Span {
    const void* p;
    size_t n;
};

// True when two byte ranges share a byte (an empty range shares none).
inline bool overlap(Span a, Span b) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a.p), y = reinterpret_cast<uintptr_t>(b.p);
    return a.n > 0 && b.n > 0 && x < y + b.n && y < x + a.n;
}

// True when an output range overlaps any of the ranges in ins[0, n) (kernels
// read their inputs while other CTAs already write their outputs).
inline bool overlaps_any(Span out, const Span* ins, int n) {
    for (int i = 0; i < n; ++i)
        if (overlap(out, ins[i])) return true;
    return false;
}
}  // namespace

void set_last_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int>(e); }

namespace {
using PFN_ctxGetCurrent = CUresult (*)(CUcontext*);
using PFN_ctxGetId = CUresult (*)(CUcontext, unsigned long long*);

// A driver API function by name, or nullptr.
void* driver_entry(const char* name) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return p;
}

// The internal stream of PCP_ATTN_DECODE_SMS with its fork and join events, one
// per CUDA context (streams and events belong to the context that made them).
// Kept for the life of the process and never freed, so a pointer handed out
// stays valid even if its table entry is later reused for another context.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t forked = nullptr, done = nullptr;
    std::mutex mu;  // one call's fork, launches and join at a time
};
CtxTable<32> g_side;
std::mutex g_side_create;

// The current context's side stream, created on first use; nullptr if it
// cannot be had (the call then runs its decode rows in sequence).
SideStream* side_stream() {
    uint64_t id = 0;
    if (!current_ctx_id(&id)) return nullptr;
    if (void* p = g_side.find(id)) return static_cast<SideStream*>(p);
    std::lock_guard<std::mutex> lock(g_side_create);
    if (void* p = g_side.find(id)) return static_cast<SideStream*>(p);
    SideStream* ss = new SideStream();
    if (cudaStreamCreateWithFlags(&ss->stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss->forked, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss->done, cudaEventDisableTiming) != cudaSuccess) {
        if (ss->done) cudaEventDestroy(ss->done);
        if (ss->forked) cudaEventDestroy(ss->forked);
        if (ss->stream) cudaStreamDestroy(ss->stream);
        delete ss;
        cudaGetLastError();
        return nullptr;
    }
    g_side.put(id, ss);
    return ss;
}
}  // namespace

bool current_ctx_id(uint64_t* id) {
    // resolved once (thread-safe static initialisation)
    static const PFN_ctxGetCurrent get_current =
        reinterpret_cast<PFN_ctxGetCurrent>(driver_entry("cuCtxGetCurrent"));
    static const PFN_ctxGetId get_id = reinterpret_cast<PFN_ctxGetId>(driver_entry("cuCtxGetId"));
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    unsigned long long v = 0;
    if (get_id(ctx, &v) != CUDA_SUCCESS) return false;
    *id = v;
    return true;
}

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

WorkspaceLayout workspace_layout(int32_t num_rows, int32_t total_q, int32_t num_q_heads,
                                 int32_t head_dim, int32_t max_kv_len, int32_t flags) {
    WorkspaceLayout w{};
    w.nparts = attn_partials(flags) > 0 ? attn_partials(flags) : 0;
    const int64_t passes = w.nparts > 0 ? w.nparts : 1;
    w.max_units = passes * ((int64_t)(total_q + kBlockM - 1) / kBlockM + num_rows);
    w.max_splits = max_kv_len > 0 ? (max_kv_len + kDecodeChunk - 1) / kDecodeChunk : 1;
    size_t o = 0;
    w.header = o;
    o = align256(o + 64 * sizeof(int32_t));
    w.row_ok = o;
    o = align256(o + (size_t)num_rows * sizeof(int32_t));
    w.dec_pre = o;
    o = align256(o + (2 * (size_t)num_rows + 1) * sizeof(int32_t));
    w.units = o;
    o = align256(o + (size_t)w.max_units * sizeof(Unit));
    w.units_sorted = o;
    o = align256(o + (size_t)w.max_units * sizeof(Unit));
    const size_t part = (size_t)total_q * num_q_heads * head_dim * sizeof(float);
    const size_t plse = (size_t)total_q * num_q_heads * sizeof(float);
    w.part_out = o;
    o = align256(o + (size_t)w.nparts * part);
    w.part_lse = o;
    o = align256(o + (size_t)w.nparts * plse);
    // two partials per decode split: the tensor-core decode writes one per softmax warpgroup
    const size_t dec = (size_t)num_rows * num_q_heads * 2 * w.max_splits;
    w.dec_out = o;
    o = align256(o + dec * head_dim * sizeof(float));
    w.dec_lse = o;
    o = align256(o + dec * sizeof(float));
    w.total = o;
    return w;
}

}  // namespace pcp

using namespace pcp;

extern "C" int pcp_last_cuda_error(void) { return g_last_cuda_error; }

extern "C" const char* pcp_status_string(int status) {
    switch (status) {
        case PCP_OK: return "ok";
        case PCP_ERR_ARG: return "invalid argument";
        case PCP_ERR_RANGE: return "index out of range";
        case PCP_ERR_UNSUPPORTED: return "unsupported configuration";
        case PCP_ERR_ALIGN: return "misaligned pointer";
        case PCP_ERR_CUDA: return "CUDA error";
        case PCP_ERR_TIMEOUT: return "device wait timed out";
        case PCP_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

extern "C" int pcp_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping,
                                  int32_t num_tokens, void* key_cache, void* value_cache,
                                  int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t* status, pcp_stream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || block_size < 1 || num_kv_heads < 1 || head_dim < 1)
        return PCP_ERR_ARG;
    if (num_tokens == 0) return PCP_OK;
    if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PCP_ERR_ARG;
    if (((int64_t)head_dim * 2 * num_kv_heads) % 16 != 0) return PCP_ERR_UNSUPPORTED;
    if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PCP_ERR_ALIGN;
    const size_t tok_bytes = (size_t)num_tokens * num_kv_heads * head_dim * 2;
    const size_t cache_bytes = (size_t)num_blocks * block_size * num_kv_heads * head_dim * 2;
    const Span ins[3] = {{k, tok_bytes}, {v, tok_bytes}, {slot_mapping, (size_t)num_tokens * 8}};
    if (overlaps_any({key_cache, cache_bytes}, ins, 3) || overlaps_any({value_cache, cache_bytes}, ins, 3) ||
        overlap({key_cache, cache_bytes}, {value_cache, cache_bytes}))
        return PCP_ERR_ARG;
    const int32_t vec_per_tok = (int32_t)((int64_t)head_dim * 2 * num_kv_heads / 16);
    return launch_cache_write(k, v, slot_mapping, num_tokens, vec_per_tok, key_cache, value_cache,
                              num_blocks * block_size, status, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" int pcp_kv_cache_write_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                                      int32_t num_tokens, void* key_cache, void* value_cache,
                                      int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                      int32_t head_dim, float k_scale, float v_scale, int32_t* status,
                                      pcp_stream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || block_size < 1 || num_kv_heads < 1 || head_dim < 1)
        return PCP_ERR_ARG;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !isfinite(k_scale) || !isfinite(v_scale)) return PCP_ERR_ARG;
    if (num_tokens == 0) return PCP_OK;
    if (!k || !v || !slot_mapping || !key_cache || !value_cache) return PCP_ERR_ARG;
    if (((int64_t)head_dim * num_kv_heads) % 16 != 0) return PCP_ERR_UNSUPPORTED;
    if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
        return PCP_ERR_ALIGN;
    const size_t tok_bytes = (size_t)num_tokens * num_kv_heads * head_dim * 2;
    const size_t cache_bytes = (size_t)num_blocks * block_size * num_kv_heads * head_dim;
    const Span ins[3] = {{k, tok_bytes}, {v, tok_bytes}, {slot_mapping, (size_t)num_tokens * 8}};
    if (overlaps_any({key_cache, cache_bytes}, ins, 3) || overlaps_any({value_cache, cache_bytes}, ins, 3) ||
        overlap({key_cache, cache_bytes}, {value_cache, cache_bytes}))
        return PCP_ERR_ARG;
    const int32_t vec_per_tok = (int32_t)((int64_t)head_dim * num_kv_heads / 16);
    return launch_cache_write_fp8(k, v, slot_mapping, num_tokens, vec_per_tok, key_cache, value_cache,
                                  num_blocks * block_size, k_scale, v_scale, status,
                                  reinterpret_cast<cudaStream_t>(stream));
}

extern "C" size_t pcp_attn_workspace_size(int32_t num_rows, int32_t total_q, int32_t num_q_heads,
                                          int32_t head_dim, int32_t max_kv_len, int32_t flags) {
    if (num_rows < 0 || total_q < 0 || num_q_heads < 1 || head_dim < 1 || max_kv_len < 0) return 0;
    if (attn_partials(flags) < 0) return 0;
    return workspace_layout(num_rows, total_q, num_q_heads, head_dim, max_kv_len, flags).total;
}

// One attention call over a bf16 cache (k_descale == v_descale == nullptr) or
// an FP8 one (both set). With a workspace provider, the workspace arguments are
// ignored and, once every argument check has passed, the provider supplies the
// workspace for the call's size.
int pcp::attn_call(const void* q, const void* key_cache, const void* value_cache, const float* k_descale,
              const float* v_descale, const int32_t* block_table, int32_t num_reqs,
              int32_t max_blocks_per_req, int64_t num_blocks, int32_t block_size, const pcp_row_t* rows,
              int32_t num_rows, int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
              int32_t head_dim, float scale, void* out, float* lse, void* workspace,
              size_t workspace_bytes, int32_t flags, int32_t* status, cudaStream_t s,
              WorkspaceProvider provide) {
    if (num_rows < 0 || total_q < 0 || num_reqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || max_blocks_per_req < 0 ||
        num_blocks < 0 || block_size < 1)
        return PCP_ERR_ARG;
    if (attn_partials(flags) < 0 || !isfinite(scale)) return PCP_ERR_ARG;
    if (num_q_heads % num_kv_heads != 0) return PCP_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PCP_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
        return PCP_ERR_UNSUPPORTED;
    if (num_q_heads / num_kv_heads > 16) return PCP_ERR_UNSUPPORTED;
    if (num_rows == 0 || total_q == 0) return PCP_OK;
    if (provide) {
        workspace = nullptr;
        workspace_bytes = 0;
    }
    if (!q || !key_cache || !value_cache || !block_table || !rows || !out || !lse || (!workspace && !provide))
        return PCP_ERR_ARG;
    if (!aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(rows) & 3u))
        return PCP_ERR_ALIGN;
    if (num_blocks * (int64_t)block_size > INT32_MAX || (int64_t)total_q * num_q_heads > INT32_MAX)
        return PCP_ERR_ARG;
    const int64_t max_kv = (int64_t)max_blocks_per_req * block_size;
    if (max_kv > INT32_MAX) return PCP_ERR_ARG;
    const WorkspaceLayout w =
        workspace_layout(num_rows, total_q, num_q_heads, head_dim, (int32_t)max_kv, flags);
    if (provide) {
        const int rc = provide(w.total, &workspace, &workspace_bytes);
        if (rc != PCP_OK) return rc;
        if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PCP_ERR_ALIGN;
    }
    if (workspace_bytes < w.total) return PCP_ERR_WORKSPACE;
    {
        const size_t esize = k_descale ? 1 : 2;
        const size_t out_bytes = (size_t)total_q * num_q_heads * head_dim * 2;
        const size_t lse_bytes = (size_t)total_q * num_q_heads * 4;
        const size_t cache_bytes = (size_t)num_blocks * block_size * num_kv_heads * head_dim * esize;
        const size_t descale_bytes = k_descale ? (size_t)num_reqs * num_kv_heads * 4 : 0;
        const Span ins[8] = {{q, out_bytes},
                             {key_cache, cache_bytes},
                             {value_cache, cache_bytes},
                             {block_table, (size_t)num_reqs * max_blocks_per_req * 4},
                             {rows, (size_t)num_rows * sizeof(pcp_row_t)},
                             {workspace, w.total},
                             {k_descale, descale_bytes},
                             {v_descale, descale_bytes}};
        if (overlaps_any({out, out_bytes}, ins, 8) || overlaps_any({lse, lse_bytes}, ins, 8) ||
            overlap({out, out_bytes}, {lse, lse_bytes}))
            return PCP_ERR_ARG;
    }

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    PrefillArgs a{};
    a.q = q;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.block_table = block_table;
    a.num_reqs = num_reqs;
    a.max_blocks = max_blocks_per_req;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.rows = rows;
    a.num_rows = num_rows;
    a.total_q = total_q;
    a.hq = num_q_heads;
    a.hkv = num_kv_heads;
    a.d = head_dim;
    a.scale = scale;
    a.out = out;
    a.lse = lse;
    a.part_out = reinterpret_cast<float*>(ws + w.part_out);
    a.part_lse = reinterpret_cast<float*>(ws + w.part_lse);
    a.nparts = w.nparts;
    a.row_ok = reinterpret_cast<const int32_t*>(ws + w.row_ok);
    a.units = reinterpret_cast<const Unit*>(ws + w.units_sorted);
    a.num_units = reinterpret_cast<const int32_t*>(ws + w.header);
    a.dec_pre = reinterpret_cast<const int32_t*>(ws + w.dec_pre);
    a.status = status;
    a.k_descale = k_descale;
    a.v_descale = v_descale;

    int rc = launch_schedule(a, flags, reinterpret_cast<Unit*>(ws + w.units),
                             reinterpret_cast<Unit*>(ws + w.units_sorted),
                             reinterpret_cast<int32_t*>(ws + w.header),
                             reinterpret_cast<int32_t*>(ws + w.row_ok),
                             reinterpret_cast<int32_t*>(ws + w.dec_pre), w.max_units, s);
    if (rc != PCP_OK) return rc;
    float* dec_out = reinterpret_cast<float*>(ws + w.dec_out);
    float* dec_lse = reinterpret_cast<float*>(ws + w.dec_lse);
    const int nsm = num_sms();
    const int kdec = attn_decode_sms(flags);
    SideStream* side = (kdec > 0 && kdec < nsm && decode_side_applies(a)) ? side_stream() : nullptr;
    if (side) {
        // decode rows on kdec SMs of the side stream, prefill rows on the others
        std::lock_guard<std::mutex> lock(side->mu);
        cudaError_t e = cudaEventRecord(side->forked, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side->stream, side->forked, 0);
        if (e != cudaSuccess) {
            set_last_cuda_error(e);
            return PCP_ERR_CUDA;
        }
        if (g_profile[2]) cudaEventRecord(g_profile[2], side->stream);
        rc = launch_decode(a, dec_out, dec_lse, w.max_splits, side->stream, kdec);
        if (rc == PCP_OK) {
            if (g_profile[3]) cudaEventRecord(g_profile[3], side->stream);
            if (g_profile[0]) cudaEventRecord(g_profile[0], s);
            rc = launch_prefill(a, s, nsm - kdec);
            if (rc == PCP_OK && g_profile[1]) cudaEventRecord(g_profile[1], s);
        }
        // joined even after a failed launch: nothing of this call runs on after the
        // caller's stream has moved past it
        e = cudaEventRecord(side->done, side->stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, side->done, 0);
        if (rc != PCP_OK) return rc;
        if (e != cudaSuccess) {
            set_last_cuda_error(e);
            return PCP_ERR_CUDA;
        }
    } else {
        if (g_profile[2]) cudaEventRecord(g_profile[2], s);
        rc = launch_decode(a, dec_out, dec_lse, w.max_splits, s);
        if (rc != PCP_OK) return rc;
        if (g_profile[3]) cudaEventRecord(g_profile[3], s);
        if (g_profile[0]) cudaEventRecord(g_profile[0], s);
        rc = launch_prefill(a, s);
        if (rc != PCP_OK) return rc;
        if (g_profile[1]) cudaEventRecord(g_profile[1], s);
    }
    if (a.nparts > 0) rc = launch_separate_merge(a, s);
    return rc;
}

extern "C" int pcp_attn_varlen(const void* q, const void* key_cache, const void* value_cache,
                               const int32_t* block_table, int32_t num_reqs,
                               int32_t max_blocks_per_req, int64_t num_blocks, int32_t block_size,
                               const pcp_row_t* rows, int32_t num_rows, int32_t total_q,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, float scale,
                               void* out, float* lse, void* workspace, size_t workspace_bytes,
                               int32_t flags, int32_t* status, pcp_stream_t stream) {
    return attn_call(q, key_cache, value_cache, nullptr, nullptr, block_table, num_reqs, max_blocks_per_req,
                     num_blocks, block_size, rows, num_rows, total_q, num_q_heads, num_kv_heads, head_dim,
                     scale, out, lse, workspace, workspace_bytes, flags, status,
                     reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int pcp_attn_varlen_fp8kv(const void* q, const void* key_cache, const void* value_cache,
                                     const float* k_descale, const float* v_descale,
                                     const int32_t* block_table, int32_t num_reqs, int32_t max_blocks_per_req,
                                     int64_t num_blocks, int32_t block_size, const pcp_row_t* rows,
                                     int32_t num_rows, int32_t total_q, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_dim, float scale, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes, int32_t flags,
                                     int32_t* status, pcp_stream_t stream) {
    if (num_rows > 0 && total_q > 0 && (!k_descale || !v_descale)) return PCP_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_descale) & 3u) || (reinterpret_cast<uintptr_t>(v_descale) & 3u))
        return PCP_ERR_ALIGN;
    return attn_call(q, key_cache, value_cache, k_descale, v_descale, block_table, num_reqs, max_blocks_per_req, num_blocks, block_size, rows, num_rows, total_q,
                     num_q_heads, num_kv_heads, head_dim, scale, out, lse, workspace, workspace_bytes, flags,
                     status, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" int pcp_set_profile_events(void* prefill_begin, void* prefill_end, void* decode_begin,
                                      void* decode_end) {
    g_profile[0] = static_cast<cudaEvent_t>(prefill_begin);
    g_profile[1] = static_cast<cudaEvent_t>(prefill_end);
    g_profile[2] = static_cast<cudaEvent_t>(decode_begin);
    g_profile[3] = static_cast<cudaEvent_t>(decode_end);
    return PCP_OK;
}

extern "C" int pcp_lse_merge(const float* out_a, const float* lse_a, const float* out_b,
                             const float* lse_b, void* out, float* lse, int32_t total_q,
                             int32_t num_q_heads, int32_t head_dim, pcp_stream_t stream) {
    if (total_q < 0 || num_q_heads < 1 || head_dim < 1) return PCP_ERR_ARG;
    if (head_dim % 8 != 0) return PCP_ERR_UNSUPPORTED;
    if (total_q == 0) return PCP_OK;
    if (!out_a || !lse_a || !out_b || !lse_b || !out || !lse) return PCP_ERR_ARG;
    if (!aligned16(out_a) || !aligned16(out_b) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse_a) & 3u) || (reinterpret_cast<uintptr_t>(lse_b) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return PCP_ERR_ALIGN;
    const size_t part_bytes = (size_t)total_q * num_q_heads * head_dim * 4;
    const size_t lse_bytes = (size_t)total_q * num_q_heads * 4;
    const Span ins[4] = {{out_a, part_bytes}, {out_b, part_bytes}, {lse_a, lse_bytes}, {lse_b, lse_bytes}};
    const Span o = {out, part_bytes / 2};
    if (overlaps_any(o, ins, 4) || overlaps_any({lse, lse_bytes}, ins, 4) || overlap(o, {lse, lse_bytes}))
        return PCP_ERR_ARG;
    return launch_lse_merge(out_a, lse_a, out_b, lse_b, out, lse, total_q, num_q_heads, head_dim,
                            reinterpret_cast<cudaStream_t>(stream));
}
