// pcp_attn_varlen_noalloc: the attention call for callers that cannot allocate
// device memory at all — a host framework that owns every byte of device
// memory through its own allocator and forbids cudaMalloc, or a latency-bound
// serving loop where cudaMalloc/cudaFree is not allowed after start-up
// because it can synchronise the device and take an unbounded time. Such a
// caller cannot provide the workspace pcp_attn_varlen asks for.
//
// This entry point instead uses one fixed scratch array that lives in the
// library's own device image: kStaticScratchBytes per GPU, reserved on every
// GPU that loads this library until the process exits. It runs the same host
// checks (in the same order) and the same launch sequence as pcp_attn_varlen
// (schedule, split-KV decode, prefill, optional LSE merge) with that array as
// the workspace. The scratch needs no clearing: every byte the kernels read is
// written earlier in the same call. All calls on a device share the one array,
// so two calls whose kernels overlap on the GPU (different streams without
// ordering between them, or different host threads) race on it; order them on
// one stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ctx_table.h"
#include "pcp.h"
#include "pcp_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

__device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

// Device address of g_scratch per CUDA context (the host-side symbol is only a
// stand-in and must never be passed to a kernel). Keyed by the context's ID, so
// a context created after a device reset looks the address up again.
pcp::CtxTable<32> g_scratch_addr;

// The workspace provider of pcp_attn_varlen_noalloc: the scratch array of the
// current device, if the call fits in it.
int scratch_workspace(size_t need, void** ws, size_t* bytes) {
    if (need > kStaticScratchBytes) return PCP_ERR_WORKSPACE;
    uint64_t id = 0;
    bool have_id = pcp::current_ctx_id(&id);
    void* p = have_id ? g_scratch_addr.find(id) : nullptr;
    if (!p) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || p == nullptr) {
            pcp::set_last_cuda_error(e);
            return PCP_ERR_CUDA;
        }
        if (!have_id) have_id = pcp::current_ctx_id(&id);  // the lookup made the context current
        if (have_id) g_scratch_addr.put(id, p);
    }
    *ws = p;
    *bytes = kStaticScratchBytes;
    return PCP_OK;
}

}  // namespace

extern "C" int pcp_attn_varlen_noalloc(const void* q, const void* key_cache, const void* value_cache,
                                       const int32_t* block_table, int32_t num_reqs,
                                       int32_t max_blocks_per_req, int64_t num_blocks,
                                       int32_t block_size, const pcp_row_t* rows, int32_t num_rows,
                                       int32_t total_q, int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, float scale, void* out, float* lse,
                                       int32_t flags, int32_t* status, pcp_stream_t stream) {
    return pcp::attn_call(q, key_cache, value_cache, nullptr, nullptr, block_table, num_reqs, max_blocks_per_req,
                          num_blocks, block_size, rows, num_rows, total_q, num_q_heads, num_kv_heads, head_dim,
                          scale, out, lse, nullptr, 0, flags, status, reinterpret_cast<cudaStream_t>(stream),
                          scratch_workspace);
}
