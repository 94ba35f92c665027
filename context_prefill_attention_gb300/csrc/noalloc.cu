// pcp_attn_varlen_noalloc: the attention call for callers that cannot allocate
// device memory at all — a host framework that owns every byte of device
// memory through its own allocator and forbids cudaMalloc, or a latency-bound
// serving loop where cudaMalloc/cudaFree is not allowed after start-up
// because it can synchronise the device and take an unbounded time. Such a
// caller cannot provide the workspace pcp_attn_varlen asks for.
//
// This entry point instead uses one fixed scratch array that lives in the
// library's own device image: kStaticScratchBytes per GPU, reserved on every
// GPU that loads this library until the process exits. It then runs exactly
// the same launch sequence as pcp_attn_varlen (schedule, split-KV decode,
// prefill, optional LSE merge) with that array as the workspace. The scratch
// needs no clearing: every byte the kernels read is written earlier in the
// same call. All calls on a device share the one array, so two calls whose
// kernels overlap on the GPU (different streams without ordering between them,
// or different host threads) race on it; order them on one stream.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "pcp.h"
#include "pcp_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;  // 64 MiB

__device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

// Device address of g_scratch for each device (the host-side symbol is only a
// stand-in and must never be passed to a kernel).
void* g_scratch_addr[128] = {};
std::mutex g_scratch_mu;

int scratch_for_current_device(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        pcp::set_last_cuda_error(e);
        return PCP_ERR_CUDA;
    }
    if (dev < 0 || dev >= 128) return PCP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || p == nullptr) {
            pcp::set_last_cuda_error(e);
            return PCP_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
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
    if (max_blocks_per_req < 0 || block_size < 1) return PCP_ERR_ARG;
    const int64_t max_kv = (int64_t)max_blocks_per_req * block_size;
    if (max_kv > INT32_MAX) return PCP_ERR_ARG;
    const size_t need = pcp_attn_workspace_size(num_rows, total_q, num_q_heads, head_dim, (int32_t)max_kv, flags);
    if (need == 0) return PCP_ERR_ARG;
    if (need > kStaticScratchBytes) return PCP_ERR_WORKSPACE;
    void* scratch = nullptr;
    const int rc = scratch_for_current_device(&scratch);
    if (rc != PCP_OK) return rc;
    return pcp_attn_varlen(q, key_cache, value_cache, block_table, num_reqs, max_blocks_per_req, num_blocks,
                           block_size, rows, num_rows, total_q, num_q_heads, num_kv_heads, head_dim, scale, out,
                           lse, scratch, kStaticScratchBytes, flags, status, stream);
}
