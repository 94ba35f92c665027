// Two HBM-bound kernels of the PCP step.
//
// cache_write_kernel: scatter the new tokens' K/V rows into the paged cache at
// their slots, skipping negative (PAD) slots ("[MRv2][PCP] Carry the row plan
// ...", commit "drop pcp_has_prefill"). A token's K (or V) for all kv heads is
// one contiguous Hkv * D * 2-byte row in both the packed input and the cache
// slot, so every thread moves one 16-byte vector and a warp moves 512
// contiguous bytes: fully coalesced reads and writes.
//
// cache_write_fp8_kernel: the same scatter into an FP8 (e4m3) cache, each
// value stored as e4m3(x / scale) with the division correctly rounded in fp32,
// round to nearest even and saturation at +-448 (the layer's k / v scale of
// "[MRv2] FlashAttention PCP support ...", context-pass call). A thread turns
// 16 bf16 values (two 16-byte loads) into one 16-byte store.
//
// lse_merge_kernel: out = (w_a out_a + w_b out_b) / (w_a + w_b) with
// w_x = exp(lse_x - max(lse_a, lse_b)) ("[MRv2] FlashAttention PCP support
// ...": (ctx_out, ctx_lse) combined with the new-token pass). One thread per
// 4 head-dims of one (token, head): two float4 loads, one 8-byte bf16 store.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

__global__ void __launch_bounds__(256)
    cache_write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                       const int64_t* __restrict__ slot, int64_t total_vec, int32_t vec_per_tok,
                       uint4* __restrict__ kc, uint4* __restrict__ vc, int64_t num_slots,
                       int32_t* status) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_vec;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / vec_per_tok;
        const int32_t e = (int32_t)(i - t * vec_per_tok);
        const int64_t s = __ldg(slot + t);
        if (s < 0) continue;
        if (s >= num_slots) {
            if (e == 0) report_status(status, PCP_ERR_RANGE);
            continue;
        }
        const uint4 kv = __ldcs(k + i);
        const uint4 vv = __ldcs(v + i);
        kc[s * vec_per_tok + e] = kv;
        vc[s * vec_per_tok + e] = vv;
    }
}

__device__ __forceinline__ uint32_t quant4(uint32_t a, uint32_t b, float scale) {
    // a, b: two bf16 pairs (elements 0-1, 2-3) -> four codes, element i in byte i
    const uint32_t c01 = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(a << 16), scale),
                                         __fdiv_rn(__uint_as_float(a & 0xFFFF0000u), scale));
    const uint32_t c23 = f32x2_to_e4m3x2(__fdiv_rn(__uint_as_float(b << 16), scale),
                                         __fdiv_rn(__uint_as_float(b & 0xFFFF0000u), scale));
    return c01 | (c23 << 16);
}

__device__ __forceinline__ uint4 quant16(uint4 x, uint4 y, float scale) {
    return make_uint4(quant4(x.x, x.y, scale), quant4(x.z, x.w, scale), quant4(y.x, y.y, scale),
                      quant4(y.z, y.w, scale));
}

__global__ void __launch_bounds__(256)
    cache_write_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                           const int64_t* __restrict__ slot, int64_t total_vec, int32_t vec_per_tok,
                           uint4* __restrict__ kc, uint4* __restrict__ vc, int64_t num_slots, float k_scale,
                           float v_scale, int32_t* status) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_vec;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / vec_per_tok;
        const int32_t e = (int32_t)(i - t * vec_per_tok);
        const int64_t s = __ldg(slot + t);
        if (s < 0) continue;
        if (s >= num_slots) {
            if (e == 0) report_status(status, PCP_ERR_RANGE);
            continue;
        }
        const uint4 k0 = __ldcs(k + 2 * i), k1 = __ldcs(k + 2 * i + 1);
        const uint4 v0 = __ldcs(v + 2 * i), v1 = __ldcs(v + 2 * i + 1);
        kc[s * vec_per_tok + e] = quant16(k0, k1, k_scale);
        vc[s * vec_per_tok + e] = quant16(v0, v1, v_scale);
    }
}

__global__ void __launch_bounds__(256)
    lse_merge_kernel(const float* __restrict__ out_a, const float* __restrict__ lse_a,
                     const float* __restrict__ out_b, const float* __restrict__ lse_b,
                     __nv_bfloat16* __restrict__ out, float* lse, int32_t total_q, int32_t hq,
                     int32_t d) {
    const int chunks = d / 4;
    const int64_t n = (int64_t)total_q * hq * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % chunks);
        const int64_t th = i / chunks;
        const int h = (int)(th % hq);
        const int64_t t = th / hq;
        const float la = lse_a[(size_t)h * total_q + t];
        const float lb = lse_b[(size_t)h * total_q + t];
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        float l = -INFINITY;
        if (!(la == -INFINITY && lb == -INFINITY)) {
            const float M = fmaxf(la, lb);
            const float wa = __expf(la - M), wb = __expf(lb - M);
            const float inv = 1.f / (wa + wb);
            const float4 xa = *reinterpret_cast<const float4*>(out_a + th * d + 4 * c);
            const float4 xb = *reinterpret_cast<const float4*>(out_b + th * d + 4 * c);
            r = make_float4((wa * xa.x + wb * xb.x) * inv, (wa * xa.y + wb * xb.y) * inv,
                            (wa * xa.z + wb * xb.z) * inv, (wa * xa.w + wb * xb.w) * inv);
            l = M + __logf(wa + wb);
        }
        uint2 w;
        w.x = pack_bf16x2(r.x, r.y);
        w.y = pack_bf16x2(r.z, r.w);
        *reinterpret_cast<uint2*>(out + th * d + 4 * c) = w;
        if (c == 0) lse[(size_t)h * total_q + t] = l;
    }
}

}  // namespace pcp

namespace pcp {

int launch_cache_write(const void* k, const void* v, const int64_t* slot, int32_t num_tokens,
                       int32_t vec_per_tok, void* key_cache, void* value_cache, int64_t num_slots,
                       int32_t* status, cudaStream_t stream) {
    const int64_t total_vec = (int64_t)num_tokens * vec_per_tok;
    int64_t blocks = (total_vec + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    cache_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), slot, total_vec,
        vec_per_tok, reinterpret_cast<uint4*>(key_cache), reinterpret_cast<uint4*>(value_cache),
        num_slots, status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

int launch_cache_write_fp8(const void* k, const void* v, const int64_t* slot, int32_t num_tokens,
                           int32_t vec_per_tok, void* key_cache, void* value_cache, int64_t num_slots,
                           float k_scale, float v_scale, int32_t* status, cudaStream_t stream) {
    const int64_t total_vec = (int64_t)num_tokens * vec_per_tok;
    int64_t blocks = (total_vec + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    cache_write_fp8_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), slot, total_vec,
        vec_per_tok, reinterpret_cast<uint4*>(key_cache), reinterpret_cast<uint4*>(value_cache),
        num_slots, k_scale, v_scale, status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

int launch_lse_merge(const float* out_a, const float* lse_a, const float* out_b, const float* lse_b,
                     void* out, float* lse, int32_t total_q, int32_t hq, int32_t d,
                     cudaStream_t stream) {
    const int64_t n = (int64_t)total_q * hq * (d / 4);
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 16;
    if (blocks > cap) blocks = cap;
    lse_merge_kernel<<<(unsigned)blocks, 256, 0, stream>>>(out_a, lse_a, out_b, lse_b,
                                                            static_cast<__nv_bfloat16*>(out), lse,
                                                            total_q, hq, d);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

}  // namespace pcp
