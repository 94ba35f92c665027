// Decode rows of a mixed PCP batch: one new token attending all keys [0, C)
// of its request ("[MRv2] FlashAttention PCP support for GQA on MRv2",
// overview: mixed-batch decode handled next to the prefill rows; "[MRv2][PCP]
// Carry the row plan ...", "drop pcp_has_prefill": decode rows carried in the
// same plan). A single query row cannot fill a 128-row MMA, so this path is
// bandwidth-bound CUDA-core code:
//  * split-KV: CTA (split, kv head, row) streams keys [512 s, 512 (s+1)) of one
//    kv head, every key's K and V row read once for all G q heads of the group;
//  * 16 lanes per key, each lane one 16-byte (128-bit) load of K and of V
//    (8 bf16 of D = 128), two keys per warp, four keys in flight per half-warp;
//  * fp32 online softmax per head, partial (out, lse) per split in the
//    workspace, merged by log-sum-exp in decode_merge_kernel.
// Also here: the LSE merge of the two prefill partials when the context and
// new-token parts are computed separately.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

namespace {

constexpr int kDecThreads = 128;
constexpr int kUnroll = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int VEC>
struct VecLoad;
template <>
struct VecLoad<8> {  // 16 bytes
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&f)[8]) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
};
template <>
struct VecLoad<4> {  // 8 bytes
    __device__ __forceinline__ static void load(const __nv_bfloat16* p, float (&f)[4]) {
        const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xFFFF0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xFFFF0000u);
    }
};

template <int D, int GMAX>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(PrefillArgs a, float* __restrict__ dec_out, float* __restrict__ dec_lse, int max_splits) {
    constexpr int VEC = D / 16;
    const int split = blockIdx.x, hk = blockIdx.y, ri = blockIdx.z;
    if (!a.row_ok[ri]) return;
    const pcp_row_t row = a.rows[ri];
    if (!row.is_decode) return;
    const int32_t C = row.kv_end;
    const int32_t lo = split * kDecodeChunk;
    if (lo >= C) return;
    const int32_t hi = min(C, lo + kDecodeChunk);
    const int G = a.hq / a.hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int half = lane / 16, dl = lane % 16;
    const float sl2 = a.scale * kLog2e;
    const int32_t bs = a.block_size;

    __shared__ float s_m[4][GMAX], s_l[4][GMAX];
    __shared__ float s_acc[4][GMAX][D];

    float qf[GMAX][VEC];
    const __nv_bfloat16* qbase = reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                 ((size_t)row.q_start * a.hq + (size_t)hk * G) * D + dl * VEC;
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        if (g < G) {
            VecLoad<VEC>::load(qbase + (size_t)g * D, qf[g]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qf[g][e] *= sl2;
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) qf[g][e] = 0.f;
        }
    }
    float m[GMAX], l[GMAX], acc[GMAX][VEC];
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
    }
    const int32_t* table = a.block_table + (size_t)row.req * a.max_blocks;
    const __nv_bfloat16* kc = reinterpret_cast<const __nv_bfloat16*>(a.key_cache);
    const __nv_bfloat16* vc = reinterpret_cast<const __nv_bfloat16*>(a.value_cache);
    const int32_t stride = 8 * kUnroll;  // keys per CTA iteration over all half-warps
    // The trip count depends on the warp only, never on the half-warp, so both
    // halves always run the full-warp shuffles below together.
    for (int32_t kw = lo + warp * 2; kw < hi; kw += stride) {
        float kf[kUnroll][VEC], vf[kUnroll][VEC];
        bool live[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int32_t k = kw + half + 8 * u;
            live[u] = false;
            if (k < hi) {
                const int32_t pg = k / bs;
                const int32_t id = pg < a.max_blocks ? __ldg(table + pg) : -1;
                if (id >= 0 && id < a.num_blocks) {
                    const size_t off = (((size_t)id * bs + (k - pg * bs)) * a.hkv + hk) * D + dl * VEC;
                    VecLoad<VEC>::load(kc + off, kf[u]);
                    VecLoad<VEC>::load(vc + off, vf[u]);
                    live[u] = true;
                } else {
                    report_status(a.status, PCP_ERR_RANGE);
                }
            }
            if (!live[u]) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) kf[u][e] = vf[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int g = 0; g < GMAX; ++g) {
            if (g >= G) break;
            float s[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < VEC; ++e) d = fmaf(qf[g][e], kf[u][e], d);
                d += __shfl_xor_sync(0xffffffffu, d, 8);
                d += __shfl_xor_sync(0xffffffffu, d, 4);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                s[u] = live[u] ? d : -INFINITY;
            }
            float mx = s[0];
#pragma unroll
            for (int u = 1; u < kUnroll; ++u) mx = fmaxf(mx, s[u]);
            const float m_new = fmaxf(m[g], mx);
            const float mu = m_new == -INFINITY ? 0.f : m_new;  // no key yet: every weight is 0
            const float alpha = fast_exp2(m[g] - mu);
            float p[kUnroll], ps = 0.f;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                p[u] = fast_exp2(s[u] - mu);
                ps += p[u];
            }
            l[g] = l[g] * alpha + ps;
            m[g] = m_new;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                float x = acc[g][e] * alpha;
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) x = fmaf(p[u], vf[u][e], x);
                acc[g][e] = x;
            }
        }
    }
    // combine the two half-warps of each warp (lane i and lane i ^ 16 hold the
    // same dims), then the four warps of the CTA through shared memory
#pragma unroll
    for (int g = 0; g < GMAX; ++g) {
        if (g >= G) break;
        const float mo = __shfl_xor_sync(0xffffffffu, m[g], 16);
        const float lo2 = __shfl_xor_sync(0xffffffffu, l[g], 16);
        const float M = fmaxf(m[g], mo);
        const float fa = M == -INFINITY ? 0.f : fast_exp2(m[g] - M);
        const float fb = M == -INFINITY ? 0.f : fast_exp2(mo - M);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float ao = __shfl_xor_sync(0xffffffffu, acc[g][e], 16);
            acc[g][e] = fa * acc[g][e] + fb * ao;
        }
        m[g] = M;
        l[g] = fa * l[g] + fb * lo2;
        if (half == 0) {
            if (dl == 0) {
                s_m[warp][g] = m[g];
                s_l[warp][g] = l[g];
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) s_acc[warp][g][dl * VEC + e] = acc[g][e];
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * D; i += kDecThreads) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, s_m[w][g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float f = fast_exp2(s_m[w][g] - M);
                L += f * s_l[w][g];
                O += f * s_acc[w][g][d];
            }
        }
        const int h = hk * G + g;
        const size_t slot = ((size_t)ri * a.hq + h) * max_splits + split;
        dec_out[slot * D + d] = L > 0.f ? O / L : 0.f;
        if (d == 0) dec_lse[slot] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    }
}

// Merge the per-split partials of every decode row into out (bf16) and lse.
template <int D>
__global__ void __launch_bounds__(D)
    decode_merge_kernel(PrefillArgs a, const float* __restrict__ dec_out, const float* __restrict__ dec_lse,
                        int max_splits) {
    const int ri = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
    if (!a.row_ok[ri]) return;
    const pcp_row_t row = a.rows[ri];
    if (!row.is_decode) return;
    const int n = min(max_splits, (row.kv_end + kDecodeChunk - 1) / kDecodeChunk);
    const size_t base = ((size_t)ri * a.hq + h) * max_splits;
    float M = -INFINITY;
    for (int s = 0; s < n; ++s) M = fmaxf(M, dec_lse[base + s]);
    float W = 0.f, O = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n; ++s) {
            const float w = __expf(dec_lse[base + s] - M);
            W += w;
            O += w * dec_out[(base + s) * D + d];
        }
    }
    const int32_t t = row.q_start;
    reinterpret_cast<__nv_bfloat16*>(a.out)[((size_t)t * a.hq + h) * D + d] = __float2bfloat16_rn(W > 0.f ? O / W : 0.f);
    if (d == 0) a.lse[(size_t)h * a.total_q + t] = W > 0.f ? M + __logf(W) : -INFINITY;
}

// LSE merge of the two prefill partials of every non-decode row.
__global__ void __launch_bounds__(256)
    separate_merge_kernel(PrefillArgs a) {
    if (!a.row_ok[blockIdx.y]) return;
    const pcp_row_t row = a.rows[blockIdx.y];
    if (row.is_decode) return;
    const int D = a.d, chunks = D / 4;
    const int64_t n = (int64_t)row.q_len * a.hq * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % chunks);
        const int64_t th = i / chunks;
        const int h = (int)(th % a.hq);
        const int32_t t = row.q_start + (int32_t)(th / a.hq);
        const float la = a.part_lse[0][(size_t)h * a.total_q + t];
        const float lb = a.part_lse[1][(size_t)h * a.total_q + t];
        const size_t o = ((size_t)t * a.hq + h) * D + 4 * c;
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse = -INFINITY;
        if (!(la == -INFINITY && lb == -INFINITY)) {
            const float M = fmaxf(la, lb);
            const float wa = __expf(la - M), wb = __expf(lb - M);
            const float inv = 1.f / (wa + wb);
            const float4 xa = *reinterpret_cast<const float4*>(a.part_out[0] + o);
            const float4 xb = *reinterpret_cast<const float4*>(a.part_out[1] + o);
            r = make_float4((wa * xa.x + wb * xb.x) * inv, (wa * xa.y + wb * xb.y) * inv,
                            (wa * xa.z + wb * xb.z) * inv, (wa * xa.w + wb * xb.w) * inv);
            lse = M + __logf(wa + wb);
        }
        uint2 w;
        w.x = pack_bf16x2(r.x, r.y);
        w.y = pack_bf16x2(r.z, r.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + o) = w;
        if (c == 0) a.lse[(size_t)h * a.total_q + t] = lse;
    }
}

template <int D, int GMAX>
int launch_decode_dg(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                     cudaStream_t stream) {
    dim3 grid(max_splits, a.hkv, a.num_rows);
    decode_kernel<D, GMAX><<<grid, kDecThreads, 0, stream>>>(a, dec_out, dec_lse, max_splits);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    decode_merge_kernel<D><<<dim3(a.num_rows, a.hq), D, 0, stream>>>(a, dec_out, dec_lse, max_splits);
    e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

template <int D>
int launch_decode_d(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                    cudaStream_t stream) {
    const int G = a.hq / a.hkv;
    if (G <= 4) return launch_decode_dg<D, 4>(a, dec_out, dec_lse, max_splits, stream);
    if (G <= 8) return launch_decode_dg<D, 8>(a, dec_out, dec_lse, max_splits, stream);
    if (G <= 16) return launch_decode_dg<D, 16>(a, dec_out, dec_lse, max_splits, stream);
    return PCP_ERR_UNSUPPORTED;
}

}  // namespace

int launch_decode(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                  cudaStream_t stream) {
    if (a.d == 64) return launch_decode_d<64>(a, dec_out, dec_lse, max_splits, stream);
    if (a.d == 128) return launch_decode_d<128>(a, dec_out, dec_lse, max_splits, stream);
    return PCP_ERR_UNSUPPORTED;
}

int launch_separate_merge(const PrefillArgs& a, cudaStream_t stream) {
    separate_merge_kernel<<<dim3(64, a.num_rows), 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

}  // namespace pcp
