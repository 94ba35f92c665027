// Decode rows of a mixed PCP batch: one new token attending all keys [0, C)
// of its request ("[MRv2] FlashAttention PCP support for GQA on MRv2",
// overview: mixed-batch decode handled next to the prefill rows; "[MRv2][PCP]
// Carry the row plan ...", "drop pcp_has_prefill": decode rows carried in the
// same plan). A single query row cannot fill a 128-row MMA and the work is
// bound by HBM bandwidth (every key's K and V read once per kv head), so this
// path is CUDA-core code built around the memory system:
//  * split-KV: CTA (split, kv head, row) streams keys [C s, C (s+1)) of one
//    kv head for all G q heads of its group (C = kDecodeChunk = 2048 keys);
//  * a producer warp reads the chunk's block-table entries once, then streams
//    32-key slabs of K and V into a 4-stage shared-memory ring with TMA: one
//    unswizzled box per page (the head's D contiguous elements of each of its
//    rows), completion on mbarriers;
//  * four consumer warps share each slab, a half-warp per group of keys: each
//    lane one 128-bit (D = 128) or 64-bit (D = 64) shared load per K and V row,
//    packed fp32 dot products, a butterfly reduce-scatter over the 16 lanes so
//    that each lane ends with one (key, head) score, one exponential per lane,
//    fp32 online softmax per q head with lazy rescaling;
//  * partial (out, lse) per split in the workspace, merged by log-sum-exp in
//    decode_merge_kernel;
//  * FP8 (e4m3) cache: the slabs hold the codes (rows of D bytes), each lane
//    converts its 8 (D = 128) or 4 (D = 64) codes to fp32 after the shared
//    load; the K descale folds into the query scale, the V descale into the
//    split's output.
// Also here: the LSE merge of the two prefill partials when the context and
// new-token parts are computed separately.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

namespace {

#ifndef PCP_DECODE_STAGES
#define PCP_DECODE_STAGES 4
#endif
constexpr int kSlab = 32;                  // keys per pipeline stage
constexpr int kStages = PCP_DECODE_STAGES;  // slabs in flight per CTA
constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxPages = kDecodeChunk / 8;  // block-table entries of one chunk (block_size >= 8)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int D, int GMAX, bool F8 = false>
struct DecCfg {
    static constexpr int kRowBytes = F8 ? D : 2 * D;                // one key of one head
    static constexpr int kSlabBytes = kSlab * kRowBytes;            // K (or V) of one slab
    static constexpr int kStageBytes = 2 * kSlabBytes;
    static constexpr int kBars = kStages * kStageBytes;
    static constexpr int kPages = kBars + 2 * kStages * 8;
    static constexpr int kComb = kPages + kMaxPages * 4 + 16;
    static constexpr int kSmem = kComb + (2 * kConsumerWarps * GMAX + kConsumerWarps * GMAX * D) * 4 + 1024;
};

// VEC consecutive elements (first dim e0) of row kr of a slab whose rows are
// VEC * 16 elements (D), as fp32: bf16 widened by a shift, FP8 codes converted.
template <int VEC, bool F8>
__device__ __forceinline__ void load_row(const uint8_t* slab, int kr, int e0, float (&f)[VEC]) {
    if constexpr (F8) {
        const uint8_t* p = slab + kr * (VEC * 16) + e0;
        if constexpr (VEC == 8) {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            float a[4], b[4];
            e4m3x4_to_f32(u.x, a);
            e4m3x4_to_f32(u.y, b);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[i] = a[i];
                f[4 + i] = b[i];
            }
        } else {
            float a[4];
            e4m3x4_to_f32(*reinterpret_cast<const uint32_t*>(p), a);
#pragma unroll
            for (int i = 0; i < 4; ++i) f[i] = a[i];
        }
    } else {
        const uint8_t* p = slab + kr * (VEC * 32) + e0 * 2;
        if constexpr (VEC == 8) {
            const uint4 u = *reinterpret_cast<const uint4*>(p);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = __uint_as_float(w[i] << 16);
                f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
            }
        } else {
            const uint2 u = *reinterpret_cast<const uint2*>(p);
            f[0] = __uint_as_float(u.x << 16);
            f[1] = __uint_as_float(u.x & 0xFFFF0000u);
            f[2] = __uint_as_float(u.y << 16);
            f[3] = __uint_as_float(u.y & 0xFFFF0000u);
        }
    }
}

template <int D, int GMAX, bool F8>
__global__ void __launch_bounds__(kDecThreads)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  PrefillArgs a, float* __restrict__ dec_out, float* __restrict__ dec_lse, int max_splits,
                  int box_rows) {
    using C = DecCfg<D, GMAX, F8>;
    constexpr int VEC = D / 16;
    const int split = blockIdx.x, hk = blockIdx.y, ri = blockIdx.z;
    if (!a.row_ok[ri]) return;
    const pcp_row_t row = a.rows[ri];
    if (!row.is_decode) return;
    const int32_t C_len = row.kv_end;
    const int32_t lo = split * kDecodeChunk;
    if (lo >= C_len) return;
    const int32_t hi = min(C_len, lo + kDecodeChunk);
    const int nslab = (hi - lo + kSlab - 1) / kSlab;
    const int G = a.hq / a.hkv;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int32_t bs = a.block_size;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto full_bar = [&](int s) { return sbase + C::kBars + 8 * s; };
    auto empty_bar = [&](int s) { return sbase + C::kBars + 8 * (kStages + s); };
    int32_t* page_row = reinterpret_cast<int32_t*>(smem + C::kPages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kPages + kMaxPages * 4);
    float* s_m = reinterpret_cast<float*>(smem + C::kComb);
    float* s_l = s_m + kConsumerWarps * GMAX;
    float* s_acc = s_l + kConsumerWarps * GMAX;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    bool ok = true;
    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------------- producer
        // every block-table entry of the chunk once (lane p: pages p and p + 32)
        const int32_t* table = a.block_table + (size_t)row.req * a.max_blocks;
        const int32_t oob = (int32_t)(a.num_blocks * bs);  // a row past the cache: zero fill
        const int32_t pg0 = lo / bs;
        const int npages = (hi - 1) / bs - pg0 + 1;
        for (int p = lane; p < npages; p += 32) {
            const int32_t pg = pg0 + p;
            const int32_t id = pg < a.max_blocks ? __ldg(table + pg) : -1;
            int32_t y = oob;
            if (id >= 0 && id < a.num_blocks) y = id * bs;
            else report_status(a.status, PCP_ERR_RANGE);
            page_row[p] = y;
        }
        __syncwarp();
        if (lane == 0) {
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            for (int i = 0; i < nslab; ++i) {
                const int st = i % kStages;
                if (!(ok = mbar_wait(empty_bar(st), ((i / kStages) & 1) ^ 1, abort_flag))) break;
                mbar_arrive_expect_tx(full_bar(st), C::kStageBytes);
                const uint32_t dst = sbase + st * C::kStageBytes;
                for (int b = 0; b < kSlab / box_rows; ++b) {
                    const int32_t key = lo + i * kSlab + b * box_rows;
                    int32_t y = oob;
                    if (key < hi) {
                        const int32_t base = page_row[key / bs - pg0];
                        if (base != oob) y = base + (key % bs);
                    }
                    tma_load_3d(dst + b * box_rows * C::kRowBytes, &tm_k, full_bar(st), 0, hk, y);
                    tma_load_3d(dst + C::kSlabBytes + b * box_rows * C::kRowBytes, &tm_v, full_bar(st), 0, hk, y);
                }
            }
            if (!ok) report_status(a.status, PCP_ERR_TIMEOUT);
        }
        __syncwarp();
    }

    const int half = lane / 16, dl = lane % 16;
    // Each half-warp handles KPI keys per step: its 16 lanes hold 8 (D = 128) or 4
    // (D = 64) dims each, so every lane forms KPI x GP partial dot products; a
    // butterfly reduce-scatter over the 16 lanes leaves lane dl with the full score
    // of key dl / GP for head dl % GP (15 shuffles for all 16 scores).
    constexpr int GP = GMAX;        // heads of a group, padded to a power of two
    constexpr int KPI = 16 / GP;    // keys per half-warp and step
    constexpr int NSUB = (kSlab + 8 * KPI - 1) / (8 * KPI);
    const int g_own = dl % GP, kk_own = dl / GP;
    float m_own = -INFINITY, l_part = 0.f;
    float acc[GP][VEC];
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
    if (warp < kConsumerWarps) {
        // ---------------------------------------------------------------- consumers
        const float kd = F8 ? __ldg(a.k_descale + (size_t)row.req * a.hkv + hk) : 1.f;
        const float sl2 = a.scale * kd * kLog2e;
        float qf[GP][VEC];
        const __nv_bfloat16* qbase = reinterpret_cast<const __nv_bfloat16*>(a.q) +
                                     ((size_t)row.q_start * a.hq + (size_t)hk * G) * D + dl * VEC;
#pragma unroll
        for (int g = 0; g < GP; ++g) {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                qf[g][e] = g < G ? __bfloat162float(qbase[(size_t)g * D + e]) * sl2 : 0.f;
        }
        for (int i = 0; i < nslab; ++i) {
            const int st = i % kStages;
            if (!(ok = mbar_wait_warp(full_bar(st), (i / kStages) & 1, abort_flag))) break;
            const uint8_t* kslab = smem + st * C::kStageBytes;
            const uint8_t* vslab = kslab + C::kSlabBytes;
            const int32_t key_base = lo + i * kSlab;
#pragma unroll
            for (int sub = 0; sub < NSUB; ++sub) {
                const int base_r = sub * 8 * KPI + (warp * 2 + half) * KPI;
                // partial dot products of this lane's dims: v[kk * GP + g]
                float v[16];
#pragma unroll
                for (int kk = 0; kk < KPI; ++kk) {
                    const int r = base_r + kk;
                    float kf[VEC];
                    if (r < kSlab) {
                        load_row<VEC, F8>(kslab, r, dl * VEC, kf);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) kf[e] = 0.f;
                    }
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        float2 d2 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int e = 0; e < VEC; e += 2)
                            d2 = ffma2(make_float2(qf[g][e], qf[g][e + 1]), make_float2(kf[e], kf[e + 1]), d2);
                        v[kk * GP + g] = d2.x + d2.y;
                    }
                }
                // reduce-scatter: after the step with offset o a lane keeps the half of its
                // values selected by bit o of its lane index
#pragma unroll
                for (int o = 8, n = 16; o >= 1; o >>= 1, n >>= 1) {
                    const bool upper = (dl & o) != 0;
#pragma unroll
                    for (int t = 0; t < n / 2; ++t) {
                        const float send = upper ? v[t] : v[t + n / 2];
                        const float keep = upper ? v[t + n / 2] : v[t];
                        v[t] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
                }
                const int r_own = base_r + kk_own;
                const bool live_own = g_own < G && r_own < kSlab && key_base + r_own < hi;
                const float s_own = live_own ? v[0] : -INFINITY;
                // running max of this head over the lanes holding it (lanes dl = g_own mod GP)
                float mx = s_own;
#pragma unroll
                for (int o = GP; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_new = fmaxf(m_own, mx);
                // lazy rescaling: keep the old reference max unless the new one exceeds it by 2^8
                const bool need = m_new > m_own + 8.0f;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? fast_exp2(m_own - m_new) : 1.f;
                    if (need) {
                        m_own = m_new;
                        l_part *= alpha;
                    }
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        const float ag = __shfl_sync(0xffffffffu, alpha, half * 16 + g);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[g][e] *= ag;
                    }
                }
                const float mu = m_own == -INFINITY ? 0.f : m_own;  // no key yet: every weight is 0
                const float p_own = fast_exp2(s_own - mu);
                l_part += p_own;
#pragma unroll
                for (int kk = 0; kk < KPI; ++kk) {
                    const int r = base_r + kk;
                    float vf[VEC];
                    if (r < kSlab && key_base + r < hi) {
                        load_row<VEC, F8>(vslab, r, dl * VEC, vf);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) vf[e] = 0.f;  // rows past the end may hold anything
                    }
#pragma unroll
                    for (int g = 0; g < GP; ++g) {
                        const float p = __shfl_sync(0xffffffffu, p_own, half * 16 + kk * GP + g);
#pragma unroll
                        for (int e = 0; e < VEC; e += 2) {
                            const float2 r2 = ffma2(make_float2(p, p), make_float2(vf[e], vf[e + 1]),
                                                    make_float2(acc[g][e], acc[g][e + 1]));
                            acc[g][e] = r2.x;
                            acc[g][e + 1] = r2.y;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(st));
        }
        if (!ok) report_status(a.status, PCP_ERR_TIMEOUT);
        // the sum of this lane's head over its lanes, then combine the two half-warps
        // (lane i and lane i ^ 16 hold the same dims) and hand the warp's state over
#pragma unroll
        for (int o = GP; o < 16; o <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, o);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float mg = __shfl_sync(0xffffffffu, m_own, half * 16 + g);
            const float lg = __shfl_sync(0xffffffffu, l_part, half * 16 + g);
            const float mo = __shfl_xor_sync(0xffffffffu, mg, 16);
            const float lo2 = __shfl_xor_sync(0xffffffffu, lg, 16);
            const float M = fmaxf(mg, mo);
            const float fa = M == -INFINITY ? 0.f : fast_exp2(mg - M);
            const float fb = M == -INFINITY ? 0.f : fast_exp2(mo - M);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[g][e], 16);
                acc[g][e] = fa * acc[g][e] + fb * ao;
            }
            if (half == 0 && g < G) {
                if (dl == 0) {
                    s_m[warp * GMAX + g] = M;
                    s_l[warp * GMAX + g] = fa * lg + fb * lo2;
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) s_acc[(warp * GMAX + g) * D + dl * VEC + e] = acc[g][e];
            }
        }
    }
    __syncthreads();
    // combine the consumer warps and write this split's partial
    const float vd = F8 ? __ldg(a.v_descale + (size_t)row.req * a.hkv + hk) : 1.f;
    for (int i = threadIdx.x; i < G * D; i += kDecThreads) {
        const int g = i / D, d = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, s_m[w * GMAX + g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float f = fast_exp2(s_m[w * GMAX + g] - M);
                L += f * s_l[w * GMAX + g];
                O += f * s_acc[(w * GMAX + g) * D + d];
            }
        }
        const int h = hk * G + g;
        const size_t slot = ((size_t)ri * a.hq + h) * (2 * max_splits) + split;  // one partial per split
        dec_out[slot * D + d] = L > 0.f ? O / L * vd : 0.f;
        if (d == 0) dec_lse[slot] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    }
}

// Merge the partials of every decode row into out (bf16) and lse: parts_per_split
// partials for each of the row's splits (the first ones of its 2 x max_splits
// slots).
template <int D>
__global__ void __launch_bounds__(D)
    decode_merge_kernel(PrefillArgs a, const float* __restrict__ dec_out, const float* __restrict__ dec_lse,
                        int max_splits, int parts_per_split) {
    const int ri = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
    if (!a.row_ok[ri]) return;
    const pcp_row_t row = a.rows[ri];
    if (!row.is_decode) return;
    const int n = parts_per_split * min(max_splits, (row.kv_end + kDecodeChunk - 1) / kDecodeChunk);
    const size_t base = ((size_t)ri * a.hq + h) * (2 * max_splits);
    // the loads of several partials in flight at once (each loop is a chain of
    // loads otherwise)
    float M = -INFINITY;
#pragma unroll 8
    for (int s = 0; s < n; ++s) M = fmaxf(M, dec_lse[base + s]);
    float W = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll 8
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

// LSE merge of the nparts prefill partials of every non-decode row:
// M = max lse_i, w_i = exp(lse_i - M), out = sum w_i out_i / sum w_i,
// lse = M + log sum w_i; parts with lse = -inf weigh 0, all -inf give (0, -inf).
__global__ void __launch_bounds__(256)
    separate_merge_kernel(PrefillArgs a) {
    if (!a.row_ok[blockIdx.y]) return;
    const pcp_row_t row = a.rows[blockIdx.y];
    if (row.is_decode) return;
    const int D = a.d, chunks = D / 4;
    const size_t out_stride = (size_t)a.total_q * a.hq * D, lse_stride = (size_t)a.hq * a.total_q;
    const int64_t n = (int64_t)row.q_len * a.hq * chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % chunks);
        const int64_t th = i / chunks;
        const int h = (int)(th % a.hq);
        const int32_t t = row.q_start + (int32_t)(th / a.hq);
        const size_t li = (size_t)h * a.total_q + t;
        const size_t o = ((size_t)t * a.hq + h) * D + 4 * c;
        float M = -INFINITY;
        for (int p = 0; p < a.nparts; ++p) M = fmaxf(M, a.part_lse[p * lse_stride + li]);
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse = -INFINITY;
        if (M != -INFINITY) {
            float W = 0.f;
            for (int p = 0; p < a.nparts; ++p) {
                const float w = __expf(a.part_lse[p * lse_stride + li] - M);
                const float4 x = *reinterpret_cast<const float4*>(a.part_out + p * out_stride + o);
                r.x += w * x.x;
                r.y += w * x.y;
                r.z += w * x.z;
                r.w += w * x.w;
                W += w;
            }
            const float inv = 1.f / W;
            r = make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
            lse = M + __logf(W);
        }
        uint2 w;
        w.x = pack_bf16x2(r.x, r.y);
        w.y = pack_bf16x2(r.z, r.w);
        *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(a.out) + o) = w;
        if (c == 0) a.lse[(size_t)h * a.total_q + t] = lse;
    }
}

template <int D, int GMAX, bool F8>
int launch_decode_dgf(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                      cudaStream_t stream) {
    const int box_rows = a.block_size < kSlab ? a.block_size : kSlab;
    const int64_t slots = a.num_blocks * a.block_size;
    CUtensorMap tk, tv;
    const int esize = F8 ? 1 : 2;
    const bool maps = make_kv_row_map(&tk, a.key_cache, D, esize, a.hkv, slots, box_rows) &&
                      make_kv_row_map(&tv, a.value_cache, D, esize, a.hkv, slots, box_rows);
    if (!maps) return PCP_ERR_CUDA;
    const int smem = DecCfg<D, GMAX, F8>::kSmem;
    cudaError_t e =
        cudaFuncSetAttribute(decode_kernel<D, GMAX, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    dim3 grid(max_splits, a.hkv, a.num_rows);
    decode_kernel<D, GMAX, F8><<<grid, kDecThreads, smem, stream>>>(tk, tv, a, dec_out, dec_lse, max_splits,
                                                                    box_rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

int launch_merge(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits, int pps,
                 cudaStream_t stream) {
    if (a.d == 64)
        decode_merge_kernel<64><<<dim3(a.num_rows, a.hq), 64, 0, stream>>>(a, dec_out, dec_lse, max_splits, pps);
    else
        decode_merge_kernel<128><<<dim3(a.num_rows, a.hq), 128, 0, stream>>>(a, dec_out, dec_lse, max_splits, pps);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

template <int D, int GMAX>
int launch_decode_dg(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                     cudaStream_t stream) {
    return a.k_descale ? launch_decode_dgf<D, GMAX, true>(a, dec_out, dec_lse, max_splits, stream)
                       : launch_decode_dgf<D, GMAX, false>(a, dec_out, dec_lse, max_splits, stream);
}

template <int D>
int launch_decode_d(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                    cudaStream_t stream) {
    const int G = a.hq / a.hkv;
    if (G <= 2) return launch_decode_dg<D, 2>(a, dec_out, dec_lse, max_splits, stream);
    if (G <= 4) return launch_decode_dg<D, 4>(a, dec_out, dec_lse, max_splits, stream);
    if (G <= 8) return launch_decode_dg<D, 8>(a, dec_out, dec_lse, max_splits, stream);
    if (G <= 16) return launch_decode_dg<D, 16>(a, dec_out, dec_lse, max_splits, stream);
    return PCP_ERR_UNSUPPORTED;
}

}  // namespace

#ifndef PCP_DECODE_TC
#define PCP_DECODE_TC 1  // 1: the tensor-core decode where it applies (head_dim 128, G <= 8)
#endif

bool decode_side_applies(const PrefillArgs& a) { return PCP_DECODE_TC && decode_tc_applies(a); }

int launch_decode(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                  cudaStream_t stream, int grid) {
    if (a.d != 64 && a.d != 128) return PCP_ERR_UNSUPPORTED;
    int rc = PCP_DECODE_TC ? launch_decode_tc(a, dec_out, dec_lse, max_splits, stream, grid) : PCP_ERR_UNSUPPORTED;
    // partials per split: the tensor-core kernel writes one per softmax warpgroup
    // over an FP8 cache and with more than 8 q heads per kv head
    int pps = (a.k_descale || a.hq / a.hkv > 8) ? 2 : 1;
    if (rc == PCP_ERR_UNSUPPORTED) {
        rc = a.d == 64 ? launch_decode_d<64>(a, dec_out, dec_lse, max_splits, stream)
                       : launch_decode_d<128>(a, dec_out, dec_lse, max_splits, stream);
        pps = 1;
    }
    if (rc != PCP_OK) return rc;
    return launch_merge(a, dec_out, dec_lse, max_splits, pps, stream);
}

int launch_separate_merge(const PrefillArgs& a, cudaStream_t stream) {
    separate_merge_kernel<<<dim3(64, a.num_rows), 256, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

}  // namespace pcp
