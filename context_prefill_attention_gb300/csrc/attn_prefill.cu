// Prefill / context attention of PCP rows on the 5th-generation tensor cores.
//
// What it computes ("Feat/pcp qwen36 hybrid", "Changes": end-aligned causal
// attention of a rank's contiguous slice over the reconstructed K/V; "[MRv2]
// FlashAttention PCP support for GQA on MRv2", overview: cached-prefix context
// attention combined by log-sum-exp; "[MRv2][PCP] Carry the row plan ...",
// "What made it removable": a row's seq_len is its end position): for query j
// of a row at position p = kv_end - q_len + j, the softmax of
// scale * q . k over keys k in [k_lo, min(k_hi, p + 1)), its weighted sum of V,
// and the natural-log LSE.
//
// Design (sm_103a):
//  * persistent grid, one CTA per SM; work items = (row tile of 128 tokens,
//    pass, pair of q heads sharing one kv head), longest first;
//  * warp 8 produces: TMA loads of the Q tiles and of K/V pages (one 3-D box
//    of block_size keys x 64 dims per page and half head-dim) straight from the
//    paged cache through the block table, 128-byte swizzled; K(j) and V(j) land
//    on one barrier;
//  * lane 0 of warp 9 alone issues the tcgen05 MMAs: S = Q K^T into TMEM (A and
//    B from shared memory), then O += P V with P read from TMEM (it overwrites
//    S) and V from shared memory. The issuing thread is the throughput limit
//    (each barrier read, commit or extra instruction there leaves the tensor
//    pipe idle), so it reads one barrier per tile for K and V, builds its
//    descriptors once per stage, and commits only S and O completions;
//  * warps 0-3 and 4-7 are two softmax warpgroups, one per q head of the item,
//    one thread per query row: they read S from TMEM, mask, exponentiate
//    against the row's reference max without a max reduction first once it is
//    known (falling back to an exact pass that rescales O in TMEM), write P
//    back as bf16, and finally normalise O and store out and lse; the last
//    head's warpgroup releases the K, V and Q stages;
//  * the two heads' MMAs interleave (S0 S1 | PV0 S0' PV1 S1' | ...) so each
//    warpgroup's softmax overlaps the other head's MMAs;
//  * every mbarrier wait is bounded: a wait that runs out sets PCP_ERR_TIMEOUT
//    in the status word and the CTA winds down, freeing its TMEM;
//  * FP8 (e4m3) cache: the producer's TMA brings the codes in. D = 128: the K
//    codes land 128-byte swizzled and S takes them as e4m3 operands (kind::
//    f8f6f4) against each item's q, which the softmax threads rewrite (a row
//    each) as two e4m3 terms per element after a power-of-two scale per row
//    (their sum is the bf16 q);
//    the V codes land in the upper half of their stage and warps 10-11 widen
//    them to f16 (one conversion per two codes, exact). D = 64: K and V codes
//    are widened to f16 from a staging area and q converted to f16. P is
//    stored as f16 and PV takes f16 operands; the per-(request, kv head)
//    descales fold into the softmax scale (K) and the epilogue's normalisation
//    (V).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

namespace {

constexpr int kThreads = 384;  // 12 warps: two softmax warpgroups, producer, MMA, two converters
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kConvWarp0 = 10;  // warps 10-11: FP8 code -> bf16 conversion (FP8 cache only)
constexpr int kConvThreads = 64;
// Tuning knobs (compile-time; the defaults are the measured best on GB300).
#ifndef PCP_PREFILL_K_STAGES
#define PCP_PREFILL_K_STAGES 2
#endif
#ifndef PCP_PREFILL_V_STAGES
#define PCP_PREFILL_V_STAGES 3
#endif
#ifndef PCP_POLY_EXP_EVERY
// Off: on GB300 the exponential unit keeps up with the tensor cores, and the
// polynomial only costs issue slots (measured: 1 pair in 4 -> 9% slower).
#define PCP_POLY_EXP_EVERY 1000000
#endif
#ifndef PCP_PREFILL_MAXFREE
#define PCP_PREFILL_MAXFREE 1
#endif
// 1: once a row has a finite reference max, a tile's exponentials use it
// directly (no row-max reduction before them); a tile whose row sum reaches
// kMaxFreeLimit falls back to the exact path (max, rescale). 0: every tile
// computes its row max first.
constexpr bool kMaxFree = PCP_PREFILL_MAXFREE != 0;
// p <= 2^64 keeps O (<= p x keys x |v|) and l far inside fp32 for any bf16 V of
// moderate size and any sequence length this library accepts
constexpr float kMaxFreeLimit = 18446744073709551616.0f;  // 2^64
constexpr int kNK = PCP_PREFILL_K_STAGES;  // K stages
constexpr int kNV = PCP_PREFILL_V_STAGES;  // V stages
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
// one pair in kPolyEvery of a tile uses the polynomial exp2 (a large value turns it off)
constexpr int kPolyEvery = PCP_POLY_EXP_EVERY;

template <int D, bool F8 = false>
struct Cfg {
    static constexpr int kHalves = D / 64;                 // 64-column (128-byte) sub-tiles
    static constexpr int kHalfBytes = 128 * 128;           // 128 rows x 128 bytes
    static constexpr int kTileBytes = kHalves * kHalfBytes;
    static constexpr int kQ = 0;
    static constexpr int kK = kQ + 2 * kTileBytes;
    static constexpr int kV = kK + kNK * kTileBytes;
    // FP8 codes of one tile: 128 rows x D bytes. D = 128: in the upper half of
    // the stage they are converted into (row r of the codes overlays row r of
    // that half, so a row is read whole before it is written); D = 64: their own
    // staging area after the V stages.
    static constexpr int kCodeBytes = kBlockN * D;
    static constexpr bool kInPlace = D == 128;
    // FP8, D = 128: S takes the K codes as e4m3 operands (128 bytes per key, one
    // 128-byte swizzle atom wide, at the start of the K stage) against q written
    // as two e4m3 terms per element; only V is widened to f16
    static constexpr bool kE4 = F8 && D == 128;
    static constexpr int kCK = kV + kNV * kTileBytes;
    static constexpr int kCV = kCK + (F8 && !kInPlace ? kNK * kCodeBytes : 0);
    static constexpr int kBar = kCV + (F8 && !kInPlace ? kNV * kCodeBytes : 0);
    __host__ __device__ static constexpr int code_k(int s) {
        return kE4 ? kK + s * kTileBytes : kInPlace ? kK + s * kTileBytes + kHalfBytes : kCK + s * kCodeBytes;
    }
    __host__ __device__ static constexpr int code_v(int s) {
        return kInPlace ? kV + s * kTileBytes + kHalfBytes : kCV + s * kCodeBytes;
    }
    static constexpr int kNumBars = 2 + 2 * kNK + 2 * kNV + 8 + kNK + kNV + 1;  // + FP8: Q landed
    static constexpr int kMisc = kBar + kNumBars * 8;      // tmem address, abort flag
    static constexpr int kSmem = kMisc + 16 + 1024;  // + alignment slack
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t tmem_s(int g) { return g ? 128u : 0u; }
    __host__ __device__ static constexpr uint32_t tmem_o(int g) { return g ? 256u + D : 256u; }
    // FP8 cache: the codes are widened to f16 (exact), q converted to f16 and P
    // stored as f16, so the MMAs take f16 operands; bf16 cache: bf16 operands
    static constexpr uint32_t kIdescS =
        kE4 ? idesc_e4m3(128, 128) : F8 ? idesc_f16(128, 128, false, false) : idesc_bf16(128, 128, false, false);
    static constexpr uint32_t kIdescO = F8 ? idesc_f16(128, D, false, true) : idesc_bf16(128, D, false, true);
};

struct Item {
    int32_t req, q_tok0, rows_valid, pos0, k_lo, k_hi, k_end, kb, n_tiles, pass, h0, hk, nslots;
};

__device__ __forceinline__ int32_t tiles_of(int32_t k_lo, int32_t k_end, int32_t bs) {
    if (k_end <= k_lo) return 0;
    const int32_t kb = (k_lo / bs) * bs;
    return (k_end - kb + kBlockN - 1) / kBlockN;
}

// Item idx of the sorted unit list. A unit naming a row outside [0, num_rows)
// (never written by the scheduler; a guard against a corrupted list) becomes an
// empty item with no valid query row, which every role skips without a write.
__device__ __forceinline__ Item decode_item(const Unit* units, int32_t idx, int32_t slots_per_unit,
                                            bool dual, int32_t G, const pcp_row_t* rows,
                                            int32_t num_rows, int32_t bs) {
    const Unit u = units[idx / slots_per_unit];
    const int32_t hs = idx % slots_per_unit;
    Item it;
    if (u.row < 0 || u.row >= num_rows) {
        it = Item{};
        it.nslots = dual ? 2 : 1;
        it.h0 = dual ? 2 * hs : hs;
        it.hk = it.h0 / G;
        return it;
    }
    const pcp_row_t r = rows[u.row];
    const int32_t mt = u.mt_pass & 0xFFFFFF;
    it.pass = u.mt_pass >> 24;
    it.req = r.req;
    it.q_tok0 = r.q_start + mt * kBlockM;
    it.rows_valid = min(kBlockM, r.q_len - mt * kBlockM);
    it.pos0 = r.kv_end - r.q_len + mt * kBlockM;
    it.k_lo = u.k_lo;
    it.k_hi = u.k_hi;
    it.k_end = min(u.k_hi, it.pos0 + it.rows_valid);
    it.kb = (u.k_lo / bs) * bs;
    it.n_tiles = tiles_of(u.k_lo, it.k_end, bs);
    it.nslots = dual ? 2 : 1;
    it.h0 = dual ? 2 * hs : hs;
    it.hk = it.h0 / G;
    return it;
}

// One tile of FP8 codes (128 rows x D bytes, row-major) -> bf16 in the
// 128-byte-swizzled K-major layout of a K or V stage (dims 64h..64h+63 of row
// r in half h, 16-byte chunk c of that row at chunk c ^ (r & 7)). Run by the 64
// converter threads (ct = 0..63): D / 16 threads per row, each converting 16
// codes (one 16-byte load) into two 16-byte chunks. In place (D = 128) the codes
// of row r sit where half 1 of row r goes; the threads of a row are in one warp
// and all of them load before any of them stores.
template <int D>
__device__ __forceinline__ void convert_codes(const uint8_t* codes, uint8_t* dst, int ct) {
    constexpr int kTpr = D / 16;             // threads per row
    constexpr int kRpp = kConvThreads / kTpr;  // rows per pass
    constexpr int kBatch = 4;                // rows per thread between warp barriers
    const int t = ct % kTpr, rsub = ct / kTpr;
    const int h = t / 4, c0 = 2 * (t % 4);
    // threads of the second half store their odd chunk first, so the eight
    // threads of a row hit eight different bank groups in each store
    const int first = c0 + (t >= 4 ? 1 : 0), second = c0 + (t >= 4 ? 0 : 1);
#pragma unroll 1
    for (int r0 = 0; r0 < kBlockN; r0 += kRpp * kBatch) {
        uint4 c[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b)
            c[b] = *reinterpret_cast<const uint4*>(codes + (r0 + kRpp * b + rsub) * D + 16 * t);
        __syncwarp();
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = r0 + kRpp * b + rsub;
            const uint2 w0 = e4m3x4_to_f16x4(c[b].x), w1 = e4m3x4_to_f16x4(c[b].y);
            const uint2 w2 = e4m3x4_to_f16x4(c[b].z), w3 = e4m3x4_to_f16x4(c[b].w);
            const uint4 lo = make_uint4(w0.x, w0.y, w1.x, w1.y);  // dims 16t .. 16t+7
            const uint4 hi = make_uint4(w2.x, w2.y, w3.x, w3.y);  // dims 16t+8 .. 16t+15
            uint8_t* row = dst + h * (128 * 128) + r * 128;
            const bool lo_first = first == c0;
            *reinterpret_cast<uint4*>(row + ((first ^ (r & 7)) << 4)) = lo_first ? lo : hi;
            *reinterpret_cast<uint4*>(row + ((second ^ (r & 7)) << 4)) = lo_first ? hi : lo;
        }
        __syncwarp();
    }
}

// The bf16 Q tiles of an item (nslots x kTileBytes bytes from q_base) turned
// into f16 in place, by the 64 converter threads (ct = 0..63): each 16-byte
// chunk holds 8 elements whatever the swizzle, so the conversion is
// elementwise. Values beyond the largest finite f16 saturate to it; the
// return value says whether any did.
__device__ __forceinline__ bool convert_q_f16(uint8_t* q_base, int bytes, int ct) {
    bool over = false;
#pragma unroll 4
    for (int off = ct * 16; off < bytes; off += kConvThreads * 16) {
        uint4 w = *reinterpret_cast<const uint4*>(q_base + off);
        uint32_t* e = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float lo = __uint_as_float(e[i] << 16), hi = __uint_as_float(e[i] & 0xFFFF0000u);
            over |= fabsf(lo) > 65504.f || fabsf(hi) > 65504.f;
            e[i] = pack_f16x2_satfinite(lo, hi);
        }
        *reinterpret_cast<uint4*>(q_base + off) = w;
    }
    return over;
}

// FP8, D = 128: row r of a head's Q tile (bf16, two 64-dim halves of 128 rows,
// 128-byte swizzled) rewritten in place as two e4m3 terms: term t at
// t * kHalfBytes + r * 128, 16-byte chunk c at c ^ (r & 7), the K-major layout
// of an e4m3 MMA operand. The row is first scaled by 2^(8 - ex), ex the binary
// exponent of its largest magnitude (frexp), so that its elements lie below
// 256; the first term is the e4m3 rounding of a scaled element x (4 significant
// bits), and the remainder, a multiple of x's last bit no larger than 8 of them
// (x has bf16's 8 significant bits), is an e4m3 value too: the terms sum to x
// exactly unless the remainder falls under e4m3's smallest subnormal (2^-9 of
// the scaled unit, where the largest element lies in [128, 256): only an element
// below 2^-9 of its row's largest can lose bits, at most 2^-17 of that largest).
// Run by the row's own softmax thread, which
// reads the whole row before writing it. Returns 2^(ex - 8), the factor that
// undoes the scaling; *over is set if an element lies beyond +-65504.
__device__ __forceinline__ float q_row_to_e4m3(uint8_t* tile, int r, bool* over) {
    constexpr int kHalf = 128 * 128;
    uint4 raw[16];  // bf16 chunk c of half h (dims 64h + 8c ..) in raw[8h + c]
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c = 0; c < 8; ++c)
            raw[8 * h + c] = *reinterpret_cast<const uint4*>(tile + h * kHalf + r * 128 + ((c ^ (r & 7)) << 4));
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m = fmax3(m, fabsf(__uint_as_float(w[k] << 16)), fabsf(__uint_as_float(w[k] & 0xFFFF0000u)));
    }
    *over = m > 65504.f;
    int ex = 0;
    frexpf(m, &ex);
    const float f = ldexpf(1.f, 8 - ex);
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {  // codes 16 cc .. 16 cc + 15 = bf16 chunks 2 cc, 2 cc + 1
        uint32_t c1[4], c2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint4 u = raw[2 * cc + k / 2];
            const uint32_t w0 = (k & 1) ? u.z : u.x, w1 = (k & 1) ? u.w : u.y;
            const float v0 = __uint_as_float(w0 << 16) * f, v1 = __uint_as_float(w0 & 0xFFFF0000u) * f;
            const float v2 = __uint_as_float(w1 << 16) * f, v3 = __uint_as_float(w1 & 0xFFFF0000u) * f;
            c1[k] = f32x2_to_e4m3x2(v0, v1) | (f32x2_to_e4m3x2(v2, v3) << 16);
            float back[4];
            e4m3x4_to_f32(c1[k], back);
            c2[k] = f32x2_to_e4m3x2(v0 - back[0], v1 - back[1]) | (f32x2_to_e4m3x2(v2 - back[2], v3 - back[3]) << 16);
        }
        const int chunk = (cc ^ (r & 7)) << 4;
        *reinterpret_cast<uint4*>(tile + r * 128 + chunk) = make_uint4(c1[0], c1[1], c1[2], c1[3]);
        *reinterpret_cast<uint4*>(tile + kHalf + r * 128 + chunk) = make_uint4(c2[0], c2[1], c2[2], c2[3]);
    }
    return ldexpf(1.f, ex - 8);
}

// S = Q_slot K^T over D (K-major A and B, 128-byte swizzle). q_desc / k_desc are
// the descriptors of the tiles' first k-step; a later k-step only moves the start
// address (the descriptor's low 14 bits, in 16-byte units), so each MMA costs one
// add of a constant (the issuing thread's instruction count per MMA is on the
// critical path of the tensor pipe).
template <int D, bool F8>
__device__ __forceinline__ void issue_qk(uint32_t tmem_s, uint64_t q_desc, uint64_t k_desc) {
    if constexpr (Cfg<D, F8>::kE4) {
        // e4m3: q's two term tiles (term t at + t * kHalfBytes) against the K codes,
        // 32 dims (32 bytes of each 128-byte row) per MMA: the same 8 MMAs
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int ks = 0; ks < D / 32; ++ks)
                mma_ss_e4m3(tmem_s, q_desc + (uint32_t)((t * Cfg<D>::kHalfBytes + ks * 32) >> 4),
                            k_desc + (uint32_t)(ks * 2), Cfg<D, F8>::kIdescS, (t | ks) ? 1u : 0u);
    } else {
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            const uint32_t off = ((ks / 4) * Cfg<D>::kHalfBytes + (ks % 4) * 32) >> 4;
            mma_ss(tmem_s, q_desc + off, k_desc + off, Cfg<D, F8>::kIdescS, ks > 0 ? 1u : 0u);
        }
    }
}

// O (+)= P V: P from TMEM (bf16 pairs in the S columns), V MN-major in shared
// memory (v_desc: the descriptor of the tile's first 16 keys).
template <int D, bool F8>
__device__ __forceinline__ void issue_pv(uint32_t tmem_o, uint32_t tmem_p, uint64_t v_desc, bool accumulate) {
#pragma unroll
    for (int ks = 0; ks < kBlockN / 16; ++ks)
        mma_ts(tmem_o, tmem_p + ks * 8, v_desc + (uint32_t)(ks * 2048 >> 4), Cfg<D, F8>::kIdescO,
               (accumulate || ks > 0) ? 1u : 0u);
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, PrefillArgs a) {
    using C = Cfg<D, F8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kBar;
    // barrier addresses
    const uint32_t q_full = bar0, q_empty = bar0 + 8;
    auto k_full = [&](int s) { return bar0 + 16 + 8 * s; };
    auto k_empty = [&](int s) { return bar0 + 16 + 8 * (kNK + s); };
    auto v_full = [&](int s) { return bar0 + 16 + 8 * (2 * kNK + s); };
    auto v_empty = [&](int s) { return bar0 + 16 + 8 * (2 * kNK + kNV + s); };
    const uint32_t bx = bar0 + 16 + 8 * (2 * kNK + 2 * kNV);
    auto s_full = [&](int g) { return bx + 8 * g; };
    auto p_full = [&](int g) { return bx + 16 + 8 * g; };
    auto o_done = [&](int g) { return bx + 32 + 8 * g; };
    auto o_free = [&](int g) { return bx + 48 + 8 * g; };
    // FP8: the codes of K / V stage s have landed
    auto kc_full = [&](int s) { return bx + 64 + 8 * s; };
    auto vc_full = [&](int s) { return bx + 64 + 8 * (kNK + s); };
    // FP8: the bf16 Q tiles have landed (the converters turn them into f16, then arrive on q_full)
    const uint32_t qc_full = bx + 64 + 8 * (kNK + kNV);
    // bf16: K(j) and V(j) land together on v_full(stage of V(j)), so the MMA
    // issuer reads one barrier per tile for both (every barrier read by the issuer
    // costs tensor-pipe time); FP8: the converters fill k_full and v_full apart
    constexpr bool kMerged = !F8;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = a.hq / a.hkv;
    const bool dual = (G % 2) == 0;
    const int slots_per_unit = dual ? a.hq / 2 : a.hq;
    const int slots_per_item = dual ? 2 : 1;  // q heads per item (Item::nslots)
    const int32_t bs = a.block_size;

    if (threadIdx.x == 0) {
        // q_full: the TMA (bf16), the converter warps (FP8, D = 64) or the softmax
        // warps of the item's head slots (FP8, D = 128)
        mbar_init(q_full, C::kE4 ? (dual ? 8 : 4) : F8 ? kConvThreads / 32 : 1);
        if (F8) mbar_init(qc_full, 1);
        // both head slots' warpgroups free Q when an item has two (each reads its
        // rows' q scales at the item's start, before its last tile)
        mbar_init(q_empty, dual ? 2 : 1);
        // FP8: a stage is full when both converter warps have arrived
        const uint32_t fill_count = F8 ? kConvThreads / 32 : 1;
        // (FP8, D = 128: the K codes are the MMA operand, full once TMA has landed them)
        for (int s = 0; s < kNK; ++s) { mbar_init(k_full(s), C::kE4 ? 1 : fill_count); mbar_init(k_empty(s), 1); }
        for (int s = 0; s < kNV; ++s) { mbar_init(v_full(s), fill_count); mbar_init(v_empty(s), 1); }
        if (F8) {
            for (int s = 0; s < kNK; ++s) mbar_init(kc_full(s), 1);
            for (int s = 0; s < kNV; ++s) mbar_init(vc_full(s), 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(s_full(g), 1);
            mbar_init(p_full(g), 128);
            mbar_init(o_done(g), 1);
            mbar_init(o_free(g), 128);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int32_t total_items = (*a.num_units) * slots_per_unit;
    // Item of this CTA in round r: the longest-first list is dealt out in snake
    // order (forward on even rounds, backward on odd ones), which balances the
    // per-CTA totals far better than plain round robin, with no atomics.
    auto item_of_round = [&](int32_t r) -> int32_t {
        return r * (int32_t)gridDim.x + ((r & 1) ? (int32_t)(gridDim.x - 1 - blockIdx.x) : (int32_t)blockIdx.x);
    };
    // Registers: the launch gives 168 per thread (384 threads); the producer /
    // MMA / converter warpgroup gives back to 104 so the softmax warpgroups can
    // hold a full 128-column score row and the 64 packed P words of the max-free
    // path (200): 128 x 104 + 256 x 200 = 384 x 168. setmaxnreg sits at the top
    // of each warpgroup's branch so that each role's code is compiled against its
    // own register limit.

    if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 104;");
    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop: lane p owns page p of every key tile. It
        // reads that page's block-table entry (all lanes in parallel, before the
        // stage is free, so the table read overlaps the wait) and issues that
        // page's TMA boxes for K and then V.
        uint32_t kt = 0, vt = 0, c = 0;
        const int32_t oob = (int32_t)(a.num_blocks * bs);  // a row past the cache: zero fill
        const int pages = kBlockN / bs;
        bool ok = true;
        for (int32_t round = 0; ok; ++round) {
            const int32_t idx = item_of_round(round);
            if (idx >= total_items) break;
            const Item it = decode_item(a.units, idx, slots_per_unit, dual, G, a.rows, a.num_rows, bs);
            if (it.n_tiles == 0) continue;
            if (c > 0 && !(ok = mbar_wait_warp(q_empty, (c - 1) & 1, abort_flag))) break;
            if (lane == 0) {
                const uint32_t qbar = F8 ? qc_full : q_full;
                mbar_arrive_expect_tx(qbar, it.nslots * C::kTileBytes);
                for (int g = 0; g < it.nslots; ++g)
                    for (int h = 0; h < C::kHalves; ++h)
                        tma_load_3d(sbase + C::kQ + g * C::kTileBytes + h * C::kHalfBytes, &tm_q,
                                    qbar, h * 64, it.h0 + g, it.q_tok0);
            }
            const int32_t* table = a.block_table + (size_t)it.req * a.max_blocks;
            for (int32_t j = 0; j < it.n_tiles && ok; ++j) {
                // this lane's page -> first cache row of the page; pages past k_end (and
                // bad ids) map to a row past the cache, which TMA fills with zeros
                int32_t y = oob;
                const int32_t k = it.kb + j * kBlockN + lane * bs;
                if (lane < pages && k < it.k_end) {
                    const int32_t pg = k / bs;
                    const int32_t id = pg < a.max_blocks ? __ldg(table + pg) : -1;
                    if (id >= 0 && id < a.num_blocks) y = id * bs;
                    else report_status(a.status, PCP_ERR_RANGE);
                }
                const int ks = kt % kNK;
                if (!(ok = mbar_wait_warp(k_empty(ks), ((kt / kNK) & 1) ^ 1, abort_flag))) break;
                if constexpr (F8) {
                    // codes: one box of bs rows x D bytes per page (D = 128: 128-byte
                    // swizzled, the e4m3 operand itself; else for the converters)
                    const uint32_t kb = C::kE4 ? k_full(ks) : kc_full(ks);
                    if (lane == 0) mbar_arrive_expect_tx(kb, C::kCodeBytes);
                    __syncwarp();
                    if (lane < pages)
                        tma_load_3d(sbase + C::code_k(ks) + lane * bs * D, &tm_k, kb, 0, it.hk, y);
                } else {
                    // K(j) and V(j) on one barrier: wait for both stages first
                    const int vs = vt % kNV;
                    if (!(ok = mbar_wait_warp(v_empty(vs), ((vt / kNV) & 1) ^ 1, abort_flag))) break;
                    if (lane == 0) mbar_arrive_expect_tx(v_full(vs), 2 * C::kTileBytes);
                    __syncwarp();
                    if (lane < pages)
                        for (int h = 0; h < C::kHalves; ++h)
                            tma_load_3d(sbase + C::kK + ks * C::kTileBytes + h * C::kHalfBytes + lane * bs * 128,
                                        &tm_k, v_full(vs), h * 64, it.hk, y);
                }
                ++kt;
                const int vs = vt % kNV;
                if (!F8) {
                    if (lane < pages)
                        for (int h = 0; h < C::kHalves; ++h)
                            tma_load_3d(sbase + C::kV + vs * C::kTileBytes + h * C::kHalfBytes + lane * bs * 128,
                                        &tm_v, v_full(vs), h * 64, it.hk, y);
                    ++vt;
                    continue;
                }
                if (!(ok = mbar_wait_warp(v_empty(vs), ((vt / kNV) & 1) ^ 1, abort_flag))) break;
                if (lane == 0) mbar_arrive_expect_tx(vc_full(vs), C::kCodeBytes);
                __syncwarp();
                if (lane < pages)
                    tma_load_3d(sbase + C::code_v(vs) + lane * bs * D, &tm_v, vc_full(vs), 0, it.hk, y);
                ++vt;
            }
            ++c;
        }
        if (!ok && lane == 0) report_status(a.status, PCP_ERR_TIMEOUT);
    } else if (F8 && warp >= kConvWarp0) {
        // ------------------------------------------------------------ FP8 converters
        // Same walk over items and tiles as the producer: per K (then V) stage wait
        // for the codes, convert them to bf16 in place, make the generic-proxy
        // stores visible to the tensor cores' async proxy, then mark the stage full.
        const int ct = threadIdx.x - kConvWarp0 * 32;
        uint32_t kt = 0, vt = 0, cq = 0;
        bool ok = true;
        for (int32_t round = 0; ok; ++round) {
            const int32_t idx = item_of_round(round);
            if (idx >= total_items) break;
            const Item it = decode_item(a.units, idx, slots_per_unit, dual, G, a.rows, a.num_rows, bs);
            if (it.n_tiles == 0) continue;
            // the item's Q tiles: bf16 -> f16 in place, then ready for the MMAs
            // (D = 128: the softmax threads write each row's e4m3 terms instead)
            if constexpr (!C::kE4) {
                if (!(ok = mbar_wait_warp(qc_full, cq & 1, abort_flag))) break;
                ++cq;
                if (__any_sync(0xffffffffu, convert_q_f16(smem + C::kQ, it.nslots * C::kTileBytes, ct)) && lane == 0)
                    report_status(a.status, PCP_ERR_RANGE);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(q_full);
            }
            for (int32_t j = 0; j < it.n_tiles && ok; ++j) {
                if constexpr (!C::kE4) {
                    const int ks = kt % kNK;
                    if (!(ok = mbar_wait_warp(kc_full(ks), (kt / kNK) & 1, abort_flag))) break;
                    convert_codes<D>(smem + C::code_k(ks), smem + C::kK + ks * C::kTileBytes, ct);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(k_full(ks));
                    ++kt;
                }
                const int vs = vt % kNV;
                if (!(ok = mbar_wait_warp(vc_full(vs), (vt / kNV) & 1, abort_flag))) break;
                convert_codes<D>(smem + C::code_v(vs), smem + C::kV + vs * C::kTileBytes, ct);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(v_full(vs));
                ++vt;
            }
        }
        if (!ok && lane == 0) report_status(a.status, PCP_ERR_TIMEOUT);
    } else if (warp == kMmaWarp && lane == 0) {
        // ------------------------------------------------------------ MMA issuer
        // Lane 0 alone runs this role, in a fixed order that staggers the two
        // heads (S0 S1 | PV0 S0' PV1 S1' | ...) so each softmax warpgroup works
        // while the other head's MMAs run. Measured on GB300: the same pattern run
        // warp-wide (every lane waiting, a vote and a reconvergence around each
        // batch) holds the tensor pipe to ~89 cycles per 128x128x16 MMA against
        // ~70 from a single thread; one issuer thread per head (independent
        // order) ran 11% slower end to end, the heads' softmaxes falling into
        // step. The other lanes only take part in the TMEM allocation and release.
        uint32_t kt = 0, vt = 0, c = 0;
        uint32_t pph[2] = {0, 0}, nslot_items[2] = {0, 0};
        bool ok = true;
        // shared-memory descriptors of the first k-step of every Q, K and V tile
        auto q_desc = [&](int g) { return sdesc_sw128(sbase + C::kQ + g * C::kTileBytes, 16, 1024); };
        auto k_desc = [&](int s2) { return sdesc_sw128(sbase + C::kK + s2 * C::kTileBytes, 16, 1024); };
        auto v_desc = [&](int s2) { return sdesc_sw128(sbase + C::kV + s2 * C::kTileBytes, C::kHalfBytes, 1024); };
        const uint64_t qd0 = q_desc(0), qd1 = q_desc(1);
        for (int32_t round = 0; ok; ++round) {
            const int32_t idx = item_of_round(round);
            if (idx >= total_items) break;
            const Item it = decode_item(a.units, idx, slots_per_unit, dual, G, a.rows, a.num_rows, bs);
            const int n = it.n_tiles;
            if (n == 0) continue;
            if (!(ok = mbar_wait(q_full, c & 1, abort_flag))) break;
            int ks = kt % kNK;
            // K(0) (bf16: with V(0))
            if (!(ok = kMerged ? mbar_wait(v_full(vt % kNV), (vt / kNV) & 1, abort_flag)
                               : mbar_wait(k_full(ks), (kt / kNK) & 1, abort_flag)))
                break;
            tc_fence_after();
            for (int g = 0; g < it.nslots; ++g) {
                issue_qk<D, F8>(tmem + C::tmem_s(g), g ? qd1 : qd0, k_desc(ks));
                mma_commit(s_full(g));
            }
            ++kt;
            for (int j = 0; j < n && ok; ++j) {
                const int vs = vt % kNV;
                if (!kMerged && !(ok = mbar_wait(v_full(vs), (vt / kNV) & 1, abort_flag))) break;
                if (j == n - 1 && (it.k_end % bs) != 0) {
                    // Keys at or past k_end inside the last loaded page may never have been
                    // written: zero their V rows so that P = 0 cannot meet a NaN.
                    const int32_t rel = it.k_end - (it.kb + j * kBlockN);
                    const int32_t r1 = ((rel + bs - 1) / bs) * bs;
                    const int nbytes = (r1 - rel) * 128;
                    for (int h = 0; h < C::kHalves; ++h) {
                        uint8_t* base = smem + C::kV + vs * C::kTileBytes + h * C::kHalfBytes + rel * 128;
                        for (int off = 0; off < nbytes; off += 16)
                            *reinterpret_cast<uint4*>(base + off) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                for (int g = 0; g < it.nslots && ok; ++g) {
                    // O += P V once the softmax has written P
                    if (!(ok = mbar_wait(p_full(g), pph[g], abort_flag))) break;
                    if (j == 0 && nslot_items[g] > 0) {
                        if (!(ok = mbar_wait(o_free(g), (nslot_items[g] - 1) & 1, abort_flag))) break;
                    }
                    tc_fence_after();
                    pph[g] ^= 1;
                    issue_pv<D, F8>(tmem + C::tmem_o(g), tmem + C::tmem_s(g), v_desc(vs), j > 0);
                    if (j + 1 < n) {
                        if (g == 0) {
                            // K(j + 1) (bf16: with V(j + 1))
                            ks = kt % kNK;
                            if (!(ok = kMerged ? mbar_wait(v_full((vt + 1) % kNV), ((vt + 1) / kNV) & 1, abort_flag)
                                               : mbar_wait(k_full(ks), (kt / kNK) & 1, abort_flag)))
                                break;
                            tc_fence_after();
                        }
                        issue_qk<D, F8>(tmem + C::tmem_s(g), g ? qd1 : qd0, k_desc(ks));
                        mma_commit(s_full(g));
                        if (g == it.nslots - 1) ++kt;
                    } else {
                        mma_commit(o_done(g));
                    }
                }
                ++vt;
            }
            for (int g = 0; g < it.nslots; ++g) ++nslot_items[g];
            ++c;
        }
        if (!ok) report_status(a.status, PCP_ERR_TIMEOUT);
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
        // ------------------------------------------------------------ softmax
        const int g = warp / 4;                 // head slot of this warpgroup
        const int r = threadIdx.x % 128;        // query row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp % 4) * 32) << 16;
        const uint32_t t_s = tmem + lane_base + C::tmem_s(g);
        const uint32_t t_o = tmem + lane_base + C::tmem_o(g);
        uint32_t sph = 0, oph = 0;
        // The warpgroup of the last head slot releases the shared stages: S of tile j
        // complete means every MMA issued before it is complete (K(j), V(j - 1) and,
        // on the last tile, Q are free); O done frees the item's last V. Its thread 0
        // arrives, so that the MMA issuer spends no commits on them.
        const bool releaser = g == slots_per_item - 1;
        uint32_t rel_k = 0, rel_v = 0, cq = 0;
        bool ok = true;
        for (int32_t round = 0; ok; ++round) {
            const int32_t idx = item_of_round(round);
            if (idx >= total_items) break;
            const Item it = decode_item(a.units, idx, slots_per_unit, dual, G, a.rows, a.num_rows, bs);
            const uint32_t my_q = cq;  // Q loads so far (items with key tiles)
            if (it.n_tiles > 0) ++cq;
            if (g >= it.nslots) continue;
            const int h = it.h0 + g;
            // FP8: the K descale scales every score (the V descale the output, below);
            // it is re-read per tile (an L1 hit) rather than held across the loop,
            // which keeps the score row within the register budget
            const float* kd_ptr = F8 ? a.k_descale + (size_t)it.req * a.hkv + it.hk : nullptr;
            const bool valid = r < it.rows_valid;
            const int32_t pos = it.pos0 + min(r, it.rows_valid - 1);
            const int32_t tok = it.q_tok0 + r;
            float m = -INFINITY, l = 0.f;
            const int n = it.n_tiles;
            // FP8, D = 128: once the item's bf16 Q has landed, this thread rewrites its
            // own row as e4m3 terms (the softmax warps are idle until the item's first S)
            // and keeps the row's q scale
            float qs_row = 1.f;
            if constexpr (C::kE4) {
                if (n > 0) {
                    if (!(ok = mbar_wait_warp(qc_full, my_q & 1, abort_flag))) break;
                    bool over = false;
                    qs_row = q_row_to_e4m3(smem + C::kQ + g * C::kTileBytes, r, &over);
                    if (over) report_status(a.status, PCP_ERR_RANGE);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if ((threadIdx.x & 31) == 0) mbar_arrive(q_full);
                }
            }
            for (int j = 0; j < n && ok; ++j) {
                if (!(ok = mbar_wait_warp(s_full(g), sph, abort_flag))) break;
                sph ^= 1;
                if (releaser) {
                    if (r == 0) {
                        mbar_arrive(k_empty(rel_k % kNK));
                        if (j > 0) mbar_arrive(v_empty(rel_v % kNV));
                    }
                    ++rel_k;
                    if (j > 0) ++rel_v;
                }
                if (j == n - 1 && (releaser || dual) && r == 0) mbar_arrive(q_empty);
                tc_fence_after();
                uint32_t s[128];
                float* sf = reinterpret_cast<float*>(s);
                const float sl2 = F8 ? a.scale * __ldg(kd_ptr) * kLog2e * qs_row : a.scale * kLog2e;
                const int32_t key0 = it.kb + j * kBlockN;
                const bool full = key0 >= it.k_lo && key0 + kBlockN <= it.k_hi &&
                                  key0 + kBlockN - 1 <= it.pos0;
                // S row of this thread into registers, keys outside [k_lo, min(k_hi, pos + 1)) at -inf
                auto load_scores = [&]() {
                    tmem_ld32(t_s + 0, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
                    tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                    tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
                    tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
                    tmem_wait_ld();
                    if (!full) {
                        const int32_t lo = it.k_lo - key0;
                        const int32_t hi = min(it.k_hi, pos + 1) - key0;
#pragma unroll
                        for (int c2 = 0; c2 < 128; ++c2)
                            if (c2 < lo || c2 >= hi) sf[c2] = -INFINITY;
                    }
                };
                // p of a pair: ex2, or (polynomial knob) the FMA-pipe exp2 for every
                // kPolyEvery-th pair (a masked key then gets ~1e-38, not 0)
                auto exp_pair = [&](float2 x, int c2) -> float2 {
                    if (c2 % kPolyEvery == kPolyEvery - 1) return exp2_poly2(x);
                    return make_float2(fast_exp2(x.x), fast_exp2(x.y));
                };
                load_scores();
                // Fast path: every row of the warp already has a finite reference max m;
                // p = 2^(s * scale * log2 e - m) straight away, no row max first. With a
                // bf16 cache, P of keys 0-63 goes to TMEM as soon as it is computed, so
                // that store overlaps the second half's exponentials (measured: prefill
                // 0.9 % faster). If a row's tile sum reaches 2^64 (its scores rose by ~64
                // in log2 units) the warp takes the exact path: the scores of keys 0-31
                // (whose columns P has overwritten) from registers, the rest from S again.
                bool exact = true;
                if (kMaxFree && __all_sync(0xffffffffu, m != -INFINITY)) {
                    const float2 sl2v = make_float2(sl2, sl2), nmu = make_float2(-m, -m);
                    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                     make_float2(0.f, 0.f)};
                    uint32_t p[64];
#pragma unroll
                    for (int c2 = 0; c2 < 64; ++c2) {
                        const float2 e = exp_pair(ffma2(make_float2(sf[2 * c2], sf[2 * c2 + 1]), sl2v, nmu), c2);
                        acc[c2 % 4] = fadd2(acc[c2 % 4], e);
                        p[c2] = F8 ? pack_f16x2(e.x, e.y) : pack_bf16x2(e.x, e.y);
                        if (!F8 && c2 == 31) tmem_st32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                    }
                    const float2 a03 = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
                    const float ts = a03.x + a03.y;
                    // f16 P (FP8 cache) must stay below 65504: a lower limit there
                    if (!__any_sync(0xffffffffu, !(ts < (F8 ? 32768.0f : kMaxFreeLimit)))) {
                        if (F8) tmem_st32(t_s, *reinterpret_cast<uint32_t(*)[32]>(&p[0]));
                        tmem_st32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&p[32]));
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(p_full(g));
                        l += ts;
                        exact = false;
                    } else if (F8) {
                        load_scores();
                    } else {
                        // columns 0-31 now hold P of keys 0-63; the scores of keys 0-31 are
                        // still in registers, those of keys 32-127 in columns 32-127
                        tmem_wait_st();
                        tmem_ld32(t_s + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
                        tmem_ld32(t_s + 64, *reinterpret_cast<uint32_t(*)[32]>(&s[64]));
                        tmem_ld32(t_s + 96, *reinterpret_cast<uint32_t(*)[32]>(&s[96]));
                        tmem_wait_ld();
                        if (!full) {
                            const int32_t lo = it.k_lo - key0;
                            const int32_t hi = min(it.k_hi, pos + 1) - key0;
#pragma unroll
                            for (int c2 = 32; c2 < 128; ++c2)
                                if (c2 < lo || c2 >= hi) sf[c2] = -INFINITY;
                        }
                    }
                }
                if (!exact) continue;
                // row max: eight independent chains of three-input maxima
                float part[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float t = sf[16 * i];
#pragma unroll
                    for (int k2 = 1; k2 < 15; k2 += 2) t = fmax3(t, sf[16 * i + k2], sf[16 * i + k2 + 1]);
                    part[i] = fmaxf(t, sf[16 * i + 15]);
                }
                const float mx = fmax3(fmax3(part[0], part[1], part[2]), fmax3(part[3], part[4], part[5]),
                                       fmaxf(part[6], part[7]));
                const float m_new = fmaxf(m, mx * sl2);
                // Lazy rescaling: keep the old reference max unless the new one exceeds
                // it by more than 2^8; O and l then stay consistent with that max.
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m = m_new;
                } else {
                    const bool need = m_new > m + kRescaleThreshold;
                    rescale = __any_sync(0xffffffffu, need);
                    if (need) {
                        alpha = fast_exp2(m - m_new);
                        l *= alpha;
                        m = m_new;
                    }
                }
                const float mu = (m == -INFINITY) ? 0.f : m;
                // O must be rescaled before the first half of this tile's PV runs (16
                // columns at a time: the score row is still live in registers)
                if (rescale) {
#pragma unroll 1
                    for (int c2 = 0; c2 < D / 16; ++c2) {
                        uint32_t o[16];
                        tmem_ld16(t_o + 16 * c2, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st16(t_o + 16 * c2, o);
                    }
                }
                // Exact path: p = 2^(s * scale * log2 e - m) with m this row's lazily
                // updated max, two lanes per instruction; P goes back to TMEM in two
                // halves (keys 0-63, then 64-127).
                const float2 sl2v = make_float2(sl2, sl2), nmu = make_float2(-mu, -mu);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t p[32];
#pragma unroll
                    for (int c3 = 0; c3 < 32; ++c3) {
                        const int c2 = half * 32 + c3;
                        const float2 e = exp_pair(ffma2(make_float2(sf[2 * c2], sf[2 * c2 + 1]), sl2v, nmu), c2);
                        acc[c2 % 4] = fadd2(acc[c2 % 4], e);
                        p[c3] = F8 ? pack_f16x2(e.x, e.y) : pack_bf16x2(e.x, e.y);
                    }
                    tmem_st32(t_s + 32 * half, p);
                    if (half == 1) {
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(p_full(g));
                    }
                }
                const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
                const float2 a03 = fadd2(a01, a23);
                l += a03.x + a03.y;
            }
            if (!ok) break;
            // ---- epilogue: out = O / l, lse = ln 2 * (m + log2 l)
            const bool has = l > 0.f;
            const float vd = F8 ? __ldg(a.v_descale + (size_t)it.req * a.hkv + it.hk) : 1.f;
            const float inv = has ? vd / l : 0.f;
            const float lse_v = has ? (m + __log2f(l)) * kLn2 : -INFINITY;
            if (n > 0) {
                if (!(ok = mbar_wait_warp(o_done(g), oph, abort_flag))) break;
                oph ^= 1;
                if (releaser) {
                    if (r == 0) mbar_arrive(v_empty(rel_v % kNV));
                    ++rel_v;
                }
                tc_fence_after();
            }
            const size_t orow = ((size_t)tok * a.hq + h) * D;
            // the whole O row into registers first, so the accumulator can be handed
            // back to the MMA warp (next item) before the global stores
            uint32_t orow_regs[D];
            if (n > 0) {
#pragma unroll
                for (int c2 = 0; c2 < D / 32; ++c2)
                    tmem_ld32(t_o + 32 * c2, *reinterpret_cast<uint32_t(*)[32]>(&orow_regs[32 * c2]));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(o_free(g));
            } else {
#pragma unroll
                for (int e = 0; e < D; ++e) orow_regs[e] = 0u;
            }
#pragma unroll
            for (int c2 = 0; c2 < D / 32; ++c2) {
                const uint32_t* o = &orow_regs[32 * c2];
                if (valid) {
                    if (it.pass == 0) {
                        uint4* dst = reinterpret_cast<uint4*>(
                            reinterpret_cast<__nv_bfloat16*>(a.out) + orow + 32 * c2);
#pragma unroll
                        for (int v4 = 0; v4 < 4; ++v4) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
                            dst[v4] = w;
                        }
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            a.part_out + (size_t)(it.pass - 1) * a.total_q * a.hq * D + orow + 32 * c2);
#pragma unroll
                        for (int v4 = 0; v4 < 8; ++v4)
                            dst[v4] = make_float4(__uint_as_float(o[4 * v4 + 0]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                                  __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
                    }
                }
            }
            if (valid) {
                float* lse_dst = it.pass == 0 ? a.lse : a.part_lse + (size_t)(it.pass - 1) * a.hq * a.total_q;
                lse_dst[(size_t)h * a.total_q + tok] = lse_v;
            }
        }
        if (!ok) report_status(a.status, PCP_ERR_TIMEOUT);
    }

    __syncwarp();  // lane 0 of the producer and of the MMA warp worked alone: reconverge first
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------ scheduler

constexpr int kSchedThreads = 1024;
// Lists of up to kSortCap units are sorted exactly (bitonic, in shared memory);
// longer ones by a counting sort over kCostBuckets cost classes (costs of
// kCostBuckets - 1 key tiles or more share the first class).
constexpr int kSortCap = 4096;
constexpr int kCostBuckets = 2 * kSortCap;  // int32 counters in the same 32 KB as the sort keys

__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* warp_sums, int32_t* total) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < kSchedThreads / 32 ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const int32_t before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[kSchedThreads / 32 - 1];
    __syncthreads();
    return before;
}

// Key tiles a unit's item walks (its cost in the schedule).
__device__ __forceinline__ int32_t unit_cost(const Unit& u, const pcp_row_t* rows, int32_t bs) {
    const pcp_row_t row = rows[u.row];
    const int32_t mt = u.mt_pass & 0xFFFFFF;
    const int32_t pos0 = row.kv_end - row.q_len + mt * kBlockM;
    const int32_t rv = min(kBlockM, row.q_len - mt * kBlockM);
    return tiles_of(u.k_lo, min(u.k_hi, pos0 + rv), bs);
}

// Partial last splits of decode rows, bucketed by their 128-key tiles (1 .. 16).
constexpr int kTailBuckets = kDecodeChunk / kBlockN;

// Check every row, then build the prefill work list: one unit per (valid
// non-decode row, 128-token tile, pass), ordered by the number of key tiles,
// longest first. Also lays out the decode work items (kv head x kDecodeChunk-key
// split of each valid decode row), full splits first and partial last splits
// after them, longest first: dec_pre[i] = full-split items of the rows before
// row i (dec_pre[num_rows]: all of them), dec_pre[num_rows + 1 + t] = the t-th
// row with a partial last split, header[1] = the number of items.
__global__ void __launch_bounds__(kSchedThreads, 1)
    schedule_kernel(PrefillArgs a, int32_t flags, Unit* units, Unit* sorted, int32_t* header,
                    int32_t* row_ok, int32_t* dec_pre, int64_t max_units) {
    __shared__ int32_t warp_sums[32];
    // decode rows with a partial last split per bucket, their first list
    // position, and the positions taken so far
    __shared__ int32_t tail_cnt[kTailBuckets + 1], tail_off[kTailBuckets + 1], tail_fill[kTailBuckets + 1];
    if (threadIdx.x <= kTailBuckets) {
        tail_cnt[threadIdx.x] = 0;
        tail_fill[threadIdx.x] = 0;
    }
    __syncthreads();
    // bitonic sort keys, or the counters of the counting sort
    __shared__ __align__(16) unsigned long long keys[kSortCap];
    const pcp_row_t* rows = a.rows;
    const int32_t num_rows = a.num_rows, bs = a.block_size;
    const int64_t max_kv = (int64_t)a.max_blocks * bs;
    const bool separate = (flags & PCP_ATTN_SEPARATE_CONTEXT) != 0;
    const bool at_row_start = (flags & PCP_ATTN_SPLIT_AT_ROW_START) != 0;
    const int nparts = a.nparts;             // 0: fused; 2: context + new; n: n key shards
    const int passes = nparts > 0 ? nparts : 1;
    int32_t base = 0, dbase = 0;
    for (int32_t r0 = 0; r0 < num_rows; r0 += kSchedThreads) {
        const int32_t ri = r0 + threadIdx.x;
        pcp_row_t row{};
        int32_t cnt = 0, dcnt = 0;
        if (ri < num_rows) {
            row = rows[ri];
            const bool ok = row.req >= 0 && row.req < a.num_reqs && row.q_len >= 1 && row.q_start >= 0 &&
                            (int64_t)row.q_start + row.q_len <= a.total_q && row.kv_end >= row.q_len &&
                            row.kv_end <= max_kv && row.ctx_len >= 0 && row.ctx_len <= row.kv_end &&
                            (row.is_decode == 0 || (row.is_decode == 1 && row.q_len == 1));
            row_ok[ri] = ok ? 1 : 0;
            if (!ok) report_status(a.status, PCP_ERR_RANGE);
            if (ok && !row.is_decode) cnt = ((row.q_len + kBlockM - 1) / kBlockM) * passes;
            if (ok && row.is_decode) {
                dcnt = (row.kv_end / kDecodeChunk) * a.hkv;
                const int32_t part = row.kv_end % kDecodeChunk;
                if (part) atomicAdd(&tail_cnt[(part + kBlockN - 1) / kBlockN], 1);
            }
        }
        int32_t dtot;
        const int32_t doff = dbase + block_exclusive_scan(dcnt, warp_sums, &dtot);
        if (ri < num_rows) dec_pre[ri] = doff;
        dbase += dtot;
        int32_t tot;
        const int32_t off = base + block_exclusive_scan(cnt, warp_sums, &tot);
        for (int32_t u = 0; u < cnt; ++u) {
            if (off + u >= max_units) break;
            const int32_t mt = u / passes, pass = nparts > 0 ? 1 + u % passes : 0;
            Unit x;
            x.row = ri;
            x.mt_pass = mt | (pass << 24);
            if (separate) {  // context [0, split) and new tokens [split, kv_end)
                const int32_t split = at_row_start ? row.kv_end - row.q_len : row.ctx_len;
                x.k_lo = pass == 2 ? split : 0;
                x.k_hi = pass == 1 ? split : row.kv_end;
            } else if (nparts > 0) {  // key shard pass - 1 of nparts: contiguous, floor bounds
                x.k_lo = (int32_t)((int64_t)row.kv_end * (pass - 1) / nparts);
                x.k_hi = (int32_t)((int64_t)row.kv_end * pass / nparts);
            } else {
                x.k_lo = 0;
                x.k_hi = row.kv_end;
            }
            units[off + u] = x;
        }
        base += tot;
    }
    const int32_t n = (int32_t)min((int64_t)base, max_units);
    __syncthreads();  // tail counts complete
    if (threadIdx.x == 0) {
        int32_t t = 0;
        for (int b = kTailBuckets; b >= 1; --b) {
            tail_off[b] = t;
            t += tail_cnt[b];
        }
        header[0] = n;
        header[1] = dbase + t * a.hkv;
        dec_pre[num_rows] = dbase;
    }
    __syncthreads();
    // the rows with a partial last split, longest first (any order within a
    // bucket: every item writes only its own partial, so the order changes no result)
    for (int32_t ri = threadIdx.x; ri < num_rows; ri += kSchedThreads) {
        if (!row_ok[ri]) continue;
        const pcp_row_t row = rows[ri];
        const int32_t part = row.kv_end % kDecodeChunk;
        if (!row.is_decode || !part) continue;
        const int b = (part + kBlockN - 1) / kBlockN;
        dec_pre[num_rows + 1 + tail_off[b] + atomicAdd(&tail_fill[b], 1)] = ri;
    }
    // every thread's units[] writes must be visible before any thread reads them
    __syncthreads();
    if (n > kSortCap) {
        // Counting sort, longest first: class c = kCostBuckets - 1 - min(cost,
        // kCostBuckets - 1); count, exclusive scan, scatter. Units of one class
        // land in any order (every item writes only its own outputs, so the
        // order changes no result).
        int32_t* cnt = reinterpret_cast<int32_t*>(keys);
        for (int32_t i = threadIdx.x; i < kCostBuckets; i += kSchedThreads) cnt[i] = 0;
        __syncthreads();
        for (int32_t i = threadIdx.x; i < n; i += kSchedThreads) {
            const int32_t c = kCostBuckets - 1 - min(unit_cost(units[i], rows, bs), kCostBuckets - 1);
            atomicAdd(&cnt[c], 1);
        }
        __syncthreads();
        constexpr int kPer = kCostBuckets / kSchedThreads;  // consecutive classes per thread
        int32_t local[kPer], sum = 0;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            local[k] = cnt[threadIdx.x * kPer + k];
            sum += local[k];
        }
        int32_t tot;
        int32_t run = block_exclusive_scan(sum, warp_sums, &tot);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            cnt[threadIdx.x * kPer + k] = run;
            run += local[k];
        }
        __syncthreads();
        for (int32_t i = threadIdx.x; i < n; i += kSchedThreads) {
            const Unit u = units[i];
            const int32_t c = kCostBuckets - 1 - min(unit_cost(u, rows, bs), kCostBuckets - 1);
            sorted[atomicAdd(&cnt[c], 1)] = u;
        }
        return;
    }
    int32_t pow2 = 1;
    while (pow2 < n) pow2 <<= 1;
    for (int32_t i = threadIdx.x; i < pow2; i += kSchedThreads) {
        unsigned long long key = ~0ull;
        if (i < n) {
            const int32_t cost = unit_cost(units[i], rows, bs);
            key = ((unsigned long long)(0x7FFFFFFF - cost) << 32) | (unsigned)i;
        }
        keys[i] = key;
    }
    __syncthreads();
    for (int32_t k = 2; k <= pow2; k <<= 1) {
        for (int32_t jj = k >> 1; jj > 0; jj >>= 1) {
            for (int32_t i = threadIdx.x; i < pow2; i += kSchedThreads) {
                const int32_t l = i ^ jj;
                if (l > i) {
                    const unsigned long long x = keys[i], y = keys[l];
                    const bool up = (i & k) == 0;
                    if ((x > y) == up) { keys[i] = y; keys[l] = x; }
                }
            }
            __syncthreads();
        }
    }
    for (int32_t i = threadIdx.x; i < n; i += kSchedThreads) sorted[i] = units[(int32_t)(keys[i] & 0xFFFFFFFFu)];
}

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// 3-D bf16 view [outer][mid][D] with a box of {64, 1, rows}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int D, int64_t mid, int64_t outer, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)mid, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)(D * 2 * mid)};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D view [outer][mid][D] of a cache with elements of esize bytes (1: FP8 codes,
// 2: bf16) and a box of {D, 1, rows}, no swizzle: a box row is one head's D
// contiguous elements (64 to 256 bytes).
bool make_row_map(CUtensorMap* m, const void* base, int D, int esize, int64_t mid, int64_t outer, int rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)mid, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)(D * esize * mid)};
    cuuint32_t box[3] = {(cuuint32_t)D, 1, (cuuint32_t)rows};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, bool F8>
int launch_prefill_d(const PrefillArgs& a, cudaStream_t stream, int grid) {
    CUtensorMap tq, tk, tv;
    const int64_t slots = a.num_blocks * a.block_size;
    // FP8: K codes 128-byte swizzled where they are the MMA operand (D = 128)
    const bool maps = F8 ? (Cfg<D, F8>::kE4 ? make_box_map(&tk, a.key_cache, D, 1, a.hkv, slots, D, 1, a.block_size, true)
                                            : make_row_map(&tk, a.key_cache, D, 1, a.hkv, slots, a.block_size)) &&
                               make_row_map(&tv, a.value_cache, D, 1, a.hkv, slots, a.block_size)
                         : make_map(&tk, a.key_cache, D, a.hkv, slots, a.block_size) &&
                               make_map(&tv, a.value_cache, D, a.hkv, slots, a.block_size);
    if (!maps || !make_map(&tq, a.q, D, a.hq, a.total_q, kBlockM)) return PCP_ERR_CUDA;
    const int smem = Cfg<D, F8>::kSmem;
    cudaError_t e =
        cudaFuncSetAttribute(prefill_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    // persistent: the work list is dealt over however many CTAs run (fewer when
    // the decode rows take some SMs beside it)
    const int ctas = grid > 0 && grid < num_sms() ? grid : num_sms();
    prefill_kernel<D, F8><<<ctas, kThreads, smem, stream>>>(tq, tk, tv, a);
    e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

}  // namespace

int launch_schedule(const PrefillArgs& a, int32_t flags, Unit* units, Unit* units_sorted,
                    int32_t* header, int32_t* row_ok, int32_t* dec_pre, int64_t max_units,
                    cudaStream_t stream) {
    schedule_kernel<<<1, kSchedThreads, 0, stream>>>(a, flags, units, units_sorted, header, row_ok,
                                                     dec_pre, max_units);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

int launch_prefill(const PrefillArgs& a, cudaStream_t stream, int grid) {
    const bool f8 = a.k_descale != nullptr;
    if (a.d == 64)
        return f8 ? launch_prefill_d<64, true>(a, stream, grid) : launch_prefill_d<64, false>(a, stream, grid);
    if (a.d == 128)
        return f8 ? launch_prefill_d<128, true>(a, stream, grid) : launch_prefill_d<128, false>(a, stream, grid);
    return PCP_ERR_UNSUPPORTED;
}

bool make_kv_row_map(CUtensorMap* m, const void* base, int D, int esize, int64_t mid, int64_t outer, int rows) {
    return make_row_map(m, base, D, esize, mid, outer, rows);
}

bool make_box_map(CUtensorMap* m, const void* base, int D, int esize, int64_t mid, int64_t outer, int box_x,
                  int box_mid, int box_outer, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)mid, (cuuint64_t)outer};
    cuuint64_t strides[2] = {(cuuint64_t)D * esize, (cuuint64_t)(D * esize * mid)};
    cuuint32_t box[3] = {(cuuint32_t)box_x, (cuuint32_t)box_mid, (cuuint32_t)box_outer};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = esize == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace pcp
