// Decode rows of a mixed PCP batch on the 5th-generation tensor cores: one new
// token attending all keys [0, C) of its request ("[MRv2] FlashAttention PCP
// support for GQA on MRv2", overview: mixed-batch decode handled next to the
// prefill rows; "[MRv2][PCP] Carry the row plan ...", "drop pcp_has_prefill":
// decode rows carried in the same plan).
//
// A decode row has one query token, so the q heads of one kv head (G <= 16;
// FP8: G <= 8) are the only other dimension an MMA can take: the kernel
// computes the transposed products, keys along M:
//   S^T [128 keys x 16] = K [128 keys x D] . Q^T      (Q^T: the G q heads, padded to 16 rows)
//   O^T [D x 16]        = V^T [D x 128 keys] . P^T    (P^T: 16 rows, P in rows 0..7 and the
//                                                      rounding remainder of P in rows 8..15;
//                                                      G > 8: 32 rows, 0..15 and 16..31)
// Over an FP8 cache S^T takes the e4m3 codes of K as they are (kind::f8f6f4,
// 32 dims per MMA) against q written as two e4m3 terms per element after a
// power-of-two scaling per head, whose sum is the bf16 q (term t of head h in
// column t * GP + h).
// The bytes of K and V, read once, set the speed; the tensor cores do the
// products so that the few instructions per key left are the softmax's.
//
// Design (sm_103a, head_dim 128, one CTA per SM, persistent):
//  * work item = (decode row, kv head, split of kDecodeChunk keys); the
//    scheduler kernel lists the full splits first and the partial last splits
//    after them, longest first (dec_pre), and the CTAs take items in snake
//    order; partial (out, lse) per split as the CUDA-core decode kernel writes
//    them, merged by decode_merge_kernel;
//  * warps 8 (K) and 9 (V) produce: per item the block-table entries of its
//    keys, then per 128-key tile one TMA box per page (bf16: two 64-dim halves,
//    128-byte swizzled; FP8: the codes, D bytes per row, into the upper half of
//    the tile), into rings of 3 K and 3 V tiles that run on across items; warp 8 also
//    loads each item's Q^T (16 q heads of the token from head hk * G, rows past
//    Hq zero filled);
//  * lane 0 of warp 10 issues every S^T (once K(g) is in and P(g - 2) has left
//    its S buffer), lane 0 of warp 11 every O^T (once P(g) is written); one
//    thread cannot issue the 16 small MMAs of a tile fast enough. Commits free
//    the K stage (after S), the V stage (after PV) and the S and O buffers;
//  * warps 0-3 and 4-7 are two softmax warpgroups taking alternate tiles, one
//    thread per key of the tile (TMEM lane) and per dim of O^T: scores -> tile
//    max per head (a reduce-scatter over the warp, then the warpgroup's four
//    warps through a named barrier) -> exact online softmax -> P = hi + lo
//    rounded to 16 bits into shared memory (P^T rows h and 8 + h; the
//    remainder keeps P's rounding out of the result); each finished tile's O^T
//    is added into registers with the running rescale; at the end of an item
//    the split's partial is written: bf16 up to 8 heads, warpgroup 0 merges the
//    two warpgroups' (max, l, O); FP8 and 16 heads, each warpgroup writes its
//    own partial (two per split, merged by decode_merge_kernel) and never waits
//    for the other;
//  * FP8 cache: the K codes land 128-byte swizzled and are the S operand; the
//    converter warps (two sets taking alternate tiles where G <= 4, else one)
//    widen each V tile's codes to f16 in place (exact; rows past the last key
//    written as zeros) for the f16 PV, and set 0 turns each item's q into its
//    e4m3 terms and per-head scales; the K descale and the q scale multiply
//    the scores, the V descale the partial;
//  * bf16 cache: V rows past a split's last key (unwritten cache slots, or a
//    stale stage) are zeroed by the softmax threads before the last PV;
//  * every wait is bounded (PCP_ERR_TIMEOUT); after a timeout the producer
//    waits, again bounded, for the copies it issued before the CTA exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pcp_device.cuh"
#include "pcp_internal.h"

namespace pcp {

namespace {

constexpr int kD = 128;          // head_dim this kernel takes
constexpr int kKeys = 128;       // keys per tile: the M of S^T
constexpr int kN = 16;           // the N of S^T (and of O^T up to 8 q heads per kv head)
constexpr int kMaxG = 16;        // q heads per kv head (FP8: 8)
constexpr int kTerms = 2;        // FP8: e4m3 terms per q element (their sum is the bf16 q exactly)
constexpr int kProdWarp = 8;     // warp 8: K tiles and Q^T; warp 9: V tiles
constexpr int kMmaWarp = 10;     // lane 0 issues the S MMAs (the warp owns the TMEM allocation)
constexpr int kPvWarp = 11;      // lane 0 issues the PV MMAs
constexpr int kConvWarp0 = 12;
constexpr int kConvThreads = 128;  // FP8: threads widening one V tile (one or two such sets)
// FP8 converter warps: two sets of four taking alternate V tiles where the
// softmax fits the registers that 20 warps leave (G <= 4), else one set
__host__ __device__ constexpr int conv_warps(bool f8, int gp) { return f8 ? (gp <= 4 ? 8 : 4) : 0; }
__host__ __device__ constexpr int tc_threads(bool f8, int gp) { return 32 * (12 + conv_warps(f8, gp)); }
constexpr int kMaxPages = kDecodeChunk / 8;  // block-table entries of one split (block_size >= 8)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <bool F8, int GP>
struct TcCfg {
    // S^T columns: the G q heads (bf16), or their kTerms e4m3 terms (FP8)
    static constexpr int kNS = 16;
    static_assert(!F8 || kTerms * GP <= kNS, "the q terms of a group fill N = 16");
    // head stride of the per-head arrays; O^T columns = P^T rows: P's hi parts in
    // rows 0 .. kGS - 1, the remainders from row kGS (N = 16, or 32 for 16 heads)
    static constexpr int kGS = GP <= 8 ? 8 : 16;
    static constexpr int kNO = 2 * kGS;
    // a partial per softmax warpgroup and split (no hand-over area): FP8, and 16
    // heads (whose hand-over area would not fit)
    static constexpr bool kSplitParts = F8 || GP > 8;
    static constexpr int kKS = F8 ? 4 : 3;                 // K tiles in flight (free after their S)
    static constexpr int kVS = (F8 && GP <= 4) ? 4 : 3;    // V tiles in flight (free after their PV)
    static constexpr int kHalfBytes = kKeys * 128;      // 128 keys x 64 dims x 2 bytes
    static constexpr int kTileBytes = 2 * kHalfBytes;   // one 16-bit K or V tile
    // FP8: a K tile is its codes, 128 keys x 128 bytes (the MMA reads them as e4m3)
    static constexpr int kKTileBytes = F8 ? kHalfBytes : kTileBytes;
    static constexpr int kRowsBytes = kN * 128;         // 16 rows x 128 bytes: one 64-element half
    static constexpr int kQBytes = 2 * kRowsBytes;      // bf16 Q^T: 16 rows x 128 dims
    static constexpr int kQCBytes = F8 ? kNS * 128 : 0;  // FP8: the e4m3 terms of Q^T, kNS rows
    static constexpr int kPBytes = 2 * kNO * 128;       // P^T: kNO rows x 128 keys
    static constexpr int kK = 0;                        // K stages
    static constexpr int kV = kKS * kKTileBytes;        // V stages
    static constexpr int kQ = kV + kVS * kTileBytes;    // two Q^T buffers (bf16)
    static constexpr int kQC = kQ + 2 * kQBytes;        // two Q^T term buffers (FP8)
    static constexpr int kP = kQC + 2 * kQCBytes;       // two P^T buffers
    static constexpr int kPre = kP + 2 * kPBytes;       // int32 [kDecTcMaxRows + 1]
    static constexpr int kPages = kPre + ((kDecTcMaxRows + 1) * 4 + 15) / 16 * 16;  // one list per producer
    static constexpr int kRed = kPages + 2 * kMaxPages * 4;  // float [2 wg][2][4][8] maxima and sums
    // bf16: warpgroup 1's max and O of an item, handed to warpgroup 0 (float [8 + 8 x 128])
    static constexpr int kXchg = kRed + (2 * 2 * 4 * kGS) * 2 * 4;
    // FP8: float [4][8] q scales, a ring of four items: the converters run at most
    // three items ahead of the softmax (they prepare item i + 3 only once S of item
    // i + 1 is done, which needs the softmax in item i at least)
    static constexpr int kQs = kXchg + (kSplitParts ? 0 : (kGS + kGS * kKeys) * 4);
    static constexpr int kBar = kQs + 4 * kGS * 4;
    static constexpr int kNumBars = 2 * kKS + 3 * kVS + 7 * 2 + 4;
    static constexpr int kMisc = kBar + kNumBars * 8;   // TMEM address, abort flag
    static constexpr int kSmem = kMisc + 16 + 1024;     // + alignment slack
    static constexpr uint32_t kTmemS = 0, kTmemO = 2 * kNS;  // S^T x 2 (kNS columns), O^T x 2 (kNO)
    static constexpr uint32_t kTmemCols = 2 * kNS + 2 * kNO <= 64 ? 64 : 128;
    static constexpr uint32_t kIdescS = F8 ? idesc_e4m3(128, kNS) : idesc_bf16(128, kN, false, false);
    static constexpr uint32_t kIdescO = F8 ? idesc_f16(128, kNO, true, false) : idesc_bf16(128, kNO, true, false);
};
static_assert(TcCfg<true, 4>::kSmem <= 232448 && TcCfg<true, 8>::kSmem <= 232448 &&
                  TcCfg<false, 8>::kSmem <= 232448 && TcCfg<false, 16>::kSmem <= 232448, "shared memory");
static_assert(TcCfg<true, 4>::kQC % 1024 == 0 && TcCfg<true, 8>::kP % 1024 == 0 &&
                  TcCfg<false, 8>::kP % 1024 == 0, "1024-byte swizzle atoms");


struct DecItem {
    int32_t ri, req, q_start, hk, split, lo, hi, nt;
};

// Item p of the decode work list: first every full kDecodeChunk-key split (row
// by row, kv head by kv head; pre[i] counts those of the rows before row i,
// pre[num_rows] all of them), then the partial last splits, hkv items per row
// in the order of tail_rows (longest partial first). Dealt in snake order, the
// CTAs then end within a fraction of a split of each other. The caller's items
// rise, so the row cursor ri only walks forward over the prefix.
__device__ __forceinline__ DecItem dec_item(const int32_t* pre, int32_t& ri, int32_t p, const pcp_row_t* rows,
                                            const int32_t* tail_rows, int32_t num_rows, int32_t hkv) {
    const int32_t nfull = pre[num_rows];
    const bool full = p < nfull;
    int32_t r, rem;
    if (full) {
        while (pre[ri + 1] <= p) ++ri;
        r = ri;
        rem = p - pre[r];
    } else {
        rem = p - nfull;
        r = tail_rows[rem / hkv];
    }
    const pcp_row_t row = rows[r];
    const int32_t nf = row.kv_end / kDecodeChunk;  // full splits of the row (>= 1 on the full side)
    DecItem it;
    it.ri = r;
    it.req = row.req;
    it.q_start = row.q_start;
    it.hk = full ? rem / nf : rem % hkv;
    it.split = full ? rem % nf : nf;
    it.lo = it.split * kDecodeChunk;
    it.hi = min(row.kv_end, it.lo + kDecodeChunk);
    it.nt = (it.hi - it.lo + kKeys - 1) / kKeys;
    return it;
}

// Named barrier 3 over the eight softmax warps that also ORs a predicate.
__device__ __forceinline__ bool bar_all_or(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 3, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Named barrier `id` over `n` threads (whole warps).
__device__ __forceinline__ void bar_sync_named(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Named barrier `id` over one softmax warpgroup (128 threads) that also ORs a
// predicate: every thread gets the same answer, so the warps leave their loops
// together.
__device__ __forceinline__ bool bar_wg_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id)
        : "memory");
    return r != 0;
}

// Max (kMax) or sum over the warp of GP values per lane, by reduce-scatter: each
// step with offset o = 16, 8, ... halves the values a lane keeps (the upper half
// where bit o of the lane is set), the remaining offsets reduce the last one.
// Lane l ends with head l / (32 / GP) reduced over all 32 lanes.
template <int GP, bool kMax>
__device__ __forceinline__ float warp_scatter(const float (&x)[GP], int lane) {
    float v[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) v[h] = x[h];
#pragma unroll
    for (int o = 16, n = GP; n > 1; o >>= 1, n >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < n / 2; ++k) {
            const float send = upper ? v[k] : v[k + n / 2];
            const float keep = upper ? v[k + n / 2] : v[k];
            const float r = __shfl_xor_sync(0xffffffffu, send, o);
            v[k] = kMax ? fmaxf(keep, r) : keep + r;
        }
    }
#pragma unroll
    for (int o = 16 / GP; o >= 1; o >>= 1) {
        const float r = __shfl_xor_sync(0xffffffffu, v[0], o);
        v[0] = kMax ? fmaxf(v[0], r) : v[0] + r;
    }
    return v[0];
}

// One tile of FP8 codes -> f16 in the 128-byte-swizzled K-major layout of a
// stage (dims 64h..64h+63 of row r in half h, 16-byte chunk c of that row at
// chunk c ^ (r & 7)). The codes of row r (128 bytes) sit where half 1 of row r
// goes; the eight threads of a row are in one warp and all load before any of
// them stores. Rows at or past nvalid are written as zeros (their codes may be
// stale or unwritten cache slots). Run by the 128 converter threads.
__device__ __forceinline__ void widen_tile(uint8_t* tile, int nvalid, int ct) {
    constexpr int kHalf = kKeys * 128;
    constexpr int kRpp = kConvThreads / 8;  // rows per pass
    constexpr int kBatch = 4;
    const int t = ct % 8, rsub = ct / 8;
    const int h = t / 4, c0 = 2 * (t % 4);
    // threads of the second half store their odd chunk first, so the eight
    // threads of a row hit eight different bank groups in each store
    const int first = c0 + (t >= 4 ? 1 : 0), second = c0 + (t >= 4 ? 0 : 1);
    const uint8_t* codes = tile + kHalf;
#pragma unroll 1
    for (int r0 = 0; r0 < kKeys; r0 += kRpp * kBatch) {
        uint4 c[kBatch];
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = r0 + kRpp * b + rsub;
            c[b] = r < nvalid ? *reinterpret_cast<const uint4*>(codes + r * kD + 16 * t) : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int r = r0 + kRpp * b + rsub;
            const uint2 w0 = e4m3x4_to_f16x4(c[b].x), w1 = e4m3x4_to_f16x4(c[b].y);
            const uint2 w2 = e4m3x4_to_f16x4(c[b].z), w3 = e4m3x4_to_f16x4(c[b].w);
            const uint4 lo = make_uint4(w0.x, w0.y, w1.x, w1.y);  // dims 16t .. 16t+7
            const uint4 hi = make_uint4(w2.x, w2.y, w3.x, w3.y);  // dims 16t+8 .. 16t+15
            uint8_t* row = tile + h * kHalf + r * 128;
            const bool lo_first = first == c0;
            *reinterpret_cast<uint4*>(row + ((first ^ (r & 7)) << 4)) = lo_first ? lo : hi;
            *reinterpret_cast<uint4*>(row + ((second ^ (r & 7)) << 4)) = lo_first ? hi : lo;
        }
        __syncwarp();
    }
}

// FP8: the group's q heads as kTerms e4m3 terms each. Input: the bf16 Q^T
// tile as TMA wrote it (two 64-dim halves of 16 rows, 128-byte swizzled).
// Output: the swizzled K-major layout of an e4m3 MMA operand, row t * GP + h
// holding term t of head h (128 codes, 16-byte chunk c of row r at chunk
// c ^ (r & 7)). Head h is first scaled by 2^(8 - ex), ex the binary exponent
// of its largest magnitude (frexp), so that every element lies below 256. The
// first term is the e4m3 rounding of the scaled element x (4 significant bits);
// the remainder x - term is a multiple of x's last bit no larger than 8 of
// them (x has 8 significant bits), so it is an e4m3 value too and the two
// terms sum to x exactly, unless the remainder falls under e4m3's smallest
// subnormal (2^-9 of the scaled unit, where the largest element lies in
// [128, 256): only elements below 2^-9 of the head's largest can lose bits, at
// most 2^-17 of it). qscale[h] = 2^(ex - 8) undoes
// the scaling. Warp w of the converter set does heads w and w + 4, lane l dims
// 4l .. 4l + 3. Returns whether an element of one of the G real heads lies
// beyond +-65504 (reported as PCP_ERR_RANGE, as the prefill rows' q is).
template <int GP>
__device__ __forceinline__ bool q_to_e4m3_terms(const uint8_t* qbf, uint8_t* qc, float* qscale, int w, int lane,
                                                int G) {
    bool over = false;
#pragma unroll
    for (int h = w; h < GP; h += 4) {
        const int d = 4 * lane, half = d >> 6, col = d & 63;
        const uint2 raw =
            *reinterpret_cast<const uint2*>(qbf + half * (kN * 128) + h * 128 + (((col >> 3) ^ (h & 7)) << 4) + (col & 7) * 2);
        float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
        float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        over |= h < G && m > 65504.f;
        int ex = 0;
        frexpf(m, &ex);
        const float f = ldexpf(1.f, 8 - ex);
        if (lane == 0) qscale[h] = ldexpf(1.f, ex - 8);
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] *= f;
#pragma unroll
        for (int t = 0; t < kTerms; ++t) {
            const uint32_t codes = f32x2_to_e4m3x2(x[0], x[1]) | (f32x2_to_e4m3x2(x[2], x[3]) << 16);
            const int row = t * GP + h;
            *reinterpret_cast<uint32_t*>(qc + row * 128 + (((d >> 4) ^ (row & 7)) << 4) + (d & 15)) = codes;
            if (t + 1 < kTerms) {
                float back[4];
                e4m3x4_to_f32(codes, back);
#pragma unroll
                for (int e = 0; e < 4; ++e) x[e] -= back[e];  // exact: both hold few significant bits
            }
        }
    }
    return over;
}

template <bool F8>
__device__ __forceinline__ uint16_t to16(float x) {
    if constexpr (F8) return __half_as_ushort(__float2half_rn(x));
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
template <bool F8>
__device__ __forceinline__ float from16(uint16_t x) {
    if constexpr (F8) return __half2float(__ushort_as_half(x));
    return __bfloat162float(__ushort_as_bfloat16(x));
}

template <bool F8, int GP>
__global__ void __launch_bounds__(tc_threads(F8, GP), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, PrefillArgs a, float* __restrict__ dec_out,
                     float* __restrict__ dec_lse, int max_splits, int q_rows) {
    using C = TcCfg<F8, GP>;
    constexpr int kKS = C::kKS, kVS = C::kVS, kNS = C::kNS;
    const int32_t total = a.num_units[1];
    if ((int32_t)blockIdx.x >= total) return;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kBar;
    // stage barriers: K tile landed, K stage free (its S is done); V tile ready
    // (FP8: widened), V stage free (its PV is done), FP8 V codes landed
    auto k_full = [&](int s) { return bar0 + 8 * s; };
    auto k_empty = [&](int s) { return bar0 + 8 * (kKS + s); };
    const uint32_t bv = bar0 + 8 * 2 * kKS;
    auto v_full = [&](int s) { return bv + 8 * s; };
    auto v_empty = [&](int s) { return bv + 8 * (kVS + s); };
    auto vc_full = [&](int s) { return bv + 8 * (2 * kVS + s); };
    // double-buffered: Q^T ready / bf16 Q^T landed (FP8) / free; S^T, P^T, O^T
    const uint32_t bx = bv + 8 * 3 * kVS;
    auto q_full = [&](int b) { return bx + 8 * b; };
    auto qc_full = [&](int b) { return bx + 16 + 8 * b; };
    auto q_empty = [&](int b) { return bx + 32 + 8 * b; };
    auto s_full = [&](int b) { return bx + 48 + 8 * b; };
    auto p_full = [&](int b) { return bx + 64 + 8 * b; };
    auto o_full = [&](int b) { return bx + 80 + 8 * b; };
    auto o_free = [&](int b) { return bx + 96 + 8 * b; };
    // FP8: the q scales of item i are in slot i % 4 (for the softmax)
    auto q_ready = [&](int b) { return bx + 112 + 8 * b; };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMisc + 4);
    int32_t* pre = reinterpret_cast<int32_t*>(smem + C::kPre);
    int32_t* pages = reinterpret_cast<int32_t*>(smem + C::kPages);
    float* red_m = reinterpret_cast<float*>(smem + C::kRed);  // [warpgroup][tile parity][warp][head]
    constexpr int kGS = C::kGS, kNO = C::kNO;
    float* red_l = red_m + 2 * 2 * 4 * kGS;                   // [item parity][8 warps][head]
    float* xchg = reinterpret_cast<float*>(smem + C::kXchg);  // bf16: [head max, head x dim O]

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int G = a.hq / a.hkv;
    const int32_t bs = a.block_size;
    const int32_t step = (int32_t)gridDim.x;
    // item of this CTA in round rd: snake order (forward on even rounds, backward
    // on odd ones) over the list, whose full splits come first and partial ones
    // longest first
    auto item_of_round = [&](int32_t rd) -> int32_t {
        return rd * step + ((rd & 1) ? step - 1 - (int32_t)blockIdx.x : (int32_t)blockIdx.x);
    };
    const int32_t* tail_rows = a.dec_pre + a.num_rows + 1;

    for (int i = threadIdx.x; i <= a.num_rows; i += tc_threads(F8, GP)) pre[i] = a.dec_pre[i];
    if (threadIdx.x == 0) {
        const uint32_t filled = F8 ? 4 : 1;  // FP8: each warp of the converter set arrives
        for (int s = 0; s < kKS; ++s) {
            mbar_init(k_full(s), 1);  // the producer's expect_tx (FP8 too: the codes are the operand)
            mbar_init(k_empty(s), 1);
        }
        for (int s = 0; s < kVS; ++s) {
            mbar_init(v_full(s), filled);
            mbar_init(v_empty(s), 1);
            mbar_init(vc_full(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(q_full(b), filled);
            mbar_init(qc_full(b), 1);
            mbar_init(q_empty(b), 1);
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 4);  // the four warps of the tile's warpgroup
            mbar_init(o_full(b), 1);
            mbar_init(o_free(b), 4);
        }
        for (int b = 0; b < 4; ++b) mbar_init(q_ready(b), 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProdWarp && lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProdWarp || warp == kProdWarp + 1) {
        // ---------------------------------------------------------------- producers
        // Warp 8 loads the K tiles (and each item's Q^T), warp 9 the V tiles: a K
        // stage is free again once its S is done, a V stage once its PV is, and
        // neither side waits for the other.
        const bool is_k = warp == kProdWarp;
        const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
        int32_t* my_pages = pages + (is_k ? 0 : kMaxPages);
        const int nst = is_k ? kKS : kVS;
        const int32_t oob = (int32_t)(a.num_blocks * bs);  // a row past the cache: zero fill
        const int ppt = kKeys / bs;                        // pages per tile
        const uint32_t q_bytes = 2u * (uint32_t)q_rows * 128u;
        // FP8: the K codes are the MMA's operand (full on landing), the V codes go
        // to the converters first
        auto full_of = [&](int st) { return is_k ? k_full(st) : (F8 ? vc_full(st) : v_full(st)); };
        uint32_t gt = 0, ic = 0;
        int32_t ri = 0;
        bool ok = true;
        for (int32_t rd = 0, p = item_of_round(0); p < total && ok; p = item_of_round(++rd)) {
            const DecItem it = dec_item(pre, ri, p, a.rows, tail_rows, a.num_rows, a.hkv);
            // the split's block-table entries as first cache rows; a bad id maps to a
            // row past the cache (zero filled) and reports PCP_ERR_RANGE
            const int32_t* table = a.block_table + (size_t)it.req * a.max_blocks;
            const int32_t pg0 = it.lo / bs;
            const int npg = (it.hi - it.lo + bs - 1) / bs;
            __syncwarp();
            for (int i = lane; i < npg; i += 32) {
                const int32_t pg = pg0 + i;
                const int32_t id = pg < a.max_blocks ? __ldg(table + pg) : -1;
                int32_t y = oob;
                if (id >= 0 && id < a.num_blocks) y = id * bs;
                else if (is_k) report_status(a.status, PCP_ERR_RANGE);
                my_pages[i] = y;
            }
            __syncwarp();
            if (is_k) {
                const int qb = ic & 1;
                if (!(ok = mbar_wait_warp(q_empty(qb), ((ic >> 1) & 1) ^ 1, abort_flag))) break;
                if (lane == 0) {
                    const uint32_t qbar = F8 ? qc_full(qb) : q_full(qb);
                    mbar_arrive_expect_tx(qbar, q_bytes);
                    for (int h = 0; h < 2; ++h)
                        tma_load_3d(sbase + C::kQ + qb * C::kQBytes + h * C::kRowsBytes, &tm_q, qbar, h * 64,
                                    it.hk * G, it.q_start);
                }
                ++ic;
            }
            for (int j = 0; j < it.nt; ++j) {
                const int st = gt % nst;
                const int nvalid = min(kKeys, it.hi - it.lo - j * kKeys);
                const int np = (nvalid + bs - 1) / bs;
                if (!(ok = mbar_wait_warp(is_k ? k_empty(st) : v_empty(st), ((gt / nst) & 1) ^ 1, abort_flag)))
                    break;
                const uint32_t fb = full_of(st);
                if (lane == 0) mbar_arrive_expect_tx(fb, (uint32_t)(np * bs) * (F8 ? kD : 2 * kD));
                __syncwarp();
                if (lane < np) {
                    const int32_t y = my_pages[j * ppt + lane];
                    const uint32_t dst = sbase + (is_k ? C::kK + st * C::kKTileBytes : C::kV + st * C::kTileBytes);
                    if constexpr (F8) {
                        // K: the codes, 128-byte swizzled, as the e4m3 operand; V: the codes
                        // where half 1 of the f16 tile goes, unswizzled, for the converters
                        tma_load_3d(dst + (is_k ? 0 : C::kHalfBytes) + lane * bs * kD, tm, fb, 0, it.hk, y);
                    } else {
                        for (int h = 0; h < 2; ++h)
                            tma_load_3d(dst + h * C::kHalfBytes + lane * bs * 128, tm, fb, h * 64, it.hk, y);
                    }
                }
                ++gt;
            }
        }
        if (!ok && lane == 0) {
            report_status(a.status, PCP_ERR_TIMEOUT);
            // wait (bounded, whatever the abort flag says) for the copies already
            // issued, so that none lands after the CTA has gone
            int no_abort = 0;
            for (uint32_t g = gt > (uint32_t)nst ? gt - nst : 0; g < gt; ++g)
                mbar_wait(full_of(g % nst), (g / nst) & 1, &no_abort, 100000000ull);
            if (is_k)
                for (uint32_t i = ic > 2 ? ic - 2 : 0; i < ic; ++i)
                    mbar_wait(F8 ? qc_full(i & 1) : q_full(i & 1), (i >> 1) & 1, &no_abort, 100000000ull);
        }
    } else if (warp == kMmaWarp || warp == kPvWarp) {
        // ---------------------------------------------------------------- MMA issuers
        // Two threads in different warps: one issues every S, the other every PV.
        // They share no operand (S reads a K stage and Q^T, PV a V stage and P^T;
        // their TMEM columns differ), and each commit covers the MMAs of the thread
        // that makes it, so the two streams need no ordering between them.
        if (lane == 0) {
            // descriptors of the first k-step; a later k-step moves the start address
            auto k_desc = [&](int s) { return sdesc_sw128(sbase + C::kK + s * C::kKTileBytes, 16, 1024); };
            auto v_desc = [&](int s) {
                return sdesc_sw128(sbase + C::kV + s * C::kTileBytes, C::kHalfBytes, 1024);
            };
            auto q_desc = [&](int b) {
                return sdesc_sw128(sbase + (F8 ? C::kQC + b * C::kQCBytes : C::kQ + b * C::kQBytes), 16, 1024);
            };
            auto p_desc = [&](int b) { return sdesc_sw128(sbase + C::kP + b * C::kPBytes, 16, 1024); };
            uint32_t g = 0, ic = 0;
            int32_t ri = 0;
            bool ok = true;
            const bool s_role = warp == kMmaWarp;
            for (int32_t rd = 0, p = item_of_round(0); p < total && ok; p = item_of_round(++rd)) {
                const DecItem it = dec_item(pre, ri, p, a.rows, tail_rows, a.num_rows, a.hkv);
                const int qb = ic & 1;
                if (s_role && !(ok = mbar_wait(q_full(qb), (ic >> 1) & 1, abort_flag))) break;
                for (int j = 0; j < it.nt; ++j, ++g) {
                    if (s_role) {
                        // S^T(g) = K(g) Q^T: A = the K tile (K-major, 128 keys), B = Q^T
                        // (K-major, 16 rows); S buffer g & 1 is free once P(g - 2) is written
                        if (g >= 2 && !(ok = mbar_wait(p_full(g & 1), ((g - 2) >> 1) & 1, abort_flag))) break;
                        if (!(ok = mbar_wait(k_full(g % kKS), (g / kKS) & 1, abort_flag))) break;
                        tc_fence_after();
                        const uint64_t kd = k_desc(g % kKS), qd = q_desc(qb);
                        const uint32_t ts = tmem + C::kTmemS + (g & 1) * kNS;
                        if constexpr (F8) {
                            // e4m3 x e4m3, 32 dims (32 bytes of each 128-byte row) per MMA
#pragma unroll
                            for (int ks = 0; ks < kD / 32; ++ks)
                                mma_ss_e4m3(ts, kd + (uint32_t)(ks * 2), qd + (uint32_t)(ks * 2), C::kIdescS,
                                            ks > 0 ? 1u : 0u);
                        } else {
#pragma unroll
                            for (int ks = 0; ks < kD / 16; ++ks) {
                                const uint32_t koff = ((ks / 4) * C::kHalfBytes + (ks % 4) * 32) >> 4;
                                const uint32_t qoff = ((ks / 4) * C::kRowsBytes + (ks % 4) * 32) >> 4;
                                mma_ss(ts, kd + koff, qd + qoff, C::kIdescS, ks > 0 ? 1u : 0u);
                            }
                        }
                        mma_commit(s_full(g & 1));
                        mma_commit(k_empty(g % kKS));
                    } else {
                        // O^T(g) = V(g)^T P^T: A = the V tile read MN-major (M = D), B = P^T
                        // (K-major, 16 rows), once P(g) is written, V(g) is in and the softmax
                        // has taken O(g - 2) out of the O buffer
                        if (!(ok = mbar_wait(p_full(g & 1), (g >> 1) & 1, abort_flag))) break;
                        if (!(ok = mbar_wait(v_full(g % kVS), (g / kVS) & 1, abort_flag))) break;
                        if (!(ok = mbar_wait(o_free(g & 1), ((g >> 1) & 1) ^ 1, abort_flag))) break;
                        tc_fence_after();
                        const uint64_t vd = v_desc(g % kVS), pd = p_desc(g & 1);
#pragma unroll
                        for (int ks = 0; ks < kKeys / 16; ++ks) {
                            const uint32_t poff = ((ks / 4) * (kNO * 128) + (ks % 4) * 32) >> 4;
                            mma_ss(tmem + C::kTmemO + (g & 1) * kNO, vd + (uint32_t)(ks * 2048 >> 4), pd + poff,
                                   C::kIdescO, ks > 0 ? 1u : 0u);
                        }
                        mma_commit(o_full(g & 1));
                        mma_commit(v_empty(g % kVS));
                    }
                }
                if (!ok) break;
                if (s_role) mma_commit(q_empty(qb));
                ++ic;
            }
            if (!ok) report_status(a.status, PCP_ERR_TIMEOUT);
        }
    } else if (F8 && warp >= kConvWarp0) {
        // ---------------------------------------------------------------- FP8 converters
        // Set 0 (warps 12-15) also turns each item's q into its e4m3 terms; the V
        // tiles are widened by set g % (number of sets).
        constexpr int kSets = F8 ? conv_warps(F8, GP) / 4 : 1;
        const int cset = (warp - kConvWarp0) / 4, cw = (warp - kConvWarp0) % 4;
        const int ct = (threadIdx.x - kConvWarp0 * 32) % kConvThreads;
        uint32_t gt = 0, ic = 0;
        int32_t ri = 0;
        bool ok = true;
        for (int32_t rd = 0, p = item_of_round(0); p < total && ok; p = item_of_round(++rd)) {
            const DecItem it = dec_item(pre, ri, p, a.rows, tail_rows, a.num_rows, a.hkv);
            const int qb = ic & 1;
            if (cset == 0) {
                if (!(ok = mbar_wait_warp(qc_full(qb), (ic >> 1) & 1, abort_flag))) break;
                if (q_to_e4m3_terms<GP>(smem + C::kQ + qb * C::kQBytes, smem + C::kQC + qb * C::kQCBytes,
                                        reinterpret_cast<float*>(smem + C::kQs) + (ic & 3) * kGS, cw, lane, G) &&
                    lane == 0)
                    report_status(a.status, PCP_ERR_RANGE);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(q_full(qb));
                    mbar_arrive(q_ready(ic & 3));
                }
            }
            ++ic;
            for (int j = 0; j < it.nt; ++j) {
                const uint32_t g = gt + j;
                if ((int)(g % kSets) != cset) continue;
                const int vs = g % kVS;
                const int nvalid = min(kKeys, it.hi - it.lo - j * kKeys);
                if (!(ok = mbar_wait_warp(vc_full(vs), (g / kVS) & 1, abort_flag))) break;
                widen_tile(smem + C::kV + vs * C::kTileBytes, nvalid, ct);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(v_full(vs));
            }
            gt += it.nt;
        }
        if (!ok && lane == 0) report_status(a.status, PCP_ERR_TIMEOUT);
    } else {
        // ---------------------------------------------------------------- softmax
        // Two warpgroups take alternate tiles (tile g: warpgroup g % 2), each with its
        // own running max, sums and O over its tiles; at the end of an item
        // warpgroup 0 merges the two and writes the split's partial.
        const int wg = warp / 4, wq = warp % 4;
        const int t = threadIdx.x % 128;  // key of the tile (S^T lane), dim (O^T lane)
        const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
        constexpr int kSpan = 32 / GP;     // lanes that end the reduce-scatter with one head
        const int hl = lane / kSpan;       // that head
        uint32_t gt = 0, ic = 0;
        int32_t ri = 0;
        bool ok = true;     // every wait of this thread so far completed
        bool stop = false;  // the joint decision to stop (FP8: the warpgroup's; bf16: both's), once per item
        for (int32_t rd = 0, p = item_of_round(0); p < total && !stop; p = item_of_round(++rd), ++ic) {
            const DecItem it = dec_item(pre, ri, p, a.rows, tail_rows, a.num_rows, a.hkv);
            const float kd = F8 ? __ldg(a.k_descale + (size_t)it.req * a.hkv + it.hk) : 1.f;
            const float sl2 = a.scale * kd * kLog2e;
            // FP8: the power of two that undoes each head's q scaling (see q_to_e4m3_terms)
            float qs[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) qs[h] = 1.f;
            if constexpr (F8) {
                ok &= mbar_wait_warp(q_ready(ic & 3), (ic >> 2) & 1, abort_flag);
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    qs[h] = reinterpret_cast<const float*>(smem + C::kQs)[(ic & 3) * kGS + h];
            }
            float m_run[GP], l_t[GP], acc[GP], a_prev[GP];
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                m_run[h] = -INFINITY;
                l_t[h] = 0.f;
                acc[h] = 0.f;
                a_prev[h] = 0.f;
            }
            // O^T of tile g (this thread's dim) into the running sums, rescaled by the
            // max update of that tile
            auto accumulate = [&](uint32_t g, const float (&alpha)[GP]) {
                ok &= mbar_wait_warp(o_full(g & 1), (g >> 1) & 1, abort_flag);
                tc_fence_after();
                uint32_t o[kNO];
                const uint32_t t_o = tmem + lane_base + C::kTmemO + (g & 1) * kNO;
                if constexpr (kNO == 32) {
                    tmem_ld32(t_o, o);
                } else {
                    tmem_ld16(t_o, o);
                }
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free(g & 1));
#pragma unroll
                for (int h = 0; h < GP; ++h)
                    acc[h] = acc[h] * alpha[h] + (__uint_as_float(o[h]) + __uint_as_float(o[kGS + h]));
            };
            uint32_t g_prev = 0;
            bool have_prev = false;
            for (int j = 0; j < it.nt; ++j) {
                const uint32_t g = gt + j;
                if ((int)(g & 1) != wg) continue;
                const int nvalid = min(kKeys, it.hi - it.lo - j * kKeys);
                const bool valid = t < nvalid;
                ok &= mbar_wait_warp(s_full(g & 1), (g >> 1) & 1, abort_flag);
                tc_fence_after();
                uint32_t s[kNS];
                tmem_ld16(tmem + lane_base + C::kTmemS + (g & 1) * kNS, s);
                tmem_wait_ld();
                float x[GP];
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    float sh = __uint_as_float(s[h]);
                    if constexpr (F8) {  // the q terms' scores, then the head's q scale
                        sh = (sh + __uint_as_float(s[GP + h])) * qs[h];
                    }
                    x[h] = valid ? sh * sl2 : -INFINITY;
                }
                // tile max per head: over the warp, then over the warpgroup's four warps
                float* rm = red_m + (wg * 2 + ((g >> 1) & 1)) * 4 * kGS;  // [warp][head]
                const float wm = warp_scatter<GP, true>(x, lane);
                if (lane % kSpan == 0) rm[wq * kGS + hl] = wm;
                bar_sync_named(1 + wg, 128);
                // O(g - 2) out of TMEM first: PV(g - 2) complete frees P buffer g & 1
                if (have_prev) accumulate(g_prev, a_prev);
                float alpha[GP];
                uint8_t* pbuf = smem + C::kP + (g & 1) * C::kPBytes;
                // this key's column of P^T: chunk (t % 64) / 8 of each row, swizzled by the row
                uint8_t* pcol = pbuf + (t >> 6) * (kNO * 128) + (t & 7) * 2;
                const int chunk = (t & 63) >> 3;
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    const float mt = fmaxf(fmaxf(rm[h], rm[kGS + h]), fmaxf(rm[2 * kGS + h], rm[3 * kGS + h]));
                    const float m_new = fmaxf(m_run[h], mt);  // finite: the tile has a valid key
                    alpha[h] = fast_exp2(m_run[h] - m_new);   // 0 on the warpgroup's first tile
                    m_run[h] = m_new;
                    const float pe = fast_exp2(x[h] - m_new);
                    l_t[h] = l_t[h] * alpha[h] + pe;
                    const uint16_t hi = to16<F8>(pe);
                    const uint16_t lo = to16<F8>(pe - from16<F8>(hi));
                    *reinterpret_cast<uint16_t*>(pcol + h * 128 + ((chunk ^ (h & 7)) << 4)) = hi;
                    *reinterpret_cast<uint16_t*>(pcol + (kGS + h) * 128 + ((chunk ^ (h & 7)) << 4)) = lo;
                }
                if (!F8 && nvalid < kKeys) {
                    // keys past the split's end: zero their V rows (unwritten cache slots in
                    // the last page, stale rows after it) once the tile has landed
                    const uint32_t vs = g % kVS;
                    ok &= mbar_wait_warp(v_full(vs), (g / kVS) & 1, abort_flag);
                    if (!valid) {
                        uint8_t* vrow = smem + C::kV + vs * C::kTileBytes + t * 128;
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4*>(vrow + h * C::kHalfBytes + c * 16) = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(g & 1));
                g_prev = g;
                have_prev = true;
#pragma unroll
                for (int h = 0; h < GP; ++h) a_prev[h] = alpha[h];
            }
            if (have_prev) accumulate(g_prev, a_prev);
            gt += it.nt;
            float* rl = red_l + (ic & 1) * 8 * kGS;  // [warp 0..7][head]
            const float wl = warp_scatter<GP, false>(l_t, lane);
            if (lane % kSpan == 0) rl[warp * kGS + hl] = wl;
            const float vd = F8 ? __ldg(a.v_descale + (size_t)it.req * a.hkv + it.hk) : 1.f;
            if constexpr (C::kSplitParts) {
                // FP8 and 16 heads: each warpgroup writes its own partial of the split (a
                // warpgroup without a tile of the item writes (0, -inf)); decode_merge_kernel
                // combines the two, so the warpgroups never wait for each other
                if ((stop = bar_wg_or(1 + wg, !ok))) break;
                const float* rw = rl + wg * 4 * kGS;
#pragma unroll
                for (int h = 0; h < GP; ++h) {
                    if (h >= G) continue;
                    const float L = rw[h] + rw[kGS + h] + rw[2 * kGS + h] + rw[3 * kGS + h];
                    const size_t slot =
                        ((size_t)it.ri * a.hq + it.hk * G + h) * (2 * max_splits) + 2 * it.split + wg;
                    dec_out[slot * kD + t] = L > 0.f ? acc[h] / L * vd : 0.f;
                    if (t == 0) dec_lse[slot] = L > 0.f ? (m_run[h] + __log2f(L)) * kLn2 : -INFINITY;
                }
            } else {
                // bf16: warpgroup 1 hands its max and O over, warpgroup 0 merges and
                // writes the split's one partial (measured faster here than two
                // partials: this decode streams near the HBM bound, where the extra
                // partials' bytes show)
                if (wg == 1) {
#pragma unroll
                    for (int h = 0; h < GP; ++h) {
                        if (t == 0) xchg[h] = m_run[h];
                        xchg[kGS + h * kKeys + t] = acc[h];
                    }
                }
                if ((stop = bar_all_or(!ok))) break;
                if (wg == 0) {
#pragma unroll
                    for (int h = 0; h < GP; ++h) {
                        if (h >= G) continue;
                        const float L0 = rl[h] + rl[kGS + h] + rl[2 * kGS + h] + rl[3 * kGS + h];
                        const float L1 = rl[4 * kGS + h] + rl[5 * kGS + h] + rl[6 * kGS + h] + rl[7 * kGS + h];
                        const float m1 = xchg[h];
                        const float M = fmaxf(m_run[h], m1);  // finite: the item has a tile
                        const float f0 = fast_exp2(m_run[h] - M), f1 = fast_exp2(m1 - M);
                        const float L = L0 * f0 + L1 * f1;
                        const float O = acc[h] * f0 + xchg[kGS + h * kKeys + t] * f1;
                        const size_t slot = ((size_t)it.ri * a.hq + it.hk * G + h) * (2 * max_splits) + it.split;
                        dec_out[slot * kD + t] = L > 0.f ? O / L : 0.f;
                        if (t == 0) dec_lse[slot] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
                    }
                }
                // warpgroup 1 writes the exchange area of the next item only after this
                bar_sync_named(4, 256);
            }
        }
        if (stop && t == 0) report_status(a.status, PCP_ERR_TIMEOUT);
    }

    __syncwarp();  // lane 0 of the MMA warp and of the producer worked alone: reconverge first
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <bool F8, int GP>
int launch_tc(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits, cudaStream_t stream,
              int grid) {
    const int64_t slots = a.num_blocks * a.block_size;
    const int q_rows = a.hq < kN ? a.hq : kN;
    CUtensorMap tq, tk, tv;
    bool maps = make_box_map(&tq, a.q, kD, 2, a.hq, a.total_q, 64, q_rows, 1, true);
    if (F8)  // K codes 128-byte swizzled (the MMA operand), V codes plain (for the converters)
        maps = maps && make_box_map(&tk, a.key_cache, kD, 1, a.hkv, slots, kD, 1, a.block_size, true) &&
               make_box_map(&tv, a.value_cache, kD, 1, a.hkv, slots, kD, 1, a.block_size, false);
    else
        maps = maps && make_box_map(&tk, a.key_cache, kD, 2, a.hkv, slots, 64, 1, a.block_size, true) &&
               make_box_map(&tv, a.value_cache, kD, 2, a.hkv, slots, 64, 1, a.block_size, true);
    if (!maps) return PCP_ERR_CUDA;
    const int smem = TcCfg<F8, GP>::kSmem;
    cudaError_t e =
        cudaFuncSetAttribute(decode_tc_kernel<F8, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    const int ctas = grid > 0 && grid < num_sms() ? grid : num_sms();
    decode_tc_kernel<F8, GP><<<ctas, tc_threads(F8, GP), smem, stream>>>(tq, tk, tv, a, dec_out, dec_lse,
                                                                              max_splits, q_rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) { set_last_cuda_error(e); return PCP_ERR_CUDA; }
    return PCP_OK;
}

}  // namespace

bool decode_tc_applies(const PrefillArgs& a) {
    const int G = a.hkv > 0 ? a.hq / a.hkv : 0;
    return a.d == kD && G >= 1 && G <= (a.k_descale ? 8 : kMaxG) && a.num_rows <= kDecTcMaxRows &&
           a.block_size <= kKeys && kKeys % a.block_size == 0;
}

int launch_decode_tc(const PrefillArgs& a, float* dec_out, float* dec_lse, int32_t max_splits,
                     cudaStream_t stream, int grid) {
    if (!decode_tc_applies(a)) return PCP_ERR_UNSUPPORTED;
    const int G = a.hq / a.hkv;
    // heads per group padded to a power of two (the padded heads' results are not written)
    const int GP = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : G <= 8 ? 8 : 16;
    if (a.k_descale) {
        if (GP == 1) return launch_tc<true, 1>(a, dec_out, dec_lse, max_splits, stream, grid);
        if (GP == 2) return launch_tc<true, 2>(a, dec_out, dec_lse, max_splits, stream, grid);
        if (GP == 4) return launch_tc<true, 4>(a, dec_out, dec_lse, max_splits, stream, grid);
        return launch_tc<true, 8>(a, dec_out, dec_lse, max_splits, stream, grid);
    }
    if (GP == 1) return launch_tc<false, 1>(a, dec_out, dec_lse, max_splits, stream, grid);
    if (GP == 2) return launch_tc<false, 2>(a, dec_out, dec_lse, max_splits, stream, grid);
    if (GP == 4) return launch_tc<false, 4>(a, dec_out, dec_lse, max_splits, stream, grid);
    if (GP == 8) return launch_tc<false, 8>(a, dec_out, dec_lse, max_splits, stream, grid);
    return launch_tc<false, 16>(a, dec_out, dec_lse, max_splits, stream, grid);
}

}  // namespace pcp
