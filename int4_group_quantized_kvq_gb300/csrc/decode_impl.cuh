// decode_impl.cuh -- split-KV flash-decode attention over the packed INT4 cache.
//
// What it computes ("AI inference tuning: KV Cache optimisation and memory
// management", bxzpzcl.cn/news/2871434, section 3.2): for each sequence b and query
// head hq, scores z_t = softmax_scale * q . k_t over all cached positions t, softmax,
// out = sum_t p_t v_t; query head hq reads KV head hq / (Hq / Hkv).  K and V are read
// packed and dequantized inside the kernel ("LLM long-context inference: managing the
// KV cache with an INT4 state machine", pwwt.cn/news/4219524, section 5 step 5), with
// k = (nibble - 8) * k_scale[group], v = (nibble - 8) * v_scale[group] ("4-bit KV cache
// compression", lpnh.cn/news/2042373, section 2.1).  The softmax is the online
// (running max / running sum) form, so no score matrix is materialised ("4-bit KV
// cache compression" section 1.3 on Flash attention).
//
// Design for GB300 (sm_103a):
//  * A unit of work is one page of HK consecutive kv heads of one sequence: HK = 4 when
//    every query head has its own kv head (Hq == Hkv) and pages hold 16 tokens, else
//    HK = 1 and the unit serves the r = Hq / Hkv query heads that share the kv head.  The HK blocks of a unit are
//    adjacent in the pool (block index page * Hkv + head), so one bulk copy moves them.
//    Either way a unit feeds 4 (or 8) query heads, the "slots" of the MMA tiles below.
//  * A persistent grid of CTAs (SM count x resident CTAs) gives every CTA an equal
//    contiguous slice of the flattened (sequence, head group, page) units, so ragged
//    lengths and small batches keep every SM busy.  The CTA's four warps take the units
//    of its slice in turn (warp k: units k, k + 4, ...), so they move through the same
//    (sequence, head group) segments at about the same time.
//  * Each warp owns a ring of `stages` unit buffers in shared memory, filled by 1-D
//    bulk copies (the TMA engine, cp.async.bulk) that complete on per-stage mbarriers.
//    Waits are bounded in time.
//  * The arithmetic runs on the tensor cores (mma.sync m16n8k16, f16 inputs, f32
//    accumulate) and the MMA does the multiply-accumulate.  For a 16-token chunk of one
//    kv head:
//      scores  S[token, col] = K[token, :] . Qcol  with M = 16 tokens, N = 8 columns,
//              K-dim = head_dim.  Column (slot, k-group) carries the slot's q masked to
//              that group, so each group's partial dot product comes out separately
//              and is scaled by its own fp16 scale afterwards.  A K nibble n enters the
//              MMA as the f16 subnormal n * 2^-24, one mask per pair of nibbles (the
//              high nibble of a byte as 16 n * 2^-24, its q column entries divided by
//              16); the MMA gives 2^-24 sum_d n_d q_d exactly in fp32, and the code
//              offset comes off per group: sum_d (n_d - 8) q_d = 2^24 S - 8 sum_d q_d,
//              with sum_d q_d taken once per segment.  With HK = 4 each kv head's chunk
//              has its own accumulator and a thread keeps the one of its slot's head.
//      output  O^T[d, col] += V^T[d, token] . W[token, col] with M = 16 dims, N = 8
//              columns (slot, hi|lo), K-dim = 16 tokens.  W = p * v_scale is split into
//              an f16 high part and an f16 remainder, two columns of the same MMA, which
//              keeps about 22 bits of the weight.  With HK = 4 the columns of the other
//              heads' slots are zeroed for each head's MMA.  M-tiles never straddle a
//              V group.  V nibbles become exact f16 integers n - 8 in two instructions
//              per pair: the offset cannot come off afterwards as for K, since there it
//              would cancel against the sum of the weights over the whole segment.
//    The INT8 per-row cache runs on the same kernel (CODEC 1): one-head units, one group
//    per row with an fp32 scale, K codes entering the score MMA as the f16 subnormals
//    (c + 128) * 2^-24 (one byte permute per pair, the offset removed per row as above)
//    and V codes as exact f16 integers.
//    The score fragment of thread (g, c) holds tokens g, g+8 of slot c (+4), and the
//    output fragment holds slot c (+4) too, so the softmax rescale is thread-local;
//    only the weights are exchanged (four shuffles per chunk and V group).  With HK = 1
//    chunks are taken two at a time (two 16-token pages, or two chunks of a larger
//    page): the two score chains interleave and one softmax reduction covers both.
//  * Split combine.  At the end of each segment (sequence, head group) every warp writes
//    its own partial (running max, running sum and unnormalised output per slot) to the
//    workspace, straight from its accumulators; no warp waits for another, and nothing is counted or fenced on the streaming path, so a warp that
//    finishes its part of a segment early keeps its copies in flight.  A second, small
//    kernel, launched behind this one with programmatic dependent launch, merges the
//    partials of each (sequence, query head) row and writes the output.  The two q
//    buffers of a CTA (which in the decode step also carry the new token's K and V rows)
//    are reused once every warp has taken its fragments out (an mbarrier with one arrival
//    per warp), the only point where warps of a CTA meet.
#pragma once

#include <cuda_fp16.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {
namespace decode {

constexpr uint64_t kWaitLimitNs = 250000000ull;   // a page copy that takes 250 ms has failed

// Warps per CTA, and resident CTAs per SM the register budget is tuned for: 3 (up to 168
// registers) when a thread carries one query-head slot of head_dim <= 128, else 2.
template <int HS>
constexpr int cta_warps() { return 4; }
template <int HS, int D = 128>
constexpr int min_ctas() { return HS == 1 && D <= 128 ? 3 : 2; }

// CTA-wide bookkeeping in shared memory.
struct CtaCtl {
    uint64_t qbar[2];    // completion of the bulk copies of q rows into the two q buffers
    uint64_t qfree[2];   // every warp has taken its q fragments out of the buffer
    uint64_t pad[12];
};
static_assert(sizeof(CtaCtl) == 128, "the planner reserves 128 bytes");
// two buffers of kQRows rows of head_dim D fp16: a segment's query-head rows (up to 8)
// and, in the decode step, its new token's K rows and V rows (2 HK; q rows + 2 HK <= 12)
constexpr int kQRows = 12;
template <int D>
constexpr int q_buf_bytes() { return 2 * kQRows * D * 2; }

struct KParams {
    const uint8_t* pool;
    const __half* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* ws_ml;       // warp partials (one per warp and segment its CTA touches): (max, sum) per slot
    float* ws_o;        //   ... and unnormalised outputs per slot
    int32_t* ws_pre;    // the pages prefix pre[0..B], for the combine kernel
    uint32_t* status;
    int32_t B, Hq, Hkv, Hg, r, ns;  // Hg = Hkv / HK head groups; ns = HK * r query heads per unit
    int32_t P, num_pages, max_blocks, block_bytes, unit_bytes, stages;
    int32_t v_codes, k_scales, v_scales;
    float scale_log2;  // softmax_scale * log2(e)
    // fused append (decode step): one token per sequence, K and V rows [B, Hkv, D] fp16,
    // quantized into the pool at position append_pos[b] (< 0: none).  k_new == nullptr: none.
    const __half* k_new;
    const __half* v_new;
    const int32_t* append_pos;
    uint8_t* pool_w;
    int32_t lg_p, lg_lk, lg_lv;  // log2 of P, of the K and of the V group width in 8-value lanes
    // sliding window with sink tokens: the last `window` positions (window <= 0: all) and
    // the first `sinks` are attended
    int32_t window, sinks;
    // positions attended: seq_lens[b] - len_sub (the INT4 part of the mixed-precision decode
    // stops len_sub positions short of the sequence's end; 0 otherwise)
    int32_t len_sub;
    // bound of every wait on a copy, in ns; and a test of that bound: with withhold > 0 each
    // warp announces its first page copy as `withhold` bytes larger than it is, so the wait
    // for it runs out
    uint64_t wait_ns;
    uint32_t withhold;
    // q is written by the kernel ahead on the stream (the host-buffer step's copy kernel):
    // read it only after griddepcontrol.wait
    bool q_after_wait;
};

// a / b for a >= 0, b > 0, with 32-bit division when both fit (the usual case).
__device__ __forceinline__ long long div_nn(long long a, long long b) {
    if (((a | b) >> 32) == 0) return static_cast<long long>(static_cast<unsigned>(a) / static_cast<unsigned>(b));
    return a / b;
}

// The positions a sequence of L positions attends to ("AI inference tuning: KV Cache
// optimisation and memory management" section 3.2, SlidingWindowAttention, for the query at
// the last position): L is clamped to [0, max_blocks * P]; positions t < L with t >= wlo or
// t < sinks.  Its pages are listed in order: the sink pages [0, sp), then the window pages
// [wlo / P, ceil(L / P)), one run when they meet.  List index j is page j + (j >= gs ? gd : 0).
struct SeqSpan {
    int L;    // positions (clamped)
    int wlo;  // first window position; 0 when every position is attended
    int gs;   // list index at which the window pages resume after a gap (np: no gap)
    int gd;   // pages skipped by the gap
    int np;   // pages listed
};
// P = 2^lg_p.
__device__ __forceinline__ SeqSpan seq_span(int L, int lg_p, int max_blocks, int window, int sinks) {
    const int P = 1 << lg_p;
    long long Lc = L < 0 ? 0 : L;
    if (Lc > (static_cast<long long>(max_blocks) << lg_p)) Lc = static_cast<long long>(max_blocks) << lg_p;
    SeqSpan sp;
    sp.L = static_cast<int>(Lc);
    const int npl = (sp.L + P - 1) >> lg_p;
    sp.wlo = 0;
    sp.gs = npl;
    sp.gd = 0;
    sp.np = npl;
    if (window > 0 && sp.L > window) {
        sp.wlo = sp.L - window;
        const int sk = sinks > 0 ? (sinks < sp.L ? sinks : sp.L) : 0;
        const int s_pages = (sk + P - 1) >> lg_p;
        const int w_first = sp.wlo >> lg_p;
        if (w_first > s_pages) {
            sp.gs = s_pages;
            sp.gd = w_first - s_pages;
            sp.np = s_pages + (npl - w_first);
        }
    }
    return sp;
}
// Page of list index j, and list index of page r (-1 when r is not attended).
__device__ __forceinline__ int span_page(const SeqSpan& sp, int j) { return j + (j >= sp.gs ? sp.gd : 0); }
__device__ __forceinline__ int span_index(const SeqSpan& sp, int r) {
    if (r < sp.gs) return r;
    return (r >= sp.gs + sp.gd && r < sp.np + sp.gd) ? r - sp.gd : -1;
}

// Exclusive prefix sums of pages per sequence into pre[0..B], the lengths (negative ones
// as 0) into lens[0..B-1] and the append positions (-1: none) into aps[0..B-1]; run by
// one warp.
__device__ __forceinline__ void page_prefix(const KParams& p, int32_t* pre, int32_t* lens, int32_t* aps, int lane) {
    int carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int np = 0;
        if (b < p.B) {
            int L = p.seq_lens[b] - p.len_sub;
            L = L < 0 ? 0 : L;
            lens[b] = L;
            aps[b] = p.k_new != nullptr ? p.append_pos[b] : -1;
            if (((static_cast<long long>(L) + p.P - 1) >> p.lg_p) > p.max_blocks) raise_flag(p.status, KVQ_FLAG_BAD_POSITION);
            if (p.window > 0) {
                np = seq_span(L, p.lg_p, p.max_blocks, p.window, p.sinks).np;
            } else {
                const long long npl = (static_cast<long long>(L) + p.P - 1) >> p.lg_p;
                np = static_cast<int>(npl < p.max_blocks ? npl : p.max_blocks);
            }
        }
        int x = np;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (b < p.B) pre[b] = carry + x - np;
        carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) pre[p.B] = carry;
}

// Sequence index b containing unit u (largest b with Hg * pre[b] <= u).
__device__ __forceinline__ int find_seq(const int32_t* pre, int B, int Hg, long long u) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(Hg) * pre[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Global address of the HK blocks of unit u, validating the page id.
template <bool WIN>
__device__ __forceinline__ const uint8_t* unit_block(const KParams& p, const int32_t* pre, const int32_t* lens,
                                                     long long u, int HK) {
    const int b = find_seq(pre, p.B, p.Hg, u);
    const long long rem = u - static_cast<long long>(p.Hg) * pre[b];
    const int np = pre[b + 1] - pre[b];
    const int hg = static_cast<int>(rem / np);
    int pg = static_cast<int>(rem - static_cast<long long>(hg) * np);
    if (WIN) pg = span_page(seq_span(lens[b], p.lg_p, p.max_blocks, p.window, p.sinks), pg);
    int page = p.block_table[static_cast<long long>(b) * p.max_blocks + pg];
    if (page < 0 || page >= p.num_pages) {
        raise_flag(p.status, KVQ_FLAG_BAD_PAGE);
        page = 0;
    }
    return p.pool + (static_cast<long long>(page) * p.Hkv + static_cast<long long>(hg) * HK) * p.block_bytes;
}

// The page (index in sequence sb's block-table row) taking the sequence's appended token
// when this call streams that page, else -1: no append, or an append into a page the call
// does not attend (those are written by the grid's spare warps).
template <bool WIN>
__device__ __forceinline__ int seg_append(const KParams& p, const int32_t* pre, const int32_t* lens,
                                          const int32_t* aps, int sb) {
    const int apos = aps[sb];
    if (apos < 0) return -1;
    const long long apg = static_cast<long long>(apos) >> p.lg_p;
    if (apg >= p.max_blocks) return -1;
    if (WIN)
        return span_index(seq_span(lens[sb], p.lg_p, p.max_blocks, p.window, p.sinks), static_cast<int>(apg)) >= 0
                   ? static_cast<int>(apg)
                   : -1;
    return apg < pre[sb + 1] - pre[sb] ? static_cast<int>(apg) : -1;
}

// unit_block for the INT4 kernel, as an integer whose bit 0 marks a bad page id (the
// address is then page 0's, 16-byte aligned, and the flag is raised): the producer clears
// the bit before the copy, the fused append skips such a page.
template <bool WIN>
__device__ __forceinline__ unsigned long long unit_addr_tagged(const KParams& p, const int32_t* pre,
                                                               const int32_t* lens, long long u, int HK) {
    const int b = find_seq(pre, p.B, p.Hg, u);
    const long long rem = u - static_cast<long long>(p.Hg) * pre[b];
    const int np = pre[b + 1] - pre[b];
    const int hg = static_cast<int>(rem / np);
    int pg = static_cast<int>(rem - static_cast<long long>(hg) * np);
    if (WIN) pg = span_page(seq_span(lens[b], p.lg_p, p.max_blocks, p.window, p.sinks), pg);
    int page = p.block_table[static_cast<long long>(b) * p.max_blocks + pg];
    unsigned long long bad = 0;
    if (page < 0 || page >= p.num_pages) {
        raise_flag(p.status, KVQ_FLAG_BAD_PAGE);
        page = 0;
        bad = 1;
    }
    return reinterpret_cast<unsigned long long>(
               p.pool + (static_cast<long long>(page) * p.Hkv + static_cast<long long>(hg) * HK) * p.block_bytes) |
           bad;
}

// First unit of slice w of U units split over W slices.
__device__ __forceinline__ long long slice_start(long long w, long long U, long long W) { return div_nn(w * U, W); }

// The slice containing unit u (the largest w with slice_start(w) <= u).
__device__ __forceinline__ long long slice_of(long long u, long long U, long long W) { return div_nn((u + 1) * W - 1, U); }

// The chunks of one step: chunk X is chunk chk[X] of the unit buffer blk[X] and holds
// sequence positions t0[X] .. t0[X] + 15; a chunk with !live[X] is masked out whole.
template <int TG>
struct Step {
    const uint8_t* blk[TG];
    int chk[TG];
    int t0[TG];
    bool live[TG];
};

// Fused append of the decode step: quantize the new token's K rows (krows: HK rows of D
// fp16, one per kv head of the unit) and V rows (vrows) into slot `slot` of the HK
// consecutive blocks at gblk in the pool and, when the page is staged in shared memory at
// sblk, into that copy too.  The rows are read through generic pointers: from global
// memory for an append into a page the call does not stream, from the segment's q buffer
// (where they were copied with q) for one it does.  All lanes call this.  A row takes
// D / 8 lanes, 8 values each (the same arithmetic and bytes as the quantize-append
// kernel): for D <= 128 the K row and the V row in one pass (lanes past 2 D / 8 idle), for
// D = 256 one after the other.  Out of line: it runs once per segment at most, and inlined
// into the streaming loop its code would crowd the instruction cache.
template <int D, int HK>
__device__ __noinline__ void append_rows(const KParams& p, const __half* krows, const __half* vrows, uint8_t* gblk,
                                         uint8_t* sblk, int slot) {
    constexpr int LPR = D / 8;                 // lanes per row
    constexpr int ROWS = LPR <= 16 ? 2 : 1;    // rows per pass
    const int lane = threadIdx.x & 31;
    const int rsel = lane / LPR;               // this lane's row in the pass
    const int tl = lane % LPR;                 // lane within the row
    for (int a = 0; a < HK; ++a) {
#pragma unroll
        for (int pass = 0; pass < 2 / ROWS; ++pass) {
            const int half = ROWS == 2 ? (rsel & 1) : pass;  // 0: the K row, 1: the V row
            const bool active = ROWS == 2 ? rsel < 2 : true;
            const int lg = half ? p.lg_lv : p.lg_lk;
            const int ng = D >> (lg + 3);
            const int code_off = (half ? p.v_codes : 0) + slot * (D / 2) + tl * 4;
            const int scale_off = (half ? p.v_scales : p.k_scales) + slot * ng * 2 + (tl >> lg) * 2;
            const bool writes_scale = (tl & ((1 << lg) - 1)) == 0;
            uint4 raw = make_uint4(0, 0, 0, 0);
            if (active) raw = *reinterpret_cast<const uint4*>((half ? vrows : krows) + a * D + tl * 8);
            __half s16;
            const uint32_t word = quant_lane8<LPR>(raw, lg, s16);
            if (active) {
                uint8_t* gb = gblk + a * p.block_bytes;
                *reinterpret_cast<uint32_t*>(gb + code_off) = word;
                if (writes_scale) *reinterpret_cast<__half*>(gb + scale_off) = s16;
                if (sblk != nullptr) {
                    uint8_t* sa = sblk + a * p.block_bytes;
                    *reinterpret_cast<uint32_t*>(sa + code_off) = word;
                    if (writes_scale) *reinterpret_cast<__half*>(sa + scale_off) = s16;
                }
            }
        }
    }
    if (sblk != nullptr) {
        fence_proxy_async_smem();  // the stage is refilled by the bulk copy engine later
        __syncwarp();
    }
}

// The N scales of a token row at p (fp16 per group for the INT4 cache, fp32 per row for
// the INT8 cache) and those of the row 8 tokens further: fp16 pairs read as one word.
template <bool F32, int N>
__device__ __forceinline__ void load_scales(const uint8_t* p, float (&a)[N], float (&b)[N]) {
    if constexpr (F32) {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            a[i] = reinterpret_cast<const float*>(p)[i];
            b[i] = reinterpret_cast<const float*>(p)[8 * N + i];
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float2 fa = __half22float2(reinterpret_cast<const __half2*>(p)[i / 2]);
            const float2 fb = __half22float2(reinterpret_cast<const __half2*>(p)[(8 * N + i) / 2]);
            a[i] = fa.x;
            a[i + 1] = fa.y;
            b[i] = fb.x;
            b[i + 1] = fb.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) {
            a[i] = __half2float(reinterpret_cast<const __half*>(p)[i]);
            b[i] = __half2float(reinterpret_cast<const __half*>(p)[8 * N + i]);
        }
    }
}

// P16: the pages hold 16 tokens (P == 16), so two one-head units, i.e. two pages, make a
// step; the instances for larger pages (P16 false) take two 16-token chunks of one page.
// Each instance carries only its own path, which keeps the loop's code small.
// CODEC 0: the INT4 cache (nibble codes, fp16 scales per group).  CODEC 1: the INT8
// per-row cache ("AI inference tuning: KV Cache optimisation and memory management"
// section 3.1): K codes P x D int8, V codes P x D int8, K scales P fp32, V scales P fp32
// per block, a value being code * scale; it runs with one group per row (GK = GV = D) and
// one-head units, and has no fused append.
template <int D, int GK, int GV, int HK, int HS, bool WIN, bool P16, int CODEC = 0>
__global__ void __launch_bounds__(cta_warps<HS>() * 32, min_ctas<HS, D>()) decode_splitkv_kernel(KParams p) {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim 64, 128 or 256");
    static_assert(CODEC == 0 || (CODEC == 1 && D == 128 && GK == D && GV == D && HK == 1), "INT8: d 128, rows");
    static_assert(D <= 128 || (HK == 1 && HS == 1), "head_dim 256: one-head units, up to 4 query heads each");
    static_assert(HK == 1 || HS == 1, "several kv heads per unit only with one query head each");
    static_assert(HK == 1 || P16, "four-head units only for 16-token pages");
    static_assert(4 * HS + 2 * HK <= kQRows, "q rows and the appended token's K and V rows fit a q buffer");
    constexpr int NGK = D / GK;               // K groups per row
    constexpr int NGV = D / GV;               // V groups per row
    constexpr bool I8 = CODEC == 1;
    constexpr int KW = I8 ? D / 16 : D / 32;  // K code words per thread per token row
    constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim
    constexpr int NTQ = (HS * NGK + 1) / 2;   // score n-tiles
    constexpr int VB = GV / 16;               // V code bytes per thread per group per row
    constexpr int MT = D / 16;                // output m-tiles
    constexpr int ROW = I8 ? D : D / 2;       // bytes of one token's codes
    constexpr int SB = I8 ? 4 : 2;            // bytes of one scale (fp32 per row, fp16 per group)
    constexpr float kOff = I8 ? 128.f : 8.f;  // the offset of the codes entering the score MMA
    constexpr int TG = HK == 1 ? 2 : 1;       // 16-token chunks per step
    constexpr int kWarps = cta_warps<HS>();   // warps per CTA
    static_assert(NGV * VB == MT, "m-tiles cover head_dim");

    // a kernel launched behind this one may start its set-up; it waits for this grid
    // before it reads what this grid writes
    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;   // fragment row group
    const int c = lane & 3;    // thread in group
    const int stages = p.stages;
    // block layout: with 16-token pages it is fixed by the template (K codes, V codes, K
    // scales, V scales, the block rounded up to 16 bytes), so offsets fold into the loads
    constexpr int kVC = 16 * ROW, kKS = 32 * ROW, kVS = kKS + 16 * NGK * SB;
    constexpr int kBB = (kVS + 16 * NGV * SB + 15) / 16 * 16;
    const int bbytes = P16 ? kBB : p.block_bytes;
    const int ubytes = P16 ? HK * kBB : p.unit_bytes;
    const int l_vcodes = P16 ? kVC : p.v_codes;
    const int l_kscales = P16 ? kKS : p.k_scales;
    const int l_vscales = P16 ? kVS : p.v_scales;
    const size_t ring_all = static_cast<size_t>(kWarps) * stages * ubytes;
    uint8_t* ring = smem + static_cast<size_t>(warp) * stages * ubytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_all) + warp * stages;
    // the (tagged) pool address of the unit each stage holds, kept for the fused append
    unsigned long long* uaddr = reinterpret_cast<unsigned long long*>(smem + ring_all) + kWarps * stages + warp * stages;
    CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + ring_all + 2 * kWarps * stages * sizeof(uint64_t));
    __half* qbuf = reinterpret_cast<__half*>(ctl + 1);  // [2][kQRows][D]
    int32_t* pre = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(qbuf) + q_buf_bytes<D>());
    int32_t* lens = pre + p.B + 1;
    int32_t* aps = lens + p.B;
    const uint32_t qbar0 = smem_u32(&ctl->qbar[0]);

    // Until griddepcontrol.wait below, the kernel ahead of this one on the stream may still be
    // running.  Only the read-only inputs are read before it: seq_lens, the block table and
    // q.  The pool (written by quantize-append), the output and the workspace come after.
    if (warp == 0) page_prefix(p, pre, lens, aps, lane);
    const uint32_t qfree0 = smem_u32(&ctl->qfree[0]);
    if (threadIdx.x == 0) {
        mbar_init(qbar0, 1);
        mbar_init(qbar0 + 8, 1);
        mbar_init(qfree0, kWarps);
        mbar_init(qfree0 + 8, kWarps);
        fence_mbar_init();
    }
    __syncthreads();

    const long long U = static_cast<long long>(p.Hg) * pre[p.B];
    const long long C = gridDim.x;
    const long long cta = blockIdx.x;
    const long long c0 = slice_start(cta, U, C);
    const long long c1 = slice_start(cta + 1, U, C);

    // Appends whose page this call does not attend (or positions out of the table) are
    // handled here, spread over all warps of the grid; the others by the warp that streams
    // the page, which also patches its staged copy before using it.
    auto orphan_appends = [&]() {
        if (p.k_new == nullptr) return;
        const long long W = C * kWarps;
        const long long nseg = static_cast<long long>(p.B) * p.Hg;
        for (long long t = cta * kWarps + warp; t < nseg; t += W) {
            const int sb = static_cast<int>(t / p.Hg);
            const int shg = static_cast<int>(t - static_cast<long long>(sb) * p.Hg);
            const int apos = aps[sb];
            if (apos < 0) continue;
            const long long apg = static_cast<long long>(apos) >> p.lg_p;
            if (apg >= p.max_blocks) {
                if (lane == 0 && shg == 0) raise_flag(p.status, KVQ_FLAG_BAD_POSITION);
                continue;
            }
            if (WIN ? span_index(seq_span(lens[sb], p.lg_p, p.max_blocks, p.window, p.sinks), static_cast<int>(apg)) >= 0
                    : apg < pre[sb + 1] - pre[sb])
                continue;  // streamed by this call
            const int page = p.block_table[static_cast<long long>(sb) * p.max_blocks + apg];
            if (page < 0 || page >= p.num_pages) {
                if (lane == 0) raise_flag(p.status, KVQ_FLAG_BAD_PAGE);
                continue;
            }
            if constexpr (!I8) {
                const long long row = static_cast<long long>(sb) * p.Hkv + static_cast<long long>(shg) * HK;
                append_rows<D, HK>(p, p.k_new + row * D, p.v_new + row * D,
                                   p.pool_w + (static_cast<long long>(page) * p.Hkv + shg * HK) * p.block_bytes,
                                   nullptr, apos & ((1 << p.lg_p) - 1));
            }
        }
    };

    // the combine kernel finds each segment's partials from the pages prefix
    auto publish_prefix = [&]() {
        if (cta == 0 && warp == 0)
            for (int i = lane; i <= p.B; i += 32) p.ws_pre[i] = pre[i];
    };
    if (c0 >= c1) {
        // no units: only appends nobody streams, after the kernel ahead has finished
        asm volatile("griddepcontrol.wait;" ::: "memory");
        publish_prefix();
        orphan_appends();
        return;  // the whole CTA leaves together
    }
    const int span = static_cast<int>(c1 - c0);
    const int nm = span > warp ? (span - warp + kWarps - 1) / kWarps : 0;  // this warp's units

    const uint32_t bar0 = smem_u32(bars);
    const uint32_t ring0 = smem_u32(ring);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- producer: lane l holds the block address of this warp's unit wbase + l; the next
    // window's addresses are looked up one window ahead so their loads overlap work ----
    auto unit_of = [&](int i) { return c0 + warp + static_cast<long long>(kWarps) * i; };
    int wbase = 0;
    unsigned long long waddr = lane < nm ? unit_addr_tagged<WIN>(p, pre, lens, unit_of(lane), HK) : 0ull;
    unsigned long long wnext = 32 + lane < nm ? unit_addr_tagged<WIN>(p, pre, lens, unit_of(32 + lane), HK) : 0ull;
    int issued = 0;
    const uint64_t l2_stream = l2_policy_evict_first();  // pages are read once per call
    auto issue = [&](int i, int st) {  // this warp's unit i into stage st; i increases call by call
        if (i - wbase >= 32) {
            wbase += 32;
            waddr = wnext;
            wnext = wbase + 32 + lane < nm ? unit_addr_tagged<WIN>(p, pre, lens, unit_of(wbase + 32 + lane), HK) : 0ull;
        }
        const unsigned long long src = __shfl_sync(0xffffffffu, waddr, i - wbase);
        if (lane == 0) {
            uaddr[st] = src;
            const uint32_t bar = bar0 + 8 * st;
            mbar_arrive_expect_tx(bar, ubytes);
            bulk_g2s_hint(ring0 + st * ubytes, reinterpret_cast<const void*>(src & ~1ull), ubytes, bar, l2_stream);
        }
        ++issued;
    };
    // The q rows of segment (sb, shg) into q buffer k & 1 (thread 0), and in the decode step,
    // when the segment's new token lands in a page this call streams, that token's K and V
    // rows of the segment's HK kv heads after them (rows ns .. ns + 2 HK - 1): the warp that
    // streams the page quantizes them from there, instead of loading them from global memory
    // in the middle of the stream, where a load waits behind the SM's page copies in flight.
    const uint32_t q_bytes = static_cast<uint32_t>(p.ns) * D * 2;
    auto issue_q = [&](int sb, int shg, int k) {
        const uint32_t bar = qbar0 + 8 * (k & 1);
        __half* dst = qbuf + (k & 1) * kQRows * D;
        const bool rows = !I8 && seg_append<WIN>(p, pre, lens, aps, sb) >= 0;
        const uint32_t r_bytes = HK * D * 2;
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, q_bytes + (rows ? 2 * r_bytes : 0));
        bulk_g2s(smem_u32(dst), p.q + (static_cast<long long>(sb) * p.Hq + shg * p.ns) * D, q_bytes, bar);
        if (rows) {
            const long long row = static_cast<long long>(sb) * p.Hkv + static_cast<long long>(shg) * HK;
            bulk_g2s(smem_u32(dst + p.ns * D), p.k_new + row * D, r_bytes, bar);
            bulk_g2s(smem_u32(dst + (p.ns + HK) * D), p.v_new + row * D, r_bytes, bar);
        }
    };
    // the first segment's q rows (read-only input) can move before the wait, unless the kernel
    // ahead on the stream writes them (q_after_wait) or the decode step appends (its K and V
    // rows may be written by that kernel)
    const bool q_late = p.q_after_wait || p.k_new != nullptr;
    auto issue_first_q = [&]() {
        int b0 = find_seq(pre, p.B, p.Hg, c0);
        const int np0 = pre[b0 + 1] - pre[b0];
        const int hg0 = static_cast<int>(div_nn(c0 - static_cast<long long>(p.Hg) * pre[b0], np0));
        if (threadIdx.x == 0) issue_q(b0, hg0, 0);
    };
    if (!q_late) issue_first_q();

    // ---- from here on the pool, the output and the workspace are used ----
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (q_late) issue_first_q();
    publish_prefix();
    orphan_appends();
    {
        const int pro = nm < stages ? nm : stages;
        if (p.withhold != 0 && lane == 0 && pro > 0) mbar_expect_tx(bar0, p.withhold);  // before the copy is issued
        for (int k = 0; k < pro; ++k) issue(k, k);
    }

    uint32_t qb[KSTEPS][NTQ][2];
    float q8[NTQ][2];  // kOff * the sum of q over the group of this thread's score columns 2c, 2c + 1,
                       // times softmax_scale * log2 e
    const float s24 = 16777216.0f * p.scale_log2;  // 2^24 * softmax_scale * log2 e
    float m[HS], l[HS];
    float o[MT][HS][4];
    int Leff = 0;  // positions of the segment's sequence (clamped to its block table)
    int wlo = 0;   // its first window position (0: all attended)
    SeqSpan sspan{};  // attended positions and listed pages of the segment's sequence

    // the kv head (within the unit) of this thread's score slot, and of its B-fragment
    // column (HK > 1 only when every slot is its own kv head)
    const int a_row = HK == 1 ? 0 : c;
    const int a_col = HK == 1 ? 0 : (g >> 1);
    // per-thread byte offsets inside a unit buffer (chunk 0)
    const int k_off = g * ROW + c * (KW * 4);
    const int ks_off = a_row * bbytes + l_kscales + g * NGK * SB;
    const int vs_off = a_row * bbytes + l_vscales + g * NGV * SB;
    const int v_off = l_vcodes + c * ROW + g * (I8 ? 16 : VB);
    const int src0 = 4 * c + (g >> 1);
    const int src1 = 4 * (c + 4) + (g >> 1);
    const bool want_lo = (g & 1) != 0;

    // One step: TG 16-token chunks, chunk X being chunk chk[X] of the unit buffer blk[X]
    // and holding sequence positions t0[X] .. t0[X] + 15, each over the HK kv heads of the
    // unit.  With MASKED, positions at or past Leff (and all of chunk X when !live[X]) are
    // excluded; without it every position is valid.
    auto process = [&](auto masked, const Step<TG>& in) {
        constexpr bool MASKED = decltype(masked)::value;
        const uint8_t* const* blk = in.blk;
        const int* chk = in.chk;
        const int* t0 = in.t0;
        const bool* live = in.live;
        bool vg[TG], vg8[TG];
        if (MASKED) {
#pragma unroll
            for (int X = 0; X < TG; ++X) {
                const int ta = t0[X] + g, tb = ta + 8;
                vg[X] = live[X] && ta < Leff && (!WIN || ta >= wlo || ta < p.sinks);
                vg8[X] = live[X] && tb < Leff && (!WIN || tb >= wlo || tb < p.sinks);
            }
        }

        // -------- scores: S = K . Q (per k-group columns), one MMA chain per chunk and head --------
        float acc[TG][HK][NTQ][4];
        {
            uint32_t kg[TG][HK][KW], kg8[TG][HK][KW];
#pragma unroll
            for (int X = 0; X < TG; ++X)
#pragma unroll
                for (int a = 0; a < HK; ++a) {
                    const uint8_t* kb = blk[X] + a * bbytes + chk[X] * 16 * ROW + k_off;
                    if constexpr (KW == 2) {
                        const uint2 x0 = *reinterpret_cast<const uint2*>(kb);
                        const uint2 x1 = *reinterpret_cast<const uint2*>(kb + 8 * ROW);
                        kg[X][a][0] = x0.x; kg[X][a][1] = x0.y;
                        kg8[X][a][0] = x1.x; kg8[X][a][1] = x1.y;
                    } else {
#pragma unroll
                        for (int w4 = 0; w4 < KW / 4; ++w4) {
                            const uint4 x0 = *reinterpret_cast<const uint4*>(kb + 16 * w4);
                            const uint4 x1 = *reinterpret_cast<const uint4*>(kb + 8 * ROW + 16 * w4);
                            kg[X][a][4 * w4 + 0] = x0.x; kg[X][a][4 * w4 + 1] = x0.y;
                            kg[X][a][4 * w4 + 2] = x0.z; kg[X][a][4 * w4 + 3] = x0.w;
                            kg8[X][a][4 * w4 + 0] = x1.x; kg8[X][a][4 * w4 + 1] = x1.y;
                            kg8[X][a][4 * w4 + 2] = x1.z; kg8[X][a][4 * w4 + 3] = x1.w;
                        }
                    }
#pragma unroll
                    for (int t = 0; t < NTQ; ++t)
                        acc[X][a][t][0] = acc[X][a][t][1] = acc[X][a][t][2] = acc[X][a][t][3] = 0.f;
                }
            if constexpr (I8) {
                // word j of a row is k-step j: its bytes' codes c, as c + 128, become the f16
                // subnormals (c + 128) * 2^-24 (bytes 0, 1 and bytes 2, 3 paired)
#pragma unroll
                for (int j = 0; j < KW; ++j)
#pragma unroll
                    for (int X = 0; X < TG; ++X) {
                        const uint32_t x = kg[X][0][j] ^ 0x80808080u, y = kg8[X][0][j] ^ 0x80808080u;
                        const uint32_t a0 = prmt(x, 0u, 0x5140u), a1 = prmt(y, 0u, 0x5140u);
                        const uint32_t a2 = prmt(x, 0u, 0x7362u), a3 = prmt(y, 0u, 0x7362u);
#pragma unroll
                        for (int t = 0; t < NTQ; ++t) mma_f16_16816(acc[X][0][t], a0, a1, a2, a3, qb[j][t][0], qb[j][t][1]);
                    }
            } else {
#pragma unroll
                for (int wi = 0; wi < KW; ++wi)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
#pragma unroll
                        for (int X = 0; X < TG; ++X)
#pragma unroll
                            for (int a = 0; a < HK; ++a) {
                                // nibbles of bytes e and e + 2 as f16 subnormals: the low ones
                                // n * 2^-24, the high ones 16 n * 2^-24
                                const uint32_t x = kg[X][a][wi] >> (8 * e);
                                const uint32_t y = kg8[X][a][wi] >> (8 * e);
                                const uint32_t a0 = x & 0x000F000Fu, a1 = y & 0x000F000Fu;
                                const uint32_t a2 = x & 0x00F000F0u, a3 = y & 0x00F000F0u;
#pragma unroll
                                for (int t = 0; t < NTQ; ++t)
                                    mma_f16_16816(acc[X][a][t], a0, a1, a2, a3, qb[2 * wi + e][t][0],
                                                  qb[2 * wi + e][t][1]);
                            }
            }
        }
        float z[TG][HS][2];
#pragma unroll
        for (int X = 0; X < TG; ++X) {
            // this thread's slot lives in the accumulator of kv head a_row
            float sacc[NTQ][4];
#pragma unroll
            for (int t = 0; t < NTQ; ++t)
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float v = acc[X][0][t][k];
#pragma unroll
                    for (int a = 1; a < HK; ++a) v = a_row == a ? acc[X][a][t][k] : v;
                    sacc[t][k] = v;
                }
            const uint8_t* s0 = blk[X] + chk[X] * 16 * NGK * SB + ks_off;
            float skg[NGK], skg8[NGK];
            load_scales<I8, NGK>(s0, skg, skg8);
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                float z0 = 0.f, z1 = 0.f;
#pragma unroll
                for (int R = 0; R < NGK; ++R) {
                    // the group's code dot product sum (n - off) q = 2^24 S - off sum q
                    const int pi = s * NGK + R;
                    // (times softmax_scale * log2 e, folded into both terms)
                    const float qo = q8[pi >> 1][pi & 1];
                    z0 = fmaf(skg[R], fmaf(sacc[pi >> 1][pi & 1], s24, -qo), z0);
                    z1 = fmaf(skg8[R], fmaf(sacc[pi >> 1][2 + (pi & 1)], s24, -qo), z1);
                }
                z[X][s][0] = z0;
                z[X][s][1] = z1;
                if (MASKED) {
                    z[X][s][0] = vg[X] ? z[X][s][0] : -INFINITY;
                    z[X][s][1] = vg8[X] ? z[X][s][1] : -INFINITY;
                }
            }
        }

        // -------- online softmax over the step's positions (per slot, lanes with the same c) --------
        // The slot's maximum over the step is reduced across lanes only when some lane holds a
        // score above the running maximum; otherwise the reduced value could not raise it, and
        // the running maximum stays as it is (most steps once a segment is under way).
        float cm[HS];
        bool up = false;
#pragma unroll
        for (int s = 0; s < HS; ++s) {
            cm[s] = fmaxf(z[0][s][0], z[0][s][1]);
#pragma unroll
            for (int X = 1; X < TG; ++X) cm[s] = fmaxf(cm[s], fmaxf(z[X][s][0], z[X][s][1]));
            up |= cm[s] > m[s];
        }
        if (__any_sync(0xffffffffu, up)) {
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                float r = cm[s];
                r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, 4));
                r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, 8));
                r = fmaxf(r, __shfl_xor_sync(0xffffffffu, r, 16));
                const float mn = fmaxf(m[s], r);
                const float alpha = fast_exp2(m[s] - mn);
                l[s] *= alpha;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mt][s][e] *= alpha;
                m[s] = mn;
            }
        }
        float pr[TG][HS][2];
#pragma unroll
        for (int s = 0; s < HS; ++s) {
#pragma unroll
            for (int X = 0; X < TG; ++X) {
                pr[X][s][0] = fast_exp2(z[X][s][0] - m[s]);
                pr[X][s][1] = fast_exp2(z[X][s][1] - m[s]);
                l[s] += pr[X][s][0] + pr[X][s][1];
            }
        }

        // -------- weights W = p * v_scale as f16 hi + lo, moved into B fragments --------
        uint32_t bv[TG][HS][NGV][2];
#pragma unroll
        for (int X = 0; X < TG; ++X) {
            const uint8_t* s0 = blk[X] + chk[X] * 16 * NGV * SB + vs_off;
            float svg[NGV], svg8[NGV];
            load_scales<I8, NGV>(s0, svg, svg8);
#pragma unroll
            for (int s = 0; s < HS; ++s) {
#pragma unroll
                for (int R = 0; R < NGV; ++R) {
                    float w0 = pr[X][s][0] * svg[R];
                    float w1 = pr[X][s][1] * svg8[R];
                    if (MASKED) {
                        w0 = vg[X] ? w0 : 0.f;  // a masked slot's scale may be any bit pattern
                        w1 = vg8[X] ? w1 : 0.f;
                    }
                    const uint32_t phi = pack_h2(w0, w1);
                    const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&phi));
                    const uint32_t plo = pack_h2(w0 - back.x, w1 - back.y);
                    const uint32_t x0 = __shfl_sync(0xffffffffu, phi, src0);
                    const uint32_t y0 = __shfl_sync(0xffffffffu, plo, src0);
                    const uint32_t x1 = __shfl_sync(0xffffffffu, phi, src1);
                    const uint32_t y1 = __shfl_sync(0xffffffffu, plo, src1);
                    bv[X][s][R][0] = want_lo ? y0 : x0;
                    bv[X][s][R][1] = want_lo ? y1 : x1;
                }
            }
        }

        // -------- output: O^T += V^T . W, every chunk and kv head --------
#pragma unroll
        for (int X = 0; X < TG; ++X)
#pragma unroll
            for (int a = 0; a < HK; ++a)
#pragma unroll
                for (int R = 0; R < NGV; ++R) {
                    // B fragment of kv head a: the columns of other heads' slots are zero
                    uint32_t b0[HS], b1[HS];
#pragma unroll
                    for (int s = 0; s < HS; ++s) {
                        b0[s] = (HK == 1 || a_col == a) ? bv[X][s][R][0] : 0u;
                        b1[s] = (HK == 1 || a_col == a) ? bv[X][s][R][1] : 0u;
                    }
                    if constexpr (I8) {
                        // this thread's 16 bytes of the rows of tokens c, c + 8, c + 4, c + 12;
                        // m-tile mt takes bytes 2 mt (rows g) and 2 mt + 1 (rows g + 8), a code c
                        // as the exact f16 integer (1024 + c + 128) - 1152
                        const uint8_t* vcodes = blk[X] + chk[X] * 16 * ROW + v_off;
                        const uint4 ta = *reinterpret_cast<const uint4*>(vcodes);
                        const uint4 tb = *reinterpret_cast<const uint4*>(vcodes + 8 * ROW);
                        const uint4 tc = *reinterpret_cast<const uint4*>(vcodes + 4 * ROW);
                        const uint4 td = *reinterpret_cast<const uint4*>(vcodes + 12 * ROW);
                        const uint32_t va[4] = {ta.x, ta.y, ta.z, ta.w}, vb[4] = {tb.x, tb.y, tb.z, tb.w};
                        const uint32_t vc[4] = {tc.x, tc.y, tc.z, tc.w}, vd[4] = {td.x, td.y, td.z, td.w};
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const uint32_t bo = 2u * static_cast<uint32_t>(mt % 2);
                            const uint32_t sel = bo | ((bo + 4) << 4) | ((bo + 1) << 8) | ((bo + 5) << 12);
                            const uint32_t tac = prmt(va[mt / 2], vb[mt / 2], sel) ^ 0x80808080u;  // tokens c, c+8
                            const uint32_t tbd = prmt(vc[mt / 2], vd[mt / 2], sel) ^ 0x80808080u;  // c+4, c+12
                            const uint32_t a0 = h2_sub(prmt(tac, 0x64646464u, 0x5140u), 0x64806480u);
                            const uint32_t a1 = h2_sub(prmt(tac, 0x64646464u, 0x7362u), 0x64806480u);
                            const uint32_t a2 = h2_sub(prmt(tbd, 0x64646464u, 0x5140u), 0x64806480u);
                            const uint32_t a3 = h2_sub(prmt(tbd, 0x64646464u, 0x7362u), 0x64806480u);
#pragma unroll
                            for (int s = 0; s < HS; ++s) mma_f16_16816(o[mt][s], a0, a1, a2, a3, b0[s], b1[s]);
                        }
                        continue;
                    }
                    uint32_t va[(VB + 3) / 4], vb[(VB + 3) / 4], vc[(VB + 3) / 4], vd[(VB + 3) / 4];
                    const uint8_t* vcodes = blk[X] + a * bbytes + chk[X] * 16 * ROW + v_off + R * (GV / 2);
                    if constexpr (VB == 8) {
                        const uint2 ta = *reinterpret_cast<const uint2*>(vcodes);
                        const uint2 tb = *reinterpret_cast<const uint2*>(vcodes + 8 * ROW);
                        const uint2 tc = *reinterpret_cast<const uint2*>(vcodes + 4 * ROW);
                        const uint2 td = *reinterpret_cast<const uint2*>(vcodes + 12 * ROW);
                        va[0] = ta.x; va[1] = ta.y; vb[0] = tb.x; vb[1] = tb.y;
                        vc[0] = tc.x; vc[1] = tc.y; vd[0] = td.x; vd[1] = td.y;
                    } else if constexpr (VB == 4) {
                        va[0] = *reinterpret_cast<const uint32_t*>(vcodes);
                        vb[0] = *reinterpret_cast<const uint32_t*>(vcodes + 8 * ROW);
                        vc[0] = *reinterpret_cast<const uint32_t*>(vcodes + 4 * ROW);
                        vd[0] = *reinterpret_cast<const uint32_t*>(vcodes + 12 * ROW);
                    } else {
                        va[0] = *reinterpret_cast<const uint16_t*>(vcodes);
                        vb[0] = *reinterpret_cast<const uint16_t*>(vcodes + 8 * ROW);
                        vc[0] = *reinterpret_cast<const uint16_t*>(vcodes + 4 * ROW);
                        vd[0] = *reinterpret_cast<const uint16_t*>(vcodes + 12 * ROW);
                    }
#pragma unroll
                    for (int jb = 0; jb < VB; jb += 2) {
                        const int wi = jb / 4;
                        const uint32_t bb = static_cast<uint32_t>(jb % 4);
                        const uint32_t sel = bb | ((bb + 1) << 4) | ((bb + 4) << 8) | ((bb + 5) << 12);
                        const int mt0 = R * VB + jb;
                        const uint32_t yac = prmt(va[wi], vb[wi], sel);  // tokens c, c+8
                        const uint32_t ybd = prmt(vc[wi], vd[wi], sel);  // tokens c+4, c+12
                        {
                            const uint32_t a0 = unpack_lo(yac), a1 = unpack_hi(yac);
                            const uint32_t a2 = unpack_lo(ybd), a3 = unpack_hi(ybd);
#pragma unroll
                            for (int s = 0; s < HS; ++s) mma_f16_16816(o[mt0][s], a0, a1, a2, a3, b0[s], b1[s]);
                        }
                        {
                            const uint32_t y1 = yac >> 8, y2 = ybd >> 8;
                            const uint32_t a0 = unpack_lo(y1), a1 = unpack_hi(y1);
                            const uint32_t a2 = unpack_lo(y2), a3 = unpack_hi(y2);
#pragma unroll
                            for (int s = 0; s < HS; ++s) mma_f16_16816(o[mt0 + 1][s], a0, a1, a2, a3, b0[s], b1[s]);
                        }
                    }
                }
    };

    // ---- walk the segments this CTA's slice touches ----
    int b = find_seq(pre, p.B, p.Hg, c0);
    int np = pre[b + 1] - pre[b];
    int hg = static_cast<int>(div_nn(c0 - static_cast<long long>(p.Hg) * pre[b], np));
    long long sfirst = static_cast<long long>(p.Hg) * pre[b] + static_cast<long long>(hg) * np;
    int consumed = 0;     // this warp's units taken out of the ring
    int cst = 0;          // stage of the next unit to consume
    uint32_t cpar = 0;    // its phase parity
    bool failed = false;  // a copy did not arrive in time: stop waiting, keep the barriers
    int f_st = 0, f_out = 0;  // where consumption stopped, and the copies still in flight then
    uint32_t f_par = 0;
    int f_consumed = 0;   // units consumed when it stopped
    constexpr bool p16 = P16;

    // q rows of a segment go to shared memory by a bulk copy issued one segment ahead
    // (thread 0, issue_q above); segment k of this CTA uses buffer k & 1 at phase (k >> 1) & 1
    // the segment after (sb, shg), skipping sequences without positions; sb == B when none
    auto next_seg = [&](int& sb, int& shg) {
        if (++shg == p.Hg) {
            shg = 0;
            do {
                ++sb;
            } while (sb < p.B && pre[sb + 1] == pre[sb]);
        }
    };
    int segk = 0;  // segments of this CTA started so far (segment 0's q copy is already issued)
    int apg_seg = -1;  // page index (within the segment's sequence) of its append, if streamed here
    bool my_app = false;  // this warp streams that page: it keeps the q buffer (which holds the
                          // token's K and V rows) until it has quantized them

    while (sfirst < c1) {
        const long long ua = sfirst > c0 ? sfirst : c0;
        const long long ue = sfirst + np < c1 ? sfirst + np : c1;
        const long long fu = ua + (((c0 + warp - ua) % kWarps) + kWarps) % kWarps;  // my first unit here
        const int cnt = fu < ue ? static_cast<int>((ue - fu + kWarps - 1) / kWarps) : 0;
        const int pg0 = static_cast<int>(fu - sfirst);
        my_app = false;

        // the next segment's q rows start moving now, into the buffer of segment segk - 1
        // once every warp has taken its fragments out of it
        if (threadIdx.x == 0 && sfirst + np < c1) {
            int nb = b, nhg = hg;
            next_seg(nb, nhg);
            if (segk >= 1 && !mbar_wait(qfree0 + 8 * ((segk - 1) & 1), ((segk - 1) >> 1) & 1, p.wait_ns))
                raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
            issue_q(nb, nhg, segk + 1);
        }
        // Every warp waits for the segment's q copy, units here or not: that copy is issued
        // only once every warp has released the buffer two segments back, so no warp can
        // arrive on a qfree barrier while the phase of two segments back is still open.
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(qbar0 + 8 * (segk & 1), (segk >> 1) & 1, p.wait_ns))) {
            if (lane == 0) raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
            failed = true;
            f_st = cst;
            f_par = cpar;
            f_out = issued - consumed;
            f_consumed = consumed;
        }
        if (cnt > 0) {
            // new (sequence, head group): q fragments and a fresh softmax state
            if constexpr (WIN) {
                sspan = seq_span(lens[b], p.lg_p, p.max_blocks, p.window, p.sinks);
                Leff = sspan.L;
                wlo = sspan.wlo;
            } else {
                Leff = min(lens[b], p.max_blocks * p.P);
            }
            apg_seg = -1;
            if constexpr (!I8) {
                apg_seg = seg_append<WIN>(p, pre, lens, aps, b);
                if (apg_seg >= 0) {
                    // its unit, and whether it is one of this warp's (units fu, fu + kWarps, ... < ue)
                    const long long u = sfirst + (WIN ? span_index(sspan, apg_seg) : apg_seg);
                    my_app = u >= fu && u < ue && (u - fu) % kWarps == 0;
                }
            }
            const __half* qseg = qbuf + (segk & 1) * kQRows * D;
#pragma unroll
            for (int t = 0; t < NTQ; ++t) {
                const int pi = 2 * t + (g & 1);
                const int sigma = pi / NGK;
                const int R = pi % NGK;
                const int j = (g >> 1) + 4 * sigma;
                const bool colv = sigma < HS && j < p.ns;
                const __half* qrow = qseg + (colv ? j : 0) * D;
                float qs = 0.f;  // this thread's part of the column's sum of q
                if constexpr (I8) {
                    // k-step j: dimensions c (D / 4) + 4 j .. + 3, in order
#pragma unroll
                    for (int j = 0; j < KW; ++j) {
                        uint2 w2 = make_uint2(0, 0);
                        if (colv) w2 = *reinterpret_cast<const uint2*>(qrow + c * (D / 4) + 4 * j);
                        const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w2.x));
                        const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w2.y));
                        qs += f0.x + f0.y + f1.x + f1.y;
                        qb[j][t][0] = w2.x;
                        qb[j][t][1] = w2.y;
                    }
                }
#pragma unroll
                for (int wi = 0; wi < (I8 ? 0 : KW); ++wi) {
                    const int dbase = c * (D / 4) + 8 * wi;
                    uint4 w4 = make_uint4(0, 0, 0, 0);
                    if (colv && dbase / GK == R) w4 = *reinterpret_cast<const uint4*>(qrow + dbase);
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&(&w4.x)[h]));
                        qs += f.x + f.y;
                    }
                    // the entries meeting high nibbles (odd dimensions) are divided by 16
                    qb[2 * wi][t][0] = prmt(w4.x, w4.z, 0x5410u);
                    qb[2 * wi][t][1] = h2_mul(prmt(w4.x, w4.z, 0x7632u), 0x2C002C00u /* 1/16 */);
                    qb[2 * wi + 1][t][0] = prmt(w4.y, w4.w, 0x5410u);
                    qb[2 * wi + 1][t][1] = h2_mul(prmt(w4.y, w4.w, 0x7632u), 0x2C002C00u);
                }
                // column g of n-tile t: its sum over the row group's four threads; this
                // thread's score columns 2c and 2c + 1 are those of the threads with g = 2c, 2c + 1
                qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                q8[t][0] = (kOff * p.scale_log2) * __shfl_sync(0xffffffffu, qs, 8 * c);
                q8[t][1] = (kOff * p.scale_log2) * __shfl_sync(0xffffffffu, qs, 8 * c + 4);
            }
        }
        // this warp is done with the segment's q buffer (a warp with units here has waited
        // for its copy, so the buffer is only reused after the copy has landed); the warp
        // that appends the segment's token releases it after the append
        __syncwarp();
        if (lane == 0 && !my_app) mbar_arrive(qfree0 + 8 * (segk & 1));
#pragma unroll
        for (int s = 0; s < HS; ++s) {
            m[s] = -INFINITY;
            l[s] = 0.f;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) o[mt][s][e] = 0.f;
        }

        for (int j = 0; j < cnt;) {
            // HK = 1 with 16-token pages: two units per step when there are two
            const int n = (HK == 1 && p16 && j + 1 < cnt) ? 2 : 1;
            int st1 = cst;
            uint32_t par1 = cpar;
            if (n == 2 && ++st1 == stages) {
                st1 = 0;
                par1 ^= 1u;
            }
            if (!failed) {
                bool ok = mbar_wait(bar0 + 8 * cst, cpar, p.wait_ns);
                if (n == 2) ok = ok && mbar_wait(bar0 + 8 * st1, par1, p.wait_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    if (lane == 0) raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
                    failed = true;
                    f_st = cst;
                    f_par = cpar;
                    f_out = issued - consumed;
                    f_consumed = consumed;
                }
            }
            if (!failed) {
                const uint8_t* blkA = ring + cst * ubytes;
                const uint8_t* blkB = ring + st1 * ubytes;
                const int pg = pg0 + kWarps * j;
                // pages of the two units (list indices past a window gap skip it)
                const int rA = WIN ? span_page(sspan, pg) : pg;
                const int rB = WIN ? span_page(sspan, pg + kWarps) : pg + kWarps;
                // the page taking this step's appended token: the token is quantized from the
                // rows copied with q, written to the pool (the unit's address was kept when its
                // copy was issued) and patched into the staged copy before the page is used
                if constexpr (!I8)
                    if (my_app && (rA == apg_seg || (n == 2 && rB == apg_seg))) {
                        const int ast = rA == apg_seg ? cst : st1;
                        const unsigned long long ga = uaddr[ast];
                        const __half* arow = qbuf + (segk & 1) * kQRows * D + p.ns * D;
                        if ((ga & 1ull) == 0)  // a bad page id: no append (flagged at its lookup)
                            append_rows<D, HK>(p, arow, arow + HK * D,
                                               p.pool_w + (ga - reinterpret_cast<unsigned long long>(p.pool)),
                                               ring + ast * ubytes, aps[b] & ((1 << p.lg_p) - 1));
                        __syncwarp();
                        if (lane == 0) mbar_arrive(qfree0 + 8 * (segk & 1));
                        my_app = false;
                    }
                // every position of [t, t + w) attended, and some of it attended
                auto all_in = [&](int t, int w) { return t + w <= Leff && (!WIN || t >= wlo || t + w <= p.sinks); };
                auto any_in = [&](int t, int w) { return !WIN || (min(t + w, Leff) > wlo || t < p.sinks); };
                if constexpr (HK == 1) {
                    if constexpr (P16) {
                        const int t0A = rA * 16, t0B = rB * 16;
                        const Step<TG> st = {{blkA, blkB}, {0, 0}, {t0A, t0B}, {true, n == 2}};
                        // (without a window, page B comes after page A, so B whole implies A whole)
                        if (n == 2 && (WIN ? all_in(t0A, 16) && all_in(t0B, 16) : t0B + 16 <= Leff))
                            process(std::false_type{}, st);
                        else process(std::true_type{}, st);
                    } else {
                        for (int chunk = 0; chunk < p.P / 16; chunk += 2) {
                            const int t0 = rA * p.P + chunk * 16;
                            if (t0 >= Leff) break;
                            // an odd last chunk pairs with a re-read of itself, masked out
                            const bool two = chunk + 1 < p.P / 16;
                            if (!any_in(t0, two ? 32 : 16)) continue;  // wholly before the window
                            const Step<TG> st = {{blkA, blkA}, {chunk, two ? chunk + 1 : chunk}, {t0, t0 + 16}, {true, two}};
                            if (two && all_in(t0, 32)) process(std::false_type{}, st);
                            else process(std::true_type{}, st);
                        }
                    }
                } else {
                    for (int chunk = 0; chunk < p.P / 16; ++chunk) {
                        const int t0 = rA * p.P + chunk * 16;
                        if (t0 >= Leff) break;
                        if (!any_in(t0, 16)) continue;  // wholly before the window
                        const Step<TG> st = {{blkA}, {chunk}, {t0}, {true}};
                        if (all_in(t0, 16)) process(std::false_type{}, st);
                        else process(std::true_type{}, st);
                    }
                }
            }

            // ---- release the stages and refill them with the units `stages` ahead ----
            if (!failed) {
                __syncwarp();
                if (lane == 0) fence_proxy_async_smem();
                if (consumed + stages < nm) issue(consumed + stages, cst);
                if (n == 2 && consumed + 1 + stages < nm) issue(consumed + 1 + stages, st1);
            }
            consumed += n;
            cst = st1;
            cpar = par1;
            if (++cst == stages) {
                cst = 0;
                cpar ^= 1u;
            }
            j += n;
        }

        // ---- segment end: this warp's part of the segment goes out as one partial ----
        // (running max and sum per slot, unnormalised output per slot), at index
        // kWarps * (CTA + segment) + warp; the combine kernel merges them.  No other warp
        // is waited for, so a warp that reaches the end early keeps streaming.
        {
            const long long seg = static_cast<long long>(b) * p.Hg + hg;
            const long long piece = static_cast<long long>(kWarps) * (cta + seg) + warp;
            float lt[HS];
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                lt[s] = l[s];
                lt[s] += __shfl_xor_sync(0xffffffffu, lt[s], 4);
                lt[s] += __shfl_xor_sync(0xffffffffu, lt[s], 8);
                lt[s] += __shfl_xor_sync(0xffffffffu, lt[s], 16);
            }
            if (cnt > 0 && !failed) {
                // straight from the accumulators: thread (g, c) holds dimensions dd, dd + 1 of
                // slot c for each P.V tile; its VB tiles of a V group give it 2 VB consecutive
                // floats and thread (g + 1, c) continues them, so every 32-byte sector of a row
                // is written whole by one store instruction or by one thread's stores in a row.
                // (Staging the rows through a ring stage for 16-byte stores kept that stage
                // from being refilled until the partial was out: a gap in the ring at every
                // segment end.)
#pragma unroll
                for (int s = 0; s < HS; ++s) {
                    const int nsr = min(4, p.ns - 4 * s);  // slots in this round
                    if (c < nsr) {
                        float* orow = p.ws_o + (piece * p.ns + 4 * s + c) * D;
#pragma unroll
                        for (int R = 0; R < NGV; ++R)
#pragma unroll
                            for (int jb = 0; jb < VB; ++jb) {
                                const int mt = R * VB + jb;
                                const int dd = 2 * (R * (GV / 2) + g * VB + jb);
                                *reinterpret_cast<float2*>(orow + dd) =
                                    make_float2(o[mt][s][0] + o[mt][s][1], o[mt][s][2] + o[mt][s][3]);
                            }
                    }
                    if (g == 0 && c < nsr)
                        *reinterpret_cast<float2*>(p.ws_ml + (piece * p.ns + 4 * s + c) * 2) = make_float2(m[s], lt[s]);
                }
            } else {
                // no units of this segment here (or a failed wait): an empty partial
                if (lane < p.ns)
                    *reinterpret_cast<float2*>(p.ws_ml + (piece * p.ns + lane) * 2) = make_float2(-INFINITY, 0.f);
                for (int k = 0; k < p.ns; ++k)
#pragma unroll
                    for (int f = lane; f < D / 4; f += 32)
                        reinterpret_cast<float4*>(p.ws_o + (piece * p.ns + k) * D)[f] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }

        // a warp that was to append but did not (a failed wait) releases the q buffer now
        if (my_app) {
            __syncwarp();
            if (lane == 0) mbar_arrive(qfree0 + 8 * (segk & 1));
            my_app = false;
        }

        // ---- next segment ----
        ++segk;
        sfirst += np;
        if (++hg == p.Hg) {
            hg = 0;
            do {
                ++b;
            } while (b < p.B && pre[b + 1] == pre[b]);
        }
        if (b < p.B) np = pre[b + 1] - pre[b];
        else break;
    }

    // ---- no q copy may still be landing when the CTA leaves (they all have, unless a
    // wait failed) ----
    if (threadIdx.x == 0) {
        for (int k = segk - 2; k < segk; ++k)
            if (k >= 0) mbar_wait(qbar0 + 8 * (k & 1), (k >> 1) & 1, p.wait_ns);
    }
    // ---- after a failed wait: let the copies already issued land before leaving ----
    if (failed) {
        // the withheld bytes of the first copy's phase, as a 16-byte copy of its own, so that
        // the phase completes once both copies have landed
        if (p.withhold != 0 && f_consumed == 0 && f_out > 0 && lane == 0)
            bulk_g2s(ring0, p.pool, p.withhold, bar0);
        int st = f_st;
        uint32_t par = f_par;
        for (int k = 0; k < f_out; ++k) {
            mbar_wait(bar0 + 8 * st, par, p.wait_ns);
            if (++st == stages) {
                st = 0;
                par ^= 1u;
            }
        }
    }
}

// Raise the kernel's dynamic shared-memory limit once to the largest size asked for,
// so repeated calls (and calls under stream capture) only launch.
template <int D, int GK, int GV, int HK, int HS, bool WIN, bool P16, int CODEC = 0>
cudaError_t ensure_smem_attr(size_t smem) {
    static std::atomic<long long> granted{-1};
    if (static_cast<long long>(smem) <= granted.load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(decode_splitkv_kernel<D, GK, GV, HK, HS, WIN, P16, CODEC>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) cudaGetLastError();  // a refused size must not linger as the last error
    if (err == cudaSuccess) {
        long long cur = granted.load();
        while (static_cast<long long>(smem) > cur && !granted.compare_exchange_weak(cur, static_cast<long long>(smem))) {
        }
    }
    return err;
}

// Resident CTAs per SM for a given shared-memory size, memoised per size (a few sizes
// per shape are asked for; the slots fill once and later calls only read them).
template <int D, int GK, int GV, int HK, int HS, bool WIN, bool P16, int CODEC = 0>
int occupancy(size_t smem) {
    constexpr int kSlots = 32;
    static std::atomic<long long> memo[kSlots];  // (smem << 8) | ctas, 0 = empty
    for (int i = 0; i < kSlots; ++i) {
        const long long m = memo[i].load(std::memory_order_acquire);
        if (m == 0) break;
        if ((m >> 8) == static_cast<long long>(smem)) return static_cast<int>(m & 0xff);
    }
    if (ensure_smem_attr<D, GK, GV, HK, HS, WIN, P16, CODEC>(smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_splitkv_kernel<D, GK, GV, HK, HS, WIN, P16, CODEC>, cta_warps<HS>() * 32,
                                                      smem) != cudaSuccess)
        return 0;
    const long long entry = (static_cast<long long>(smem) << 8) | (n & 0xff);
    for (int i = 0; i < kSlots; ++i) {
        long long expect = 0;
        if (memo[i].compare_exchange_strong(expect, entry) || expect == entry) break;
    }
    return n;
}

template <int D, int GK, int GV, int HK, int HS, bool WIN, bool P16, int CODEC = 0>
cudaError_t run(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    KParams p;
    p.pool = a.pool;
    p.q = a.q;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.ws_ml = reinterpret_cast<float*>(a.workspace + plan.ws_ml_offset);
    p.ws_o = reinterpret_cast<float*>(a.workspace + plan.ws_o_offset);
    p.ws_pre = reinterpret_cast<int32_t*>(a.workspace + plan.ws_pre_offset);
    p.status = a.status ? a.status : reinterpret_cast<uint32_t*>(a.workspace);
    p.len_sub = a.len_sub;
    p.wait_ns = a.wait_ns != 0 ? a.wait_ns : kWaitLimitNs;
    p.withhold = a.withhold_first_copy ? 16u : 0u;
    p.q_after_wait = a.q_after_wait;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.Hg = a.Hkv / HK;
    p.r = a.Hq / a.Hkv;
    p.ns = HK * p.r;
    p.P = a.L.P;
    p.num_pages = a.num_pages;
    p.max_blocks = a.max_blocks;
    p.block_bytes = a.L.bytes;
    p.v_codes = a.L.v_codes;
    p.k_scales = a.L.k_scales;
    p.v_scales = a.L.v_scales;
    if (CODEC == 1) {  // the INT8 block: K codes, V codes (P x D bytes each), K and V scales (P fp32 each)
        p.block_bytes = 2 * a.L.P * D + 8 * a.L.P;
        p.v_codes = a.L.P * D;
        p.k_scales = 2 * a.L.P * D;
        p.v_scales = 2 * a.L.P * D + 4 * a.L.P;
    }
    p.unit_bytes = p.block_bytes * HK;
    p.stages = plan.stages;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.append_pos = a.append_pos;
    p.pool_w = a.pool_w;
    p.window = a.window;
    p.sinks = a.sinks;
    p.lg_p = 0;
    while ((1 << p.lg_p) < a.L.P) ++p.lg_p;
    p.lg_lk = 0;
    while ((8 << p.lg_lk) < a.L.Gk) ++p.lg_lk;
    p.lg_lv = 0;
    while ((8 << p.lg_lv) < a.L.Gv) ++p.lg_lv;
    cudaError_t err = ensure_smem_attr<D, GK, GV, HK, HS, WIN, P16, CODEC>(plan.smem_bytes);
    if (err != cudaSuccess) return err;
    // The launch may start before the kernel ahead of it on the stream finishes
    // (programmatic dependent launch); the kernel waits with griddepcontrol.wait before
    // it reads any input.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.ctas));
    cfg.blockDim = dim3(cta_warps<HS>() * 32);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<D, GK, GV, HK, HS, WIN, P16, CODEC>, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace decode

// Dispatch entry points, one per translation unit: per K group size for head_dim 128, per
// head_dim for 64 and 256 (the _win ones serve calls with a sliding window).
cudaError_t decode_run_gk32(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk64(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk128(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_gk32(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk64(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk128(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
cudaError_t decode_run_gk32_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk64_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk128_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_gk32_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk64_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk128_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
cudaError_t decode_run_d64(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_d64_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_d256(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_d256_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_d64(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_d64_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_d256(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_d256_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);

}  // namespace kvq

// Dispatch key of an instance: K and V group sizes, unit shape (HK kv heads, HS query-head
// slots per thread) and whether pages hold 16 tokens.
#define KVQ_DECODE_KEY(GK, GV, HK, HS, P16) (((GK) << 13) + (GV) * 32 + (HK) * 8 + (HS) * 2 + (P16))
// The instances of one (head_dim D_, GK_, GV_): the three unit shapes (HK, HS) in
// {(1, 1), (1, 2), (4, 1)} and, for one-head units, 16-token pages or larger ones; W_
// selects the window instances.
#define KVQ_DECODE_CASES(D_, GK_, GV_, W_, CALL)                                                    \
    case KVQ_DECODE_KEY(GK_, GV_, 1, 1, 1): return CALL(D_, GK_, GV_, 1, 1, W_, true);              \
    case KVQ_DECODE_KEY(GK_, GV_, 1, 1, 0): return CALL(D_, GK_, GV_, 1, 1, W_, false);             \
    case KVQ_DECODE_KEY(GK_, GV_, 1, 2, 1): return CALL(D_, GK_, GV_, 1, 2, W_, true);              \
    case KVQ_DECODE_KEY(GK_, GV_, 1, 2, 0): return CALL(D_, GK_, GV_, 1, 2, W_, false);             \
    case KVQ_DECODE_KEY(GK_, GV_, 4, 1, 1): return CALL(D_, GK_, GV_, 4, 1, W_, true);
// Head_dim 256: one-head units with one query-head slot per thread only.
#define KVQ_DECODE_CASES_1H(D_, GK_, GV_, W_, CALL)                                                 \
    case KVQ_DECODE_KEY(GK_, GV_, 1, 1, 1): return CALL(D_, GK_, GV_, 1, 1, W_, true);              \
    case KVQ_DECODE_KEY(GK_, GV_, 1, 1, 0): return CALL(D_, GK_, GV_, 1, 1, W_, false);
#define KVQ_DECODE_RUN(D_, GK_, GV_, HK_, HS_, W_, P16_) decode::run<D_, GK_, GV_, HK_, HS_, W_, P16_>(a, plan, s)
#define KVQ_DECODE_OCC(D_, GK_, GV_, HK_, HS_, W_, P16_) decode::occupancy<D_, GK_, GV_, HK_, HS_, W_, P16_>(smem)
// One translation unit's entry points over the cases CASES(CALL) lists.
#define KVQ_DECODE_TU(CASES, RUN_NAME, OCC_NAME)                                                     \
    namespace kvq {                                                                                  \
    cudaError_t RUN_NAME(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s) {              \
        switch (KVQ_DECODE_KEY(a.L.Gk, a.L.Gv, plan.hk, plan.hs, a.L.P == 16 ? 1 : 0)) {             \
            CASES(KVQ_DECODE_RUN)                                                                    \
            default: return cudaErrorInvalidValue;                                                   \
        }                                                                                            \
    }                                                                                                \
    int OCC_NAME(const DecodeArgs& a, const DecodePlan& plan, size_t smem) {                         \
        switch (KVQ_DECODE_KEY(a.L.Gk, a.L.Gv, plan.hk, plan.hs, a.L.P == 16 ? 1 : 0)) {             \
            CASES(KVQ_DECODE_OCC)                                                                    \
            default: return 0;                                                                       \
        }                                                                                            \
    }                                                                                                \
    }
