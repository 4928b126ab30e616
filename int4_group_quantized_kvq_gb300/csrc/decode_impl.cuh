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
//  * Work is the flattened list of (sequence, kv head, page) units.  A persistent grid
//    of W warps (SM count x resident CTAs x 4) gives every warp an equal contiguous
//    slice, so ragged lengths and small batches still keep every SM busy.
//  * Each warp owns a ring of `stages` page buffers in shared memory, filled by 1-D
//    bulk copies (the TMA engine, cp.async.bulk) that complete on per-stage mbarriers.
//    A (page, head) block is contiguous (2144 bytes at d=128, P=16), so one copy moves
//    a whole page of K codes, V codes and scales.  Waits are bounded in time.
//  * The arithmetic runs on the tensor cores (mma.sync m16n8k16, f16 inputs, f32
//    accumulate), which keeps the per-element ALU work near one instruction: nibbles
//    become exact f16 integers in two instructions per pair, and the MMA does the
//    multiply-accumulate.  For a 16-token chunk:
//      scores  S[token, col] = K[token, :] . Qcol  with M = 16 tokens, N = 8 columns,
//              K-dim = head_dim.  Column (head, k-group) carries q masked to that group,
//              so each group's partial dot product comes out separately and is scaled
//              by its own fp16 scale afterwards (codes and q are exact in f16; products
//              and sums are fp32).
//      output  O^T[d, col] += V^T[d, token] . W[token, col] with M = 16 dims, N = 8
//              columns (head, hi|lo), K-dim = 16 tokens.  W = p * v_scale is split into
//              an f16 high part and an f16 remainder, two columns of the same MMA, which
//              keeps about 22 bits of the weight.  M-tiles never straddle a V group.
//    The score fragment of thread (g, c) holds tokens g, g+8 of head c (+4), and the
//    output fragment holds head c (+4) too, so the softmax rescale is thread-local;
//    only the weights are exchanged (four shuffles per chunk and V group).
//    Chunks are taken two at a time (two 16-token pages, or two chunks of a larger
//    page): the two score chains interleave and one softmax reduction covers both.
//  * Split combine, fused: a warp that finishes its part of a (sequence, kv head)
//    segment writes a partial (running max, running sum, unnormalised output), then
//    bumps a counter (fence + atomic add, never waiting on other warps; the result is
//    looked at one segment later so the round trip overlaps streaming).  The warp that
//    counted last merges: all partials of a segment spread over at most 32 warps, or,
//    for longer segments, its group of 32 partials into a level-2 partial, the last
//    group then merging those.  Counters return to zero for the next call.  A segment
//    covered by one warp is written directly from registers.
#pragma once

#include <cuda_fp16.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace decode {

constexpr int kWarps = 4;                         // warps per CTA
constexpr int kMergeFanIn = 32;                   // longest segment (in warps) merged in-kernel

// Per-warp values needed only at segment ends, kept in shared memory rather than in
// registers (the hot loop needs every register it can get).
struct WarpCtx {
    long long U, W, wid;
    int pend_kind, pend_b, pend_h, pend_gi, pend_target;
    int pad;
};
constexpr uint64_t kWaitLimitNs = 250000000ull;   // a page copy that takes 250 ms has failed

struct KParams {
    const uint8_t* pool;
    const __half* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* out;
    float* ws_ml;       // level-1 partials (one per warp and segment it touches): (max, sum)
    float* ws_o;        //   ... and unnormalised outputs
    float* ws_gml;      // level-2 partials (one per group of 32 warps of a long segment)
    float* ws_go;
    int32_t* counters;  // per segment; zero between calls
    int32_t* gcounters; // per group of a long segment; zero between calls
    uint32_t* status;
    int32_t B, Hq, Hkv, r, P, num_pages, max_blocks, block_bytes, stages;
    int32_t v_codes, k_scales, v_scales;
    float scale_log2;  // softmax_scale * log2(e)
};

// Exclusive prefix sums of pages per sequence into pre[0..B]; run by one warp.
__device__ __forceinline__ void page_prefix(const KParams& p, int32_t* pre, int lane) {
    int carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int b = b0 + lane;
        int np = 0;
        if (b < p.B) {
            int L = p.seq_lens[b];
            L = L < 0 ? 0 : L;
            long long npl = (static_cast<long long>(L) + p.P - 1) / p.P;
            if (npl > p.max_blocks) {
                raise_flag(p.status, KVQ_FLAG_BAD_POSITION);
                npl = p.max_blocks;
            }
            np = static_cast<int>(npl);
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

// Sequence index b containing unit u (largest b with Hkv * pre[b] <= u).
__device__ __forceinline__ int find_seq(const int32_t* pre, int B, int Hkv, long long u) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(Hkv) * pre[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Global address of the block of unit u, validating the page id.
__device__ __forceinline__ const uint8_t* unit_block(const KParams& p, const int32_t* pre, long long u) {
    const int b = find_seq(pre, p.B, p.Hkv, u);
    const long long rem = u - static_cast<long long>(p.Hkv) * pre[b];
    const int np = pre[b + 1] - pre[b];
    const int h = static_cast<int>(rem / np);
    const int pg = static_cast<int>(rem - static_cast<long long>(h) * np);
    int page = p.block_table[static_cast<long long>(b) * p.max_blocks + pg];
    if (page < 0 || page >= p.num_pages) {
        raise_flag(p.status, KVQ_FLAG_BAD_PAGE);
        page = 0;
    }
    return p.pool + (static_cast<long long>(page) * p.Hkv + h) * p.block_bytes;
}

// First unit of warp w's slice of U units split over W warps.
__device__ __forceinline__ long long slice_start(long long w, long long U, long long W) { return w * U / W; }

// The warp whose slice contains unit u (the largest w with slice_start(w) <= u).
__device__ __forceinline__ long long slice_of(long long u, long long U, long long W) { return ((u + 1) * W - 1) / U; }

// What a warp ending its part of segment (b, h) needs to know: the warps sharing the
// segment (n), whether it alone holds it, and which counter stands for its partial (the
// segment's, or that of its group of 32 when n > kMergeFanIn) with how many partials.
struct SegEnd {
    int n;            // warps whose slices touch the segment
    int alone;        // 1: this warp holds the whole segment
    int kind;         // 1: segment counter, 2: group counter
    int gi;           // group index within the segment (kind 2)
    int target;       // partials the counter stands for
    long long cidx;   // counter index (segment, or group's first partial slot)
};

static __device__ __noinline__ SegEnd segment_end(const int32_t* pre, int b, int h, int Hkv, long long U, long long W,
                                           long long wid, int lane) {
    SegEnd e;
    const int np = pre[b + 1] - pre[b];
    const long long seg = static_cast<long long>(b) * Hkv + h;
    const long long a_unit = static_cast<long long>(Hkv) * pre[b] + static_cast<long long>(h) * np;
    const long long wf = slice_of(a_unit, U, W);
    const long long wl = slice_of(a_unit + np - 1, U, W);
    const bool dense = U >= W;  // every slice non-empty
    e.n = static_cast<int>(wl - wf + 1);
    e.gi = e.n > kMergeFanIn ? static_cast<int>((wid - wf) / 32) : 0;
    const long long c0 = e.n > kMergeFanIn ? wf + 32LL * e.gi : wf;
    const long long c1 = e.n > kMergeFanIn ? (c0 + 31 < wl ? c0 + 31 : wl) : wl;
    int pieces = static_cast<int>(c1 - c0 + 1);
    if (!dense) {
        pieces = 0;
        for (long long w0 = c0; w0 <= c1; w0 += 32) {
            const long long w = w0 + lane;
            pieces += __popc(__ballot_sync(0xffffffffu, w <= c1 && slice_start(w, U, W) < slice_start(w + 1, U, W)));
        }
    }
    e.alone = (e.n == 1 || (!dense && e.n <= kMergeFanIn && pieces == 1)) ? 1 : 0;
    e.kind = e.n > kMergeFanIn ? 2 : 1;
    e.target = pieces;
    e.cidx = e.n > kMergeFanIn ? c0 + seg : seg;
    return e;
}

// Merge n partials (max, sum, unnormalised output) of one segment, read through index(k)
// (partial k's slot; -1 = empty), for each of the r query heads.  The result goes to the
// normalised output of (b, h) when final, else to the level-2 slot `dst`.  Lane i takes
// partials i, i + 32, ... for the maxima and sums; the outputs are folded 4 dimensions
// per lane with 8 loads in flight.
template <int D, typename Index>
__device__ __forceinline__ void merge_partials(const KParams& p, const float* src_ml, const float* src_o, int n,
                                               Index index, bool final_out, long long dst, int b, int h, int lane) {
    for (int j = 0; j < p.r; ++j) {
        float M = -INFINITY;
        for (int k0 = 0; k0 < n; k0 += 32) {
            const long long ix = k0 + lane < n ? index(k0 + lane) : -1;
            if (ix >= 0) M = fmaxf(M, __ldcg(src_ml + (ix * p.r + j) * 2));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float Lsum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const long long stride4 = static_cast<long long>(p.r) * D / 4;
        for (int k0 = 0; k0 < n; k0 += 32) {
            const long long ix = k0 + lane < n ? index(k0 + lane) : -1;
            float f = 0.f;
            if (ix >= 0) {
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(src_ml + (ix * p.r + j) * 2));
                f = fast_exp2(ml.x - M);
                Lsum = fmaf(f, ml.y, Lsum);
            }
            const int cnt = n - k0 < 32 ? n - k0 : 32;
            for (int i0 = 0; i0 < cnt; i0 += 8) {
                float4 ov[8];
                float fi[8];
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    fi[kk] = __shfl_sync(0xffffffffu, f, (i0 + kk) & 31);
                    const long long ik = __shfl_sync(0xffffffffu, ix, (i0 + kk) & 31);
                    ov[kk] = (i0 + kk < cnt && fi[kk] != 0.f)
                                 ? __ldcg(reinterpret_cast<const float4*>(src_o + (ik * p.r + j) * D) + lane)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                    (void)stride4;
                }
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const float gk = (i0 + kk < cnt) ? fi[kk] : 0.f;
                    acc.x = fmaf(gk, ov[kk].x, acc.x);
                    acc.y = fmaf(gk, ov[kk].y, acc.y);
                    acc.z = fmaf(gk, ov[kk].z, acc.z);
                    acc.w = fmaf(gk, ov[kk].w, acc.w);
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, off);
        if (final_out) {
            const float inv = 1.f / Lsum;
            float4* o4 = reinterpret_cast<float4*>(p.out + (static_cast<long long>(b) * p.Hq + h * p.r + j) * D) + lane;
            *o4 = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        } else {
            if (lane == 0) *reinterpret_cast<float2*>(p.ws_gml + (dst * p.r + j) * 2) = make_float2(M, Lsum);
            reinterpret_cast<float4*>(p.ws_go + (dst * p.r + j) * D)[lane] = acc;
        }
    }
}

// A warp that was last to count a partial merges what its counter stood for.  kind 1:
// the <= 32 warps of a short segment -> output.  kind 2: one group of up to 32 warps of a
// long segment -> level-2 partial; the group that is counted last at the segment level
// then merges the group partials -> output.  Counters return to zero once used.
template <int D>
__device__ __noinline__ void merge_after_count(const KParams& p, int kind, int b, int h, int gi, long long U,
                                               long long W, const int32_t* pre, int lane) {
    const int np = pre[b + 1] - pre[b];
    const long long seg = static_cast<long long>(b) * p.Hkv + h;
    const long long a_unit = static_cast<long long>(p.Hkv) * pre[b] + static_cast<long long>(h) * np;
    const long long wf = slice_of(a_unit, U, W);
    const long long wl = slice_of(a_unit + np - 1, U, W);
    const int n = static_cast<int>(wl - wf + 1);
    const bool dense = U >= W;
    auto slice_ix = [&](long long w) -> long long {
        return (dense || slice_start(w, U, W) < slice_start(w + 1, U, W)) ? w + seg : -1;
    };
    __threadfence();  // the partials counted before this warp are visible
    if (kind == 1) {
        merge_partials<D>(p, p.ws_ml, p.ws_o, n, [&](int k) { return slice_ix(wf + k); }, true, 0, b, h, lane);
        if (lane == 0) p.counters[seg] = 0;
        return;
    }
    const long long gs = wf + 32LL * gi;
    const int gn = static_cast<int>(wl - gs + 1 < 32 ? wl - gs + 1 : 32);
    merge_partials<D>(p, p.ws_ml, p.ws_o, gn, [&](int k) { return slice_ix(gs + k); }, false, gs + seg, b, h,
                      lane);
    if (lane == 0) p.gcounters[gs + seg] = 0;
    // count this group at the segment level; groups holding no non-empty slice never count
    const int ng = (n + 31) / 32;
    auto group_live = [&](int k) {
        if (dense) return true;
        const long long g0 = wf + 32LL * k, g1 = g0 + 31 < wl ? g0 + 31 : wl;
        return slice_start(g0, U, W) < slice_start(g1 + 1, U, W);
    };
    int live = 0;
    for (int k0 = 0; k0 < ng; k0 += 32) live += __popc(__ballot_sync(0xffffffffu, k0 + lane < ng && group_live(k0 + lane)));
    __threadfence();
    __syncwarp();
    int arrived = 0;
    if (lane == 0) arrived = atomicAdd(p.counters + seg, 1);
    arrived = __shfl_sync(0xffffffffu, arrived, 0);
    if (arrived >= live && lane == 0) raise_flag(p.status, KVQ_FLAG_STALE_WORKSPACE);
    if (arrived != live - 1) return;
    __threadfence();
    merge_partials<D>(p, p.ws_gml, p.ws_go, ng,
                      [&](int k) { return group_live(k) ? wf + 32LL * k + seg : -1LL; }, true, 0, b, h, lane);
    if (lane == 0) p.counters[seg] = 0;
}

// Resident CTAs the register budget is tuned for (3 gives up to 168 registers, enough
// for the single-head-slot fragments without spilling).
template <int GK, int HS>
constexpr int min_ctas() { return HS == 1 ? 3 : 2; }

template <int D, int GK, int GV, int HS>
__global__ void __launch_bounds__(kWarps * 32, min_ctas<GK, HS>()) decode_splitkv_kernel(KParams p) {
    static_assert(D == 128, "the fragment mapping below is written for head_dim 128");
    constexpr int NGK = D / GK;               // K groups per row
    constexpr int NGV = D / GV;               // V groups per row
    constexpr int KW = D / 32;                // K code words per thread per token row
    constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim
    constexpr int NTQ = (HS * NGK + 1) / 2;   // score n-tiles
    constexpr int VB = GV / 16;               // V code bytes per thread per group per row
    constexpr int MT = D / 16;                // output m-tiles
    constexpr int ROW = D / 2;                // bytes of one token's codes
    static_assert(NGV * VB == MT, "m-tiles cover head_dim");

    // let the combine pass launch now; it waits for this grid before reading anything
    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;   // fragment row group
    const int c = lane & 3;    // thread in group
    const int stages = p.stages;
    const int bytes = p.block_bytes;
    const size_t ring_bytes = static_cast<size_t>(kWarps) * stages * bytes;
    uint8_t* ring = smem + static_cast<size_t>(warp) * stages * bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * stages;
    WarpCtx* ctx_all = reinterpret_cast<WarpCtx*>(smem + ring_bytes + kWarps * stages * sizeof(uint64_t));
    volatile WarpCtx* ctx = ctx_all + warp;
    int32_t* pre = reinterpret_cast<int32_t*>(ctx_all + kWarps);

    // every input may come from the kernel ahead of this one on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp == 0) page_prefix(p, pre, lane);
    __syncthreads();

    const long long U = static_cast<long long>(p.Hkv) * pre[p.B];
    const long long W = static_cast<long long>(gridDim.x) * kWarps;
    const long long wid = static_cast<long long>(blockIdx.x) * kWarps + warp;
    const long long u0 = slice_start(wid, U, W);
    const long long u1 = slice_start(wid + 1, U, W);
    // sequences with no positions get zeros (no slice visits them)
    for (long long bb = wid; bb < p.B; bb += W) {
        if (pre[bb + 1] == pre[bb]) {
            float4* z4 = reinterpret_cast<float4*>(p.out + bb * p.Hq * D);
            for (int i = lane; i < p.Hq * D / 4; i += 32) z4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (u0 >= u1) return;
    const int n_units = static_cast<int>(u1 - u0);
    ctx->U = U;
    ctx->W = W;
    ctx->wid = wid;
    ctx->pend_kind = 0;

    const uint32_t bar0 = smem_u32(bars);
    const uint32_t ring0 = smem_u32(ring);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- producer: lane l holds the block address of unit wbase + l; the next window's
    // addresses are looked up one window ahead so their block-table loads overlap work ----
    int wbase = 0;
    unsigned long long waddr =
        lane < n_units ? reinterpret_cast<unsigned long long>(unit_block(p, pre, u0 + lane)) : 0ull;
    unsigned long long wnext =
        32 + lane < n_units ? reinterpret_cast<unsigned long long>(unit_block(p, pre, u0 + 32 + lane)) : 0ull;
    auto issue = [&](int i, int st) {  // unit u0 + i into stage st; i increases call by call
        if (i - wbase >= 32) {
            wbase += 32;
            waddr = wnext;
            wnext = wbase + 32 + lane < n_units
                        ? reinterpret_cast<unsigned long long>(unit_block(p, pre, u0 + wbase + 32 + lane))
                        : 0ull;
        }
        const unsigned long long src = __shfl_sync(0xffffffffu, waddr, i - wbase);
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * st;
            mbar_arrive_expect_tx(bar, bytes);
            bulk_g2s(ring0 + st * bytes, reinterpret_cast<const void*>(src), bytes, bar);
        }
    };

    // ---- consumer cursor ----
    int b = find_seq(pre, p.B, p.Hkv, u0);
    int np = pre[b + 1] - pre[b];
    int h = static_cast<int>((u0 - static_cast<long long>(p.Hkv) * pre[b]) / np);
    int pg = static_cast<int>(u0 - static_cast<long long>(p.Hkv) * pre[b] - static_cast<long long>(h) * np);
    int Leff = 0;
    bool seg_start = true;

    const int pro = n_units < stages ? n_units : stages;
    for (int k = 0; k < pro; ++k) issue(k, k);

    uint32_t qb[KSTEPS][NTQ][2];
    float m[HS], l[HS];
    float o[MT][HS][4];

    // per-thread byte offsets inside a page buffer (chunk 0)
    const int k_off = g * ROW + c * (D / 8);
    const int ks_off = p.k_scales + g * NGK * 2;
    const int vs_off = p.v_scales + g * NGV * 2;
    const int v_off = p.v_codes + c * ROW + g * VB;
    const int src0 = 4 * c + (g >> 1);
    const int src1 = 4 * (c + 4) + (g >> 1);
    const bool want_lo = (g & 1) != 0;

    // Two 16-token chunks, X = 0 and X = 1, processed together: chunk X is chunk chk[X]
    // of the page buffer blk[X] and holds sequence positions t0[X] .. t0[X] + 15.  With
    // MASKED, positions at or past Leff (and all of chunk 1 when !liveB) are excluded;
    // without it every position is valid.  The two score MMA chains are independent and
    // interleave; the softmax reduction covers all 32 positions at once.
    auto process_pair = [&](auto masked, const uint8_t* blkA, int chA, int t0A, const uint8_t* blkB, int chB,
                            int t0B, bool liveB) {
        constexpr bool MASKED = decltype(masked)::value;
        const uint8_t* blk[2] = {blkA, blkB};
        const int chk[2] = {chA, chB};
        bool vg[2], vg8[2];
        if (MASKED) {
            vg[0] = t0A + g < Leff;
            vg8[0] = t0A + g + 8 < Leff;
            vg[1] = liveB && t0B + g < Leff;
            vg8[1] = liveB && t0B + g + 8 < Leff;
        }

        // -------- scores: S = K . Q (per k-group columns), one MMA chain per chunk --------
        uint32_t kg[2][KW], kg8[2][KW];
#pragma unroll
        for (int X = 0; X < 2; ++X) {
            const uint8_t* kb = blk[X] + chk[X] * 16 * ROW + k_off;
            const uint4 x0 = *reinterpret_cast<const uint4*>(kb);
            const uint4 x1 = *reinterpret_cast<const uint4*>(kb + 8 * ROW);
            kg[X][0] = x0.x; kg[X][1] = x0.y; kg[X][2] = x0.z; kg[X][3] = x0.w;
            kg8[X][0] = x1.x; kg8[X][1] = x1.y; kg8[X][2] = x1.z; kg8[X][3] = x1.w;
        }
        float acc[2][NTQ][4];
#pragma unroll
        for (int X = 0; X < 2; ++X)
#pragma unroll
            for (int t = 0; t < NTQ; ++t) acc[X][t][0] = acc[X][t][1] = acc[X][t][2] = acc[X][t][3] = 0.f;
#pragma unroll
        for (int wi = 0; wi < KW; ++wi) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    const uint32_t x = kg[X][wi] >> (8 * e);
                    const uint32_t y = kg8[X][wi] >> (8 * e);
                    const uint32_t a0 = unpack_lo(x), a1 = unpack_lo(y), a2 = unpack_hi(x), a3 = unpack_hi(y);
#pragma unroll
                    for (int t = 0; t < NTQ; ++t)
                        mma_f16_16816(acc[X][t], a0, a1, a2, a3, qb[2 * wi + e][t][0], qb[2 * wi + e][t][1]);
                }
            }
        }
        float z[2][HS][2];
#pragma unroll
        for (int X = 0; X < 2; ++X) {
            const __half* s0 = reinterpret_cast<const __half*>(blk[X] + chk[X] * 16 * NGK * 2 + ks_off);
            const __half* s1 = s0 + 8 * NGK;
            float skg[NGK], skg8[NGK];
#pragma unroll
            for (int R = 0; R < NGK; ++R) {
                skg[R] = __half2float(s0[R]);
                skg8[R] = __half2float(s1[R]);
            }
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                float z0 = 0.f, z1 = 0.f;
#pragma unroll
                for (int R = 0; R < NGK; ++R) {
                    const int pi = s * NGK + R;
                    z0 = fmaf(skg[R], acc[X][pi >> 1][pi & 1], z0);
                    z1 = fmaf(skg8[R], acc[X][pi >> 1][2 + (pi & 1)], z1);
                }
                z[X][s][0] = z0 * p.scale_log2;
                z[X][s][1] = z1 * p.scale_log2;
                if (MASKED) {
                    z[X][s][0] = vg[X] ? z[X][s][0] : -INFINITY;
                    z[X][s][1] = vg8[X] ? z[X][s][1] : -INFINITY;
                }
            }
        }

        // -------- online softmax over the 32 positions (per head, lanes with the same c) --------
        float mn[HS];
        bool grow = false;
#pragma unroll
        for (int s = 0; s < HS; ++s) {
            float cm = fmaxf(fmaxf(z[0][s][0], z[0][s][1]), fmaxf(z[1][s][0], z[1][s][1]));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 4));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 8));
            cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, 16));
            mn[s] = fmaxf(m[s], cm);
            grow |= mn[s] > m[s];
        }
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                const float alpha = fast_exp2(m[s] - mn[s]);
                l[s] *= alpha;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mt][s][e] *= alpha;
            }
        }
        float pr[2][HS][2];
#pragma unroll
        for (int s = 0; s < HS; ++s) {
            m[s] = mn[s];
#pragma unroll
            for (int X = 0; X < 2; ++X) {
                pr[X][s][0] = fast_exp2(z[X][s][0] - mn[s]);
                pr[X][s][1] = fast_exp2(z[X][s][1] - mn[s]);
                l[s] += pr[X][s][0] + pr[X][s][1];
            }
        }

        // -------- weights W = p * v_scale as f16 hi + lo, moved into B fragments --------
        uint32_t bv[2][HS][NGV][2];
#pragma unroll
        for (int X = 0; X < 2; ++X) {
            const __half* s0 = reinterpret_cast<const __half*>(blk[X] + chk[X] * 16 * NGV * 2 + vs_off);
            const __half* s1 = s0 + 8 * NGV;
            float svg[NGV], svg8[NGV];
#pragma unroll
            for (int R = 0; R < NGV; ++R) {
                svg[R] = __half2float(s0[R]);
                svg8[R] = __half2float(s1[R]);
            }
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

        // -------- output: O^T += V^T . W, both chunks --------
#pragma unroll
        for (int R = 0; R < NGV; ++R) {
            uint32_t va[2][(VB + 3) / 4], vb[2][(VB + 3) / 4], vc[2][(VB + 3) / 4], vd[2][(VB + 3) / 4];
#pragma unroll
            for (int X = 0; X < 2; ++X) {
                const uint8_t* vcodes = blk[X] + chk[X] * 16 * ROW + v_off + R * (GV / 2);
                if constexpr (VB == 8) {
                    const uint2 ta = *reinterpret_cast<const uint2*>(vcodes);
                    const uint2 tb = *reinterpret_cast<const uint2*>(vcodes + 8 * ROW);
                    const uint2 tc = *reinterpret_cast<const uint2*>(vcodes + 4 * ROW);
                    const uint2 td = *reinterpret_cast<const uint2*>(vcodes + 12 * ROW);
                    va[X][0] = ta.x; va[X][1] = ta.y; vb[X][0] = tb.x; vb[X][1] = tb.y;
                    vc[X][0] = tc.x; vc[X][1] = tc.y; vd[X][0] = td.x; vd[X][1] = td.y;
                } else if constexpr (VB == 4) {
                    va[X][0] = *reinterpret_cast<const uint32_t*>(vcodes);
                    vb[X][0] = *reinterpret_cast<const uint32_t*>(vcodes + 8 * ROW);
                    vc[X][0] = *reinterpret_cast<const uint32_t*>(vcodes + 4 * ROW);
                    vd[X][0] = *reinterpret_cast<const uint32_t*>(vcodes + 12 * ROW);
                } else {
                    va[X][0] = *reinterpret_cast<const uint16_t*>(vcodes);
                    vb[X][0] = *reinterpret_cast<const uint16_t*>(vcodes + 8 * ROW);
                    vc[X][0] = *reinterpret_cast<const uint16_t*>(vcodes + 4 * ROW);
                    vd[X][0] = *reinterpret_cast<const uint16_t*>(vcodes + 12 * ROW);
                }
            }
#pragma unroll
            for (int jb = 0; jb < VB; jb += 2) {
                const int wi = jb / 4;
                const uint32_t bb = static_cast<uint32_t>(jb % 4);
                const uint32_t sel = bb | ((bb + 1) << 4) | ((bb + 4) << 8) | ((bb + 5) << 12);
                const int mt0 = R * VB + jb;
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    const uint32_t yac = prmt(va[X][wi], vb[X][wi], sel);  // tokens c, c+8
                    const uint32_t ybd = prmt(vc[X][wi], vd[X][wi], sel);  // tokens c+4, c+12
                    {
                        const uint32_t a0 = unpack_lo(yac), a1 = unpack_hi(yac);
                        const uint32_t a2 = unpack_lo(ybd), a3 = unpack_hi(ybd);
#pragma unroll
                        for (int s = 0; s < HS; ++s)
                            mma_f16_16816(o[mt0][s], a0, a1, a2, a3, bv[X][s][R][0], bv[X][s][R][1]);
                    }
                    {
                        const uint32_t y1 = yac >> 8, y2 = ybd >> 8;
                        const uint32_t a0 = unpack_lo(y1), a1 = unpack_hi(y1);
                        const uint32_t a2 = unpack_lo(y2), a3 = unpack_hi(y2);
#pragma unroll
                        for (int s = 0; s < HS; ++s)
                            mma_f16_16816(o[mt0 + 1][s], a0, a1, a2, a3, bv[X][s][R][0], bv[X][s][R][1]);
                    }
                }
            }
        }
    };

    // Counting a partial is deferred: the atomic add is issued at the end of a segment and
    // its result looked at when the next segment ends (or the slice does), so the round
    // trip overlaps streaming.  pend_kind 0 = nothing pending.
    int pend_arrived = 0;
    auto resolve = [&]() {
        const int kind = ctx->pend_kind;
        if (kind == 0) return;
        const int arrived = __shfl_sync(0xffffffffu, pend_arrived, 0);
        const int target = ctx->pend_target;
        if (arrived >= target && lane == 0) raise_flag(p.status, KVQ_FLAG_STALE_WORKSPACE);
        if (arrived == target - 1)
            merge_after_count<D>(p, kind, ctx->pend_b, ctx->pend_h, ctx->pend_gi, ctx->U, ctx->W, pre, lane);
        __syncwarp();
        ctx->pend_kind = 0;
    };

    // End of this warp's part of segment (b, h): write it, or hand over a partial.
    auto flush = [&]() {
        const SegEnd e = segment_end(pre, b, h, p.Hkv, ctx->U, ctx->W, ctx->wid, lane);
        const long long seg = static_cast<long long>(b) * p.Hkv + h;
        float lt[HS];
#pragma unroll
        for (int s = 0; s < HS; ++s) {
            lt[s] = l[s];
            lt[s] += __shfl_xor_sync(0xffffffffu, lt[s], 4);
            lt[s] += __shfl_xor_sync(0xffffffffu, lt[s], 8);
            lt[s] += __shfl_xor_sync(0xffffffffu, lt[s], 16);
        }
        if (e.alone) {
            // the whole segment is in this warp's registers: normalise and write
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                const int j = c + 4 * s;
                if (j < p.r) {
                    const float inv = 1.f / lt[s];
                    float* od = p.out + (static_cast<long long>(b) * p.Hq + h * p.r + j) * D;
#pragma unroll
                    for (int R = 0; R < NGV; ++R)
#pragma unroll
                        for (int jb = 0; jb < VB; ++jb) {
                            const int mt = R * VB + jb;
                            const int dd = 2 * (R * (GV / 2) + g * VB + jb);
                            *reinterpret_cast<float2*>(od + dd) = make_float2((o[mt][s][0] + o[mt][s][1]) * inv,
                                                                             (o[mt][s][2] + o[mt][s][3]) * inv);
                        }
                }
            }
            return;
        }
        const long long piece = ctx->wid + seg;
#pragma unroll
        for (int s = 0; s < HS; ++s) {
            const int j = c + 4 * s;
            if (j < p.r) {
                if (g == 0) *reinterpret_cast<float2*>(p.ws_ml + (piece * p.r + j) * 2) = make_float2(m[s], lt[s]);
                float* od = p.ws_o + (piece * p.r + j) * D;
#pragma unroll
                for (int R = 0; R < NGV; ++R)
#pragma unroll
                    for (int jb = 0; jb < VB; ++jb) {
                        const int mt = R * VB + jb;
                        const int dd = 2 * (R * (GV / 2) + g * VB + jb);
                        *reinterpret_cast<float2*>(od + dd) =
                            make_float2(o[mt][s][0] + o[mt][s][1], o[mt][s][2] + o[mt][s][3]);
                    }
            }
        }
        resolve();  // the previous segment's count has had time to come back
        __threadfence();  // publish this partial before counting it
        __syncwarp();
        if (lane == 0) {
            pend_arrived = atomicAdd((e.kind == 2 ? p.gcounters : p.counters) + e.cidx, 1);
            ctx->pend_kind = e.kind;
            ctx->pend_b = b;
            ctx->pend_h = h;
            ctx->pend_gi = e.gi;
            ctx->pend_target = e.target;
        }
        __syncwarp();
    };

    int cst = 0;          // stage of the next unit to consume
    uint32_t cpar = 0;    // its phase parity
    const bool p16 = p.P == 16;

    for (int i = 0; i < n_units;) {
        if (seg_start) {
            // new (sequence, kv head): q fragments and a fresh softmax state
            int L = p.seq_lens[b];
            L = L < 0 ? 0 : L;
            Leff = min(L, p.max_blocks * p.P);
#pragma unroll
            for (int t = 0; t < NTQ; ++t) {
                const int pi = 2 * t + (g & 1);
                const int sigma = pi / NGK;
                const int R = pi % NGK;
                const int j = (g >> 1) + 4 * sigma;
                const bool colv = sigma < HS && j < p.r;
                const __half* qrow = p.q + (static_cast<long long>(b) * p.Hq + h * p.r + (colv ? j : 0)) * D;
#pragma unroll
                for (int wi = 0; wi < KW; ++wi) {
                    const int dbase = c * (D / 4) + 8 * wi;
                    uint4 w4 = make_uint4(0, 0, 0, 0);
                    if (colv && dbase / GK == R) w4 = *reinterpret_cast<const uint4*>(qrow + dbase);
                    qb[2 * wi][t][0] = prmt(w4.x, w4.z, 0x5410u);
                    qb[2 * wi][t][1] = prmt(w4.x, w4.z, 0x7632u);
                    qb[2 * wi + 1][t][0] = prmt(w4.y, w4.w, 0x5410u);
                    qb[2 * wi + 1][t][1] = prmt(w4.y, w4.w, 0x7632u);
                }
            }
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                m[s] = -INFINITY;
                l[s] = 0.f;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mt][s][e] = 0.f;
            }
            seg_start = false;
        }

        // 16-token pages: two pages of the same segment per iteration when there are two;
        // larger pages: one page, its chunks two at a time.
        const int n = (p16 && i + 1 < n_units && pg + 1 < np) ? 2 : 1;
        int st1 = cst;
        uint32_t par1 = cpar;
        bool ok = mbar_wait(bar0 + 8 * cst, cpar, kWaitLimitNs);
        if (n == 2) {
            if (++st1 == stages) {
                st1 = 0;
                par1 ^= 1u;
            }
            ok = ok && mbar_wait(bar0 + 8 * st1, par1, kWaitLimitNs);
        }
        if (!__all_sync(0xffffffffu, ok)) {
            // give up on this slice: flag it, then let the copies already issued land
            if (lane == 0) raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
            const int pending = n_units - i < stages ? n_units - i : stages;
            int st = cst;
            uint32_t par = cpar;
            for (int k = 0; k < pending; ++k) {
                mbar_wait(bar0 + 8 * st, par, kWaitLimitNs);
                if (++st == stages) {
                    st = 0;
                    par ^= 1u;
                }
            }
            return;
        }
        const uint8_t* blkA = ring + cst * bytes;
        const uint8_t* blkB = ring + st1 * bytes;
        if (p16) {
            const int t0 = pg * 16;
            if (n == 2 && t0 + 32 <= Leff)
                process_pair(std::false_type{}, blkA, 0, t0, blkB, 0, t0 + 16, true);
            else
                process_pair(std::true_type{}, blkA, 0, t0, blkB, 0, t0 + 16, n == 2);
        } else {
            for (int chunk = 0; chunk < p.P / 16; chunk += 2) {
                const int t0 = pg * p.P + chunk * 16;
                if (t0 >= Leff) break;
                if (t0 + 32 <= Leff)
                    process_pair(std::false_type{}, blkA, chunk, t0, blkA, chunk + 1, t0 + 16, true);
                else
                    process_pair(std::true_type{}, blkA, chunk, t0, blkA, chunk + 1, t0 + 16, true);
            }
        }

        // ---- release the stages and refill them with the pages `stages` units ahead ----
        __syncwarp();
        if (lane == 0) fence_proxy_async_smem();
        if (i + stages < n_units) issue(i + stages, cst);
        if (n == 2 && i + 1 + stages < n_units) issue(i + 1 + stages, st1);
        cst = st1;
        cpar = par1;
        if (++cst == stages) {
            cst = 0;
            cpar ^= 1u;
        }
        i += n;

        // ---- end of a segment or of this warp's slice ----
        pg += n;
        const bool seg_end = (pg == np);
        if (seg_end || i == n_units) flush();
        if (seg_end) {
            pg = 0;
            if (++h == p.Hkv) {
                h = 0;
                do {
                    ++b;
                } while (b < p.B && pre[b + 1] == pre[b]);
            }
            if (b < p.B) np = pre[b + 1] - pre[b];
            seg_start = true;
        }
    }
    resolve();
}

// Raise the kernel's dynamic shared-memory limit once to the largest size asked for,
// so repeated calls (and calls under stream capture) only launch.
template <int D, int GK, int GV, int HS>
cudaError_t ensure_smem_attr(size_t smem) {
    static std::atomic<long long> granted{-1};
    if (static_cast<long long>(smem) <= granted.load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(decode_splitkv_kernel<D, GK, GV, HS>,
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
template <int D, int GK, int GV, int HS>
int occupancy(size_t smem) {
    constexpr int kSlots = 32;
    static std::atomic<long long> memo[kSlots];  // (smem << 8) | ctas, 0 = empty
    for (int i = 0; i < kSlots; ++i) {
        const long long m = memo[i].load(std::memory_order_acquire);
        if (m == 0) break;
        if ((m >> 8) == static_cast<long long>(smem)) return static_cast<int>(m & 0xff);
    }
    if (ensure_smem_attr<D, GK, GV, HS>(smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_splitkv_kernel<D, GK, GV, HS>, kWarps * 32, smem) !=
        cudaSuccess)
        return 0;
    const long long entry = (static_cast<long long>(smem) << 8) | (n & 0xff);
    for (int i = 0; i < kSlots; ++i) {
        long long expect = 0;
        if (memo[i].compare_exchange_strong(expect, entry) || expect == entry) break;
    }
    return n;
}

template <int D, int GK, int GV, int HS>
cudaError_t run(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    KParams p;
    p.pool = a.pool;
    p.q = a.q;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.ws_ml = reinterpret_cast<float*>(a.workspace + plan.ws_ml_offset);
    p.ws_o = reinterpret_cast<float*>(a.workspace + plan.ws_o_offset);
    p.ws_gml = reinterpret_cast<float*>(a.workspace + plan.ws_gml_offset);
    p.ws_go = reinterpret_cast<float*>(a.workspace + plan.ws_go_offset);
    p.counters = reinterpret_cast<int32_t*>(a.workspace + plan.ws_cnt_offset);
    p.gcounters = reinterpret_cast<int32_t*>(a.workspace + plan.ws_gcnt_offset);
    p.status = reinterpret_cast<uint32_t*>(a.workspace);
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.r = a.Hq / a.Hkv;
    p.P = a.L.P;
    p.num_pages = a.num_pages;
    p.max_blocks = a.max_blocks;
    p.block_bytes = a.L.bytes;
    p.stages = plan.stages;
    p.v_codes = a.L.v_codes;
    p.k_scales = a.L.k_scales;
    p.v_scales = a.L.v_scales;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    cudaError_t err = ensure_smem_attr<D, GK, GV, HS>(plan.smem_bytes);
    if (err != cudaSuccess) return err;
    // The launch may start before the kernel ahead of it on the stream finishes
    // (programmatic dependent launch); the kernel waits with griddepcontrol.wait before
    // it reads any input.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.ctas));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, decode_splitkv_kernel<D, GK, GV, HS>, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace decode

// Per-K-group dispatch entry points, one per translation unit.
cudaError_t decode_run_gk32(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk64(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk128(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_gk32(const DecodeArgs& a, size_t smem);
int decode_occupancy_gk64(const DecodeArgs& a, size_t smem);
int decode_occupancy_gk128(const DecodeArgs& a, size_t smem);

}  // namespace kvq

// Instantiates the dispatch for one K group size GK_ over GV in {32, 64, 128}, HS in {1, 2}.
#define KVQ_DECODE_TU(GK_)                                                                           \
    namespace kvq {                                                                                  \
    cudaError_t decode_run_gk##GK_(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s) {    \
        const int hs = (a.Hq / a.Hkv) > 4 ? 2 : 1;                                                   \
        switch (a.L.Gv * 4 + hs) {                                                                   \
            case 32 * 4 + 1: return decode::run<128, GK_, 32, 1>(a, plan, s);                        \
            case 32 * 4 + 2: return decode::run<128, GK_, 32, 2>(a, plan, s);                        \
            case 64 * 4 + 1: return decode::run<128, GK_, 64, 1>(a, plan, s);                        \
            case 64 * 4 + 2: return decode::run<128, GK_, 64, 2>(a, plan, s);                        \
            case 128 * 4 + 1: return decode::run<128, GK_, 128, 1>(a, plan, s);                      \
            case 128 * 4 + 2: return decode::run<128, GK_, 128, 2>(a, plan, s);                      \
            default: return cudaErrorInvalidValue;                                                   \
        }                                                                                            \
    }                                                                                                \
    int decode_occupancy_gk##GK_(const DecodeArgs& a, size_t smem) {                                 \
        const int hs = (a.Hq / a.Hkv) > 4 ? 2 : 1;                                                   \
        switch (a.L.Gv * 4 + hs) {                                                                   \
            case 32 * 4 + 1: return decode::occupancy<128, GK_, 32, 1>(smem);                        \
            case 32 * 4 + 2: return decode::occupancy<128, GK_, 32, 2>(smem);                        \
            case 64 * 4 + 1: return decode::occupancy<128, GK_, 64, 1>(smem);                        \
            case 64 * 4 + 2: return decode::occupancy<128, GK_, 64, 2>(smem);                        \
            case 128 * 4 + 1: return decode::occupancy<128, GK_, 128, 1>(smem);                      \
            case 128 * 4 + 2: return decode::occupancy<128, GK_, 128, 2>(smem);                      \
            default: return 0;                                                                       \
        }                                                                                            \
    }                                                                                                \
    }
