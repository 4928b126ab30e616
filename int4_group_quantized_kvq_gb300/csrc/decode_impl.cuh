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
//    slice, so ragged lengths and small batches still keep every SM busy.  A warp
//    writes one partial (running max, running sum, unnormalised output) per (sequence,
//    kv head) segment its slice touches; the combine pass merges them.
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
#pragma once

#include <cuda_fp16.h>

#include <atomic>
#include <cstdint>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace decode {

constexpr int kWarps = 4;                         // warps per CTA
constexpr uint64_t kWaitLimitNs = 250000000ull;   // a page copy that takes 250 ms has failed

struct KParams {
    const uint8_t* pool;
    const __half* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* ws_ml;
    float* ws_o;
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

template <int D, int GK, int GV, int HS>
__global__ void __launch_bounds__(kWarps * 32) decode_splitkv_kernel(KParams p) {
    static_assert(D == 128, "the fragment mapping below is written for head_dim 128");
    constexpr int NGK = D / GK;               // K groups per row
    constexpr int NGV = D / GV;               // V groups per row
    constexpr int KW = D / 32;                // K code words per thread per token row
    constexpr int KSTEPS = D / 16;            // MMA k-steps over head_dim
    constexpr int NTQ = (HS * NGK + 1) / 2;   // score n-tiles
    constexpr int VB = GV / 16;               // V code bytes per thread per group per row
    constexpr int MT = D / 16;                // output m-tiles
    static_assert(NGV * VB == MT, "m-tiles cover head_dim");

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;   // fragment row group
    const int c = lane & 3;    // thread in group
    const int stages = p.stages;
    const size_t ring_bytes = static_cast<size_t>(kWarps) * stages * p.block_bytes;
    uint8_t* ring = smem + static_cast<size_t>(warp) * stages * p.block_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_bytes) + warp * stages;
    int32_t* pre = reinterpret_cast<int32_t*>(smem + ring_bytes + kWarps * stages * sizeof(uint64_t));

    if (warp == 0) page_prefix(p, pre, lane);
    __syncthreads();

    const long long U = static_cast<long long>(p.Hkv) * pre[p.B];
    const long long W = static_cast<long long>(gridDim.x) * kWarps;
    const long long wid = static_cast<long long>(blockIdx.x) * kWarps + warp;
    const long long u0 = wid * U / W;
    const long long u1 = (wid + 1) * U / W;
    if (u0 >= u1) return;

    const uint32_t bar0 = smem_u32(bars);
    const uint32_t ring0 = smem_u32(ring);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- producer: lane l keeps the block address of unit win + l ----
    long long win = u0;
    const uint8_t* waddr = (u0 + lane < u1) ? unit_block(p, pre, u0 + lane) : nullptr;
    int istage = 0;
    auto issue = [&](long long u) {
        if (u - win >= 32) {
            win += 32;
            waddr = (win + lane < u1) ? unit_block(p, pre, win + lane) : nullptr;
        }
        const uint8_t* src = reinterpret_cast<const uint8_t*>(
            __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(waddr), static_cast<int>(u - win)));
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * istage;
            mbar_arrive_expect_tx(bar, p.block_bytes);
            bulk_g2s(ring0 + istage * p.block_bytes, src, p.block_bytes, bar);
        }
        istage = (istage + 1 == stages) ? 0 : istage + 1;
    };

    const long long n_units = u1 - u0;
    const int pro = static_cast<int>(n_units < stages ? n_units : stages);
    for (int k = 0; k < pro; ++k) issue(u0 + k);

    // ---- consumer cursor ----
    int b = find_seq(pre, p.B, p.Hkv, u0);
    int np = pre[b + 1] - pre[b];
    long long rem0 = u0 - static_cast<long long>(p.Hkv) * pre[b];
    int h = static_cast<int>(rem0 / np);
    int pg = static_cast<int>(rem0 - static_cast<long long>(h) * np);
    int Leff = 0;
    bool seg_start = true;

    uint32_t qb[KSTEPS][NTQ][2];
    float m[HS], l[HS];
    float o[MT][HS][4];

    int cstage = 0;
    uint32_t cparity = 0;

    for (long long u = u0; u < u1; ++u) {
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

        // ---- wait for this unit's page ----
        bool ok = mbar_wait(bar0 + 8 * cstage, cparity, kWaitLimitNs);
        if (!__all_sync(0xffffffffu, ok)) {
            // give up on this slice: flag it, then let copies already issued land
            if (lane == 0) raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
            long long pending = (u1 - u < stages) ? (u1 - u) : stages;
            int s = cstage;
            uint32_t par = cparity;
            for (long long k = 0; k < pending; ++k) {
                mbar_wait(bar0 + 8 * s, par, kWaitLimitNs);
                if (++s == stages) { s = 0; par ^= 1u; }
            }
            return;
        }
        const uint8_t* blk = ring + static_cast<size_t>(cstage) * p.block_bytes;

        for (int chunk = 0; chunk < p.P / 16; ++chunk) {
            const int t0 = pg * p.P + chunk * 16;
            if (t0 >= Leff) break;
            const bool vg = t0 + g < Leff;
            const bool vg8 = t0 + g + 8 < Leff;
            const int rg = chunk * 16 + g;  // slot rows in the page

            // -------- scores: S = K . Q (per k-group columns) --------
            uint32_t kg[KW], kg8[KW];
            {
                const uint4 x0 = *reinterpret_cast<const uint4*>(blk + rg * (D / 2) + c * (D / 8));
                const uint4 x1 = *reinterpret_cast<const uint4*>(blk + (rg + 8) * (D / 2) + c * (D / 8));
                kg[0] = x0.x; kg[1] = x0.y; kg[2] = x0.z; kg[3] = x0.w;
                kg8[0] = x1.x; kg8[1] = x1.y; kg8[2] = x1.z; kg8[3] = x1.w;
            }
            float acc[NTQ][4];
#pragma unroll
            for (int t = 0; t < NTQ; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
#pragma unroll
            for (int wi = 0; wi < KW; ++wi) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t x = kg[wi] >> (8 * e);
                    const uint32_t y = kg8[wi] >> (8 * e);
                    const uint32_t a0 = unpack_lo(x), a1 = unpack_lo(y), a2 = unpack_hi(x), a3 = unpack_hi(y);
#pragma unroll
                    for (int t = 0; t < NTQ; ++t)
                        mma_f16_16816(acc[t], a0, a1, a2, a3, qb[2 * wi + e][t][0], qb[2 * wi + e][t][1]);
                }
            }
            float skg[NGK], skg8[NGK];
            {
                const __half* s0 = reinterpret_cast<const __half*>(blk + p.k_scales + rg * NGK * 2);
                const __half* s1 = reinterpret_cast<const __half*>(blk + p.k_scales + (rg + 8) * NGK * 2);
#pragma unroll
                for (int R = 0; R < NGK; ++R) {
                    skg[R] = __half2float(s0[R]);
                    skg8[R] = __half2float(s1[R]);
                }
            }
            float z[HS][2];
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int R = 0; R < NGK; ++R) {
                    const int pi = s * NGK + R;
                    s0 = fmaf(skg[R], acc[pi >> 1][pi & 1], s0);
                    s1 = fmaf(skg8[R], acc[pi >> 1][2 + (pi & 1)], s1);
                }
                z[s][0] = vg ? s0 * p.scale_log2 : -INFINITY;
                z[s][1] = vg8 ? s1 * p.scale_log2 : -INFINITY;
            }

            // -------- online softmax (per head, over lanes with the same c) --------
            float mn[HS];
            bool grow = false;
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                float cm = fmaxf(z[s][0], z[s][1]);
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
            float pr[HS][2];
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                m[s] = mn[s];
                pr[s][0] = fast_exp2(z[s][0] - mn[s]);
                pr[s][1] = fast_exp2(z[s][1] - mn[s]);
                l[s] += pr[s][0] + pr[s][1];
            }

            // -------- weights W = p * v_scale as f16 hi + lo, moved into B fragments --------
            float svg[NGV], svg8[NGV];
            {
                const __half* s0 = reinterpret_cast<const __half*>(blk + p.v_scales + rg * NGV * 2);
                const __half* s1 = reinterpret_cast<const __half*>(blk + p.v_scales + (rg + 8) * NGV * 2);
#pragma unroll
                for (int R = 0; R < NGV; ++R) {
                    svg[R] = __half2float(s0[R]);
                    svg8[R] = __half2float(s1[R]);
                }
            }
            const int src0 = 4 * c + (g >> 1);
            const int src1 = 4 * (c + 4) + (g >> 1);
            const bool want_lo = (g & 1) != 0;
            uint32_t bv[HS][NGV][2];
#pragma unroll
            for (int s = 0; s < HS; ++s) {
#pragma unroll
                for (int R = 0; R < NGV; ++R) {
                    const float w0 = vg ? pr[s][0] * svg[R] : 0.f;
                    const float w1 = vg8 ? pr[s][1] * svg8[R] : 0.f;
                    const __half h0 = __float2half_rn(w0);
                    const __half h1 = __float2half_rn(w1);
                    const float r0 = w0 - __half2float(h0);
                    const float r1 = w1 - __half2float(h1);
                    __half2 hp = __halves2half2(h0, h1);
                    const uint32_t phi = *reinterpret_cast<uint32_t*>(&hp);
                    const uint32_t plo = pack_h2(r0, r1);
                    const uint32_t x0 = __shfl_sync(0xffffffffu, phi, src0);
                    const uint32_t y0 = __shfl_sync(0xffffffffu, plo, src0);
                    const uint32_t x1 = __shfl_sync(0xffffffffu, phi, src1);
                    const uint32_t y1 = __shfl_sync(0xffffffffu, plo, src1);
                    bv[s][R][0] = want_lo ? y0 : x0;
                    bv[s][R][1] = want_lo ? y1 : x1;
                }
            }

            // -------- output: O^T += V^T . W --------
            const uint8_t* vcodes = blk + p.v_codes + (chunk * 16) * (D / 2);
#pragma unroll
            for (int R = 0; R < NGV; ++R) {
                const int off = R * (GV / 2) + g * VB;
                uint32_t va[(VB + 3) / 4], vb[(VB + 3) / 4], vc[(VB + 3) / 4], vd[(VB + 3) / 4];
                if constexpr (VB == 8) {
                    const uint2 ta = *reinterpret_cast<const uint2*>(vcodes + c * (D / 2) + off);
                    const uint2 tb = *reinterpret_cast<const uint2*>(vcodes + (c + 8) * (D / 2) + off);
                    const uint2 tc = *reinterpret_cast<const uint2*>(vcodes + (c + 4) * (D / 2) + off);
                    const uint2 td = *reinterpret_cast<const uint2*>(vcodes + (c + 12) * (D / 2) + off);
                    va[0] = ta.x; va[1] = ta.y; vb[0] = tb.x; vb[1] = tb.y;
                    vc[0] = tc.x; vc[1] = tc.y; vd[0] = td.x; vd[1] = td.y;
                } else if constexpr (VB == 4) {
                    va[0] = *reinterpret_cast<const uint32_t*>(vcodes + c * (D / 2) + off);
                    vb[0] = *reinterpret_cast<const uint32_t*>(vcodes + (c + 8) * (D / 2) + off);
                    vc[0] = *reinterpret_cast<const uint32_t*>(vcodes + (c + 4) * (D / 2) + off);
                    vd[0] = *reinterpret_cast<const uint32_t*>(vcodes + (c + 12) * (D / 2) + off);
                } else {
                    va[0] = *reinterpret_cast<const uint16_t*>(vcodes + c * (D / 2) + off);
                    vb[0] = *reinterpret_cast<const uint16_t*>(vcodes + (c + 8) * (D / 2) + off);
                    vc[0] = *reinterpret_cast<const uint16_t*>(vcodes + (c + 4) * (D / 2) + off);
                    vd[0] = *reinterpret_cast<const uint16_t*>(vcodes + (c + 12) * (D / 2) + off);
                }
#pragma unroll
                for (int jb = 0; jb < VB; jb += 2) {
                    const int wi = jb / 4;
                    const uint32_t bb = static_cast<uint32_t>(jb % 4);
                    const uint32_t sel = bb | ((bb + 1) << 4) | ((bb + 4) << 8) | ((bb + 5) << 12);
                    const uint32_t yac = prmt(va[wi], vb[wi], sel);  // tokens c, c+8
                    const uint32_t ybd = prmt(vc[wi], vd[wi], sel);  // tokens c+4, c+12
                    const int mt0 = R * VB + jb;
                    {
                        const uint32_t a0 = unpack_lo(yac), a1 = unpack_hi(yac);
                        const uint32_t a2 = unpack_lo(ybd), a3 = unpack_hi(ybd);
#pragma unroll
                        for (int s = 0; s < HS; ++s) mma_f16_16816(o[mt0][s], a0, a1, a2, a3, bv[s][R][0], bv[s][R][1]);
                    }
                    {
                        const uint32_t y1 = yac >> 8, y2 = ybd >> 8;
                        const uint32_t a0 = unpack_lo(y1), a1 = unpack_hi(y1);
                        const uint32_t a2 = unpack_lo(y2), a3 = unpack_hi(y2);
#pragma unroll
                        for (int s = 0; s < HS; ++s)
                            mma_f16_16816(o[mt0 + 1][s], a0, a1, a2, a3, bv[s][R][0], bv[s][R][1]);
                    }
                }
            }
        }

        // ---- release the stage and refill it with the page `stages` units ahead ----
        __syncwarp();
        if (u + stages < u1) {
            if (lane == 0) fence_proxy_async_smem();
            issue(u + stages);
        }
        if (++cstage == stages) {
            cstage = 0;
            cparity ^= 1u;
        }

        // ---- end of a segment or of this warp's slice: write the partial ----
        ++pg;
        const bool seg_end = (pg == np);
        if (seg_end || u + 1 == u1) {
            const long long piece = wid + static_cast<long long>(b) * p.Hkv + h;
#pragma unroll
            for (int s = 0; s < HS; ++s) {
                float lt = l[s];
                lt += __shfl_xor_sync(0xffffffffu, lt, 4);
                lt += __shfl_xor_sync(0xffffffffu, lt, 8);
                lt += __shfl_xor_sync(0xffffffffu, lt, 16);
                const int j = c + 4 * s;
                if (j < p.r) {
                    float* ml = p.ws_ml + (piece * p.r + j) * 2;
                    if (g == 0) {
                        ml[0] = m[s];
                        ml[1] = lt;
                    }
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
        }
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
}

// Merge the per-warp partials of each (sequence, query head).
template <int D>
__global__ void __launch_bounds__(128) decode_combine_kernel(KParams p, float* out, int32_t W) {
    extern __shared__ __align__(16) int32_t cpre[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) page_prefix(p, cpre, lane);
    __syncthreads();
    const long long item = static_cast<long long>(blockIdx.x) * 4 + warp;
    if (item >= static_cast<long long>(p.B) * p.Hq) return;
    const int b = static_cast<int>(item / p.Hq);
    const int hq = static_cast<int>(item % p.Hq);
    const int h = hq / p.r, j = hq % p.r;
    const int np = cpre[b + 1] - cpre[b];
    const long long U = static_cast<long long>(p.Hkv) * cpre[p.B];
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    float* dst = out + item * D + lane * PER;
    if (np == 0 || U == 0) {
        *reinterpret_cast<float4*>(dst) = make_float4(0.f, 0.f, 0.f, 0.f);
        return;
    }
    const long long a = static_cast<long long>(p.Hkv) * cpre[b] + static_cast<long long>(h) * np;
    const long long e = a + np - 1;
    const long long wf = ((a + 1) * W - 1) / U;
    const long long wl = ((e + 1) * W - 1) / U;
    const long long seg = static_cast<long long>(b) * p.Hkv + h;
    float M = -INFINITY;
    for (long long w = wf; w <= wl; ++w) {
        if (w * U / W == (w + 1) * U / W) continue;  // empty slice: wrote nothing
        M = fmaxf(M, p.ws_ml[((w + seg) * p.r + j) * 2]);
    }
    float Lsum = 0.f;
    for (long long w = wf; w <= wl; ++w) {
        if (w * U / W == (w + 1) * U / W) continue;
        const float* ml = p.ws_ml + ((w + seg) * p.r + j) * 2;
        const float f = fast_exp2(ml[0] - M);
        Lsum = fmaf(f, ml[1], Lsum);
        const float4 ov = *reinterpret_cast<const float4*>(p.ws_o + ((w + seg) * p.r + j) * D + lane * PER);
        acc[0] = fmaf(f, ov.x, acc[0]);
        acc[1] = fmaf(f, ov.y, acc[1]);
        acc[2] = fmaf(f, ov.z, acc[2]);
        acc[3] = fmaf(f, ov.w, acc[3]);
    }
    const float inv = 1.f / Lsum;
    *reinterpret_cast<float4*>(dst) = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
}

template <int D, int GK, int GV, int HS>
cudaError_t ensure_smem_attr(size_t smem);

template <int D, int GK, int GV, int HS>
cudaError_t run(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    KParams p;
    p.pool = a.pool;
    p.q = a.q;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.ws_ml = reinterpret_cast<float*>(a.workspace + plan.ws_ml_offset);
    p.ws_o = reinterpret_cast<float*>(a.workspace + plan.ws_o_offset);
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
    auto kern = decode_splitkv_kernel<D, GK, GV, HS>;
    cudaError_t err = ensure_smem_attr<D, GK, GV, HS>(plan.smem_bytes);
    if (err != cudaSuccess) return err;
    kern<<<plan.ctas, kWarps * 32, plan.smem_bytes, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const long long items = static_cast<long long>(a.B) * a.Hq;
    const unsigned cblocks = static_cast<unsigned>((items + 3) / 4);
    decode_combine_kernel<D><<<cblocks, 128, (a.B + 1) * sizeof(int32_t), stream>>>(p, a.out, plan.warps);
    return cudaGetLastError();
}

// Raise the kernel's dynamic shared-memory limit once to the largest size asked for,
// so repeated calls (and calls under stream capture) only launch.
template <int D, int GK, int GV, int HS>
cudaError_t ensure_smem_attr(size_t smem) {
    static std::atomic<long long> granted{-1};
    if (static_cast<long long>(smem) <= granted.load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(decode_splitkv_kernel<D, GK, GV, HS>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err == cudaSuccess) {
        long long cur = granted.load();
        while (static_cast<long long>(smem) > cur && !granted.compare_exchange_weak(cur, static_cast<long long>(smem))) {
        }
    }
    return err;
}

// Resident CTAs per SM for a given shared-memory size (memoised for the last size asked).
template <int D, int GK, int GV, int HS>
int occupancy(size_t smem) {
    static std::atomic<long long> memo{-1};  // (smem << 8) | ctas
    const long long m = memo.load(std::memory_order_acquire);
    if (m >= 0 && (m >> 8) == static_cast<long long>(smem)) return static_cast<int>(m & 0xff);
    if (ensure_smem_attr<D, GK, GV, HS>(smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_splitkv_kernel<D, GK, GV, HS>, kWarps * 32, smem) !=
        cudaSuccess)
        return 0;
    memo.store((static_cast<long long>(smem) << 8) | (n & 0xff), std::memory_order_release);
    return n;
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
