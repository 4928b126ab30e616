// decode_fp16.cuh -- split-KV decode attention over the FP16 paged cache: the FP16 baseline
// of the latency comparison in "LLM long-context inference: managing the KV cache with an
// INT4 state machine", section 7.4 (FP16 attention; INT4 dequantized first and then attended
// through this kernel; INT4 dequantized inside the operator, decode_impl.cuh).
//
// The FP16 cache keeps the INT4 cache's pages: block (page, kv head) at
// (page * Hkv + h) * 4 * P * d bytes holds K rows P x d fp16, then V rows P x d fp16.
//
// The grid, the unit slices, the per-warp rings of bulk copies, the q staging and the
// per-warp partials (and so the combine kernel) are those of decode_splitkv_kernel; a
// unit is one page of one kv head (8 KB at P = 16, d = 128).  The arithmetic runs on the
// CUDA cores, which at 512 bytes per token and head keeps far below the HBM time:
//  * lane l owns dimensions 4l .. 4l + 3 of q (prescaled by softmax_scale * log2 e), of
//    each K and V row it reads (8 bytes per row: conflict-free shared loads) and of the
//    output;
//  * the T token dot products of a step (T = 16, or 8 with 8 query heads per kv head)
//    are reduced across the warp by a butterfly that halves the values a lane keeps at
//    each exchange (T shuffles in all instead of 5 T), leaving token (lane >> 1) (T = 16)
//    or (lane >> 2) (T = 8) in every lane;
//  * the online softmax runs per query head on those lanes; each weight is then
//    broadcast by a shuffle to the V accumulation.
//
// The same kernel serves the rotated 4-bit cache (codec 2; the INT8 per-row cache runs on
// the tensor-core kernel of decode_impl.cuh): only the row reader differs, and for the
// rotated codec ("LARQL KV cache engines", engine three; wht_codec.cu) the arithmetic runs
// in the rotated domain.  A row there is
// x^ = H (sigma c) / d with H symmetric, so q . x^ = (H q / d) . (sigma c): each segment's
// q is rotated once (and divided by d), the rows are read as sigma * c_code, and the
// accumulated output sum_t p_t sigma_t c_t is rotated back (H / d) when the warp writes
// its partial; the combine is linear and never sees the rotated domain.
#pragma once

#include "decode_impl.cuh"

namespace kvq {
namespace decode {

// Parameters of the CUDA-core kernel: the split-KV kernel's, and the rotated codec's
// codebook levels.
struct FParams {
    KParams p;
    float lut[16];
};

// fp32 Walsh-Hadamard transform of a 128-vector held 4 per lane (lane l: elements 4l ..
// 4l + 3): stages of span 1 and 2 inside the lane, then 4 .. 64 across lanes at xor
// distances 1 .. 16, the lower element of each pair becoming a + b and the upper a - b.
__device__ __forceinline__ void wht128_lane4(float (&y)[4], int lane) {
    const float t0 = y[0] + y[1], t1 = y[0] - y[1], t2 = y[2] + y[3], t3 = y[2] - y[3];
    y[0] = t0 + t2;
    y[2] = t0 - t2;
    y[1] = t1 + t3;
    y[3] = t1 - t3;
#pragma unroll
    for (int X = 1; X < 32; X <<= 1) {
        const bool upper = (lane & X) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, y[j], X);
            y[j] = upper ? other - y[j] : y[j] + other;
        }
    }
}

// One row of a staged block: this lane's 4 values (dimensions 4l .. 4l + 3) of row `row`
// of K (is_v 0) or V (is_v 1).  CODEC 0, FP16 blocks: K rows then V rows, P x D fp16
// each.  CODEC 2, rotated 4-bit blocks: K codes P x D/2 (nibbles, element 2j low), V codes,
// K sigma P fp32, V sigma P fp32; a value is sigma * lut[code], in the rotated domain.
// The reader returns lut[code] only: the row's sigma (row_sigma) multiplies the reduced
// score and the softmax weight instead of every value.
template <int CODEC, int D>
__device__ __forceinline__ void block_row4(const uint8_t* blk, int P, int is_v, int row, int lane, float (&x)[4],
                                           const float* lut) {
    if constexpr (CODEC == 2) {
        const uint32_t w = *reinterpret_cast<const uint16_t*>(blk + (is_v * P + row) * (D / 2) + 2 * lane);
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = lut[(w >> (4 * j)) & 15u];
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(blk + ((is_v * P + row) * D + 4 * lane) * 2);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
        x[0] = a.x;
        x[1] = a.y;
        x[2] = b.x;
        x[3] = b.y;
    }
}

// sigma of row `row` of K (is_v 0) or V (is_v 1) in a rotated 4-bit block
template <int D>
__device__ __forceinline__ float row_sigma(const uint8_t* blk, int P, int is_v, int row) {
    return *reinterpret_cast<const float*>(blk + P * D + 4 * (is_v * P + row));
}

// R: query heads per kv head, rounded up to 1, 2, 4 or 8.  WIN: the sequences list only
// their window and sink pages (p.window > 0), as in decode_splitkv_kernel.  CODEC: 0 FP16,
// 2 rotated 4-bit blocks.
template <int D, int R, bool WIN, int CODEC = 0>
__global__ void __launch_bounds__(128, 1) decode_fp16_kernel(const __grid_constant__ FParams f) {
    static_assert(D == 128, "four dimensions per lane");
    static_assert(CODEC == 0 || CODEC == 2, "FP16 or rotated 4-bit blocks");
    const KParams& p = f.p;
    constexpr int kWarps = 4;
    constexpr int T = R == 8 ? 8 : 16;   // tokens per step
    constexpr int LG_T = R == 8 ? 3 : 4;
    constexpr int TSH = 5 - LG_T;        // lane of token tau: tau << TSH

    asm volatile("griddepcontrol.launch_dependents;");

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int stages = p.stages;
    const int ubytes = p.unit_bytes;
    const size_t ring_all = static_cast<size_t>(kWarps) * stages * ubytes;
    uint8_t* ring = smem + static_cast<size_t>(warp) * stages * ubytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ring_all) + warp * stages;
    CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + ring_all + kWarps * stages * sizeof(uint64_t));
    __half* qbuf = reinterpret_cast<__half*>(ctl + 1);  // [2][8][D]
    int32_t* pre = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(qbuf) + q_buf_bytes<D>());
    int32_t* lens = pre + p.B + 1;
    int32_t* aps = lens + p.B;
    const uint32_t qbar0 = smem_u32(&ctl->qbar[0]);
    const uint32_t qfree0 = smem_u32(&ctl->qfree[0]);
    float* lut = reinterpret_cast<float*>(ctl->pad);  // the rotated codec's levels (64 of its 96 bytes)

    // read-only inputs only until griddepcontrol.wait (seq_lens, block table, q)
    if (warp == 0) page_prefix(p, pre, lens, aps, lane);
    if (CODEC == 2 && threadIdx.x < 16) lut[threadIdx.x] = f.lut[threadIdx.x];
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
    auto publish_prefix = [&]() {
        if (cta == 0 && warp == 0)
            for (int i = lane; i <= p.B; i += 32) p.ws_pre[i] = pre[i];
    };
    if (c0 >= c1) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        publish_prefix();
        return;
    }
    const int span = static_cast<int>(c1 - c0);
    const int nm = span > warp ? (span - warp + kWarps - 1) / kWarps : 0;

    const uint32_t bar0 = smem_u32(bars);
    const uint32_t ring0 = smem_u32(ring);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncwarp();

    // ---- producer: as in decode_splitkv_kernel (addresses a window of 32 units ahead) ----
    auto unit_of = [&](int i) { return c0 + warp + static_cast<long long>(kWarps) * i; };
    int wbase = 0;
    unsigned long long waddr =
        lane < nm ? reinterpret_cast<unsigned long long>(unit_block<WIN>(p, pre, lens, unit_of(lane), 1)) : 0ull;
    unsigned long long wnext =
        32 + lane < nm ? reinterpret_cast<unsigned long long>(unit_block<WIN>(p, pre, lens, unit_of(32 + lane), 1))
                       : 0ull;
    int issued = 0;
    const uint64_t l2_stream = l2_policy_evict_first();
    auto issue = [&](int i, int st) {
        if (i - wbase >= 32) {
            wbase += 32;
            waddr = wnext;
            wnext = wbase + 32 + lane < nm
                        ? reinterpret_cast<unsigned long long>(unit_block<WIN>(p, pre, lens, unit_of(wbase + 32 + lane), 1))
                        : 0ull;
        }
        const unsigned long long src = __shfl_sync(0xffffffffu, waddr, i - wbase);
        if (lane == 0) {
            const uint32_t bar = bar0 + 8 * st;
            mbar_arrive_expect_tx(bar, ubytes);
            bulk_g2s_hint(ring0 + st * ubytes, reinterpret_cast<const void*>(src), ubytes, bar, l2_stream);
        }
        ++issued;
    };
    const uint32_t q_bytes = static_cast<uint32_t>(p.ns) * D * 2;
    auto issue_q = [&](int sb, int shg, int k) {
        const uint32_t bar = qbar0 + 8 * (k & 1);
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(bar, q_bytes);
        bulk_g2s(smem_u32(qbuf + (k & 1) * 8 * D), p.q + (static_cast<long long>(sb) * p.Hq + shg * p.ns) * D, q_bytes,
                 bar);
    };
    auto next_seg = [&](int& sb, int& shg) {
        if (++shg == p.Hg) {
            shg = 0;
            do {
                ++sb;
            } while (sb < p.B && pre[sb + 1] == pre[sb]);
        }
    };
    int b = find_seq(pre, p.B, p.Hg, c0);
    int np = pre[b + 1] - pre[b];
    int hg = static_cast<int>(div_nn(c0 - static_cast<long long>(p.Hg) * pre[b], np));
    long long sfirst = static_cast<long long>(p.Hg) * pre[b] + static_cast<long long>(hg) * np;
    if (threadIdx.x == 0) issue_q(b, hg, 0);

    asm volatile("griddepcontrol.wait;" ::: "memory");
    publish_prefix();
    {
        const int pro = nm < stages ? nm : stages;
        for (int k = 0; k < pro; ++k) issue(k, k);
    }

    // ---- consumer ----
    float qv[R][4];  // this lane's q dimensions, scaled to log2 units
    float m[R], l[R], o[R][4];
    int consumed = 0, cst = 0;
    uint32_t cpar = 0;
    bool failed = false;
    int f_st = 0, f_out = 0;
    uint32_t f_par = 0;
    int segk = 0;
    auto fail_here = [&]() {
        if (lane == 0) raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
        failed = true;
        f_st = cst;
        f_par = cpar;
        f_out = issued - consumed;
    };

    while (sfirst < c1) {
        const long long ua = sfirst > c0 ? sfirst : c0;
        const long long ue = sfirst + np < c1 ? sfirst + np : c1;
        const long long fu = ua + (((c0 + warp - ua) % kWarps) + kWarps) % kWarps;
        const int cnt = fu < ue ? static_cast<int>((ue - fu + kWarps - 1) / kWarps) : 0;
        const int pg0 = static_cast<int>(fu - sfirst);
        const SeqSpan sspan = seq_span(lens[b], p.lg_p, p.max_blocks, WIN ? p.window : 0, WIN ? p.sinks : 0);
        const int Leff = sspan.L;
        const int wlo = sspan.wlo;  // 0 without a window

        if (threadIdx.x == 0 && sfirst + np < c1) {
            int nb = b, nhg = hg;
            next_seg(nb, nhg);
            if (segk >= 1 && !mbar_wait(qfree0 + 8 * ((segk - 1) & 1), ((segk - 1) >> 1) & 1, kWaitLimitNs))
                raise_flag(p.status, KVQ_FLAG_WAIT_TIMEOUT);
            issue_q(nb, nhg, segk + 1);
        }
        // Every warp waits for the segment's q copy, units here or not: that copy is issued
        // only once every warp has released the buffer two segments back, so no warp can
        // arrive on a qfree barrier while the phase of two segments back is still open.
        if (!failed && !__all_sync(0xffffffffu, mbar_wait(qbar0 + 8 * (segk & 1), (segk >> 1) & 1, kWaitLimitNs)))
            fail_here();
        if (cnt > 0) {
            const __half* qseg = qbuf + (segk & 1) * 8 * D;
#pragma unroll
            for (int s = 0; s < R; ++s) {
                const int sl = s < p.ns ? s : 0;
                const uint2 w = *reinterpret_cast<const uint2*>(qseg + sl * D + 4 * lane);
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
                qv[s][0] = f0.x * p.scale_log2;
                qv[s][1] = f0.y * p.scale_log2;
                qv[s][2] = f1.x * p.scale_log2;
                qv[s][3] = f1.y * p.scale_log2;
            }
            if constexpr (CODEC == 2) {
                // scores against the rotated rows: (H q / d) . (sigma c)
#pragma unroll
                for (int s = 0; s < R; ++s) {
                    wht128_lane4(qv[s], lane);
#pragma unroll
                    for (int j = 0; j < 4; ++j) qv[s][j] *= 1.0f / D;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(qfree0 + 8 * (segk & 1));
#pragma unroll
        for (int s = 0; s < R; ++s) {
            m[s] = -INFINITY;
            l[s] = 0.f;
            o[s][0] = o[s][1] = o[s][2] = o[s][3] = 0.f;
        }

        int last_st = cst;
        for (int j = 0; j < cnt; ++j) {
            if (!failed && !__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * cst, cpar, kWaitLimitNs))) fail_here();
            if (!failed) {
                const uint8_t* blk = ring + cst * ubytes;
                const int pg = pg0 + kWarps * j;
                const int rp = WIN ? span_page(sspan, pg) : pg;  // the page (past a window gap)
                for (int t0 = 0; t0 < p.P; t0 += T) {
                    const int tpos = rp * p.P + t0;
                    if (tpos >= Leff) break;
                    // a step wholly outside the window and the sinks is skipped, so every
                    // processed step holds an attended token
                    if (WIN && !(min(tpos + T, Leff) > wlo || tpos < p.sinks)) continue;
                    // the attended tokens of the step (bit t); the others' V rows are skipped, since
                    // slots past a sequence's end may hold any bit pattern, which a zero weight
                    // would not cancel (0 * inf)
                    uint32_t vmask = 0xffffffffu;
                    if (!(tpos + T <= Leff && (!WIN || tpos >= wlo || tpos + T <= p.sinks))) {
                        vmask = 0u;
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            const int tt2 = tpos + t;
                            if (tt2 < Leff && (!WIN || tt2 >= wlo || tt2 < p.sinks)) vmask |= 1u << t;
                        }
                    }
                    // partial dot products of this lane's 4 dimensions, T tokens, R heads
                    float a[R][T];
#pragma unroll
                    for (int t = 0; t < T; ++t) {
                        float kx[4];
                        block_row4<CODEC, D>(blk, p.P, 0, t0 + t, lane, kx, lut);
                        const float2 k0 = make_float2(kx[0], kx[1]);
                        const float2 k1 = make_float2(kx[2], kx[3]);
#pragma unroll
                        for (int s = 0; s < R; ++s)
                            a[s][t] = fmaf(qv[s][3], k1.y, fmaf(qv[s][2], k1.x, fmaf(qv[s][1], k0.y, qv[s][0] * k0.x)));
                    }
                    // butterfly: at exchange X a lane keeps the half of its values whose token
                    // index has bit (X >> TSH) equal to its lane bit X, adding the partner's half
#pragma unroll
                    for (int s = 0; s < R; ++s) {
#pragma unroll
                        for (int X = 16, n = T; n > 1; X >>= 1, n >>= 1) {
                            const bool up = (lane & X) != 0;
#pragma unroll
                            for (int i = 0; i < n / 2; ++i) {
                                const float keep = up ? a[s][i + n / 2] : a[s][i];
                                const float give = up ? a[s][i] : a[s][i + n / 2];
                                a[s][i] = keep + __shfl_xor_sync(0xffffffffu, give, X);
                            }
                        }
                        // the remaining lanes of a token hold partial sums of different dimensions
#pragma unroll
                        for (int X = (1 << TSH) >> 1; X > 0; X >>= 1) a[s][0] += __shfl_xor_sync(0xffffffffu, a[s][0], X);
                    }
                    // online softmax per head on the token this lane holds
                    const int tau = lane >> TSH;
                    if constexpr (CODEC == 2) {
                        const float sk = row_sigma<D>(blk, p.P, 0, t0 + tau);
#pragma unroll
                        for (int s = 0; s < R; ++s) a[s][0] *= sk;
                    }
                    const int tt = tpos + tau;
                    const bool valid = tt < Leff && (!WIN || tt >= wlo || tt < p.sinks);
                    float pw[R];
#pragma unroll
                    for (int s = 0; s < R; ++s) {
                        const float z = valid ? a[s][0] : -INFINITY;
                        float cm = z;
#pragma unroll
                        for (int X = 16; X >= (1 << TSH); X >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, X));
                        const float mn = fmaxf(m[s], cm);  // finite: the step holds a valid token
                        const float alpha = fast_exp2(m[s] - mn);
                        pw[s] = fast_exp2(z - mn);
                        float ps = pw[s];
#pragma unroll
                        for (int X = 16; X >= (1 << TSH); X >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, X);
                        l[s] = fmaf(l[s], alpha, ps);
                        m[s] = mn;
                        o[s][0] *= alpha;
                        o[s][1] *= alpha;
                        o[s][2] *= alpha;
                        o[s][3] *= alpha;
                    }
                    // o += sum_tau p_tau v_tau; a step with unattended tokens skips their rows
                    // (MASKED), every other step runs without a test per token
                    auto accumulate = [&](auto masked) {
                        constexpr bool MASKED = decltype(masked)::value;
#pragma unroll
                        for (int t = 0; t < T; ++t) {
                            if (MASKED && !((vmask >> t) & 1u)) continue;
                            float vx[4];
                            block_row4<CODEC, D>(blk, p.P, 1, t0 + t, lane, vx, lut);
                            // the rotated codec's row sigma goes into the weight (up to 4 query
                            // heads per kv head) or into the values
                            const float sv = CODEC == 2 ? row_sigma<D>(blk, p.P, 1, t0 + t) : 1.f;
                            if (CODEC == 2 && R > 4) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) vx[j] *= sv;
                            }
                            const float2 v0 = make_float2(vx[0], vx[1]);
                            const float2 v1 = make_float2(vx[2], vx[3]);
#pragma unroll
                            for (int s = 0; s < R; ++s) {
                                float pt = __shfl_sync(0xffffffffu, pw[s], t << TSH);
                                if (CODEC == 2 && R <= 4) pt *= sv;
                                o[s][0] = fmaf(pt, v0.x, o[s][0]);
                                o[s][1] = fmaf(pt, v0.y, o[s][1]);
                                o[s][2] = fmaf(pt, v1.x, o[s][2]);
                                o[s][3] = fmaf(pt, v1.y, o[s][3]);
                            }
                        }
                    };
                    if (vmask == 0xffffffffu) accumulate(std::false_type{});
                    else accumulate(std::true_type{});
                }
                __syncwarp();
                if (lane == 0) fence_proxy_async_smem();
                if (consumed + stages < nm) issue(consumed + stages, cst);
            }
            last_st = cst;
            ++consumed;
            if (++cst == stages) {
                cst = 0;
                cpar ^= 1u;
            }
        }
        (void)last_st;

        // ---- segment end: this warp's partial, index kWarps * (CTA + segment) + warp ----
        {
            const long long seg = static_cast<long long>(b) * p.Hg + hg;
            const long long piece = static_cast<long long>(kWarps) * (cta + seg) + warp;
            const bool mine = cnt > 0 && !failed;
#pragma unroll
            for (int s = 0; s < R; ++s) {
                if constexpr (CODEC == 2) {
                    // back from the rotated domain: H o / d
                    wht128_lane4(o[s], lane);
#pragma unroll
                    for (int j = 0; j < 4; ++j) o[s][j] *= 1.0f / D;
                }
                if (s < p.ns) {
                    if (lane == 0)
                        *reinterpret_cast<float2*>(p.ws_ml + (piece * p.ns + s) * 2) =
                            mine ? make_float2(m[s], l[s]) : make_float2(-INFINITY, 0.f);
                    reinterpret_cast<float4*>(p.ws_o + (piece * p.ns + s) * D)[lane] =
                        mine ? make_float4(o[s][0], o[s][1], o[s][2], o[s][3]) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }

        ++segk;
        sfirst += np;
        next_seg(b, hg);
        if (b < p.B) np = pre[b + 1] - pre[b];
        else break;
    }

    // ---- no q copy may still be landing when the CTA leaves ----
    if (threadIdx.x == 0) {
        for (int k = segk - 2; k < segk; ++k)
            if (k >= 0) mbar_wait(qbar0 + 8 * (k & 1), (k >> 1) & 1, kWaitLimitNs);
    }
    if (failed) {
        int st = f_st;
        uint32_t par = f_par;
        for (int k = 0; k < f_out; ++k) {
            mbar_wait(bar0 + 8 * st, par, kWaitLimitNs);
            if (++st == stages) {
                st = 0;
                par ^= 1u;
            }
        }
    }
}

}  // namespace decode
}  // namespace kvq
