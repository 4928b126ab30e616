// decode_combine.cu -- the split-KV combine kernel and its launch: it writes the decode
// output from the warp partials the decode grid(s) leave in the workspace.
#include <algorithm>

#include "decode_impl.cuh"

namespace kvq {
namespace decode {

// ---------------------------------------------------------------------------
// Combine: the warp partials of each (sequence, query head) row into its output.
// ---------------------------------------------------------------------------
// One source of partials: a decode grid's workspace region and how that grid listed
// each sequence's pages and laid out its partials.
struct CSource {
    const float* ws_ml;
    const float* ws_o;
    const int32_t* ws_pre;  // the pages prefix the grid publishes (used above kCombineLocalB)
    int32_t Hg, ns;         // head groups of the grid's units, query heads per unit
    int32_t C, W;           // the grid's CTAs, and warps per CTA (partials per CTA and segment)
    int32_t max_blocks, window, sinks, len_sub;  // as in KParams
};

struct CParams {
    CSource src[2];
    int32_t nsrc;  // 1, or 2 for the mixed-precision decode (INT4 history, FP16 recent tokens)
    const int32_t* seq_lens;
    float* out;
    float* out_host;  // device address of mapped pinned host memory that also receives out, or nullptr
    int32_t B, Hq, lg_p;
};

constexpr int kCombineMaxWarps = 16;
constexpr int kCombineLocalB = 256;   // up to this batch the row metadata is computed before the wait

// One CTA per output row (b, hq).  In source s the row's partials sit at W * (cf + seg) + j
// for j < W * (cl - cf + 1), where CTAs cf..cl of that grid hold the units of segment
// seg = (b, hq / ns); when some CTA slices are empty (fewer units than CTAs) their partials
// do not exist.  Warp w of the CTA takes partials w, w + nw, ..., NB at a time, keeping
// a running maximum M and sum L and an unnormalised output (lane l: dimensions 4f .. 4f + 3
// for f = l, l + 32, ... below D / 4),
// over the sources in turn; the warps' results are then merged with weights 2^(M_w - max M).
// Sequences without positions have no partials and get zeros.  This is the split-KV
// combine of flash decoding: out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i.
// NSRC: sources of partials (p.nsrc), a template parameter so the one-source combine
// carries no code for a second.
// NB: partials a warp loads together, 8 or 4.  The 4-partial instance, held to 64
// registers (at head_dim 256 it may take more, which its rows need), serves the rows of
// many partials (16-warp CTAs): at up to 128 registers such a CTA would hold a whole SM's
// register file and keep the next call's decode CTAs off that SM until it leaves; at 64
// it holds half.  Rows of 4- and 8-warp CTAs (up to 64 partials) load 8 at a time, in
// one round.
template <int D, int NSRC, int NB>
__global__ void __launch_bounds__(kCombineMaxWarps * 32, NB == 8 || D == 256 ? 1 : 2)
combine_kernel(CParams p) {
    static_assert(D == 64 || D == 128 || D == 256, "head_dim 64, 128 or 256");
    static_assert(NB == 8 || NB == 4, "8 partials a batch, or 4 for the 4-warp CTAs");
    constexpr int NV = (D / 4 + 31) / 32;                 // float4 of the row per lane
    constexpr int NA = NB == 4 ? 1 : (NV == 1 ? 4 : 2);  // independent sums per float4 (shorter fma chains)
    auto lane_has = [](int lane, int v) { return D / 4 >= 32 || lane + 32 * v < D / 4; };
    // the next decode call may start its set-up; it waits for this grid before it
    // touches the workspace
    asm volatile("griddepcontrol.launch_dependents;");
    __shared__ float s_m[kCombineMaxWarps], s_l[kCombineMaxWarps];
    __shared__ float4 s_o[kCombineMaxWarps][D / 4];
    __shared__ int s_red[2][2][kCombineMaxWarps];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int b = static_cast<int>(blockIdx.x / p.Hq);
    const int hq = static_cast<int>(blockIdx.x - static_cast<long long>(b) * p.Hq);

    // Pages of sequence i as source s listed them, and the row's range of partials.
    auto pages_of = [&](const CSource& s, int i) {
        return seq_span(p.seq_lens[i] - s.len_sub, p.lg_p, s.max_blocks, s.window, s.sinks).np;
    };
    auto row_range = [&](const CSource& s, int pb_, int np_, int tot_, long long& cf_, long long& base_,
                         long long& U_) {
        const int hg = hq / s.ns;
        U_ = static_cast<long long>(s.Hg) * tot_;
        const long long sf = static_cast<long long>(s.Hg) * pb_ + static_cast<long long>(hg) * np_;
        cf_ = slice_of(sf, U_, s.C);
        const long long cl = slice_of(sf + np_ - 1, U_, s.C);
        base_ = static_cast<long long>(s.W) * (cf_ + static_cast<long long>(b) * s.Hg + hg);
        return s.W * static_cast<int>(cl - cf_ + 1);
    };
    int n[2] = {0, 0};
    long long cf[2] = {0, 0}, base[2] = {0, 0}, U[2] = {1, 1};

    // The row's pages prefix: for small batches from seq_lens (a read-only input) while
    // the decode grids still run; else from the prefix each decode grid publishes.
    const bool local = p.B <= kCombineLocalB;
    if (local) {
#pragma unroll
        for (int si = 0; si < NSRC; ++si) {
            int before = 0, all = 0;
            for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
                const int n_i = pages_of(p.src[si], i);
                all += n_i;
                if (i < b) before += n_i;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                before += __shfl_xor_sync(0xffffffffu, before, off);
                all += __shfl_xor_sync(0xffffffffu, all, off);
            }
            if (lane == 0) {
                s_red[si][0][warp] = before;
                s_red[si][1][warp] = all;
            }
        }
        __syncthreads();
#pragma unroll
        for (int si = 0; si < NSRC; ++si) {
            int pb = 0, tot = 0;
            for (int w = 0; w < nw; ++w) {
                pb += s_red[si][0][w];
                tot += s_red[si][1][w];
            }
            const int np = pages_of(p.src[si], b);
            if (np > 0) n[si] = row_range(p.src[si], pb, np, tot, cf[si], base[si], U[si]);
        }
    }

    // the partials (and the published prefixes) are written by the decode grids ahead of this one
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!local) {
#pragma unroll
        for (int si = 0; si < NSRC; ++si) {
            const int32_t* pre = p.src[si].ws_pre;
            const int pb = __ldcg(pre + b);
            const int np = __ldcg(pre + b + 1) - pb;
            const int tot = __ldcg(pre + p.B);
            if (np > 0) n[si] = row_range(p.src[si], pb, np, tot, cf[si], base[si], U[si]);
        }
    }

    float M = -INFINITY, L = 0.f;
    float4 acc[NV][NA];
#pragma unroll
    for (int v = 0; v < NV; ++v)
#pragma unroll
        for (int a = 0; a < NA; ++a) acc[v][a] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int si = 0; si < NSRC; ++si) {
        const CSource& s = p.src[si];
        const int sl = hq - (hq / s.ns) * s.ns;
        const bool dense = U[si] >= s.C;  // every CTA slice holds units
        const long long stride_ml = static_cast<long long>(s.ns) * 2;
        const long long stride_o = static_cast<long long>(s.ns) * D;
        const float* ml0 = s.ws_ml + (base[si] * s.ns + sl) * 2;
        const float* o0 = s.ws_o + (base[si] * s.ns + sl) * D + 4 * lane;
        for (int j0 = warp; j0 < n[si]; j0 += NB * nw) {
            float2 ml[NB];
            float4 ov[NB][NV];
#pragma unroll
            for (int kk = 0; kk < NB; ++kk) {
                const int j = j0 + kk * nw;
                bool have = j < n[si];
                if (have && !dense) {
                    const long long k = cf[si] + j / s.W;
                    have = slice_start(k, U[si], s.C) < slice_start(k + 1, U[si], s.C);
                }
                ml[kk] = have ? __ldcg(reinterpret_cast<const float2*>(ml0 + j * stride_ml)) : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    ov[kk][v] = have && lane_has(lane, v) ? __ldcg(reinterpret_cast<const float4*>(o0 + j * stride_o) + 32 * v)
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float mb = M;
#pragma unroll
            for (int kk = 0; kk < NB; ++kk) mb = fmaxf(mb, ml[kk].x);
            if (mb == -INFINITY) continue;  // only empty partials so far
            if (mb > M) {  // a larger running maximum: rescale what has been summed
                const float f = fast_exp2(M - mb);
                L *= f;
#pragma unroll
                for (int v = 0; v < NV; ++v)
#pragma unroll
                    for (int a = 0; a < NA; ++a) {
                        acc[v][a].x *= f;
                        acc[v][a].y *= f;
                        acc[v][a].z *= f;
                        acc[v][a].w *= f;
                    }
                M = mb;
            }
#pragma unroll
            for (int kk = 0; kk < NB; ++kk) {
                const float f = fast_exp2(ml[kk].x - M);
                L = fmaf(f, ml[kk].y, L);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float4& A = acc[v][kk % NA];
                    A.x = fmaf(f, ov[kk][v].x, A.x);
                    A.y = fmaf(f, ov[kk][v].y, A.y);
                    A.z = fmaf(f, ov[kk][v].z, A.z);
                    A.w = fmaf(f, ov[kk][v].w, A.w);
                }
            }
        }
    }
    if (lane == 0) {
        s_m[warp] = M;
        s_l[warp] = L;
    }
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        float4 t = acc[v][0];
#pragma unroll
        for (int a = 1; a < NA; ++a) {
            t.x += acc[v][a].x;
            t.y += acc[v][a].y;
            t.z += acc[v][a].z;
            t.w += acc[v][a].w;
        }
        if (lane_has(lane, v)) s_o[warp][lane + 32 * v] = t;
    }
    __syncthreads();
    if (warp == 0) {
        float Mx = -INFINITY;
        for (int w = 0; w < nw; ++w) Mx = fmaxf(Mx, s_m[w]);
        float Ls = 0.f;
        if (Mx != -INFINITY)
            for (int w = 0; w < nw; ++w) Ls = fmaf(fast_exp2(s_m[w] - Mx), s_l[w], Ls);
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        const long long row = static_cast<long long>(b) * p.Hq + hq;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            if (!lane_has(lane, v)) continue;
            const int f4 = lane + 32 * v;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
            if (Mx != -INFINITY) {
                for (int w = 0; w < nw; ++w) {
                    const float f = fast_exp2(s_m[w] - Mx);
                    const float4 ow = s_o[w][f4];
                    O.x = fmaf(f, ow.x, O.x);
                    O.y = fmaf(f, ow.y, O.y);
                    O.z = fmaf(f, ow.z, O.z);
                    O.w = fmaf(f, ow.w, O.w);
                }
            }
            const float4 r = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
            reinterpret_cast<float4*>(p.out + row * D)[f4] = r;
            if (p.out_host != nullptr) reinterpret_cast<float4*>(p.out_host + row * D)[f4] = r;
        }
    }
}

}  // namespace decode

namespace {

// The partials one decode grid (arguments a, plan) leaves in its workspace.
decode::CSource source_of(const DecodeArgs& a, const DecodePlan& plan) {
    decode::CSource s;
    s.ws_ml = reinterpret_cast<const float*>(a.workspace + plan.ws_ml_offset);
    s.ws_o = reinterpret_cast<const float*>(a.workspace + plan.ws_o_offset);
    s.ws_pre = reinterpret_cast<const int32_t*>(a.workspace + plan.ws_pre_offset);
    s.Hg = a.Hkv / plan.hk;
    s.ns = plan.hk * (a.Hq / a.Hkv);
    s.C = plan.ctas;
    s.W = 4;
    s.max_blocks = a.max_blocks;
    s.window = a.window;
    s.sinks = a.sinks;
    s.len_sub = a.len_sub;
    return s;
}

cudaError_t launch(const decode::CParams& p, int d, int warps, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.B) * p.Hq;
    if (rows <= 0) return cudaSuccess;
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    // Launched while the decode grid runs (programmatic dependent launch); the kernel
    // waits with griddepcontrol.wait before it reads the workspace.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(static_cast<unsigned>(warps) * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err;
    const bool light = warps == 16;  // the 64-register instance
    if (p.nsrc == 2) err = cudaLaunchKernelEx(&cfg, decode::combine_kernel<128, 2, 8>, p);  // mixed: head_dim 128 only
    else if (d == 64) err = light ? cudaLaunchKernelEx(&cfg, decode::combine_kernel<64, 1, 4>, p)
                                  : cudaLaunchKernelEx(&cfg, decode::combine_kernel<64, 1, 8>, p);
    else if (d == 256) err = light ? cudaLaunchKernelEx(&cfg, decode::combine_kernel<256, 1, 4>, p)
                                   : cudaLaunchKernelEx(&cfg, decode::combine_kernel<256, 1, 8>, p);
    else if (d == 128) err = light ? cudaLaunchKernelEx(&cfg, decode::combine_kernel<128, 1, 4>, p)
                                   : cudaLaunchKernelEx(&cfg, decode::combine_kernel<128, 1, 8>, p);
    else return cudaErrorInvalidValue;
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

int lg2(int P) {
    int l = 0;
    while ((1 << l) < P) ++l;
    return l;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    decode::CParams p{};
    p.src[0] = source_of(a, plan);
    p.nsrc = 1;
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.out_host = a.out_host;
    p.B = a.B;
    p.Hq = a.Hq;
    p.lg_p = lg2(a.L.P);
    return launch(p, a.L.d, plan.combine_warps, stream);
}

// The mixed-precision decode: the partials of the INT4 grid (a0, plan0) and of the FP16
// grid (a1, plan1) merged per row.
cudaError_t launch_combine2(const DecodeArgs& a0, const DecodePlan& plan0, const DecodeArgs& a1,
                            const DecodePlan& plan1, cudaStream_t stream) {
    decode::CParams p{};
    p.src[0] = source_of(a0, plan0);
    p.src[1] = source_of(a1, plan1);
    p.nsrc = 2;
    p.seq_lens = a0.seq_lens;
    p.out = a0.out;
    p.B = a0.B;
    p.Hq = a0.Hq;
    p.lg_p = lg2(a0.L.P);
    const int warps = std::max(plan0.combine_warps, plan1.combine_warps);
    return launch(p, a0.L.d, warps, stream);
}

}  // namespace kvq
