// quantize.cu -- quantize-on-append: fp16 K/V rows -> packed INT4 codes + fp16 group
// scales written into their (page, kv-head) blocks.
//
// "4-bit KV cache compression" (lpnh.cn/news/2042373), section 2.1: per group of G
// elements along head_dim, scale = amax / 7 (an all-zero group gets 1), code =
// round(x / scale) clamped to [-7, 7].  Here scale = fp16_rne(fp32(amax) / 7.0f), the
// zero test is on that fp16 value, and code = round_half_even(fp32(x) / fp32(scale))
// with an IEEE division, so codes and scales are bit-exact functions of the input.
//
// Work mapping: a "row job" is one K or one V row of d fp16 values for one (sequence,
// new token, kv head).  A team of d/8 lanes takes a job; each lane loads 16 bytes
// (8 values), the group maximum is a shuffle-xor reduction over the G/8 lanes of a
// group, and each lane stores its 8 codes as one 32-bit word, so a team writes the
// row's d/2 code bytes contiguously.  The job loop is grid-strided.
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

template <int D>
__global__ void __launch_bounds__(256) quantize_append_kernel(QuantizeArgs a) {
    // a decode launched behind this kernel may start its own set-up now; it waits for
    // this grid to finish before it reads the pool
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int LPR = D / 8;            // lanes per row
    constexpr int TEAMS = 32 / LPR;       // row jobs per warp at a time
    const int lane = threadIdx.x & 31;
    const int team = lane / LPR;
    const int tl = lane % LPR;            // lane within the team
    const int lanes_k = a.L.Gk / 8;       // lanes per K group
    const int lanes_v = a.L.Gv / 8;
    const long long jobs = 2LL * a.B * a.n_new * a.Hkv;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const long long warps_total = static_cast<long long>(gridDim.x) * blockDim.x / 32;

    for (long long base = warp_global * TEAMS; base < jobs; base += warps_total * TEAMS) {
        const long long job = base + team;
        const bool active = job < jobs;
        // job -> (row index, K or V); rows ordered as the input [B, n_new, Hkv]
        const long long row = job >> 1;
        const int is_v = static_cast<int>(job & 1);
        const int G = is_v ? a.L.Gv : a.L.Gk;
        const int glanes = is_v ? lanes_v : lanes_k;

        // load 8 fp16 values
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (active) {
            const __half* src = (is_v ? a.v : a.k) + row * D + tl * 8;
            raw = *reinterpret_cast<const uint4*>(src);
        }
        float x[8];
        {
            const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __half22float2(h2[i]);
                x[2 * i] = f.x;
                x[2 * i + 1] = f.y;
            }
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
        // group maximum over the group's lanes (groups are aligned within the team).  The
        // K and V teams of a warp have different group widths, so every lane runs the
        // same shuffles and only folds in partners inside its own group.
#pragma unroll
        for (int off = 1; off < LPR; off <<= 1) {
            const float other = __shfl_xor_sync(0xffffffffu, amax, off);
            if (off < glanes) amax = fmaxf(amax, other);
        }

        if (!active) continue;
        __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
        if ((__half_as_ushort(s16) & 0x7fffu) == 0) s16 = __ushort_as_half(0x3c00u);
        const float s = __half2float(s16);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int c = __float2int_rn(__fdiv_rn(x[i], s));
            c = max(-7, min(7, c));
            word |= static_cast<uint32_t>(c + 8) << (4 * i);
        }

        // destination: position, page, slot
        const int h = static_cast<int>(row % a.Hkv);
        const long long bt_row = row / a.Hkv;  // (b, t)
        const int t = static_cast<int>(bt_row % a.n_new);
        const int b = static_cast<int>(bt_row / a.n_new);
        const long long pos = static_cast<long long>(a.start_pos[b]) + t;
        const long long pidx = pos >= 0 ? pos / a.L.P : -1;
        if (pos < 0 || pidx >= a.max_blocks) {
            if (tl == 0) raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
            continue;
        }
        const int page = a.block_table[static_cast<long long>(b) * a.max_blocks + pidx];
        if (page < 0 || page >= a.num_pages) {
            if (tl == 0) raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
            continue;
        }
        const int slot = static_cast<int>(pos % a.L.P);
        uint8_t* blk = a.pool + (static_cast<long long>(page) * a.Hkv + h) * a.L.bytes;
        uint8_t* codes = blk + (is_v ? a.L.v_codes : 0) + slot * (D / 2);
        reinterpret_cast<uint32_t*>(codes)[tl] = word;
        if ((tl % glanes) == 0) {
            uint8_t* scales = blk + (is_v ? a.L.v_scales : a.L.k_scales) + slot * (D / G) * 2;
            reinterpret_cast<__half*>(scales)[tl / glanes] = s16;
        }
    }
}

template <int D>
cudaError_t launch_q(const QuantizeArgs& a, cudaStream_t stream) {
    const long long jobs = 2LL * a.B * a.n_new * a.Hkv;
    if (jobs == 0) return cudaSuccess;
    constexpr int threads = 256;
    constexpr int jobs_per_block = (threads / 32) * (32 / (D / 8));
    long long blocks = (jobs + jobs_per_block - 1) / jobs_per_block;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 8;  // 8 blocks of 256 per SM
    if (blocks > cap) blocks = cap;
    quantize_append_kernel<D><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_append(const QuantizeArgs& a, cudaStream_t stream) {
    switch (a.L.d) {
        case 64: return launch_q<64>(a, stream);
        case 128: return launch_q<128>(a, stream);
        case 256: return launch_q<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvq
