// fp16_cache.cu -- the FP16 paged cache of the latency comparison ("LLM long-context
// inference: managing the KV cache with an INT4 state machine", section 7.4): its append,
// and the dequantization of the INT4 cache into it (the "dequantize first, then attend"
// arm).  Block (page, kv head) at (page * Hkv + h) * 4 * P * d bytes: K rows P x d fp16,
// then V rows P x d fp16.
//
// Both kernels move 16-byte pieces: one thread per 8 elements of one row.
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

__device__ __forceinline__ uint8_t* fp16_row(uint8_t* pool16, int Hkv, int d, int P, long long page, int h, int is_v,
                                             int slot) {
    return pool16 + (page * Hkv + h) * (4LL * P * d) + (static_cast<long long>(is_v) * P + slot) * d * 2;
}

// rows k, v [B, n_new, Hkv, d] fp16 -> the FP16 pool at start_pos[b] + t
__global__ void __launch_bounds__(256) fp16_append_kernel(Fp16AppendArgs a) {
    const int words = a.d / 8;
    const long long total = 2LL * a.B * a.n_new * a.Hkv * words;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int w = static_cast<int>(i % words);
        const long long r = i / words;  // ((b * n_new + t) * Hkv + h) * 2 + is_v
        const int is_v = static_cast<int>(r & 1);
        const long long row = r >> 1;
        const int h = static_cast<int>(row % a.Hkv);
        const long long bt_ = row / a.Hkv;
        const int t = static_cast<int>(bt_ % a.n_new);
        const int b = static_cast<int>(bt_ / a.n_new);
        const long long pos = static_cast<long long>(a.start_pos[b]) + t;
        const long long pidx = pos >= 0 ? pos / a.P : -1;
        if (pidx < 0 || pidx >= a.max_blocks) {
            if (w == 0 && is_v == 0) raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
            continue;
        }
        const int page = a.block_table[static_cast<long long>(b) * a.max_blocks + pidx];
        if (page < 0 || page >= a.num_pages) {
            if (w == 0 && is_v == 0) raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
            continue;
        }
        const uint4 src = reinterpret_cast<const uint4*>((is_v ? a.v : a.k) + row * a.d)[w];
        uint8_t* dst = fp16_row(a.pool16, a.Hkv, a.d, a.P, page, h, is_v, static_cast<int>(pos % a.P));
        reinterpret_cast<uint4*>(dst)[w] = src;
    }
}

// positions 0 .. seq_lens[b]-1 of the INT4 pool -> the FP16 pool, same pages and slots.
// One CTA per (page index j, sequence b) covers the Hkv blocks of that page; each value
// is (nibble - 8) * scale, exact in fp32, rounded to fp16 (nearest even).
__global__ void __launch_bounds__(256) dequantize_to_fp16_kernel(Fp16DequantArgs a) {
    const int b = blockIdx.y;
    const long long j = blockIdx.x;
    int len = a.seq_lens[b];
    len = len < 0 ? 0 : len;
    const long long need = (static_cast<long long>(len) + a.L.P - 1) / a.L.P;
    if (j >= need) return;
    if (j >= a.max_blocks) {
        if (threadIdx.x == 0) raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
        return;
    }
    const int page = a.block_table[static_cast<long long>(b) * a.max_blocks + j];
    if (page < 0 || page >= a.num_pages) {
        if (threadIdx.x == 0) raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
        return;
    }
    const int d = a.L.d;
    const int words = d / 8;
    const long long rows_here = static_cast<long long>(len) - j * a.L.P;  // positions in this page
    const int slots = rows_here < a.L.P ? static_cast<int>(rows_here) : a.L.P;
    const int total = a.Hkv * 2 * slots * words;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int w = i % words;
        const int r = i / words;  // (h * 2 + is_v) * slots + slot
        const int slot = r % slots;
        const int is_v = (r / slots) & 1;
        const int h = r / (2 * slots);
        const uint8_t* blk = a.pool + (static_cast<long long>(page) * a.Hkv + h) * a.L.bytes;
        const int G = is_v ? a.L.Gv : a.L.Gk;
        const uint32_t word = reinterpret_cast<const uint32_t*>(blk + (is_v ? a.L.v_codes : 0) + slot * (d / 2))[w];
        const float s = __half2float(
            reinterpret_cast<const __half*>(blk + (is_v ? a.L.v_scales : a.L.k_scales) + slot * (d / G) * 2)[(w * 8) / G]);
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = static_cast<float>(static_cast<int>((word >> (4 * k)) & 0xFu) - 8) * s;
        uint4 pk;
        pk.x = pack_h2(v[0], v[1]);
        pk.y = pack_h2(v[2], v[3]);
        pk.z = pack_h2(v[4], v[5]);
        pk.w = pack_h2(v[6], v[7]);
        reinterpret_cast<uint4*>(fp16_row(a.pool16, a.Hkv, d, a.L.P, page, h, is_v, slot))[w] = pk;
    }
}

// INT8 per-row codec ("AI inference tuning: KV Cache optimisation and memory management"
// section 3.1): rows k, v [B, n_new, Hkv, d] fp16 -> the INT8 pool at start_pos[b] + t,
// scale = amax / 127 (IEEE division, floor 1e-8), code = clamp(rne(x / scale), -128, 127)
// with x / scale the IEEE quotient.  Block (page, kv head): K codes P x d int8, V codes
// P x d int8, K scales P fp32, V scales P fp32.
//
// The 16 values a lane holds (row values 16 tl .. 16 tl + 15) as 16 code bytes, and the
// row's scale.  With rs = rcp(s) (relative error below 2^-22) the exact product p = x rs is
// within |q| 2^-22 < 2^-14.9 of the quotient q = x / s (|q| <= 127 (1 + 2^-24), since
// s >= amax / 127 rounded), and the IEEE quotient is within 2^-18 of q (|q| < 128):
//  * m = fma(x, rs, 1.5 * 2^23) rounds p to an integer r once; m's bit pattern is
//    0x4B400000 + r, so its low byte is r as a two's-complement byte (|r| <= 127);
//  * e = fma(x, rs, -r) is p - r rounded once.  When |e| <= 1/2 - 2^-13 for all of the
//    lane's values, the IEEE quotient is within 1/2 - 2^-13 + 2^-14.9 + 2^-18 + 2^-25 < 1/2
//    of r, so rounding it gives r (no tie, no clamp); otherwise the lane takes the IEEE
//    division and the clamp for all its values.  A NaN or infinite input, or an infinite
//    scale, gives a NaN e for that input, so those rows take the same slower path.
// The slower path: the IEEE quotient of each value by s, rounded half to even, clamped.
// Out of line, so the common path keeps its registers.
__device__ __noinline__ uint4 int8_slow16(uint4 r0, uint4 r1, float s) {
    const uint32_t words[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
    uint32_t out[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&words[w]));
        const float c0 = fminf(fmaxf(rintf(__fdiv_rn(f.x, s)), -128.f), 127.f);
        const float c1 = fminf(fmaxf(rintf(__fdiv_rn(f.y, s)), -128.f), 127.f);
        const uint32_t b = (static_cast<uint32_t>(static_cast<int>(c0)) & 0xffu) |
                           ((static_cast<uint32_t>(static_cast<int>(c1)) & 0xffu) << 8);
        out[w >> 1] |= b << (16 * (w & 1));
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

template <int LPR>
__device__ __forceinline__ uint4 int8_lane16(const uint4 (&raw)[2], float& scale_out) {
    float x[16];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint4 r4 = raw[w >> 2];
        const uint32_t word = (w & 3) == 0 ? r4.x : (w & 3) == 1 ? r4.y : (w & 3) == 2 ? r4.z : r4.w;
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&word));
        x[2 * w] = f.x;
        x[2 * w + 1] = f.y;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int off = 1; off < LPR; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    float s = __fdiv_rn(amax, 127.0f);
    if (s < 1e-8f) s = 1e-8f;
    scale_out = s;
    float rs;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rs) : "f"(s));
    constexpr float kMagic = 12582912.0f;          // 1.5 * 2^23
    constexpr float kBand = 0.4998779296875f;      // 1/2 - 2^-13
    uint32_t m[16];
    float emax = 0.f;  // the largest |e|, NaN if any e is NaN
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float mi = fmaf(x[i], rs, kMagic);
        const float e = fmaf(x[i], rs, kMagic - mi);  // kMagic - mi = -r exactly
        emax = max_abs_nan(emax, e);
        m[i] = __float_as_uint(mi);
    }
    const bool slow = !(emax <= kBand);
    if (slow) return int8_slow16(raw[0], raw[1], s);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        w[k] = prmt(prmt(m[4 * k], m[4 * k + 1], 0x0040u), prmt(m[4 * k + 2], m[4 * k + 3], 0x0040u), 0x5410u);
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Work mapping as in the INT4 quantize kernel: rows (a token of one kv head) go to warps
// in blocks of 32, lane l first looking up where row l of the block goes (its block and
// slot); a job is the K or the V row of a row, held by a team of LPR = D / 16 lanes, 16
// values a lane; the warp takes a block's 64 jobs TEAMS * 2 at a time, loading the next
// pass's fp16 rows before it computes the current one.  Blocks are grid-strided over one
// wave of resident CTAs.
template <int D>
__global__ void __launch_bounds__(256, 3) int8_quantize_kernel(Fp16AppendArgs a) {
    constexpr int LPR = D / 16;
    constexpr int TEAMS = 32 / LPR;
    constexpr int U = 2;
    constexpr int JPP = TEAMS * U;
    constexpr int PASSES = 64 / JPP;
    const int lane = threadIdx.x & 31;
    const int team = lane / LPR;
    const int tl = lane % LPR;
    const long long rows = static_cast<long long>(a.B) * a.n_new * a.Hkv;
    const long long blocks = (rows + 31) / 32;
    const long long block_bytes = 2LL * a.P * D + 8LL * a.P;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const long long warps_total = static_cast<long long>(gridDim.x) * blockDim.x / 32;
    auto load = [&](long long row0, int ps, uint4 (&raw)[U][2]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jl = ps * JPP + u * TEAMS + team;
            const long long row = row0 + (jl >> 1);
            raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);
            if (row < rows) {
                const __half* src = ((jl & 1) ? a.v : a.k) + row * D + tl * 16;
                raw[u][0] = __ldcs(reinterpret_cast<const uint4*>(src));
                raw[u][1] = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
            }
        }
    };
    for (long long blk = warp_global; blk < blocks; blk += warps_total) {
        const long long row0 = blk * 32;
        // row row0 + lane: ((b * n_new + t) * Hkv + h); its block address and slot, or 0 when
        // the row is past the end or skipped (flagged)
        unsigned long long my_dst = 0ull;
        int my_slot = 0;
        if (row0 + lane < rows) {
            const long long row = row0 + lane;
            const int h = static_cast<int>(row % a.Hkv);
            const long long tok = row / a.Hkv;
            const int b = static_cast<int>(tok / a.n_new);
            const long long pos = static_cast<long long>(a.start_pos[b]) + (tok - static_cast<long long>(b) * a.n_new);
            const long long pidx = pos >= 0 ? pos / a.P : -1;
            if (pidx < 0 || pidx >= a.max_blocks) {
                raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
            } else {
                const int page = a.block_table[static_cast<long long>(b) * a.max_blocks + pidx];
                if (page < 0 || page >= a.num_pages) {
                    raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
                } else {
                    my_slot = static_cast<int>(pos - pidx * a.P);
                    my_dst = reinterpret_cast<unsigned long long>(a.pool16 +
                                                                  (static_cast<long long>(page) * a.Hkv + h) * block_bytes);
                }
            }
        }
        uint4 raw[U][2];
        load(row0, 0, raw);
#pragma unroll 1
        for (int ps = 0; ps < PASSES; ++ps) {
            uint4 nxt[U][2];
            if (ps + 1 < PASSES) load(row0, ps + 1, nxt);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int jl = ps * JPP + u * TEAMS + team;
                const int is_v = jl & 1;
                float sc;
                const uint4 codes = int8_lane16<LPR>(raw[u], sc);
                const unsigned long long dst = __shfl_sync(0xffffffffu, my_dst, jl >> 1);
                const int slot = __shfl_sync(0xffffffffu, my_slot, jl >> 1);
                if (dst == 0ull) continue;
                uint8_t* blkp = reinterpret_cast<uint8_t*>(dst);
                reinterpret_cast<uint4*>(blkp + (static_cast<long long>(is_v) * a.P + slot) * D)[tl] = codes;
                if (tl == 0) *reinterpret_cast<float*>(blkp + 2LL * a.P * D + 4LL * (is_v * a.P + slot)) = sc;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                raw[u][0] = nxt[u][0];
                raw[u][1] = nxt[u][1];
            }
        }
    }
}

}  // namespace

cudaError_t launch_int8_quantize_append(const Fp16AppendArgs& a, cudaStream_t stream) {
    const long long rows = 2LL * a.B * a.n_new * a.Hkv;
    if (rows == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    // one wave of 256-thread CTAs (3 per SM), 8 warps each taking blocks of 32 rows
    const long long rows32 = (rows / 2 + 31) / 32;
    const long long want = (rows32 + 7) / 8;
    const long long grid = want < 3LL * sms ? want : 3LL * sms;
    switch (a.d) {
        case 64: int8_quantize_kernel<64><<<static_cast<unsigned>(grid), 256, 0, stream>>>(a); break;
        case 128: int8_quantize_kernel<128><<<static_cast<unsigned>(grid), 256, 0, stream>>>(a); break;
        case 256: int8_quantize_kernel<256><<<static_cast<unsigned>(grid), 256, 0, stream>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_fp16_append(const Fp16AppendArgs& a, cudaStream_t stream) {
    const long long total = 2LL * a.B * a.n_new * a.Hkv * (a.d / 8);
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long want = (total + 255) / 256;
    const long long grid = want < 8LL * sms ? want : 8LL * sms;
    fp16_append_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_dequantize_to_fp16(const Fp16DequantArgs& a, long long max_pages, cudaStream_t stream) {
    if (max_pages <= 0 || a.B <= 0) return cudaSuccess;
    if (max_pages > 0x7fffffffLL || a.B > 65535) return cudaErrorInvalidValue;
    dequantize_to_fp16_kernel<<<dim3(static_cast<unsigned>(max_pages), static_cast<unsigned>(a.B)), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvq
