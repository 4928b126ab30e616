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
// section 3.1): rows k, v [B, n_new, Hkv, d] fp16 -> the INT8 pool at start_pos[b] + t.
// One warp per K or V row, lane l on values 4l .. 4l + 3 (and 128 + 4l .. for d = 256):
// scale = amax / 127 (IEEE division, floor 1e-8), code = clamp(rne(x / scale), -128, 127).
// Block (page, kv head): K codes P x d int8, V codes P x d int8, K scales P fp32, V
// scales P fp32.
__global__ void __launch_bounds__(256) int8_quantize_kernel(Fp16AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const long long rows = 2LL * a.B * a.n_new * a.Hkv;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long block_bytes = 2LL * a.P * a.d + 8LL * a.P;
    for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const int is_v = static_cast<int>(r & 1);
        const long long row = r >> 1;  // (b * n_new + t) * Hkv + h
        const int h = static_cast<int>(row % a.Hkv);
        const long long bt_ = row / a.Hkv;
        const int t = static_cast<int>(bt_ % a.n_new);
        const int b = static_cast<int>(bt_ / a.n_new);
        const long long pos = static_cast<long long>(a.start_pos[b]) + t;
        const long long pidx = pos >= 0 ? pos / a.P : -1;
        if (pidx < 0 || pidx >= a.max_blocks) {
            if (lane == 0 && is_v == 0) raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
            continue;
        }
        const int page = a.block_table[static_cast<long long>(b) * a.max_blocks + pidx];
        if (page < 0 || page >= a.num_pages) {
            if (lane == 0 && is_v == 0) raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
            continue;
        }
        const int slot = static_cast<int>(pos % a.P);
        const __half* src = (is_v ? a.v : a.k) + row * a.d;
        float x[2][4];
        float amax = 0.f;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const int c = lane + 32 * c2;  // 4-value chunk
            if (4 * c < a.d) {
                const uint2 w = reinterpret_cast<const uint2*>(src)[c];
                const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
                const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
                x[c2][0] = f0.x;
                x[c2][1] = f0.y;
                x[c2][2] = f1.x;
                x[c2][3] = f1.y;
#pragma unroll
                for (int j = 0; j < 4; ++j) amax = fmaxf(amax, fabsf(x[c2][j]));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        float sc = __fdiv_rn(amax, 127.0f);
        if (sc < 1e-8f) sc = 1e-8f;
        uint8_t* blk = a.pool16 + (static_cast<long long>(page) * a.Hkv + h) * block_bytes;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
            const int c = lane + 32 * c2;
            if (4 * c < a.d) {
                uint32_t w = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float q = rintf(__fdiv_rn(x[c2][j], sc));
                    q = fminf(fmaxf(q, -128.f), 127.f);
                    w |= (static_cast<uint32_t>(static_cast<int>(q)) & 0xffu) << (8 * j);
                }
                *reinterpret_cast<uint32_t*>(blk + (static_cast<long long>(is_v) * a.P + slot) * a.d + 4 * c) = w;
            }
        }
        if (lane == 0) *reinterpret_cast<float*>(blk + 2LL * a.P * a.d + 4LL * (is_v * a.P + slot)) = sc;
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
    const long long want = (rows + 7) / 8;
    const long long grid = want < 8LL * sms ? want : 8LL * sms;
    int8_quantize_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(a);
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
