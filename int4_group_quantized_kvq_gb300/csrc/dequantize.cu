// dequantize.cu -- packed INT4 pages -> dense K/V rows.
//
// "4-bit KV cache compression" (lpnh.cn/news/2042373), section 2.1: the stored
// value is code * scale.  With code in [-7, 7] and an fp16 scale the product is
// exact in fp32; the fp16 output is that product rounded to nearest even.
//
// One thread produces 8 consecutive elements of one row (one 32-bit word of codes).
#include <cuda_fp16.h>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

__global__ void __launch_bounds__(256) dequantize_kernel(DequantArgs a) {
    const int d = a.L.d;
    const int words = d / 8;  // per row
    const long long total = 2LL * a.n * a.Hkv * words;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int w = static_cast<int>(i % words);
        const long long rowkv = i / words;       // ((t * Hkv + h) * 2 + is_v)
        const int is_v = static_cast<int>(rowkv & 1);
        const long long row = rowkv >> 1;        // t * Hkv + h
        const int h = static_cast<int>(row % a.Hkv);
        const int t = static_cast<int>(row / a.Hkv);
        const long long pos = static_cast<long long>(a.start) + t;
        long long pidx = pos / a.L.P;
        int page = 0;
        if (pidx >= a.max_blocks) {
            if (w == 0) raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
            pidx = -1;
        } else {
            page = a.block_table[static_cast<long long>(a.b) * a.max_blocks + pidx];
            if (page < 0 || page >= a.num_pages) {
                if (w == 0) raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
                page = 0;
            }
        }
        const int slot = static_cast<int>(pos % a.L.P);
        const uint8_t* blk = a.pool + (static_cast<long long>(page) * a.Hkv + h) * a.L.bytes;
        const int G = is_v ? a.L.Gv : a.L.Gk;
        const uint32_t word =
            reinterpret_cast<const uint32_t*>(blk + (is_v ? a.L.v_codes : 0) + slot * (d / 2))[w];
        const __half s16 =
            reinterpret_cast<const __half*>(blk + (is_v ? a.L.v_scales : a.L.k_scales) + slot * (d / G) * 2)[(w * 8) / G];
        const float s = __half2float(s16);
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = static_cast<float>(static_cast<int>((word >> (4 * k)) & 0xFu) - 8) * s;
        if (pidx < 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = 0.f;
        }
        const long long o = row * d + w * 8;
        void* dst = is_v ? a.out_v : a.out_k;
        if (a.out_fp32) {
            float4* p = reinterpret_cast<float4*>(static_cast<float*>(dst) + o);
            p[0] = make_float4(v[0], v[1], v[2], v[3]);
            p[1] = make_float4(v[4], v[5], v[6], v[7]);
        } else {
            uint4 pk;
            pk.x = pack_h2(v[0], v[1]);
            pk.y = pack_h2(v[2], v[3]);
            pk.z = pack_h2(v[4], v[5]);
            pk.w = pack_h2(v[6], v[7]);
            *reinterpret_cast<uint4*>(static_cast<__half*>(dst) + o) = pk;
        }
    }
}

}  // namespace

cudaError_t launch_dequantize(const DequantArgs& a, cudaStream_t stream) {
    const long long total = 2LL * a.n * a.Hkv * (a.L.d / 8);
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    dequantize_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvq
