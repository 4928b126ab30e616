// wht_codec.cu -- the rotated 4-bit codec ("LARQL KV cache engines", engine three,
// codec/turbo-quant: each K or V row of a head is rotated by a Walsh-Hadamard transform
// and quantized with a Lloyd-Max codebook; head_dim a power of two; about 0.9954 per-row
// cosine at 4 bits): its codebook, quantize-on-append and dequantization.
//
// Per row x (d = 128 values, fp16 in, fp32 arithmetic, each operation rounded once):
//   y = H x, H the unnormalised Sylvester-order Walsh-Hadamard matrix, by the fast
//     transform with stages of span 1, 2, 4, .., 64;
//   sigma = sqrt(sum x_i^2), the squares summed in fixed pairs: lane l of a warp holds
//     x_{4l} .. x_{4l+3} and forms (x0^2 + x1^2) + (x2^2 + x3^2), then the lanes add
//     their partners' sums at xor distances 16, 8, 4, 2, 1 (sigma is the RMS of y, as
//     H H = d I);
//   code_i = #{j : y_i / sigma >= T_j}, T_j the fp32 midpoints of the 16 Lloyd-Max
//     levels of the standard normal; sigma = 0 gives codes 0;
//   stored: the codes as nibbles (element 2j low), then sigma as fp32.
// Dequantized: x^ = H (sigma * c_code) / d, c the fp32 levels.  The decode kernel never
// dequantizes: it scores against H q and accumulates sigma * c in the rotated domain,
// rotating each partial back at its segment end (decode_fp16.cuh).
//
// Block (page, kv head): K codes P x 64 bytes, V codes P x 64, K sigma P fp32, V sigma
// P fp32: P * (d + 8) bytes.
#include <cmath>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// Standard normal density and upper tail, in double.
double npdf(double t) { return std::exp(-0.5 * t * t) * 0.39894228040143267794; }
double nupper(double t) { return 0.5 * std::erfc(t * 0.70710678118654752440); }

// The 16-level Lloyd-Max quantizer of the standard normal.  The law is symmetric, so
// only the 8 positive levels are iterated: level k (k = 0..7) is the mean of the normal
// on [b_k, b_{k+1}), b_0 = 0, b_k the midpoint of levels k-1 and k, b_8 = infinity;
// the mean of the normal on [a, b) is (pdf(a) - pdf(b)) / (upper(a) - upper(b)).
// Iterated from evenly spaced levels until no level moves by more than 1e-15.
Wht4Codebook make_codebook() {
    double pos[8];
    for (int k = 0; k < 8; ++k) pos[k] = 0.375 * (k + 0.5);
    for (int it = 0; it < 200000; ++it) {
        double lo = 0.0, moved = 0.0;
        for (int k = 0; k < 8; ++k) {
            const double hi = k + 1 < 8 ? 0.5 * (pos[k] + pos[k + 1]) : INFINITY;
            const double num = npdf(lo) - (std::isinf(hi) ? 0.0 : npdf(hi));
            const double den = nupper(lo) - (std::isinf(hi) ? 0.0 : nupper(hi));
            const double nk = num / den;
            moved = std::fmax(moved, std::fabs(nk - pos[k]));
            lo = hi;  // the next cell starts at the old midpoint (Jacobi-style sweep)
            pos[k] = nk;
        }
        if (moved <= 1e-15) break;
    }
    Wht4Codebook cb;
    double lv[16];
    for (int k = 0; k < 8; ++k) {
        lv[8 + k] = pos[k];
        lv[7 - k] = -pos[k];
    }
    for (int j = 0; j < 16; ++j) cb.levels[j] = static_cast<float>(lv[j]);
    for (int j = 1; j < 16; ++j) cb.thresholds[j - 1] = static_cast<float>(0.5 * (lv[j - 1] + lv[j]));
    return cb;
}

struct Wht4QuantArgs {
    Fp16AppendArgs a;
    float thr[15];
};

// fp32 fast Walsh-Hadamard transform of a 128-vector held 4 per lane (lane l: elements
// 4l .. 4l + 3), stages of span 1, 2 inside the lane, 4 .. 64 across lanes at xor
// distances 1 .. 16: the lower element of a pair becomes a + b, the upper a - b.
__device__ __forceinline__ void wht128(float (&y)[4], int lane) {
    float t0 = __fadd_rn(y[0], y[1]), t1 = __fsub_rn(y[0], y[1]);
    float t2 = __fadd_rn(y[2], y[3]), t3 = __fsub_rn(y[2], y[3]);
    y[0] = __fadd_rn(t0, t2);
    y[2] = __fsub_rn(t0, t2);
    y[1] = __fadd_rn(t1, t3);
    y[3] = __fsub_rn(t1, t3);
#pragma unroll
    for (int X = 1; X < 32; X <<= 1) {
        const bool upper = (lane & X) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float other = __shfl_xor_sync(0xffffffffu, y[j], X);
            y[j] = upper ? __fsub_rn(other, y[j]) : __fadd_rn(y[j], other);
        }
    }
}

// The row's codes for the 8 values a lane holds (row elements 8 tl .. 8 tl + 7, a team of
// 16 lanes per row), and the row's sigma.  Every step is the oracle's, in its order:
//  * sigma^2: squares summed in fours ((y0^2 + y1^2) + (y2^2 + y3^2), elements 4g .. 4g+3),
//    then the 32 sums pairwise at index distances 16, 8, 4, 2, 1 -- here lane distances 8,
//    4, 2, 1 for both of the lane's sums, then the lane's two sums;
//  * the transform's stages of span 1, 2, 4 inside the lane and 8 .. 64 across lanes at xor
//    distances 1 .. 8, the lower element of a pair becoming a + b and the upper a - b;
//  * u = y / sigma (IEEE division), the code the number of thresholds <= u, found by a
//    binary search over the 15 ascending thresholds (the same count as a linear scan, NaN
//    counting none); no codes (all 0) when sigma is not positive.
__device__ __forceinline__ uint32_t wht4_lane8(uint4 raw, const float* thr, int tl, float& sigma_out) {
    float y[8];
    {
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
            y[2 * k] = f.x;
            y[2 * k + 1] = f.y;
        }
    }
    float s0 = __fadd_rn(__fadd_rn(__fmul_rn(y[0], y[0]), __fmul_rn(y[1], y[1])),
                         __fadd_rn(__fmul_rn(y[2], y[2]), __fmul_rn(y[3], y[3])));
    float s1 = __fadd_rn(__fadd_rn(__fmul_rn(y[4], y[4]), __fmul_rn(y[5], y[5])),
                         __fadd_rn(__fmul_rn(y[6], y[6]), __fmul_rn(y[7], y[7])));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) {
        s0 = __fadd_rn(s0, __shfl_xor_sync(0xffffffffu, s0, off));
        s1 = __fadd_rn(s1, __shfl_xor_sync(0xffffffffu, s1, off));
    }
    const float sigma = __fsqrt_rn(__fadd_rn(s0, s1));
    sigma_out = sigma;
#pragma unroll
    for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if ((j & h) == 0) {
                const float a = y[j], b = y[j + h];
                y[j] = __fadd_rn(a, b);
                y[j + h] = __fsub_rn(a, b);
            }
    // across lanes: lower a + b, upper a - b, as other + sgn * mine with sgn = +-1 (one
    // rounding of the exact sum, so the same value as the add or the subtract)
#pragma unroll
    for (int X = 1; X < 16; X <<= 1) {
        const float sgn = (tl & X) != 0 ? -1.f : 1.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) y[j] = fmaf(y[j], sgn, __shfl_xor_sync(0xffffffffu, y[j], X));
    }
    uint32_t packed = 0;
    if (sigma > 0.f) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float u = __fdiv_rn(y[j], sigma);
            int c = u >= thr[7] ? 8 : 0;
            c += u >= thr[c + 3] ? 4 : 0;
            c += u >= thr[c + 1] ? 2 : 0;
            c += u >= thr[c] ? 1 : 0;
            packed |= static_cast<uint32_t>(c) << (4 * j);
        }
    }
    return packed;
}

// Work mapping as in the INT4 quantize kernel: rows (a token of one kv head, in the order
// (b, t, h)) go to warps in blocks of 32, lane l looking up where row l goes; a job is the
// K or the V row of a row, held by a team of 16 lanes, 8 values a lane; the warp takes a
// block's 64 jobs four at a time, loading the next pass's rows before it computes.
__global__ void __launch_bounds__(256) wht4_quantize_kernel(Wht4QuantArgs w) {
    const Fp16AppendArgs& a = w.a;
    __shared__ float thr[16];
    if (threadIdx.x < 15) thr[threadIdx.x] = w.thr[threadIdx.x];
    __syncthreads();
    constexpr int LPR = 16, TEAMS = 2, U = 2, JPP = TEAMS * U, PASSES = 64 / JPP;
    const int lane = threadIdx.x & 31;
    const int team = lane / LPR;
    const int tl = lane % LPR;
    const long long rows = static_cast<long long>(a.B) * a.n_new * a.Hkv;
    const long long blocks = (rows + 31) / 32;
    const long long block_bytes = static_cast<long long>(a.P) * (128 + 8);
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const long long warps_total = static_cast<long long>(gridDim.x) * blockDim.x / 32;
    auto load = [&](long long row0, int ps, uint4 (&raw)[U]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jl = ps * JPP + u * TEAMS + team;
            const long long row = row0 + (jl >> 1);
            raw[u] = make_uint4(0, 0, 0, 0);
            if (row < rows) raw[u] = __ldcs(reinterpret_cast<const uint4*>(((jl & 1) ? a.v : a.k) + row * 128) + tl);
        }
    };
    for (long long blk = warp_global; blk < blocks; blk += warps_total) {
        const long long row0 = blk * 32;
        unsigned long long my_dst = 0ull;  // the row's block, or 0 when past the end or skipped (flagged)
        int my_slot = 0;
        if (row0 + lane < rows) {
            const long long row = row0 + lane;  // (b * n_new + t) * Hkv + h
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
        uint4 raw[U];
        load(row0, 0, raw);
#pragma unroll 1
        for (int ps = 0; ps < PASSES; ++ps) {
            uint4 nxt[U];
            if (ps + 1 < PASSES) load(row0, ps + 1, nxt);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int jl = ps * JPP + u * TEAMS + team;
                const int is_v = jl & 1;
                float sigma;
                const uint32_t codes = wht4_lane8(raw[u], thr, tl, sigma);
                const unsigned long long dst = __shfl_sync(0xffffffffu, my_dst, jl >> 1);
                const int slot = __shfl_sync(0xffffffffu, my_slot, jl >> 1);
                if (dst == 0ull) continue;
                uint8_t* blkp = reinterpret_cast<uint8_t*>(dst);
                reinterpret_cast<uint32_t*>(blkp + (static_cast<long long>(is_v) * a.P + slot) * 64)[tl] = codes;
                if (tl == 0) *reinterpret_cast<float*>(blkp + 128LL * a.P + 4LL * (is_v * a.P + slot)) = sigma;
            }
#pragma unroll
            for (int u = 0; u < U; ++u) raw[u] = nxt[u];
        }
    }
}

struct Wht4DequantArgs {
    const uint8_t* pool;
    const int32_t* block_table;
    float* out_k;
    float* out_v;
    uint32_t* status;
    int32_t max_blocks, b, start, n, Hkv, P, num_pages;
    float lut[16];
};

// One warp per (position, kv head, K or V): x^ = H (sigma * c_code) / 128 in fp32.
__global__ void __launch_bounds__(256) wht4_dequantize_kernel(Wht4DequantArgs w) {
    const int lane = threadIdx.x & 31;
    const long long rows = 2LL * w.n * w.Hkv;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    const long long block_bytes = static_cast<long long>(w.P) * (128 + 8);
    for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += nwarps) {
        const int is_v = static_cast<int>(r & 1);
        const long long row = r >> 1;  // t * Hkv + h
        const int h = static_cast<int>(row % w.Hkv);
        const int t = static_cast<int>(row / w.Hkv);
        const long long pos = static_cast<long long>(w.start) + t;
        float* dst = (is_v ? w.out_v : w.out_k) + row * 128;
        const int page = pos / w.P < w.max_blocks
                             ? w.block_table[static_cast<long long>(w.b) * w.max_blocks + pos / w.P]
                             : -1;
        if (page < 0 || page >= w.num_pages) {
            if (lane == 0 && is_v == 0) raise_flag(w.status, KVQ_FLAG_BAD_PAGE);
            reinterpret_cast<float4*>(dst)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        const int slot = static_cast<int>(pos % w.P);
        const uint8_t* blk = w.pool + (static_cast<long long>(page) * w.Hkv + h) * block_bytes;
        const uint32_t code = *reinterpret_cast<const uint16_t*>(blk + (static_cast<long long>(is_v) * w.P + slot) * 64 +
                                                                 2 * lane);
        const float sigma = *reinterpret_cast<const float*>(blk + 128LL * w.P + 4LL * (is_v * w.P + slot));
        float y[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) y[j] = sigma * w.lut[(code >> (4 * j)) & 15];
        wht128(y, lane);
        reinterpret_cast<float4*>(dst)[lane] =
            make_float4(y[0] * 0.0078125f, y[1] * 0.0078125f, y[2] * 0.0078125f, y[3] * 0.0078125f);
    }
}

int resident_grid(long long rows_per_8) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    const long long grid = rows_per_8 < 8LL * sms ? rows_per_8 : 8LL * sms;
    return static_cast<int>(grid);
}

}  // namespace

const Wht4Codebook& wht4_codebook() {
    static const Wht4Codebook cb = make_codebook();
    return cb;
}

cudaError_t launch_wht4_quantize_append(const Fp16AppendArgs& a, cudaStream_t stream) {
    const long long rows = 2LL * a.B * a.n_new * a.Hkv;
    if (rows == 0) return cudaSuccess;
    const int grid = resident_grid(((rows / 2 + 31) / 32 + 7) / 8);  // CTAs of 8 warps, blocks of 32 rows
    if (grid < 0) return cudaErrorUnknown;
    Wht4QuantArgs w;
    w.a = a;
    const Wht4Codebook& cb = wht4_codebook();
    for (int k = 0; k < 15; ++k) w.thr[k] = cb.thresholds[k];
    wht4_quantize_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(w);
    return cudaGetLastError();
}

cudaError_t launch_wht4_dequantize(const uint8_t* pool, const int32_t* block_table, int32_t max_blocks, int32_t b,
                                   int32_t start, int32_t n, float* out_k, float* out_v, uint32_t* status,
                                   int32_t Hkv, int32_t P, int32_t num_pages, cudaStream_t stream) {
    const long long rows = 2LL * n * Hkv;
    if (rows == 0) return cudaSuccess;
    const int grid = resident_grid((rows + 7) / 8);
    if (grid < 0) return cudaErrorUnknown;
    Wht4DequantArgs w;
    w.pool = pool;
    w.block_table = block_table;
    w.out_k = out_k;
    w.out_v = out_v;
    w.status = status;
    w.max_blocks = max_blocks;
    w.b = b;
    w.start = start;
    w.n = n;
    w.Hkv = Hkv;
    w.P = P;
    w.num_pages = num_pages;
    const Wht4Codebook& cb = wht4_codebook();
    for (int k = 0; k < 16; ++k) w.lut[k] = cb.levels[k];
    wht4_dequantize_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(w);
    return cudaGetLastError();
}

}  // namespace kvq
