// quantize.cu -- quantize-on-append: fp16 K/V rows -> packed INT4 codes + fp16 group
// scales written into their (page, kv-head) blocks.
//
// "4-bit KV cache compression" (lpnh.cn/news/2042373), section 2.1: per group of G
// elements along head_dim, scale = amax / 7 (an all-zero group gets 1), code =
// round(x / scale) clamped to [-7, 7].  Here scale = fp16_rne(fp32(amax) / 7.0f), the
// zero test is on that fp16 value, and code = round_half_even(fp32(x) / fp32(scale)),
// computed exactly without a per-element division (quant_code below), so codes and
// scales are bit-exact functions of the input.
#include <cuda_fp16.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

// round_half_even(fp32(x) / s) without a division per element.  x and s are fp16
// values (s > 0), so the quotient q = x / s is either exactly a half-integer or more
// than 2^-13 away from every half-integer: with x = X 2^a and s = S 2^b (integers
// X, S < 2048), q - (k + 1/2) = (2 X 2^(a-b) - (2k + 1) S) / (2 S), whose numerator is
// a nonzero multiple of min(1, 2^(a-b)), and 2^(a-b) > S / 4096 whenever |q| >= 1/2.
// The fp32 quotient the definition rounds is therefore on the same side of every
// half-integer as q.  y = x * rs, with rs within 2 ulp of 1/s, is within 2^-18 of q for
// |q| < 16 (the quotient never reaches 16 for finite input: the fp16 scale is at least
// two thirds of amax / 7), so rounding y gives the same code unless y is within 2^-10
// of a half-integer h; there the sign of x - h s, exact in one fma because h s has at
// most 15 significant bits, decides, with ties to even.
__device__ __forceinline__ int exact_code(float x, float s, float y) {
    const float h = floorf(y) + 0.5f;    // the half-integer next to y (when y is near one)
    const float r = fmaf(-h, s, x);      // sign of x - h s, exact
    const int lo = __float2int_rd(h);
    return r > 0.f ? lo + 1 : (r < 0.f ? lo : lo + (lo & 1));
}

// The 8 codes of one lane as nibbles (code + 8, low nibble first) of a 32-bit word.
__device__ __forceinline__ uint32_t quant8(const float (&x)[8], float s, bool plain) {
    int c[8];
    if (plain) {
        // an infinite scale or a NaN input: the plain conversion of the IEEE quotient
        // (a NaN quotient converts to 0)
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = __float2int_rn(__fdiv_rn(x[i], s));
    } else {
        float rs;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rs) : "f"(s));
        constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer, ties to even
        bool near = false;
        float y[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            y[i] = x[i] * rs;
            const float m = y[i] + kMagic;
            c[i] = __float_as_int(m) - 0x4B400000;
            near |= fabsf(y[i] - (m - kMagic)) > 0.4990234375f;
        }
        if (near) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (fabsf(y[i] - rintf(y[i])) > 0.4990234375f) c[i] = exact_code(x[i], s, y[i]);
        }
    }
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) word |= static_cast<uint32_t>(max(-7, min(7, c[i])) + 8) << (4 * i);
    return word;
}

// Quantize one row job (a K or V row of one (sequence, token, kv head)) held as 8
// values per lane, and store its codes and scales.  Every lane of the warp calls this
// together (the group maximum is a shuffle reduction); `active` marks real jobs.
template <int D>
__device__ __forceinline__ void quantize_row(const QuantizeArgs& a, uint4 raw, uint32_t job, bool active, int tl) {
    constexpr int LPR = D / 8;  // lanes per row
    const int is_v = static_cast<int>(job & 1u);
    const int lg = is_v ? a.lg_lanes_v : a.lg_lanes_k;  // log2 of the lanes per group
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
    // group maximum over the group's lanes (groups are aligned within the team).  The K
    // and V teams of a warp have different group widths, so every lane runs the same
    // shuffles and only folds in partners inside its own group.
#pragma unroll
    for (int off = 1; off < LPR; off <<= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, amax, off);
        if (off < (1 << lg)) amax = fmaxf(amax, other);
    }
    if (!active) return;
    __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
    if ((__half_as_ushort(s16) & 0x7fffu) == 0) s16 = __ushort_as_half(0x3c00u);
    const float s = __half2float(s16);
    bool nan = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) nan |= x[i] != x[i];
    const uint32_t word = quant8(x, s, nan || isinf(s));

    // destination: row = (b * n_new + t) * Hkv + h -> position, page, slot
    const uint32_t row = job >> 1;
    const uint32_t bt = fast_div(row, a.div_h);
    const int h = static_cast<int>(row - bt * static_cast<uint32_t>(a.Hkv));
    const uint32_t b = fast_div(bt, a.div_n);
    const int t = static_cast<int>(bt - b * static_cast<uint32_t>(a.n_new));
    const long long pos = static_cast<long long>(a.start_pos[b]) + t;
    const long long pidx = pos >> a.lg_p;
    if (pos < 0 || pidx >= a.max_blocks) {
        if (tl == 0) raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
        return;
    }
    const int page = a.block_table[static_cast<long long>(b) * a.max_blocks + pidx];
    if (page < 0 || page >= a.num_pages) {
        if (tl == 0) raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
        return;
    }
    const int slot = static_cast<int>(pos & ((1 << a.lg_p) - 1));
    uint8_t* blk = a.pool + (static_cast<long long>(page) * a.Hkv + h) * a.L.bytes;
    uint8_t* codes = blk + (is_v ? a.L.v_codes : 0) + slot * (D / 2);
    reinterpret_cast<uint32_t*>(codes)[tl] = word;
    if ((tl & ((1 << lg) - 1)) == 0) {
        const int ngroups = D >> (lg + 3);
        uint8_t* scales = blk + (is_v ? a.L.v_scales : a.L.k_scales) + slot * ngroups * 2;
        reinterpret_cast<__half*>(scales)[tl >> lg] = s16;
    }
}

// Work mapping: jobs are (row, K or V) pairs, K and V of a row adjacent.  A warp takes
// TEAMS jobs at a time, U times over, loading all U x 16 bytes per lane before it
// computes, so enough loads are in flight to stream from HBM.  The job loop is
// grid-strided over a grid of one wave of resident CTAs.
template <int D, int U>
__global__ void __launch_bounds__(256) quantize_append_kernel(QuantizeArgs a) {
    // a decode launched behind this kernel may start its own set-up now; it waits for
    // this grid to finish before it reads the pool
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int LPR = D / 8;            // lanes per row
    constexpr int TEAMS = 32 / LPR;       // row jobs per warp at a time
    const int lane = threadIdx.x & 31;
    const int team = lane / LPR;
    const int tl = lane % LPR;            // lane within the team
    const uint32_t jobs = 2u * a.rows;
    const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const uint32_t warps_total = gridDim.x * blockDim.x / 32;
    for (uint32_t base = warp_global * TEAMS * U; base < jobs; base += warps_total * TEAMS * U) {
        uint4 raw[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t job = base + u * TEAMS + team;
            raw[u] = make_uint4(0, 0, 0, 0);
            if (job < jobs) {
                const __half* src = ((job & 1u) ? a.v : a.k) + static_cast<size_t>(job >> 1) * D + tl * 8;
                raw[u] = __ldcs(reinterpret_cast<const uint4*>(src));  // read once: stream past the caches
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t job = base + u * TEAMS + team;
            quantize_row<D>(a, raw[u], job, job < jobs, tl);
        }
    }
}

// Resident 256-thread CTAs per SM of an instance, looked up once.
template <int D, int U>
int quantize_ctas_per_sm() {
    static std::atomic<int> memo{0};
    int n = memo.load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, quantize_append_kernel<D, U>, 256, 0) != cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        n = 1;
    }
    memo.store(n, std::memory_order_relaxed);
    return n;
}

template <int D>
cudaError_t launch_q(const QuantizeArgs& a, cudaStream_t stream) {
    constexpr int U = 4;
    const long long jobs = 2LL * a.rows;
    if (jobs == 0) return cudaSuccess;
    constexpr int threads = 256;
    constexpr int jobs_per_block = (threads / 32) * (32 / (D / 8)) * U;
    long long blocks = (jobs + jobs_per_block - 1) / jobs_per_block;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * quantize_ctas_per_sm<D, U>();
    if (blocks > cap) blocks = cap;
    quantize_append_kernel<D, U><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
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
