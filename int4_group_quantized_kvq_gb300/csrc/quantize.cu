// quantize.cu -- quantize-on-append: fp16 K/V rows -> packed INT4 codes + fp16 group
// scales written into their (page, kv-head) blocks.
//
// "4-bit KV cache compression" (lpnh.cn/news/2042373), section 2.1: per group of G
// elements along head_dim, scale = amax / 7 (an all-zero group gets 1), code =
// round(x / scale) clamped to [-7, 7].  Here scale = fp16_rne(fp32(amax) / 7.0f), the
// zero test is on that fp16 value, and code = round_half_even(fp32(x) / fp32(scale)),
// computed exactly without a per-element division (kvq_quant.cuh, shared with the decode
// step's fused append), so codes and scales are bit-exact functions of the input.
#include <cuda_fp16.h>

#include <atomic>

#include "kvq_device.cuh"
#include "kvq_internal.h"
#include "kvq_quant.cuh"

namespace kvq {
namespace {

// The 16 values a lane holds (row values 16 tl .. 16 tl + 15, inside one group) as 16
// nibbles (code + 8, element 2j low), low word first, and the group's fp16 scale.  The
// codes are those of quant_lane8 (kvq_quant.cuh, which the decode step's fused append
// uses), computed with fewer instructions for the common case:
//  * y = x * rcp(s) plus 1.5 * 2^23 + 8 rounds y + 8 to an integer, ties to even (8 is
//    even), whose low four bits are the nibble whenever the code needs no clamp;
//  * a lane takes the slower path of quant_lane8's arithmetic (the exact half-integer
//    check and the clamp) for all its values when one of them lies within 2^-16 of a
//    half-integer or the group's largest |y| exceeds 7.49.  The band is safe: y is
//    within 2^-17.6 of the quotient q for |q| < 16 (kvq_quant.cuh), and q is either a
//    half-integer or more than 2^-13 from every one, so outside the band y and q round
//    alike; and it is narrow, so a warp's 512 values rarely send it down the slower path
//    (a 2^-10 band did for most warps);
//  * a NaN input makes its |y - round(y)| NaN, and an infinite scale (from an infinite
//    input) makes that input's y = inf * 0 = NaN, so both reach the slower path through
//    the same test (written to hold for NaN); there they take the IEEE division, as in
//    quant_lane8;
//  * nibbles are paired into bytes by one shift and one bit select, and four bytes
//    gathered into a word by three byte permutes.
// LPR lanes hold a row; a group spans 1 << lg16 lanes.
template <int LPR>
__device__ __forceinline__ uint2 quant_lane16(const uint4 (&raw)[2], int lg16, __half& scale_out) {
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
    for (int off = 1; off < LPR; off <<= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, amax, off);
        if (off < (1 << lg16)) amax = fmaxf(amax, other);
    }
    __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
    if ((__half_as_ushort(s16) & 0x7fffu) == 0) s16 = __ushort_as_half(0x3c00u);
    const float s = __half2float(s16);
    scale_out = s16;
    float rs;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rs) : "f"(s));
    constexpr float kMagic8 = 12582920.0f;  // 1.5 * 2^23 + 8
    constexpr float kBand = 0.4999847412109375f;  // 1/2 - 2^-16
    bool slow = amax * rs > 7.49f;
    uint32_t byt[8];  // byte j (low 8 bits): the nibbles of values 2j and 2j + 1
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const float y0 = x[2 * j] * rs, y1 = x[2 * j + 1] * rs;
        const float m0 = y0 + kMagic8, m1 = y1 + kMagic8;
        slow |= !(fabsf(y0 - (m0 - kMagic8)) <= kBand);
        slow |= !(fabsf(y1 - (m1 - kMagic8)) <= kBand);
        byt[j] = (__float_as_uint(m0) & 0xFu) | ((__float_as_uint(m1) << 4) & ~0xFu);
    }
    uint32_t lo = prmt(prmt(byt[0], byt[1], 0x0040u), prmt(byt[2], byt[3], 0x0040u), 0x5410u);
    uint32_t hi = prmt(prmt(byt[4], byt[5], 0x0040u), prmt(byt[6], byt[7], 0x0040u), 0x5410u);
    if (slow) {
        bool plain = isinf(s);
#pragma unroll
        for (int i = 0; i < 16; ++i) plain |= x[i] != x[i];
        lo = quant8(*reinterpret_cast<const float(*)[8]>(&x[0]), s, plain);
        hi = quant8(*reinterpret_cast<const float(*)[8]>(&x[8]), s, plain);
    }
    return make_uint2(lo, hi);
}

// Quantize one row job (a K or V row of one (sequence, token, kv head)) held as 16
// values per lane, and store its codes and scales.  Every lane of the warp calls this
// together (the group maximum is a shuffle reduction); `active` marks real jobs.
template <int D>
__device__ __forceinline__ void quantize_row(const QuantizeArgs& a, const uint4 (&raw)[2], uint32_t job, bool active,
                                             int tl) {
    const int is_v = static_cast<int>(job & 1u);
    const int lg = (is_v ? a.lg_lanes_v : a.lg_lanes_k) - 1;  // log2 of the 16-value lanes per group
    __half s16;
    const uint2 words = quant_lane16<D / 16>(raw, lg, s16);
    if (!active) return;

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
    reinterpret_cast<uint2*>(codes)[tl] = words;
    if ((tl & ((1 << lg) - 1)) == 0) {
        const int ngroups = D >> (lg + 4);
        uint8_t* scales = blk + (is_v ? a.L.v_scales : a.L.k_scales) + slot * ngroups * 2;
        reinterpret_cast<__half*>(scales)[tl >> lg] = s16;
    }
}

// Work mapping: jobs are (row, K or V) pairs, K and V of a row adjacent.  A warp takes
// TEAMS jobs at a time, U times over, loading all U x 32 bytes per lane before it
// computes, so enough loads are in flight to stream from HBM.  The job loop is
// grid-strided over a grid of one wave of resident CTAs.
template <int D, int U>
__global__ void __launch_bounds__(256, 4) quantize_append_kernel(QuantizeArgs a) {
    // A decode launched behind this kernel may start its own set-up now; it waits for this
    // grid to finish before it reads the pool.  This kernel itself may start before the
    // kernel ahead of it (a decode that reads the pool) has finished: it waits for it
    // before anything else.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int LPR = D / 16;           // lanes per row
    constexpr int TEAMS = 32 / LPR;       // row jobs per warp at a time
    const int lane = threadIdx.x & 31;
    const int team = lane / LPR;
    const int tl = lane % LPR;            // lane within the team
    const uint32_t jobs = 2u * a.rows;
    const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const uint32_t warps_total = gridDim.x * blockDim.x / 32;
    for (uint32_t base = warp_global * TEAMS * U; base < jobs; base += warps_total * TEAMS * U) {
        uint4 raw[U][2];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t job = base + u * TEAMS + team;
            raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);
            if (job < jobs) {
                const __half* src = ((job & 1u) ? a.v : a.k) + static_cast<size_t>(job >> 1) * D + tl * 16;
                raw[u][0] = __ldcs(reinterpret_cast<const uint4*>(src));  // read once: stream past the caches
                raw[u][1] = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
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
    constexpr int U = 2;
    const long long jobs = 2LL * a.rows;
    if (jobs == 0) return cudaSuccess;
    constexpr int threads = 256;
    constexpr int jobs_per_block = (threads / 32) * (32 / (D / 16)) * U;
    long long blocks = (jobs + jobs_per_block - 1) / jobs_per_block;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * quantize_ctas_per_sm<D, U>();
    if (blocks > cap) blocks = cap;
    // programmatic dependent launch: the CTAs may become resident while the kernel ahead
    // drains; the kernel waits for it with griddepcontrol.wait before touching memory
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, quantize_append_kernel<D, U>, a);
    if (err != cudaSuccess) return err;
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
