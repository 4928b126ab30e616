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

// fp32(1/7).  For every fp16 value a >= 0 (subnormals and +inf included),
// fp16_rne(a * kInv7) == fp16_rne(fp32_rn(a / 7)): the product and the IEEE quotient
// may differ in the last fp32 bit, but never across an fp16 rounding boundary.  The
// domain is 31,745 values and the CPU tests check every one of them, so one multiply
// stands in for the division of the definition.
constexpr float kInv7 = 0.142857149f;  // 0x3E124925

// The 16 values a lane holds (row values 16 tl .. 16 tl + 15, inside one group) as 16
// nibbles (code + 8, element 2j low), low word first, and the group's fp16 scale.  The
// codes are those of quant_lane8 (kvq_quant.cuh, which the decode step's fused append
// uses), computed with fewer instructions for the common case.  With rs = rcp(s), within
// 2 ulp of 1/s, the exact product p = x rs is within |q| 2^-23 < 2^-19 of the quotient
// q = x / s for |q| < 16 (kvq_quant.cuh shows the quotient stays below 16).
//  * m = fma(x, rs, 1.5 * 2^23 + 8) rounds p + 8 to an integer once, ties to even (8 is
//    even), so r = m - (1.5 * 2^23 + 8) is the integer nearest p, and the low four bits of
//    m's bit pattern are the nibble r + 8 whenever the code needs no clamp;
//  * e = fma(x, rs, -r) is p - r rounded once (|p - r| <= 1/2, so within 2^-26).  When
//    |e| <= 1/2 - 2^-16 for all of the lane's values, q is within 1/2 - 2^-16 + 2^-26 +
//    2^-19 < 1/2 of r, so r is the nearest integer to q and no tie is possible; otherwise
//    (or when the group's largest |p| may exceed 7.49 and a clamp is possible) the lane takes
//    the slower path of quant_lane8's arithmetic, the exact half-integer check and the clamp,
//    for all its values.  The band is narrow: a warp's 512 values rarely send it there;
//  * a NaN input makes its e NaN, and an infinite scale (from an infinite input) makes that
//    input's e = inf * 0 = NaN, so both reach the slower path through the same test: the
//    lane's largest |e| is kept by a NaN-propagating maximum (one instruction a value) and
//    the test is written to hold for NaN; there they take the IEEE division, as in
//    quant_lane8;
//  * on the fast path a nibble n = r + 8 is in [1, 15] and m's bit pattern is 0x4B4000 << 8
//    | n: bits 4 .. 21 are zero.  So m0 + 16 m1 holds the byte of two nibbles in its low 8
//    bits with zeros above up to bit 21, b0 + 256 b1 holds two such bytes in its low 16 bits,
//    and one byte permute joins two of those into the word (shift-adds, no masks).
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
    __half s16 = __float2half_rn(amax * kInv7);
    if ((__half_as_ushort(s16) & 0x7fffu) == 0) s16 = __ushort_as_half(0x3c00u);
    const float s = __half2float(s16);
    scale_out = s16;
    float rs;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rs) : "f"(s));
    constexpr float kMagic8 = 12582920.0f;  // 1.5 * 2^23 + 8
    constexpr float kBand = 0.4999847412109375f;  // 1/2 - 2^-16
    uint32_t m[16];
    float emax = 0.f;  // the largest |e|, NaN if any e is NaN
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float mi = fmaf(x[i], rs, kMagic8);
        const float e = fmaf(x[i], rs, kMagic8 - mi);  // kMagic8 - mi = -r exactly
        emax = max_abs_nan(emax, e);
        m[i] = __float_as_uint(mi);
    }
    const bool slow = amax * rs > 7.49f || !(emax <= kBand);
    uint32_t h[4];  // h[k]: the nibbles of values 4k .. 4k + 3 in its low 16 bits
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t b0 = m[4 * k] + 16u * m[4 * k + 1];
        const uint32_t b1 = m[4 * k + 2] + 16u * m[4 * k + 3];
        h[k] = b0 + 256u * b1;
    }
    uint32_t lo = prmt(h[0], h[1], 0x5410u);
    uint32_t hi = prmt(h[2], h[3], 0x5410u);
    if (slow) {
        bool plain = isinf(s);
#pragma unroll
        for (int i = 0; i < 16; ++i) plain |= x[i] != x[i];
        lo = quant8(*reinterpret_cast<const float(*)[8]>(&x[0]), s, plain);
        hi = quant8(*reinterpret_cast<const float(*)[8]>(&x[8]), s, plain);
    }
    return make_uint2(lo, hi);
}

// Destination of one row (a (token, kv head) pair): the address of its (page, kv head)
// block and its slot in the page, or block 0 when the row is skipped (its position or
// page is out of range, which raises a flag).  Token tok belongs to sequence b: with
// cu_rows the last b whose first token cu_rows[b] is <= tok, else tok / n_new.
__device__ __forceinline__ unsigned long long row_dest(const QuantizeArgs& a, uint32_t row, int& slot) {
    const uint32_t tok = fast_div(row, a.div_h);
    const int h = static_cast<int>(row - tok * static_cast<uint32_t>(a.Hkv));
    int b;
    long long t;
    if (a.cu_rows != nullptr) {
        int lo = 0, hi = a.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(a.cu_rows + mid) <= static_cast<int>(tok)) lo = mid;
            else hi = mid - 1;
        }
        b = lo;
        t = static_cast<long long>(tok) - __ldg(a.cu_rows + b);
    } else {
        b = static_cast<int>(fast_div(tok, a.div_n));
        t = static_cast<long long>(tok) - static_cast<long long>(b) * a.n_new;
    }
    const long long pos = static_cast<long long>(__ldg(a.start_pos + b)) + t;
    const long long pidx = pos >> a.lg_p;
    if (pos < 0 || pidx >= a.max_blocks) {
        raise_flag(a.status, KVQ_FLAG_BAD_POSITION);
        return 0ull;
    }
    const int page = __ldg(a.block_table + static_cast<long long>(b) * a.max_blocks + pidx);
    if (page < 0 || page >= a.num_pages) {
        raise_flag(a.status, KVQ_FLAG_BAD_PAGE);
        return 0ull;
    }
    slot = static_cast<int>(pos & ((1 << a.lg_p) - 1));
    return reinterpret_cast<unsigned long long>(a.pool + (static_cast<long long>(page) * a.Hkv + h) * a.L.bytes);
}

// Work mapping.  Rows go to warps in blocks of 32; a job is the K or the V row of one row
// (K and V of a row adjacent), held by a team of LPR = D / 16 lanes, 16 values a lane.
// Lane l of the warp first works out where row l of the block goes (one block-table
// lookup per row, shared by its K and V jobs and by the lanes of their teams through
// shuffles), then the warp quantizes the block's 64 jobs TEAMS * U at a time.  A pass's
// fp16 rows are loaded (all U x 32 bytes per lane) before it computes, and with PF the
// next pass's rows are loaded before this pass computes, so enough loads are in flight to
// stream from HBM.  The block loop is grid-strided over one wave of resident CTAs.
template <int D, int U, bool PF, int MINB>
__global__ void __launch_bounds__(256, MINB) quantize_append_kernel(QuantizeArgs a) {
    // A decode launched behind this kernel may start its own set-up now; it waits for this
    // grid to finish before it reads the pool.  This kernel itself may start before the
    // kernel ahead of it (a decode that reads the pool) has finished: it waits for it
    // before anything else.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    constexpr int LPR = D / 16;           // lanes per job
    constexpr int TEAMS = 32 / LPR;       // jobs per warp at a time
    constexpr int JPP = TEAMS * U;        // jobs per pass
    constexpr int PASSES = 64 / JPP;      // passes over a block's 64 jobs
    const int lane = threadIdx.x & 31;
    const int team = lane / LPR;
    const int tl = lane % LPR;            // lane within the team
    const uint32_t blocks = (a.rows + 31u) / 32u;
    const uint32_t warp_global = (blockIdx.x * blockDim.x + threadIdx.x) / 32;
    const uint32_t warps_total = gridDim.x * blockDim.x / 32;
    // the fp16 rows of pass ps of the block at row0
    auto load = [&](uint32_t row0, int ps, uint4 (&raw)[U][2]) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int jl = ps * JPP + u * TEAMS + team;  // job within the block
            const uint32_t row = row0 + static_cast<uint32_t>(jl >> 1);
            raw[u][0] = raw[u][1] = make_uint4(0, 0, 0, 0);
            if (row < a.rows) {
                const __half* src = ((jl & 1) ? a.v : a.k) + static_cast<size_t>(row) * D + tl * 16;
                raw[u][0] = __ldcs(reinterpret_cast<const uint4*>(src));  // read once: stream past the caches
                raw[u][1] = __ldcs(reinterpret_cast<const uint4*>(src) + 1);
            }
        }
    };
    for (uint32_t blk = warp_global; blk < blocks; blk += warps_total) {
        const uint32_t row0 = blk * 32u;
        int my_slot = 0;
        const unsigned long long my_dst = row0 + lane < a.rows ? row_dest(a, row0 + lane, my_slot) : 0ull;
        uint4 raw[U][2];
        if (PF) load(row0, 0, raw);
#pragma unroll 1
        for (int ps = 0; ps < PASSES; ++ps) {
            uint4 nxt[U][2];
            if (PF) {
                if (ps + 1 < PASSES) load(row0, ps + 1, nxt);
            } else {
                load(row0, ps, raw);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int jl = ps * JPP + u * TEAMS + team;
                const int is_v = jl & 1;
                const int lg = (is_v ? a.lg_lanes_v : a.lg_lanes_k) - 1;  // log2 of the 16-value lanes per group
                __half s16;
                const uint2 words = quant_lane16<LPR>(raw[u], lg, s16);
                const unsigned long long dst = __shfl_sync(0xffffffffu, my_dst, jl >> 1);
                const int slot = __shfl_sync(0xffffffffu, my_slot, jl >> 1);
                if (dst == 0ull) continue;  // past the end, or skipped and flagged
                uint8_t* blkp = reinterpret_cast<uint8_t*>(dst);
                uint8_t* codes = blkp + (is_v ? a.L.v_codes : 0) + slot * (D / 2);
                reinterpret_cast<uint2*>(codes)[tl] = words;
                if ((tl & ((1 << lg) - 1)) == 0) {
                    const int ngroups = D >> (lg + 4);
                    uint8_t* scales = blkp + (is_v ? a.L.v_scales : a.L.k_scales) + slot * ngroups * 2;
                    reinterpret_cast<__half*>(scales)[tl >> lg] = s16;
                }
            }
            if (PF) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    raw[u][0] = nxt[u][0];
                    raw[u][1] = nxt[u][1];
                }
            }
        }
    }
}

// The instance launched: jobs per lane per pass, next-pass prefetch, resident CTAs per SM
// the register budget is set for.
constexpr int kQuantU = 2;
constexpr bool kQuantPrefetch = true;
constexpr int kQuantMinBlocks = 3;

// Resident 256-thread CTAs per SM of an instance, looked up once.
template <int D>
int quantize_ctas_per_sm() {
    static std::atomic<int> memo{0};
    int n = memo.load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, quantize_append_kernel<D, kQuantU, kQuantPrefetch, kQuantMinBlocks>, 256, 0) != cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        n = 1;
    }
    memo.store(n, std::memory_order_relaxed);
    return n;
}

template <int D>
cudaError_t launch_q(const QuantizeArgs& a, cudaStream_t stream) {
    const long long blocks32 = (static_cast<long long>(a.rows) + 31) / 32;
    if (blocks32 == 0) return cudaSuccess;
    constexpr int threads = 256;
    long long blocks = (blocks32 + threads / 32 - 1) / (threads / 32);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = static_cast<long long>(sms > 0 ? sms : 1) * quantize_ctas_per_sm<D>();
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
    const cudaError_t err =
        cudaLaunchKernelEx(&cfg, quantize_append_kernel<D, kQuantU, kQuantPrefetch, kQuantMinBlocks>, a);
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
