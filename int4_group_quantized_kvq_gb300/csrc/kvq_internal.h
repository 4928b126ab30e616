// kvq_internal.h -- launchers shared between the kernel files and the C ABI layer.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq.h"

namespace kvq {

// Byte offsets of the four sections of a (page, kv-head) block.
struct BlockLayout {
    int32_t d, P, Gk, Gv;
    int32_t v_codes;   // P * d / 2
    int32_t k_scales;  // P * d
    int32_t v_scales;  // P * d + P * (d / Gk) * 2
    int32_t bytes;     // padded to 16
};

inline BlockLayout block_layout(const kvq_cache_config& c) {
    BlockLayout L;
    L.d = c.head_dim;
    L.P = c.page_size;
    L.Gk = c.group_k;
    L.Gv = c.group_v;
    L.v_codes = c.page_size * c.head_dim / 2;
    L.k_scales = c.page_size * c.head_dim;
    L.v_scales = L.k_scales + c.page_size * (c.head_dim / c.group_k) * 2;
    const int32_t raw = L.v_scales + c.page_size * (c.head_dim / c.group_v) * 2;
    L.bytes = (raw + 15) / 16 * 16;
    return L;
}

// Division of 32-bit n < 2^31 by a fixed divisor d >= 1 as a multiply-high, add and
// shift: with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1,
// n / d = (umulhi(n, m) + n) >> l, and the sum stays below 2^32 because n < 2^31.
struct FastDiv {
    uint32_t d, m, l;
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while ((1ull << f.l) < d) ++f.l;
    f.m = static_cast<uint32_t>(((1ull << 32) * ((1ull << f.l) - d)) / d + 1);
    return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
    return (__umulhi(n, f.m) + n) >> f.l;
}
#endif

struct QuantizeArgs {
    uint8_t* pool;
    const __half* k;
    const __half* v;
    const int32_t* block_table;
    const int32_t* start_pos;
    // ragged batches: sequence b owns tokens cu_rows[b] .. cu_rows[b + 1] - 1 of the row
    // arrays (nullptr: every sequence owns n_new tokens, sequence b from b * n_new)
    const int32_t* cu_rows;
    uint32_t* status;
    int32_t max_blocks, B, n_new, Hkv, num_pages;
    uint32_t rows;          // tokens * Hkv (< 2^30)
    FastDiv div_h, div_n;   // by Hkv, by n_new (unused with cu_rows)
    int32_t lg_p;           // log2 page_size
    int32_t lg_lanes_k, lg_lanes_v;  // log2 of group_k / 8 and group_v / 8 (lanes of 8 values per group)
    BlockLayout L;
};
cudaError_t launch_quantize_append(const QuantizeArgs& a, cudaStream_t stream);

struct DequantArgs {
    const uint8_t* pool;
    const int32_t* block_table;
    void* out_k;
    void* out_v;
    uint32_t* status;
    int32_t max_blocks, b, start, n, Hkv, num_pages, out_fp32;
    BlockLayout L;
};
cudaError_t launch_dequantize(const DequantArgs& a, cudaStream_t stream);

// Copy n16 16-byte words from src (device address of mapped pinned host memory) to dst on
// the device, as a kernel launched with programmatic dependent launch: it reads src while
// the kernel ahead of it on the stream finishes and writes dst only after that kernel has.
cudaError_t launch_stage_in(const void* src, void* dst, size_t n16, cudaStream_t stream);

// Decode attention: the persistent split-KV kernel with the split combine fused in.
struct DecodePlan {
    int32_t hk;           // kv heads per unit of work (4 when Hq == Hkv, Hkv % 4 == 0, P == 16; else 1)
    int32_t hs;           // query-head slots per score thread: 1 (up to 4 per unit) or 2 (up to 8)
    int32_t ctas;         // CTAs of the persistent grid (4 warps each)
    int32_t stages;       // bulk-copy ring depth per warp, in units
    size_t smem_bytes;    // dynamic shared memory per CTA
    int32_t combine_warps; // warps per CTA of the combine kernel (one CTA per output row)
    size_t ws_pre_offset; // pages prefix per sequence, published by the decode grid
    size_t ws_ml_offset;  // (max, sum) of the warp partials
    size_t ws_o_offset;   // unnormalised outputs of the warp partials
    size_t ws_bytes;      // total workspace bytes
};

struct DecodeArgs {
    const uint8_t* pool;
    const __half* q;
    const int32_t* block_table;
    const int32_t* seq_lens;
    float* out;
    uint8_t* workspace;
    int32_t max_blocks, B, Hq, Hkv, num_pages, max_len;
    float softmax_scale;
    BlockLayout L;
    // the decode step's fused append of one token per sequence (k_new == nullptr: none)
    const __half* k_new = nullptr;
    const __half* v_new = nullptr;
    const int32_t* append_pos = nullptr;
    uint8_t* pool_w = nullptr;
    // sliding window with sink tokens: the last `window` positions (0: all) and the first `sinks`
    int32_t window = 0;
    int32_t sinks = 0;
    // attention over the FP16 cache instead of the INT4 one (the comparison's baseline), or
    // (with int8 or wht also set) over the INT8 per-row cache or the rotated 4-bit cache;
    // all three take the CUDA-core kernel
    bool fp16 = false;
    bool int8 = false;
    bool wht = false;
    // attend seq_lens[b] - len_sub positions (the INT4 part of the mixed-precision decode)
    int32_t len_sub = 0;
    // status word (nullptr: the first word of the workspace)
    uint32_t* status = nullptr;
    // device address of mapped pinned host memory the combine also writes the output to
    // (the host-buffer decode step), or nullptr
    float* out_host = nullptr;
    // q (and the new rows) are written by the kernel just ahead on the stream, which lets
    // this grid start early: the grid reads q only after griddepcontrol.wait
    bool q_after_wait = false;
    // bound of the INT4 kernel's waits on copies in ns (0: the default, 250 ms), and the test
    // of that bound (each warp's first page copy announced 16 bytes larger than it is)
    uint64_t wait_ns = 0;
    bool withhold_first_copy = false;
};

// The FP16 cache of the latency comparison: block (page, kv head) holds K rows P x d fp16,
// then V rows P x d fp16.
struct Fp16AppendArgs {
    uint8_t* pool16;
    const __half* k;
    const __half* v;
    const int32_t* block_table;
    const int32_t* start_pos;
    uint32_t* status;
    int32_t max_blocks, B, n_new, Hkv, d, P, num_pages;
};
struct Fp16DequantArgs {
    const uint8_t* pool;
    uint8_t* pool16;
    const int32_t* block_table;
    const int32_t* seq_lens;
    uint32_t* status;
    int32_t max_blocks, B, Hkv, num_pages;
    BlockLayout L;
};
cudaError_t launch_fp16_append(const Fp16AppendArgs& a, cudaStream_t stream);
// INT8 per-row cache: quantize-append, arguments as for the FP16 append
cudaError_t launch_int8_quantize_append(const Fp16AppendArgs& a, cudaStream_t stream);
cudaError_t launch_dequantize_to_fp16(const Fp16DequantArgs& a, long long max_pages, cudaStream_t stream);

// The rotated 4-bit codec (wht_codec.cu): its fp32 codebook (the 16 Lloyd-Max levels of
// the standard normal, ascending, and the 15 midpoints between them), computed once;
// quantize-append with the FP16 append's arguments (pool16 the codec's pool, d = 128);
// dequantization of positions [start, start + n) of sequence b to fp32 [n, Hkv, 128].
struct Wht4Codebook {
    float levels[16];
    float thresholds[15];
};
const Wht4Codebook& wht4_codebook();
cudaError_t launch_wht4_quantize_append(const Fp16AppendArgs& a, cudaStream_t stream);
cudaError_t launch_wht4_dequantize(const uint8_t* pool, const int32_t* block_table, int32_t max_blocks, int32_t b,
                                   int32_t start, int32_t n, float* out_k, float* out_v, uint32_t* status,
                                   int32_t Hkv, int32_t P, int32_t num_pages, cudaStream_t stream);

// Returns cudaErrorInvalidValue for a geometry no kernel instance covers.
cudaError_t plan_decode(const DecodeArgs& a, DecodePlan* plan);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);
// the decode grid alone (its partials stay in the workspace), and the combine of two grids'
// partials (the mixed-precision decode)
cudaError_t launch_decode_grid(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream);
cudaError_t launch_combine2(const DecodeArgs& a0, const DecodePlan& plan0, const DecodeArgs& a1,
                            const DecodePlan& plan1, cudaStream_t stream);

}  // namespace kvq
