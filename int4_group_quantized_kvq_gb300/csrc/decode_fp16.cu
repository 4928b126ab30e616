// decode_fp16.cu -- launch of the FP16-cache decode kernel (decode_fp16.cuh) and its
// occupancy query, dispatched on the query heads per kv head.
#include <atomic>

#include "decode_fp16.cuh"

namespace kvq {
namespace decode {
namespace {

template <int R, bool WIN, int CODEC>
cudaError_t fp16_smem_attr(size_t smem) {
    static std::atomic<long long> granted{-1};
    if (static_cast<long long>(smem) <= granted.load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t err = cudaFuncSetAttribute(decode_fp16_kernel<128, R, WIN, CODEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
    if (err != cudaSuccess) {
        cudaGetLastError();
        return err;
    }
    long long cur = granted.load();
    while (static_cast<long long>(smem) > cur && !granted.compare_exchange_weak(cur, static_cast<long long>(smem))) {
    }
    return cudaSuccess;
}

template <int R, bool WIN, int CODEC>
int fp16_occupancy(size_t smem) {
    if (fp16_smem_attr<R, WIN, CODEC>(smem) != cudaSuccess) return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_fp16_kernel<128, R, WIN, CODEC>, 128, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

template <int R, bool WIN, int CODEC>
cudaError_t fp16_run(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    FParams fp{};
    KParams& p = fp.p;
    p.pool = a.pool;
    p.q = a.q;
    p.block_table = a.block_table;
    p.seq_lens = a.seq_lens;
    p.ws_ml = reinterpret_cast<float*>(a.workspace + plan.ws_ml_offset);
    p.ws_o = reinterpret_cast<float*>(a.workspace + plan.ws_o_offset);
    p.ws_pre = reinterpret_cast<int32_t*>(a.workspace + plan.ws_pre_offset);
    p.status = a.status ? a.status : reinterpret_cast<uint32_t*>(a.workspace);
    p.len_sub = a.len_sub;
    p.window = a.window;
    p.sinks = a.sinks;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.Hg = a.Hkv;
    p.r = a.Hq / a.Hkv;
    p.ns = p.r;
    p.P = a.L.P;
    p.num_pages = a.num_pages;
    p.max_blocks = a.max_blocks;
    p.block_bytes = CODEC == 2 ? a.L.P * (a.L.d + 8) : 4 * a.L.P * a.L.d;
    if (CODEC == 2) {
        const Wht4Codebook& cb = wht4_codebook();
        for (int j = 0; j < 16; ++j) fp.lut[j] = cb.levels[j];
    }
    p.unit_bytes = p.block_bytes;
    p.stages = plan.stages;
    p.scale_log2 = a.softmax_scale * 1.4426950408889634f;
    p.lg_p = 0;
    while ((1 << p.lg_p) < a.L.P) ++p.lg_p;
    cudaError_t err = fp16_smem_attr<R, WIN, CODEC>(plan.smem_bytes);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.ctas));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = plan.smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, decode_fp16_kernel<128, R, WIN, CODEC>, fp);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace
}  // namespace decode

// query heads per kv head r in 1..8, rounded up to 1, 2, 4 or 8; window instances when a
// window is given; rotated 4-bit blocks for that cache
template <bool WIN, int CODEC>
cudaError_t run_r(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s) {
    const int r = a.Hq / a.Hkv;
    if (r <= 1) return decode::fp16_run<1, WIN, CODEC>(a, plan, s);
    if (r <= 2) return decode::fp16_run<2, WIN, CODEC>(a, plan, s);
    if (r <= 4) return decode::fp16_run<4, WIN, CODEC>(a, plan, s);
    if (r <= 8) return decode::fp16_run<8, WIN, CODEC>(a, plan, s);
    return cudaErrorInvalidValue;
}
template <bool WIN, int CODEC>
int occ_r(const DecodeArgs& a, size_t smem) {
    const int r = a.Hq / a.Hkv;
    if (r <= 1) return decode::fp16_occupancy<1, WIN, CODEC>(smem);
    if (r <= 2) return decode::fp16_occupancy<2, WIN, CODEC>(smem);
    if (r <= 4) return decode::fp16_occupancy<4, WIN, CODEC>(smem);
    if (r <= 8) return decode::fp16_occupancy<8, WIN, CODEC>(smem);
    return 0;
}

cudaError_t decode_run_fp16(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s) {
    if (a.wht) return a.window > 0 ? run_r<true, 2>(a, plan, s) : run_r<false, 2>(a, plan, s);
    return a.window > 0 ? run_r<true, 0>(a, plan, s) : run_r<false, 0>(a, plan, s);
}

int decode_occupancy_fp16(const DecodeArgs& a, const DecodePlan& plan, size_t smem) {
    (void)plan;
    if (a.wht) return a.window > 0 ? occ_r<true, 2>(a, smem) : occ_r<false, 2>(a, smem);
    return a.window > 0 ? occ_r<true, 0>(a, smem) : occ_r<false, 0>(a, smem);
}

}  // namespace kvq
