// decode_int8.cu -- decode attention kernel instances for the INT8 per-row cache: the split-KV
// tensor-core kernel of decode_impl.cuh with 8-bit codes and one fp32 scale per row (one-head
// units; one or two query-head slots per thread; 16-token pages or larger ones; the INT8
// calls attend to every position).
#include "decode_impl.cuh"

namespace kvq {

#define KVQ_INT8_CASES(CALL)                                                                     \
    case 0: return CALL(1, false, false);                                                        \
    case 1: return CALL(1, false, true);                                                         \
    case 2: return CALL(2, false, false);                                                        \
    case 3: return CALL(2, false, true);
#define KVQ_INT8_KEY ((plan.hk != 1 || plan.hs < 1 || plan.hs > 2 || a.L.d != 128 || a.window > 0) ? -1 \
                      : (plan.hs - 1) * 2 + (a.L.P == 16 ? 1 : 0))
#define KVQ_INT8_RUN(HS_, W_, P16_) decode::run<128, 128, 128, 1, HS_, W_, P16_, 1>(a, plan, s)
#define KVQ_INT8_OCC(HS_, W_, P16_) decode::occupancy<128, 128, 128, 1, HS_, W_, P16_, 1>(smem)

cudaError_t decode_run_int8(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s) {
    switch (KVQ_INT8_KEY) {
        KVQ_INT8_CASES(KVQ_INT8_RUN)
        default: return cudaErrorInvalidValue;
    }
}

int decode_occupancy_int8(const DecodeArgs& a, const DecodePlan& plan, size_t smem) {
    switch (KVQ_INT8_KEY) {
        KVQ_INT8_CASES(KVQ_INT8_OCC)
        default: return 0;
    }
}

}  // namespace kvq
