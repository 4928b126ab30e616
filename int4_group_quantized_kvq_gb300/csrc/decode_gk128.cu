// decode_gk128.cu -- decode attention kernel instances for K groups of 128.
#include "decode_impl.cuh"

#define KVQ_GK128_CASES(CALL)                        \
    KVQ_DECODE_CASES(128, 128, 32, false, CALL)  \
    KVQ_DECODE_CASES(128, 128, 64, false, CALL)  \
    KVQ_DECODE_CASES(128, 128, 128, false, CALL)
KVQ_DECODE_TU(KVQ_GK128_CASES, decode_run_gk128, decode_occupancy_gk128)
