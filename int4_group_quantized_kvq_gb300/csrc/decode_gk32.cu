// decode_gk32.cu -- decode attention kernel instances for K groups of 32.
#include "decode_impl.cuh"

#define KVQ_GK32_CASES(CALL)                        \
    KVQ_DECODE_CASES(128, 32, 32, false, CALL)  \
    KVQ_DECODE_CASES(128, 32, 64, false, CALL)  \
    KVQ_DECODE_CASES(128, 32, 128, false, CALL)
KVQ_DECODE_TU(KVQ_GK32_CASES, decode_run_gk32, decode_occupancy_gk32)
