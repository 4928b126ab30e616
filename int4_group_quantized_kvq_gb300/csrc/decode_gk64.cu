// decode_gk64.cu -- decode attention kernel instances for K groups of 64.
#include "decode_impl.cuh"

#define KVQ_GK64_CASES(CALL)                        \
    KVQ_DECODE_CASES(128, 64, 32, false, CALL)  \
    KVQ_DECODE_CASES(128, 64, 64, false, CALL)  \
    KVQ_DECODE_CASES(128, 64, 128, false, CALL)
KVQ_DECODE_TU(KVQ_GK64_CASES, decode_run_gk64, decode_occupancy_gk64)
