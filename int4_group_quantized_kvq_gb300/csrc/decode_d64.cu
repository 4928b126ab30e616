// decode_d64.cu -- decode attention kernel instances for head_dim 64: K and V
// groups of 32 or 64.
#include "decode_impl.cuh"

#define KVQ_D64_CASES(CALL)                       \
    KVQ_DECODE_CASES(64, 32, 32, false, CALL)  \
    KVQ_DECODE_CASES(64, 32, 64, false, CALL)  \
    KVQ_DECODE_CASES(64, 64, 32, false, CALL)  \
    KVQ_DECODE_CASES(64, 64, 64, false, CALL)
KVQ_DECODE_TU(KVQ_D64_CASES, decode_run_d64, decode_occupancy_d64)
