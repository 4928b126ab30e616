// decode_d256_win.cu -- decode attention kernel instances for head_dim 256 (one-head units,
// up to 4 query heads per kv head; K groups of 64 or 128, V groups of 32, 64 or 128), sliding
// window with sink tokens.
#include "decode_impl.cuh"

#define KVQ_D256_WIN_CASES(CALL) \
    KVQ_DECODE_CASES_1H(256, 64, 32, true, CALL) \
    KVQ_DECODE_CASES_1H(256, 64, 64, true, CALL) \
    KVQ_DECODE_CASES_1H(256, 64, 128, true, CALL) \
    KVQ_DECODE_CASES_1H(256, 128, 32, true, CALL) \
    KVQ_DECODE_CASES_1H(256, 128, 64, true, CALL) \
    KVQ_DECODE_CASES_1H(256, 128, 128, true, CALL)
KVQ_DECODE_TU(KVQ_D256_WIN_CASES, decode_run_d256_win, decode_occupancy_d256_win)
