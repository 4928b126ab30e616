// decode_d64_win.cu -- decode attention kernel instances for head_dim 64 (K and V groups of
// 32 or 64), sliding window with sink tokens.
#include "decode_impl.cuh"

#define KVQ_D64_WIN_CASES(CALL)                       \
    KVQ_DECODE_CASES(64, 32, 32, true, CALL)  \
    KVQ_DECODE_CASES(64, 32, 64, true, CALL)  \
    KVQ_DECODE_CASES(64, 64, 32, true, CALL)  \
    KVQ_DECODE_CASES(64, 64, 64, true, CALL)
KVQ_DECODE_TU(KVQ_D64_WIN_CASES, decode_run_d64_win, decode_occupancy_d64_win)
