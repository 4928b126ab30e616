// decode_gk128_win.cu -- decode attention kernel instances for K groups of 128, sliding window
// with sink tokens.
#include "decode_impl.cuh"

#define KVQ_GK128_WIN_CASES(CALL)                        \
    KVQ_DECODE_CASES(128, 128, 32, true, CALL)  \
    KVQ_DECODE_CASES(128, 128, 64, true, CALL)  \
    KVQ_DECODE_CASES(128, 128, 128, true, CALL)
KVQ_DECODE_TU(KVQ_GK128_WIN_CASES, decode_run_gk128_win, decode_occupancy_gk128_win)
