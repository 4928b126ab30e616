// decode_gk32_win.cu -- decode attention kernel instances for K groups of 32, sliding window
// with sink tokens.
#include "decode_impl.cuh"

#define KVQ_GK32_WIN_CASES(CALL)                        \
    KVQ_DECODE_CASES(128, 32, 32, true, CALL)  \
    KVQ_DECODE_CASES(128, 32, 64, true, CALL)  \
    KVQ_DECODE_CASES(128, 32, 128, true, CALL)
KVQ_DECODE_TU(KVQ_GK32_WIN_CASES, decode_run_gk32_win, decode_occupancy_gk32_win)
