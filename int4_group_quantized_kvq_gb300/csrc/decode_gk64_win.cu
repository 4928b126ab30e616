// decode_gk64_win.cu -- decode attention kernel instances for K groups of 64, sliding window
// with sink tokens.
#include "decode_impl.cuh"

#define KVQ_GK64_WIN_CASES(CALL)                        \
    KVQ_DECODE_CASES(128, 64, 32, true, CALL)  \
    KVQ_DECODE_CASES(128, 64, 64, true, CALL)  \
    KVQ_DECODE_CASES(128, 64, 128, true, CALL)
KVQ_DECODE_TU(KVQ_GK64_WIN_CASES, decode_run_gk64_win, decode_occupancy_gk64_win)
