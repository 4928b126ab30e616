// decode_gk128_win.cu -- decode attention kernel instances for K groups of 128, sliding window
// with sink tokens.
#include "decode_impl.cuh"

KVQ_DECODE_TU(128, true, decode_run_gk128_win, decode_occupancy_gk128_win)
