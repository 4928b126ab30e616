// decode_gk32_win.cu -- decode attention kernel instances for K groups of 32, sliding window
// with sink tokens.
#include "decode_impl.cuh"

KVQ_DECODE_TU(32, true, decode_run_gk32_win, decode_occupancy_gk32_win)
