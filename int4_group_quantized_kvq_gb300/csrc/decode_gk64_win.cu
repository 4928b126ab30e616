// decode_gk64_win.cu -- decode attention kernel instances for K groups of 64, sliding window
// with sink tokens.
#include "decode_impl.cuh"

KVQ_DECODE_TU(64, true, decode_run_gk64_win, decode_occupancy_gk64_win)
