// decode_gk64.cu -- decode attention kernel instances for K groups of 64.
#include "decode_impl.cuh"

KVQ_DECODE_TU(64, false, decode_run_gk64, decode_occupancy_gk64)
