// decode_gk32.cu -- decode attention kernel instances for K groups of 32.
#include "decode_impl.cuh"

KVQ_DECODE_TU(32, false, decode_run_gk32, decode_occupancy_gk32)
