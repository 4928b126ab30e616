// decode_gk128.cu -- decode attention kernel instances for K groups of 128.
#include "decode_impl.cuh"

KVQ_DECODE_TU(128, false, decode_run_gk128, decode_occupancy_gk128)
