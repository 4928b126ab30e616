// decode_gk64.cu -- decode attention kernel instances for K groups of 64.
#include "decode_impl.cuh"

KVQ_DECODE_TU(64)
