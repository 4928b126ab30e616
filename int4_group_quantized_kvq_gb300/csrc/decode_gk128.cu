// decode_gk128.cu -- decode attention kernel instances for K groups of 128.
#include "decode_impl.cuh"

KVQ_DECODE_TU(128)
