// host_stage.cu -- moving a decode step's inputs in from pinned host memory inside the
// stream's chain of kernels (the host-buffer decode step, "4-bit KV cache compression"
// section 1.1: the new token's q, K and V arrive, the step runs, the output leaves).
#include <cuda_runtime.h>

#include <cstdint>

#include "kvq_internal.h"

namespace kvq {
namespace {

// Thread i copies word i, and then words i + stride, ...: the first word of each thread is
// read before griddepcontrol.wait, so the read from host memory overlaps the end of the
// kernel ahead on the stream; nothing is written before that kernel has finished (it may
// still read dst, the previous step's inputs).
__global__ void __launch_bounds__(256) stage_in_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                       unsigned long long n) {
    asm volatile("griddepcontrol.launch_dependents;");
    const unsigned long long stride = static_cast<unsigned long long>(gridDim.x) * blockDim.x;
    const unsigned long long i0 = static_cast<unsigned long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint4 first = make_uint4(0, 0, 0, 0);
    if (i0 < n) first = src[i0];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (i0 < n) dst[i0] = first;
    for (unsigned long long i = i0 + stride; i < n; i += stride) dst[i] = src[i];
}

}  // namespace

cudaError_t launch_stage_in(const void* src, void* dst, size_t n16, cudaStream_t stream) {
    if (n16 == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    unsigned long long blocks = (n16 + 255) / 256;
    const unsigned long long cap = static_cast<unsigned long long>(sms > 0 ? sms : 1) * 4;
    if (blocks > cap) blocks = cap;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, stage_in_kernel, static_cast<const uint4*>(src),
                                               static_cast<uint4*>(dst), static_cast<unsigned long long>(n16));
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace kvq
