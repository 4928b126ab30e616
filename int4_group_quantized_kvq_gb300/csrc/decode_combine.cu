// decode_combine.cu -- launch of the split-KV combine kernel, which writes the decode
// output from the warp partials the decode grid leaves in the workspace.
#include "decode_impl.cuh"

namespace kvq {

cudaError_t launch_combine(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    decode::CParams p;
    p.ws_ml = reinterpret_cast<const float*>(a.workspace + plan.ws_ml_offset);
    p.ws_o = reinterpret_cast<const float*>(a.workspace + plan.ws_o_offset);
    p.ws_pre = reinterpret_cast<const int32_t*>(a.workspace + plan.ws_pre_offset);
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.P = a.L.P;
    p.lg_p = 0;
    while ((1 << p.lg_p) < a.L.P) ++p.lg_p;
    p.max_blocks = a.max_blocks;
    p.window = a.window;
    p.sinks = a.sinks;
    p.B = a.B;
    p.Hq = a.Hq;
    p.Hg = a.Hkv / plan.hk;
    p.ns = plan.hk * (a.Hq / a.Hkv);
    p.C = plan.ctas;
    p.W = 4;
    const long long rows = static_cast<long long>(a.B) * a.Hq;
    if (rows <= 0) return cudaSuccess;
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    // Launched while the decode grid runs (programmatic dependent launch); the kernel
    // waits with griddepcontrol.wait before it reads the workspace.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(static_cast<unsigned>(plan.combine_warps) * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, decode::combine_kernel<128>, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

}  // namespace kvq
