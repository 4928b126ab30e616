// decode_combine.cu -- launch of the split-KV combine kernel, which writes the decode
// output from the warp partials the decode grid(s) leave in the workspace.
#include <algorithm>

#include "decode_impl.cuh"

namespace kvq {
namespace {

// The partials one decode grid (arguments a, plan) leaves in its workspace.
decode::CSource source_of(const DecodeArgs& a, const DecodePlan& plan) {
    decode::CSource s;
    s.ws_ml = reinterpret_cast<const float*>(a.workspace + plan.ws_ml_offset);
    s.ws_o = reinterpret_cast<const float*>(a.workspace + plan.ws_o_offset);
    s.ws_pre = reinterpret_cast<const int32_t*>(a.workspace + plan.ws_pre_offset);
    s.Hg = a.Hkv / plan.hk;
    s.ns = plan.hk * (a.Hq / a.Hkv);
    s.C = plan.ctas;
    s.W = 4;
    s.max_blocks = a.max_blocks;
    s.window = a.window;
    s.sinks = a.sinks;
    s.len_sub = a.len_sub;
    return s;
}

cudaError_t launch(const decode::CParams& p, int warps, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.B) * p.Hq;
    if (rows <= 0) return cudaSuccess;
    if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
    // Launched while the decode grid runs (programmatic dependent launch); the kernel
    // waits with griddepcontrol.wait before it reads the workspace.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows));
    cfg.blockDim = dim3(static_cast<unsigned>(warps) * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t err = cudaLaunchKernelEx(&cfg, decode::combine_kernel<128>, p);
    if (err != cudaSuccess) return err;
    return cudaGetLastError();
}

int lg2(int P) {
    int l = 0;
    while ((1 << l) < P) ++l;
    return l;
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    decode::CParams p{};
    p.src[0] = source_of(a, plan);
    p.nsrc = 1;
    p.seq_lens = a.seq_lens;
    p.out = a.out;
    p.B = a.B;
    p.Hq = a.Hq;
    p.lg_p = lg2(a.L.P);
    return launch(p, plan.combine_warps, stream);
}

// The mixed-precision decode: the partials of the INT4 grid (a0, plan0) and of the FP16
// grid (a1, plan1) merged per row.
cudaError_t launch_combine2(const DecodeArgs& a0, const DecodePlan& plan0, const DecodeArgs& a1,
                            const DecodePlan& plan1, cudaStream_t stream) {
    decode::CParams p{};
    p.src[0] = source_of(a0, plan0);
    p.src[1] = source_of(a1, plan1);
    p.nsrc = 2;
    p.seq_lens = a0.seq_lens;
    p.out = a0.out;
    p.B = a0.B;
    p.Hq = a0.Hq;
    p.lg_p = lg2(a0.L.P);
    const int warps = std::max(plan0.combine_warps, plan1.combine_warps);
    return launch(p, warps, stream);
}

}  // namespace kvq
