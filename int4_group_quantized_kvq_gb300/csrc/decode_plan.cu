// decode_plan.cu -- sizing of the persistent split-KV grid and of its workspace.
//
// The grid is W warps (4 per CTA).  W is the number of warps the device can keep
// resident (SMs x resident CTAs x 4), reduced for small problems so that a warp gets
// at least two pages; every warp receives an equal contiguous slice of the flattened
// (sequence, kv head, page) units.  Each warp writes at most one partial per
// (sequence, kv head) segment its slice touches.  Partial index = warp + segment is
// unique: if warp w touches segment s and warp w-1 touches segment s+1, warp w-1 would
// hold a later unit than warp w, which contiguous ordered slices rule out.  So the
// workspace holds W + B * Hkv partials, each r (query heads per KV head) x (2 + d) floats,
// plus one split counter per (sequence, KV head) and, for segments spread over more than
// 32 warps, a second level: one counter and one partial per group of 32 warps (indexed
// by the group's first partial, so the same W + B * Hkv slots suffice).  The counters
// must be zero when a call starts; each is reset by the warp that consumes it, so they
// stay zero from one call to the next while the workspace serves the same shape.
#include <algorithm>

#include "kvq_internal.h"

namespace kvq {

cudaError_t decode_run_gk32(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk64(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk128(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_gk32(const DecodeArgs& a, size_t smem);
int decode_occupancy_gk64(const DecodeArgs& a, size_t smem);
int decode_occupancy_gk128(const DecodeArgs& a, size_t smem);

namespace {
constexpr int kWarpsPerCta = 4;
constexpr int kMaxStages = 8;  // deepest page ring per warp
constexpr size_t kWarpCtxBytes = 64;  // per-warp shared context of the decode kernel
constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

cudaError_t plan_decode(const DecodeArgs& a, DecodePlan* plan) {
    if (a.L.d != 128) return cudaErrorInvalidValue;
    if (a.L.P % 16 != 0) return cudaErrorInvalidValue;
    const int r = a.Hq / a.Hkv;
    if (r < 1 || r > 8) return cudaErrorInvalidValue;
    // Resident CTAs are limited by registers; give each warp as deep a ring of page
    // buffers as the shared memory left at that occupancy allows (up to 8 stages).
    auto smem_for = [&](int st) {
        return static_cast<size_t>(kWarpsPerCta) * st * a.L.bytes + static_cast<size_t>(kWarpsPerCta) * st * 8 +
               static_cast<size_t>(kWarpsPerCta) * kWarpCtxBytes + static_cast<size_t>(a.B + 1) * 4;
    };
    auto occ_for = [&](size_t smem) {
        switch (a.L.Gk) {
            case 32: return decode_occupancy_gk32(a, smem);
            case 64: return decode_occupancy_gk64(a, smem);
            case 128: return decode_occupancy_gk128(a, smem);
            default: return 0;
        }
    };
    int dev = 0, sms = 0, smem_max = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    int stages = 2;
    if (smem_for(stages) > static_cast<size_t>(smem_max)) return cudaErrorInvalidConfiguration;
    int occ = occ_for(smem_for(stages));
    if (occ <= 0) return a.L.Gk == 32 || a.L.Gk == 64 || a.L.Gk == 128 ? cudaErrorInvalidConfiguration
                                                                    : cudaErrorInvalidValue;
    for (int st = kMaxStages; st > 2; --st) {
        if (smem_for(st) <= static_cast<size_t>(smem_max) && occ_for(smem_for(st)) >= occ) {
            stages = st;
            break;
        }
    }
    const size_t smem = smem_for(stages);
    const long long w_max = static_cast<long long>(sms) * occ * kWarpsPerCta;
    const long long pages_max = (static_cast<long long>(std::max(a.max_len, 0)) + a.L.P - 1) / a.L.P;
    const long long u_max = static_cast<long long>(a.Hkv) * a.B * pages_max;
    long long w = std::min(w_max, std::max<long long>(kWarpsPerCta, (u_max + 1) / 2));
    w = round_up(static_cast<size_t>(w), kWarpsPerCta);
    plan->warps = static_cast<int32_t>(w);
    plan->ctas = static_cast<int32_t>(w / kWarpsPerCta);
    plan->stages = stages;
    plan->smem_bytes = smem;
    const size_t pieces = static_cast<size_t>(w) + static_cast<size_t>(a.B) * a.Hkv;
    const size_t segs = static_cast<size_t>(a.B) * a.Hkv;
    const size_t part_ml = round_up(pieces * r * 2 * sizeof(float), kAlign);
    const size_t part_o = round_up(pieces * r * a.L.d * sizeof(float), kAlign);
    plan->ws_cnt_offset = kAlign;  // the first 256 bytes hold the status word
    plan->ws_gcnt_offset = plan->ws_cnt_offset + round_up(segs * sizeof(int32_t), kAlign);
    plan->ws_ml_offset = plan->ws_gcnt_offset + round_up(pieces * sizeof(int32_t), kAlign);
    plan->ws_o_offset = plan->ws_ml_offset + part_ml;
    plan->ws_gml_offset = plan->ws_o_offset + part_o;
    plan->ws_go_offset = plan->ws_gml_offset + part_ml;
    plan->ws_bytes = plan->ws_go_offset + part_o;
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    switch (a.L.Gk) {
        case 32: return decode_run_gk32(a, plan, stream);
        case 64: return decode_run_gk64(a, plan, stream);
        case 128: return decode_run_gk128(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kvq
