// decode_plan.cu -- sizing of the persistent split-KV grid and of its workspace.
//
// A unit of work is one page of HK consecutive kv heads: HK = 4 when every query head
// has its own kv head, Hkv is a multiple of 4 and pages hold 16 tokens, else HK = 1.
// The grid is C CTAs of 4 warps: C is the number of CTAs the device keeps resident (SMs
// x resident CTAs), reduced for small problems so that a warp gets at least two units;
// every CTA receives an equal contiguous slice of the flattened (sequence, head group,
// page) units.  Each warp writes one partial per segment (sequence, head group) its
// CTA's slice touches, at index 4 * (CTA + segment) + warp, which is unique (CTA +
// segment is: if CTA k touches segment s and CTA k - 1 touches s + 1, CTA k - 1 would
// hold a later unit than CTA k, which ordered slices rule out).  So the workspace holds
// 4 * (C + B * Hg) partials of ns = HK * r query heads, each (max, sum) plus d floats,
// and the pages prefix the decode grid publishes for the combine kernel, which runs
// next with one CTA per (sequence, query head) row.  Nothing in the workspace carries
// over from one call to the next.
#include <algorithm>

#include "kvq_internal.h"

namespace kvq {

cudaError_t decode_run_gk32(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk64(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk128(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_gk32(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk64(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk128(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
cudaError_t decode_run_gk32_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk64_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_gk128_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_gk32_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk64_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_gk128_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
cudaError_t decode_run_d64(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_d64_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_d256(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_d256_win(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_d64(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_d64_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_d256(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
int decode_occupancy_d256_win(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
cudaError_t launch_combine(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
cudaError_t decode_run_fp16(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_fp16(const DecodeArgs& a, const DecodePlan& plan, size_t smem);
cudaError_t decode_run_int8(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t s);
int decode_occupancy_int8(const DecodeArgs& a, const DecodePlan& plan, size_t smem);

namespace {
constexpr int kMaxStages = 8;           // deepest unit ring per warp
constexpr size_t kMaxRingBytes = 8 * 2144;  // per warp: deeper rings gain nothing
constexpr int kMinUnitsPerWarp = 2;
constexpr size_t kAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
}  // namespace

cudaError_t plan_decode(const DecodeArgs& a, DecodePlan* plan) {
    // the INT4 kernels take head_dim 64, 128 or 256 (256: up to 4 query heads per kv head);
    // the other caches and the mixed decode head_dim 128
    if (a.L.d != 128 && (a.fp16 || (a.L.d != 64 && a.L.d != 256))) return cudaErrorInvalidValue;
    if (a.L.P % 16 != 0) return cudaErrorInvalidValue;
    const int r = a.Hq / a.Hkv;
    if (r < 1 || r > (a.L.d == 256 ? 4 : 8)) return cudaErrorInvalidValue;
    // four kv heads per unit for 16-token pages (a 4-block unit then stays near the size
    // of one larger page); larger pages are big enough copies on their own
    plan->hk = (!a.fp16 && r == 1 && a.Hkv % 4 == 0 && a.L.P == 16 && a.L.d <= 128) ? 4 : 1;
    plan->hs = (plan->hk == 1 && r > 4) ? 2 : 1;
    // CTA bookkeeping (128 bytes) and the two q buffers of 12 rows of head_dim fp16 (the q
    // rows of a segment and, in the decode step, the new token's K and V rows)
    const size_t kCtlBytes = 128 + static_cast<size_t>(2) * 12 * a.L.d * 2;
    const int hg = a.Hkv / plan->hk;
    const int kWarpsPerCta = 4;  // the kernel's CTA size
    const int ns = plan->hk * r;
    // the FP16 cache's unit is one page of one kv head: K and V rows, P x d fp16 each
    // (the INT8 cache's: K and V codes P x d each, then 2 P fp32 scales)
    const size_t unit = !a.fp16 ? static_cast<size_t>(a.L.bytes) * plan->hk
                        : a.wht  ? static_cast<size_t>(a.L.P) * (a.L.d + 8)
                        : a.int8 ? static_cast<size_t>(2) * a.L.P * a.L.d + static_cast<size_t>(8) * a.L.P
                                 : static_cast<size_t>(4) * a.L.P * a.L.d;
    // Resident CTAs are limited by registers; give each warp as deep a ring of unit
    // buffers as the shared memory left at that occupancy allows.
    // per warp and stage: the unit buffer, its mbarrier and the unit's pool address
    auto smem_for = [&](int st) {
        return static_cast<size_t>(kWarpsPerCta) * st * unit + static_cast<size_t>(kWarpsPerCta) * st * 16 +
               kCtlBytes + round_up(static_cast<size_t>(3 * a.B + 1) * 4, 16);
    };
    auto occ_for = [&](size_t smem) {
        if (a.int8) return decode_occupancy_int8(a, *plan, smem);
        if (a.fp16) return decode_occupancy_fp16(a, *plan, smem);
        const bool w = a.window > 0;
        if (a.L.d == 64) return w ? decode_occupancy_d64_win(a, *plan, smem) : decode_occupancy_d64(a, *plan, smem);
        if (a.L.d == 256) return w ? decode_occupancy_d256_win(a, *plan, smem) : decode_occupancy_d256(a, *plan, smem);
        switch (a.L.Gk) {
            case 32: return w ? decode_occupancy_gk32_win(a, *plan, smem) : decode_occupancy_gk32(a, *plan, smem);
            case 64: return w ? decode_occupancy_gk64_win(a, *plan, smem) : decode_occupancy_gk64(a, *plan, smem);
            case 128: return w ? decode_occupancy_gk128_win(a, *plan, smem) : decode_occupancy_gk128(a, *plan, smem);
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
    // a 64-token FP16 page (32 KB) leaves room for one stage per warp only: its copy is
    // then not overlapped with the arithmetic
    if (a.fp16 && smem_for(stages) > static_cast<size_t>(smem_max)) stages = 1;
    if (smem_for(stages) > static_cast<size_t>(smem_max)) return cudaErrorInvalidConfiguration;
    const int occ = occ_for(smem_for(stages));
    if (occ <= 0) return a.L.Gk == 32 || a.L.Gk == 64 || a.L.Gk == 128 ? cudaErrorInvalidConfiguration
                                                                    : cudaErrorInvalidValue;
    for (int st = kMaxStages; st > 2; --st) {
        if (static_cast<size_t>(st) * unit > std::max(kMaxRingBytes, 3 * unit)) continue;
        if (smem_for(st) <= static_cast<size_t>(smem_max) && occ_for(smem_for(st)) >= occ) {
            stages = st;
            break;
        }
    }
    const long long c_max = static_cast<long long>(sms) * occ;
    long long pages_max = (static_cast<long long>(std::max(a.max_len, 0)) + a.L.P - 1) / a.L.P;
    if (a.window > 0) {  // a sequence lists its sink pages and at most window / P + 1 window pages
        const long long sink_pages = (std::min<long long>(std::max(a.sinks, 0), std::max(a.max_len, 0)) + a.L.P - 1) / a.L.P;
        pages_max = std::min(pages_max, sink_pages + a.window / a.L.P + 2);
    }
    const long long u_max = static_cast<long long>(hg) * a.B * pages_max;
    const long long ctas = std::min(c_max, std::max<long long>(1, u_max / (kMinUnitsPerWarp * kWarpsPerCta)));
    plan->ctas = static_cast<int32_t>(ctas);
    // Combine CTA size from the most partials a row can have: a segment of pages_max
    // units spans about pages_max / (u_max / ctas) + 2 CTA slices, 4 partials each; a
    // warp folds 8 partials per round trip, so give it about 8 of them.
    {
        const long long per_cta = std::max<long long>(1, u_max / ctas);
        const long long parts = kWarpsPerCta * (pages_max / per_cta + 2);
        plan->combine_warps = parts <= 32 ? 4 : (parts <= 64 ? 8 : 16);
    }
    plan->stages = stages;
    plan->smem_bytes = smem_for(stages);
    const size_t pieces = static_cast<size_t>(kWarpsPerCta) * (static_cast<size_t>(ctas) + static_cast<size_t>(a.B) * hg);
    plan->ws_pre_offset = kAlign;  // the first 256 bytes hold the status word
    plan->ws_ml_offset = plan->ws_pre_offset + round_up((static_cast<size_t>(a.B) + 1) * sizeof(int32_t), kAlign);
    plan->ws_o_offset = plan->ws_ml_offset + round_up(pieces * ns * 2 * sizeof(float), kAlign);
    plan->ws_bytes = plan->ws_o_offset + round_up(pieces * ns * a.L.d * sizeof(float), kAlign);
    return cudaSuccess;
}

cudaError_t launch_decode_grid(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    if (a.int8) return decode_run_int8(a, plan, stream);
    if (a.fp16) return decode_run_fp16(a, plan, stream);
    const bool w = a.window > 0;
    if (a.L.d == 64) return w ? decode_run_d64_win(a, plan, stream) : decode_run_d64(a, plan, stream);
    if (a.L.d == 256) return w ? decode_run_d256_win(a, plan, stream) : decode_run_d256(a, plan, stream);
    switch (a.L.Gk) {
        case 32: return w ? decode_run_gk32_win(a, plan, stream) : decode_run_gk32(a, plan, stream);
        case 64: return w ? decode_run_gk64_win(a, plan, stream) : decode_run_gk64(a, plan, stream);
        case 128: return w ? decode_run_gk128_win(a, plan, stream) : decode_run_gk128(a, plan, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t stream) {
    cudaError_t e = launch_decode_grid(a, plan, stream);
    if (e != cudaSuccess) return e;
    return launch_combine(a, plan, stream);
}

}  // namespace kvq
