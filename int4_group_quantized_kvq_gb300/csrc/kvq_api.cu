// kvq_api.cu -- the extern "C" boundary: argument validation, geometry checks,
// dispatch to the kernels and error reporting.  No allocation, no hidden state
// except a per-thread error string.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "kvq.h"
#include "kvq_internal.h"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int ok() {
    g_err[0] = '\0';
    return KVQ_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool is_pow2_in(int x, int lo, int hi) { return x >= lo && x <= hi && (x & (x - 1)) == 0; }

// Geometry shared by every call.  Returns KVQ_OK or an error (with the message set).
int check_cfg(const kvq_cache_config* c) {
    if (!c) return fail(KVQ_EINVAL, "cfg is NULL");
    if (c->num_kv_heads < 1) return fail(KVQ_EINVAL, "num_kv_heads %d < 1", c->num_kv_heads);
    if (c->num_pages < 1) return fail(KVQ_EINVAL, "num_pages %d < 1", c->num_pages);
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256)
        return fail(KVQ_EUNSUPPORTED, "head_dim %d not in {64, 128, 256}", c->head_dim);
    if (!is_pow2_in(c->page_size, 16, 64)) return fail(KVQ_EUNSUPPORTED, "page_size %d not in {16, 32, 64}", c->page_size);
    if (!is_pow2_in(c->group_k, 32, 128) || c->group_k > c->head_dim)
        return fail(KVQ_EUNSUPPORTED, "group_k %d not in {32, 64, 128} or > head_dim", c->group_k);
    if (!is_pow2_in(c->group_v, 32, 128) || c->group_v > c->head_dim)
        return fail(KVQ_EUNSUPPORTED, "group_v %d not in {32, 64, 128} or > head_dim", c->group_v);
    const size_t blocks = static_cast<size_t>(c->num_pages) * c->num_kv_heads;
    if (blocks * kvq::block_layout(*c).bytes > (static_cast<size_t>(1) << 46))
        return fail(KVQ_EINVAL, "pool larger than 64 TiB");
    return KVQ_OK;
}

// Shapes the decode kernels take: the INT4 cache at head_dim 64, 128 or 256 (256: up to 4
// query heads per kv head and K groups of 64 or 128, the register budget of one warp's
// fragments); the other caches at head_dim 128.
int check_decode_shape(const kvq_cache_config* c, int r, int codec) {
    if (codec != 0 && c->head_dim != 128)
        return fail(KVQ_EUNSUPPORTED, "decode attention over this cache supports head_dim 128");
    if (c->head_dim == 256 && r > 4)
        return fail(KVQ_EUNSUPPORTED, "head_dim 256: query heads per KV head %d > 4", r);
    if (c->head_dim == 256 && c->group_k < 64)
        return fail(KVQ_EUNSUPPORTED, "head_dim 256: group_k %d < 64", c->group_k);
    return KVQ_OK;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(KVQ_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// The device address of page-locked host memory (cudaHostAlloc / cudaHostRegister), or
// nullptr for any other pointer (pageable host memory, device memory).
void* mapped_host_address(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // not a pointer the runtime knows: no lingering error
        return nullptr;
    }
    if (at.type != cudaMemoryTypeHost) return nullptr;
    return at.devicePointer;
}

}  // namespace

extern "C" {

size_t kvq_block_bytes(const kvq_cache_config* cfg) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    return static_cast<size_t>(kvq::block_layout(*cfg).bytes);
}

size_t kvq_pool_bytes(const kvq_cache_config* cfg) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    return static_cast<size_t>(cfg->num_pages) * cfg->num_kv_heads * kvq::block_layout(*cfg).bytes;
}

}  // extern "C"

namespace {
// The quantize-append of both entry points: `tokens` rows of [Hkv, d] in k and v, owned by
// the sequences as cu_rows says (nullptr: n_new each).
int quantize_append_impl(const kvq_cache_config* cfg, void* pool, const void* k, const void* v,
                         const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos,
                         const int32_t* cu_rows, int32_t batch, int32_t n_new, int64_t tokens, uint32_t* status,
                         kvq_stream_t stream, const char* name) {
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool || !k || !v || !block_table || !start_pos) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(k, 16) || !aligned(v, 16))
        return fail(KVQ_EINVAL, "pool, k and v must be 16-byte aligned");
    if (!aligned(block_table, 4) || !aligned(start_pos, 4) || (status && !aligned(status, 4)) ||
        (cu_rows && !aligned(cu_rows, 4)))
        return fail(KVQ_EINVAL, "int32/uint32 arguments must be 4-byte aligned");
    if (tokens * cfg->num_kv_heads >= (int64_t{1} << 30))
        return fail(KVQ_EINVAL, "tokens * num_kv_heads must be below 2^30 per call");
    kvq::QuantizeArgs a;
    a.pool = static_cast<uint8_t*>(pool);
    a.k = static_cast<const __half*>(k);
    a.v = static_cast<const __half*>(v);
    a.block_table = block_table;
    a.start_pos = start_pos;
    a.cu_rows = cu_rows;
    a.status = status;
    a.max_blocks = max_blocks;
    a.B = batch;
    a.n_new = n_new;
    a.Hkv = cfg->num_kv_heads;
    a.num_pages = cfg->num_pages;
    a.rows = static_cast<uint32_t>(tokens) * static_cast<uint32_t>(cfg->num_kv_heads);
    a.div_h = kvq::make_fastdiv(static_cast<uint32_t>(cfg->num_kv_heads));
    a.div_n = kvq::make_fastdiv(static_cast<uint32_t>(n_new > 0 ? n_new : 1));
    a.lg_p = 0;
    while ((1 << a.lg_p) < cfg->page_size) ++a.lg_p;
    a.lg_lanes_k = 0;
    while ((8 << a.lg_lanes_k) < cfg->group_k) ++a.lg_lanes_k;
    a.lg_lanes_v = 0;
    while ((8 << a.lg_lanes_v) < cfg->group_v) ++a.lg_lanes_v;
    a.L = kvq::block_layout(*cfg);
    cudaError_t e = kvq::launch_quantize_append(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, name);
    return ok();
}
}  // namespace

extern "C" {

int kvq_quantize_append(const kvq_cache_config* cfg, void* pool, const void* k, const void* v,
                        const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos, int32_t batch,
                        int32_t n_new, uint32_t* status, kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || n_new < 0) return fail(KVQ_EINVAL, "batch %d / n_new %d negative", batch, n_new);
    if (batch == 0 || n_new == 0) return ok();
    return quantize_append_impl(cfg, pool, k, v, block_table, max_blocks, start_pos, nullptr, batch, n_new,
                                static_cast<int64_t>(batch) * n_new, status, stream, "kvq_quantize_append launch");
}

int kvq_quantize_append_varlen(const kvq_cache_config* cfg, void* pool, const void* k_rows, const void* v_rows,
                               const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos,
                               const int32_t* cu_rows, int32_t batch, int32_t total_rows, uint32_t* status,
                               kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || total_rows < 0)
        return fail(KVQ_EINVAL, "batch %d / total_rows %d negative", batch, total_rows);
    if (batch == 0 || total_rows == 0) return ok();
    if (!cu_rows) return fail(KVQ_EINVAL, "NULL device pointer");
    return quantize_append_impl(cfg, pool, k_rows, v_rows, block_table, max_blocks, start_pos, cu_rows, batch, 0,
                                total_rows, status, stream, "kvq_quantize_append_varlen launch");
}

namespace {
// codec: 0 the INT4 cache, 1 the FP16 cache, 2 the INT8 per-row cache, 3 the rotated
// 4-bit cache
size_t workspace_bytes_impl(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads, int32_t max_len,
                            int codec) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    if (batch < 1 || num_q_heads < 1 || max_len < 0 || num_q_heads % cfg->num_kv_heads) {
        fail(KVQ_EINVAL, "invalid batch / num_q_heads / max_len");
        return 0;
    }
    if (check_decode_shape(cfg, num_q_heads / cfg->num_kv_heads, codec) != KVQ_OK) return 0;
    kvq::DecodeArgs a{};
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = cfg->num_kv_heads;
    a.max_len = max_len;
    a.fp16 = codec != 0;
    a.int8 = codec == 2;
    a.wht = codec == 3;
    a.L = kvq::block_layout(*cfg);
    kvq::DecodePlan plan;
    cudaError_t e = kvq::plan_decode(a, &plan);
    if (e != cudaSuccess) {
        fail(e == cudaErrorInvalidValue ? KVQ_EUNSUPPORTED : KVQ_ECUDA, "no decode kernel for this shape: %s",
             cudaGetErrorString(e));
        return 0;
    }
    ok();
    return plan.ws_bytes;
}
}  // namespace

size_t kvq_decode_workspace_bytes(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads,
                                  int32_t max_len) {
    return workspace_bytes_impl(cfg, batch, num_q_heads, max_len, 0);
}

size_t kvq_fp16_decode_workspace_bytes(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads,
                                       int32_t max_len) {
    return workspace_bytes_impl(cfg, batch, num_q_heads, max_len, 1);
}

size_t kvq_int8_decode_workspace_bytes(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads,
                                       int32_t max_len) {
    return workspace_bytes_impl(cfg, batch, num_q_heads, max_len, 2);
}

size_t kvq_wht4_decode_workspace_bytes(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads,
                                       int32_t max_len) {
    return workspace_bytes_impl(cfg, batch, num_q_heads, max_len, 3);
}

namespace {
int decode_attention_impl(const kvq_cache_config* cfg, const void* pool, const void* q, const int32_t* block_table,
                          int32_t max_blocks, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                          int32_t max_len, float softmax_scale, int32_t window, int32_t sinks, float* out,
                          void* workspace, size_t workspace_bytes, kvq_stream_t stream, int codec = 0,
                          uint64_t test_wait_ns = 0) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || num_q_heads < 1 || max_len < 0)
        return fail(KVQ_EINVAL, "batch %d, num_q_heads %d, max_len %d", batch, num_q_heads, max_len);
    if (window < 0 || sinks < 0) return fail(KVQ_EINVAL, "window %d, sinks %d", window, sinks);
    if (num_q_heads % cfg->num_kv_heads)
        return fail(KVQ_EINVAL, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, cfg->num_kv_heads);
    if (num_q_heads / cfg->num_kv_heads > 8)
        return fail(KVQ_EUNSUPPORTED, "query heads per KV head %d > 8", num_q_heads / cfg->num_kv_heads);
    if (int e = check_decode_shape(cfg, num_q_heads / cfg->num_kv_heads, codec)) return e;
    if (batch > 4096) return fail(KVQ_EUNSUPPORTED, "batch %d > 4096", batch);
    if (batch == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool || !q || !block_table || !seq_lens || !out || !workspace) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(q, 16) || !aligned(out, 16))
        return fail(KVQ_EINVAL, "pool, q and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(KVQ_EINVAL, "workspace must be 256-byte aligned");
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4)) return fail(KVQ_EINVAL, "int32 arguments must be aligned");
    kvq::DecodeArgs a;
    a.pool = static_cast<const uint8_t*>(pool);
    a.q = static_cast<const __half*>(q);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = out;
    a.workspace = static_cast<uint8_t*>(workspace);
    a.max_blocks = max_blocks;
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = cfg->num_kv_heads;
    a.num_pages = cfg->num_pages;
    a.max_len = max_len;
    a.softmax_scale = softmax_scale;
    a.window = window;
    a.sinks = sinks;
    a.fp16 = codec != 0;
    a.int8 = codec == 2;
    a.wht = codec == 3;
    a.L = kvq::block_layout(*cfg);
    if (test_wait_ns != 0) {
        a.wait_ns = test_wait_ns;
        a.withhold_first_copy = true;
    }
    kvq::DecodePlan plan;
    cudaError_t e = kvq::plan_decode(a, &plan);
    if (e == cudaErrorInvalidValue) return fail(KVQ_EUNSUPPORTED, "no decode kernel for this shape");
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention plan");
    if (workspace_bytes < plan.ws_bytes)
        return fail(KVQ_EWORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, plan.ws_bytes);
    e = kvq::launch_decode(a, plan, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention launch");
    return ok();
}

int decode_step_impl(const kvq_cache_config* cfg, void* pool, const void* k_new, const void* v_new,
                     const int32_t* append_pos, const void* q, const int32_t* block_table, int32_t max_blocks,
                     const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                     int32_t window, int32_t sinks, float* out, void* workspace, size_t workspace_bytes,
                     kvq_stream_t stream, float* out_host = nullptr, bool q_after_wait = false) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || num_q_heads < 1 || max_len < 0)
        return fail(KVQ_EINVAL, "batch %d, num_q_heads %d, max_len %d", batch, num_q_heads, max_len);
    if (window < 0 || sinks < 0) return fail(KVQ_EINVAL, "window %d, sinks %d", window, sinks);
    if (num_q_heads % cfg->num_kv_heads)
        return fail(KVQ_EINVAL, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, cfg->num_kv_heads);
    if (num_q_heads / cfg->num_kv_heads > 8)
        return fail(KVQ_EUNSUPPORTED, "query heads per KV head %d > 8", num_q_heads / cfg->num_kv_heads);
    if (int e = check_decode_shape(cfg, num_q_heads / cfg->num_kv_heads, 0)) return e;
    if (batch > 4096) return fail(KVQ_EUNSUPPORTED, "batch %d > 4096", batch);
    if (batch == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool || !k_new || !v_new || !append_pos || !q || !block_table || !seq_lens || !out || !workspace)
        return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(q, 16) || !aligned(out, 16) || !aligned(k_new, 16) || !aligned(v_new, 16))
        return fail(KVQ_EINVAL, "pool, k_new, v_new, q and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(KVQ_EINVAL, "workspace must be 256-byte aligned");
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(append_pos, 4))
        return fail(KVQ_EINVAL, "int32 arguments must be aligned");
    kvq::DecodeArgs a;
    a.pool = static_cast<const uint8_t*>(pool);
    a.q = static_cast<const __half*>(q);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = out;
    a.workspace = static_cast<uint8_t*>(workspace);
    a.max_blocks = max_blocks;
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = cfg->num_kv_heads;
    a.num_pages = cfg->num_pages;
    a.max_len = max_len;
    a.softmax_scale = softmax_scale;
    a.L = kvq::block_layout(*cfg);
    a.k_new = static_cast<const __half*>(k_new);
    a.v_new = static_cast<const __half*>(v_new);
    a.append_pos = append_pos;
    a.pool_w = static_cast<uint8_t*>(pool);
    a.window = window;
    a.sinks = sinks;
    a.out_host = out_host;
    a.q_after_wait = q_after_wait;
    kvq::DecodePlan plan;
    cudaError_t e = kvq::plan_decode(a, &plan);
    if (e == cudaErrorInvalidValue) return fail(KVQ_EUNSUPPORTED, "no decode kernel for this shape");
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_step plan");
    if (workspace_bytes < plan.ws_bytes)
        return fail(KVQ_EWORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, plan.ws_bytes);
    e = kvq::launch_decode(a, plan, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_step launch");
    return ok();
}
}  // namespace

int kvq_decode_attention(const kvq_cache_config* cfg, const void* pool, const void* q, const int32_t* block_table,
                         int32_t max_blocks, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                         int32_t max_len, float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                         kvq_stream_t stream) {
    return decode_attention_impl(cfg, pool, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                 softmax_scale, 0, 0, out, workspace, workspace_bytes, stream);
}

int kvq_test_decode_wait_timeout(const kvq_cache_config* cfg, const void* pool, const void* q,
                                 const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                                 int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale, float* out,
                                 void* workspace, size_t workspace_bytes, uint64_t wait_limit_ns,
                                 kvq_stream_t stream) {
    if (wait_limit_ns < 1000 || wait_limit_ns > 10000000)
        return fail(KVQ_EINVAL, "wait_limit_ns %llu outside [1 us, 10 ms]", static_cast<unsigned long long>(wait_limit_ns));
    return decode_attention_impl(cfg, pool, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                 softmax_scale, 0, 0, out, workspace, workspace_bytes, stream, 0, wait_limit_ns);
}

int kvq_decode_attention_window(const kvq_cache_config* cfg, const void* pool, const void* q,
                                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                                int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                                int32_t window, int32_t sinks, float* out, void* workspace, size_t workspace_bytes,
                                kvq_stream_t stream) {
    return decode_attention_impl(cfg, pool, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                 softmax_scale, window, sinks, out, workspace, workspace_bytes, stream);
}

int kvq_fp16_decode_attention(const kvq_cache_config* cfg, const void* pool16, const void* q,
                              const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                              int32_t num_q_heads, int32_t max_len, float softmax_scale, float* out, void* workspace,
                              size_t workspace_bytes, kvq_stream_t stream) {
    return decode_attention_impl(cfg, pool16, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                 softmax_scale, 0, 0, out, workspace, workspace_bytes, stream, 1);
}

int kvq_int8_decode_attention(const kvq_cache_config* cfg, const void* pool8, const void* q,
                              const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                              int32_t num_q_heads, int32_t max_len, float softmax_scale, float* out, void* workspace,
                              size_t workspace_bytes, kvq_stream_t stream) {
    return decode_attention_impl(cfg, pool8, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                 softmax_scale, 0, 0, out, workspace, workspace_bytes, stream, 2);
}

int kvq_wht4_decode_attention(const kvq_cache_config* cfg, const void* pool4r, const void* q,
                              const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                              int32_t num_q_heads, int32_t max_len, float softmax_scale, float* out, void* workspace,
                              size_t workspace_bytes, kvq_stream_t stream) {
    return decode_attention_impl(cfg, pool4r, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                 softmax_scale, 0, 0, out, workspace, workspace_bytes, stream, 3);
}

int kvq_decode_step(const kvq_cache_config* cfg, void* pool, const void* k_new, const void* v_new,
                    const int32_t* append_pos, const void* q, const int32_t* block_table, int32_t max_blocks,
                    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                    float* out, void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
    return decode_step_impl(cfg, pool, k_new, v_new, append_pos, q, block_table, max_blocks, seq_lens, batch,
                            num_q_heads, max_len, softmax_scale, 0, 0, out, workspace, workspace_bytes, stream);
}

int kvq_decode_step_host(const kvq_cache_config* cfg, void* pool, const void* host_in, void* dev_in,
                         const int32_t* append_pos, const int32_t* block_table, int32_t max_blocks,
                         const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len,
                         float softmax_scale, float* out, void* host_out, void* workspace, size_t workspace_bytes,
                         kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || num_q_heads < 1) return fail(KVQ_EINVAL, "batch %d, num_q_heads %d", batch, num_q_heads);
    if (batch == 0) return ok();
    if (!host_in || !dev_in || !host_out || !out) return fail(KVQ_EINVAL, "NULL buffer");
    if (!aligned(dev_in, 16)) return fail(KVQ_EINVAL, "dev_in must be 16-byte aligned");
    const size_t d = static_cast<size_t>(cfg->head_dim);
    const size_t q_bytes = static_cast<size_t>(batch) * num_q_heads * d * 2;
    const size_t kv_bytes = static_cast<size_t>(batch) * cfg->num_kv_heads * d * 2;
    const size_t in_bytes = q_bytes + 2 * kv_bytes;
    const size_t out_bytes = static_cast<size_t>(batch) * num_q_heads * d * 4;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint8_t* din = static_cast<uint8_t*>(dev_in);
    // Pinned host memory is read and written by the kernels themselves (through its device
    // address), so the step stays one chain of kernels launched behind each other; pageable
    // memory takes a copy on the stream.
    const void* in_dev = mapped_host_address(host_in);
    float* out_dev = static_cast<float*>(mapped_host_address(host_out));
    if (!aligned(in_dev, 16) || in_bytes % 16) in_dev = nullptr;
    if (!aligned(out_dev, 16)) out_dev = nullptr;
    cudaError_t e = in_dev ? kvq::launch_stage_in(in_dev, din, in_bytes / 16, st)
                           : cudaMemcpyAsync(din, host_in, in_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_step_host input copy");
    if (int rc = decode_step_impl(cfg, pool, din + q_bytes, din + q_bytes + kv_bytes, append_pos, din, block_table,
                                  max_blocks, seq_lens, batch, num_q_heads, max_len, softmax_scale, 0, 0, out,
                                  workspace, workspace_bytes, stream, out_dev, in_dev != nullptr))
        return rc;
    if (!out_dev) {
        e = cudaMemcpyAsync(host_out, out, out_bytes, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_step_host output copy");
    }
    return ok();
}

int kvq_decode_step_host_pipelined(const kvq_cache_config* cfg, void* pool, const void* host_in, void* dev_in,
                                   const int32_t* append_pos, const int32_t* block_table, int32_t max_blocks,
                                   const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len,
                                   float softmax_scale, float* out, void* host_out, void* workspace,
                                   size_t workspace_bytes, kvq_stream_t stream, kvq_stream_t copy_in,
                                   kvq_stream_t copy_out, kvq_event_t events[3]) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || num_q_heads < 1) return fail(KVQ_EINVAL, "batch %d, num_q_heads %d", batch, num_q_heads);
    if (batch == 0) return ok();
    if (!host_in || !dev_in || !host_out || !out || !events || !events[0] || !events[1] || !events[2])
        return fail(KVQ_EINVAL, "NULL buffer or event");
    if (!aligned(dev_in, 16)) return fail(KVQ_EINVAL, "dev_in must be 16-byte aligned");
    if (stream == copy_in || stream == copy_out || copy_in == copy_out)
        return fail(KVQ_EINVAL, "stream, copy_in and copy_out must be three distinct streams");
    const size_t d = static_cast<size_t>(cfg->head_dim);
    const size_t q_bytes = static_cast<size_t>(batch) * num_q_heads * d * 2;
    const size_t kv_bytes = static_cast<size_t>(batch) * cfg->num_kv_heads * d * 2;
    const size_t out_bytes = static_cast<size_t>(batch) * num_q_heads * d * 4;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const cudaStream_t ci = reinterpret_cast<cudaStream_t>(copy_in);
    const cudaStream_t co = reinterpret_cast<cudaStream_t>(copy_out);
    cudaEvent_t ev_in = reinterpret_cast<cudaEvent_t>(events[0]);
    cudaEvent_t ev_step = reinterpret_cast<cudaEvent_t>(events[1]);
    cudaEvent_t ev_out = reinterpret_cast<cudaEvent_t>(events[2]);
    uint8_t* din = static_cast<uint8_t*>(dev_in);
    cudaError_t e = cudaStreamWaitEvent(ci, ev_step, 0);  // the slot's last step has read dev_in
    if (e == cudaSuccess) e = cudaMemcpyAsync(din, host_in, q_bytes + 2 * kv_bytes, cudaMemcpyHostToDevice, ci);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, ci);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_out, 0);  // the slot's last output copy has read out
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_step_host_pipelined input copy");
    if (int rc = decode_step_impl(cfg, pool, din + q_bytes, din + q_bytes + kv_bytes, append_pos, din, block_table,
                                  max_blocks, seq_lens, batch, num_q_heads, max_len, softmax_scale, 0, 0, out,
                                  workspace, workspace_bytes, stream))
        return rc;
    e = cudaEventRecord(ev_step, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(co, ev_step, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(host_out, out, out_bytes, cudaMemcpyDeviceToHost, co);
    if (e == cudaSuccess) e = cudaEventRecord(ev_out, co);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_step_host_pipelined output copy");
    return ok();
}

int kvq_decode_step_window(const kvq_cache_config* cfg, void* pool, const void* k_new, const void* v_new,
                           const int32_t* append_pos, const void* q, const int32_t* block_table, int32_t max_blocks,
                           const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, int32_t max_len,
                           float softmax_scale, int32_t window, int32_t sinks, float* out, void* workspace,
                           size_t workspace_bytes, kvq_stream_t stream) {
    return decode_step_impl(cfg, pool, k_new, v_new, append_pos, q, block_table, max_blocks, seq_lens, batch,
                            num_q_heads, max_len, softmax_scale, window, sinks, out, workspace, workspace_bytes,
                            stream);
}

int kvq_dequantize(const kvq_cache_config* cfg, const void* pool, const int32_t* block_table, int32_t max_blocks,
                   int32_t b, int32_t start, int32_t n, void* out_k, void* out_v, int32_t out_dtype, uint32_t* status,
                   kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (b < 0 || start < 0 || n < 0) return fail(KVQ_EINVAL, "b %d, start %d, n %d", b, start, n);
    if (out_dtype != 0 && out_dtype != 1) return fail(KVQ_EINVAL, "out_dtype %d not 0 (fp16) or 1 (fp32)", out_dtype);
    if (n == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool || !block_table || !out_k || !out_v) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(out_k, 16) || !aligned(out_v, 16))
        return fail(KVQ_EINVAL, "pool, out_k and out_v must be 16-byte aligned");
    kvq::DequantArgs a;
    a.pool = static_cast<const uint8_t*>(pool);
    a.block_table = block_table;
    a.out_k = out_k;
    a.out_v = out_v;
    a.status = status;
    a.max_blocks = max_blocks;
    a.b = b;
    a.start = start;
    a.n = n;
    a.Hkv = cfg->num_kv_heads;
    a.num_pages = cfg->num_pages;
    a.out_fp32 = out_dtype;
    a.L = kvq::block_layout(*cfg);
    cudaError_t e = kvq::launch_dequantize(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kvq_dequantize launch");
    return ok();
}

size_t kvq_fp16_pool_bytes(const kvq_cache_config* cfg) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    return static_cast<size_t>(cfg->num_pages) * cfg->num_kv_heads * 4u * cfg->page_size * cfg->head_dim;
}

size_t kvq_int8_pool_bytes(const kvq_cache_config* cfg) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    return static_cast<size_t>(cfg->num_pages) * cfg->num_kv_heads *
           (2u * cfg->page_size * cfg->head_dim + 8u * cfg->page_size);
}

size_t kvq_wht4_pool_bytes(const kvq_cache_config* cfg) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    return static_cast<size_t>(cfg->num_pages) * cfg->num_kv_heads * cfg->page_size * (cfg->head_dim + 8u);
}

void kvq_wht4_codebook(float* levels16, float* thresholds15) {
    const kvq::Wht4Codebook& cb = kvq::wht4_codebook();
    for (int j = 0; j < 16 && levels16; ++j) levels16[j] = cb.levels[j];
    for (int j = 0; j < 15 && thresholds15; ++j) thresholds15[j] = cb.thresholds[j];
}

namespace {
// rows into the FP16 cache unchanged (codec 1), or quantized into the INT8 per-row cache
// (codec 2) or the rotated 4-bit cache (codec 3)
int rows_append_impl(const kvq_cache_config* cfg, void* pool16, const void* k, const void* v,
                    const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos, int32_t batch,
                    int32_t n_new, uint32_t* status, kvq_stream_t stream, int codec) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || n_new < 0) return fail(KVQ_EINVAL, "batch %d / n_new %d negative", batch, n_new);
    if (batch == 0 || n_new == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool16 || !k || !v || !block_table || !start_pos) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool16, 16) || !aligned(k, 16) || !aligned(v, 16))
        return fail(KVQ_EINVAL, "pool16, k and v must be 16-byte aligned");
    if (!aligned(block_table, 4) || !aligned(start_pos, 4) || (status && !aligned(status, 4)))
        return fail(KVQ_EINVAL, "int32/uint32 arguments must be 4-byte aligned");
    kvq::Fp16AppendArgs a;
    a.pool16 = static_cast<uint8_t*>(pool16);
    a.k = static_cast<const __half*>(k);
    a.v = static_cast<const __half*>(v);
    a.block_table = block_table;
    a.start_pos = start_pos;
    a.status = status;
    a.max_blocks = max_blocks;
    a.B = batch;
    a.n_new = n_new;
    a.Hkv = cfg->num_kv_heads;
    a.d = cfg->head_dim;
    a.P = cfg->page_size;
    a.num_pages = cfg->num_pages;
    if (codec == 2 && (cfg->head_dim % 4 || cfg->head_dim > 256))
        return fail(KVQ_EUNSUPPORTED, "the INT8 cache needs head_dim a multiple of 4, at most 256");
    if (codec == 3 && cfg->head_dim != 128) return fail(KVQ_EUNSUPPORTED, "the rotated 4-bit cache needs head_dim 128");
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = codec == 3   ? kvq::launch_wht4_quantize_append(a, st)
                    : codec == 2 ? kvq::launch_int8_quantize_append(a, st)
                                 : kvq::launch_fp16_append(a, st);
    if (e != cudaSuccess)
        return cuda_fail(e, codec == 3   ? "kvq_wht4_quantize_append launch"
                            : codec == 2 ? "kvq_int8_quantize_append launch"
                                         : "kvq_fp16_append launch");
    return ok();
}

}  // namespace

int kvq_fp16_append(const kvq_cache_config* cfg, void* pool16, const void* k, const void* v,
                    const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos, int32_t batch,
                    int32_t n_new, uint32_t* status, kvq_stream_t stream) {
    return rows_append_impl(cfg, pool16, k, v, block_table, max_blocks, start_pos, batch, n_new, status, stream, 1);
}

int kvq_int8_quantize_append(const kvq_cache_config* cfg, void* pool8, const void* k, const void* v,
                             const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos, int32_t batch,
                             int32_t n_new, uint32_t* status, kvq_stream_t stream) {
    return rows_append_impl(cfg, pool8, k, v, block_table, max_blocks, start_pos, batch, n_new, status, stream, 2);
}

int kvq_wht4_quantize_append(const kvq_cache_config* cfg, void* pool4r, const void* k, const void* v,
                             const int32_t* block_table, int32_t max_blocks, const int32_t* start_pos, int32_t batch,
                             int32_t n_new, uint32_t* status, kvq_stream_t stream) {
    return rows_append_impl(cfg, pool4r, k, v, block_table, max_blocks, start_pos, batch, n_new, status, stream, 3);
}

int kvq_wht4_dequantize(const kvq_cache_config* cfg, const void* pool4r, const int32_t* block_table,
                        int32_t max_blocks, int32_t b, int32_t start, int32_t n, float* out_k, float* out_v,
                        uint32_t* status, kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (cfg->head_dim != 128) return fail(KVQ_EUNSUPPORTED, "the rotated 4-bit cache needs head_dim 128");
    if (b < 0 || start < 0 || n < 0) return fail(KVQ_EINVAL, "b %d, start %d, n %d", b, start, n);
    if (n == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool4r || !block_table || !out_k || !out_v) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool4r, 16) || !aligned(out_k, 16) || !aligned(out_v, 16))
        return fail(KVQ_EINVAL, "pool, out_k and out_v must be 16-byte aligned");
    if (!aligned(block_table, 4) || (status && !aligned(status, 4)))
        return fail(KVQ_EINVAL, "int32/uint32 arguments must be 4-byte aligned");
    cudaError_t e = kvq::launch_wht4_dequantize(static_cast<const uint8_t*>(pool4r), block_table, max_blocks, b, start,
                                                n, out_k, out_v, status, cfg->num_kv_heads, cfg->page_size,
                                                cfg->num_pages, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kvq_wht4_dequantize launch");
    return ok();
}

int kvq_dequantize_to_fp16_pool(const kvq_cache_config* cfg, const void* pool, void* pool16,
                                const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                                int32_t batch, int32_t max_len, uint32_t* status, kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || max_len < 0) return fail(KVQ_EINVAL, "batch %d / max_len %d negative", batch, max_len);
    if (batch > 65535) return fail(KVQ_EUNSUPPORTED, "batch %d > 65535", batch);
    if (batch == 0 || max_len == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool || !pool16 || !block_table || !seq_lens) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(pool16, 16)) return fail(KVQ_EINVAL, "pool and pool16 must be 16-byte aligned");
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || (status && !aligned(status, 4)))
        return fail(KVQ_EINVAL, "int32/uint32 arguments must be 4-byte aligned");
    kvq::Fp16DequantArgs a;
    a.pool = static_cast<const uint8_t*>(pool);
    a.pool16 = static_cast<uint8_t*>(pool16);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.status = status;
    a.max_blocks = max_blocks;
    a.B = batch;
    a.Hkv = cfg->num_kv_heads;
    a.num_pages = cfg->num_pages;
    a.L = kvq::block_layout(*cfg);
    const long long max_pages = (static_cast<long long>(max_len) + cfg->page_size - 1) / cfg->page_size;
    cudaError_t e = kvq::launch_dequantize_to_fp16(a, max_pages, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "kvq_dequantize_to_fp16_pool launch");
    return ok();
}

namespace {
// The two grids of the mixed-precision decode: INT4 over positions [0, L - residual),
// FP16 over [L - residual, L); their workspaces back to back, one status word.
struct MixedPlan {
    kvq::DecodeArgs a4, a16;
    kvq::DecodePlan p4, p16;
    size_t off16, bytes;
};
cudaError_t plan_mixed(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads, int32_t max_len,
                       int32_t residual, MixedPlan* m) {
    kvq::DecodeArgs a{};
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = cfg->num_kv_heads;
    a.max_len = max_len;
    a.L = kvq::block_layout(*cfg);
    m->a4 = a;
    m->a4.len_sub = residual;
    m->a16 = a;
    m->a16.fp16 = true;
    m->a16.window = residual;
    cudaError_t e = kvq::plan_decode(m->a4, &m->p4);
    if (e != cudaSuccess) return e;
    e = kvq::plan_decode(m->a16, &m->p16);
    if (e != cudaSuccess) return e;
    m->off16 = (m->p4.ws_bytes + 255) / 256 * 256;
    m->bytes = m->off16 + m->p16.ws_bytes;
    return cudaSuccess;
}
}  // namespace

size_t kvq_mixed_decode_workspace_bytes(const kvq_cache_config* cfg, int32_t batch, int32_t num_q_heads,
                                        int32_t max_len, int32_t residual) {
    if (check_cfg(cfg) != KVQ_OK) return 0;
    if (batch < 1 || num_q_heads < 1 || max_len < 0 || residual < 0 || num_q_heads % cfg->num_kv_heads) {
        fail(KVQ_EINVAL, "invalid batch / num_q_heads / max_len / residual");
        return 0;
    }
    if (residual == 0) return kvq_decode_workspace_bytes(cfg, batch, num_q_heads, max_len);
    MixedPlan m;
    cudaError_t e = plan_mixed(cfg, batch, num_q_heads, max_len, residual, &m);
    if (e != cudaSuccess) {
        fail(e == cudaErrorInvalidValue ? KVQ_EUNSUPPORTED : KVQ_ECUDA, "no decode kernel for this shape: %s",
             cudaGetErrorString(e));
        return 0;
    }
    ok();
    return m.bytes;
}

int kvq_mixed_decode_attention(const kvq_cache_config* cfg, const void* pool, const int32_t* block_table,
                               int32_t max_blocks, const void* pool16, const int32_t* block_table16,
                               int32_t max_blocks16, int32_t num_pages16, const void* q, const int32_t* seq_lens,
                               int32_t batch, int32_t num_q_heads, int32_t max_len, int32_t residual,
                               float softmax_scale, float* out, void* workspace, size_t workspace_bytes,
                               kvq_stream_t stream) {
    if (residual < 0) return fail(KVQ_EINVAL, "residual %d < 0", residual);
    if (residual == 0)
        return kvq_decode_attention(cfg, pool, q, block_table, max_blocks, seq_lens, batch, num_q_heads, max_len,
                                    softmax_scale, out, workspace, workspace_bytes, stream);
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || num_q_heads < 1 || max_len < 0)
        return fail(KVQ_EINVAL, "batch %d, num_q_heads %d, max_len %d", batch, num_q_heads, max_len);
    if (num_q_heads % cfg->num_kv_heads)
        return fail(KVQ_EINVAL, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, cfg->num_kv_heads);
    if (num_q_heads / cfg->num_kv_heads > 8)
        return fail(KVQ_EUNSUPPORTED, "query heads per KV head %d > 8", num_q_heads / cfg->num_kv_heads);
    if (cfg->head_dim != 128) return fail(KVQ_EUNSUPPORTED, "decode attention supports head_dim 128");
    if (batch > 4096) return fail(KVQ_EUNSUPPORTED, "batch %d > 4096", batch);
    if (batch == 0) return ok();
    if (max_blocks < 1 || max_blocks16 < 1 || num_pages16 < 1)
        return fail(KVQ_EINVAL, "max_blocks %d, max_blocks16 %d, num_pages16 %d", max_blocks, max_blocks16,
                    num_pages16);
    if (!pool || !pool16 || !q || !block_table || !block_table16 || !seq_lens || !out || !workspace)
        return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(pool16, 16) || !aligned(q, 16) || !aligned(out, 16))
        return fail(KVQ_EINVAL, "pools, q and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(KVQ_EINVAL, "workspace must be 256-byte aligned");
    if (!aligned(block_table, 4) || !aligned(block_table16, 4) || !aligned(seq_lens, 4))
        return fail(KVQ_EINVAL, "int32 arguments must be aligned");
    MixedPlan m;
    cudaError_t e = plan_mixed(cfg, batch, num_q_heads, max_len, residual, &m);
    if (e == cudaErrorInvalidValue) return fail(KVQ_EUNSUPPORTED, "no decode kernel for this shape");
    if (e != cudaSuccess) return cuda_fail(e, "kvq_mixed_decode_attention plan");
    if (workspace_bytes < m.bytes)
        return fail(KVQ_EWORKSPACE, "workspace %zu bytes < %zu required", workspace_bytes, m.bytes);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    for (kvq::DecodeArgs* a : {&m.a4, &m.a16}) {
        a->q = static_cast<const __half*>(q);
        a->seq_lens = seq_lens;
        a->out = out;
        a->num_pages = cfg->num_pages;
        a->softmax_scale = softmax_scale;
        a->status = reinterpret_cast<uint32_t*>(ws);
    }
    m.a4.pool = static_cast<const uint8_t*>(pool);
    m.a4.block_table = block_table;
    m.a4.max_blocks = max_blocks;
    m.a4.workspace = ws;
    m.a16.pool = static_cast<const uint8_t*>(pool16);
    m.a16.block_table = block_table16;
    m.a16.max_blocks = max_blocks16;
    m.a16.num_pages = num_pages16;
    m.a16.workspace = ws + m.off16;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    e = kvq::launch_decode_grid(m.a4, m.p4, s);
    if (e == cudaSuccess) e = kvq::launch_decode_grid(m.a16, m.p16, s);
    if (e == cudaSuccess) e = kvq::launch_combine2(m.a4, m.p4, m.a16, m.p16, s);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_mixed_decode_attention launch");
    return ok();
}

int kvq_read_status(const void* status_word, uint32_t* flags, kvq_stream_t stream) {
    if (!status_word || !flags) return fail(KVQ_EINVAL, "NULL pointer");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(flags, status_word, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_read_status");
    return ok();
}

const char* kvq_last_error(void) { return g_err; }

const char* kvq_version(void) { return "kvq 0.1 (sm_103a)"; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode attention without any allocation.
//
// Some callers cannot hand the library a workspace.  A plugin inside a host
// engine may own no device allocator.  An embedded or real-time runtime may run
// with a fixed memory budget and forbid allocation once serving starts.  Code on
// an out-of-memory path cannot ask for more memory.  For them this entry point
// keeps its scratch in one array compiled into the library
// (kNoAllocScratchBytes = 8 MiB, held on every GPU that loads the library until
// the process exits) and never calls cudaMalloc, cudaFree or any allocating
// routine.
//
// The first call on a device looks up that device's address of the array
// (cudaGetSymbolAddress, with the device current); make that first call before
// any stream capture.  Every call on a device uses the same array, and the array
// keeps what the last call left in it.  Calls whose work overlaps on the GPU
// (other streams, other threads) race on it: serialize them.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(8) << 20;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t noalloc_scratch(void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (dev >= 0 && dev < kMaxDevices && g_noalloc_ptr[dev]) {
        *ptr = g_noalloc_ptr[dev];
        return cudaSuccess;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices) g_noalloc_ptr[dev] = p;
    *ptr = p;
    return cudaSuccess;
}

}  // namespace

extern "C" int kvq_decode_attention_noalloc(const kvq_cache_config* cfg, const void* pool, const void* q,
                                            const int32_t* block_table, int32_t max_blocks, const int32_t* seq_lens,
                                            int32_t batch, int32_t num_q_heads, int32_t max_len, float softmax_scale,
                                            float* out, uint32_t* status, kvq_stream_t stream) {
    if (int e = check_cfg(cfg)) return e;
    if (batch < 0 || num_q_heads < 1 || max_len < 0)
        return fail(KVQ_EINVAL, "batch %d, num_q_heads %d, max_len %d", batch, num_q_heads, max_len);
    if (num_q_heads % cfg->num_kv_heads)
        return fail(KVQ_EINVAL, "num_q_heads %d not a multiple of num_kv_heads %d", num_q_heads, cfg->num_kv_heads);
    if (num_q_heads / cfg->num_kv_heads > 8)
        return fail(KVQ_EUNSUPPORTED, "query heads per KV head %d > 8", num_q_heads / cfg->num_kv_heads);
    if (int e = check_decode_shape(cfg, num_q_heads / cfg->num_kv_heads, 0)) return e;
    if (batch > 4096) return fail(KVQ_EUNSUPPORTED, "batch %d > 4096", batch);
    if (batch == 0) return ok();
    if (max_blocks < 1) return fail(KVQ_EINVAL, "max_blocks %d < 1", max_blocks);
    if (!pool || !q || !block_table || !seq_lens || !out) return fail(KVQ_EINVAL, "NULL device pointer");
    if (!aligned(pool, 16) || !aligned(q, 16) || !aligned(out, 16))
        return fail(KVQ_EINVAL, "pool, q and out must be 16-byte aligned");
    if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || (status && !aligned(status, 4)))
        return fail(KVQ_EINVAL, "int32/uint32 arguments must be 4-byte aligned");
    kvq::DecodeArgs a;
    a.pool = static_cast<const uint8_t*>(pool);
    a.q = static_cast<const __half*>(q);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.out = out;
    a.max_blocks = max_blocks;
    a.B = batch;
    a.Hq = num_q_heads;
    a.Hkv = cfg->num_kv_heads;
    a.num_pages = cfg->num_pages;
    a.max_len = max_len;
    a.softmax_scale = softmax_scale;
    a.L = kvq::block_layout(*cfg);
    kvq::DecodePlan plan;
    cudaError_t e = kvq::plan_decode(a, &plan);
    if (e == cudaErrorInvalidValue) return fail(KVQ_EUNSUPPORTED, "no decode kernel for this shape");
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention_noalloc plan");
    if (plan.ws_bytes > kNoAllocScratchBytes)
        return fail(KVQ_EWORKSPACE,
                    "this shape needs %zu bytes of scratch; the built-in scratch of kvq_decode_attention_noalloc "
                    "holds %zu bytes (use kvq_decode_attention with a workspace)",
                    plan.ws_bytes, kNoAllocScratchBytes);
    // The scratch used is the current device's copy of the array: the arguments must live on
    // that device (q stands for them), or the kernel would pair them with another GPU's array.
    {
        int cur = 0;
        cudaPointerAttributes attr{};
        e = cudaGetDevice(&cur);
        if (e == cudaSuccess) e = cudaPointerGetAttributes(&attr, q);
        if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention_noalloc device check");
        if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
            return fail(KVQ_EINVAL, "kvq_decode_attention_noalloc: q is not device memory");
        if (attr.device != cur)
            return fail(KVQ_EINVAL,
                        "kvq_decode_attention_noalloc: q is on device %d but device %d is current; make the device "
                        "of the stream and the buffers current",
                        attr.device, cur);
    }
    void* scratch = nullptr;
    e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention_noalloc scratch lookup");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The status word must start each call at zero (the partial results and the pages
    // prefix behind it are written before they are read).
    e = cudaMemsetAsync(scratch, 0, plan.ws_ml_offset, s);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention_noalloc scratch clear");
    a.workspace = static_cast<uint8_t*>(scratch);
    e = kvq::launch_decode(a, plan, s);
    if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention_noalloc launch");
    if (status) {
        e = cudaMemcpyAsync(status, scratch, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "kvq_decode_attention_noalloc status copy");
    }
    return ok();
}
