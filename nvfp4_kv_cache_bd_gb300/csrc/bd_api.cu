// Host side of the C ABI declared in include/bd.h: argument validation,
// context state and kernel launches.  Every error in a host-side argument is
// detected here, before any CUDA call, and returned as a status code;
// device-resident indexes are checked by the kernels (device error word).
#include <math.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#include "bd_copy.h"
#include "bd_internal.h"

struct bd_ctx {
    bd_config cfg;
    std::mutex mu_lock;
    int device = -1;
    float* d_mu = nullptr;   // [num_layers][num_kv_heads][128], zero-initialised
    int* d_err = nullptr;    // device error word
};

namespace {

using bd::kD;

bool finite_in(float x, float lo, float hi) { return isfinite(x) && x >= lo && x <= hi; }

int check_cfg(const bd_config* c) {
    if (!c) return BD_ERR_INVALID_ARG;
    if (c->num_layers < 1 || c->num_layers > 4096) return BD_ERR_INVALID_ARG;
    if (c->num_kv_heads < 1 || c->num_q_heads < 1) return BD_ERR_INVALID_ARG;
    if (c->format != BD_FORMAT_NVFP4 && c->format != BD_FORMAT_MXFP4) return BD_ERR_INVALID_ARG;
    if ((c->key_search | c->rotation | c->centering) & ~1) return BD_ERR_INVALID_ARG;
    if (c->query_terms != 1 && c->query_terms != 2) return BD_ERR_INVALID_ARG;
    if (c->p_mode < BD_P_NONE || c->p_mode > BD_P_AMAX2_OR_AMAX6) return BD_ERR_INVALID_ARG;
    // the probability kernel supports c = 1 or c = 8 (config.py probability_environment)
    if (c->p_c != 1 && c->p_c != 8) return BD_ERR_INVALID_ARG;
    if (c->pool_pages < 0) return BD_ERR_INVALID_ARG;
    if (c->head_dim != 128 || c->page_size != 128 || c->sink_tokens != 16) return BD_ERR_UNSUPPORTED;
    if (c->num_q_heads != bd::kGroup * c->num_kv_heads || c->num_kv_heads > 16) return BD_ERR_UNSUPPORTED;
    return BD_OK;
}

// Allocate the context's device state on the current device (first launch).
int ensure_device(bd_ctx* ctx) {
    std::lock_guard<std::mutex> g(ctx->mu_lock);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BD_ERR_CUDA;
    if (ctx->d_mu) return dev == ctx->device ? BD_OK : BD_ERR_INVALID_ARG;
    const size_t mu_bytes = (size_t)ctx->cfg.num_layers * ctx->cfg.num_kv_heads * kD * sizeof(float);
    if (cudaMalloc(&ctx->d_mu, mu_bytes) != cudaSuccess) return BD_ERR_CUDA;
    if (cudaMalloc(&ctx->d_err, sizeof(int)) != cudaSuccess) {
        cudaFree(ctx->d_mu);
        ctx->d_mu = nullptr;
        return BD_ERR_CUDA;
    }
    if (cudaMemset(ctx->d_mu, 0, mu_bytes) != cudaSuccess || cudaMemset(ctx->d_err, 0, sizeof(int)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return BD_ERR_CUDA;
    ctx->device = dev;
    return BD_OK;
}

const float* layer_mu(const bd_ctx* ctx, int layer) {
    return ctx->d_mu + (size_t)layer * ctx->cfg.num_kv_heads * kD;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? BD_OK : BD_ERR_CUDA; }

}  // namespace

extern "C" {

int bd_create(const bd_config* cfg, bd_ctx** out) {
    if (!out) return BD_ERR_INVALID_ARG;
    const int st = check_cfg(cfg);
    if (st != BD_OK) return st;
    bd_ctx* ctx = new (std::nothrow) bd_ctx;
    if (!ctx) return BD_ERR_INVALID_ARG;
    ctx->cfg = *cfg;
    *out = ctx;
    return BD_OK;
}

void bd_destroy(bd_ctx* ctx) {
    if (!ctx) return;
    if (ctx->d_mu) cudaFree(ctx->d_mu);
    if (ctx->d_err) cudaFree(ctx->d_err);
    delete ctx;
}

const char* bd_status_string(int status) {
    switch (status) {
        case BD_OK: return "ok";
        case BD_ERR_INVALID_ARG: return "invalid argument";
        case BD_ERR_UNSUPPORTED: return "unsupported configuration";
        case BD_ERR_CUDA: return "CUDA runtime error";
        case BD_ERR_WORKSPACE: return "workspace too small";
        case BD_ERR_TIMEOUT: return "device-side wait timed out";
        default: return "unknown status";
    }
}

int bd_set_key_shift(bd_ctx* ctx, int layer, const float* mu_host) {
    if (!ctx || !mu_host || layer < 0 || layer >= ctx->cfg.num_layers) return BD_ERR_INVALID_ARG;
    const size_t n = (size_t)ctx->cfg.num_kv_heads * kD;
    for (size_t i = 0; i < n; ++i)
        if (!isfinite(mu_host[i])) return BD_ERR_INVALID_ARG;
    int st = ensure_device(ctx);
    if (st != BD_OK) return st;
    // A copy from pageable memory may return before its DMA lands; wait for
    // it so that every kernel launched afterwards reads the new mean.
    cudaError_t e = cudaMemcpyAsync((void*)layer_mu(ctx, layer), mu_host, n * sizeof(float), cudaMemcpyHostToDevice, 0);
    if (e == cudaSuccess) e = cudaStreamSynchronize(0);
    return cuda_status(e);
}

size_t bd_record_bytes(const bd_ctx* ctx) { return ctx ? (size_t)bd::record_bytes(ctx->cfg.format) : 0; }

size_t bd_query_packed_bytes(const bd_ctx* ctx) { return ctx ? bd::qpack_stride(ctx->cfg.num_q_heads) : 0; }

int bd_quantize_kv_pages(bd_ctx* ctx, int layer, const void* k, const void* v, const int32_t* dst_pages, int n,
                         float k_gscale, float v_gscale, void* kv_pool, void* stream) {
    if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers || n < 0 || n > (1 << 24)) return BD_ERR_INVALID_ARG;
    if (!finite_in(k_gscale, 1e-30f, 1e30f) || !finite_in(v_gscale, 1e-30f, 1e30f)) return BD_ERR_INVALID_ARG;
    if (n == 0) return BD_OK;
    if (!k || !v || !dst_pages || !kv_pool) return BD_ERR_INVALID_ARG;
    if (((uintptr_t)k | (uintptr_t)v) & 15u || ((uintptr_t)kv_pool & 15u)) return BD_ERR_INVALID_ARG;
    int st = ensure_device(ctx);
    if (st != BD_OK) return st;
    bd::WriterArgs a;
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.dst_pages = dst_pages;
    a.mu = layer_mu(ctx, layer);
    a.pool = static_cast<uint8_t*>(kv_pool);
    a.n = n;
    a.hkv = ctx->cfg.num_kv_heads;
    a.format = ctx->cfg.format;
    a.key_search = ctx->cfg.key_search;
    a.rotation = ctx->cfg.rotation;
    a.centering = ctx->cfg.centering;
    a.pool_pages = ctx->cfg.pool_pages;
    a.gk = k_gscale;
    a.gv = v_gscale;
    a.err = ctx->d_err;
    return cuda_status(bd::launch_writer(a, static_cast<cudaStream_t>(stream)));
}

int bd_append_kv(bd_ctx* ctx, int layer, const void* k_new, const void* v_new, const int32_t* seq_lens,
                 const int32_t* block_table, int max_blocks, void* sink_k, void* sink_v, void* tail_k, void* tail_v,
                 int B, float k_gscale, float v_gscale, void* kv_pool, void* stream) {
    if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers || B < 0 || B > (1 << 20)) return BD_ERR_INVALID_ARG;
    if (max_blocks < 0 || max_blocks > (1 << 22)) return BD_ERR_INVALID_ARG;
    if (!finite_in(k_gscale, 1e-30f, 1e30f) || !finite_in(v_gscale, 1e-30f, 1e30f)) return BD_ERR_INVALID_ARG;
    if (B == 0) return BD_OK;
    if (!k_new || !v_new || !seq_lens || !sink_k || !sink_v || !tail_k || !tail_v) return BD_ERR_INVALID_ARG;
    if (max_blocks > 0 && (!block_table || !kv_pool)) return BD_ERR_INVALID_ARG;
    const uintptr_t align = (uintptr_t)k_new | (uintptr_t)v_new | (uintptr_t)sink_k | (uintptr_t)sink_v |
                            (uintptr_t)tail_k | (uintptr_t)tail_v | (uintptr_t)kv_pool;
    if (align & 15u) return BD_ERR_INVALID_ARG;
    int st = ensure_device(ctx);
    if (st != BD_OK) return st;
    bd::WriterArgs a;
    a.k = static_cast<const uint16_t*>(tail_k);
    a.v = static_cast<const uint16_t*>(tail_v);
    a.dst_pages = nullptr;
    a.mu = layer_mu(ctx, layer);
    a.pool = static_cast<uint8_t*>(kv_pool);
    a.n = B;
    a.hkv = ctx->cfg.num_kv_heads;
    a.format = ctx->cfg.format;
    a.key_search = ctx->cfg.key_search;
    a.rotation = ctx->cfg.rotation;
    a.centering = ctx->cfg.centering;
    a.pool_pages = ctx->cfg.pool_pages;
    a.gk = k_gscale;
    a.gv = v_gscale;
    a.seq_lens = seq_lens;
    a.block_table = block_table;
    a.max_blocks = max_blocks;
    a.k_new = static_cast<const uint16_t*>(k_new);
    a.v_new = static_cast<const uint16_t*>(v_new);
    a.sink_k = static_cast<uint16_t*>(sink_k);
    a.sink_v = static_cast<uint16_t*>(sink_v);
    a.tail_k = static_cast<uint16_t*>(tail_k);
    a.tail_v = static_cast<uint16_t*>(tail_v);
    a.err = ctx->d_err;
    return cuda_status(bd::launch_writer(a, static_cast<cudaStream_t>(stream)));
}

int bd_quantize_query(bd_ctx* ctx, int layer, const void* q, int B, void* q_packed, void* stream) {
    if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers || B < 0 || B > (1 << 20)) return BD_ERR_INVALID_ARG;
    if (B == 0) return BD_OK;
    if (!q || !q_packed || ((uintptr_t)q & 15u) || ((uintptr_t)q_packed & 15u)) return BD_ERR_INVALID_ARG;
    int st = ensure_device(ctx);
    if (st != BD_OK) return st;
    bd::QueryArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.mu = layer_mu(ctx, layer);
    a.qp = static_cast<uint8_t*>(q_packed);
    a.B = B;
    a.hq = ctx->cfg.num_q_heads;
    a.format = ctx->cfg.format;
    a.rotation = ctx->cfg.rotation;
    a.centering = ctx->cfg.centering;
    a.terms = ctx->cfg.query_terms;
    a.stride = bd::qpack_stride(a.hq);
    return cuda_status(bd::launch_query(a, static_cast<cudaStream_t>(stream)));
}

size_t bd_decode_workspace_size(const bd_ctx* ctx, int B, int max_blocks) {
    if (!ctx || B <= 0 || max_blocks < 0) return 0;
    int ns = 0, pps = 0;
    bd::decode_splits(B, ctx->cfg.num_kv_heads, max_blocks, &ns, &pps);
    return bd::decode_ws_bytes(B, ctx->cfg.num_q_heads, ctx->cfg.num_kv_heads, ns);
}

int bd_decode_attention(bd_ctx* ctx, int layer, const void* q_packed, const void* q, const void* kv_pool,
                        const int32_t* block_table, int max_blocks, const int32_t* seq_lens, const void* sink_k,
                        const void* sink_v, const void* tail_k, const void* tail_v, int B, float tau,
                        float k_gscale, float v_gscale, float* out, void* ws, size_t ws_bytes, void* stream) {
    if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers || B < 0 || B > (1 << 20)) return BD_ERR_INVALID_ARG;
    if (max_blocks < 0 || max_blocks > (1 << 22)) return BD_ERR_INVALID_ARG;
    // tau must be a finite number between 0 and 448 (config.py probability_environment)
    if (!finite_in(tau, 0.0f, 448.0f)) return BD_ERR_INVALID_ARG;
    if (!finite_in(k_gscale, 1e-30f, 1e30f) || !finite_in(v_gscale, 1e-30f, 1e30f)) return BD_ERR_INVALID_ARG;
    if (B == 0) return BD_OK;
    if (!q || !seq_lens || !sink_k || !sink_v || !tail_k || !tail_v || !out || !ws) return BD_ERR_INVALID_ARG;
    // no packed query: the decode quantizes q itself, for up to 32 query heads
    if (!q_packed && ctx->cfg.num_q_heads > 32) return BD_ERR_UNSUPPORTED;
    if (max_blocks > 0 && (!block_table || !kv_pool)) return BD_ERR_INVALID_ARG;
    const uintptr_t align = (uintptr_t)q_packed | (uintptr_t)kv_pool | (uintptr_t)q | (uintptr_t)sink_k |
                            (uintptr_t)sink_v | (uintptr_t)tail_k | (uintptr_t)tail_v | (uintptr_t)out | (uintptr_t)ws;
    if (align & 15u) return BD_ERR_INVALID_ARG;
    if (ws_bytes < bd_decode_workspace_size(ctx, B, max_blocks)) return BD_ERR_WORKSPACE;
    int st = ensure_device(ctx);
    if (st != BD_OK) return st;
    bd::DecodeArgs a;
    a.qp = static_cast<const uint8_t*>(q_packed);
    a.q = static_cast<const uint16_t*>(q);
    a.mu = layer_mu(ctx, layer);
    a.rotation = ctx->cfg.rotation;
    a.terms = ctx->cfg.query_terms;
    a.pool = static_cast<const uint8_t*>(kv_pool);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.sink_k = static_cast<const uint16_t*>(sink_k);
    a.sink_v = static_cast<const uint16_t*>(sink_v);
    a.tail_k = static_cast<const uint16_t*>(tail_k);
    a.tail_v = static_cast<const uint16_t*>(tail_v);
    a.out = out;
    a.parts = static_cast<float*>(ws);
    a.err = ctx->d_err;
    a.qstride = bd::qpack_stride(ctx->cfg.num_q_heads);
    a.B = B;
    a.hq = ctx->cfg.num_q_heads;
    a.hkv = ctx->cfg.num_kv_heads;
    a.max_blocks = max_blocks;
    bd::decode_splits(B, a.hkv, max_blocks, &a.nsplit, &a.pages_per_split);
    a.counters = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(ws) +
                                                       bd::decode_parts_bytes(B, a.hq, a.nsplit));
    a.tag = bd::next_decode_tag();
    a.pool_pages = ctx->cfg.pool_pages;
    a.format = ctx->cfg.format;
    a.centering = ctx->cfg.centering;
    a.p_mode = ctx->cfg.p_mode;
    a.p_c = ctx->cfg.p_c;
    a.tau = tau;
    a.gk = k_gscale;
    a.gv = v_gscale;
    return cuda_status(bd::launch_decode(a, static_cast<cudaStream_t>(stream)));
}

int bd_decode_attention_noalloc(bd_ctx* ctx, int layer, const void* q_packed, const void* q, const void* kv_pool,
                                const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                                const void* sink_k, const void* sink_v, const void* tail_k, const void* tail_v, int B,
                                float tau, float k_gscale, float v_gscale, float* out, void* stream) {
    // Same checks as bd_decode_attention; no cudaMalloc, cudaFree or other
    // allocating call is made on this path.
    if (!ctx || layer < 0 || layer >= ctx->cfg.num_layers || B < 0 || B > (1 << 20)) return BD_ERR_INVALID_ARG;
    if (max_blocks < 0 || max_blocks > (1 << 22)) return BD_ERR_INVALID_ARG;
    if (!finite_in(tau, 0.0f, 448.0f)) return BD_ERR_INVALID_ARG;
    if (!finite_in(k_gscale, 1e-30f, 1e30f) || !finite_in(v_gscale, 1e-30f, 1e30f)) return BD_ERR_INVALID_ARG;
    if (B == 0) return BD_OK;
    if (!q || !seq_lens || !sink_k || !sink_v || !tail_k || !tail_v || !out) return BD_ERR_INVALID_ARG;
    if (!q_packed && ctx->cfg.num_q_heads > 32) return BD_ERR_UNSUPPORTED;
    if (max_blocks > 0 && (!block_table || !kv_pool)) return BD_ERR_INVALID_ARG;
    const uintptr_t align = (uintptr_t)q_packed | (uintptr_t)kv_pool | (uintptr_t)q | (uintptr_t)sink_k |
                            (uintptr_t)sink_v | (uintptr_t)tail_k | (uintptr_t)tail_v | (uintptr_t)out;
    if (align & 15u) return BD_ERR_INVALID_ARG;
    // the fixed scratch must hold this call's split partials
    const size_t need = bd_decode_workspace_size(ctx, B, max_blocks);
    if (need > bd::kNoAllocScratchBytes) return BD_ERR_WORKSPACE;
    {
        // a context is bound to the device of its first launch: its error word
        // lives there
        std::lock_guard<std::mutex> g(ctx->mu_lock);
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess) return BD_ERR_CUDA;
        if (ctx->d_mu && dev != ctx->device) return BD_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    if (bd::noalloc_scratch(&scratch) != cudaSuccess) return BD_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bd::DecodeArgs a;
    a.qp = static_cast<const uint8_t*>(q_packed);
    a.q = static_cast<const uint16_t*>(q);
    // this path never creates the key-mean array: without it no shift was set
    // (q.mu = 0)
    a.mu = ctx->d_mu ? layer_mu(ctx, layer) : nullptr;
    a.rotation = ctx->cfg.rotation;
    a.terms = ctx->cfg.query_terms;
    a.pool = static_cast<const uint8_t*>(kv_pool);
    a.block_table = block_table;
    a.seq_lens = seq_lens;
    a.sink_k = static_cast<const uint16_t*>(sink_k);
    a.sink_v = static_cast<const uint16_t*>(sink_v);
    a.tail_k = static_cast<const uint16_t*>(tail_k);
    a.tail_v = static_cast<const uint16_t*>(tail_v);
    a.out = out;
    a.parts = static_cast<float*>(scratch);
    // a bounded wait that runs out is recorded only if the context already
    // has its device error word (this path never creates it)
    a.err = ctx->d_err;
    a.qstride = bd::qpack_stride(ctx->cfg.num_q_heads);
    a.B = B;
    a.hq = ctx->cfg.num_q_heads;
    a.hkv = ctx->cfg.num_kv_heads;
    a.max_blocks = max_blocks;
    bd::decode_splits(B, a.hkv, max_blocks, &a.nsplit, &a.pages_per_split);
    a.counters = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(scratch) +
                                                       bd::decode_parts_bytes(B, a.hq, a.nsplit));
    a.tag = bd::next_decode_tag();
    a.pool_pages = ctx->cfg.pool_pages;
    a.format = ctx->cfg.format;
    a.centering = ctx->cfg.centering;
    a.p_mode = ctx->cfg.p_mode;
    a.p_c = ctx->cfg.p_c;
    a.tau = tau;
    a.gk = k_gscale;
    a.gv = v_gscale;
    return cuda_status(bd::launch_decode(a, s));
}

int bd_read_device_error(bd_ctx* ctx, void* stream, int* out) {
    if (!ctx || !out) return BD_ERR_INVALID_ARG;
    if (!ctx->d_err) {
        *out = BD_OK;
        return BD_OK;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return BD_ERR_CUDA;
    if (cudaMemcpy(&v, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return BD_ERR_CUDA;
    if (cudaMemset(ctx->d_err, 0, sizeof(int)) != cudaSuccess) return BD_ERR_CUDA;
    *out = v;
    return BD_OK;
}

int bd_copy_async(void* dst, const void* src, size_t bytes, void* stream) {
    if (bytes == 0) return BD_OK;
    if (!dst || !src) return BD_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) return BD_ERR_INVALID_ARG;
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst), s0 = reinterpret_cast<uintptr_t>(src);
    if (d0 < s0 + bytes && s0 < d0 + bytes) return BD_ERR_INVALID_ARG;   // overlapping ranges
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BD_ERR_CUDA;
    // first and last byte of each range: device memory of this device, or
    // pinned host memory the device reaches at the same address
    const void* ends[4] = {dst, static_cast<const uint8_t*>(dst) + bytes - 1, src,
                           static_cast<const uint8_t*>(src) + bytes - 1};
    for (const void* p : ends) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
            cudaGetLastError();   // an unknown pointer: clear the (non-sticky) error it left
            return BD_ERR_INVALID_ARG;
        }
        const bool on_dev = at.type == cudaMemoryTypeDevice && at.device == dev;
        const bool mapped_host = at.type == cudaMemoryTypeHost && at.devicePointer == p;
        if (!on_dev && !mapped_host) return BD_ERR_INVALID_ARG;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return BD_ERR_CUDA;
    return cuda_status(bd::launch_copy(dst, src, bytes, sms, static_cast<cudaStream_t>(stream)));
}

int bd_selftest_bounded_wait(bd_ctx* ctx, int timeout_us, void* stream) {
    if (!ctx || timeout_us < 1 || timeout_us > 2000000) return BD_ERR_INVALID_ARG;
    int st = ensure_device(ctx);
    if (st != BD_OK) return st;
    return cuda_status(
        bd::launch_bounded_wait_selftest(ctx->d_err, (uint64_t)timeout_us * 1000ull, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
