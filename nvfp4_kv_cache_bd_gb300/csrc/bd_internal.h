// Internal declarations shared by the host API and the kernel launchers.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/bd.h"

namespace bd {

constexpr int kD = 128;          // head_dim
constexpr int kPage = 128;       // tokens per FP4 page
constexpr int kSink = 16;        // BF16 sink tokens
constexpr int kGroup = 4;        // query heads per kv head
constexpr int kCodeBytes = 8192; // codes of one record
constexpr int kPartStride = 132; // floats per split partial: m, l, pad, pad, O[128]
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // bounded waits give up after 1 s
constexpr int kMaxDevices = 64;  // per-device host caches (attributes, SM counts, scratch addresses)

__host__ __device__ inline int nblocks(int format) { return format == BD_FORMAT_NVFP4 ? 8 : 4; }
__host__ __device__ inline int record_bytes(int format) { return kCodeBytes + kPage * nblocks(format); }
inline size_t qpack_stride(int hq) { return ((size_t)hq * (2 * 64 + 2 * 8 + 4) + 16 + 255) / 256 * 256; }

struct WriterArgs {
    const uint16_t* k;
    const uint16_t* v;
    const int32_t* dst_pages;
    const float* mu;          // [Hkv][128] of this layer (device)
    uint8_t* pool;
    int n, hkv, format, key_search, rotation, centering;
    int pool_pages;           // 0: only negative destination pages are rejected
    float gk, gv;
    // -0.0f, read by the kernel at run time: the addend of the fma that forms
    // a product which is summed later, so that the compiler cannot see the
    // addend is zero and fold the product into the sum (x*y + -0 = RN(x*y)).
    float zero_addend = -0.0f;
    // Append mode (bd_append_kv) when seq_lens is set: n = B sequences, k/v
    // are the BF16 tail buffers [B][128][Hkv][128]; the new token is stored
    // at position seq_lens[b] and the tail page it completes is packed into
    // block_table[b][(L - 16) / 128].
    const int32_t* seq_lens = nullptr;
    const int32_t* block_table = nullptr;
    int max_blocks = 0;
    const uint16_t* k_new = nullptr;   // [B][Hkv][128]
    const uint16_t* v_new = nullptr;
    uint16_t* sink_k = nullptr;        // [B][16][Hkv][128]
    uint16_t* sink_v = nullptr;
    uint16_t* tail_k = nullptr;        // [B][128][Hkv][128] (the same buffers as k, v)
    uint16_t* tail_v = nullptr;
    int* err = nullptr;
};

struct QueryArgs {
    const uint16_t* q;
    const float* mu;          // [Hkv][128] of this layer (device)
    uint8_t* qp;
    int B, hq, format, rotation, centering, terms;
    size_t stride;
    float zero_addend = -0.0f;   // as in WriterArgs
};

struct DecodeArgs {
    const uint8_t* qp;        // packed query; nullptr: the decode quantizes q itself
    const uint16_t* q;
    const float* mu;          // the layer's key mean [Hkv][128] (fused query quantization)
    int rotation, terms;      // query recipe (fused query quantization)
    const uint8_t* pool;
    const int32_t* block_table;
    const int32_t* seq_lens;
    const uint16_t* sink_k;
    const uint16_t* sink_v;
    const uint16_t* tail_k;
    const uint16_t* tail_v;
    float* out;
    float* parts;             // [B][Hq][nsplit + 1][kPartStride]
    unsigned long long* counters;   // [B][Hkv] split arrival counters (tag << 24 | count)
    unsigned long long tag;   // this call's 40-bit counter tag (never 0)
    int* err;
    size_t qstride;
    int B, hq, hkv, max_blocks, nsplit, pages_per_split;
    int pool_pages;           // 0: only negative block-table entries are rejected
    int format, centering, p_mode, p_c;
    float tau, gk, gv;
    float zero_addend = -0.0f;   // as in WriterArgs (fused query quantization)
};

cudaError_t launch_writer(const WriterArgs& a, cudaStream_t s);
cudaError_t launch_query(const QueryArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_bounded_wait_selftest(int* err, uint64_t limit_ns, cudaStream_t s);
void decode_splits(int B, int hkv, int max_blocks, int* nsplit, int* pages_per_split);
size_t decode_ws_bytes(int B, int hq, int hkv, int nsplit);
size_t decode_parts_bytes(int B, int hq, int nsplit);
unsigned long long next_decode_tag();

// Fixed device scratch of bd_decode_attention_noalloc (see bd_decode.cu).
constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;
cudaError_t noalloc_scratch(void** out);

// A pool page index the kernels may dereference: in [0, pool_pages), or any
// non-negative int when the pool size is not declared.
__host__ __device__ inline bool page_ok(int64_t phys, int pool_pages) {
    return phys >= 0 && (pool_pages <= 0 || phys < pool_pages);
}

}  // namespace bd
