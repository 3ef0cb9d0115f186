/*
 * bd.h -- C ABI of the GB300 (sm_103a) NVFP4 KV-cache hot path:
 *   - the page-fill writer that quantizes freshly filled 128-token KV pages,
 *   - the two-term FP4 query quantizer,
 *   - paged single-token decode attention that reads the packed FP4 K/V.
 *
 * Method sources (cited by page title and section):
 *  [cfg]  BitDecoding-FP4 "evaluation/config.py": RECIPE (key smoothing,
 *         Hadamard rotation, adaptive {4,6} block-scale search, dual residual
 *         query quantization, underflow-aware probability scaling),
 *         recipe_additional_config, probability_environment, KV_MODES
 *         ("bitdecoding-nvfp4": 16-token BF16 sink, key_scale_geometry
 *         "local"; "bitdecoding-mxfp4": scale_mode "mxfp4_search"),
 *         PARITY_ENGINE_KWARGS (block_size 128).
 *  [ab]   kv-landlords "scripts/quant_ab.py": module docstring (each page is
 *         quantized once when it fills; the partial hot page stays BF16),
 *         mem_ratio (4-bit codes plus one 1-byte scale per 16 elements).
 *  [arch] "How openbitsys/bitdecoding-fp4 works": KV cache writer ->
 *         KV quantization ("quantizes pages"), decode interface -> paged
 *         attention kernel, hybrid cache.
 *
 * Conventions shared by every call:
 *  - Every call returns an int status (BD_OK or a negative BD_ERR_*); no C++
 *    exception crosses this boundary.  Argument errors in host-side values
 *    are detected before anything is launched and leave device memory
 *    untouched.  Device-resident indexes (block tables, destination pages,
 *    sequence lengths) are checked by the kernels themselves: an entry out of
 *    range is skipped, never dereferenced, and recorded in the device error
 *    word.
 *  - All tensors are caller-owned device memory unless a parameter says
 *    "host".  The library owns only the bd_ctx, its per-layer key-shift copy
 *    and its device error word.
 *  - Launch calls take a cudaStream_t as void*, are asynchronous and never
 *    synchronize.  Device-side failures (a bounded wait that ran out, an
 *    out-of-range device-resident index) are recorded in the context's device
 *    error word; read it with bd_read_device_error().
 *  - bf16 tensors are raw 16-bit bfloat16 bit patterns (const void*).
 *  - The first launch call on a device allocates the context's device state
 *    (key-shift table, error word) with cudaMalloc; make that first call, or
 *    bd_set_key_shift(), before capturing a stream into a CUDA graph.  A
 *    context then belongs to that device: a later call made while another
 *    device is current returns BD_ERR_INVALID_ARG (one context per device).
 *
 * ---------------------------------------------------------------------------
 * Byte layouts (both the CUDA path and the independent CPU oracle write these)
 * ---------------------------------------------------------------------------
 *  E2M1 code: bit 3 = sign, bits 2..0 index {0, .5, 1, 1.5, 2, 3, 4, 6}.
 *  NVFP4 block: 16 consecutive head-dim elements share one E4M3 (FN) scale
 *    byte; the tensor also has one fp32 per-tensor scale g (k_gscale /
 *    v_gscale, or the query's own g1/g2).  value = E2M1 * E4M3 * g.
 *  MXFP4 block: 32 consecutive head-dim elements share one UE8M0 byte
 *    (value 2^(byte-127)); no per-tensor scale.  value = E2M1 * 2^(byte-127).
 *
 *  KV pool of one layer: records ordered [physical page][kv head][K, V].
 *    record bytes R = 8192 + 128*nb, nb = 8 (NVFP4) or 4 (MXFP4):
 *    R = 9216 (NVFP4), 8704 (MXFP4).  bd_record_bytes() returns R.
 *    The K record (the layout the decode's block-scaled tensor-core MMA
 *    reads straight from shared memory):
 *      codes: 128 tokens x 128 dims in groups of 8 tokens x 32 dims, each
 *        group 128 contiguous bytes (16 per token): the byte of dims d, d+1
 *        (d even, d in the low nibble) of token t is at
 *        (t/8)*512 + (d/32)*128 + (t%8)*16 + (d%32)/2.  Elements are in the
 *        rotated, centered domain when rotation / centering are on.
 *      scales: nb/4 groups of 512 bytes (NVFP4 2, MXFP4 1), each 32 lines of
 *        16 bytes; line i holds tokens i, i+32, i+64, i+96, four blocks each:
 *        the byte of block b of token t is at
 *        8192 + (b/4)*512 + (t%32)*16 + (t/32)*4 + b%4.
 *    The V record pairs token tau = 16 i + 2 p with token tau + 1
 *    (16-token group i = 0..7, p = 0..7):
 *      codes [8 i][8 p][8 slots][16 B]: the byte of head dim d is
 *        code(tau, d) | code(tau + 1, d) << 4, at slot (d/16) XOR 2(p mod 4),
 *        byte d mod 16 of the slot.  (A byte is one f16x2 of the decode's
 *        P V operand; the XOR spreads its 16-byte reads over all
 *        shared-memory banks.)
 *      scales[8 i][8 p][nb][2]: scale bytes of block b, token tau first.
 *    FP4 page p of a sequence holds its tokens 16 + 128 p ... 16 + 128 p + 127
 *    (tokens 0..15 are the BF16 sink).
 *
 *  Packed query of one token (stride bd_query_packed_bytes(), a multiple of
 *  256): for Hq query heads and terms t = 0, 1:
 *      codes  at (t*Hq + j)*64                 [64 B] (same nibble order as K)
 *      scales at 2*Hq*64 + (t*Hq + j)*nb       [nb B]
 *      g      at 2*Hq*64 + 2*Hq*8              float[2] (g1, g2; MXFP4: 1, 1)
 *      q.mu   at 2*Hq*64 + 2*Hq*8 + 16         float[Hq] (unrotated bf16 q
 *                                              times the layer's key mean)
 *    all other bytes zero.  With query_terms = 1 the second term's codes and
 *    scales are zero and g2 = 0.
 */
#ifndef BD_H
#define BD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    BD_OK = 0,
    BD_ERR_INVALID_ARG = -1,  /* null pointer, size out of range, non-finite or out-of-range scalar */
    BD_ERR_UNSUPPORTED = -2,  /* a configuration this library does not implement */
    BD_ERR_CUDA = -3,         /* a CUDA runtime call failed */
    BD_ERR_WORKSPACE = -4,    /* the caller's workspace is smaller than required */
    BD_ERR_TIMEOUT = -5       /* a bounded device-side wait ran out (reported via the error word) */
};

enum { BD_FORMAT_NVFP4 = 0, BD_FORMAT_MXFP4 = 1 };

/* Probability quantization modes ([cfg] probability_environment):
 * BD_P_AMAX6 is the mode used when underflow-aware scaling is disabled;
 * BD_P_AMAX2_OR_AMAX6 is "amax2_or_amax6" (p_c = 1) or "..._c8" (p_c = 8);
 * BD_P_NONE keeps probabilities unquantized (ablation). */
enum { BD_P_NONE = 0, BD_P_AMAX6 = 1, BD_P_AMAX2_OR_AMAX6 = 2 };

typedef struct bd_config {
    int num_layers;    /* >= 1: number of key-shift tables held by the context */
    int num_q_heads;   /* must equal 4 * num_kv_heads (GQA group of 4) */
    int num_kv_heads;  /* 1..16 */
    int head_dim;      /* must be 128 */
    int page_size;     /* must be 128 ([cfg] PARITY_ENGINE_KWARGS block_size) */
    int sink_tokens;   /* must be 16 ([cfg] KV_MODES sink_tokens) */
    int format;        /* BD_FORMAT_NVFP4 or BD_FORMAT_MXFP4 */
    int key_search;    /* NVFP4 keys: 1 = adaptive {4,6} search ("four_six"), 0 = "amax6" */
    int rotation;      /* 1 = Hadamard rotation of K and Q along head_dim ("hadamard"), 0 = "none" */
    int centering;     /* 1 = key smoothing: subtract the static per-channel key mean */
    int query_terms;   /* 2 = dual residual query (Q ~ Q1 + Q2), 1 = single term */
    int p_mode;        /* BD_P_* */
    int p_c;           /* 1 or 8 ([cfg] probability_environment: "supports c=1 or c=8") */
    int pool_pages;    /* physical pages in each layer's pool, or 0 = not declared.  Kernels never
                          touch a pool page outside [0, pool_pages) (with 0: outside [0, 2^31)):
                          a block-table or destination entry there is skipped and
                          BD_ERR_INVALID_ARG is recorded in the device error word.  Negative
                          entries are always skipped this way. */
} bd_config;

typedef struct bd_ctx bd_ctx;

/* Validate cfg and create a context (host memory only; no CUDA call).
 * Returns BD_ERR_INVALID_ARG for null pointers or values out of range,
 * BD_ERR_UNSUPPORTED for head_dim / page_size / sink / GQA ratios this library
 * does not implement.  *out is set only on success. */
int bd_create(const bd_config* cfg, bd_ctx** out);

/* Free the context and its device state (safe on NULL). */
void bd_destroy(bd_ctx* ctx);

/* Static text for a status code. */
const char* bd_status_string(int status);

/* Copy one layer's static key mean mu [num_kv_heads][128] fp32 from HOST
 * memory into the context ([cfg] RECIPE key_smoothing; KEY_SHIFT_SIDECAR holds
 * these means).  The default mean of every layer is zero.  Synchronous: it
 * returns once the copy has landed in device memory, so every later launch
 * reads the new mean.  Do not call it while a launch that reads this layer's
 * mean may still be running. */
int bd_set_key_shift(bd_ctx* ctx, int layer, const float* mu_host);

/* Bytes of one pool record (9216 NVFP4, 8704 MXFP4); a layer's pool holds
 * pages * num_kv_heads * 2 records. */
size_t bd_record_bytes(const bd_ctx* ctx);

/* Bytes of one packed query token (a multiple of 256). */
size_t bd_query_packed_bytes(const bd_ctx* ctx);

/* Page-fill writer ([ab] freeze-at-fill; [arch] KV cache writer -> KV
 * quantization).  Quantizes n freshly filled pages of one layer, K and V in
 * one launch:
 *   k, v      : bf16 [n][128 tokens][num_kv_heads][128], device, read only.
 *   dst_pages : int32 [n], device: physical page of each input page in kv_pool.
 *               An entry outside [0, pool_pages) (negative, with pool_pages 0)
 *               is skipped and BD_ERR_INVALID_ARG is recorded in the device
 *               error word.
 *   K = rotate(bf16 - mu[layer]) (per config), then per 16-element block the
 *   {4,6} search (or amax6) with per-tensor scale k_gscale; NVFP4 V uses
 *   amax6 with v_gscale; MXFP4 uses the mxfp4 search for both and ignores the
 *   g scales.  The records of the given pages are overwritten; nothing else
 *   in kv_pool is touched.  g scales must be finite and in [1e-30, 1e30].
 *   n = 0 is a no-op.  Destination pages must be distinct. */
int bd_quantize_kv_pages(bd_ctx* ctx, int layer, const void* k, const void* v,
                         const int32_t* dst_pages, int n, float k_gscale, float v_gscale,
                         void* kv_pool, void* stream);

/* Two-term query quantization ([cfg] RECIPE dual_residual_query_quantization,
 * query scale mode "amax6"): per token, q -> rotate -> Q1 with g1 =
 * amax/2688 over the token's num_q_heads*128 values -> residual R = q_rot -
 * Q1hat -> Q2 with g2 = amax(R)/2688 (a zero amax gives g = 1).
 *   q        : bf16 [B][num_q_heads][128], device.
 *   q_packed : B * bd_query_packed_bytes() bytes, device, written entirely.
 *   B = 0 is a no-op. */
int bd_quantize_query(bd_ctx* ctx, int layer, const void* q, int B, void* q_packed, void* stream);

/* Append one decode-step token per sequence to the hybrid cache and pack the
 * FP4 page it completes ([arch] hybrid cache: BF16 sink and tail, frozen
 * FP4 pages; kv-landlords quant_ab.py freeze-at-fill).  One launch:
 *   k_new, v_new : bf16 [B][num_kv_heads][128], device: the new token.
 *   seq_lens     : int32 [B], device: each sequence's length L BEFORE this
 *                  token; the token takes position L.  Not modified: advance
 *                  it by one before the next decode reads the token.  A
 *                  negative L stores nothing and records BD_ERR_INVALID_ARG.
 *   sink_k/v     : bf16 [B][16][num_kv_heads][128], device, updated in place
 *                  (the token goes to row L when L < 16).
 *   tail_k/v     : bf16 [B][128][num_kv_heads][128], device, updated in place
 *                  (row (L-16) mod 128 otherwise).
 *   block_table  : int32 [B][max_blocks], device.  When the token completes
 *                  tail page p = (L-16) div 128 (its row is 127), the page's
 *                  128 tokens are quantized into pool page block_table[b][p]
 *                  exactly as bd_quantize_kv_pages would; a page whose slot
 *                  lies beyond max_blocks, or whose entry lies outside
 *                  [0, pool_pages), is skipped and BD_ERR_INVALID_ARG is
 *                  recorded in the device error word.
 *   k/v_gscale, kv_pool : as bd_quantize_kv_pages.
 * This kernel does not allow the next grid to launch early, so a following
 * decode sees the packed page and the new rows. */
int bd_append_kv(bd_ctx* ctx, int layer, const void* k_new, const void* v_new, const int32_t* seq_lens,
                 const int32_t* block_table, int max_blocks, void* sink_k, void* sink_v, void* tail_k,
                 void* tail_v, int B, float k_gscale, float v_gscale, void* kv_pool, void* stream);

/* Workspace bytes bd_decode_attention needs for B sequences whose block
 * table rows hold max_blocks entries (0 if B == 0): the split partials, one
 * 8-byte arrival counter per (sequence, kv head) and room for B packed
 * queries. */
size_t bd_decode_workspace_size(const bd_ctx* ctx, int B, int max_blocks);

/* Paged single-token decode attention over the hybrid cache ([arch] decode
 * interface -> paged attention kernel; [cfg] sink_tokens, block_size):
 *   q_packed    : from bd_quantize_query, device; or NULL (num_q_heads <= 32,
 *                 else BD_ERR_UNSUPPORTED): the call quantizes q itself into
 *                 the bytes bd_quantize_query would write -- inside the
 *                 decode kernel when its grid fits one wave of the GPU, else
 *                 with the query kernel into ws first -- and the output is
 *                 bit-identical to passing those bytes.
 *   q           : bf16 [B][num_q_heads][128], device (raw query, used by the
 *                 BF16 sink and tail tokens).
 *   kv_pool     : the layer's pool (layout above), device.
 *   block_table : int32 [B][max_blocks], device: physical page of each FP4
 *                 page of each sequence.  A page whose entry lies outside
 *                 [0, pool_pages) (negative, with pool_pages 0) is left out of
 *                 the attention, nothing is read for it, and BD_ERR_INVALID_ARG
 *                 is recorded in the device error word.
 *   seq_lens    : int32 [B], device: context length L of each sequence
 *                 (0 <= L <= 16 + 128*max_blocks + 127); L = 0 gives zeros.
 *                 A negative L is taken as 0 and a longer one keeps only its
 *                 first max_blocks FP4 pages (and its tail rows); both record
 *                 BD_ERR_INVALID_ARG in the device error word.
 *   sink_k/v    : bf16 [B][16][num_kv_heads][128]: tokens 0..min(L,16)-1.
 *   tail_k/v    : bf16 [B][128][num_kv_heads][128]: the partial page, tokens
 *                 16 + 128*npages ... L-1 in rows 0.., npages = max(0,L-16) div 128.
 *   tau         : probability threshold, finite, in [0, 448]
 *                 ([cfg] probability_environment).
 *   k/v_gscale  : the per-tensor scales the layer's pages were written with.
 *   out         : fp32 [B][num_q_heads][128], device.
 *   ws          : device scratch of at least bd_decode_workspace_size(ctx, B,
 *                 max_blocks) bytes for the split partials, the split
 *                 arrival counters and (q_packed NULL) the packed queries;
 *                 it needs no initialization (a counter
 *                 carries a per-call tag: bytes from earlier calls or never
 *                 written count as zero).  Calls that share a workspace must
 *                 not overlap on the GPU.
 * Query head j reads kv head j / 4; softmax scale 1/sqrt(128).
 * One decode kernel is launched on `stream` (preceded by the query kernel
 * in the one case above): each split holding pages (and the
 * split of the BF16 sink and tail) writes its partial to ws and counts
 * itself in at its (sequence, kv head)'s counter, and the split that
 * completes the count merges that group's partials into out.
 * Ordering: the kernel may start reading kv_pool, block_table and seq_lens
 * while the preceding grid in the stream, if it allows programmatic early
 * launch, still runs (this library's query and decode kernels do); those
 * inputs must be written by work that completes before that grid starts
 * (bd_quantize_kv_pages and bd_append_kv never allow early launch).  q_packed, q, the sink and
 * tail rows, out and ws are touched only after the preceding grid has
 * completed. */
int bd_decode_attention(bd_ctx* ctx, int layer, const void* q_packed, const void* q,
                        const void* kv_pool, const int32_t* block_table, int max_blocks,
                        const int32_t* seq_lens, const void* sink_k, const void* sink_v,
                        const void* tail_k, const void* tail_v, int B, float tau,
                        float k_gscale, float v_gscale, float* out, void* ws, size_t ws_bytes,
                        void* stream);

/* bd_decode_attention without a caller workspace and without any device
 * allocation.  No page of the method has a counterpart: this entry point
 * exists for callers that cannot call cudaMalloc -- code that runs inside
 * another framework's memory pool or allocator, a plugin that is handed only
 * its input and output buffers, or a process whose GPU memory is reserved up
 * front -- and so cannot provide the workspace bd_decode_attention needs.
 * Arguments are those of bd_decode_attention minus ws / ws_bytes; inputs and
 * out are still caller-owned device memory.
 *  - The split partials and arrival counters live in one fixed 4 MiB device
 *    array inside the library (every GPU that loads the library holds it
 *    until the process exits).  A call whose workspace would need more
 *    (bd_decode_workspace_size(ctx, B, max_blocks) > 4 MiB) is rejected with
 *    BD_ERR_WORKSPACE before anything is launched: use bd_decode_attention
 *    with a workspace instead.
 *  - Nothing in that array has to start at zero: each call writes every
 *    partial it reads, and its counters carry the call's own tag.  Every
 *    call shares the array, so calls that overlap on the GPU (other
 *    streams, other threads) race and must be serialized by the caller.
 *  - The first call on a device looks up the array's device address; make
 *    that first call before capturing a stream into a CUDA graph.
 *  - Like every launch call it must run on the context's device (the device
 *    of the context's first launch), else it returns BD_ERR_INVALID_ARG.
 *  - No cudaMalloc, cudaFree or allocating library routine is called.  A
 *    bounded device wait that runs out is recorded in the context's error
 *    word only if that word already exists (any other launch call or
 *    bd_set_key_shift creates it); this call never creates it. */
int bd_decode_attention_noalloc(bd_ctx* ctx, int layer, const void* q_packed, const void* q,
                                const void* kv_pool, const int32_t* block_table, int max_blocks,
                                const int32_t* seq_lens, const void* sink_k, const void* sink_v,
                                const void* tail_k, const void* tail_v, int B, float tau,
                                float k_gscale, float v_gscale, float* out, void* stream);

/* Synchronize `stream`, copy the context's device error word into *out
 * (BD_OK, BD_ERR_TIMEOUT or BD_ERR_INVALID_ARG: the first error a kernel
 * recorded since the last read) and reset it to BD_OK. */
int bd_read_device_error(bd_ctx* ctx, void* stream, int* out);

/* Copy `bytes` bytes from src to dst by a kernel on `stream` (asynchronous).
 * Each pointer is device memory of the current device or pinned host memory
 * mapped at the same address (cudaHostAlloc / cudaHostRegister on a system
 * with unified addressing); the kernel's loads and stores reach host memory
 * through the CPU-GPU link.  On a Grace-Blackwell node this moves a decode
 * step's queries in and its outputs out (a few hundred kilobytes) faster than
 * a DMA copy, whose start-up dominates at that size.
 *  - dst and src: 16-byte aligned; each range lies inside one allocation
 *    (the call checks its two ends, not what lies between); the two ranges
 *    must not overlap; any byte count (0 does nothing).
 *  - The first and last byte of both ranges are checked with
 *    cudaPointerGetAttributes before anything is launched: pageable host
 *    memory, another device's memory, a null, unaligned or overlapping
 *    range returns BD_ERR_INVALID_ARG and nothing is copied.
 *  - Host memory written by the copy is complete once the stream reaches
 *    the point after it (synchronize or wait on an event before reading).
 *  - The kernel is a programmatic dependent launch, like this library's
 *    other kernels: it lets the next kernel in the stream start early and
 *    waits for the preceding grid before it reads src.  A kernel launched
 *    after it with programmatic stream serialization must execute
 *    griddepcontrol.wait before reading dst (this library's kernels do);
 *    every other stream-ordered operation sees the copy complete. */
int bd_copy_async(void* dst, const void* src, size_t bytes, void* stream);

/* Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier phase nothing will complete, for at most timeout_us microseconds
 * (1..2000000), then records BD_ERR_TIMEOUT in the device error word and
 * returns.  Read the result with bd_read_device_error(). */
int bd_selftest_bounded_wait(bd_ctx* ctx, int timeout_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BD_H */
