// Two-term FP4 query quantization.
//
// Method: BitDecoding-FP4 evaluation config (config.py) RECIPE
// dual_residual_query_quantization with nvfp4_query_terms = 2, query scale
// mode "amax6", Hadamard rotation (nvfp4_rotation); MXFP4 queries use the
// "mxfp4_search" rule.  Per token: q -> rotate -> Q1 (per-tensor scale
// g1 = amax/2688 over the token's Hq*128 values) -> R = q_rot - Q1hat -> Q2
// (g2 = amax(R)/2688); a zero amax gives g = 1.  Also stores q.mu (unrotated
// bf16 q times the layer's key mean, fp32) so the decode can restore the key
// mean's contribution to the FP4 logits.
//
// The quantization itself lives in bd_query.cuh (the decode kernel's fused
// path runs the same code).
#include "bd_query.cuh"

namespace bd {
namespace {

// One CTA per token, one thread per (query head j, 16-dim chunk c).
__global__ void __launch_bounds__(512) query_kernel(const QueryArgs a) {
    __shared__ float red[16];
    const int b = blockIdx.x;
    // Programmatic dependent launch: let the dependent decode launch at once
    // (it streams the layer's static FP4 pages and waits for this grid before
    // it reads the packed query), then wait for the grid that precedes us in
    // the stream, whose outputs may feed q.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    qquant::quantize_token<1>(a, a.q + (size_t)b * a.hq * kD, a.mu, a.qp + (size_t)b * a.stride, (int)threadIdx.x,
                              (int)blockDim.x, red, [] { __syncthreads(); });
}

}  // namespace

cudaError_t launch_query(const QueryArgs& a, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B);
    cfg.blockDim = dim3((unsigned)(a.hq * 8));
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, query_kernel, a);
}

}  // namespace bd
