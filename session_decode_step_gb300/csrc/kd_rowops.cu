// kd_rowops.cu -- the row-parallel operations of the decode step: embedding
// gather, RMSNorm (fp32 in, fp16 out) and the greedy argmax.
//
// memra-engine decode_batch.rs: "Row-parallel ops (norm/rope/quantize/activation)
// batch trivially -- they are the SAME kernels prefill already runs at T rows";
// one CTA per row, so row b's bytes never depend on B.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

// x[b][i] = q * d of the token's canonical Q8_0 row (exact in fp32).
__global__ void embed_kernel(const uint8_t* __restrict__ emb, const int* __restrict__ token, int H,
                             float* __restrict__ x) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const uint8_t* row = emb + (size_t)token[b] * (H / 32) * 34;
    for (int i = threadIdx.x; i < H; i += blockDim.x) {
        const uint8_t* blk = row + (i >> 5) * 34;
        const __half_raw hr{(unsigned short)(blk[0] | (blk[1] << 8))};
        const float d = __half2float(__half(hr));
        const float q = (float)(int8_t)blk[2 + (i & 31)];
        x[(size_t)b * H + i] = __fmul_rn(q, d);
    }
}

constexpr int NORM_THREADS = 256;

// out = fp16(x * (1 / sqrt(mean(x^2) + eps)) * w), sum of squares in a fixed order:
// per-thread strided partials, a fixed shuffle tree, then warps in order.
__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_kernel(const float* __restrict__ x,
                                                               const float* __restrict__ w,
                                                               __half* __restrict__ out, int H,
                                                               float eps) {
    __shared__ float wsum[NORM_THREADS / 32];
    __shared__ float rs;
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x;
    const float4* xr = reinterpret_cast<const float4*>(x + (size_t)b * H);
    float ss = 0.0f;
    for (int i = tid; i < H / 4; i += NORM_THREADS) {
        const float4 v = xr[i];
        ss = __fmaf_rn(v.x, v.x, ss);
        ss = __fmaf_rn(v.y, v.y, ss);
        ss = __fmaf_rn(v.z, v.z, ss);
        ss = __fmaf_rn(v.w, v.w, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(FULL_MASK, ss, o));
    if ((tid & 31) == 0) wsum[tid >> 5] = ss;
    __syncthreads();
    if (tid == 0) {
        float t = wsum[0];
        for (int i = 1; i < NORM_THREADS / 32; ++i) t = __fadd_rn(t, wsum[i]);
        rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)H), eps)));
    }
    __syncthreads();
    const float r = rs;
    const float4* wr = reinterpret_cast<const float4*>(w);
    __half2* o2 = reinterpret_cast<__half2*>(out + (size_t)b * H);
    for (int i = tid; i < H / 4; i += NORM_THREADS) {
        const float4 v = xr[i], g = wr[i];
        o2[2 * i] = __floats2half2_rn(__fmul_rn(__fmul_rn(v.x, r), g.x), __fmul_rn(__fmul_rn(v.y, r), g.y));
        o2[2 * i + 1] = __floats2half2_rn(__fmul_rn(__fmul_rn(v.z, r), g.z), __fmul_rn(__fmul_rn(v.w, r), g.w));
    }
}

constexpr int ARGMAX_THREADS = 1024;

// (value, index) order for the greedy pick: larger value wins, equal values go
// to the lower index, NaN never wins.
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    if (v != v) return false;
    if (bi < 0) return true;
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_kernel(const float* __restrict__ logits,
                                                                int V, int* __restrict__ out) {
    __shared__ float sv[ARGMAX_THREADS / 32];
    __shared__ int si[ARGMAX_THREADS / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x;
    const float* row = logits + (size_t)b * V;
    float bv = 0.0f;
    int bi = -1;
    for (int i = tid; i < V; i += ARGMAX_THREADS) {
        const float v = row[i];
        if (better(v, i, bv, bi)) { bv = v; bi = i; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(FULL_MASK, bv, o);
        const int oi = __shfl_xor_sync(FULL_MASK, bi, o);
        if (oi >= 0 && better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if ((tid & 31) == 0) { sv[tid >> 5] = bv; si[tid >> 5] = bi; }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < ARGMAX_THREADS / 32; ++w)
            if (si[w] >= 0 && better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
        out[b] = bi;
    }
}

static void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, bool pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
}

cudaError_t launch_embed(const uint8_t* tok_embd, const int* token, int B, int H, float* x, bool pdl,
                         cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, embed_kernel, tok_embd, token, H, x);
}

cudaError_t launch_rmsnorm(const float* x, const float* w, __half* out, int B, int H, float eps,
                           bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(NORM_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, x, w, out, H, eps);
}

cudaError_t launch_argmax(const float* logits, int B, int V, int* out, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(ARGMAX_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, argmax_kernel, logits, V, out);
}

}  // namespace kd
