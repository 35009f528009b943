// kd_rowops.cu -- the row-parallel operations of the decode step: embedding
// gather (with the row's sum of squares for the first fused RMSNorm) and the
// greedy argmax.  RMSNorm itself is fused into the projections' activation load.
//
// memra-engine decode_batch.rs: "Row-parallel ops (norm/rope/quantize/activation)
// batch trivially -- they are the SAME kernels prefill already runs at T rows";
// one CTA per row, so row b's bytes never depend on B.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int EMBED_THREADS = 256;

// out[i] = fp16(x[i] / sqrt(mean(x^2) + eps) * w[i]) for the row x[0..H) already
// in global memory (written by this CTA); the sum of squares in a fixed order:
// per-thread strided, a fixed shuffle tree, then warps in order.
__device__ __forceinline__ void norm_row(const float* x, int H, const float* w, float eps, __half* out,
                                         float ss_thread) {
    __shared__ float wsum[EMBED_THREADS / 32];
    __shared__ float rsh;
    const int tid = threadIdx.x;
    float s = ss_thread;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
    if ((tid & 31) == 0) wsum[tid >> 5] = s;
    __syncthreads();
    if (tid == 0) {
        float t = wsum[0];
        for (int i = 1; i < EMBED_THREADS / 32; ++i) t = __fadd_rn(t, wsum[i]);
        rsh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)H), eps)));
    }
    __syncthreads();
    const float r = rsh;
    for (int i = tid; i < H; i += EMBED_THREADS) out[i] = __float2half_rn(__fmul_rn(__fmul_rn(x[i], r), w[i]));
}

// x[b][i] = q * d of the token's canonical Q8_0 row (exact in fp32), then the
// first layer's normed input xn[b] = fp16(rmsnorm(x[b]) * w).
__global__ void __launch_bounds__(EMBED_THREADS) embed_kernel(const uint8_t* __restrict__ emb,
                                                              const int* __restrict__ token, int H,
                                                              float* __restrict__ x, const float* __restrict__ w,
                                                              float eps, __half* __restrict__ xn) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x, tid = threadIdx.x;
    const uint8_t* row = emb + (size_t)token[b] * (H / 32) * 34;
    float* xr = x + (size_t)b * H;
    float s = 0.0f;
    for (int i = tid; i < H; i += EMBED_THREADS) {
        const uint8_t* blk = row + (i >> 5) * 34;
        const __half_raw hr{(unsigned short)(blk[0] | (blk[1] << 8))};
        const float d = __half2float(__half(hr));
        const float q = (float)(int8_t)blk[2 + (i & 31)];
        const float v = __fmul_rn(q, d);
        xr[i] = v;
        s = __fmaf_rn(v, v, s);
    }
    norm_row(xr, H, w, eps, xn + (size_t)b * H, s);  // each thread re-reads only what it wrote
}

// The same norm for residual rows supplied from outside.
__global__ void __launch_bounds__(EMBED_THREADS) row_norm_kernel(const float* __restrict__ x, int H,
                                                                 const float* __restrict__ w, float eps,
                                                                 __half* __restrict__ xn) {
    const int b = blockIdx.x, tid = threadIdx.x;
    const float* xr = x + (size_t)b * H;
    float s = 0.0f;
    for (int i = tid; i < H; i += EMBED_THREADS) s = __fmaf_rn(xr[i], xr[i], s);
    norm_row(xr, H, w, eps, xn + (size_t)b * H, s);
}

cudaError_t launch_row_norm(const float* x, int B, int H, const float* w, float eps, __half* xn, cudaStream_t s) {
    row_norm_kernel<<<B, EMBED_THREADS, 0, s>>>(x, H, w, eps, xn);
    return cudaGetLastError();
}

// RMSNorm of residual rows whose per-group sums of squares were left by the
// kernel that wrote them: r_b = 1 / sqrt(sum_g ssq[g][b] / H + eps) (groups in
// order: lane-strided, then a fixed shuffle tree), then elementwise
// xn = fp16(x * r_b * w).  Block (c, b) covers columns [1024c, 1024c + 1024) of row b.
constexpr int NORM_THREADS = 256;
constexpr int NORM_COLS = NORM_THREADS * 4;

__global__ void __launch_bounds__(NORM_THREADS) norm_from_ssq_kernel(const float* __restrict__ x,
                                                                     const float* __restrict__ ssq, int H,
                                                                     const float* __restrict__ w, float eps,
                                                                     __half* __restrict__ xn) {
    __shared__ float rsh;
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.y, tid = threadIdx.x;
    if (tid < 32) {
        float s = 0.0f;
        for (int g = tid; g < H / 32; g += 32) s = __fadd_rn(s, ssq[(size_t)g * MAX_NORM_SLOTS + b]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
        if (tid == 0) rsh = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)H), eps)));
    }
    const int i = blockIdx.x * NORM_COLS + tid * 4;
    const float4 v = i < H ? *reinterpret_cast<const float4*>(x + (size_t)b * H + i) : make_float4(0, 0, 0, 0);
    const float4 g = i < H ? *reinterpret_cast<const float4*>(w + i) : make_float4(0, 0, 0, 0);
    __syncthreads();
    if (i >= H) return;
    const float r = rsh;
    __half2* o = reinterpret_cast<__half2*>(xn + (size_t)b * H + i);
    o[0] = __floats2half2_rn(__fmul_rn(__fmul_rn(v.x, r), g.x), __fmul_rn(__fmul_rn(v.y, r), g.y));
    o[1] = __floats2half2_rn(__fmul_rn(__fmul_rn(v.z, r), g.z), __fmul_rn(__fmul_rn(v.w, r), g.w));
}

cudaError_t launch_norm_from_ssq(const float* x, const float* ssq, int B, int H, const float* w, float eps,
                                 __half* xn, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((H + NORM_COLS - 1) / NORM_COLS, B);
    cfg.blockDim = dim3(NORM_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, norm_from_ssq_kernel, x, ssq, H, w, eps, xn);
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

cudaError_t rowops_init_attributes() {
    // One shared-memory carveout for every kernel of the step, so consecutive
    // kernels never wait for an SM to reconfigure its L1/shared split.
    for (const void* f : {(const void*)embed_kernel, (const void*)row_norm_kernel, (const void*)norm_from_ssq_kernel,
                          (const void*)argmax_kernel}) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

static void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, bool pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
}

cudaError_t launch_embed(const uint8_t* tok_embd, const int* token, int B, int H, float* x, const float* w,
                         float eps, __half* xn, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(EMBED_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, embed_kernel, tok_embd, token, H, x, w, eps, xn);
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
