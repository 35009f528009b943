// kd_rowops.cu -- the row-parallel operations of the decode step: embedding
// gather with the first RMSNorm, the same norm for rows supplied from outside,
// and the greedy argmax.  (The norms inside the layer stack have no kernel of
// their own: NormLink splits them between the residual writer and the next
// projection.)
//
// memra-engine decode_batch.rs treats the row-parallel ops as the same kernels
// run at B rows; here every row's arithmetic is its own, so row b's bytes never
// depend on B.
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
    constexpr int U = 16;  // loads issued together
    for (int i0 = 0; i0 < H; i0 += EMBED_THREADS * U) {
        float xv[U], wv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + tid + EMBED_THREADS * u;
            xv[u] = i < H ? x[i] : 0.0f;
            wv[u] = i < H ? w[i] : 0.0f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + tid + EMBED_THREADS * u;
            if (i < H) out[i] = __float2half_rn(__fmul_rn(__fmul_rn(xv[u], r), wv[u]));
        }
    }
}

// Sum of squares of one 32-column group held one value per lane of a warp:
// a fixed shuffle tree; lane 0 writes it to both NormLink tables ([16][H/32]).
__device__ __forceinline__ void group_ssq(float v, int b, int gi, int ng, float* ssq0, float* ssq1) {
    float s = __fmul_rn(v, v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
    if ((threadIdx.x & 31) == 0 && gi < ng) {
        ssq0[(size_t)b * ng + gi] = s;
        ssq1[(size_t)b * ng + gi] = s;
    }
}

// x[b][i] = q * d of the token's canonical Q8_0 row (exact in fp32), then the
// first layer's normed input xn[b] = fp16(rmsnorm(x[b]) * w) and the per-group
// sums of squares of x[b] in both tables.  Element i = i0 + tid + 256u: for a
// fixed u each warp holds one whole 32-column group.
__global__ void __launch_bounds__(EMBED_THREADS) embed_kernel(const uint8_t* __restrict__ emb,
                                                              const int* __restrict__ token, int H,
                                                              float* __restrict__ x, const float* __restrict__ w,
                                                              float eps, __half* __restrict__ xn,
                                                              float* __restrict__ ssq0, float* __restrict__ ssq1,
                                                              int* __restrict__ zero, int n_zero) {
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    const int b = blockIdx.x, tid = threadIdx.x;
    for (int i = b * EMBED_THREADS + tid; i < n_zero; i += gridDim.x * EMBED_THREADS) zero[i] = 0;
    const uint8_t* row = emb + (size_t)token[b] * (H / 32) * 34;
    float* xr = x + (size_t)b * H;
    constexpr int U = 16;  // elements per thread whose loads are issued together
    float s = 0.0f;
    for (int i0 = 0; i0 < H; i0 += EMBED_THREADS * U) {
        int8_t q[U];
        unsigned short dbits[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + tid + EMBED_THREADS * u;
            const uint8_t* blk = row + (i >> 5) * 34;
            q[u] = i < H ? (int8_t)blk[2 + (i & 31)] : (int8_t)0;
            dbits[u] = i < H ? (unsigned short)(blk[0] | (blk[1] << 8)) : (unsigned short)0;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + tid + EMBED_THREADS * u;
            float v = 0.0f;
            if (i < H) {
                const __half_raw hr{dbits[u]};
                v = __fmul_rn((float)q[u], __half2float(__half(hr)));
                xr[i] = v;
                s = __fmaf_rn(v, v, s);
            }
            group_ssq(v, b, (i0 + EMBED_THREADS * u) / 32 + (tid >> 5), H / 32, ssq0, ssq1);
        }
    }
    norm_row(xr, H, w, eps, xn + (size_t)b * H, s);  // each thread re-reads only what it wrote
}

// The same norm and tables for residual rows supplied from outside.
__global__ void __launch_bounds__(EMBED_THREADS) row_norm_kernel(const float* __restrict__ x, int H,
                                                                 const float* __restrict__ w, float eps,
                                                                 __half* __restrict__ xn, float* __restrict__ ssq0,
                                                                 float* __restrict__ ssq1) {
    const int b = blockIdx.x, tid = threadIdx.x;
    const float* xr = x + (size_t)b * H;
    float s = 0.0f;
    for (int i0 = 0; i0 < H; i0 += EMBED_THREADS) {  // H is a multiple of 32: warps stay converged
        const int i = i0 + tid;
        const float v = i < H ? xr[i] : 0.0f;
        s = __fmaf_rn(v, v, s);
        group_ssq(v, b, i0 / 32 + (tid >> 5), H / 32, ssq0, ssq1);
    }
    norm_row(xr, H, w, eps, xn + (size_t)b * H, s);
}

cudaError_t launch_row_norm(const float* x, int B, int H, const float* w, float eps, __half* xn, float* ssq0,
                            float* ssq1, cudaStream_t s) {
    row_norm_kernel<<<B, EMBED_THREADS, 0, s>>>(x, H, w, eps, xn, ssq0, ssq1);
    return cudaGetLastError();
}

// Greedy argmax over many CTAs.  Each (value, index) maps to a 64-bit key whose
// unsigned order is the pick order -- larger value first, then lower index; -0
// counts as +0; NaN maps to 0 and never wins -- so every CTA can merge its best
// key into keys[b] with an atomic maximum, in any order, with one result.  The
// last CTA to finish turns keys into indices (-1 if nothing but NaN) and resets
// keys and the counter for the next launch.
constexpr int ARGMAX_THREADS = 256;
constexpr int ARGMAX_CHUNK = ARGMAX_THREADS * 8;  // logits per CTA: two float4 per thread

__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
    if (v != v) return 0ull;
    if (v == 0.0f) v = 0.0f;
    const unsigned u = __float_as_uint(v);
    const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(~(unsigned)i);
}

__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_kernel(const float* __restrict__ logits, int V,
                                                                unsigned long long* keys, unsigned* done,
                                                                int* __restrict__ out) {
    __shared__ unsigned long long wbest[ARGMAX_THREADS / 32];
    __shared__ bool last;
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    const int b = blockIdx.y, tid = threadIdx.x;
    const float* row = logits + (size_t)b * V;
    const int i0 = blockIdx.x * ARGMAX_CHUNK + tid * 4;
    float4 v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = i0 + h * ARGMAX_THREADS * 4;
        v[h] = i < V ? __ldcg(reinterpret_cast<const float4*>(row + i)) : make_float4(NAN, NAN, NAN, NAN);
    }
    unsigned long long best = 0ull;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = i0 + h * ARGMAX_THREADS * 4;
        best = max(best, argmax_key(v[h].x, i));
        best = max(best, argmax_key(v[h].y, i + 1));
        best = max(best, argmax_key(v[h].z, i + 2));
        best = max(best, argmax_key(v[h].w, i + 3));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(FULL_MASK, best, o));
    if ((tid & 31) == 0) wbest[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < ARGMAX_THREADS / 32; ++w) best = max(best, wbest[w]);
        if (best) atomicMax(&keys[b], best);
        __threadfence();
        last = atomicAdd(done, 1u) == gridDim.x * gridDim.y - 1;
    }
    __syncthreads();
    if (last && tid < (int)gridDim.y) {
        __threadfence();
        const unsigned long long k = atomicExch(&keys[tid], 0ull);
        out[tid] = k ? (int)(~(unsigned)(k & 0xffffffffull)) : -1;
        if (tid == 0) *done = 0u;
    }
}

cudaError_t rowops_init_attributes() {
    // One shared-memory carveout for every kernel of the step, so consecutive
    // kernels never wait for an SM to reconfigure its L1/shared split.
    for (const void* f : {(const void*)embed_kernel, (const void*)row_norm_kernel, (const void*)argmax_kernel}) {
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
                         float eps, __half* xn, float* ssq0, float* ssq1, int* zero, int n_zero, bool pdl,
                         cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(EMBED_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, embed_kernel, tok_embd, token, H, x, w, eps, xn, ssq0, ssq1, zero, n_zero);
}

cudaError_t launch_argmax(const float* logits, int B, int V, int* out, unsigned long long* keys, unsigned* done,
                          bool pdl, cudaStream_t s) {
    if (V % 4) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3((V + ARGMAX_CHUNK - 1) / ARGMAX_CHUNK, B);
    cfg.blockDim = dim3(ARGMAX_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, argmax_kernel, logits, V, keys, done, out);
}

}  // namespace kd
