// kd_rowops.cu -- the row-parallel operations of the decode step: embedding
// gather with the first RMSNorm, the RMSNorm between a residual writer and the
// next projection, and the greedy argmax.
//
// memra-engine decode_batch.rs treats the row-parallel ops as the same kernels
// run at B rows; here every row's arithmetic is its own, so row b's bytes never
// depend on B.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int EMBED_THREADS = 1024;
constexpr int EMBED_U = 4;  // columns per thread and pass (4096 per pass)

// x[b] = q * d of the token's canonical Q8_0 row (exact in fp32), and the
// per-group sums of squares ssq[g][b] of the row, as a residual writer leaves
// them for the next RMSNorm.  With w: also the first RMSNorm of the row,
// xn[b] = fp16(x * r_b * w), r_b formed from those sums in the RMSNorm kernel's
// order and roundings (the same bits as the norm kernel run after this one).
// Block b covers row b.  The row's bytes are first copied to shared memory in
// 8-byte words (a row is 136 (H / 128) bytes, so 8-byte aligned); in pass p warp
// w then holds elements 4096p + 1024u + 32w + lane, i.e. group 128p + 32u + w
// with lane = row, added by the residual writers' shuffle tree.
__global__ void __launch_bounds__(EMBED_THREADS) embed_kernel(const uint8_t* __restrict__ emb,
                                                              const int* __restrict__ token, int H,
                                                              float* __restrict__ x, float* __restrict__ ssq,
                                                              const float* __restrict__ w, float eps,
                                                              __half* __restrict__ xn, unsigned long long* tl) {
    extern __shared__ uint2 rowsh[];  // [H / 32 * 34 / 8] the row's bytes, then [H / 32] the group sums
    __shared__ float rsh;
    tl_entry(tl);
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(tl);
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nw = H / 32 * 34 / 8;  // 8-byte words of the row
    float* gsq = reinterpret_cast<float*>(rowsh + nw);
    float* xr = x + (size_t)b * H;
    {
        const uint2* src = reinterpret_cast<const uint2*>(emb + (size_t)token[b] * (H / 32) * 34);
        for (int i = tid; i < nw; i += EMBED_THREADS) rowsh[i] = __ldcs(src + i);
    }
    float w0[EMBED_U];  // the first pass's norm weights, loaded while the row arrives
    if (w) {
#pragma unroll
        for (int u = 0; u < EMBED_U; ++u) {
            const int i = tid + EMBED_THREADS * u;
            w0[u] = i < H ? w[i] : 0.0f;
        }
    }
    __syncthreads();
    const uint8_t* row = reinterpret_cast<const uint8_t*>(rowsh);
    auto elem = [&](int i) {
        const uint8_t* blk = row + (i >> 5) * 34;
        const __half_raw hr{(unsigned short)(blk[0] | (blk[1] << 8))};
        return __fmul_rn((float)(int8_t)blk[2 + (i & 31)], __half2float(__half(hr)));
    };
    constexpr int PASS = EMBED_THREADS * EMBED_U;
    float v0[EMBED_U];  // the first pass, kept for the norm
    for (int p0 = 0; p0 < H; p0 += PASS) {
#pragma unroll
        for (int u = 0; u < EMBED_U; ++u) {
            const int i = p0 + tid + EMBED_THREADS * u;
            if (p0 + EMBED_THREADS * u + 32 * warp < H) {  // the warp's 32 elements: one whole group
                const float v = elem(i);
                if (p0 == 0) v0[u] = v;
                xr[i] = v;
                float s = __fmul_rn(v, v);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
                if (lane == 0) {
                    ssq[(size_t)(i >> 5) * MAX_NORM_SLOTS + b] = s;
                    gsq[i >> 5] = s;
                }
            } else if (p0 == 0) {
                v0[u] = 0.0f;
            }
        }
    }
    if (w) {
        __syncthreads();  // every group sum is in gsq
        if (warp == 0) {
            const float r = rms_factor_of([&](int g) { return gsq[g]; }, lane, H, eps);
            if (lane == 0) rsh = r;
        }
        __syncthreads();
        const float r = rsh;
        __half* o = xn + (size_t)b * H;
#pragma unroll
        for (int u = 0; u < EMBED_U; ++u) {
            const int i = tid + EMBED_THREADS * u;
            if (i < H) o[i] = __float2half_rn(__fmul_rn(__fmul_rn(v0[u], r), w0[u]));
        }
        for (int p0 = PASS; p0 < H; p0 += PASS)
#pragma unroll
            for (int u = 0; u < EMBED_U; ++u) {
                const int i = p0 + tid + EMBED_THREADS * u;
                if (i < H) o[i] = __float2half_rn(__fmul_rn(__fmul_rn(elem(i), r), w[i]));
            }
    }
    tl_exit(tl);
}

// Per-group sums of squares of residual rows supplied from outside, in the
// layout and order the residual writers' epilogues leave them: one warp per
// (32-row group g, row b), lane r holding x[b][32g + r]^2, added by a fixed
// shuffle tree.  The step's own RMSNorm kernel then forms the normed input
// from them (so a layer run alone goes through the same norm as in a step).
constexpr int SSQ_WARPS = 8;

__global__ void __launch_bounds__(SSQ_WARPS * 32) ssq_rows_kernel(const float* __restrict__ x, int H,
                                                                  float* __restrict__ ssq) {
    const int lane = threadIdx.x & 31;
    const int g = blockIdx.x * SSQ_WARPS + (threadIdx.x >> 5), b = blockIdx.y;
    if (g >= H / 32) return;
    const float v = x[(size_t)b * H + (size_t)g * 32 + lane];
    float s = __fmul_rn(v, v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
    if (lane == 0) ssq[(size_t)g * MAX_NORM_SLOTS + b] = s;
}

cudaError_t launch_ssq_rows(const float* x, int B, int H, float* ssq, cudaStream_t s) {
    ssq_rows_kernel<<<dim3((H / 32 + SSQ_WARPS - 1) / SSQ_WARPS, B), SSQ_WARPS * 32, 0, s>>>(x, H, ssq);
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
                                                                     __half* __restrict__ xn,
                                                                     unsigned long long* tl) {
    __shared__ float rsh;
    tl_entry(tl);
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(tl);
    const int b = blockIdx.y, tid = threadIdx.x;
    const int i = blockIdx.x * NORM_COLS + tid * 4;
    const float4 v = i < H ? *reinterpret_cast<const float4*>(x + (size_t)b * H + i) : make_float4(0, 0, 0, 0);
    const float4 g = i < H ? *reinterpret_cast<const float4*>(w + i) : make_float4(0, 0, 0, 0);
    if (tid < 32) {
        const float r = rms_factor_from_ssq(ssq, b, tid, H, eps);  // the shared order (kd_device.cuh)
        if (tid == 0) rsh = r;
    }
    __syncthreads();
    if (i < H) {
        const float r = rsh;
        __half2* o = reinterpret_cast<__half2*>(xn + (size_t)b * H + i);
        o[0] = __floats2half2_rn(__fmul_rn(__fmul_rn(v.x, r), g.x), __fmul_rn(__fmul_rn(v.y, r), g.y));
        o[1] = __floats2half2_rn(__fmul_rn(__fmul_rn(v.z, r), g.z), __fmul_rn(__fmul_rn(v.w, r), g.w));
    }
    tl_exit(tl);
}

cudaError_t launch_norm_from_ssq(const float* x, const float* ssq, int B, int H, const float* w, float eps,
                                 __half* xn, bool pdl, cudaStream_t s, unsigned long long* tl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((H + NORM_COLS - 1) / NORM_COLS, B);
    cfg.blockDim = dim3(NORM_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, norm_from_ssq_kernel, x, ssq, H, w, eps, xn, tl);
}

// Greedy argmax over many CTAs.  Each (value, index) maps to a 64-bit key whose
// unsigned order is the pick order -- larger value first, then lower index; -0
// counts as +0; NaN maps to 0 and never wins -- so every CTA can merge its best
// key into keys[b] with an atomic maximum, in any order, with one result.  The
// last CTA to finish turns keys into indices (-1 if nothing but NaN) and resets
// keys and the counter for the next launch.
constexpr int ARGMAX_THREADS = 256;
constexpr int ARGMAX_CHUNK = ARGMAX_THREADS * 8;  // logits per CTA: two float4 per thread

__global__ void __launch_bounds__(ARGMAX_THREADS) argmax_kernel(const float* __restrict__ logits, int V,
                                                                unsigned long long* keys, unsigned* done,
                                                                int* __restrict__ out, unsigned long long* tl,
                                                                const int* __restrict__ samp) {
    __shared__ unsigned long long wbest[ARGMAX_THREADS / 32];
    __shared__ bool last;
    tl_entry(tl);
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(tl);
    const int b = blockIdx.y, tid = threadIdx.x;
    const float* row = logits + (size_t)b * V;
    const int i0 = blockIdx.x * ARGMAX_CHUNK + tid * 4;
    float4 v[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int i = i0 + h * ARGMAX_THREADS * 4;
        v[h] = i < V ? __ldcg(reinterpret_cast<const float4*>(row + i)) : make_float4(NAN, NAN, NAN, NAN);
    }
    // Temperature sampling: the row's entries get their Gumbel perturbation
    // (entry v: word v mod 4 of the Philox block at counter (v / 4, counter, 0, 0)
    // under key (seed, 0)); the pick is then the same argmax.
    const PickParams pp = pick_params(samp, b);
    if (pp.T > 0.0f) {  // one Philox block serves the four entries of a float4
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = i0 + h * ARGMAX_THREADS * 4;
            if (i < V) {
                uint64_t w[4];
                philox4x64_10((uint64_t)(i >> 2), pp.ctr, 0, 0, pp.seed, 0, w);
                v[h].x = gumbel_perturb(v[h].x, pp.T, w[0]);
                v[h].y = gumbel_perturb(v[h].y, pp.T, w[1]);
                v[h].z = gumbel_perturb(v[h].z, pp.T, w[2]);
                v[h].w = gumbel_perturb(v[h].w, pp.T, w[3]);
            }
        }
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
    tl_exit(tl);
}

cudaError_t rowops_init_attributes() {
    // One shared-memory carveout for every kernel of the step, so consecutive
    // kernels never wait for an SM to reconfigure its L1/shared split.
    for (const void* f : {(const void*)embed_kernel, (const void*)ssq_rows_kernel, (const void*)norm_from_ssq_kernel,
                          (const void*)argmax_kernel}) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    // the embedding stages a whole row (and its group sums) in shared memory
    return cudaFuncSetAttribute(embed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
}

static void pdl_attr(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, bool pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
}

cudaError_t launch_embed(const uint8_t* tok_embd, const int* token, int B, int H, float* x, float* ssq,
                         const float* w, float eps, __half* xn, bool pdl, cudaStream_t s, unsigned long long* tl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(EMBED_THREADS);
    cfg.dynamicSmemBytes = (size_t)(H / 32) * 34 + (size_t)(H / 32) * sizeof(float);  // the row, its group sums
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, embed_kernel, tok_embd, token, H, x, ssq, w, eps, xn, tl);
}

cudaError_t launch_argmax(const float* logits, int B, int V, int* out, unsigned long long* keys, unsigned* done,
                          bool pdl, cudaStream_t s, unsigned long long* tl, const int* samp) {
    if (V % 4) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr, pdl);
    cfg.gridDim = dim3((V + ARGMAX_CHUNK - 1) / ARGMAX_CHUNK, B);
    cfg.blockDim = dim3(ARGMAX_THREADS);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, argmax_kernel, logits, V, keys, done, out, tl, samp);
}

}  // namespace kd
