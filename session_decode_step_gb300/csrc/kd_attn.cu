// kd_attn.cu -- ragged GQA split-K flash-decode over slot-indexed fp16 KV.
//
// Phase B of memra-engine decode_batch.rs `decode_batch_layers` ("phase B attends
// all B sequences (one blockIdx.z launch + one combine)") and hf2q ADR-040's
// batched flash-vec kernel (one dispatch for N queries, each with its own slot
// and kv_seq_len), for B sessions of unrelated lengths.
//
// Work item = (session b, KV head, split s): keys [s*C, min((s+1)*C, pos_b+1)),
// with C fixed, so the number of splits and every split's arithmetic depend on
// the session's own length only -- the result does not depend on what else is
// in the batch.  One CTA takes a work item at a time from a fixed-size grid:
// it bulk-copies the split's K rows and V rows (contiguous in the arena) into
// shared memory, computes the scores of the GQA group's query heads, a local
// softmax (max m, sum l) and the weighted V sum, and writes (o, m, l).  A second
// kernel merges a session-head's splits in split order (online-softmax combine).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int ATT_THREADS = 128;  // one key per thread in the score pass
constexpr int ATT_WARPS = ATT_THREADS / 32;
static_assert(ATT_CHUNK == ATT_THREADS, "score pass assumes one key per thread");

template <int HD, int GQ>
struct AttnSmem {
    static constexpr int KV_BYTES = ATT_CHUNK * HD * 2;              // one K or V tile
    static constexpr int RED_BYTES = ATT_WARPS * GQ * HD * 4;        // PV partials (alias K tile)
    static constexpr int Q_BYTES = GQ * HD * 4;
    static constexpr int P_BYTES = ATT_CHUNK * GQ * 4;
    static constexpr int STAT_BYTES = 2 * ATT_WARPS * GQ * 4 + 2 * GQ * 4;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + KV_BYTES;
    static constexpr int Q_OFF = V_OFF + KV_BYTES;
    static constexpr int P_OFF = Q_OFF + Q_BYTES;
    static constexpr int STAT_OFF = P_OFF + P_BYTES;
    static constexpr int BAR_OFF = (STAT_OFF + STAT_BYTES + 15) / 16 * 16;
    static constexpr int TOTAL = BAR_OFF + 16;
    static_assert(RED_BYTES <= KV_BYTES, "PV partials must fit in the K tile");
};

// Work-item decode: items are ordered session-major, then split, then KV head.
__device__ __forceinline__ bool attn_item(const AttnArgs& a, int item, int& b, int& s, int& kvh) {
    int base = 0;
    for (int i = 0; i < a.B; ++i) {
        const int ns = (a.pos[i] + ATT_CHUNK) / ATT_CHUNK;  // ceil((pos+1)/C)
        const int cnt = ns * a.nkv;
        if (item < base + cnt) {
            b = i;
            const int r = item - base;
            s = r / a.nkv;
            kvh = r - s * a.nkv;
            return true;
        }
        base += cnt;
    }
    return false;
}

__device__ __forceinline__ int attn_items(const AttnArgs& a) {
    int n = 0;
    for (int i = 0; i < a.B; ++i) n += (a.pos[i] + ATT_CHUNK) / ATT_CHUNK * a.nkv;
    return n;
}

template <int HD, int GQ>
__global__ void __launch_bounds__(ATT_THREADS) attn_split_kernel(const AttnArgs a) {
    using L = AttnSmem<HD, GQ>;
    extern __shared__ __align__(128) uint8_t smem[];
    __half* Ks = reinterpret_cast<__half*>(smem + L::K_OFF);
    __half* Vs = reinterpret_cast<__half*>(smem + L::V_OFF);
    float* red = reinterpret_cast<float*>(smem + L::K_OFF);   // aliases Ks after the score pass
    float4* qs = reinterpret_cast<float4*>(smem + L::Q_OFF);  // [GQ][2][HD/8] float4
    float* ps = reinterpret_cast<float*>(smem + L::P_OFF);    // [C][GQ]
    float* wstat = reinterpret_cast<float*>(smem + L::STAT_OFF);  // [2][WARPS][GQ]
    float* hstat = wstat + 2 * ATT_WARPS * GQ;                // [2][GQ]: m, l
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);  // [0]=K, [1]=V

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NCH = HD / 8;  // 16-byte chunks per row

    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();  // q and the appended KV rows come from the previous kernel
    pdl_launch_dependents();

    const int n_items = attn_items(a);
    uint32_t parity = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x, parity ^= 1u) {
        int b, s, kvh;
        attn_item(a, item, b, s, kvh);
        const int t_kv = a.pos[b] + 1;
        const int t0 = s * ATT_CHUNK;
        const int n = min(ATT_CHUNK, t_kv - t0);
        const size_t row0 = (((size_t)a.slot[b] * a.nkv + kvh) * a.cap + t0) * HD;

        if (tid == 0) {
            const uint32_t bytes = (uint32_t)n * HD * 2;
            mbar_arrive_expect_tx(&bar[0], bytes);
            bulk_g2s(Ks, a.kc + row0, bytes, &bar[0]);
            mbar_arrive_expect_tx(&bar[1], bytes);
            bulk_g2s(Vs, a.vc + row0, bytes, &bar[1]);
        }
        // q of the group's heads, split into chunk halves: qs[h][half][c] = q[h][8c + 4*half .. +3]
        const float* qg = a.q + ((size_t)b * a.nh + (size_t)kvh * GQ) * HD;
        for (int i = tid; i < GQ * HD / 4; i += ATT_THREADS) {
            const int h = i / (HD / 4), w = i - h * (HD / 4);  // float4 index within the head
            const int c = w >> 1, hf = w & 1;
            qs[(h * 2 + hf) * NCH + c] = *reinterpret_cast<const float4*>(qg + (size_t)h * HD + 4 * w);
        }
        __syncthreads();

        // every thread polls; the CTA agrees on one outcome
        const bool k_ok = __syncthreads_and(mbar_wait_bounded(&bar[0], parity)) != 0;
        // ---- scores: thread t owns key t; chunks visited in a rotated order so the
        // 8 lanes of a shared-memory phase touch 8 different banks groups.
        float sc[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) sc[h] = 0.0f;
        const int t = tid;
        if (k_ok && t < n) {
            const __half* krow = Ks + (size_t)t * HD;
#pragma unroll 4
            for (int cc = 0; cc < NCH; ++cc) {
                const int c = (cc + t) & (NCH - 1);
                const uint4 kv = lds_v4(krow + c * 8);
                const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kv.x));
                const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kv.y));
                const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kv.z));
                const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kv.w));
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    const float4 qa = qs[(h * 2 + 0) * NCH + c];
                    const float4 qb = qs[(h * 2 + 1) * NCH + c];
                    float d = sc[h];
                    d = __fmaf_rn(qa.x, k01.x, d);
                    d = __fmaf_rn(qa.y, k01.y, d);
                    d = __fmaf_rn(qa.z, k23.x, d);
                    d = __fmaf_rn(qa.w, k23.y, d);
                    d = __fmaf_rn(qb.x, k45.x, d);
                    d = __fmaf_rn(qb.y, k45.y, d);
                    d = __fmaf_rn(qb.z, k67.x, d);
                    d = __fmaf_rn(qb.w, k67.y, d);
                    sc[h] = d;
                }
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) sc[h] = __fmul_rn(sc[h], a.scale);
        } else {
#pragma unroll
            for (int h = 0; h < GQ; ++h) sc[h] = -INFINITY;
        }
        // ---- per-head max over the split, fixed reduction tree
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            float m = sc[h];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, o));
            if (lane == 0) wstat[warp * GQ + h] = m;
        }
        __syncthreads();
        if (tid < GQ) {
            float m = wstat[tid];
            for (int w = 1; w < ATT_WARPS; ++w) m = fmaxf(m, wstat[w * GQ + tid]);
            hstat[tid] = m;
        }
        __syncthreads();
        // ---- probabilities and their sum
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float p = (t < n) ? expf(__fsub_rn(sc[h], hstat[h])) : 0.0f;
            ps[t * GQ + h] = p;
            float l = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l = __fadd_rn(l, __shfl_xor_sync(FULL_MASK, l, o));
            if (lane == 0) wstat[ATT_WARPS * GQ + warp * GQ + h] = l;
        }
        __syncthreads();
        if (tid < GQ) {
            float l = wstat[ATT_WARPS * GQ + tid];
            for (int w = 1; w < ATT_WARPS; ++w) l = __fadd_rn(l, wstat[ATT_WARPS * GQ + w * GQ + tid]);
            hstat[GQ + tid] = l;
        }
        // ---- o = sum_t p_t V_t: warp w takes keys w, w+4, ...; lane owns HD/32 dims
        const bool v_ok = __syncthreads_and(mbar_wait_bounded(&bar[1], parity)) != 0;
        constexpr int DPL = HD / 32;  // dims per lane (2 or 4)
        float o[GQ][DPL];
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int j = 0; j < DPL; ++j) o[h][j] = 0.0f;
        if (v_ok) {
            for (int tk = warp; tk < n; tk += ATT_WARPS) {
                float vf[DPL];
                if constexpr (DPL == 4) {
                    const uint2 vv = *reinterpret_cast<const uint2*>(Vs + (size_t)tk * HD + lane * 4);
                    const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
                    const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
                    vf[0] = v01.x; vf[1] = v01.y; vf[2] = v23.x; vf[3] = v23.y;
                } else {
                    const uint32_t vv = *reinterpret_cast<const uint32_t*>(Vs + (size_t)tk * HD + lane * 2);
                    const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv));
                    vf[0] = v01.x; vf[1] = v01.y;
                }
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    const float p = ps[tk * GQ + h];
#pragma unroll
                    for (int j = 0; j < DPL; ++j) o[h][j] = __fmaf_rn(p, vf[j], o[h][j]);
                }
            }
        }
        if (!(k_ok && v_ok) && tid == 0) atomicOr(a.err, ERR_WAIT_TIMEOUT);
        __syncthreads();  // every thread is done with Ks before it becomes `red`
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int j = 0; j < DPL; ++j) red[(warp * GQ + h) * HD + lane * DPL + j] = o[h][j];
        __syncthreads();
        for (int i = tid; i < GQ * HD; i += ATT_THREADS) {
            const int h = i / HD, d = i - h * HD;
            float v = red[h * HD + d];
            for (int w = 1; w < ATT_WARPS; ++w) v = __fadd_rn(v, red[(w * GQ + h) * HD + d]);
            float* dst = a.part + (((size_t)b * a.nh + kvh * GQ + h) * a.max_splits + s) * (HD + 2);
            dst[d] = v;
            if (d == 0) {
                dst[HD] = hstat[h];
                dst[HD + 1] = hstat[GQ + h];
            }
        }
        // The next item's bulk copies overwrite Ks (written above as `red`): order
        // these generic-proxy accesses before them.
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (!(k_ok && v_ok)) {
            // Let any copy still in flight land before the CTA (and its smem) goes away.
            (void)mbar_wait_bounded(&bar[0], parity);
            (void)mbar_wait_bounded(&bar[1], parity);
            return;
        }
    }
}

// Merge a (session, head)'s splits in split order:
//   M = max_s m_s,  out = fp16( sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s ).
template <int HD>
__global__ void attn_combine_kernel(const AttnArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.y, h = blockIdx.x, d = threadIdx.x;
    if (b >= a.B) return;
    const int ns = (a.pos[b] + ATT_CHUNK) / ATT_CHUNK;
    const float* p = a.part + ((size_t)b * a.nh + h) * a.max_splits * (HD + 2);
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, p[(size_t)s * (HD + 2) + HD]);
    float num = 0.0f, den = 0.0f;
    for (int s = 0; s < ns; ++s) {
        const float* ps = p + (size_t)s * (HD + 2);
        const float w = expf(__fsub_rn(ps[HD], M));
        num = __fmaf_rn(w, ps[d], num);
        den = __fmaf_rn(w, ps[HD + 1], den);
    }
    a.out[(size_t)b * a.nh * HD + (size_t)h * HD + d] = __float2half_rn(__fdiv_rn(num, den));
}

// Standalone append (the op-level entry point; the step appends in the QKV epilogue).
__global__ void kv_append_kernel(const float* __restrict__ k, const float* __restrict__ v,
                                 __half* kc, __half* vc, const int* slot, const int* pos, int nkv,
                                 int hd, int cap) {
    const int b = blockIdx.y, h = blockIdx.x;
    const size_t dst = (((size_t)slot[b] * nkv + h) * cap + pos[b]) * hd;
    const size_t src = ((size_t)b * nkv + h) * hd;
    for (int i = threadIdx.x; i < hd; i += blockDim.x) {
        kc[dst + i] = __float2half_rn(k[src + i]);
        vc[dst + i] = __float2half_rn(v[src + i]);
    }
}

bool attn_supported(int hd, int group) {
    return (hd == 64 || hd == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

#define KD_ATT_DISPATCH(HD_, MACRO)                  \
    switch (group) {                                 \
        case 1: MACRO(HD_, 1); break;                \
        case 2: MACRO(HD_, 2); break;                \
        case 4: MACRO(HD_, 4); break;                \
        case 8: MACRO(HD_, 8); break;                \
        default: return cudaErrorInvalidValue;       \
    }

cudaError_t attn_init_attributes() {
    cudaError_t e = cudaSuccess;
#define KD_SET(HD_, GQ_)                                                                         \
    e = cudaFuncSetAttribute(attn_split_kernel<HD_, GQ_>,                                        \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem<HD_, GQ_>::TOTAL); \
    if (e != cudaSuccess) return e;
    for (int group : {1, 2, 4, 8}) {
        KD_ATT_DISPATCH(64, KD_SET)
        KD_ATT_DISPATCH(128, KD_SET)
    }
#undef KD_SET
    return cudaSuccess;
}

int attn_split_grid(int num_sms, int hd, int group) {
    int per_sm = 1;
    cudaError_t e = cudaSuccess;
#define KD_OCC(HD_, GQ_)                                                                       \
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<HD_, GQ_>,   \
                                                      ATT_THREADS, AttnSmem<HD_, GQ_>::TOTAL);
    auto run = [&]() -> cudaError_t {
        if (hd == 64) { KD_ATT_DISPATCH(64, KD_OCC) } else { KD_ATT_DISPATCH(128, KD_OCC) }
        return e;
    };
#undef KD_OCC
    if (run() != cudaSuccess || per_sm < 1) per_sm = 1;
    return num_sms * per_sm;
}

static cudaError_t launch_cfg(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, bool pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaSuccess;
}

cudaError_t launch_attn_split(const AttnArgs& a, int grid, bool pdl, cudaStream_t s) {
    const int group = a.nh / a.nkv;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    launch_cfg(cfg, attr, pdl);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(ATT_THREADS);
    cfg.stream = s;
#define KD_LAUNCH(HD_, GQ_)                                  \
    cfg.dynamicSmemBytes = AttnSmem<HD_, GQ_>::TOTAL;        \
    return cudaLaunchKernelEx(&cfg, attn_split_kernel<HD_, GQ_>, a);
    if (a.hd == 64) { KD_ATT_DISPATCH(64, KD_LAUNCH) } else if (a.hd == 128) { KD_ATT_DISPATCH(128, KD_LAUNCH) }
#undef KD_LAUNCH
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_combine(const AttnArgs& a, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    launch_cfg(cfg, attr, pdl);
    cfg.gridDim = dim3(a.nh, a.B);
    cfg.blockDim = dim3(a.hd);
    cfg.stream = s;
    if (a.hd == 64) return cudaLaunchKernelEx(&cfg, attn_combine_kernel<64>, a);
    if (a.hd == 128) return cudaLaunchKernelEx(&cfg, attn_combine_kernel<128>, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_kv_append(const float* k, const float* v, __half* kc, __half* vc, const int* slot,
                             const int* pos, int B, int nkv, int hd, int cap, cudaStream_t s) {
    kv_append_kernel<<<dim3(nkv, B), 128, 0, s>>>(k, v, kc, vc, slot, pos, nkv, hd, cap);
    return cudaGetLastError();
}

}  // namespace kd
