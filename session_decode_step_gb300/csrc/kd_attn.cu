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
// in the batch.  A persistent CTA per SM walks its items through a ring of
// shared-memory stages: the split's K rows arrive by tensor-map copies with the
// 128-byte swizzle (conflict-free reads while q is broadcast), its V rows by a
// plain bulk copy.  Per item: the GQA group's scores, a local softmax (max m,
// sum l) and the weighted V sum, written as (o, m, l).  A second kernel merges
// a session-head's splits in split order (online-softmax combine).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int AT_THREADS = 256;  // 8 warps
constexpr int AT_WARPS = AT_THREADS / 32;
constexpr int AT_STAGES = 2;     // work items in flight per CTA (several CTAs per SM)
constexpr int AT_C = ATT_CHUNK;  // keys per work item (split)
static_assert(AT_C == 64, "the score pass maps 2 x 32 keys onto the 8 warps");

// Shared memory of one CTA.  A stage holds one work item: its K rows as 64-dim
// halves written by the tensor-map copy with the 128-byte swizzle (row r's
// 16-byte chunk c sits at chunk c ^ (r & 7)), then its V rows as written by a
// plain bulk copy ([key][head_dim] fp16).
template <int HD, int GQ>
struct AttnSmem {
    static constexpr int NREG = HD / 64;                   // 128-byte K halves per row
    static constexpr int KREG_BYTES = AT_C * 128;          // one half of the K tile
    static constexpr int K_BYTES = NREG * KREG_BYTES;
    static constexpr int V_BYTES = AT_C * HD * 2;
    static constexpr int STAGE = K_BYTES + V_BYTES;        // 1024-byte multiple
    static constexpr int Q_OFF = AT_STAGES * STAGE;        // q, double-buffered [2][GQ][HD]
    static constexpr int SP_OFF = Q_OFF + 2 * GQ * HD * 4; // score partials [4][C][GQ]
    static constexpr int SS_OFF = SP_OFF + 4 * AT_C * GQ * 4;  // probabilities [C][GQ]
    static constexpr int BAR_OFF = (SS_OFF + AT_C * GQ * 4 + 15) / 16 * 16;
    static constexpr int TOTAL = BAR_OFF + AT_STAGES * 8 + 1024;  // + alignment slack
    static_assert(STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
};

// Work items are ordered session-major, then split, then KV head.
__device__ __forceinline__ int attn_items(const AttnArgs& a) {
    int n = 0;
    for (int i = 0; i < a.B; ++i) n += (a.pos[i] + AT_C) / AT_C * a.nkv;
    return n;
}

struct AttnItem {
    int b, s, kvh, n, ns;  // session, split, KV head, keys in this split, splits of the session
};

__device__ __forceinline__ AttnItem attn_item(const AttnArgs& a, int item) {
    AttnItem it{0, 0, 0, 0, 0};
    int base = 0;
    for (int i = 0; i < a.B; ++i) {
        const int ns = (a.pos[i] + AT_C) / AT_C;  // ceil((pos+1)/C)
        const int cnt = ns * a.nkv;
        if (item < base + cnt) {
            const int r = item - base;
            it.b = i;
            it.s = r / a.nkv;
            it.kvh = r - it.s * a.nkv;
            it.n = min(AT_C, a.pos[i] + 1 - it.s * AT_C);
            it.ns = ns;
            return it;
        }
        base += cnt;
    }
    return it;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

template <int HD, int GQ>
__global__ void __launch_bounds__(AT_THREADS, GQ <= 4 ? 3 : 2)
    attn_split_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmk8) {
    using L = AttnSmem<HD, GQ>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base for the swizzled tiles
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    float* qsb = reinterpret_cast<float*>(smem + L::Q_OFF);  // [2][GQ][HD]
    float* sp = reinterpret_cast<float*>(smem + L::SP_OFF);  // [4][C][GQ]
    float* ss = reinterpret_cast<float*>(smem + L::SS_OFF);  // [C][GQ]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < AT_STAGES; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    __syncthreads();

    // Issue the copies of this CTA's j-th work item into stage j % AT_STAGES.
    auto issue = [&](const AttnItem& it, int j) {
        uint8_t* stg = smem + (j % AT_STAGES) * L::STAGE;
        const int t0 = it.s * AT_C;
        const long row = a.row0 + ((long)a.slot[it.b] * a.nkv + it.kvh) * a.cap + t0;
        const bool full = it.n == AT_C;
        const int krows = full ? AT_C : (it.n + 7) / 8 * 8;
        const uint32_t bytes = (uint32_t)(L::NREG * krows * 128 + it.n * HD * 2);
        uint64_t* b = &bar[j % AT_STAGES];
        mbar_arrive_expect_tx(b, bytes);
        for (int r = 0; r < L::NREG; ++r) {
            uint8_t* kdst = stg + r * L::KREG_BYTES;
            if (full) {
                tma_load_2d(kdst, &tmk, r * 64, (int)row, b);
            } else {
                for (int k8 = 0; k8 < krows; k8 += 8) tma_load_2d(kdst + k8 * 128, &tmk8, r * 64, (int)(row + k8), b);
            }
        }
        bulk_g2s(stg + L::K_BYTES, a.vc + (row - a.row0) * HD, (uint32_t)(it.n * HD * 2), b);
    };

    // History rows (keys < pos) were written by earlier steps: the items that do
    // not hold this step's new row can be fetched before waiting on the QKV kernel.
    int n_items = attn_items(a);
    int issued = 0;
    if (tid == 0) {
        for (int j = 0; j < AT_STAGES; ++j) {
            const int item = blockIdx.x + j * gridDim.x;
            if (item >= n_items) break;
            const AttnItem it = attn_item(a, item);
            if (it.s == it.ns - 1) break;  // holds the new row: after the wait
            issue(it, j);
            issued = j + 1;
        }
    }
    pdl_wait();
    pdl_launch_dependents();
    if (tid == 0)
        for (int j = issued; j < AT_STAGES; ++j) {
            const int item = blockIdx.x + j * gridDim.x;
            if (item >= n_items) break;
            issue(attn_item(a, item), j);
        }
    constexpr int QN = GQ * HD;                                 // q floats per item
    constexpr int QPT = (QN + AT_THREADS - 1) / AT_THREADS;    // per thread (1..4)
    if ((int)blockIdx.x < n_items) {  // q of the first item
        const AttnItem it = attn_item(a, blockIdx.x);
        const float* qg = a.q + ((size_t)it.b * a.nh + (size_t)it.kvh * GQ) * HD;
#pragma unroll
        for (int i = 0; i < QPT; ++i)
            if (tid + i * AT_THREADS < QN) qsb[tid + i * AT_THREADS] = qg[tid + i * AT_THREADS];
    }

    constexpr int QCH = HD / 32;  // 16-byte K chunks per dim quarter
    // PV mapping: warp -> (head, dim range); lane -> 8 dims x keys of one residue class.
    constexpr int WPH = AT_WARPS / GQ;         // warps per head
    constexpr int DPW = HD / WPH;              // dims per warp
    constexpr int LPK = DPW / 8 < 1 ? 1 : DPW / 8;  // lanes per key
    constexpr int KGR = 32 / LPK;              // key residue classes per warp
    const int kh = warp & 1, qd = warp >> 1;
    const int pv_h = warp / WPH, pv_d0 = (warp % WPH) * DPW + (lane % LPK) * 8, pv_kr = lane / LPK;
    const bool pv_on = (lane % LPK) * 8 < DPW;

    for (int j = 0;; ++j) {
        const int item = blockIdx.x + j * gridDim.x;
        if (item >= n_items) break;
        const AttnItem it = attn_item(a, item);
        uint8_t* stg = smem + (j % AT_STAGES) * L::STAGE;
        const float* qs = qsb + (j & 1) * GQ * HD;
        const bool ok = __syncthreads_and(mbar_wait_bounded(&bar[j % AT_STAGES], (uint32_t)(j / AT_STAGES) & 1u)) != 0;
        if (!ok) {
            // Flag it, let every copy already issued (items j .. j+STAGES-1) land, leave.
            if (tid == 0) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                for (int t = j; t < j + AT_STAGES; ++t)
                    if (blockIdx.x + t * gridDim.x < n_items)
                        (void)mbar_wait_bounded(&bar[t % AT_STAGES], (uint32_t)(t / AT_STAGES) & 1u);
            }
            __syncthreads();
            break;
        }
        // ---- scores: warp (kh, qd) takes keys 32kh + lane over dim quarter qd;
        // q is read warp-uniformly (broadcast), K conflict-free through the swizzle.
        {
            const int k = 32 * kh + lane;
            float dot[GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) dot[h] = 0.0f;
#pragma unroll
            for (int jj = 0; jj < QCH; ++jj) {
                const int c = qd * QCH + jj;
                const uint8_t* kp = stg + (c >> 3) * L::KREG_BYTES + k * 128 + (((c & 7) ^ (k & 7)) << 4);
                const uint4 kv = lds_v4(kp);
                const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kv.x));
                const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kv.y));
                const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kv.z));
                const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kv.w));
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    const float4 qa = *reinterpret_cast<const float4*>(qs + h * HD + c * 8);
                    const float4 qb = *reinterpret_cast<const float4*>(qs + h * HD + c * 8 + 4);
                    float d = dot[h];
                    d = __fmaf_rn(qa.x, k01.x, d);
                    d = __fmaf_rn(qa.y, k01.y, d);
                    d = __fmaf_rn(qa.z, k23.x, d);
                    d = __fmaf_rn(qa.w, k23.y, d);
                    d = __fmaf_rn(qb.x, k45.x, d);
                    d = __fmaf_rn(qb.y, k45.y, d);
                    d = __fmaf_rn(qb.z, k67.x, d);
                    d = __fmaf_rn(qb.w, k67.y, d);
                    dot[h] = d;
                }
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) sp[(qd * AT_C + k) * GQ + h] = dot[h];
        }
        __syncthreads();
        // ---- softmax over the item's keys: warp h takes head h (quarters summed in order)
        float m_h = 0.0f, l_h = 0.0f;
        if (warp < GQ) {
            const int h = warp;
            float v[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int k = lane + 32 * u, i = k * GQ + h;
                const float sum = __fadd_rn(__fadd_rn(__fadd_rn(sp[i], sp[AT_C * GQ + i]), sp[2 * AT_C * GQ + i]),
                                            sp[3 * AT_C * GQ + i]);
                v[u] = k < it.n ? __fmul_rn(sum, a.scale) : -INFINITY;
            }
            float m = fmaxf(v[0], v[1]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, o));
            const float p0 = lane < it.n ? expf(__fsub_rn(v[0], m)) : 0.0f;
            const float p1 = lane + 32 < it.n ? expf(__fsub_rn(v[1], m)) : 0.0f;
            float l = __fadd_rn(p0, p1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l = __fadd_rn(l, __shfl_xor_sync(FULL_MASK, l, o));
            ss[lane * GQ + h] = p0;
            ss[(lane + 32) * GQ + h] = p1;
            m_h = m;
            l_h = l;
        }
        __syncthreads();
        // q of the next item: issue its loads now, land them after the PV loop.
        float qn[QPT];
        const int item_n = blockIdx.x + (j + 1) * gridDim.x;
        if (item_n < n_items) {
            const AttnItem nx = attn_item(a, item_n);
            const float* qg = a.q + ((size_t)nx.b * a.nh + (size_t)nx.kvh * GQ) * HD;
#pragma unroll
            for (int i = 0; i < QPT; ++i) qn[i] = tid + i * AT_THREADS < QN ? qg[tid + i * AT_THREADS] : 0.0f;
        }
        // ---- o = sum_k p_k V_k for head pv_h, dims pv_d0 .. +7, keys k = pv_kr (mod KGR)
        {
            float o[8];
#pragma unroll
            for (int d = 0; d < 8; ++d) o[d] = 0.0f;
            const __half* vs = reinterpret_cast<const __half*>(stg + L::K_BYTES);
            if (pv_on)
                for (int k = pv_kr; k < it.n; k += KGR) {
                    const uint4 vv = lds_v4(vs + k * HD + pv_d0);
                    const float pk = ss[k * GQ + pv_h];
                    const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
                    const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
                    const float2 v45 = __half22float2(*reinterpret_cast<const __half2*>(&vv.z));
                    const float2 v67 = __half22float2(*reinterpret_cast<const __half2*>(&vv.w));
                    o[0] = __fmaf_rn(pk, v01.x, o[0]);
                    o[1] = __fmaf_rn(pk, v01.y, o[1]);
                    o[2] = __fmaf_rn(pk, v23.x, o[2]);
                    o[3] = __fmaf_rn(pk, v23.y, o[3]);
                    o[4] = __fmaf_rn(pk, v45.x, o[4]);
                    o[5] = __fmaf_rn(pk, v45.y, o[5]);
                    o[6] = __fmaf_rn(pk, v67.x, o[6]);
                    o[7] = __fmaf_rn(pk, v67.y, o[7]);
                }
            // sum the key residue classes (lanes LPK, 2*LPK, ... apart), fixed tree
#pragma unroll
            for (int off = LPK; off < 32; off <<= 1)
#pragma unroll
                for (int d = 0; d < 8; ++d) o[d] = __fadd_rn(o[d], __shfl_xor_sync(FULL_MASK, o[d], off));
            float* dst = a.part + (((size_t)it.b * a.nh + it.kvh * GQ + pv_h) * a.max_splits + it.s) * ATT_REC(HD);
            if (pv_on && pv_kr == 0) {
                *reinterpret_cast<float4*>(dst + pv_d0) = make_float4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<float4*>(dst + pv_d0 + 4) = make_float4(o[4], o[5], o[6], o[7]);
            }
        }
        if (warp < GQ && lane == 0) {
            float* dst = a.part + (((size_t)it.b * a.nh + it.kvh * GQ + warp) * a.max_splits + it.s) * ATT_REC(HD);
            dst[HD] = m_h;
            dst[HD + 1] = l_h;
        }
        if (item_n < n_items) {
            float* qd_next = qsb + ((j + 1) & 1) * GQ * HD;
#pragma unroll
            for (int i = 0; i < QPT; ++i)
                if (tid + i * AT_THREADS < QN) qd_next[tid + i * AT_THREADS] = qn[i];
        }
        __syncthreads();  // the stage is consumed: refill it
        if (tid == 0) {
            const int nxt = blockIdx.x + (j + AT_STAGES) * gridDim.x;
            if (nxt < n_items) issue(attn_item(a, nxt), j + AT_STAGES);
        }
    }
}

// Merge a (session, head)'s splits in split order:
//   M = max_s m_s,  out = fp16( sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s ).
// The per-split (m, l) pairs are staged in shared memory by parallel loads; the
// weights e^{m_s - M} are computed once; each thread then sums its dimension
// over the splits with independent loads.
constexpr int COMB_MAX_SPLITS = ATT_MAX_SPLITS;

template <int HD>
__global__ void __launch_bounds__(HD) attn_combine_kernel(const AttnArgs a) {
    __shared__ float wts[COMB_MAX_SPLITS];
    __shared__ float ls[COMB_MAX_SPLITS];
    __shared__ float red[HD / 32];
    __shared__ float Msh, Lsh;
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.y, h = blockIdx.x, d = threadIdx.x;
    if (b >= a.B) return;
    const int ns = (a.pos[b] + ATT_CHUNK) / ATT_CHUNK;
    const float* p = a.part + ((size_t)b * a.nh + h) * a.max_splits * ATT_REC(HD);
    float mloc = -INFINITY;
    for (int s = d; s < ns; s += HD) {
        const float2 ml = *reinterpret_cast<const float2*>(p + (size_t)s * ATT_REC(HD) + HD);
        wts[s] = ml.x;
        ls[s] = ml.y;
        mloc = fmaxf(mloc, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(FULL_MASK, mloc, o));
    if ((d & 31) == 0) red[d >> 5] = mloc;
    __syncthreads();
    if (d == 0) {
        float M = red[0];
        for (int w = 1; w < HD / 32; ++w) M = fmaxf(M, red[w]);
        Msh = M;
    }
    __syncthreads();
    const float M = Msh;
    for (int s = d; s < ns; s += HD) wts[s] = expf(__fsub_rn(wts[s], M));
    __syncthreads();
    if (d == 0) {
        float den = 0.0f;
        for (int s = 0; s < ns; ++s) den = __fmaf_rn(wts[s], ls[s], den);
        Lsh = den;
    }
    float num = 0.0f;
    int s = 0;
    for (; s + 4 <= ns; s += 4) {
        const float o0 = p[(size_t)(s + 0) * ATT_REC(HD) + d], o1 = p[(size_t)(s + 1) * ATT_REC(HD) + d];
        const float o2 = p[(size_t)(s + 2) * ATT_REC(HD) + d], o3 = p[(size_t)(s + 3) * ATT_REC(HD) + d];
        num = __fmaf_rn(wts[s + 0], o0, num);
        num = __fmaf_rn(wts[s + 1], o1, num);
        num = __fmaf_rn(wts[s + 2], o2, num);
        num = __fmaf_rn(wts[s + 3], o3, num);
    }
    for (; s < ns; ++s) num = __fmaf_rn(wts[s], p[(size_t)s * ATT_REC(HD) + d], num);
    __syncthreads();
    a.out[(size_t)b * a.nh * HD + (size_t)h * HD + d] = __float2half_rn(__fdiv_rn(num, Lsh));
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
#define KD_SET(HD_, GQ_)                                                                             \
    e = cudaFuncSetAttribute(attn_split_kernel<HD_, GQ_>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             AttnSmem<HD_, GQ_>::TOTAL);                                             \
    if (e != cudaSuccess) return e;                                                                  \
    e = cudaFuncSetAttribute(attn_split_kernel<HD_, GQ_>, cudaFuncAttributePreferredSharedMemoryCarveout, \
                             cudaSharedmemCarveoutMaxShared);                                        \
    if (e != cudaSuccess) return e;
    for (int group : {1, 2, 4, 8}) {
        KD_ATT_DISPATCH(64, KD_SET)
        KD_ATT_DISPATCH(128, KD_SET)
    }
#undef KD_SET
    for (const void* f : {(const void*)attn_combine_kernel<64>, (const void*)attn_combine_kernel<128>,
                          (const void*)kv_append_kernel})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return e;
    return cudaSuccess;
}

int attn_split_grid(int num_sms, int hd, int group) {
    // persistent: as many CTAs as fit on every SM at once
    int per_sm = 1;
    cudaError_t e = cudaSuccess;
#define KD_OCC(HD_, GQ_)                                                                     \
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_kernel<HD_, GQ_>, \
                                                      AT_THREADS, AttnSmem<HD_, GQ_>::TOTAL);
    auto run = [&]() -> cudaError_t {
        if (hd == 64) { KD_ATT_DISPATCH(64, KD_OCC) } else { KD_ATT_DISPATCH(128, KD_OCC) }
        return e;
    };
#undef KD_OCC
    if (run() != cudaSuccess || per_sm < 1) per_sm = 1;
    return num_sms * per_sm;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link to libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t make_attn_maps(const __half* k_arena, long rows, int hd, AttnMaps* out) {
    static EncodeTiledFn encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (rows < 1 || rows > 0x7fffffffL || (hd != 64 && hd != 128)) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)hd, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)hd * 2};
    const cuuint32_t estr[2] = {1, 1};
    const cuuint32_t box_full[2] = {64, (cuuint32_t)ATT_CHUNK};
    const cuuint32_t box_tail[2] = {64, 8};
    void* base = const_cast<__half*>(k_arena);
    CUresult r = encode(&out->k, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box_full, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    r = encode(&out->k8, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides, box_tail, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

static cudaError_t launch_cfg(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, bool pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaSuccess;
}

cudaError_t launch_attn_split(const AttnArgs& a, const AttnMaps& maps, int grid, bool pdl, cudaStream_t s) {
    const int group = a.nh / a.nkv;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    launch_cfg(cfg, attr, pdl);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(AT_THREADS);
    cfg.stream = s;
#define KD_LAUNCH(HD_, GQ_)                               \
    cfg.dynamicSmemBytes = AttnSmem<HD_, GQ_>::TOTAL;     \
    return cudaLaunchKernelEx(&cfg, attn_split_kernel<HD_, GQ_>, a, maps.k, maps.k8);
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
