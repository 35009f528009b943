// kd_mmvq.cu -- Q8_0 weight-only matrix x (m <= 16) activations, one numeric
// program for every m.
//
// This is the batched mmvq of memra-engine's decode_batch.rs (module header:
// every projection at m = B reads the weights once for all B rows; each row is
// "bit-identical per (token,row) to m=1").  The Q8_0 weights stream from HBM
// through a per-warp ring of shared-memory stages filled by 1-D bulk copies
// (TMA); each 16-row x 32-column Q8_0 block is converted to fp16 in registers
// (exact) and multiplied on the tensor cores by two m16n8k16 MMAs whose eight
// columns are eight sessions; the block's fp32 result is then scaled by its
// fp16 block scale and accumulated in fp32.  Sessions 8..15 use a second
// column tile with the same weight fragments.
//
// Why per-row exactness holds: a column of an MMA result depends only on that
// column's activations; tile shape, k-split, reduction order and epilogue are
// functions of the matrix shape alone, never of m; rows beyond m are zeros.
//
// K is split into S ranges (shape-dependent); each warp task writes its fp32
// partial for a row group, and the last of the S tasks to arrive (counted with
// one atomic per task, no waiting) adds the partials in split order 0..S-1 and
// runs the fused epilogue: plain store, residual add, SwiGLU, or RoPE + KV append.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int MMVQ_WARPS = 16;
constexpr int RING = 3;  // stages in flight per warp

size_t mmvq_smem_bytes() {
    return (size_t)MMVQ_WARPS * RING * STAGE_BYTES + (size_t)MMVQ_WARPS * RING * sizeof(uint64_t);
}

void choose_split(PackedQ8& m) {
    // Tasks of kpt k-groups; prefer enough tasks to fill a nominal 152-SM GPU with
    // 16 warps each several times over, evenly (the choice ignores m).
    const double warps = 152.0 * MMVQ_WARPS;
    int best = 1;
    double best_score = -1.0;
    for (int kpt = 1; kpt <= 8; ++kpt) {
        if (m.KG % kpt) continue;
        const double tasks = (double)m.G * (m.KG / kpt);
        const double rounds = tasks / warps;
        const double balance = rounds / std::ceil(rounds);           // last-round fill
        const double overhead = 1.0 / (1.0 + 0.5 / kpt);             // per-task cost
        const double score = balance * overhead;
        if (score > best_score + 1e-9) { best_score = score; best = kpt; }
    }
    m.kpt = best;
    m.S = m.KG / best;
}

// ---------------------------------------------------------------- repack ----
__global__ void repack_q8_0_kernel(const uint8_t* __restrict__ src, int K,
                                   const int* __restrict__ tile_src, int G,
                                   uint8_t* __restrict__ dst) {
    const int KG = K / KGROUP;
    const int nbk = K / 32;  // Q8_0 blocks per source row
    const size_t total = (size_t)G * KG * MT * 136;
    for (size_t idx = blockIdx.x * (size_t)blockDim.x + threadIdx.x; idx < total;
         idx += (size_t)gridDim.x * blockDim.x) {
        const int unit = (int)(idx % 136);
        size_t rest = idx / 136;
        const int mt = (int)(rest % MT);
        rest /= MT;
        const int kg = (int)(rest % KG);
        const int g = (int)(rest / KG);
        const int r0 = tile_src[g * MT + mt];
        uint8_t* out = dst + (((size_t)g * KG + kg) * MT + mt) * TILE_KG_BYTES;
        uint8_t v[16];
        if (unit < 128) {
            const int kb = unit >> 5, ln = unit & 31, gq = ln >> 2, cq = ln & 3;
            const int blk = kg * 4 + kb;
            for (int h = 0; h < 2; ++h) {
                const uint8_t* b = src + ((size_t)(r0 + gq + 8 * h) * nbk + blk) * 34 + 2 + 8 * cq;
                for (int j = 0; j < 8; ++j) v[8 * h + j] = (uint8_t)(b[j] ^ 0x80u);
            }
            out += kb * 512 + ln * 16;
        } else {
            const int gq = unit - 128;
            for (int kb = 0; kb < 4; ++kb) {
                const int blk = kg * 4 + kb;
                const uint8_t* b0 = src + ((size_t)(r0 + gq) * nbk + blk) * 34;
                const uint8_t* b1 = src + ((size_t)(r0 + gq + 8) * nbk + blk) * 34;
                v[4 * kb + 0] = b0[0];
                v[4 * kb + 1] = b0[1];
                v[4 * kb + 2] = b1[0];
                v[4 * kb + 3] = b1[1];
            }
            out += 2048 + gq * 16;
        }
        uint4 w;
        w.x = v[0] | (v[1] << 8) | (v[2] << 16) | ((uint32_t)v[3] << 24);
        w.y = v[4] | (v[5] << 8) | (v[6] << 16) | ((uint32_t)v[7] << 24);
        w.z = v[8] | (v[9] << 8) | (v[10] << 16) | ((uint32_t)v[11] << 24);
        w.w = v[12] | (v[13] << 8) | (v[14] << 16) | ((uint32_t)v[15] << 24);
        *reinterpret_cast<uint4*>(out) = w;
    }
}

cudaError_t launch_repack(const uint8_t* src, int K, const int* tile_src, int G, uint8_t* dst,
                          cudaStream_t s) {
    const size_t total = (size_t)G * (K / KGROUP) * MT * 136;
    const int threads = 256;
    const int blocks = (int)std::min<size_t>((total + threads - 1) / threads, 65535 * 4);
    repack_q8_0_kernel<<<blocks, threads, 0, s>>>(src, K, tile_src, G, dst);
    return cudaGetLastError();
}

// ------------------------------------------------------------ epilogues ----
// v[mt][nt][i]: fragment element i of tile mt, column tile nt:
//   row  = mt*16 + gq + (i >= 2 ? 8 : 0)   (within the group of 32 rows)
//   col  = nt*8 + 2*cq + (i & 1)           (the session index n)
template <int NT>
__device__ __forceinline__ void epilogue(const MmvqArgs& a, int epi, int g, int gq, int cq,
                                         float (&v)[MT][NT][4]) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = nt * 8 + 2 * cq + (i & 1);
            if (n >= a.B) continue;
            const int r = gq + ((i >> 1) << 3);  // row within a 16-row tile
            if (epi == EPI_STORE || epi == EPI_RESID) {
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    float* dst = a.y + (size_t)n * a.ld + (size_t)g * GROUP_ROWS + mt * TILE_ROWS + r;
                    *dst = (epi == EPI_STORE) ? v[mt][nt][i] : __fadd_rn(*dst, v[mt][nt][i]);
                }
            } else if (epi == EPI_SWIGLU) {
                const float gt = v[0][nt][i], up = v[1][nt][i];
                const float sg = __fdiv_rn(gt, __fadd_rn(1.0f, expf(-gt)));
                a.act[(size_t)n * a.ld + (size_t)g * TILE_ROWS + r] = __float2half_rn(__fmul_rn(sg, up));
            } else {  // EPI_QKV: tile 0 = dims [16j, 16j+16), tile 1 = the same + hd/2
                const int per_head = a.hd / GROUP_ROWS;
                const int head = g / per_head;
                const int dim = (g - head * per_head) * TILE_ROWS + r;
                const int half = a.hd >> 1;
                const float x0 = v[0][nt][i], x1 = v[1][nt][i];
                const int p = a.pos[n];
                if (head < a.nh + a.nkv) {
                    const float2 cs = a.rope[(size_t)p * half + dim];
                    const float y0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
                    const float y1 = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
                    if (head < a.nh) {
                        float* q = a.q_out + ((size_t)n * a.nh + head) * a.hd;
                        q[dim] = y0;
                        q[dim + half] = y1;
                    } else {
                        __half* k = a.kc + (((size_t)a.slot[n] * a.nkv + (head - a.nh)) * a.cap + p) * a.hd;
                        k[dim] = __float2half_rn(y0);
                        k[dim + half] = __float2half_rn(y1);
                    }
                } else {
                    __half* vv = a.vc + (((size_t)a.slot[n] * a.nkv + (head - a.nh - a.nkv)) * a.cap + p) * a.hd;
                    vv[dim] = __float2half_rn(x0);
                    vv[dim + half] = __float2half_rn(x1);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ mmvq ----
template <int NT, int EPI>
__global__ void __launch_bounds__(MMVQ_WARPS * 32, 1) mmvq_kernel(const MmvqArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    uint8_t* ring = smem + (size_t)warp * RING * STAGE_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + (size_t)MMVQ_WARPS * RING * STAGE_BYTES) + warp * RING;

    const int gw = blockIdx.x * MMVQ_WARPS + warp;
    const int nw = gridDim.x * MMVQ_WARPS;
    const int ntasks = a.G * a.S;
    const int my_tasks = gw < ntasks ? (ntasks - 1 - gw) / nw + 1 : 0;
    const int total = my_tasks * a.kpt;

    if (lane == 0) {
        for (int i = 0; i < RING; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    __syncwarp();

    // Stage sidx of this warp -> (group, split, k-group).  Tasks are split-major
    // (task = s * G + g) so warps running side by side share activation columns.
    auto stage_coords = [&](int sidx, int& g, int& s, int& kg) {
        const int ti = sidx / a.kpt, j = sidx - ti * a.kpt;
        const int task = gw + ti * nw;
        s = task / a.G;
        g = task - s * a.G;
        kg = s * a.kpt + j;
    };
    const uint64_t policy = l2_policy_evict_first();
    auto issue = [&](int sidx) {
        int g, s, kg;
        stage_coords(sidx, g, s, kg);
        const int slot = sidx % RING;
        mbar_arrive_expect_tx(&bar[slot], STAGE_BYTES);
        bulk_g2s_hint(ring + slot * STAGE_BYTES, a.w + ((size_t)g * a.KG + kg) * STAGE_BYTES,
                      STAGE_BYTES, &bar[slot], policy);
    };

    // The weights do not depend on earlier kernels: start streaming them before
    // waiting for the producer of the activations.
    if (lane == 0)
        for (int i = 0; i < RING && i < total; ++i) issue(i);
    pdl_wait();
    pdl_launch_dependents();

    // Activation fragments: lane (gq, cq) multiplies session n = gq + 8*nt at
    // columns 8cq .. 8cq+7 of each 32-column block (the k permutation the
    // packed weights use).  Sessions >= B read as zeros.
    const __half* xrow[NT];
    bool xok[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int n = gq + 8 * nt;
        xok[nt] = n < a.B;
        xrow[nt] = a.x + (size_t)(xok[nt] ? n : 0) * a.K + cq * 8;
    }
    auto load_x = [&](int sidx, uint4 (&xv)[4][NT]) {
        int g, s, kg;
        stage_coords(sidx, g, s, kg);
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                xv[kb][nt] = xok[nt] ? ldg_nc_v4(xrow[nt] + kg * KGROUP + kb * 32) : make_uint4(0, 0, 0, 0);
    };

    uint4 xcur[4][NT], xnext[4][NT];
    if (total > 0) load_x(0, xcur);

    float acc[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;

    for (int sidx = 0; sidx < total; ++sidx) {
        const int slot = sidx % RING;
        if (sidx + 1 < total) load_x(sidx + 1, xnext);

        const bool ok = mbar_wait_bounded(&bar[slot], (uint32_t)(sidx / RING) & 1u);
        if (__any_sync(FULL_MASK, !ok)) {
            // Give up: flag it, let every copy already issued land, and leave.
            if (lane == 0) atomicOr(a.err, ERR_WAIT_TIMEOUT);
            for (int t = sidx; t < total && t < sidx + RING; ++t)
                (void)mbar_wait_bounded(&bar[t % RING], (uint32_t)(t / RING) & 1u);
            return;
        }

        const uint8_t* st = ring + slot * STAGE_BYTES;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const uint8_t* tb = st + mt * TILE_KG_BYTES;
            const uint4 sc = lds_v4(tb + 2048 + gq * 16);
            const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                const uint4 wq = lds_v4(tb + kb * 512 + lane * 16);
                // k-half 0: columns 8cq+0..3; k-half 1: columns 8cq+4..7
                const uint32_t a00 = u8x2_lo_to_half2(wq.x), a01 = u8x2_lo_to_half2(wq.z);
                const uint32_t a02 = u8x2_hi_to_half2(wq.x), a03 = u8x2_hi_to_half2(wq.z);
                const uint32_t a10 = u8x2_lo_to_half2(wq.y), a11 = u8x2_lo_to_half2(wq.w);
                const uint32_t a12 = u8x2_hi_to_half2(wq.y), a13 = u8x2_hi_to_half2(wq.w);
                const float2 d = __half22float2(*reinterpret_cast<const __half2*>(&scw[kb]));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float t[4];
                    mma_16816_zero(t, a00, a01, a02, a03, xcur[kb][nt].x, xcur[kb][nt].y);
                    mma_16816_acc(t, a10, a11, a12, a13, xcur[kb][nt].z, xcur[kb][nt].w);
                    acc[mt][nt][0] = __fmaf_rn(d.x, t[0], acc[mt][nt][0]);
                    acc[mt][nt][1] = __fmaf_rn(d.x, t[1], acc[mt][nt][1]);
                    acc[mt][nt][2] = __fmaf_rn(d.y, t[2], acc[mt][nt][2]);
                    acc[mt][nt][3] = __fmaf_rn(d.y, t[3], acc[mt][nt][3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && sidx + RING < total) issue(sidx + RING);

#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) xcur[kb][nt] = xnext[kb][nt];

        const int ti = sidx / a.kpt;
        if (sidx - ti * a.kpt != a.kpt - 1) continue;  // task not finished yet

        // ---- task done: combine the split-K partials, then the epilogue ----
        int g, s, kg;
        stage_coords(sidx, g, s, kg);
        if (a.S == 1) {
            epilogue<NT>(a, EPI, g, gq, cq, acc);
        } else {
            float* pt = a.part + ((size_t)g * a.S + s) * (GROUP_ROWS * 16);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int r0 = mt * TILE_ROWS + gq, c0 = nt * 8 + 2 * cq;
                    *reinterpret_cast<float2*>(pt + r0 * 16 + c0) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
                    *reinterpret_cast<float2*>(pt + (r0 + 8) * 16 + c0) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
                }
            __threadfence();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = (atomicAdd(&a.cnt[g], 1) == a.S - 1);
            last = __shfl_sync(FULL_MASK, last, 0);
            if (last) {
                __threadfence();
                float v[MT][NT][4];
                const float* p0 = a.part + (size_t)g * a.S * (GROUP_ROWS * 16);
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int r0 = mt * TILE_ROWS + gq, c0 = nt * 8 + 2 * cq;
                        float2 lo = ldcg_f2(p0 + r0 * 16 + c0), hi = ldcg_f2(p0 + (r0 + 8) * 16 + c0);
                        for (int ss = 1; ss < a.S; ++ss) {
                            const float* ps = p0 + (size_t)ss * (GROUP_ROWS * 16);
                            const float2 l2 = ldcg_f2(ps + r0 * 16 + c0), h2 = ldcg_f2(ps + (r0 + 8) * 16 + c0);
                            lo.x = __fadd_rn(lo.x, l2.x);
                            lo.y = __fadd_rn(lo.y, l2.y);
                            hi.x = __fadd_rn(hi.x, h2.x);
                            hi.y = __fadd_rn(hi.y, h2.y);
                        }
                        v[mt][nt][0] = lo.x;
                        v[mt][nt][1] = lo.y;
                        v[mt][nt][2] = hi.x;
                        v[mt][nt][3] = hi.y;
                    }
                epilogue<NT>(a, EPI, g, gq, cq, v);
                if (lane == 0) a.cnt[g] = 0;  // ready for the next launch
            }
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;
    }
}

template <int NT, int EPI>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(mmvq_kernel<NT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)mmvq_smem_bytes());
}

cudaError_t mmvq_init_attributes() {
    cudaError_t e;
#define KD_ATTR(NT, EPI) \
    if ((e = set_attr<NT, EPI>()) != cudaSuccess) return e;
    KD_ATTR(1, EPI_STORE) KD_ATTR(2, EPI_STORE) KD_ATTR(1, EPI_RESID) KD_ATTR(2, EPI_RESID)
    KD_ATTR(1, EPI_SWIGLU) KD_ATTR(2, EPI_SWIGLU) KD_ATTR(1, EPI_QKV) KD_ATTR(2, EPI_QKV)
#undef KD_ATTR
    return cudaSuccess;
}

template <int NT, int EPI>
static cudaError_t launch_t(const MmvqArgs& a, int grid, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(MMVQ_WARPS * 32);
    cfg.dynamicSmemBytes = mmvq_smem_bytes();
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mmvq_kernel<NT, EPI>, a);
}

cudaError_t launch_mmvq(const MmvqArgs& a, int epi, int num_sms, bool pdl, cudaStream_t s) {
    const int ntasks = a.G * a.S;
    const int grid = std::max(1, std::min(num_sms, (ntasks + MMVQ_WARPS - 1) / MMVQ_WARPS));
    const bool wide = a.B > 8;
    switch (epi) {
        case EPI_STORE: return wide ? launch_t<2, EPI_STORE>(a, grid, pdl, s) : launch_t<1, EPI_STORE>(a, grid, pdl, s);
        case EPI_RESID: return wide ? launch_t<2, EPI_RESID>(a, grid, pdl, s) : launch_t<1, EPI_RESID>(a, grid, pdl, s);
        case EPI_SWIGLU: return wide ? launch_t<2, EPI_SWIGLU>(a, grid, pdl, s) : launch_t<1, EPI_SWIGLU>(a, grid, pdl, s);
        case EPI_QKV: return wide ? launch_t<2, EPI_QKV>(a, grid, pdl, s) : launch_t<1, EPI_QKV>(a, grid, pdl, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kd
