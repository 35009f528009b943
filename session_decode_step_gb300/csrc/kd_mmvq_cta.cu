// kd_mmvq_cta.cu -- Q8_0 mmvq, "group" schedule: for matrices whose 32-row
// groups spread evenly over the SMs (q|k|v, o-proj, gate|up, down).
//
// CTA c owns row groups c, c + grid, ...; within a group its 8 warps split the
// K range into 8 contiguous k-group ranges (fixed by the shape), each streamed
// through the warp's own ring of shared-memory stages.  At the end of a group
// the warps' fp32 partials meet in shared memory and are added in warp order;
// no global partials, fences or atomics.  Nothing depends on m.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_mmvq_common.cuh"

namespace kd {

// PAIR: a launch of two CTAs per SM for G > SMs (B <= 8, where it gives no SM
// more groups than one CTA per SM would): one CTA per group up to 2 * SMs
// groups, else 2 * SMs CTAs taking groups c, c + grid, ...  A shallower ring
// lets two CTAs share an SM: twice the warps and more weight bytes in flight
// per SM for the stage pipeline, which (not HBM) bounds the one-CTA launch.
// NIN: the RMSNorm fused into the activation load (MmvqArgs::nx): each warp
// forms its whole k-range of normed tiles once, after the dependency wait, and
// keeps them for all its groups; the ring then carries weights only.
// Shared memory: per warp a ring of RD stages of weights, and its activation
// tiles (one per ring stage, or NIN: one per k-group of its range); then the
// barriers and the partial-sum buffer.
template <int NT, bool PAIR, bool NIN>
struct CtaSmem {
    static_assert(!(PAIR && NIN), "the fused norm's tiles do not fit two CTAs per SM");
    static constexpr int RD = PAIR || (NIN && NT == 2) ? 2 : 3;  // stages in flight per warp (measured best)
    static constexpr int RS = NT == 1 ? 9 : 16;  // partial-row stride (floats), padded against bank conflicts
    static constexpr int XT = NIN ? NORM_IN_MAX_KG : RD;  // activation tiles per warp
    static constexpr size_t X_BYTES = (size_t)MMVQ_WARPS * XT * NT * XTILE_BYTES;  // at a 1024-byte boundary
    static constexpr size_t W_OFF = X_BYTES;
    static constexpr size_t RING_BYTES = (size_t)MMVQ_WARPS * RD * STAGE_BYTES;
    static constexpr size_t BAR_OFF = W_OFF + RING_BYTES;
    static constexpr size_t RED_BYTES = (size_t)MMVQ_WARPS * GROUP_ROWS * RS * sizeof(float);
    static constexpr size_t RED_OFF = BAR_OFF + MMVQ_WARPS * RD * sizeof(uint64_t);
    static constexpr size_t TOTAL = RED_OFF + RED_BYTES + 1024;  // + alignment slack
    static_assert(!PAIR || 2 * (TOTAL + 1024) <= 228 * 1024, "two CTAs per SM");
};

template <int NT, int EPI, bool PAIR, bool NIN>
__global__ void __launch_bounds__(MMVQ_WARPS * 32, NT == 1 && !NIN ? 2 : 1)
    mmvq_cta_kernel(const MmvqArgs a, const __grid_constant__ CUtensorMap xm) {
    using L = CtaSmem<NT, PAIR, NIN>;
    constexpr int RD = L::RD;
    constexpr uint32_t SB = STAGE_BYTES + (NIN ? 0 : NT * XTILE_BYTES);  // bytes a stage's barrier waits for
    static_assert(!PAIR || NT == 1, "two CTAs per SM need the one-tile register budget");
    extern __shared__ uint8_t smem_raw[];
    tl_entry(a.tl);
    uint8_t* smem = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    uint8_t* xring = smem + (size_t)warp * L::XT * NT * XTILE_BYTES;
    uint8_t* ring = smem + L::W_OFF + (size_t)warp * RD * STAGE_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF) + warp * RD;
    float* red = reinterpret_cast<float*>(smem + L::RED_OFF);  // [warp][32 rows][RS]

    const int kg0 = warp * a.KG / MMVQ_WARPS, nk = (warp + 1) * a.KG / MMVQ_WARPS - kg0;
    const int ngrp = (int)blockIdx.x < a.G ? (a.G - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int total = ngrp * nk;

    if (lane == 0) {
        for (int i = 0; i < RD; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    __syncwarp();

    const uint64_t policy = l2_policy_evict_first();
    // Issue cursor: stage (group ii of this CTA, k-group kg0 + ikk).
    int ii = 0, ikk = 0;
    auto issue_w = [&](int slot_) {
        const int g = blockIdx.x + ii * gridDim.x;
        mbar_arrive_expect_tx(&bar[slot_], SB);
        bulk_g2s_hint(ring + slot_ * STAGE_BYTES, a.w + ((size_t)g * a.KG + kg0 + ikk) * STAGE_BYTES, STAGE_BYTES,
                      &bar[slot_], policy);
        if (++ikk == nk) { ikk = 0; ++ii; }
    };
    // The weights do not depend on earlier kernels: start streaming them before
    // waiting for the producer of the activations.  Each barrier expects the
    // stage's weights and activations; the activations follow after the wait.
    if (lane == 0) {
        if (a.inject_tx && blockIdx.x == 0 && total > 0) {  // debug fault hook: CTA 0's first warp with stages
            int fw = 0;
            while ((fw + 1) * a.KG / MMVQ_WARPS == fw * a.KG / MMVQ_WARPS) ++fw;
            if (warp == fw) mbar_expect_tx(&bar[0], (uint32_t)a.inject_tx);
        }
        for (int i = 0; i < RD && i < total; ++i) issue_w(i);
        prefetch_tmap(&xm);
    }
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(a.tl);
    if constexpr (NIN) {
        // the warp's normed k-range, once (the partial buffer holds the norm factors meanwhile)
        norm_tiles<NT>(a, warp, lane, kg0, ngrp > 0 ? nk : 0, xring, red);
        __syncthreads();  // red is the partial buffer again
    } else {
        if (lane == 0)
            for (int i = 0; i < RD && i < total; ++i)
                tma_x_tile<NT>(xring + i * NT * XTILE_BYTES, &xm, kg0 + i % nk, &bar[i]);
    }

    int sidx = 0, slot = 0;
    uint32_t phase = 0;
    bool failed = false;
    for (int gi = 0; gi < ngrp; ++gi) {
        const int g = blockIdx.x + gi * gridDim.x;
        // What the epilogue reads from global memory, loaded now so the group's end
        // does not wait for it: the residual rows (thread (warp, lane) takes session
        // warp + 8j, row lane) or the q|k|v epilogue's positions and cos/sin pairs.
        float xold[NT];
        QkvIn qin{};
        if constexpr (EPI == EPI_RESID) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int n = warp + MMVQ_WARPS * j;
                xold[j] = n < a.B ? resid_load(a, g, lane, n) : 0.0f;
            }
        } else if constexpr (EPI == EPI_QKV) {
            if (tid < a.B * TILE_ROWS) qin = qkv_load(a, g, tid & 15, tid >> 4);
        }
        float acc[MT][NT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;
        for (int kk = 0; kk < nk && !failed; ++kk, ++sidx) {
            const bool ok = mbar_wait_bounded(&bar[slot], phase);
            if (__any_sync(FULL_MASK, !ok)) {
                // Give up: flag it, let every copy already issued land, stop computing.
                if (lane == 0) atomicOr(a.err, ERR_WAIT_TIMEOUT);
                for (int t = sidx; t < total && t < sidx + RD; ++t)
                    (void)mbar_wait_bounded(&bar[t % RD], (uint32_t)(t / RD) & 1u);
                failed = true;
                break;
            }
            uint4 xv[4][NT];
            lds_x_tile<NT>(xring + (NIN ? kk : slot) * NT * XTILE_BYTES, gq, cq, xv);
            mma_stage<NT>(ring + slot * STAGE_BYTES, lane, gq, xv, acc);
            __syncwarp();
            if (lane == 0 && sidx + RD < total) {
                issue_w(slot);
                if constexpr (!NIN)
                    tma_x_tile<NT>(xring + slot * NT * XTILE_BYTES, &xm, kg0 + (sidx + RD) % nk, &bar[slot]);
            }
            if (++slot == RD) { slot = 0; phase ^= 1u; }
        }
        // ---- the group's partials meet in shared memory (every warp takes part) ----
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int r0 = mt * TILE_ROWS + gq, c0 = nt * 8 + 2 * cq;
                float* rw = red + ((size_t)warp * GROUP_ROWS) * L::RS;
                rw[r0 * L::RS + c0] = acc[mt][nt][0];
                rw[r0 * L::RS + c0 + 1] = acc[mt][nt][1];
                rw[(r0 + 8) * L::RS + c0] = acc[mt][nt][2];
                rw[(r0 + 8) * L::RS + c0 + 1] = acc[mt][nt][3];
            }
        __syncthreads();
        auto sum_rows = [&](int row, int n) {  // session n's column, warps 0..7 in order
            const int col = (n & ~7) | session_col(n & 7);
            float v = red[row * L::RS + col];
#pragma unroll
            for (int w = 1; w < MMVQ_WARPS; ++w) v = __fadd_rn(v, red[((size_t)w * GROUP_ROWS + row) * L::RS + col]);
            return v;
        };
        if constexpr (EPI == EPI_STORE || EPI == EPI_RESID) {
            for (int n = warp; n < a.B; n += MMVQ_WARPS) {  // a warp per session, a lane per row
                const float v = sum_rows(lane, n);
                if constexpr (EPI == EPI_STORE) {
                    epi_store(a, g, lane, n, v);
                } else {
                    const float x = epi_resid_apply(a, g, lane, n, n >= MMVQ_WARPS ? xold[NT - 1] : xold[0], v);
                    float s = __fmul_rn(x, x);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
                    if (lane == 0) a.ssq_out[(size_t)g * NORM_SLOTS + n] = s;
                }
            }
        } else {
            for (int e = tid; e < a.B * TILE_ROWS; e += MMVQ_WARPS * 32) {  // (row pair, session)
                const int n = e >> 4, rr = e & 15;
                const float v0 = sum_rows(rr, n), v1 = sum_rows(rr + TILE_ROWS, n);
                if constexpr (EPI == EPI_SWIGLU)
                    epi_swiglu(a, g, rr, n, v0, v1);
                else
                    epi_qkv_in(a, g, rr, n, v0, v1, e == tid ? qin : qkv_load(a, g, rr, n));
            }
        }
        __syncthreads();  // the partial buffer is reused by the next group
    }
    tl_exit(a.tl);
}

template <int NT, int EPI, bool PAIR, bool NIN>
static cudaError_t cta_attr() {
    cudaError_t e = cudaFuncSetAttribute(mmvq_cta_kernel<NT, EPI, PAIR, NIN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)CtaSmem<NT, PAIR, NIN>::TOTAL);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mmvq_cta_kernel<NT, EPI, PAIR, NIN>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

template <int NT, int EPI, bool PAIR, bool NIN>
static cudaError_t cta_launch(const MmvqArgs& a, const CUtensorMap& xm, int grid, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(MMVQ_WARPS * 32);
    cfg.dynamicSmemBytes = CtaSmem<NT, PAIR, NIN>::TOTAL;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mmvq_cta_kernel<NT, EPI, PAIR, NIN>, a, xm);
}

#define KD_CTA_CASES(X, NT_, PAIR_) \
    X(NT_, EPI_STORE, PAIR_, false) X(NT_, EPI_SWIGLU, PAIR_, false) X(NT_, EPI_QKV, PAIR_, false) \
    X(NT_, EPI_RESID, PAIR_, false)
// the fused norm feeds the projections after an RMSNorm: q|k|v and gate|up
#define KD_CTA_NIN_CASES(X, NT_) X(NT_, EPI_SWIGLU, false, true) X(NT_, EPI_QKV, false, true)

cudaError_t mmvq_cta_init_attributes() {
    cudaError_t e;
#define KD_A(NT_, EPI_, PAIR_, NIN_) \
    if ((e = cta_attr<NT_, EPI_, PAIR_, NIN_>()) != cudaSuccess) return e;
    KD_CTA_CASES(KD_A, 1, false)
    KD_CTA_CASES(KD_A, 2, false)
    KD_CTA_CASES(KD_A, 1, true)
    KD_CTA_NIN_CASES(KD_A, 1)
    KD_CTA_NIN_CASES(KD_A, 2)
#undef KD_A
    return cudaSuccess;
}

// The one-tile kernel (B <= 8) runs two CTAs per SM when the groups outnumber
// the SMs and the pair of CTAs on an SM takes no more groups than one CTA per SM
// would: one CTA per group up to 2 x SMs groups, else 2 x SMs CTAs.  Otherwise
// min(G, SMs) CTAs.  A CTA takes groups c, c + grid, ...
int mmvq_cta_grid(int G, int B, int num_sms, bool fused_norm, bool* pair) {
    const int per_sm = (G + num_sms - 1) / num_sms, per_pair = 2 * ((G + 2 * num_sms - 1) / (2 * num_sms));
    *pair = !fused_norm && B <= 8 && G > num_sms && per_pair <= per_sm;
    if (*pair) return G < 2 * num_sms ? G : 2 * num_sms;
    return G < num_sms ? G : num_sms;
}

cudaError_t launch_mmvq_cta(const MmvqArgs& a, const CUtensorMap& xm, int epi, int num_sms, bool pdl, cudaStream_t s) {
    const bool wide = a.B > 8, nin = a.nx != nullptr;
    if (nin && (a.KG > MMVQ_WARPS * NORM_IN_MAX_KG || (epi != EPI_QKV && epi != EPI_SWIGLU)))
        return cudaErrorInvalidValue;
    bool pair = false;
    const int grid = mmvq_cta_grid(a.G, a.B, num_sms, nin, &pair);
#define KD_L(NT_, EPI_, PAIR_, NIN_)                                  \
    if (epi == EPI_ && (NT_ == 2) == wide && PAIR_ == pair && NIN_ == nin) \
        return cta_launch<NT_, EPI_, PAIR_, NIN_>(a, xm, grid, pdl, s);
    KD_CTA_CASES(KD_L, 1, false)
    KD_CTA_CASES(KD_L, 2, false)
    KD_CTA_CASES(KD_L, 1, true)
    KD_CTA_NIN_CASES(KD_L, 1)
    KD_CTA_NIN_CASES(KD_L, 2)
#undef KD_L
    return cudaErrorInvalidValue;
}

}  // namespace kd
