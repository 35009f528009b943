// kd_ffn.cu -- the feed-forward block of a layer as one launch: the gate|up
// product with SwiGLU, then the down product with the residual add (and the
// next RMSNorm's NormLink outputs), on the group schedule of kd_mmvq_cta.cu.
//
// memra-engine decode_batch.rs runs the FFN of all B rows as two batched mmvq
// calls.  Here both products stream through the same per-warp rings of one
// persistent grid: when a warp has issued its last gate|up stage it goes on to
// its down stages' weights, so the HBM stream does not stop at the boundary
// between the two products.  The down stages' activation tiles (the SwiGLU
// output) are requested once every CTA has stored its gate|up part: a CTA that
// finishes its gate|up groups adds one to an arrival counter, and one thread
// of each CTA with down work polls it (bounded, with a short sleep between
// reads) before that CTA's warps request their tiles.  The arithmetic and the
// split of K over the warps are the group schedule's (kd_mmvq_cta.cu), so the
// results are those of the two products launched one after the other.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "kd_mmvq_common.cuh"

namespace kd {

template <int NT>
struct FfnSmem {
    static constexpr int RD = 3;                                              // stages in flight per warp
    static constexpr int RS = NT == 1 ? 9 : 16;                               // partial-row stride (floats)
    static constexpr size_t X_BYTES = (size_t)MMVQ_WARPS * RD * NT * XTILE_BYTES;  // 1024-byte aligned
    static constexpr size_t W_OFF = X_BYTES;
    static constexpr size_t BAR_OFF = W_OFF + (size_t)MMVQ_WARPS * RD * STAGE_BYTES;
    static constexpr size_t RED_OFF = BAR_OFF + MMVQ_WARPS * RD * sizeof(uint64_t);
    static constexpr size_t RED_BYTES = (size_t)MMVQ_WARPS * GROUP_ROWS * RS * sizeof(float);
    static constexpr size_t SC_OFF = RED_OFF + RED_BYTES;  // two [16] factor arrays: gate|up, down
    static constexpr size_t FLAG_OFF = SC_OFF + 2 * MAX_NORM_SLOTS * sizeof(float);  // the arrival wait's outcome
    static constexpr size_t TOTAL = FLAG_OFF + 16 + 1024;  // + alignment slack
};

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Order this thread's generic-proxy global accesses with its tensor-map copies.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
// Bounded poll until *p >= target (false: gave up), sleeping briefly between
// reads so that many pollers leave the line's L2 slice to the writers.
__device__ __forceinline__ bool wait_count(const int* p, int target) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0;; ++i) {
        if (ld_acquire_gpu(p) >= target) return true;
        if (i >= WAIT_MAX_POLLS || ((i & 15u) == 15u && global_timer_ns() - t0 > WAIT_MAX_NS)) return false;
        __nanosleep(64);
    }
}

// gu: gate|up (EPI_SWIGLU into gu.act, a NormLink consumer); dn: down (EPI_RESID,
// its x is gu.act); *ready: CTAs done with gate|up, zero at launch.  Grid: at
// most one CTA per SM and no more than gu.G CTAs, all resident together.
template <int NT>
__global__ void __launch_bounds__(MMVQ_WARPS * 32, 1)
    ffn_kernel(const MmvqArgs gu, const MmvqArgs dn, int* ready,
               const __grid_constant__ CUtensorMap xm_gu,
               const __grid_constant__ CUtensorMap xm_dn) {
    using L = FfnSmem<NT>;
    constexpr int RD = L::RD;
    constexpr uint32_t SB = STAGE_BYTES + NT * XTILE_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const int c = blockIdx.x, grid = gridDim.x;
    uint8_t* xring = smem + (size_t)warp * RD * NT * XTILE_BYTES;
    uint8_t* ring = smem + L::W_OFF + (size_t)warp * RD * STAGE_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF) + warp * RD;
    float* red = reinterpret_cast<float*>(smem + L::RED_OFF);
    float* sc0 = reinterpret_cast<float*>(smem + L::SC_OFF);  // gate|up: r_cur / r_pre
    float* sc1 = sc0 + MAX_NORM_SLOTS;                         // down: r_pre of the xs it writes
    volatile int* act_ok = reinterpret_cast<volatile int*>(smem + L::FLAG_OFF);

    // This warp's stages: gate|up groups c, c + grid, ..., then down groups
    // c, c + grid, ..., each over the warp's contiguous k-group range.
    const int kg0 = warp * gu.KG / MMVQ_WARPS, nk0 = (warp + 1) * gu.KG / MMVQ_WARPS - kg0;
    const int kg1 = warp * dn.KG / MMVQ_WARPS, nk1 = (warp + 1) * dn.KG / MMVQ_WARPS - kg1;
    const int ngrp0 = c < gu.G ? (gu.G - 1 - c) / grid + 1 : 0;
    const int ngrp1 = c < dn.G ? (dn.G - 1 - c) / grid + 1 : 0;
    const int tot0 = ngrp0 * nk0, total = tot0 + ngrp1 * nk1;

    if (lane == 0) {
        for (int i = 0; i < RD; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    __syncwarp();

    const uint64_t policy = l2_policy_evict_first();
    // Issue cursor (lane 0's copy is the one used): the next stage whose weights
    // are requested, as (phase, group index, k-group index).
    int wt = 0, wph = 0, wii = 0, wkk = 0;
    auto advance = [&]() {
        ++wt;
        if (++wkk == (wph ? nk1 : nk0)) {
            wkk = 0;
            if (++wii == (wph ? ngrp1 : ngrp0)) { wii = 0; ++wph; }
        }
        if (wph == 0 && wt == tot0) { wph = 1; wii = 0; wkk = 0; }  // no gate|up stages for this warp
    };
    auto x_tile = [&](int u, int ph, int kg) {  // stage u's activation tile
        if (ph)
            tma_x_tile<NT>(xring + (u % RD) * NT * XTILE_BYTES, &xm_dn, kg, &bar[u % RD]);
        else
            tma_x_tile<NT>(xring + (u % RD) * NT * XTILE_BYTES, &xm_gu, kg, &bar[u % RD]);
    };
    // Stage wt's weights, and its activation tile unless it is a down stage and
    // the SwiGLU output is not complete yet (then the phase boundary requests it).
    auto issue = [&](bool x_ok) {
        const int slot_ = wt % RD;
        mbar_arrive_expect_tx(&bar[slot_], SB);
        const int g = c + wii * grid;
        if (wph) {
            bulk_g2s_hint(ring + slot_ * STAGE_BYTES, dn.w + ((size_t)g * dn.KG + kg1 + wkk) * STAGE_BYTES,
                          STAGE_BYTES, &bar[slot_], policy);
            if (x_ok) x_tile(wt, 1, kg1 + wkk);
        } else {
            bulk_g2s_hint(ring + slot_ * STAGE_BYTES, gu.w + ((size_t)g * gu.KG + kg0 + wkk) * STAGE_BYTES,
                          STAGE_BYTES, &bar[slot_], policy);
            if (x_ok) x_tile(wt, 0, kg0 + wkk);
        }
        advance();
    };
    if (tot0 == 0) wph = 1;

    // Weights depend on nothing: the ring fills before the wait for the producer
    // of the gate|up input; the gate|up stages' activation tiles follow the wait.
    const int first = RD < total ? RD : total;
    if (lane == 0)
        for (int i = 0; i < first; ++i) {
            mbar_arrive_expect_tx(&bar[wt % RD], SB);  // (issue() without the activations)
            const int g = c + wii * grid;
            if (wph)
                bulk_g2s_hint(ring + (wt % RD) * STAGE_BYTES, dn.w + ((size_t)g * dn.KG + kg1 + wkk) * STAGE_BYTES,
                              STAGE_BYTES, &bar[wt % RD], policy);
            else
                bulk_g2s_hint(ring + (wt % RD) * STAGE_BYTES, gu.w + ((size_t)g * gu.KG + kg0 + wkk) * STAGE_BYTES,
                              STAGE_BYTES, &bar[wt % RD], policy);
            advance();
        }
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    if (lane == 0)
        for (int u = 0; u < first && u < tot0; ++u) x_tile(u, 0, kg0 + u % nk0);
    // The sessions' norm factors, while the first activation tiles are in flight.
    norm_scales<EPI_SWIGLU>(gu, sc0, warp, lane);
    norm_scales<EPI_RESID>(dn, sc1, warp, lane);
    __syncthreads();

    int t = 0, slot = 0;
    uint32_t phase = 0;
    bool failed = false;

    // One product's groups; each phase is compiled on its own.
    auto run_phase = [&](auto phc, const MmvqArgs& a) {
        constexpr int ph = decltype(phc)::value;
        const int ngrp = ph ? ngrp1 : ngrp0, nk = ph ? nk1 : nk0;
        if constexpr (ph == 1) {
            // This CTA's SwiGLU outputs are stored (the last gate|up epilogue ends
            // with a barrier): publish them, then wait until every CTA has.
            if (tid == 0) {
                __threadfence();
                atomicAdd(ready, 1);
                *act_ok = ngrp1 > 0 ? (int)wait_count(ready, grid) : 1;
            }
            __syncthreads();
            if (!*act_ok) {
                if (lane == 0) atomicOr(gu.err, ERR_WAIT_TIMEOUT);
                failed = true;
            }
            // The down stages whose weights are already requested get their
            // activation tiles now (whatever they hold if the wait gave up, so
            // that every requested stage lands).
            if (lane == 0) {
                fence_proxy_async_global();
                const int issued = t + RD < total ? t + RD : total;
                for (int u = tot0 > t ? tot0 : t; u < issued; ++u) {
                    const int r = u - tot0, kk = r % nk1;
                    x_tile(u, 1, kg1 + kk);
                }
            }
        }
        for (int gi = 0; gi < ngrp; ++gi) {
            const int g = c + gi * grid;
            float xold[NT];
            float nwr = 0.0f;
            if constexpr (ph == 1) {  // the residual rows and the next norm's weights, ahead of the epilogue
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int n = warp + MMVQ_WARPS * j;
                    xold[j] = n < a.B ? resid_load(a, g, lane, n) : 0.0f;
                }
                if (a.nl.xs != nullptr) nwr = a.nl.nw[(size_t)g * GROUP_ROWS + lane];
            }
            float acc[MT][NT][4];
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;
            for (int kk = 0; kk < nk && !failed; ++kk, ++t) {
                const bool ok = mbar_wait_bounded(&bar[slot], phase);
                if (__any_sync(FULL_MASK, !ok)) {
                    if (lane == 0) atomicOr(gu.err, ERR_WAIT_TIMEOUT);
                    failed = true;
                    break;
                }
                uint4 xv[4][NT];
                lds_x_tile<NT>(xring + slot * NT * XTILE_BYTES, gq, cq, xv);
                mma_stage<NT>(ring + slot * STAGE_BYTES, lane, gq, xv, acc);
                __syncwarp();
                if (lane == 0 && t + RD < total) issue(ph == 1 || t + RD < tot0);
                if (++slot == RD) { slot = 0; phase ^= 1u; }
            }
            // ---- the group's partials meet in shared memory ----
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
                for (int w = 1; w < MMVQ_WARPS; ++w)
                    v = __fadd_rn(v, red[((size_t)w * GROUP_ROWS + row) * L::RS + col]);
                return v;
            };
            if constexpr (ph == 0) {
                for (int e = tid; e < a.B * TILE_ROWS; e += MMVQ_WARPS * 32) {  // (row pair, session)
                    const int n = e >> 4, rr = e & 15;
                    const float f = sc0[n];
                    epi_swiglu(a, g, rr, n, __fmul_rn(sum_rows(rr, n), f), __fmul_rn(sum_rows(rr + TILE_ROWS, n), f));
                }
            } else {
                for (int n = warp; n < a.B; n += MMVQ_WARPS) {  // a warp per session, a lane per row
                    const float v = sum_rows(lane, n);
                    const float x = epi_resid_apply(a, g, lane, n, n >= MMVQ_WARPS ? xold[NT - 1] : xold[0], v);
                    if (a.nl.xs != nullptr) epi_xs(a, g, lane, n, x, nwr, sc1[n]);
                    float s = __fmul_rn(x, x);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
                    if (lane == 0) a.ssq_out[(size_t)n * a.G + g] = s;
                }
            }
            __syncthreads();  // the partial buffer is reused by the next group (and the stores precede the count)
        }
    };
    run_phase(std::integral_constant<int, 0>{}, gu);
    run_phase(std::integral_constant<int, 1>{}, dn);
    // After a wait gave up, copies may still be in flight: let every requested
    // stage land (bounded) before the CTA's shared memory is released.
    if (failed)
        for (int u = t; u < total && u < t + RD; ++u) (void)mbar_wait_bounded(&bar[u % RD], (uint32_t)(u / RD) & 1u);
}

size_t ffn_smem_bytes(bool wide) { return wide ? FfnSmem<2>::TOTAL : FfnSmem<1>::TOTAL; }

cudaError_t ffn_init_attributes() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(ffn_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)FfnSmem<1>::TOTAL)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(ffn_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)FfnSmem<2>::TOTAL)) != cudaSuccess)
        return e;
    for (const void* f : {(const void*)ffn_kernel<1>, (const void*)ffn_kernel<2>})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return e;
    return cudaSuccess;
}

cudaError_t launch_ffn(const MmvqArgs& gu, const MmvqArgs& dn, int* ready, const CUtensorMap& xm_gu,
                       const CUtensorMap& xm_dn, int num_sms, bool pdl, cudaStream_t s) {
    if (gu.B != dn.B || gu.B < 1 || gu.B > MAX_NORM_SLOTS || dn.K != gu.G * TILE_ROWS || dn.K % KGROUP)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gu.G < num_sms ? gu.G : num_sms);
    cfg.blockDim = dim3(MMVQ_WARPS * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (gu.B > 8) {
        cfg.dynamicSmemBytes = FfnSmem<2>::TOTAL;
        return cudaLaunchKernelEx(&cfg, ffn_kernel<2>, gu, dn, ready, xm_gu, xm_dn);
    }
    cfg.dynamicSmemBytes = FfnSmem<1>::TOTAL;
    return cudaLaunchKernelEx(&cfg, ffn_kernel<1>, gu, dn, ready, xm_gu, xm_dn);
}

}  // namespace kd
