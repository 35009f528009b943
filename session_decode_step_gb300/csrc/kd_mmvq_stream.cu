// kd_mmvq_stream.cu -- Q8_0 mmvq, "stream" schedule: for matrices with many
// more 32-row groups than SMs that do not spread evenly over them (lm_head).
//
// The matrix is a sequence of T = G * KG stages (one 128-column k-group of one
// row group, contiguous in memory).  Warp w of W takes stages [w*T/W, (w+1)*T/W),
// so every warp streams the same bytes (+-1 stage) as one contiguous range,
// through its own ring of shared-memory stages: a 1-D bulk copy of the stage's
// weights and tensor-map copies of its activation tiles, on one barrier.  A
// row group split between warps is finished by the last of them to arrive (one
// atomic per warp and group, no waiting): it adds the fp32 partials in warp
// order and runs the epilogue.  W depends on the shape and SM count, never on m.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_mmvq_common.cuh"

namespace kd {

__device__ __forceinline__ int stage_owner(long t, long T, long W) { return (int)(((t + 1) * W - 1) / T); }

// EPI_PICK state of a lane: for each of its two session columns per tile, the
// best pick key so far.
template <int NT>
struct PickLane {
    unsigned long long best[NT][2];
};

// The Gumbel words of this lane's four rows (gq + 8k, k < 4) of row group g in
// column (nt, j) -- entry e takes word e mod 4 of Philox block e / 4.  The four
// lanes gq = 4h + t (t < 4) of one cq need blocks 8g + 2k + h, k < 4, and word t
// of each: lane t computes block k = t, and four shuffle steps transpose the
// words (in step s lane t reads block (t + s) mod 4 from the lane that made it,
// which sends its word (k - s) mod 4).  Every lane takes part.  Out of line:
// only sampled steps call it, and its code stays out of the streaming loop.
__device__ __noinline__ void pick_words(const PickParams& p, int g, int gq, int lane, uint64_t (&out)[4]) {
    const int t = gq & 3, h = gq >> 2;
    uint64_t w[4];
    philox4x64_10((uint64_t)(8 * g + 2 * t + h), p.ctr, 0, 0, p.seed, 0, w);
#pragma unroll
    for (int sft = 0; sft < 4; ++sft) {
        const int q = (t - sft) & 3;  // the word this lane sends in this step
        const uint64_t send = q == 0 ? w[0] : q == 1 ? w[1] : q == 2 ? w[2] : w[3];
        const int k = (t + sft) & 3;  // the block this lane receives
        const int src = ((h * 4 + k) << 2) | (lane & 3);
        const uint64_t got = __shfl_sync(FULL_MASK, send, src);
        if (k == 0) out[0] = got;
        else if (k == 1) out[1] = got;
        else if (k == 2) out[2] = got;
        else out[3] = got;
    }
}

// Epilogue over this lane's fragment of a finished row group.
template <int NT, int EPI>
__device__ __forceinline__ void frag_epilogue(const MmvqArgs& a, int g, int gq, int cq, float (&v)[MT][NT][4],
                                              PickLane<NT>& pk) {
    if constexpr (EPI == EPI_PICK) {
        // keys of the lane's entries: rows gq + 8k (k = 2 mt + (i >> 1)) of columns (nt, i & 1)
        const int lane = (gq << 2) | cq;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const PickParams p = pick_params(a.samp, nt * 8 + col_session(2 * cq + j));
                uint64_t gw[4] = {0, 0, 0, 0};
                if (a.samp) pick_words(p, g, gq, lane, gw);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int row = gq + 8 * k;
                    float x = v[k >> 1][nt][((k & 1) << 1) | j];
                    if (p.T > 0.0f) x = gumbel_perturb(x, p.T, gw[k]);
                    pk.best[nt][j] = max(pk.best[nt][j], argmax_key(x, g * GROUP_ROWS + row));
                }
            }
    }
    float ss[NT][2];  // RESID: this lane's share of sum(x_new^2) per column
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) ss[nt][0] = ss[nt][1] = 0.0f;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = nt * 8 + col_session(2 * cq + (i & 1));
            if (n >= a.B) continue;
            const int r = gq + ((i >> 1) << 3);  // row within a 16-row tile
            if constexpr (EPI == EPI_STORE || EPI == EPI_PICK) {
                epi_store(a, g, r, n, v[0][nt][i]);
                epi_store(a, g, r + TILE_ROWS, n, v[1][nt][i]);
            } else if constexpr (EPI == EPI_RESID) {
                const float x0 = epi_resid(a, g, r, n, v[0][nt][i]);
                const float x1 = epi_resid(a, g, r + TILE_ROWS, n, v[1][nt][i]);
                ss[nt][i & 1] = __fmaf_rn(x1, x1, __fmaf_rn(x0, x0, ss[nt][i & 1]));
            } else if constexpr (EPI == EPI_SWIGLU) {
                epi_swiglu(a, g, r, n, v[0][nt][i], v[1][nt][i]);
            } else {
                epi_qkv(a, g, r, n, v[0][nt][i], v[1][nt][i]);
            }
        }
    if constexpr (EPI == EPI_RESID) {
        // sum over the 8 row lanes (gq) of each column, fixed tree; gq == 0 writes
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float s = ss[nt][j];
                s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, 4));
                s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, 8));
                s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, 16));
                const int n = nt * 8 + col_session(2 * cq + j);
                if (gq == 0 && n < a.B) a.ssq_out[(size_t)g * NORM_SLOTS + n] = s;
            }
    }
}

// The end of an EPI_PICK launch: a session's best key over the CTA's lanes
// (the 8 row lanes, then the warps) goes into pick_keys with one atomic
// maximum; the last CTA to arrive turns the keys into indices (-1 if nothing
// but NaN) and leaves the keys and the counter zero for the next launch --
// launch_argmax's merge, over keys made from the same stored values.
template <int NT>
__device__ __forceinline__ void pick_finish(const MmvqArgs& a, PickLane<NT>& pk, int warp, int lane) {
    __shared__ unsigned long long tab[MMVQ_WARPS][16];
    __shared__ bool last;
    const int gq = lane >> 2, cq = lane & 3, tid = threadIdx.x;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            unsigned long long k = pk.best[nt][j];
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) k = max(k, __shfl_xor_sync(FULL_MASK, k, o));
            if (gq == 0) tab[warp][nt * 8 + col_session(2 * cq + j)] = k;
        }
    __syncthreads();
    if (warp == 0) {  // B <= 16: the merging threads are lanes of warp 0
        if (lane < a.B) {
            unsigned long long k = tab[0][lane];
#pragma unroll
            for (int w = 1; w < MMVQ_WARPS; ++w) k = max(k, tab[w][lane]);
            if (k) atomicMax(&a.pick_keys[lane], k);
        }
        __threadfence();  // the warp's maxima are visible before its arrival
        __syncwarp();
        if (lane == 0) last = atomic_add_acq_rel(a.pick_done, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (last && tid < a.B) {  // after the acquiring arrival: every CTA's maxima are in
        const unsigned long long k = atomicExch(&a.pick_keys[tid], 0ull);
        a.pick_out[tid] = k ? (int)(~(unsigned)(k & 0xffffffffull)) : -1;
        if (tid == 0) *a.pick_done = 0u;
    }
}

// Shared memory: per warp a ring of RD stages, each the stage's weights and its
// activation tiles.
template <int NT>
struct StreamSmem {
    static constexpr int RD = NT == 1 ? RING : RING - 1;  // stages in flight per warp
    static constexpr size_t X_BYTES = (size_t)MMVQ_WARPS * RD * NT * XTILE_BYTES;  // at a 1024-byte boundary
    static constexpr size_t W_OFF = X_BYTES;
    static constexpr size_t BAR_OFF = W_OFF + (size_t)MMVQ_WARPS * RD * STAGE_BYTES;
    static constexpr size_t TOTAL = BAR_OFF + MMVQ_WARPS * RD * sizeof(uint64_t) + 1024;  // + alignment slack
};

template <int NT, int EPI>
__global__ void __launch_bounds__(MMVQ_WARPS * 32, 1)
    mmvq_stream_kernel(const MmvqArgs a, const __grid_constant__ CUtensorMap xm) {
    using L = StreamSmem<NT>;
    constexpr int RD = L::RD;
    constexpr uint32_t SB = STAGE_BYTES + NT * XTILE_BYTES;  // bytes a stage's barrier waits for
    extern __shared__ uint8_t smem_raw[];
    tl_entry(a.tl);
    uint8_t* smem = align1024(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    uint8_t* xring = smem + (size_t)warp * RD * NT * XTILE_BYTES;
    uint8_t* ring = smem + L::W_OFF + (size_t)warp * RD * STAGE_BYTES;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF) + warp * RD;

    const long T = (long)a.G * a.KG;
    const int w = blockIdx.x * MMVQ_WARPS + warp;
    const bool active = w < a.W;  // false only when the matrix has fewer stages than the grid has warps
    const long s_begin = active ? (long)w * T / a.W : 0, s_end = active ? (long)(w + 1) * T / a.W : 0;
    const int n = (int)(s_end - s_begin);

    if (lane == 0) {
        for (int i = 0; i < RD; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    __syncwarp();

    const uint64_t policy = l2_policy_evict_first();
    const uint8_t* wsrc = a.w + (size_t)s_begin * STAGE_BYTES;  // this warp's contiguous range
    // The weights do not depend on earlier kernels: start streaming them before
    // waiting for the producer of the activations.  Each barrier expects the
    // stage's weights and activations; the activations follow after the wait.
    if (lane == 0) {
        if (a.inject_tx && blockIdx.x == 0 && warp == 0 && n > 0) mbar_expect_tx(&bar[0], (uint32_t)a.inject_tx);
        for (int i = 0; i < RD && i < n; ++i) {
            mbar_arrive_expect_tx(&bar[i], SB);
            bulk_g2s_hint(ring + i * STAGE_BYTES, wsrc + (size_t)i * STAGE_BYTES, STAGE_BYTES, &bar[i], policy);
        }
        prefetch_tmap(&xm);
    }
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(a.tl);

    PickLane<NT> pk;
    if constexpr (EPI == EPI_PICK) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) pk.best[nt][j] = 0ull;
    }

    int g = (int)(s_begin / a.KG), kg = (int)(s_begin - (long)g * a.KG);
    int xkg = kg;  // k-group of the next stage whose activations are requested (lane 0)
    if (lane == 0)
        for (int i = 0; i < RD && i < n; ++i) {
            tma_x_tile<NT>(xring + i * NT * XTILE_BYTES, &xm, xkg, &bar[i]);
            if (++xkg == a.KG) xkg = 0;
        }

    float acc[MT][NT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[mt][nt][i] = 0.0f;

    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n; ++i) {
        const bool ok = mbar_wait_bounded(&bar[slot], phase);
        if (__any_sync(FULL_MASK, !ok)) {
            // Give up: flag it, let every copy already issued land, stop computing.
            if (lane == 0) atomicOr(a.err, ERR_WAIT_TIMEOUT);
            for (int t = i; t < n && t < i + RD; ++t)
                (void)mbar_wait_bounded(&bar[t % RD], (uint32_t)(t / RD) & 1u);
            // Keep the arrival counters consistent for the next launch: arrive on
            // every shared row group this warp still owns (the current one has not
            // been arrived on yet), and reset a counter when arriving last.  The
            // groups' outputs are not valid after a fault (the fault word says so).
            if (lane == 0) {
                const int g_last = (int)((s_end - 1) / a.KG);
                for (int gg = g; gg <= g_last; ++gg) {
                    const long first = (long)gg * a.KG;
                    const int w0 = stage_owner(first, T, a.W), w1 = stage_owner(first + a.KG - 1, T, a.W);
                    if (w0 != w1 && atomicAdd(&a.cnt[gg], 1) == w1 - w0) a.cnt[gg] = 0;
                }
            }
            break;
        }
        uint4 xv[4][NT];
        lds_x_tile<NT>(xring + slot * NT * XTILE_BYTES, gq, cq, xv);
        mma_stage<NT>(ring + slot * STAGE_BYTES, lane, gq, xv, acc);
        __syncwarp();
        if (lane == 0 && i + RD < n) {
            mbar_arrive_expect_tx(&bar[slot], SB);
            bulk_g2s_hint(ring + slot * STAGE_BYTES, wsrc + (size_t)(i + RD) * STAGE_BYTES, STAGE_BYTES,
                          &bar[slot], policy);
            tma_x_tile<NT>(xring + slot * NT * XTILE_BYTES, &xm, xkg, &bar[slot]);
            if (++xkg == a.KG) xkg = 0;
        }
        if (++slot == RD) { slot = 0; phase ^= 1u; }

        const bool seg_end = (kg == a.KG - 1) || (i == n - 1);
        if (!seg_end) {
            ++kg;
            continue;
        }
        // ---- this warp's part of row group g is done ----
        const long gfirst = (long)g * a.KG;
        const int w0 = stage_owner(gfirst, T, a.W), w1 = stage_owner(gfirst + a.KG - 1, T, a.W);
        // The group's finished values: the warp's own (the whole group was its),
        // or, for the last of several contributors, the sum of their partials.
        float v[MT][NT][4];
        bool finish = false;
        if (w0 == w1) {
            finish = true;
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i2 = 0; i2 < 4; ++i2) v[mt][nt][i2] = acc[mt][nt][i2];
        } else {
            const int ncontrib = w1 - w0 + 1;
            float* pt = a.part + ((size_t)g * a.maxc + (w - w0)) * (GROUP_ROWS * 16);
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
            if (lane == 0) last = (atomicAdd(&a.cnt[g], 1) == ncontrib - 1);
            last = __shfl_sync(FULL_MASK, last, 0);
            if (last) {
                __threadfence();
                // Sum the slots in contributor order; loads are issued CH slots at a
                // time so their latencies overlap.
                constexpr int CH = NT == 1 ? 4 : 4;
                const float* p0 = a.part + (size_t)g * a.maxc * (GROUP_ROWS * 16);
                for (int s0 = 0; s0 < ncontrib; s0 += CH) {
                    float2 lo[CH][MT][NT], hi[CH][MT][NT];
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        if (s0 + j >= ncontrib) break;
                        const float* ps = p0 + (size_t)(s0 + j) * (GROUP_ROWS * 16);
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const int r0 = mt * TILE_ROWS + gq, c0 = nt * 8 + 2 * cq;
                                lo[j][mt][nt] = ldcg_f2(ps + r0 * 16 + c0);
                                hi[j][mt][nt] = ldcg_f2(ps + (r0 + 8) * 16 + c0);
                            }
                    }
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        if (s0 + j >= ncontrib) break;
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                if (s0 + j == 0) {  // the first slot starts the sum
                                    v[mt][nt][0] = lo[j][mt][nt].x;
                                    v[mt][nt][1] = lo[j][mt][nt].y;
                                    v[mt][nt][2] = hi[j][mt][nt].x;
                                    v[mt][nt][3] = hi[j][mt][nt].y;
                                } else {
                                    v[mt][nt][0] = __fadd_rn(v[mt][nt][0], lo[j][mt][nt].x);
                                    v[mt][nt][1] = __fadd_rn(v[mt][nt][1], lo[j][mt][nt].y);
                                    v[mt][nt][2] = __fadd_rn(v[mt][nt][2], hi[j][mt][nt].x);
                                    v[mt][nt][3] = __fadd_rn(v[mt][nt][3], hi[j][mt][nt].y);
                                }
                            }
                    }
                }
                finish = true;
                if (lane == 0) a.cnt[g] = 0;  // ready for the next launch
            }
        }
        if (finish) frag_epilogue<NT, EPI>(a, g, gq, cq, v, pk);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i2 = 0; i2 < 4; ++i2) acc[mt][nt][i2] = 0.0f;
        ++g;
        kg = 0;
    }
    if constexpr (EPI == EPI_PICK) pick_finish<NT>(a, pk, warp, lane);
    tl_exit(a.tl);
}

template <int NT, int EPI>
static cudaError_t stream_attr() {
    cudaError_t e = cudaFuncSetAttribute(mmvq_stream_kernel<NT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)StreamSmem<NT>::TOTAL);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mmvq_stream_kernel<NT, EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

template <int NT, int EPI>
static cudaError_t stream_launch(const MmvqArgs& a, const CUtensorMap& xm, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.W + MMVQ_WARPS - 1) / MMVQ_WARPS);
    cfg.blockDim = dim3(MMVQ_WARPS * 32);
    cfg.dynamicSmemBytes = StreamSmem<NT>::TOTAL;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, mmvq_stream_kernel<NT, EPI>, a, xm);
}

#define KD_STREAM_CASES(X, NT_) \
    X(NT_, EPI_STORE) X(NT_, EPI_SWIGLU) X(NT_, EPI_QKV) X(NT_, EPI_RESID) X(NT_, EPI_PICK)

cudaError_t mmvq_stream_init_attributes() {
    cudaError_t e;
#define KD_A(NT_, EPI_) \
    if ((e = stream_attr<NT_, EPI_>()) != cudaSuccess) return e;
    KD_STREAM_CASES(KD_A, 1)
    KD_STREAM_CASES(KD_A, 2)
#undef KD_A
    return cudaSuccess;
}

cudaError_t launch_mmvq_stream(const MmvqArgs& a, const CUtensorMap& xm, int epi, bool pdl, cudaStream_t s) {
    const bool wide = a.B > 8;
#define KD_L(NT_, EPI_) \
    if (epi == EPI_ && (NT_ == 2) == wide) return stream_launch<NT_, EPI_>(a, xm, pdl, s);
    KD_STREAM_CASES(KD_L, 1)
    KD_STREAM_CASES(KD_L, 2)
#undef KD_L
    return cudaErrorInvalidValue;
}

}  // namespace kd
