// kd_attn.cu -- ragged GQA split-K flash-decode over slot-indexed fp16 KV.
//
// The attention phase of memra-engine decode_batch.rs `decode_batch_layers` (all
// sequences in one launch, then one combine) and hf2q ADR-040's
// batched flash-vec kernel (one dispatch for N queries, each with its own slot
// and kv_seq_len), for B sessions of unrelated lengths.
//
// Work item = (session b, KV head, split s): keys [s*C, min((s+1)*C, pos_b+1)),
// with C fixed, so the number of splits and every split's arithmetic depend on
// the session's own length only -- the result does not depend on what else is
// in the batch.  A persistent CTA per SM walks its items through a ring of
// shared-memory stages, filled by tensor-map copies of the split's K and V rows
// with the 128-byte swizzle; each item is computed by one warp.  Per item: the
// GQA group's scores and the weighted V sum as tensor-core products, a local
// softmax (max m, sum l) in between, written as (o, m, l).  A second kernel merges a session-head's
// splits in split order (online-softmax combine).
#include <cuda.h>

#include <type_traits>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kd_attn_common.cuh"

namespace kd {

// Shared memory of one CTA: a ring of STAGES stages shared by its warps.  A
// stage holds one work item: its K tile, then its V tile, each as 64-dim halves
// of [64 keys][128 B] written by tensor-map copies with the 128-byte swizzle
// (row r's 16-byte chunk c sits at chunk c ^ (r & 7)), so the 8 rows an
// ldmatrix phase reads always fall in 8 different bank groups.  Per stage: a
// full barrier and the CTA-local index of the item last issued into it.
template <int HD>
struct AttnSmem {
    static constexpr int NREG = HD / 64;                    // 64-dim halves of a row
    static constexpr int HALF_BYTES = AT_C * 128;           // one half of a work item's tile
    static constexpr int K_BYTES = NREG * HALF_BYTES;
    static constexpr int STAGE = 2 * K_BYTES;               // K tile, V tile
    static constexpr int STAGES = 192 * 1024 / STAGE;       // 6 at hd 128, 12 at hd 64
    static constexpr int BAR_OFF = STAGES * STAGE;           // per stage a K barrier, then per stage a V barrier
    static constexpr int ITEM_OFF = BAR_OFF + 2 * STAGES * 8;  // the same for the item words
    static constexpr int TOTAL = ITEM_OFF + 2 * STAGES * 4 + 16 + 1024;  // + flag, alignment slack
    static_assert(STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    // byte offset of (row, 16-byte chunk along the head dim) inside a tile
    static __device__ __forceinline__ uint32_t off(int row, int chunk) {
        return (uint32_t)((chunk >> 3) * HALF_BYTES + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
    }
};

// A CTA takes the items blockIdx.x + k * gridDim.x, k = 0, 1, ...: item k goes
// through stage k % STAGES and is computed by warp k % AT_WARPS, which then
// refills that stage with item k + STAGES: the K tile right after its scores,
// the V tile after its output.  For each tile a consumer first waits until the
// tile's item word says k (the copy of item k was issued, so the tile's barrier
// is in item k's phase), then for the barrier.  The scores S = Q K^T
// and the output O = P V are m16n8k16 tensor-core products taken transposed
// (S^T = K Q^T, O^T = V^T P^T): the 16 MMA rows are keys, then head dims, with
// no padding; the 8 columns are the GQA group's heads, each as q (then p)
// rounded to fp16 and the remainder of that rounding, whose two products add
// up to the fp32-accurate one.  K tiles are the A operand as stored, V tiles
// through the transposing ldmatrix.
template <int HD, int GQ>
__global__ void __launch_bounds__(AT_WARPS * 32, 1)
    attn_split_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmk8, const __grid_constant__ CUtensorMap tmv,
                      const __grid_constant__ CUtensorMap tmv8) {
    using L = AttnSmem<HD>;
    constexpr int S = L::STAGES;
    constexpr int KS = HD / 16;  // 16-dim k-steps of Q K^T
    constexpr int NU = HD / 8;   // 8-dim output tiles of P V
    static_assert(GQ == 1 || GQ == 2 || GQ == 4 || GQ == 8, "GQA group");
    extern __shared__ uint8_t smem_raw[];
    tl_entry(a.tl);
    uint8_t* smem = align1024(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    // Stage st's K tile lands on bar[st] and its V tile on bar[S + st]; item
    // words likewise (the last item whose K, resp. V, copy was issued there).
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    volatile int* stage_item = reinterpret_cast<volatile int*>(smem + L::ITEM_OFF);
    volatile int* cta_failed = stage_item + 2 * S;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2 * S; ++i) {
            mbar_init(&bar[i], 1);
            stage_item[i] = -1;
        }
        *cta_failed = 0;
        mbar_init_fence();
        if (a.inject_tx && blockIdx.x == 0) mbar_expect_tx(&bar[0], (uint32_t)a.inject_tx);  // debug fault hook
    }
    __syncthreads();

    AttnTable tab;
    tab.build(a, lane);
    const int n_items = tab.n_items;
    const int nk = (int)blockIdx.x < n_items ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto gitem = [&](int k) { return (int)blockIdx.x + k * (int)gridDim.x; };
    // Issue the copies of the CTA's item k into stage k % S (lane 0): its K tile
    // (parts & 1) and/or its V tile (parts & 2), each on its own barrier.  Cached
    // keys and values are read once per step: their lines go first when L2 needs
    // room, ahead of the step's small, often re-read activation buffers.
    const uint64_t kv_policy = l2_policy_evict_first();
    auto issue = [&](const AttnItem& it, int k, int parts) {
        const int st = k % S;
        uint8_t* stg = smem + st * L::STAGE;
        const int row = (int)(a.row0 + ((long)it.slot * a.nkv + it.kvh) * a.cap + (long)it.s * AT_C);
        const bool full = it.n == AT_C;
        const int krows = full ? AT_C : (it.n + 7) / 8 * 8;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            if (!((parts >> part) & 1)) continue;
            uint64_t* b = &bar[part * S + st];
            const CUtensorMap* tm = part ? &tmv : &tmk;
            const CUtensorMap* tm8 = part ? &tmv8 : &tmk8;
            stage_item[part * S + st] = k;
            mbar_arrive_expect_tx(b, (uint32_t)(L::NREG * krows * 128));
            for (int r = 0; r < L::NREG; ++r) {
                uint8_t* dst = stg + part * L::K_BYTES + r * L::HALF_BYTES;
                if (full)
                    tma_load_2d_hint(dst, tm, r * 64, row, b, kv_policy);
                else
                    for (int k8 = 0; k8 < krows; k8 += 8)
                        tma_load_2d_hint(dst + k8 * 128, tm8, r * 64, row + k8, b, kv_policy);
            }
        }
    };

    // The first S items fill the ring.  History rows (keys < pos) were written by
    // earlier steps: items that do not hold this step's new row are fetched before
    // waiting on the QKV kernel.
    if (threadIdx.x == 0) {  // the ragged-tail maps are often first used after the wait
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmk8);
        prefetch_tmap(&tmv8);
    }
    unsigned early = 0;
    for (int i = 0, k = warp; k < S && k < nk; ++i, k += AT_WARPS) {
        const AttnItem it = tab.item(a, lane, gitem(k));
        if (it.s != it.ns - 1) {
            if (lane == 0) issue(it, k, 3);
            early |= 1u << i;
        }
    }
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(a.tl);
    for (int i = 0, k = warp; k < S && k < nk; ++i, k += AT_WARPS)
        if (!((early >> i) & 1u)) {
            const AttnItem it = tab.item(a, lane, gitem(k));
            if (lane == 0) issue(it, k, 3);
        }

    // The MMAs' 8-wide N dimension: column 2h + part of N-tile j is head 4j + h,
    // part 0 carrying q (then p) rounded to fp16 and part 1 the remainder of that
    // rounding.  Lane (g, c) supplies column g (head 4j + g/2, part g & 1) of the
    // B fragments and holds columns 2c, 2c + 1 (both parts of head 4j + c) of
    // the results, so the two parts add up in the lane.
    constexpr int NQ = GQ > 4 ? GQ / 4 : 1;  // N-tiles of heads
    const int colh = g >> 1;
    const bool col_lo = (g & 1) != 0;
    // q of the lane's column head, dims 16 ks + 2c (+1) and 16 ks + 8 + 2c (+1)
    float2 qv[NQ][KS][2];
    auto load_q = [&](const AttnItem& it) {
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const int h = 4 * j + colh;
            if (h < GQ) {
                const float* qp = a.q + ((size_t)it.b * a.nh + (size_t)it.kvh * GQ + h) * HD + 2 * c;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    qv[j][ks][0] = *reinterpret_cast<const float2*>(qp + 16 * ks);
                    qv[j][ks][1] = *reinterpret_cast<const float2*>(qp + 16 * ks + 8);
                }
            }
        }
    };
    if (warp < nk) load_q(tab.item(a, lane, gitem(warp)));

    for (int k = warp; k < nk; k += AT_WARPS) {
        const AttnItem it = tab.item(a, lane, gitem(k));
        const int st = k % S;
        uint8_t* stg = smem + st * L::STAGE;
        const uint32_t kbase = smem_u32(stg), vbase = kbase + L::K_BYTES;

        uint32_t qb[NQ][KS][2];  // B fragments of Q^T
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const bool on = 4 * j + colh < GQ;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const float2 u = qv[j][ks][0], w = qv[j][ks][1];
                qb[j][ks][0] = !on ? 0u : (col_lo ? f2_lo(u.x, u.y) : f2_hi(u.x, u.y));
                qb[j][ks][1] = !on ? 0u : (col_lo ? f2_lo(w.x, w.y) : f2_hi(w.x, w.y));
            }
        }
        if (k + AT_WARPS < nk) load_q(tab.item(a, lane, gitem(k + AT_WARPS)));  // lands during this item

        const uint32_t par = (uint32_t)(k / S) & 1u;
        bool ok = wait_value(stage_item + st, k);
        ok = ok && mbar_wait_bounded(&bar[st], par);  // the K tile
        if (__any_sync(FULL_MASK, !ok)) {
            if (lane == 0) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                *cta_failed = 1;
            }
            break;
        }
        const int n = it.n;
        const bool refill = k + S < nk;
        AttnItem nx{};
        if (refill) nx = tab.item(a, lane, gitem(k + S));

        // ---- S^T = K Q^T: M = 16 keys (AT_KT tiles), N = the head columns, K = 16 dims.
        // k-steps outside, key tiles inside: MMAs issued back to back go to
        // different accumulators; each tile adds its k-steps in order.
        float sacc[AT_KT][NQ][4];
#pragma unroll
        for (int m = 0; m < AT_KT; ++m)
#pragma unroll
            for (int j = 0; j < NQ; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[m][j][i] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            uint32_t ka[AT_KT][4];
#pragma unroll
            for (int m = 0; m < AT_KT; ++m)
                ldsm_x4(kbase + L::off(16 * m + ((lane >> 3) & 1) * 8 + (lane & 7), 2 * ks + (lane >> 4)), ka[m][0],
                        ka[m][1], ka[m][2], ka[m][3]);
#pragma unroll
            for (int j = 0; j < NQ; ++j)
#pragma unroll
                for (int m = 0; m < AT_KT; ++m)
                    mma_16816_acc(sacc[m][j], ka[m][0], ka[m][1], ka[m][2], ka[m][3], qb[j][ks][0], qb[j][ks][1]);
        }
        // The K tile is read: refill it with item k + S's, half an item before its V.
        __syncwarp();
        if (refill && lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(nx, k + S, 1);
        }
        // ---- per head 4j + c: scores of keys 16m + g (e = 0) and 16m + g + 8 (e = 1);
        // scale, mask, softmax over the item's keys (the 8 lanes g of a head)
        float sv[NQ][AT_KT][2], mx[NQ], lsum[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            mx[j] = -INFINITY;
#pragma unroll
            for (int m = 0; m < AT_KT; ++m)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float sc = __fadd_rn(sacc[m][j][2 * e], sacc[m][j][2 * e + 1]);  // both parts
                    const int key = 16 * m + g + 8 * e;
                    sv[j][m][e] = key < n ? __fmul_rn(sc, a.scale) : -INFINITY;
                    mx[j] = fmaxf(mx[j], sv[j][m][e]);
                }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) mx[j] = fmaxf(mx[j], __shfl_xor_sync(FULL_MASK, mx[j], o));
            lsum[j] = 0.0f;
#pragma unroll
            for (int m = 0; m < AT_KT; ++m)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = 16 * m + g + 8 * e;
                    sv[j][m][e] = key < n ? expf(__fsub_rn(sv[j][m][e], mx[j])) : 0.0f;
                    lsum[j] = __fadd_rn(lsum[j], sv[j][m][e]);
                }
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) lsum[j] = __fadd_rn(lsum[j], __shfl_xor_sync(FULL_MASK, lsum[j], o));
        }

        // The V tile.
        ok = wait_value(stage_item + S + st, k);
        ok = ok && mbar_wait_bounded(&bar[S + st], par);
        if (__any_sync(FULL_MASK, !ok)) {
            if (lane == 0) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                *cta_failed = 1;
            }
            break;
        }
        if (n < AT_C) {
            // V rows [n, 16-key step end) enter the last P V step with p = 0: make
            // them zero (they hold other positions or stale data, possibly NaN).
            const int z = ((n + 15) & ~15) - n;
            for (int e = lane; e < z * L::NREG * 8; e += 32) {
                const int r = n + e / (L::NREG * 8), rem = e % (L::NREG * 8);
                *reinterpret_cast<uint4*>(stg + L::K_BYTES + (rem >> 3) * L::HALF_BYTES + r * 128 + (rem & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }

        // ---- O^T = V^T P^T: M = 16 dims (NU/2 tiles), N = the head columns, K = 16 keys,
        // over the key steps that hold keys.  P^T's B fragment of lane (g, c) wants
        // keys 2c, 2c + 1 (and + 8) of its column head: they sit in lanes
        // (2c, g/2) and (2c + 1, g/2).
        float oacc[NU / 2][NQ][4];
#pragma unroll
        for (int mt = 0; mt < NU / 2; ++mt)
#pragma unroll
            for (int j = 0; j < NQ; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) oacc[mt][j][i] = 0.0f;
        const int nsteps = (n + 15) >> 4;
        const int src0 = (2 * c) * 4 + colh, src1 = src0 + 4;
#pragma unroll
        for (int js = 0; js < AT_KT; ++js) {
            if (js < nsteps) {
                uint32_t pb[NQ][2];
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
                    const float v00 = __shfl_sync(FULL_MASK, sv[j][js][0], src0);
                    const float v01 = __shfl_sync(FULL_MASK, sv[j][js][0], src1);
                    const float v10 = __shfl_sync(FULL_MASK, sv[j][js][1], src0);
                    const float v11 = __shfl_sync(FULL_MASK, sv[j][js][1], src1);
                    const bool on = 4 * j + colh < GQ;
                    pb[j][0] = !on ? 0u : (col_lo ? f2_lo(v00, v01) : f2_hi(v00, v01));
                    pb[j][1] = !on ? 0u : (col_lo ? f2_lo(v10, v11) : f2_hi(v10, v11));
                }
                uint32_t va[NU / 2][4];
#pragma unroll
                for (int mt = 0; mt < NU / 2; ++mt)
                    ldsm_x4_trans(vbase + L::off(16 * js + (lane >> 4) * 8 + (lane & 7), 2 * mt + ((lane >> 3) & 1)),
                                  va[mt][0], va[mt][1], va[mt][2], va[mt][3]);
#pragma unroll
                for (int j = 0; j < NQ; ++j)
#pragma unroll
                    for (int mt = 0; mt < NU / 2; ++mt)
                        mma_16816_acc(oacc[mt][j], va[mt][0], va[mt][1], va[mt][2], va[mt][3], pb[j][0], pb[j][1]);
            }
        }
        // ---- both parts of head 4j + c, dims 16 mt + g and 16 mt + g + 8: write (o, m, l)
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const int h = 4 * j + c;
            if (h < GQ) {
                float* dst = a.part + (((size_t)it.b * a.nh + (size_t)it.kvh * GQ + h) * a.max_splits + it.s) *
                                          ATT_REC(HD);
#pragma unroll
                for (int mt = 0; mt < NU / 2; ++mt) {
                    dst[16 * mt + g] = __fadd_rn(oacc[mt][j][0], oacc[mt][j][1]);
                    dst[16 * mt + g + 8] = __fadd_rn(oacc[mt][j][2], oacc[mt][j][3]);
                }
                if (g == 0) *reinterpret_cast<float2*>(dst + HD) = make_float2(mx[j], lsum[j]);
            }
        }

        __syncwarp();  // the V tile is read: refill it
        if (refill && lane == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue(nx, k + S, 2);
        }
    }
    // After a wait gave up, copies may still be in flight: before the CTA's shared
    // memory is released, wait (bounded) for the last item issued into each K and
    // each V tile.
    __syncthreads();
    if (threadIdx.x == 0 && *cta_failed)
        for (int i = 0; i < 2 * S; ++i) {
            const int k = stage_item[i];
            if (k >= 0) (void)mbar_wait_bounded(&bar[i], (uint32_t)(k / S) & 1u);
        }
    tl_exit(a.tl);
}

// Merge a (session, head)'s splits (flash-decoding's reduction):
//   M = max_s m_s,  out = fp16( sum_s e^{m_s - M} o_s / sum_s e^{m_s - M} l_s ).
// NW warps.  The numerator is split into NW contiguous ranges of splits, one per
// warp, whose lanes read whole records (HD/32 dims each, 16- or 8-byte loads)
// and sum their range in split order, COMB_UNROLL records in flight; the first
// COMB_UNROLL records of every range are requested before anything else, so that
// a short session's merge waits for one batch of loads.  Each thread reads the
// (m, l) of splits t, t + 32 NW, ... into shared memory; M is a block max, the
// weights e^{m_s - M} are formed once per split and the denominator is a fixed
// tree (each thread summing its splits in order, then the warps' sums in warp
// order); the warps' numerators are added in warp order.  Every order depends on
// the session's split count and NW (fixed by the split capacity) only.
constexpr int COMB_MAX_SPLITS = ATT_MAX_SPLITS;
constexpr int COMB_UNROLL = 8;
// warps of the merge: 4 up to 64 splits (4096 positions) of capacity, 32 beyond
__host__ __device__ constexpr int comb_warps(int max_splits) { return max_splits <= 64 ? 4 : 32; }

template <int HD, int NW>
__global__ void __launch_bounds__(NW * 32) attn_combine_kernel(const AttnArgs a) {
    constexpr int DPL = HD / 32;  // dims per lane
    constexpr int NT = NW * 32;
    static_assert(DPL == 2 || DPL == 4, "head_dim 64 or 128");
    using VecT = typename std::conditional<DPL == 4, float4, float2>::type;
    __shared__ float wts[COMB_MAX_SPLITS], ls[COMB_MAX_SPLITS];
    __shared__ float red_m[NW], red_l[NW];
    __shared__ __align__(16) float part[NW][HD];
    tl_entry(a.tl);
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    const int b = blockIdx.y, h = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    // The step's positions were staged before its first kernel: read while the
    // split kernel finishes.
    const int pos_b = b < a.B ? a.pos[b] : 0;
    pdl_wait();
    tl_waited(a.tl);
    if (b >= a.B) {
        tl_exit(a.tl);
        return;
    }
    const float* p = a.part + ((size_t)b * a.nh + h) * a.max_splits * ATT_REC(HD);
    // Only the session's own split records are read: records past its split count
    // may be cold (never written).
    const int ns = (pos_b + ATT_CHUNK) / ATT_CHUNK;
    // the warp's range of splits, and its first records
    const int s0 = (int)(((long)ns * warp) / NW), s1 = (int)(((long)ns * (warp + 1)) / NW);
    const float* pl = p + lane * DPL;
    VecT o[COMB_UNROLL];
#pragma unroll
    for (int u = 0; u < COMB_UNROLL; ++u)
        if (s0 + u < s1) o[u] = __ldcg(reinterpret_cast<const VecT*>(pl + (size_t)(s0 + u) * ATT_REC(HD)));
    float mloc = -INFINITY;
    for (int s = t; s < ns; s += NT) {
        const float2 ml = __ldcg(reinterpret_cast<const float2*>(p + (size_t)s * ATT_REC(HD) + HD));
        wts[s] = ml.x;
        ls[s] = ml.y;
        mloc = fmaxf(mloc, ml.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(FULL_MASK, mloc, off));
    if (lane == 0) red_m[warp] = mloc;
    __syncthreads();
    float M = red_m[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) M = fmaxf(M, red_m[w]);
    float den = 0.0f;
    for (int s = t; s < ns; s += NT) {
        const float e = expf(__fsub_rn(wts[s], M));
        wts[s] = e;
        den = __fmaf_rn(e, ls[s], den);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) den = __fadd_rn(den, __shfl_xor_sync(FULL_MASK, den, off));
    if (lane == 0) red_l[warp] = den;
    __syncthreads();
    float L = red_l[0];
#pragma unroll
    for (int w = 1; w < NW; ++w) L = __fadd_rn(L, red_l[w]);
    float num[DPL];
#pragma unroll
    for (int i = 0; i < DPL; ++i) num[i] = 0.0f;
    for (int sb = s0; sb < s1; sb += COMB_UNROLL) {
        if (sb != s0) {
#pragma unroll
            for (int u = 0; u < COMB_UNROLL; ++u)
                if (sb + u < s1) o[u] = __ldcg(reinterpret_cast<const VecT*>(pl + (size_t)(sb + u) * ATT_REC(HD)));
        }
#pragma unroll
        for (int u = 0; u < COMB_UNROLL; ++u)
            if (sb + u < s1) {
                const float e = wts[sb + u];
                const float* ov = reinterpret_cast<const float*>(&o[u]);
#pragma unroll
                for (int i = 0; i < DPL; ++i) num[i] = __fmaf_rn(e, ov[i], num[i]);
            }
    }
#pragma unroll
    for (int i = 0; i < DPL; ++i) part[warp][lane * DPL + i] = num[i];
    __syncthreads();
    for (int d = t; d < HD; d += NT) {
        float n = part[0][d];
#pragma unroll
        for (int w = 1; w < NW; ++w) n = __fadd_rn(n, part[w][d]);
        a.out[(size_t)b * a.nh * HD + (size_t)h * HD + d] = __float2half_rn(__fdiv_rn(n, L));
    }
    tl_exit(a.tl);
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
                             AttnSmem<HD_>::TOTAL);                                                  \
    if (e != cudaSuccess) return e;                                                                  \
    e = cudaFuncSetAttribute(attn_split_kernel<HD_, GQ_>, cudaFuncAttributePreferredSharedMemoryCarveout, \
                             cudaSharedmemCarveoutMaxShared);                                        \
    if (e != cudaSuccess) return e;
    for (int group : {1, 2, 4, 8}) {
        KD_ATT_DISPATCH(64, KD_SET)
        KD_ATT_DISPATCH(128, KD_SET)
    }
#undef KD_SET
    for (const void* f : {(const void*)attn_combine_kernel<64, 4>, (const void*)attn_combine_kernel<128, 4>,
                          (const void*)attn_combine_kernel<64, 32>, (const void*)attn_combine_kernel<128, 32>,
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
                                                      AT_WARPS * 32, AttnSmem<HD_>::TOTAL);
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

cudaError_t encode_fp16_2d(CUtensorMap* out, const void* base, long inner, long rows, int box_inner, int box_rows) {
    static EncodeTiledFn encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (inner < 1 || rows < 1 || rows > 0x7fffffffL || (inner * 2) % 16 || (reinterpret_cast<uintptr_t>(base) & 15))
        return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    const cuuint32_t estr[2] = {1, 1};
    const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_attn_maps(const __half* k_arena, const __half* v_arena, long rows, int hd, AttnMaps* out) {
    if (hd != 64 && hd != 128) return cudaErrorInvalidValue;
    cudaError_t e;
    if ((e = encode_fp16_2d(&out->k, k_arena, hd, rows, 64, ATT_CHUNK)) != cudaSuccess) return e;
    if ((e = encode_fp16_2d(&out->k8, k_arena, hd, rows, 64, 8)) != cudaSuccess) return e;
    if ((e = encode_fp16_2d(&out->v, v_arena, hd, rows, 64, ATT_CHUNK)) != cudaSuccess) return e;
    return encode_fp16_2d(&out->v8, v_arena, hd, rows, 64, 8);
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
    cfg.stream = s;
#define KD_LAUNCH(HD_, GQ_)                                 \
    cfg.blockDim = dim3(AT_WARPS * 32);                     \
    cfg.dynamicSmemBytes = AttnSmem<HD_>::TOTAL;            \
    return cudaLaunchKernelEx(&cfg, attn_split_kernel<HD_, GQ_>, a, maps.k, maps.k8, maps.v, maps.v8);
    if (a.hd == 64) { KD_ATT_DISPATCH(64, KD_LAUNCH) } else if (a.hd == 128) { KD_ATT_DISPATCH(128, KD_LAUNCH) }
#undef KD_LAUNCH
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_combine(const AttnArgs& a, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    launch_cfg(cfg, attr, pdl);
    const int nw = comb_warps(a.max_splits);
    cfg.gridDim = dim3(a.nh, a.B);
    cfg.blockDim = dim3(nw * 32);
    cfg.stream = s;
    if (a.hd == 64)
        return nw == 4 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<64, 4>, a)
                       : cudaLaunchKernelEx(&cfg, attn_combine_kernel<64, 32>, a);
    if (a.hd == 128)
        return nw == 4 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel<128, 4>, a)
                       : cudaLaunchKernelEx(&cfg, attn_combine_kernel<128, 32>, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_kv_append(const float* k, const float* v, __half* kc, __half* vc, const int* slot,
                             const int* pos, int B, int nkv, int hd, int cap, cudaStream_t s) {
    kv_append_kernel<<<dim3(nkv, B), 128, 0, s>>>(k, v, kc, vc, slot, pos, nkv, hd, cap);
    return cudaGetLastError();
}

}  // namespace kd
