// kd_attn_q8.cu -- the KV cache in Q8_0 (the long-context option): quantised
// append and split-K flash-decode over Q8_0 keys and values (head_dim 128).
//
// A cached head row is 128 one-byte quants u = q + 128 and four fp16 block
// scales (one per 32 dims): 136 bytes instead of 256 in fp16, so a 64-key work
// item moves 8.5 KB per tile.  Quantisation, in fp32: per block d = max|x| / 127,
// stored as fp16(d), q = x / d rounded half away from zero, within [-127, 127]
// (memra appends quantised K/V in `decode_batch_layers` phase A; hf2q ADR-040
// measures against llama.cpp's q8_0 K/V).
//
// The attention keeps the fp16 kernel's work items, bounded waits and merge
// (kd_attn.cu), with separate rings for the K and the V parts of the items; the
// tiles and the two products differ:
//   scores Sᵀ = K Qᵀ per 32-dim block: the quants, read with ldmatrix as pairs
//   of bytes and converted to fp16 exactly, are the A operand of the block's two
//   m16n8k16 MMAs, whose k index runs over the block's dims in the fixed order
//   (4c, 4c+1 | 4c+2, 4c+3) that the query's B operand shares; the block's
//   partial scores are scaled by the key's block scale in fp32 and summed;
//   values Oᵀ = Vᵀ Pᵀ: the transposing ldmatrix, reading the quants as pairs of
//   bytes, gives a lane keys 2c, 2c+1 of dims 2g, 2g+1; one byte permute per
//   register splits them into the A operand of dim 2g (MMA row g) and of dim
//   2g + 1 (row g + 8), so a 16-dim slice's rows hold its even dims, then its
//   odd ones; the value scales multiply the probabilities instead (p_t d_t,blk,
//   split into fp16 hi + lo like p in the fp16 kernel), one B operand per
//   32-dim block.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_attn_common.cuh"

namespace kd {

struct AttnQ8Smem {
    static constexpr int HD = 128;
    static constexpr int QROW = 128;                     // bytes of a row's quants
    static constexpr int NBLK = HD / 32;                 // block scales per row
    static constexpr int TILE = AT_C * QROW;             // 8 KB of quants per tile
    static constexpr int SROW = NBLK * 2;                // 8 bytes of scales per row
    static constexpr int STILE = AT_C * SROW;            // 512 B of scales per tile
    // Separate rings for the items' K parts (SK slots) and V parts (SV slots): a V
    // part is re-issued only when its slot's previous item has finished its value
    // phase, so V needs the deeper ring (K 8 / V 18 measured best of the 26 slots'
    // splits; 13 / 13 was 1.4% slower on the long-context step, 6 / 20 2.4%).
    static constexpr int SK = 8, SV = 18;
    static constexpr int KQ_OFF = 0, VQ_OFF = SK * TILE, KS_OFF = (SK + SV) * TILE, VS_OFF = KS_OFF + SK * STILE;
    // Consumer warps per CTA (one CTA per SM): as many as the kernel's registers
    // allow without spilling -- 16 (128 registers a lane) for a group of 4, 12 for
    // groups of 1 and 2, 8 for a group of 8.
    static constexpr __host__ __device__ int warps(int group) { return group == 8 ? 8 : group == 4 ? 16 : 12; }
    // as many 17 KB stages as the opt-in shared memory holds (with barriers, item words, slack)
    static constexpr int BAR_OFF = VS_OFF + SV * STILE;
    static constexpr int ITEM_OFF = BAR_OFF + (SK + SV) * 8;
    static constexpr int TOTAL = ITEM_OFF + (SK + SV) * 4 + 16 + 1024;
    static_assert(TILE % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(TOTAL <= 227 * 1024, "opt-in shared memory");
    // quants: row r's 16-byte chunk c at chunk c ^ (r & 7) (128-byte swizzle)
    static __device__ __forceinline__ uint32_t qoff(int row, int chunk) {
        return (uint32_t)(row * QROW + ((chunk ^ (row & 7)) << 4));
    }
};

// The lane's part of an fp16 hi/lo split of the pair (x, y): hi = x with its 13
// low mantissa bits cleared (exact in fp16 for |x| in fp16's normal range), lo =
// fp16(x - hi) (x - hi is exact in fp32); hi + lo is within 2^-21 |x| of x.  A
// hi lane passes cf = 0, sgn = 0 (0 x + hi), a lo lane cf = 1, sgn = the sign bit
// (x - hi): the same four instructions and one conversion on every lane.
__device__ __forceinline__ uint32_t f2_part(float x, float y, float cf, uint32_t sgn) {
    const float tx = __uint_as_float((__float_as_uint(x) & 0xFFFFE000u) ^ sgn);
    const float ty = __uint_as_float((__float_as_uint(y) & 0xFFFFE000u) ^ sgn);
    return f2_hi(__fmaf_rn(cf, x, tx), __fmaf_rn(cf, y, ty));
}

// fp16 bit pairs as fp32 (one conversion each).
__device__ __forceinline__ float2 h2bits_to_float2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Bytes 0 and 2 (even) or 1 and 3 (odd) of v, each u = q + 128, as half2(q, q')
// exactly (the same magic-number conversion as the byte-pair helpers).
__device__ __forceinline__ uint32_t u8x2_even_to_half2(uint32_t v) {
    const uint32_t h = __byte_perm(v, 0x64646464u, 0x4240);
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}
__device__ __forceinline__ uint32_t u8x2_odd_to_half2(uint32_t v) {
    const uint32_t h = __byte_perm(v, 0x64646464u, 0x4341);
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

template <int GQ>
__global__ void __launch_bounds__(AttnQ8Smem::warps(GQ) * 32, 1)
    attn_split_q8_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmk8, const __grid_constant__ CUtensorMap tmv,
                         const __grid_constant__ CUtensorMap tmv8) {
    using L = AttnQ8Smem;
    constexpr int SK = L::SK, SV = L::SV, SMAX = SK > SV ? SK : SV;
    constexpr int HD = L::HD;
    constexpr int NU = HD / 8;  // 8-dim output tiles of P V
    constexpr int W = L::warps(GQ);
    static_assert(GQ == 1 || GQ == 2 || GQ == 4 || GQ == 8, "GQA group");
    extern __shared__ uint8_t smem_raw[];
    tl_entry(a.tl);
    uint8_t* smem = align1024(smem_raw);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
    volatile int* stage_item = reinterpret_cast<volatile int*>(smem + L::ITEM_OFF);
    volatile int* cta_failed = stage_item + SK + SV;

    if (threadIdx.x == 0) {
        for (int i = 0; i < SK + SV; ++i) {
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
    // Issue the copies of the CTA's item k (lane 0): its K part (parts & 1: quants
    // and scales) into K slot k % SK and/or its V part (parts & 2) into V slot
    // k % SV, each on its slot's barrier.  Quants by tensor map (64-row box, or 8-row boxes for a ragged
    // tail); scales by one bulk copy (8 bytes a row, rounded up to 16).
    const uint64_t kv_policy = l2_policy_evict_first();
    auto issue = [&](const AttnItem& it, int k, int parts) {
        const long row = a.row0 + ((long)it.slot * a.nkv + it.kvh) * a.cap + (long)it.s * AT_C;
        const bool full = it.n == AT_C;
        const int qrows = full ? AT_C : (it.n + 7) / 8 * 8;
        const uint32_t sbytes = (uint32_t)((it.n * L::SROW + 15) / 16 * 16);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            if (!((parts >> part) & 1)) continue;
            const int st = part ? k % SV : k % SK;
            uint64_t* b = &bar[part * SK + st];
            const CUtensorMap* tm = part ? &tmv : &tmk;
            const CUtensorMap* tm8 = part ? &tmv8 : &tmk8;
            const __half* sc = part ? a.vs : a.ks;
            stage_item[part * SK + st] = k;
            mbar_arrive_expect_tx(b, (uint32_t)(qrows * L::QROW) + sbytes);
            uint8_t* dq = smem + (part ? L::VQ_OFF : L::KQ_OFF) + st * L::TILE;
            if (full)
                tma_load_2d_hint(dq, tm, 0, (int)row, b, kv_policy);
            else
                for (int k8 = 0; k8 < qrows; k8 += 8) tma_load_2d_hint(dq + k8 * L::QROW, tm8, 0, (int)row + k8, b, kv_policy);
            bulk_g2s_hint(smem + (part ? L::VS_OFF : L::KS_OFF) + st * L::STILE, sc + row * L::NBLK, sbytes, b,
                          kv_policy);
        }
    };

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        prefetch_tmap(&tmk8);
        prefetch_tmap(&tmv8);
    }
    // History items (not holding this step's new row) are fetched before the wait.
    unsigned early = 0;
    auto first_parts = [&](int k) { return (k < SK ? 1 : 0) | (k < SV ? 2 : 0); };
    for (int i = 0, k = warp; k < SMAX && k < nk; ++i, k += W) {
        const AttnItem it = tab.item(a, lane, gitem(k));
        if (it.s != it.ns - 1) {
            if (lane == 0) issue(it, k, first_parts(k));
            early |= 1u << i;
        }
    }
    pdl_launch_dependents();  // dependents may become resident now; they still wait for this grid
    pdl_wait();
    tl_waited(a.tl);
    for (int i = 0, k = warp; k < SMAX && k < nk; ++i, k += W)
        if (!((early >> i) & 1u)) {
            const AttnItem it = tab.item(a, lane, gitem(k));
            if (lane == 0) issue(it, k, first_parts(k));
        }

    // MMA columns as in the fp16 kernel: column 2h + part of N-tile j is head 4j + h,
    // part 0 the fp16 rounding of q (then p), part 1 the remainder.
    constexpr int NQ = GQ > 4 ? GQ / 4 : 1;
    const int colh = g >> 1;
    const float cf = (g & 1) ? 1.0f : 0.0f;                // f2_part: the lane's part
    const uint32_t sgn = (g & 1) ? 0x80000000u : 0u;
    // q of the lane's column head: per 32-dim block blk and 16-dim half hf, dims
    // 32 blk + 16 hf + 4c .. + 3 (the k order of the quants' A operand)
    float4 qv[NQ][4][2];
    auto load_q = [&](const AttnItem& it) {
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const int h = 4 * j + colh;
            if (h < GQ) {
                const float* qp = a.q + ((size_t)it.b * a.nh + (size_t)it.kvh * GQ + h) * HD + 4 * c;
#pragma unroll
                for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) qv[j][blk][hf] = *reinterpret_cast<const float4*>(qp + 32 * blk + 16 * hf);
            }
        }
    };
    uint32_t qb[NQ][4][2][2];  // B fragments of Qᵀ: [blk][half][b0, b1]
    auto make_qb = [&]() {
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const bool on = 4 * j + colh < GQ;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float4 u = qv[j][blk][hf];
                    qb[j][blk][hf][0] = !on ? 0u : f2_part(u.x, u.y, cf, sgn);
                    qb[j][blk][hf][1] = !on ? 0u : f2_part(u.z, u.w, cf, sgn);
                }
        }
    };
    // The warp's next item and its q fragments: made once the scores no longer
    // need this item's.
    AttnItem it_next{};
    if (warp < nk) {
        it_next = tab.item(a, lane, gitem(warp));
        load_q(it_next);
        make_qb();
    }

    for (int k = warp; k < nk; k += W) {
        const AttnItem it = it_next;
        const int kst = k % SK, vst = k % SV;
        const uint32_t kq = smem_u32(smem + L::KQ_OFF + kst * L::TILE);
        const uint8_t* kscale = smem + L::KS_OFF + kst * L::STILE;
        const uint32_t vq = smem_u32(smem + L::VQ_OFF + vst * L::TILE);
        const uint8_t* vscale = smem + L::VS_OFF + vst * L::STILE;

        bool ok = wait_value(stage_item + kst, k);
        ok = ok && mbar_wait_bounded(&bar[kst], (uint32_t)(k / SK) & 1u);  // the K part
        if (__any_sync(FULL_MASK, !ok)) {
            if (lane == 0) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                *cta_failed = 1;
            }
            break;
        }
        const int n = it.n;

        // ---- scores: per 16-key tile m and 32-dim block, two MMAs, then the keys' block scales
        float sacc[AT_KT][NQ][4];
#pragma unroll
        for (int m = 0; m < AT_KT; ++m)
#pragma unroll
            for (int j = 0; j < NQ; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) sacc[m][j][i] = 0.0f;
#pragma unroll
        for (int m = 0; m < AT_KT; ++m) {
            const uint2 s0 = *reinterpret_cast<const uint2*>(kscale + (16 * m + g) * L::SROW);
            const uint2 s1 = *reinterpret_cast<const uint2*>(kscale + (16 * m + g + 8) * L::SROW);
            const float2 d0p[2] = {h2bits_to_float2(s0.x), h2bits_to_float2(s0.y)};  // key 16m + g, blocks 0..3
            const float2 d1p[2] = {h2bits_to_float2(s1.x), h2bits_to_float2(s1.y)};  // key 16m + g + 8
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kq + L::qoff(16 * m + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * blk + (lane >> 4)), r0, r1, r2, r3);
                const uint32_t a0 = u8x2_lo_to_half2(r0), a2 = u8x2_hi_to_half2(r0);
                const uint32_t a1 = u8x2_lo_to_half2(r1), a3 = u8x2_hi_to_half2(r1);
                const uint32_t e0 = u8x2_lo_to_half2(r2), e2 = u8x2_hi_to_half2(r2);
                const uint32_t e1 = u8x2_lo_to_half2(r3), e3 = u8x2_hi_to_half2(r3);
                const float d0 = (blk & 1) ? d0p[blk >> 1].y : d0p[blk >> 1].x;
                const float d1 = (blk & 1) ? d1p[blk >> 1].y : d1p[blk >> 1].x;
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
                    float t[4];
                    mma_16816_zero(t, a0, a1, a2, a3, qb[j][blk][0][0], qb[j][blk][0][1]);
                    mma_16816_acc(t, e0, e1, e2, e3, qb[j][blk][1][0], qb[j][blk][1][1]);
                    sacc[m][j][0] = __fmaf_rn(d0, t[0], sacc[m][j][0]);
                    sacc[m][j][1] = __fmaf_rn(d0, t[1], sacc[m][j][1]);
                    sacc[m][j][2] = __fmaf_rn(d1, t[2], sacc[m][j][2]);
                    sacc[m][j][3] = __fmaf_rn(d1, t[3], sacc[m][j][3]);
                }
            }
        }
        // The K part is read: refill it with item k + S's.
        __syncwarp();
        if (k + SK < nk) {
            const AttnItem nx = tab.item(a, lane, gitem(k + SK));
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(nx, k + SK, 1);
            }
        }
        if (k + W < nk) {
            it_next = tab.item(a, lane, gitem(k + W));
            load_q(it_next);
            make_qb();
        }
        // ---- softmax over the item's keys (as in the fp16 kernel)
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

        // The V part.
        ok = wait_value(stage_item + SK + vst, k);
        ok = ok && mbar_wait_bounded(&bar[SK + vst], (uint32_t)(k / SV) & 1u);
        if (__any_sync(FULL_MASK, !ok)) {
            if (lane == 0) {
                atomicOr(a.err, ERR_WAIT_TIMEOUT);
                *cta_failed = 1;
            }
            break;
        }

        // p d_t,blk would fall below fp16's normal range for small p: the item's
        // products carry an exact power-of-two factor 2^e, taken from its largest
        // value scale so that p d 2^e < 2^14, and the output drops it again in fp32.
        float pscale = 1.0f, pinv = 1.0f;
        {
            const uint4 w = lds_v4(vscale + 2 * lane * L::SROW);  // rows 2 lane, 2 lane + 1
            float dm = 0.0f;
            if (2 * lane < n) {
                const float2 x = h2bits_to_float2(w.x), y = h2bits_to_float2(w.y);
                dm = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(y.x), fabsf(y.y)));
            }
            if (2 * lane + 1 < n) {
                const float2 x = h2bits_to_float2(w.z), y = h2bits_to_float2(w.w);
                dm = fmaxf(dm, fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(y.x), fabsf(y.y))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) dm = fmaxf(dm, __shfl_xor_sync(FULL_MASK, dm, o));
            if (dm > 0.0f && dm <= 65504.0f) {
                // dm in [2^(E-127), 2^(E-126)): e = 140 - E, within [-2, 37] for fp16 scales
                const int e = 140 - ((__float_as_int(dm) >> 23) & 0xff);
                pscale = __int_as_float((127 + e) << 23);
                pinv = __int_as_float((127 - e) << 23);
            }
        }

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
                // Pᵀ per block: keys 2c, 2c + 1 (+ 8) of the lane's column head, each p
                // times its key's block scale (0 past the item's keys)
                // keys kb, kb + 1 and kb + 8, kb + 9: two 16-byte rows pairs of scales
                const int kb = 16 * js + 2 * c;
                const uint4 wa = lds_v4(vscale + kb * L::SROW), wb = lds_v4(vscale + (kb + 8) * L::SROW);
                float2 dk[4][2];  // [key r][blocks 0,1 | 2,3]; 0 past the item's keys
                dk[0][0] = h2bits_to_float2(kb < n ? wa.x : 0u);
                dk[0][1] = h2bits_to_float2(kb < n ? wa.y : 0u);
                dk[1][0] = h2bits_to_float2(kb + 1 < n ? wa.z : 0u);
                dk[1][1] = h2bits_to_float2(kb + 1 < n ? wa.w : 0u);
                dk[2][0] = h2bits_to_float2(kb + 8 < n ? wb.x : 0u);
                dk[2][1] = h2bits_to_float2(kb + 8 < n ? wb.y : 0u);
                dk[3][0] = h2bits_to_float2(kb + 9 < n ? wb.z : 0u);
                dk[3][1] = h2bits_to_float2(kb + 9 < n ? wb.w : 0u);
                uint32_t pb[4][NQ][2];
#pragma unroll
                for (int j = 0; j < NQ; ++j) {
                    const float v00 = __fmul_rn(__shfl_sync(FULL_MASK, sv[j][js][0], src0), pscale);
                    const float v01 = __fmul_rn(__shfl_sync(FULL_MASK, sv[j][js][0], src1), pscale);
                    const float v10 = __fmul_rn(__shfl_sync(FULL_MASK, sv[j][js][1], src0), pscale);
                    const float v11 = __fmul_rn(__shfl_sync(FULL_MASK, sv[j][js][1], src1), pscale);
                    const bool on = 4 * j + colh < GQ;
#pragma unroll
                    for (int blk = 0; blk < 4; ++blk) {
                        auto dsc = [&](int r) { return (blk & 1) ? dk[r][blk >> 1].y : dk[r][blk >> 1].x; };
                        const float p0 = __fmul_rn(v00, dsc(0)), p1 = __fmul_rn(v01, dsc(1));
                        const float p2 = __fmul_rn(v10, dsc(2)), p3 = __fmul_rn(v11, dsc(3));
                        pb[blk][j][0] = !on ? 0u : f2_part(p0, p1, cf, sgn);
                        pb[blk][j][1] = !on ? 0u : f2_part(p2, p3, cf, sgn);
                    }
                }
                // per 32-dim block: keys 0-7 / 8-15 of its two 16-dim slices, transposed
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_trans(vq + L::qoff(16 * js + (lane & 7) + ((lane >> 3) & 1) * 8, 2 * blk + (lane >> 4)), r0,
                                  r1, r2, r3);
                    const uint32_t s0a0 = u8x2_even_to_half2(r0), s0a1 = u8x2_odd_to_half2(r0);
                    const uint32_t s0a2 = u8x2_even_to_half2(r1), s0a3 = u8x2_odd_to_half2(r1);
                    const uint32_t s1a0 = u8x2_even_to_half2(r2), s1a1 = u8x2_odd_to_half2(r2);
                    const uint32_t s1a2 = u8x2_even_to_half2(r3), s1a3 = u8x2_odd_to_half2(r3);
#pragma unroll
                    for (int j = 0; j < NQ; ++j) {
                        mma_16816_acc(oacc[2 * blk][j], s0a0, s0a1, s0a2, s0a3, pb[blk][j][0], pb[blk][j][1]);
                        mma_16816_acc(oacc[2 * blk + 1][j], s1a0, s1a1, s1a2, s1a3, pb[blk][j][0], pb[blk][j][1]);
                    }
                }
            }
        }
        // ---- both parts of head 4j + c, dims 16 mt + 2g and 16 mt + 2g + 1: write (o, m, l)
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const int h = 4 * j + c;
            if (h < GQ) {
                float* dst = a.part + (((size_t)it.b * a.nh + (size_t)it.kvh * GQ + h) * a.max_splits + it.s) *
                                          ATT_REC(HD);
#pragma unroll
                for (int mt = 0; mt < NU / 2; ++mt)
                    *reinterpret_cast<float2*>(dst + 16 * mt + 2 * g) =
                        make_float2(__fmul_rn(__fadd_rn(oacc[mt][j][0], oacc[mt][j][1]), pinv),
                                    __fmul_rn(__fadd_rn(oacc[mt][j][2], oacc[mt][j][3]), pinv));
                if (g == 0) *reinterpret_cast<float2*>(dst + HD) = make_float2(mx[j], lsum[j]);
            }
        }
        __syncwarp();  // the V part is read: refill it
        if (k + SV < nk) {
            const AttnItem nx = tab.item(a, lane, gitem(k + SV));
            if (lane == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(nx, k + SV, 2);
            }
        }
    }
    // After a wait gave up, copies may still be in flight: before the CTA's shared
    // memory is released, wait (bounded) for the last item issued into each part.
    __syncthreads();
    if (threadIdx.x == 0 && *cta_failed)
        for (int i = 0; i < SK + SV; ++i) {
            const int k = stage_item[i];
            if (k >= 0) (void)mbar_wait_bounded(&bar[i], (uint32_t)(k / (i < SK ? SK : SV)) & 1u);
        }
    tl_exit(a.tl);
}

// ---- quantisation ------------------------------------------------------------
// One warp per 32-value block, a lane per value: d = max|x| / 127 (fp32), stored
// as fp16; q = x / d rounded half away from zero, within [-127, 127]; 0 for an
// all-zero block.  Returns the stored quant byte u = q + 128.
__device__ __forceinline__ uint8_t q8_quant_lane(float x, int lane, __half* scale_out) {
    float amax = fabsf(x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, o));
    const float d = __fdiv_rn(amax, 127.0f);
    int q = 0;
    if (d > 0.0f) q = max(-127, min(127, (int)roundf(__fdiv_rn(x, d))));
    if (lane == 0) *scale_out = __float2half_rn(d);
    return (uint8_t)(q + 128);
}

// The step's new K and V rows (fp32 [B][nkv][128], from the q|k|v epilogue) into
// the Q8_0 arenas at (slot[b], pos[b]).  Block (h, b): warp w quantises block
// w & 3 of K (w < 4) or of V (w >= 4).
__global__ void __launch_bounds__(256) kvq8_append_kernel(const float* __restrict__ knew, const float* __restrict__ vnew,
                                                          uint8_t* kq, __half* ks, uint8_t* vq, __half* vs,
                                                          const int* slot, const int* pos, int nkv, int cap, long row0) {
    pdl_launch_dependents();
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = warp & 3, part = warp >> 2;
    const long row = row0 + ((long)slot[b] * nkv + h) * cap + pos[b];
    const float x = (part ? vnew : knew)[((size_t)b * nkv + h) * 128 + 32 * blk + lane];
    uint8_t* q = (part ? vq : kq) + row * 128 + 32 * blk + lane;
    *q = q8_quant_lane(x, lane, (part ? vs : ks) + row * 4 + blk);
}

// Rows of fp32 or fp16 values [n_rows][128] into Q8_0 rows: source row r (layer
// l = r / (nkv * len), head h, position t) goes to arena row
// l * layer_rows + base + h * cap + t.  A warp per 32-value block.
template <typename T>
__global__ void __launch_bounds__(128) kvq8_rows_kernel(const T* __restrict__ src, long n_rows, int nkv, int len,
                                                        int cap, long layer_rows, long base, uint8_t* q, __half* sc) {
    const long r = blockIdx.x;
    if (r >= n_rows) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long lh = r / len;
    const int t = (int)(r - lh * len);
    const long l = lh / nkv;
    const int h = (int)(lh - l * nkv);
    const long row = l * layer_rows + base + (long)h * cap + t;
    float x;
    if constexpr (sizeof(T) == 2)
        x = __half2float(reinterpret_cast<const __half*>(src)[r * 128 + 32 * warp + lane]);
    else
        x = src[r * 128 + 32 * warp + lane];
    q[row * 128 + 32 * warp + lane] = q8_quant_lane(x, lane, sc + row * 4 + warp);
}

cudaError_t launch_kvq8_append(const float* knew, const float* vnew, uint8_t* kq, __half* ks, uint8_t* vq, __half* vs,
                               const int* slot, const int* pos, int B, int nkv, int cap, long row0, bool pdl,
                               cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3(nkv, B);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, kvq8_append_kernel, knew, vnew, kq, ks, vq, vs, slot, pos, nkv, cap, row0);
}

cudaError_t launch_kvq8_rows(const void* src, bool src_fp16, long n_rows, int nkv, int len, int cap, long layer_rows,
                             long base, uint8_t* q, __half* sc, cudaStream_t s) {
    if (n_rows <= 0) return cudaSuccess;
    if (n_rows > 0x7fffffffL) return cudaErrorInvalidValue;
    if (src_fp16)
        kvq8_rows_kernel<__half><<<(unsigned)n_rows, 128, 0, s>>>(reinterpret_cast<const __half*>(src), n_rows, nkv, len,
                                                                 cap, layer_rows, base, q, sc);
    else
        kvq8_rows_kernel<float><<<(unsigned)n_rows, 128, 0, s>>>(reinterpret_cast<const float*>(src), n_rows, nkv, len,
                                                                cap, layer_rows, base, q, sc);
    return cudaGetLastError();
}

// ---- tensor maps and launch -------------------------------------------------------
typedef CUresult (*EncodeTiledQ8Fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static cudaError_t encode_u8_rows(CUtensorMap* out, const void* base, long rows, int box_rows) {
    static EncodeTiledQ8Fn encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult qr;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
        if (e != cudaSuccess) return e;
        if (qr != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<EncodeTiledQ8Fn>(fn);
    }
    if (rows < 1 || rows > 0x7fffffffL || (reinterpret_cast<uintptr_t>(base) & 15)) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {128, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t estr[2] = {1, 1};
    const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_attn_q8_maps(const uint8_t* kq, const uint8_t* vq, long rows, AttnMaps* out) {
    cudaError_t e;
    if ((e = encode_u8_rows(&out->k, kq, rows, ATT_CHUNK)) != cudaSuccess) return e;
    if ((e = encode_u8_rows(&out->k8, kq, rows, 8)) != cudaSuccess) return e;
    if ((e = encode_u8_rows(&out->v, vq, rows, ATT_CHUNK)) != cudaSuccess) return e;
    return encode_u8_rows(&out->v8, vq, rows, 8);
}

bool attn_q8_supported(int hd, int group) {
    return hd == AttnQ8Smem::HD && (group == 1 || group == 2 || group == 4 || group == 8);
}

cudaError_t attn_q8_init_attributes() {
    cudaError_t e = cudaSuccess;
    for (const void* f : {(const void*)attn_split_q8_kernel<1>, (const void*)attn_split_q8_kernel<2>,
                          (const void*)attn_split_q8_kernel<4>, (const void*)attn_split_q8_kernel<8>}) {
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnQ8Smem::TOTAL)) != cudaSuccess)
            return e;
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return e;
    }
    for (const void* f : {(const void*)kvq8_append_kernel, (const void*)kvq8_rows_kernel<__half>,
                          (const void*)kvq8_rows_kernel<float>})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
            return e;
    return cudaSuccess;
}

cudaError_t launch_attn_split_q8(const AttnArgs& a, const AttnMaps& maps, int grid, bool pdl, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(AttnQ8Smem::warps(a.nh / a.nkv) * 32);
    cfg.dynamicSmemBytes = AttnQ8Smem::TOTAL;
    cfg.stream = s;
    switch (a.nh / a.nkv) {
        case 1: return cudaLaunchKernelEx(&cfg, attn_split_q8_kernel<1>, a, maps.k, maps.k8, maps.v, maps.v8);
        case 2: return cudaLaunchKernelEx(&cfg, attn_split_q8_kernel<2>, a, maps.k, maps.k8, maps.v, maps.v8);
        case 4: return cudaLaunchKernelEx(&cfg, attn_split_q8_kernel<4>, a, maps.k, maps.k8, maps.v, maps.v8);
        case 8: return cudaLaunchKernelEx(&cfg, attn_split_q8_kernel<8>, a, maps.k, maps.k8, maps.v, maps.v8);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kd
