// kd_mmvq_common.cuh -- device code shared by the two Q8_0 mmvq schedules
// (kd_mmvq_stream.cu: warps stream equal contiguous shares of the matrix;
// kd_mmvq_cta.cu: a CTA owns whole row groups and its warps split K).
//
// The arithmetic is identical in both and never depends on m (the number of
// activation rows): per 32-column Q8_0 block, the int8 quants are converted to
// fp16 exactly and multiplied on two m16n8k16 MMAs (fp32 accumulate) whose 8
// columns are 8 sessions; the block result is scaled by its fp16 scale with an
// fp32 FMA.  Only how many MMA columns are stored depends on m.
#pragma once
#include <cuda_fp16.h>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int RING = 4;        // weight stages in flight per warp
constexpr int NORM_SLOTS = MAX_NORM_SLOTS;

// One stage (one 128-column k-group of a 32-row group) into the accumulators.
// x: this lane's activation fragments for the stage's 4 blocks (k permutation
// of the packed layout); acc[mt][nt][i]: row mt*16 + gq (+8 for i >= 2),
// MMA column nt*8 + 2*cq + (i & 1), i.e. session nt*8 + col_session(2*cq + (i & 1)).
template <int NT>
__device__ __forceinline__ void mma_stage(const uint8_t* st, int lane, int gq, const uint4 (&x)[4][NT],
                                          float (&acc)[MT][NT][4]) {
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
                mma_16816_zero(t, a00, a01, a02, a03, x[kb][nt].x, x[kb][nt].y);
                mma_16816_acc(t, a10, a11, a12, a13, x[kb][nt].z, x[kb][nt].w);
                acc[mt][nt][0] = __fmaf_rn(d.x, t[0], acc[mt][nt][0]);
                acc[mt][nt][1] = __fmaf_rn(d.x, t[1], acc[mt][nt][1]);
                acc[mt][nt][2] = __fmaf_rn(d.y, t[2], acc[mt][nt][2]);
                acc[mt][nt][3] = __fmaf_rn(d.y, t[3], acc[mt][nt][3]);
            }
        }
    }
}

// ---- activation tiles -------------------------------------------------------
// A stage's activations arrive with its weights: the tensor-map copy of the
// [8 sessions][128 columns] fp16 tile for each 8 sessions, as two 64-column
// halves of [8 rows][128 B] with the 128-byte swizzle (16-byte chunk c of row r
// at chunk c ^ r), 1024-byte aligned.  Rows past the map's end read as zeros;
// rows >= B hold whatever the buffer holds and only feed MMA columns that are
// never stored.
constexpr int XTILE_BYTES = 2048;  // one stage, 8 sessions

template <int NT>
__device__ __forceinline__ void tma_x_tile(uint8_t* xt, const void* xmap, int kg, uint64_t* bar) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int h = 0; h < 2; ++h) tma_load_2d(xt + (nt * 2 + h) * 1024, xmap, kg * KGROUP + 64 * h, 8 * nt, bar);
}

// MMA column c (0..7) of an 8-session tile carries session col_session(c):
// the lanes of one shared-memory wavefront (gq = 2w, 2w + 1) then read tile
// rows w and w + 4, whose swizzled chunks fall in different bank halves.
// Which column holds a session changes nothing in its arithmetic.
__device__ __forceinline__ int col_session(int c) { return (c >> 1) | ((c & 1) << 2); }
__device__ __forceinline__ int session_col(int s) { return ((s & 3) << 1) | (s >> 2); }

// Lane (gq, cq) multiplies session 8*nt + col_session(gq) at columns 8cq .. 8cq+7
// of each 32-column block kb: the 16-byte chunk 4kb + cq of that session's row.
template <int NT>
__device__ __forceinline__ void lds_x_tile(const uint8_t* xt, int gq, int cq, uint4 (&xv)[4][NT]) {
    const int row = col_session(gq);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
            xv[kb][nt] = lds_v4(xt + (nt * 2 + (kb >> 1)) * 1024 + row * 128 + ((((kb & 1) * 4 + cq) ^ row) << 4));
}

// fp16(x * r * w) of two neighbouring elements, as an fp16 pair (first element low)
__device__ __forceinline__ uint32_t norm_pair(float x0, float x1, float r, float w0, float w1) {
    const __half2 t = __floats2half2_rn(__fmul_rn(__fmul_rn(x0, r), w0), __fmul_rn(__fmul_rn(x1, r), w1));
    return *reinterpret_cast<const uint32_t*>(&t);
}

// The fused activation load: this warp's normed input tiles for k-groups
// kg0 .. kg0 + nk - 1 (nk <= NORM_IN_MAX_KG), xn[s][k] = fp16(x[s][k] * r_s * w[k])
// for the launch's sessions (zero for the unused ones), written as the
// activation tensor map would deliver them: per k-group and 8 sessions, two
// 64-column halves of [8 rows][128 B], 16-byte chunk c of row r at chunk c ^ r.
// CTA-collective (every warp calls it, nk may be 0): warp 0 forms the sessions'
// norm factors r_s (rms_factor_from_ssq's order) into rsm[] while the other
// warps' x loads are in flight.  Lane (p, c) handles column chunk c (8 columns)
// of sessions p, p + 2, ...; two k-groups' loads are in flight at a time.
template <int NT>
__device__ __forceinline__ void norm_tiles(const MmvqArgs& a, int warp, int lane, int kg0, int nk, uint8_t* xt,
                                           float* rsm) {
    constexpr int SPL = 4 * NT;  // sessions per lane
    const int c = lane & 15, p = lane >> 4;
    float4 xv[2][SPL][2], wv[2][2];
    auto load = [&](int k0) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int kk = k0 + u;
            if (kk < nk) {
                const int col = (kg0 + kk) * KGROUP + 8 * c;
                wv[u][0] = __ldg(reinterpret_cast<const float4*>(a.nw + col));
                wv[u][1] = __ldg(reinterpret_cast<const float4*>(a.nw + col + 4));
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int s = p + 2 * j;
                    if (s < a.B) {
                        const float* xp = a.nx + (size_t)s * a.K + col;
                        xv[u][j][0] = __ldcg(reinterpret_cast<const float4*>(xp));
                        xv[u][j][1] = __ldcg(reinterpret_cast<const float4*>(xp + 4));
                    }
                }
            }
        }
    };
    load(0);
    if (warp == 0) {
        // r_s: lane l holds groups l, l + 32, l + 64, l + 96 of every session (a
        // sums-of-squares row is 16 sessions, 64 bytes), added in that order.
        const int ng = a.K / 32;
        float4 pre[NORM_IN_MAX_KG][2 * NT];
#pragma unroll
        for (int i = 0; i < NORM_IN_MAX_KG; ++i)
#pragma unroll
            for (int q = 0; q < 2 * NT; ++q)
                pre[i][q] = lane + 32 * i < ng
                                ? __ldcg(reinterpret_cast<const float4*>(a.nssq + (size_t)(lane + 32 * i) * MAX_NORM_SLOTS) + q)
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int q = 0; q < 2 * NT; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float sv = 0.0f;
#pragma unroll
                for (int i = 0; i < NORM_IN_MAX_KG; ++i) {
                    const float v = e == 0 ? pre[i][q].x : e == 1 ? pre[i][q].y : e == 2 ? pre[i][q].z : pre[i][q].w;
                    if (lane + 32 * i < ng) sv = __fadd_rn(sv, v);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sv = __fadd_rn(sv, __shfl_xor_sync(FULL_MASK, sv, o));
                if (lane == 0) rsm[4 * q + e] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(sv, (float)a.K), a.neps)));
            }
    }
    __syncthreads();
    float r[SPL];
#pragma unroll
    for (int j = 0; j < SPL; ++j) r[j] = rsm[p + 2 * j];
#pragma unroll
    for (int k0 = 0; k0 < NORM_IN_MAX_KG; k0 += 2) {
        if (k0 > 0) load(k0);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int kk = k0 + u;
            if (kk < nk) {
#pragma unroll
                for (int j = 0; j < SPL; ++j) {
                    const int s = p + 2 * j;
                    uint4 o = make_uint4(0u, 0u, 0u, 0u);
                    if (s < a.B) {
                        o.x = norm_pair(xv[u][j][0].x, xv[u][j][0].y, r[j], wv[u][0].x, wv[u][0].y);
                        o.y = norm_pair(xv[u][j][0].z, xv[u][j][0].w, r[j], wv[u][0].z, wv[u][0].w);
                        o.z = norm_pair(xv[u][j][1].x, xv[u][j][1].y, r[j], wv[u][1].x, wv[u][1].y);
                        o.w = norm_pair(xv[u][j][1].z, xv[u][j][1].w, r[j], wv[u][1].z, wv[u][1].w);
                    }
                    const int nt = s >> 3, rr = s & 7;
                    uint8_t* dst = xt + (size_t)kk * NT * XTILE_BYTES + (nt * 2 + (c >> 3)) * 1024 + rr * 128 +
                                   (((c & 7) ^ rr) << 4);
                    *reinterpret_cast<uint4*>(dst) = o;
                }
            }
        }
    }
}

// ---- epilogues on single outputs ------------------------------------------
// Row r (0..31) of row group g, session n, value v.
__device__ __forceinline__ void epi_store(const MmvqArgs& a, int g, int r, int n, float v) {
    a.y[(size_t)n * a.ld + (size_t)g * GROUP_ROWS + r] = v;
}
// Residual add; returns the updated value.
__device__ __forceinline__ float epi_resid(const MmvqArgs& a, int g, int r, int n, float v) {
    float* p = a.y + (size_t)n * a.ld + (size_t)g * GROUP_ROWS + r;
    const float x = __fadd_rn(*p, v);
    *p = x;
    return x;
}
// The same with the old value loaded ahead of time (resid_load).
__device__ __forceinline__ float resid_load(const MmvqArgs& a, int g, int r, int n) {
    return a.y[(size_t)n * a.ld + (size_t)g * GROUP_ROWS + r];
}
__device__ __forceinline__ float epi_resid_apply(const MmvqArgs& a, int g, int r, int n, float old, float v) {
    const float x = __fadd_rn(old, v);
    a.y[(size_t)n * a.ld + (size_t)g * GROUP_ROWS + r] = x;
    return x;
}
// Pair epilogues: tile 0 row r with tile 1 row r (r = 0..15).
//   SwiGLU: act = fp16(silu(gate) * up)
__device__ __forceinline__ void epi_swiglu(const MmvqArgs& a, int g, int r, int n, float gt, float up) {
    const float sg = __fdiv_rn(gt, __fadd_rn(1.0f, expf(-gt)));
    a.act[(size_t)n * a.ld + (size_t)g * TILE_ROWS + r] = __float2half_rn(__fmul_rn(sg, up));
}
//   QKV: dims (i, i + hd/2) of one head; RoPE at the row's position for q and k;
//   q to fp32, k and v appended to the session's slot at its position as fp16.
//   What it reads from global memory (the position, the slot, the cos/sin pair)
//   can be loaded ahead of time (qkv_load).
struct QkvIn {
    int p, slot;
    float2 cs;
};
__device__ __forceinline__ QkvIn qkv_load(const MmvqArgs& a, int g, int r, int n) {
    const int per_head = a.hd / GROUP_ROWS;
    const int head = g / per_head;
    const int dim = (g - head * per_head) * TILE_ROWS + r;
    QkvIn in;
    in.p = a.pos[n];
    in.slot = a.slot[n];
    in.cs = head < a.nh + a.nkv ? a.rope[(size_t)in.p * (a.hd >> 1) + dim] : make_float2(0.0f, 0.0f);
    return in;
}
__device__ __forceinline__ void epi_qkv_in(const MmvqArgs& a, int g, int r, int n, float x0, float x1, const QkvIn& in) {
    const int per_head = a.hd / GROUP_ROWS;
    const int head = g / per_head;
    const int dim = (g - head * per_head) * TILE_ROWS + r;
    const int half = a.hd >> 1;
    const int p = in.p;
    if (head < a.nh + a.nkv) {
        const float2 cs = in.cs;
        const float y0 = __fsub_rn(__fmul_rn(x0, cs.x), __fmul_rn(x1, cs.y));
        const float y1 = __fadd_rn(__fmul_rn(x0, cs.y), __fmul_rn(x1, cs.x));
        if (head < a.nh) {
            float* q = a.q_out + ((size_t)n * a.nh + head) * a.hd;
            q[dim] = y0;
            q[dim + half] = y1;
        } else if (a.k_out) {  // Q8_0 cache: the fp32 row, quantised by the append kernel
            float* k = a.k_out + ((size_t)n * a.nkv + (head - a.nh)) * a.hd;
            k[dim] = y0;
            k[dim + half] = y1;
        } else {
            __half* k = a.kc + (((size_t)in.slot * a.nkv + (head - a.nh)) * a.cap + p) * a.hd;
            k[dim] = __float2half_rn(y0);
            k[dim + half] = __float2half_rn(y1);
        }
    } else if (a.v_out) {
        float* vv = a.v_out + ((size_t)n * a.nkv + (head - a.nh - a.nkv)) * a.hd;
        vv[dim] = x0;
        vv[dim + half] = x1;
    } else {
        __half* vv = a.vc + (((size_t)in.slot * a.nkv + (head - a.nh - a.nkv)) * a.cap + p) * a.hd;
        vv[dim] = __float2half_rn(x0);
        vv[dim + half] = __float2half_rn(x1);
    }
}
__device__ __forceinline__ void epi_qkv(const MmvqArgs& a, int g, int r, int n, float x0, float x1) {
    epi_qkv_in(a, g, r, n, x0, x1, qkv_load(a, g, r, n));
}

}  // namespace kd
