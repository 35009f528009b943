// kd_device.cuh -- small sm_103a device helpers shared by the decode-step kernels:
// mbarrier + bulk-copy (TMA 1-D) staging, the legacy warp-level f16 MMA, exact
// int8 -> fp16 conversion, programmatic-dependent-launch controls, bounded waits.
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

#include "kd_kernels.h"

namespace kd {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Device fault word bits (kd_device_status reports them).
constexpr int ERR_WAIT_TIMEOUT = 1;   // a bounded mbarrier wait ran out

// Bounded waits: give up after this many polls or this much wall time, whichever
// comes first.  A healthy wait ends in microseconds.
constexpr uint32_t WAIT_MAX_POLLS = 1u << 24;
constexpr uint64_t WAIT_MAX_NS = 500ull * 1000ull * 1000ull;  // 0.5 s

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- timeline (kd_profile_timeline): optional per-CTA stamps ------------------
// A launch's records are [TL_CTAS][TL_WORDS] u64: the global timer (ns) at the
// CTA's entry, when its dependency wait returned, the latest end over its
// warps, and its SM id.  tl == nullptr (the normal case) costs one test.

__device__ __forceinline__ unsigned long long* tl_rec(unsigned long long* tl) {
    const unsigned cta = blockIdx.y * gridDim.x + blockIdx.x;
    return cta < (unsigned)TL_CTAS ? tl + (size_t)cta * TL_WORDS : nullptr;
}
__device__ __forceinline__ void tl_entry(unsigned long long* tl) {
    if (tl && threadIdx.x == 0) {
        unsigned long long* r = tl_rec(tl);
        if (r) {
            unsigned sm;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
            r[0] = global_timer_ns();
            r[3] = sm;
        }
    }
}
__device__ __forceinline__ void tl_waited(unsigned long long* tl) {
    if (tl && threadIdx.x == 0) {
        unsigned long long* r = tl_rec(tl);
        if (r) r[1] = global_timer_ns();
    }
}
// Called by every warp as it finishes (lane 0 stamps; the record keeps the latest).
__device__ __forceinline__ void tl_exit(unsigned long long* tl) {
    if (tl && (threadIdx.x & 31) == 0) {
        unsigned long long* r = tl_rec(tl);
        if (r) atomicMax(r + 2, (unsigned long long)global_timer_ns());
    }
}

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Raise the byte count the barrier's current phase waits for, without an
// arrival (the debug fault hook: a phase that expects more bytes than its
// copies deliver never completes, so the bounded wait on it runs out).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Poll until the barrier's phase with this parity completes, or give up (false).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < WAIT_MAX_POLLS; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 255u && global_timer_ns() - t0 > WAIT_MAX_NS) break;
    }
    return false;
}

// ---- bulk copy global -> shared (TMA, 1-D), completion counted on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tensor-map tile load (TMA): tile at element coordinates (x, y) of the map
// (x innermost, x * element size a multiple of 16 bytes) into dst (aligned as the
// map's swizzle requires), completing on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// The same with an L2 cache policy for the copied lines (l2_policy_*).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Fetch a tensor map's descriptor ahead of its first copy (the map itself never
// depends on an earlier kernel, so this can run before the dependency wait).
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// The first 1024-byte boundary at or after p (tiles written with the 128-byte
// swizzle need it; dynamic shared memory is only guaranteed 16-byte alignment).
__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Same, with an L2 eviction-priority hint (for data read exactly once per step).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- programmatic dependent launch ----------------------------------------
// Wait until the grids this one depends on have completed and flushed memory.
// A no-op when the kernel was launched without the PDL attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream start launching (its pre-wait prologue).
// Issued before this kernel's own wait: the dependent grid is only scheduled
// once every CTA of this grid is resident, and its griddepcontrol.wait still
// waits for this grid to complete, so the order of work is unchanged while the
// dependent's weight prefetch can start on SMs this grid leaves free.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- RMSNorm from per-group sums of squares -----------------------------------
// r = 1 / sqrt(sum_g ssq[g][b] / H + eps) for the H/32 groups a residual writer
// left: lane l adds groups l, l + 32, ... in order (the first add is exact),
// then a fixed shuffle tree; every lane returns the same value.  The RMSNorm
// kernel (rms_factor_from_ssq) and the fused activation load
// (rms_factor_from_parts, with the lane's values loaded ahead: groups
// lane + 32 i, i < 4, for H <= 4096) do exactly this arithmetic.
__device__ __forceinline__ float rms_factor_from_parts(const float (&pre)[NORM_IN_MAX_KG], int lane, int H, float eps) {
    const int ng = H / 32;
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < NORM_IN_MAX_KG; ++i)
        if (lane + 32 * i < ng) s = __fadd_rn(s, pre[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)H), eps)));
}
__device__ __forceinline__ void rms_parts_load(const float* ssq, int b, int lane, int H, float (&pre)[NORM_IN_MAX_KG]) {
    const int ng = H / 32;
#pragma unroll
    for (int i = 0; i < NORM_IN_MAX_KG; ++i)
        pre[i] = lane + 32 * i < ng ? __ldcg(ssq + (size_t)(lane + 32 * i) * MAX_NORM_SLOTS + b) : 0.0f;
}

// The sums read through `get(g)`: from global memory (the norm kernel) or from
// the shared-memory copy the embedding kernel keeps of the sums it wrote.
template <class Get>
__device__ __forceinline__ float rms_factor_of(Get get, int lane, int H, float eps) {
    const int ng = H / 32;
    float s = 0.0f;
    for (int g = lane; g < ng; g += 32) s = __fadd_rn(s, get(g));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)H), eps)));
}
__device__ __forceinline__ float rms_factor_from_ssq(const float* ssq, int b, int lane, int H, float eps) {
    return rms_factor_of([&](int g) { return __ldcg(ssq + (size_t)g * MAX_NORM_SLOTS + b); }, lane, H, eps);
}

// Device-scope atomic add with acquire-release semantics: the writes this CTA
// ordered before it (through a barrier) are visible to a CTA that reads the
// counter afterwards, and that CTA's later accesses see every write released
// into the counter before.
__device__ __forceinline__ unsigned atomic_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ---- the pick: greedy argmax and Gumbel-max sampling ---------------------------
// Each (value, index) maps to a 64-bit key whose unsigned order is the pick
// order -- larger value first, then lower index; -0 counts as +0; NaN maps to 0
// and never wins -- so partial picks merge with a maximum, in any order, with
// one result.
__device__ __forceinline__ unsigned long long argmax_key(float v, int i) {
    if (v != v) return 0ull;
    if (v == 0.0f) v = 0.0f;
    const unsigned u = __float_as_uint(v);
    const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(~(unsigned)i);
}

// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of two 64 x 64
// -> 128 multiplies mixing the four counter words with the key, the key bumped
// by the two Weyl constants between rounds.  Returns the block's four words.
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0,
                                              uint64_t k1, uint64_t (&w)[4]) {
    constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    constexpr uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += W0;
            k1 += W1;
        }
        const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0, hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
        const uint64_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    w[0] = c0; w[1] = c1; w[2] = c2; w[3] = c3;
}

// logit / T - log(-log u), u = (top 24 bits of w + 1/2) / 2^24 (exact, in (0, 1)).
__device__ __forceinline__ float gumbel_perturb(float logit, float T, uint64_t w) {
    const float u = __fmul_rn(__fadd_rn((float)(unsigned)(w >> 40), 0.5f), 0x1p-24f);
    const float g = -logf(-logf(u));
    return __fadd_rn(__fdiv_rn(logit, T), g);
}

// A row's sampling parameters in the staged descriptor block `samp`: the
// temperature's bits at [b], the seed at [16 + 2b] (low word first), the
// counter at [48 + 2b]; T <= 0 picks greedily.  Entry v of the row is perturbed
// by word v mod 4 of the Philox block at counter (v / 4, counter, 0, 0) under
// key (seed, 0).
struct PickParams {
    float T;
    uint64_t seed, ctr;
};
__device__ __forceinline__ PickParams pick_params(const int* samp, int b) {
    PickParams p{0.0f, 0, 0};
    if (!samp) return p;
    p.T = __int_as_float(samp[b]);
    p.seed = ((uint64_t)(unsigned)samp[17 + 2 * b] << 32) | (unsigned)samp[16 + 2 * b];
    p.ctr = ((uint64_t)(unsigned)samp[49 + 2 * b] << 32) | (unsigned)samp[48 + 2 * b];
    return p;
}

// ---- exact int8 -> fp16 ----------------------------------------------------
// The repacked weights hold u = q + 128 (0..255).  Placing u under the fp16
// exponent of 1024 gives the half 1024 + u exactly (the fp16 spacing there is
// 1); subtracting 1152 leaves q exactly.  This is the byte-permute /
// magic-number conversion published by Kim et al., "Who Says Elephants Can't
// Run: Bringing Large Scale MoE Models into Cloud Scale Production" (2022).
__device__ __forceinline__ uint32_t u8x2_lo_to_half2(uint32_t v) {  // bytes 0,1
    uint32_t h = __byte_perm(v, 0x64646464u, 0x4140);
    const uint32_t bias = 0x64806480u;  // half2(1152, 1152)
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(bias));
    return r;
}
__device__ __forceinline__ uint32_t u8x2_hi_to_half2(uint32_t v) {  // bytes 2,3
    uint32_t h = __byte_perm(v, 0x64646464u, 0x4342);
    const uint32_t bias = 0x64806480u;
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(bias));
    return r;
}

// ---- warp-level MMA: D = A(16x16 f16, row) * B(16x8 f16, col) + 0, f32 out --
__device__ __forceinline__ void mma_16816_zero(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_16816_acc(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint4 lds_v4(const void* p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_u32(p)));
    return r;
}

__device__ __forceinline__ float2 ldcg_f2(const float* p) { return __ldcg(reinterpret_cast<const float2*>(p)); }

}  // namespace kd
