// kd_attn_common.cuh -- pieces shared by the split-K attention kernels over
// fp16 KV (kd_attn.cu) and over Q8_0 KV (kd_attn_q8.cu): the work-item table,
// ldmatrix wrappers, the fp16 hi/lo split, bounded polls.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_device.cuh"
#include "kd_kernels.h"

namespace kd {

constexpr int AT_C = ATT_CHUNK;  // keys per work item (split)
constexpr int AT_WARPS = 8;      // consumer warps per CTA (two per SM sub-partition)
constexpr int AT_KT = AT_C / 16;  // 16-key tiles (and 16-key steps) of a work item
static_assert(AT_C % 16 == 0 && AT_C <= 64, "a work item is whole 16-key tiles, at most 4");

// Work items are ordered session-major, then split, then KV head.
struct AttnItem {
    int b, s, kvh, n, ns, slot;  // session, split, KV head, keys in this split, splits of the session, its slot
};

// The session table of a launch, held one session per lane (B <= 32): the
// session's slot, position, split count and first item.  Built once per warp
// from the step's descriptor; an item's session is then found by a ballot over
// the lanes' first items, with no memory access.
struct AttnTable {
    int slot, pos, ns, base, n_items;
    __device__ __forceinline__ void build(const AttnArgs& a, int lane) {
        slot = lane < a.B ? a.slot[lane] : 0;
        pos = lane < a.B ? a.pos[lane] : 0;
        ns = lane < a.B ? (pos + ATT_CHUNK) / ATT_CHUNK : 0;  // ceil((pos+1)/C)
        int incl = ns * a.nkv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(FULL_MASK, incl, o);
            if (lane >= o) incl += v;
        }
        base = incl - ns * a.nkv;
        n_items = __shfl_sync(FULL_MASK, incl, 31);
    }
    // Warp-uniform item index (< n_items); every lane gets the same answer.
    __device__ __forceinline__ AttnItem item(const AttnArgs& a, int lane, int x) const {
        const unsigned m = __ballot_sync(FULL_MASK, lane < a.B && base <= x);
        const int b = 31 - __clz(m);
        AttnItem it;
        it.b = b;
        const int r = x - __shfl_sync(FULL_MASK, base, b);
        it.s = r / a.nkv;
        it.kvh = r - it.s * a.nkv;
        it.n = min(ATT_CHUNK, __shfl_sync(FULL_MASK, pos, b) + 1 - it.s * ATT_CHUNK);
        it.ns = __shfl_sync(FULL_MASK, ns, b);
        it.slot = __shfl_sync(FULL_MASK, slot, b);
        return it;
    }
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                              uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// fp32 pair -> fp16 pair (low half = first element), and the fp16 pair of what
// that rounding left over: hi + lo carries about 22 significant bits.
__device__ __forceinline__ uint32_t f2_hi(float x, float y) {
    const __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t f2_lo(float x, float y) {
    const __half2 h = __floats2half2_rn(x, y);
    const float2 f = __half22float2(h);
    const __half2 l = __floats2half2_rn(__fsub_rn(x, f.x), __fsub_rn(y, f.y));
    return *reinterpret_cast<const uint32_t*>(&l);
}

// Bounded poll of a shared-memory word until it holds v (false: gave up).
__device__ __forceinline__ bool wait_value(const volatile int* p, int v) {
    if (*p == v) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; i < WAIT_MAX_POLLS; ++i) {
        if (*p == v) return true;
        if ((i & 255u) == 255u && global_timer_ns() - t0 > WAIT_MAX_NS) break;
    }
    return false;
}

}  // namespace kd
