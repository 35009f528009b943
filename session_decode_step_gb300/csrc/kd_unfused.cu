// kd_unfused.cu -- the step's epilogue operations as kernels of their own, for
// the unfused launch train (KD_FLAG_UNFUSED): each projection stores its plain
// fp32 result y (rows in the packed matrix's order: row group g holds its first
// 16-row tile at 32g .. 32g + 15 and its second at 32g + 16 .. 32g + 31), and
// one of these kernels then applies what the fused epilogue would have:
//   RoPE + KV append (after q|k|v), SwiGLU (after gate|up), the residual add
//   and the next norm's per-group sums of squares (after o-proj and down).
// They call the same per-element arithmetic as the fused epilogues, so the two
// trains give the same bits; the tests check that they do.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kd_mmvq_common.cuh"

namespace kd {

// (session n, row pair rr of group g) of a paired matrix: y rows 32g + rr and 32g + 16 + rr.
__global__ void __launch_bounds__(256) pair_epilogue_kernel(const MmvqArgs a, const float* __restrict__ y, int ldy,
                                                            int epi) {
    const int e = blockIdx.x * blockDim.x + threadIdx.x;  // over B x G x 16
    const int n = e / (a.G * TILE_ROWS), rem = e - n * (a.G * TILE_ROWS);
    const int g = rem / TILE_ROWS, rr = rem - g * TILE_ROWS;
    if (n >= a.B) return;
    const float v0 = y[(size_t)n * ldy + (size_t)g * GROUP_ROWS + rr];
    const float v1 = y[(size_t)n * ldy + (size_t)g * GROUP_ROWS + TILE_ROWS + rr];
    if (epi == EPI_SWIGLU)
        epi_swiglu(a, g, rr, n, v0, v1);
    else
        epi_qkv(a, g, rr, n, v0, v1);
}

// The residual add of row group g for session n (a warp, a lane per row), and
// the group's sum of squares of the new rows by the fused epilogue's tree.
__global__ void __launch_bounds__(256) resid_epilogue_kernel(const MmvqArgs a, const float* __restrict__ y, int ldy) {
    const int lane = threadIdx.x & 31;
    const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);  // over B x G
    const int n = w / a.G, g = w - n * a.G;
    if (n >= a.B) return;
    const float v = y[(size_t)n * ldy + (size_t)g * GROUP_ROWS + lane];
    const float x = epi_resid(a, g, lane, n, v);
    float s = __fmul_rn(x, x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(FULL_MASK, s, o));
    if (lane == 0) a.ssq_out[(size_t)g * NORM_SLOTS + n] = s;
}

cudaError_t launch_unfused_epilogue(const MmvqArgs& a, const float* y, int ldy, int epi, cudaStream_t s) {
    if (epi == EPI_RESID) {
        const int warps = a.B * a.G;
        resid_epilogue_kernel<<<(warps + 7) / 8, 256, 0, s>>>(a, y, ldy);
    } else if (epi == EPI_SWIGLU || epi == EPI_QKV) {
        const int n = a.B * a.G * TILE_ROWS;
        pair_epilogue_kernel<<<(n + 255) / 256, 256, 0, s>>>(a, y, ldy, epi);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kd
