// kd_mmvq.cu -- Q8_0 weight-only matrix x (m <= 16) activations: the device
// weight layout (repack), the choice of schedule per matrix, and dispatch.
//
// This is the batched mmvq of memra-engine's decode_batch.rs (module header):
// every projection at m = B reads the weights once for all B rows, and each row
// is bit-identical to its m = 1 result.  Two schedules share one arithmetic
// (kd_mmvq_common.cuh): "group" (kd_mmvq_cta.cu) when a matrix's 32-row groups
// spread evenly over the SMs, "stream" (kd_mmvq_stream.cu) otherwise.  The
// choice, and every split of K, depends on the matrix shape and the SM count only.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "kd_mmvq_common.cuh"

namespace kd {

cudaError_t mmvq_stream_init_attributes();
cudaError_t mmvq_cta_init_attributes();
cudaError_t launch_mmvq_stream(const MmvqArgs& a, const CUtensorMap& xm, int epi, bool pdl, cudaStream_t s);
cudaError_t launch_mmvq_cta(const MmvqArgs& a, const CUtensorMap& xm, int epi, int num_sms, bool pdl, cudaStream_t s);


// The group schedule keeps a row group's reduction in one CTA's shared memory;
// it is used when the groups spread evenly over the SMs: at most two per SM
// (one CTA per group), or up to eight per SM when the busiest SM has at most 5%
// more groups than the average.  Otherwise the stream schedule balances stages.
static int choose_mode(int G, int num_sms) {
    if (G <= 2 * num_sms) return MMVQ_GROUP;
    const long most = (long)((G + num_sms - 1) / num_sms) * num_sms;  // groups the busiest SM's share implies
    if (G <= 8 * num_sms && most * 100 <= 105L * G) return MMVQ_GROUP;
    return MMVQ_STREAM;
}

void plan_split(PackedQ8& m, int num_sms, int force_mode) {
    m.mode = force_mode >= 0 ? force_mode : choose_mode(m.G, num_sms);
    // stream: W warps, each a contiguous run of the T = G * KG stages; W never
    // exceeds T, so every warp owns at least one stage.
    const long T = (long)m.G * m.KG;
    m.W = (int)std::min<long>((long)num_sms * MMVQ_WARPS, T);
    int maxc = 1;
    if (m.mode == MMVQ_STREAM)
        for (int g = 0; g < m.G; ++g) {
            const long t0 = (long)g * m.KG, t1 = t0 + m.KG - 1;
            const int w0 = (int)(((t0 + 1) * m.W - 1) / T), w1 = (int)(((t1 + 1) * m.W - 1) / T);
            maxc = std::max(maxc, w1 - w0 + 1);
        }
    m.maxc = maxc;
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

cudaError_t mmvq_init_attributes() {
    cudaError_t e = mmvq_stream_init_attributes();
    if (e != cudaSuccess) return e;
    return mmvq_cta_init_attributes();
}

cudaError_t launch_mmvq(const MmvqArgs& a, const CUtensorMap& xmap, int mode, int epi, int num_sms, bool pdl,
                        cudaStream_t s) {
    if (mode == MMVQ_GROUP) return launch_mmvq_cta(a, xmap, epi, num_sms, pdl, s);
    return launch_mmvq_stream(a, xmap, epi, pdl, s);
}

}  // namespace kd
