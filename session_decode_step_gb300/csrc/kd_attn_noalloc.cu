// kd_attn_noalloc.cu -- kd_attn_append_decode without a workspace argument.
//
// Some callers cannot allocate device memory at the point where they decode:
// code running inside a memory pool or arena that owns every byte of the GPU,
// an embedding that forbids cudaMalloc/cudaFree on its hot path (both can
// synchronise the device and stall other streams), or a process whose allocator
// is not CUDA-aware.  For them this entry point keeps its scratch in one
// statically sized device array that the library holds from load to exit on
// every GPU it is used on, and performs no allocation of any kind: the session
// slots and positions travel to the device as kernel arguments, not through a
// host-to-device copy.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <string>

#include "kd.h"
#include "kd_kernels.h"

// The scratch: 256 bytes of descriptor (slots, positions, fault word), then the
// per-split partial results of the attention.  Every GPU that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char g_attn_scratch[KD_ATTN_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t DESC_BYTES = 256;
constexpr int MAX_DEVICES = 64;

// Per device, the scratch array's device address: stored only once the lookup
// has succeeded, so a failed lookup (a transient error, or a first call made
// during a stream capture) is retried by the next call.
std::mutex g_setup_mu;
void* g_scratch_ptr[MAX_DEVICES];

// Slots and positions arrive by value; the fault word must start at zero.
struct DescArgs {
    int slot[KD_MAX_BATCH];
    int pos[KD_MAX_BATCH];
};

__global__ void set_descriptor_kernel(const DescArgs d, int B, int* dst) {
    const int i = threadIdx.x;
    if (i < KD_MAX_BATCH) {
        dst[i] = i < B ? d.slot[i] : 0;
        dst[KD_MAX_BATCH + i] = i < B ? d.pos[i] : 0;
    }
    if (i == 0) dst[2 * KD_MAX_BATCH] = 0;  // fault word of this call
}

kd_status fail(kd_status st, const std::string& msg) {
    kd::set_last_error(msg.c_str());  // reported by kd_last_error()
    return st;
}

// The array's device address on device `dev` (current), looked up on first use.
kd_status scratch_address(int dev, cudaStream_t s, void** out) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone)
            return fail(KD_ERR_INVALID_ARG,
                        "kd_attn_append_decode_noalloc: the first call on a device looks up the scratch "
                        "array's address and must not be made during a stream capture");
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return fail(KD_ERR_CUDA, std::string("kd_attn_append_decode_noalloc: cudaGetSymbolAddress: ") +
                                         cudaGetErrorString(e));
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KD_OK;
}

}  // namespace

cudaError_t kd::noalloc_fault_word(int dev, int** out) {
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    *out = g_scratch_ptr[dev] ? reinterpret_cast<int*>(g_scratch_ptr[dev]) + 2 * KD_MAX_BATCH : nullptr;
    return cudaSuccess;
}

extern "C" kd_status kd_attn_append_decode_noalloc(const float* q, const float* k_new, const float* v_new,
                                                   uint16_t* k_cache, uint16_t* v_cache, const int32_t* slots,
                                                   const int32_t* positions, int32_t B, int32_t n_heads,
                                                   int32_t n_kv_heads, int32_t head_dim, int32_t n_slots,
                                                   int32_t cap, uint16_t* out, kd_stream stream) {
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !slots || !positions || !out)
        return fail(KD_ERR_INVALID_ARG, "kd_attn_append_decode_noalloc: null argument");
    if (B < 1 || B > KD_MAX_BATCH) return fail(KD_ERR_BATCH, "kd_attn_append_decode_noalloc: B out of range");
    if (n_kv_heads < 1 || n_heads < 1 || n_heads % n_kv_heads ||
        !kd::attn_supported(head_dim, n_heads / n_kv_heads))
        return fail(KD_ERR_UNSUPPORTED, "kd_attn_append_decode_noalloc: unsupported head layout");
    if (n_slots < 1 || cap < 1) return fail(KD_ERR_INVALID_ARG, "kd_attn_append_decode_noalloc: n_slots/cap");
    const size_t splits = (size_t)(cap + kd::ATT_CHUNK - 1) / kd::ATT_CHUNK;
    if (splits > (size_t)kd::ATT_MAX_SPLITS)
        return fail(KD_ERR_UNSUPPORTED, "kd_attn_append_decode_noalloc: cap too large");
    const size_t need = DESC_BYTES + (size_t)B * n_heads * splits * kd::ATT_REC(head_dim) * sizeof(float);
    if (need > (size_t)KD_ATTN_NOALLOC_SCRATCH_BYTES)
        return fail(KD_ERR_UNSUPPORTED,
                    "kd_attn_append_decode_noalloc: B * n_heads * ceil(cap/64) * (head_dim + 4) * 4 + 256 = " +
                        std::to_string(need) + " bytes exceeds the fixed scratch of " +
                        std::to_string((size_t)KD_ATTN_NOALLOC_SCRATCH_BYTES) + " bytes");
    if (((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) ||
        (reinterpret_cast<uintptr_t>(q) & 7))
        return fail(KD_ERR_INVALID_ARG, "kd_attn_append_decode_noalloc: caches must be 16-byte aligned, q 8-byte");
    DescArgs d{};
    for (int b = 0; b < B; ++b) {
        if (slots[b] < 0 || slots[b] >= n_slots) return fail(KD_ERR_BAD_SESSION, "slot out of range");
        for (int j = 0; j < b; ++j)
            if (slots[j] == slots[b]) return fail(KD_ERR_BAD_SESSION, "slot repeated");
        if (positions[b] < 0 || positions[b] >= cap) return fail(KD_ERR_POSITION, "position out of range");
        d.slot[b] = slots[b];
        d.pos[b] = positions[b];
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return fail(KD_ERR_CUDA, "kd_attn_append_decode_noalloc: no current CUDA device");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Once per device, with it current: the scratch array's device address.  In
    // host code the array's name only stands in for it.
    void* scratch = nullptr;
    const kd_status st = scratch_address(dev, s, &scratch);
    if (st != KD_OK) return st;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        kd::ensure_device_attributes(dev) != cudaSuccess)
        return fail(KD_ERR_CUDA, "kd_attn_append_decode_noalloc: device set-up failed");
    kd::AttnMaps maps;
    if (kd::make_attn_maps(reinterpret_cast<const __half*>(k_cache), reinterpret_cast<const __half*>(v_cache),
                           (long)n_slots * n_kv_heads * cap, head_dim, &maps) != cudaSuccess)
        return fail(KD_ERR_CUDA, "kd_attn_append_decode_noalloc: tensor map encoding failed");
    int* desc = reinterpret_cast<int*>(scratch);
    cudaError_t e;
    set_descriptor_kernel<<<1, 32, 0, s>>>(d, B, desc);
    if ((e = cudaGetLastError()) != cudaSuccess) return fail(KD_ERR_CUDA, cudaGetErrorString(e));
    if ((e = kd::launch_kv_append(k_new, v_new, reinterpret_cast<__half*>(k_cache), reinterpret_cast<__half*>(v_cache),
                                  desc, desc + KD_MAX_BATCH, B, n_kv_heads, head_dim, cap, s)) != cudaSuccess)
        return fail(KD_ERR_CUDA, cudaGetErrorString(e));
    kd::AttnArgs t{};
    t.q = q;
    t.kc = reinterpret_cast<const __half*>(k_cache);
    t.vc = reinterpret_cast<const __half*>(v_cache);
    t.row0 = 0;
    t.slot = desc;
    t.pos = desc + KD_MAX_BATCH;
    t.B = B;
    t.nh = n_heads;
    t.nkv = n_kv_heads;
    t.hd = head_dim;
    t.cap = cap;
    t.scale = 1.0f / sqrtf((float)head_dim);
    t.part = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(scratch) + DESC_BYTES);
    t.max_splits = (int)splits;
    t.out = reinterpret_cast<__half*>(out);
    t.err = desc + 2 * KD_MAX_BATCH;
    if ((e = kd::launch_attn_split(t, maps, kd::attn_split_grid(sms, head_dim, n_heads / n_kv_heads), false, s)) !=
        cudaSuccess)
        return fail(KD_ERR_CUDA, cudaGetErrorString(e));
    if ((e = kd::launch_attn_combine(t, false, s)) != cudaSuccess) return fail(KD_ERR_CUDA, cudaGetErrorString(e));
    return KD_OK;
}
