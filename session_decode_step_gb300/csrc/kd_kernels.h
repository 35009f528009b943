// kd_kernels.h -- host-side launch interface of the decode-step kernels (library internal).
#pragma once
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kd {

// ---------------------------------------------------------------------------
// Q8_0 weight layout on the device ("packed").
//
// A matrix of N rows and K columns is cut into tiles of 16 rows and k-groups
// of 128 columns.  Tiles come in pairs (a "group" of MT = 2 tiles) that one
// warp multiplies together, so a group's two tiles share every activation
// fragment.  Which source rows form a group is chosen per matrix: consecutive
// rows for plain projections, (gate, up) row tiles for the SwiGLU pair, and
// rows (i, i + head_dim/2) of one head for the RoPE pair.
//
// For one (group, k-group) the bytes are MT x 2176:
//   per tile: 4 sub-blocks (one Q8_0 block of 32 columns each) x 32 lanes x 16 B
//   of quants stored as u = q + 128, laid out so that lane L = 4*g + c holds
//   the 8 quants of row g and of row g + 8 at columns 8c .. 8c+7 of the block
//   (exactly the A fragments of two m16n8k16 MMAs, after a fixed permutation of
//   the k index that the activation fragments share); then 8 x 16 B of scales:
//   for g = 0..7, the fp16 pairs (d[g], d[g+8]) of the 4 sub-blocks.
// Groups are stored k-group-contiguous: offset ((group * KG + kg) * MT + mt) * 2176.
// ---------------------------------------------------------------------------
constexpr int TILE_ROWS = 16;
constexpr int MT = 2;
constexpr int KGROUP = 128;
constexpr int TILE_KG_BYTES = 2176;
constexpr int STAGE_BYTES = MT * TILE_KG_BYTES;
constexpr int GROUP_ROWS = MT * TILE_ROWS;

enum Epilogue : int {
    EPI_STORE = 0,   // y[n][row] = v
    EPI_RESID = 1,   // x[n][row] += v (fp32 residual stream)
    EPI_SWIGLU = 2,  // act[n][i] = fp16(silu(gate_i) * up_i)
    EPI_QKV = 3,     // RoPE q and k at each row's position, q to fp32, k/v appended as fp16
};

struct PackedQ8 {
    uint8_t* w = nullptr;   // packed bytes
    int rows = 0, K = 0;    // logical shape
    int G = 0, KG = 0;      // groups of 32 rows, k-groups of 128 columns
    int kpt = 1, S = 1;     // k-groups per task, k-splits (S = KG / kpt)
    size_t bytes() const { return (size_t)G * KG * STAGE_BYTES; }
    size_t part_floats() const { return S > 1 ? (size_t)G * S * GROUP_ROWS * 16 : 0; }
};

// Pick the split of K into tasks for an N x K matrix; depends on the shape only.
void choose_split(PackedQ8& m);

// Repack a canonical Q8_0 matrix already on the device.  tile_src[t] is the
// first source row of packed tile t (G * MT entries, device memory).
cudaError_t launch_repack(const uint8_t* src, int K, const int* tile_src, int G, uint8_t* dst,
                          cudaStream_t s);

struct MmvqArgs {
    const uint8_t* w;
    int G, KG, kpt, S, K;
    const __half* x;     // [B][K] fp16 activations
    int B;
    float* part;         // split-K partials
    int* cnt;            // [G] arrival counters, zero between launches
    int* err;            // device fault word
    int ld;              // row stride (elements) of the epilogue output
    float* y;            // EPI_STORE / EPI_RESID target
    __half* act;         // EPI_SWIGLU target
    // EPI_QKV
    float* q_out;        // [B][nh][hd]
    __half* kc;          // this layer's K arena [slots][nkv][cap][hd]
    __half* vc;
    const int* slot;     // [B]
    const int* pos;      // [B]
    const float2* rope;  // [max_ctx][hd/2] (cos, sin)
    int nh, nkv, hd, cap;
};

cudaError_t launch_mmvq(const MmvqArgs& a, int epi, int num_sms, bool pdl, cudaStream_t s);
size_t mmvq_smem_bytes();
cudaError_t mmvq_init_attributes();

// ---- attention -------------------------------------------------------------
constexpr int ATT_CHUNK = 128;  // keys per split; fixed, so a session's splits depend on its length only

struct AttnArgs {
    const float* q;       // [B][nh][hd] fp32, rotated
    const __half* kc;     // this layer's arenas [slots][nkv][cap][hd] fp16
    const __half* vc;
    const int* slot;      // [B]
    const int* pos;       // [B]; the row attends keys 0..pos
    int B, nh, nkv, hd, cap;
    float scale;
    float* part;          // [B][nh][max_splits][hd + 2]
    int max_splits;
    __half* out;          // [B][nh*hd]
    int* err;
};

bool attn_supported(int hd, int group);
cudaError_t launch_attn_split(const AttnArgs& a, int grid, bool pdl, cudaStream_t s);
cudaError_t launch_attn_combine(const AttnArgs& a, bool pdl, cudaStream_t s);
int attn_split_grid(int num_sms, int hd, int group);
cudaError_t attn_init_attributes();

// Append fp32 k/v rows [B][nkv][hd] to the fp16 arenas at (slot[b], pos[b]).
cudaError_t launch_kv_append(const float* k, const float* v, __half* kc, __half* vc, const int* slot,
                             const int* pos, int B, int nkv, int hd, int cap, cudaStream_t s);

// ---- row ops -----------------------------------------------------------------
// x[b][:] = dequant(tok_embd[token[b]])  (canonical Q8_0 rows)
cudaError_t launch_embed(const uint8_t* tok_embd, const int* token, int B, int H, float* x,
                         bool pdl, cudaStream_t s);
// out[b][i] = fp16(x[b][i] / sqrt(mean(x[b]^2) + eps) * w[i])
cudaError_t launch_rmsnorm(const float* x, const float* w, __half* out, int B, int H, float eps,
                           bool pdl, cudaStream_t s);
// out[b] = argmax_v logits[b][v] (ties -> lowest v, NaN never wins, -1 if none)
cudaError_t launch_argmax(const float* logits, int B, int V, int* out, bool pdl, cudaStream_t s);

}  // namespace kd
