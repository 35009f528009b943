// kd_kernels.h -- host-side launch interface of the decode-step kernels (library internal).
#pragma once
#include <cuda.h>
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
    EPI_PICK = 4,    // EPI_STORE, and the rows' pick from the stored values (stream schedule only)
};

// Timeline records (kd_profile_timeline): per launch [TL_CTAS][TL_WORDS] u64.
constexpr int TL_CTAS = 1024;
constexpr int TL_WORDS = 4;

constexpr int MAX_NORM_SLOTS = 16;  // sum-of-squares tables hold one entry per session slot 0..15
// The fused-norm activation load keeps a warp's whole k-range of normed tiles in
// shared memory: at most this many 128-column k-groups per warp (K <= 4096).
constexpr int NORM_IN_MAX_KG = 4;

enum MmvqMode : int {
    MMVQ_STREAM = 0,  // warps stream equal contiguous shares; partials of shared groups via global memory
    MMVQ_GROUP = 1,   // a CTA owns whole row groups; its warps split K and reduce in shared memory
};

struct PackedQ8 {
    uint8_t* w = nullptr;   // packed bytes
    int rows = 0, K = 0;    // logical shape
    int G = 0, KG = 0;      // groups of 32 rows, k-groups of 128 columns
    int mode = MMVQ_STREAM; // schedule (depends on the shape and SM count only)
    int W = 1;              // stream: warps streaming it (one contiguous stage range each)
    int maxc = 1;           // stream: most warps sharing one row group
    size_t bytes() const { return (size_t)G * KG * STAGE_BYTES; }
    size_t part_floats() const { return mode == MMVQ_STREAM && maxc > 1 ? (size_t)G * maxc * GROUP_ROWS * 16 : 0; }
};

// Split a matrix's stages over the warps of a grid of num_sms CTAs; depends on
// the shape and the SM count only.
// force_mode: -1 = choose from the shape, else MMVQ_STREAM / MMVQ_GROUP.
void plan_split(PackedQ8& m, int num_sms, int force_mode = -1);

// Repack a canonical Q8_0 matrix already on the device.  tile_src[t] is the
// first source row of packed tile t (G * MT entries, device memory).
cudaError_t launch_repack(const uint8_t* src, int K, const int* tile_src, int G, uint8_t* dst,
                          cudaStream_t s);

constexpr int MMVQ_WARPS = 8;  // warps per mmvq CTA

// Tensor map of fp16 data viewed as [rows][inner] (128-byte swizzle, box of
// box_rows x box_inner, zero fill outside); base 16-byte aligned, inner * 2 a
// multiple of 16.
cudaError_t encode_fp16_2d(CUtensorMap* out, const void* base, long inner, long rows, int box_inner, int box_rows);
// The activation map an mmvq launch reads its input x [rows][K] through: boxes
// of 8 rows x 64 columns (each stage loads 2 per 8 sessions).
inline cudaError_t make_x_map(const __half* x, int K, int rows, CUtensorMap* out) {
    return encode_fp16_2d(out, x, K, rows, 64, 8);
}

struct MmvqArgs {
    const uint8_t* w;
    int G, KG, W, maxc, K;
    const __half* x;     // [B][K] fp16 activations (the kernels read them through the launch's map of x)
    int B;
    // EPI_RESID: each group's writer also leaves sum(x_new^2) of its 32 rows per
    // session in ssq_out[g][n], so the next RMSNorm needs no row reduction.
    float* ssq_out;      // [G][16]
    float* part;         // split-K partials
    int* cnt;            // [G] arrival counters, zero between launches
                         // (part: [G][maxc][32 rows][16 columns] fp32)
    int* err;            // device fault word
    // Debug fault hook (0 in normal use): extra bytes the first stage of CTA 0,
    // warp 0 waits for, so that its bounded wait runs out (no copy is touched).
    int inject_tx;
    unsigned long long* tl;  // timeline records of this launch, or nullptr
    // RMSNorm fused into the activation load (group schedule only; nx == nullptr
    // otherwise): x is then xn = fp16(nx * r_b * nw), r_b = 1 / sqrt(sum_g
    // nssq[g][b] / K + neps), formed by each warp for its own k-groups once, in
    // the RMSNorm kernel's order and roundings (the same bits as that kernel).
    const float* nx;     // [B][K] fp32 residual rows
    const float* nssq;   // [K/32][16] per-group sums of squares the residual writer left
    const float* nw;     // [K] norm weight
    float neps;
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
    // Q8_0 KV cache: the epilogue leaves the rotated k and v rows in fp32
    // [B][nkv][hd] here (quantised into the arena by launch_kvq8_append) instead
    // of writing fp16 rows into kc / vc.
    float* k_out;
    float* v_out;
    // EPI_PICK: each row's pick (launch_argmax's result, from the stored values)
    // fused into the store; keys, done and samp as launch_argmax takes them.
    unsigned long long* pick_keys;
    unsigned* pick_done;
    int* pick_out;
    const int* samp;
};

// xmap: make_x_map of a.x with at least B rows.
cudaError_t launch_mmvq(const MmvqArgs& a, const CUtensorMap& xmap, int mode, int epi, int num_sms, bool pdl,
                        cudaStream_t s);
// Smallest dynamic shared memory any mmvq launch needs (for occupancy checks).
cudaError_t mmvq_init_attributes();
// The unfused train: apply epilogue `epi` (EPI_QKV, EPI_SWIGLU or EPI_RESID, with
// a's epilogue fields) to a projection's plain result y [B][ldy] (rows in the
// packed order), as the fused epilogue does.
cudaError_t launch_unfused_epilogue(const MmvqArgs& a, const float* y, int ldy, int epi, cudaStream_t s);

// ---- attention -------------------------------------------------------------
constexpr int ATT_CHUNK = 64;        // keys per split; fixed, so a session's splits depend on its length only
constexpr int ATT_MAX_SPLITS = 1024;  // longest context: 1024 * 64 = 65536 positions
// One split's partial result per (session, head): o[hd], then m, l, and padding
// to a 16-byte multiple so every record starts 16-byte aligned.
__host__ __device__ constexpr int ATT_REC(int hd) { return hd + 4; }

struct AttnArgs {
    const float* q;       // [B][nh][hd] fp32, rotated
    const __half* kc;     // this layer's arenas [slots][nkv][cap][hd] fp16
    const __half* vc;
    long row0;            // this layer's first row in the tensor maps ([rows][hd] over the whole arenas)
    const int* slot;      // [B]
    const int* pos;       // [B]; the row attends keys 0..pos
    int B, nh, nkv, hd, cap;
    float scale;
    float* part;          // [B][nh][max_splits][ATT_REC(hd)]
    int max_splits;
    __half* out;          // [B][nh*hd]
    int* err;
    int inject_tx;        // debug fault hook (0 in normal use): extra bytes item 0's K tile waits for
    unsigned long long* tl;  // timeline records of this launch (split or combine), or nullptr
    // Q8_0 KV cache: this layer's block-scale planes [rows][hd/32] fp16 (the
    // quants are read through the tensor maps); unused with fp16 KV.
    const __half* ks;
    const __half* vs;
};

// Tensor maps over the K and V arenas, each viewed as [rows][hd] fp16: 64-row
// boxes and 8-row boxes (ragged tails) of 64-dim halves, 128-byte swizzle.
struct AttnMaps {
    CUtensorMap k, k8, v, v8;
};
cudaError_t make_attn_maps(const __half* k_arena, const __half* v_arena, long rows, int hd, AttnMaps* out);

bool attn_supported(int hd, int group);
cudaError_t launch_attn_split(const AttnArgs& a, const AttnMaps& maps, int grid, bool pdl, cudaStream_t s);
cudaError_t launch_attn_combine(const AttnArgs& a, bool pdl, cudaStream_t s);
int attn_split_grid(int num_sms, int hd, int group);
cudaError_t attn_init_attributes();

// ---- Q8_0 KV cache (head_dim 128) -----------------------------------------------
// Arena rows are 128 quant bytes u = q + 128 ([rows][128] uint8) and 4 fp16
// block scales ([rows][4]); per 32-value block d = max|x| / 127 (fp32) stored as
// fp16, q = x / d rounded half away from zero within [-127, 127].
bool attn_q8_supported(int hd, int group);
cudaError_t attn_q8_init_attributes();
cudaError_t make_attn_q8_maps(const uint8_t* kq, const uint8_t* vq, long rows, AttnMaps* out);
cudaError_t launch_attn_split_q8(const AttnArgs& a, const AttnMaps& maps, int grid, bool pdl, cudaStream_t s);
// The step's new rows (fp32 [B][nkv][128]) into the arenas at row0 + (slot*nkv + h)*cap + pos.
cudaError_t launch_kvq8_append(const float* knew, const float* vnew, uint8_t* kq, __half* ks, uint8_t* vq, __half* vs,
                               const int* slot, const int* pos, int B, int nkv, int cap, long row0, bool pdl,
                               cudaStream_t s);
// n_rows source rows [n_rows][128] (fp16 or fp32, device) of a [layers][nkv][len]
// block into arena rows l * layer_rows + base + h * cap + t.
cudaError_t launch_kvq8_rows(const void* src, bool src_fp16, long n_rows, int nkv, int len, int cap, long layer_rows,
                             long base, uint8_t* q, __half* sc, cudaStream_t s);

// Append fp32 k/v rows [B][nkv][hd] to the fp16 arenas at (slot[b], pos[b]).
cudaError_t launch_kv_append(const float* k, const float* v, __half* kc, __half* vc, const int* slot,
                             const int* pos, int B, int nkv, int hd, int cap, cudaStream_t s);

// ---- row ops -----------------------------------------------------------------
// x[b][:] = dequant(tok_embd[token[b]])  (canonical Q8_0 rows) and, as a residual
// writer leaves them, the per-group sums of squares ssq[g][b] of those rows;
// with w (nullable), also xn[b][:] = the RMSNorm of x[b] with weight w, bit for
// bit what launch_norm_from_ssq would then form
cudaError_t launch_embed(const uint8_t* tok_embd, const int* token, int B, int H, float* x, float* ssq,
                         const float* w, float eps, __half* xn, bool pdl, cudaStream_t s,
                         unsigned long long* tl = nullptr);
// ssq[g][b] = sum of x[b][32g .. 32g+31]^2 for rows supplied from outside, in
// the residual writers' group layout and summation order
cudaError_t launch_ssq_rows(const float* x, int B, int H, float* ssq, cudaStream_t s);
// The same norm from the per-group sums of squares ssq[g][b] (g < H/32) a
// residual writer left: elementwise, spread over many CTAs.
cudaError_t launch_norm_from_ssq(const float* x, const float* ssq, int B, int H, const float* w, float eps,
                                 __half* xn, bool pdl, cudaStream_t s, unsigned long long* tl = nullptr);
cudaError_t rowops_init_attributes();
// out[b] = argmax_v logits[b][v] (ties -> lowest v, NaN never wins, -1 if none).
// keys [>= B] and done: device scratch that is zero before the first launch;
// every launch leaves it zero again.  V must be a multiple of 4.
// samp (nullable, device, SAMP_INTS words): per-row temperature sampling --
// words [0, 16) the rows' temperatures (fp32 bits; <= 0 greedy), [16 + 2b, 17 + 2b]
// row b's seed (low, high 32 bits), [48 + 2b, 49 + 2b] its counter.  A row with
// temperature T > 0 takes the argmax of logit / T plus Gumbel noise from
// Philox4x64-10 (see kd_sample_params in kd.h).
constexpr int SAMP_INTS = 80;
cudaError_t launch_argmax(const float* logits, int B, int V, int* out, unsigned long long* keys, unsigned* done,
                          bool pdl, cudaStream_t s, unsigned long long* tl = nullptr, const int* samp = nullptr);

// Device address of the allocation-free attention call's fault word on device
// dev, or nullptr if that call has not run on the device yet.
cudaError_t noalloc_fault_word(int dev, int** out);

// Set the calling thread's last-error message (what kd_last_error() returns).
void set_last_error(const char* msg);
// Kernel attributes (shared-memory sizes, carveouts) of device dev, set once.
cudaError_t ensure_device_attributes(int dev);

}  // namespace kd
