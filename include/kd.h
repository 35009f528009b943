/*
 * kd.h -- C ABI of the batched multi-session decode step for GB300 (sm_103a).
 *
 * One decode step runs B independent sessions (1 <= B <= 16) through one
 * fused forward pass of a dense, Llama-shaped decoder with Q8_0 weights.  Each
 * session owns a slot of the fp16 KV arena and sits at its own position; every
 * weight matrix is streamed from HBM once per step for all B rows.  This is
 * the batched decode step of memra-engine's `decode_batch.rs` (module header:
 * several sequences go through one fused pass that reads the weights once, and
 * each row's result must not depend on the batch; `decode_step_batch`)
 * restated for one GB300: one process, one GPU, no collectives.
 *
 * Conventions for every function:
 *   - Returns KD_OK (0) or a negative kd_status.  Nothing aborts, nothing
 *     throws across the ABI; the reason for the last failure on the calling
 *     thread is available from kd_last_error().
 *   - Arguments are validated on the host before any work is enqueued, so a
 *     call that fails leaves every piece of state as it was.
 *   - "device" pointers are CUDA device (or managed) addresses on the current
 *     device; "host" pointers are ordinary CPU memory.
 *   - A kd_stream is a cudaStream_t passed as void*; NULL is the legacy
 *     default stream.  Work is enqueued on it and the call returns without
 *     waiting, unless the function says otherwise.
 *   - A model handle is not thread-safe: callers serialise calls on it.
 */
#ifndef KD_H_
#define KD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kd_status;
enum {
    KD_OK = 0,
    KD_ERR_INVALID_ARG = -1,   /* null pointer, bad size, bad shape */
    KD_ERR_OOM = -2,           /* device or pinned-host allocation failed */
    KD_ERR_CUDA = -3,          /* a CUDA runtime call failed (message has the CUDA error) */
    KD_ERR_NO_FREE_SLOT = -4,  /* every session slot is bound */
    KD_ERR_BAD_SESSION = -5,   /* id out of range, not bound, or repeated within one step */
    KD_ERR_POSITION = -6,      /* position < 0, > the session's length, or >= max_ctx */
    KD_ERR_BATCH = -7,         /* B < 1, or above what the call accepts (see each call) */
    KD_ERR_UNSUPPORTED = -8,   /* a shape the kernels do not implement (see kd_config) */
    KD_ERR_DEVICE = -9         /* a kernel reported a device-side fault (bounded wait ran out) */
};

/* The widest batch one launch train takes: memra refuses B > 16 because above
 * it its kernels change numeric configuration and rows are no longer exact
 * (decode_batch.rs, module header).  kd_decode_step takes larger batches as
 * consecutive groups of at most KD_MAX_BATCH rows on the same kernels, so
 * every row stays exact. */
#define KD_MAX_BATCH 16

typedef void* kd_stream;          /* cudaStream_t */
typedef struct kd_model kd_model; /* opaque, library-owned */

/* Model shape.  Requirements (else KD_ERR_UNSUPPORTED): hidden, ffn and
 * n_heads*head_dim are multiples of 128; hidden is at most 131072 (the
 * embedding kernel stages a whole row on chip); head_dim is 64 or 128; n_heads is
 * 1, 2, 4 or 8 times n_kv_heads; vocab is a multiple of 32; max_ctx is at
 * most 65536.  All sizes and max_sessions, max_ctx are >= 1 (else
 * KD_ERR_INVALID_ARG).
 * rope_theta is the NeoX RoPE base; rms_eps the RMSNorm epsilon. */
typedef struct {
    int32_t n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, vocab;
    float rope_theta, rms_eps;
    int32_t max_sessions;   /* KV slots in the arena */
    int32_t max_ctx;        /* positions per slot (the slot capacity) */
    int32_t flags;          /* KD_FLAG_* */
} kd_config;

#define KD_FLAG_NO_GRAPH 1  /* launch each kernel every step instead of replaying a CUDA graph */
/* Force one projection schedule for every matrix (coverage testing; results stay
 * exact per row for every B, but the fp32 summation order differs between the
 * two schedules).  Default: chosen per matrix from its shape and the SM count. */
#define KD_FLAG_SCHEDULE_STREAM 2
#define KD_FLAG_SCHEDULE_GROUP 4
/* Fold the RMSNorm before q|k|v and gate|up into those projections' activation
 * load (each warp forms its k-range of the normed input from the fp32 residual
 * and the per-group sums of squares) instead of running it as a kernel of its
 * own.  The results are bit-identical either way.  Off by default: on GB300 the
 * folded load (every CTA reading the whole fp32 residual before its first MMA)
 * measured slower than the separate kernel, whose latency overlaps the next
 * projection's weight prefetch. */
#define KD_FLAG_FUSED_NORM 32
/* The unfused train: every projection stores its plain fp32 result, and RoPE +
 * KV append, SwiGLU and the residual add with the norm's sums of squares run
 * as kernels of their own.  Bit-identical to the fused epilogues; for testing
 * and measurement. */
#define KD_FLAG_UNFUSED 64
/* The KV cache in Q8_0 (the long-context option; memra appends quantised K/V in
 * `decode_batch_layers` phase A, hf2q ADR-040 measures llama.cpp with q8_0
 * K/V): each cached head row is 128 quants and 4 fp16 block scales (136 bytes
 * instead of 256).  Per 32-value block d = max|x| / 127 in fp32, stored as
 * fp16(d); q = x / d rounded half away from zero within [-127, 127]; value =
 * q * fp16(d).  New rows are quantised from the step's fp32 k (after RoPE) and
 * v; kd_session_load_kv quantises its fp16 input the same way.  Needs
 * head_dim 128 and an even max_ctx (else KD_ERR_UNSUPPORTED). */
#define KD_FLAG_KV_Q8_0 128

/* Host weights.  Matrices are canonical Q8_0: row-major [rows][cols/32] blocks
 * of {fp16 scale d (little-endian); int8 q[32]} (34 bytes), value = q * d, the
 * blocks running along the input dimension.  Per-layer arrays hold n_layers
 * pointers.  Shapes ([rows][cols]): tok_embd and output [vocab][hidden];
 * wq [n_heads*head_dim][hidden]; wk, wv [n_kv_heads*head_dim][hidden];
 * wo [hidden][n_heads*head_dim]; w_gate, w_up [ffn][hidden]; w_down [hidden][ffn];
 * norms fp32 [hidden].  The library copies everything; the caller may free the
 * host memory once kd_model_load returns. */
typedef struct {
    const void* tok_embd;
    const void* output;
    const float* output_norm;
    const void* const* wq;
    const void* const* wk;
    const void* const* wv;
    const void* const* wo;
    const void* const* w_gate;
    const void* const* w_up;
    const void* const* w_down;
    const float* const* attn_norm;
    const float* const* ffn_norm;
} kd_weights;

/* Copy and repack the weights into device memory and allocate the KV arena
 * (2 * n_layers * max_sessions * n_kv_heads * max_ctx * head_dim fp16) and the
 * step workspaces.  Synchronous.  On success *out owns all of it.
 * The model is the state every step shares: memra decode_batch.rs
 * `decode_step_batch(&self, e, tokens, caches)` reads one set of weights for
 * all B rows (module header: the weights are streamed once per step), while
 * each session's KV lives apart from them.  The arena is a fixed number of
 * slots of a fixed capacity each, as in hf2q ADR-040 section 0.0 ("Full-context
 * slot correction": `--max-slots` slots, each with the whole configured
 * context; weights and compute scratch kept apart from the slots' KV).
 * Errors: KD_ERR_INVALID_ARG / KD_ERR_UNSUPPORTED for a bad or unsupported
 * shape (checked before any CUDA call), KD_ERR_OOM if device or pinned memory
 * runs out, KD_ERR_CUDA otherwise; nothing is left allocated on failure. */
kd_status kd_model_load(const kd_config* cfg, const kd_weights* w, kd_model** out);

/* Wait for the model's outstanding work, then free everything it owns: the
 * teardown matching kd_model_load (the pages' engines release the weights and
 * the slots with the engine; hf2q ADR-040 section 0.0, weights and slot KV are
 * separate budgets owned by the worker).  The handle is invalid afterwards. */
kd_status kd_model_free(kd_model* m);

/* Claim a free slot (lowest free id) for a new session of length 0.
 * Slot ownership per session follows memra's per-sequence `Cache` (its own
 * position and KV) and hf2q ADR-040's KV indexed by slot. */
kd_status kd_session_bind(kd_model* m, int32_t* session_id_out);

/* Release a session's slot.  Waits on the host for the last step that used the
 * model, so a freed slot is never rebound while a step may still write it.
 * hf2q ADR-040 section 0.0 ("Agent-slot lifetime"): a slot is a retained
 * cache; a new conversation reuses an idle slot and invalidates its old state
 * first -- here a freed slot is bound again at length 0.
 * Errors: KD_ERR_BAD_SESSION if the id is not bound. */
kd_status kd_session_free(kd_model* m, int32_t session_id);

/* Fill a bound session's cache with `len` positions (its prompt history):
 * k_fp16 and v_fp16 are [n_layers][n_kv_heads][len][head_dim] fp16, host or
 * device memory (any address CUDA can copy from).  Sets the length to len.
 * Enqueued on `stream`; the source must stay valid until the stream reaches it.
 * A session's state is its own position and KV: in memra decode_batch.rs
 * `decode_step_batch`, row b carries a cache of its own holding its position
 * and its quantized KV;
 * Kakeya PR-A3c binds each batch row to a session with its own KV-cache row,
 * filled with its ~1238-token context before batched decode.  Loading a slot
 * also restores a retained history (hf2q ADR-040 section 0.0, "Agent-slot
 * lifetime": a continuation reuses its slot's KV instead of re-prefilling).
 * Errors: KD_ERR_BAD_SESSION (not bound), KD_ERR_POSITION (len outside
 * [0, max_ctx]), KD_ERR_INVALID_ARG (null cache with len > 0). */
kd_status kd_session_load_kv(kd_model* m, int32_t session_id, const void* k_fp16,
                             const void* v_fp16, int32_t len, kd_stream stream);

/* The number of positions a bound session holds: memra's `cache.pos`, which a
 * batched step moves forward by one for every row, as a single-sequence step
 * would (decode_batch.rs `decode_step_batch`); here it becomes the step's
 * position + 1.  Host only, no CUDA call.  Errors: KD_ERR_BAD_SESSION. */
kd_status kd_session_length(const kd_model* m, int32_t session_id, int32_t* len_out);

/* One batched decode step (memra decode_batch.rs `decode_step_batch`: row b is
 * session b with its own cache and position; every projection runs at m = B).
 *   B: 1 .. max_sessions.  Up to KD_MAX_BATCH rows go through one launch train;
 *     a larger B runs as consecutive groups of at most KD_MAX_BATCH rows (rows
 *     0..15, 16..31, ...), each reading the weights once, with the same
 *     per-row arithmetic (every row equal to its B = 1 result).  memra refuses
 *     B > 16 and leaves wider concurrency to its serve scheduler, which splits
 *     it into groups of at most 16 (decode_batch.rs, `decode_step_batch`). 
 *   session_ids, tokens, positions: host arrays of length B.  Ids must be bound
 *     and distinct; tokens in [0, vocab); 0 <= positions[b] <= length(session)
 *     and positions[b] < max_ctx.  The token is written to the cache at
 *     positions[b] and attends keys 0..positions[b]; afterwards the session's
 *     length is positions[b] + 1 (a position below the length rewinds).
 *   logits_out: NULL or device fp32 [B][vocab], 16-byte aligned; row b belongs
 *     to session_ids[b].
 *   argmax_out: NULL or device int32 [B]: the greedy next token (largest logit,
 *     ties to the lowest index, NaN never wins; -1 if a row is all NaN).
 * Enqueued on `stream` without a host wait; outputs are valid once the stream
 * has reached them.  Steps of one model may be issued on different streams:
 * each step waits for the previous one on the device. */
kd_status kd_decode_step(kd_model* m, const int32_t* session_ids, const int32_t* tokens,
                         const int32_t* positions, int32_t B, float* logits_out,
                         int32_t* argmax_out, kd_stream stream);

/* Per-row sampling parameters (memra decode_batch.rs `decode_step_batch_sampled`:
 * a Gumbel perturbation keyed by (seed, counter) and the temperature, then the
 * same argmax, is one categorical draw from softmax(logits / temperature); the
 * draw depends on (seed, counter) only, not on the rest of the batch).
 *   temperature <= 0 (or NaN): the greedy pick of kd_decode_step.
 *   temperature > 0: the index of the largest z_v = logit_v / temperature - log(-log u_v)
 *     (fp32; ties to the lowest index, NaN never wins), u_v = (top 24 bits of w + 1/2) / 2^24
 *     where w is word v mod 4 of the Philox4x64-10 block (Salmon et al., "Parallel
 *     random numbers: as easy as 1, 2, 3", SC'11) at counter {v / 4, counter, 0, 0}
 *     under key {seed, 0}.
 * The same (logits, temperature, seed, counter) always give the same token. */
typedef struct {
    float temperature;
    uint32_t reserved;  /* 0 */
    uint64_t seed;
    uint64_t counter;
} kd_sample_params;

/* kd_decode_step with device-side temperature sampling: row b's token is drawn
 * per params[b] (host array of B) and written to token_out[b] (device int32 [B],
 * required).  Everything else, including logits_out (the undisturbed logits),
 * as for kd_decode_step.  Errors as for kd_decode_step; KD_ERR_INVALID_ARG for
 * a null params or token_out. */
kd_status kd_decode_step_sampled(kd_model* m, const int32_t* session_ids, const int32_t* tokens,
                                 const int32_t* positions, int32_t B, const kd_sample_params* params,
                                 float* logits_out, int32_t* token_out, kd_stream stream);

/* Allocation failure, for checking that a load fails closed (hf2q ADR-040:
 * allocation overruns are refused with an error, never a crash or a half-built
 * object).  With nth >= 1, the nth device or pinned-host allocation of the next
 * kd_model_load fails as if memory had run out: that load returns KD_ERR_OOM
 * with everything it had allocated freed; the switch then disarms itself.
 * nth = 0 disarms it.  *allocs_out (nullable) receives the number of
 * allocations the most recent kd_model_load made, so that a caller can arm each
 * of them in turn.  No other thread may load a model while it is armed.
 * Errors: KD_ERR_INVALID_ARG for nth < 0. */
kd_status kd_debug_fail_alloc(int32_t nth, int32_t* allocs_out);

/* Debug: when dev_buf is not NULL, later steps also write the residual stream
 * after the embedding and after every layer to dev_buf, device fp32
 * [n_layers+1][B][hidden] (steps then launch kernel by kernel).  NULL turns it off.
 * The residual stream is the fp32 `x` of memra decode_batch.rs
 * `decode_batch_layers` (a `CudaSlice<f32>` carried from layer to layer); the
 * capture exposes it per layer so that a batched step can be compared layer by
 * layer with a reference, the way hf2q ADR-040 narrowed its N = 8 divergence
 * down to one operation (section 0.13, post-audit finding).  The buffer is
 * caller-owned and must hold B rows of the steps that run while it is set. */
kd_status kd_debug_capture_hidden(kd_model* m, float* dev_buf);

/* Debug: run decoder layer `layer` alone on the residual rows x_in (device or
 * host fp32 [B][hidden], B <= KD_MAX_BATCH) for the given sessions at the given
 * positions (same rules as kd_decode_step), writing the layer's output rows to x_out (device or
 * host fp32 [B][hidden]).  Writes that layer's K/V row at each position; does
 * not change any session's length.  The same kernels as a step run, so a layer
 * can be checked on its own against a reference, without errors carried in from
 * the layers before it.  Enqueued on `stream`. */
kd_status kd_debug_layer(kd_model* m, int32_t layer, const int32_t* session_ids,
                         const int32_t* positions, int32_t B, const float* x_in,
                         float* x_out, kd_stream stream);

/* Wait for the model's work, then read and clear its device fault word.
 * *flags_out = 0 when no kernel gave up a bounded wait; KD_ERR_DEVICE is
 * returned when one did (the outputs of that step are not valid; the model's
 * internal arrival counters are cleared as well, so the next step is correct).
 * memra returns an error for the request rather than stopping the process
 * (decode_batch.rs: every step returns a `Result`). */
kd_status kd_device_status(kd_model* m, int32_t* flags_out);

/* Debug fault hook, for testing kd_device_status: the next kd_decode_step
 * launches kernel by kernel, and the first launch of kernel class
 * `kernel_class` (one with bounded waits: KD_K_QKV, KD_K_ATTN_SPLIT, KD_K_WO,
 * KD_K_GATE_UP, KD_K_DOWN or KD_K_LM_HEAD) has one barrier expect a few bytes
 * more than its copies deliver.  Every copy still lands; the wait on that
 * barrier runs out after its time limit (about half a second), the kernel sets
 * the fault word and returns, and the step's outputs are invalid.  Nothing
 * faults or hangs.  One-shot.  Errors: KD_ERR_INVALID_ARG for another class. */
kd_status kd_debug_inject_wait_timeout(kd_model* m, int32_t kernel_class);

/* Measurement (the event-based counterpart of memra's per-phase breakdown,
 * decode_batch.rs BATCH_PHASE, without its host syncs).  While enabled, steps
 * launch kernel by kernel and bracket every kernel with CUDA events on the
 * step's stream.  kd_profile_read waits for the model's work, then returns per
 * kernel class (KD_K_*) the number of launches and their summed device time in
 * milliseconds since the previous read, and resets the sums. */
/* (KD_K_RMSNORM: the elementwise norm between a residual writer and the next
 * projection; its row reductions are fused into the residual writer.) */
enum {
    KD_K_EMBED = 0, KD_K_RMSNORM, KD_K_QKV, KD_K_ATTN_SPLIT, KD_K_ATTN_COMBINE, KD_K_WO,
    KD_K_GATE_UP, KD_K_DOWN, KD_K_LM_HEAD, KD_K_ARGMAX, KD_K_COUNT
};
kd_status kd_profile_enable(kd_model* m, int32_t on);
kd_status kd_profile_read(kd_model* m, int32_t* launches /* [KD_K_COUNT] */,
                          double* ms /* [KD_K_COUNT] */);

/* Measurement: a per-CTA timeline of later steps, in the pipelined step as it
 * runs (CUDA graph and programmatic dependent launch kept; one graph per
 * buffer).  While dev_buf is set, launch i of a step (i < max_launches) stamps
 * in dev_buf[i][cta][0..3] (device uint64 [max_launches][KD_TIMELINE_CTAS][4],
 * cta = blockIdx.y * gridDim.x + blockIdx.x < KD_TIMELINE_CTAS) the GPU global
 * timer in ns when the CTA started, when its dependency wait returned and when
 * its last warp ended, and its SM id.  Records a launch does not use are not
 * written: zero the buffer first.  Each step overwrites the records.  When
 * classes_out (host int32 [max_launches]) is not NULL it receives the kernel
 * class (KD_K_*) of each launch index of a full step (-1 past its end).  NULL
 * dev_buf turns it off.  The counterpart of memra's per-phase breakdown
 * (decode_batch.rs BATCH_PHASE) without its stream syncs. */
#define KD_TIMELINE_CTAS 1024
kd_status kd_profile_timeline(kd_model* m, uint64_t* dev_buf, int32_t max_launches, int32_t* classes_out);

/* The message of the last failure on the calling thread ("" if none).  The C
 * counterpart of the error value memra's batched calls return with their
 * `Result<_, Box<dyn Error>>` (decode_batch.rs `decode_step_batch`): a status
 * code says which kind of failure, this string says what failed.  Owned by the
 * library; valid until the thread's next failing call. */
const char* kd_last_error(void);

/* ------------------------------------------------------------------------
 * Op-level entry points: the step's kernels on their own, for isolated tests
 * and measurements.  Same conventions as above.
 * ---------------------------------------------------------------------- */

typedef struct kd_q8_matrix kd_q8_matrix; /* a repacked Q8_0 matrix on the device */

/* Copy a canonical Q8_0 matrix [rows][cols/32] (host memory) to the device in
 * the kernel's tiled layout, with a split-K workspace for m <= KD_MAX_BATCH.
 * rows must be a multiple of 32 and cols a multiple of 128.  Synchronous. */
kd_status kd_q8_matrix_create(const void* q8_0_host, int32_t rows, int32_t cols,
                              kd_q8_matrix** out);
kd_status kd_q8_matrix_free(kd_q8_matrix* w);

/* Weight-only Q8_0 matrix-vector product for m = 1..16 rows (memra's batched
 * verify-tier mmvq, whose rows must equal their m = 1 results bit for bit):
 *   y[r][o] = sum over blocks b of d[o][b] * sum_j q[o][b][j] * x[r][32b+j]
 * x: device fp16 [m][cols], 16-byte aligned; y: device fp32 [m][rows].  Row r of y is
 * bit-identical for every m.  Calls on one matrix must be stream-ordered
 * (they share its workspace). */
kd_status kd_mmvq(const kd_q8_matrix* w, const uint16_t* x, int32_t m, float* y,
                  kd_stream stream);

/* Wait for the whole device, then read and clear the fault word of the
 * matrix's kd_mmvq calls (0: no bounded wait ran out; else KD_ERR_DEVICE, and
 * the results of those calls are not valid). */
kd_status kd_q8_matrix_status(kd_q8_matrix* w, int32_t* flags_out);

/* The schedule the library picks for a Q8_0 matrix of rows x cols on a GPU with
 * num_sms SMs (host only: no CUDA call, usable without a GPU).  It depends on the
 * shape and the SM count only, never on the batch, so a row's arithmetic is the
 * same at every m.  *mode_out: 1 = group (a CTA owns whole 32-row groups and its
 * 8 warps split K), chosen when the groups number at most twice the SMs, or at
 * most 8 times the SMs with the busiest SM's share at most 5% above the average;
 * 0 = stream (warps stream equal contiguous shares of the matrix's 128-column
 * stages).  *warps_out: the streaming warps (min(8 * num_sms, stages)); *share_out:
 * the most stream warps meeting in one row group (1 on the group schedule).
 * rows a multiple of 32, cols of 128, num_sms >= 1: else KD_ERR_UNSUPPORTED /
 * KD_ERR_INVALID_ARG. */
kd_status kd_mmvq_schedule(int32_t rows, int32_t cols, int32_t num_sms, int32_t* mode_out,
                           int32_t* warps_out, int32_t* share_out);

/* Greedy pick over logit rows, as the step's argmax (memra decode_batch.rs
 * `decode_batch_epilogue`, a device argmax equal to the host one):
 *   out[b] = the index of the largest logits[b][v]; equal values go to the
 *   lowest index, -0 equals +0, NaN never wins; -1 if row b is all NaN.
 * logits: device fp32 [B][V], 16-byte aligned, V a multiple of 4; out: device
 * int32 [B]; B in [1, KD_MAX_BATCH]; workspace: device memory of
 * KD_ARGMAX_WORKSPACE_BYTES, owned by the caller, used by one call at a time. */
#define KD_ARGMAX_WORKSPACE_BYTES 256
kd_status kd_argmax(const float* logits, int32_t B, int32_t V, int32_t* out, void* workspace,
                    kd_stream stream);

/* Temperature sampling over logit rows, as kd_decode_step_sampled's pick:
 * out[b] drawn per params[b] (host array of B, see kd_sample_params; the
 * parameters are copied on the call).  logits: device fp32 [B][V], 16-byte
 * aligned, V a multiple of 4; out: device int32 [B]; B in [1, KD_MAX_BATCH];
 * workspace: device memory of KD_SAMPLE_WORKSPACE_BYTES, 16-byte aligned, owned
 * by the caller, used by one call at a time. */
#define KD_SAMPLE_WORKSPACE_BYTES 1024
kd_status kd_sample(const float* logits, int32_t B, int32_t V, const kd_sample_params* params, int32_t* out,
                    void* workspace, kd_stream stream);

/* Bytes of device workspace kd_attn_append_decode needs for these sizes. */
size_t kd_attn_workspace_bytes(int32_t B, int32_t n_heads, int32_t head_dim, int32_t cap);

/* KV append then ragged GQA split-K flash-decode (memra decode_batch_layers:
 * first every row's K/V is appended, then every sequence attends):
 *   for each row b: K[slot_b][h][pos_b] = fp16(k_new[b][h]), same for V; then
 *   out[b][qh] = fp16(sum_{t<=pos_b} softmax_t(q[b][qh] . K_t / sqrt(head_dim)) V_t)
 *   over KV head qh / (n_heads / n_kv_heads).
 * q: device fp32 [B][n_heads][head_dim] (already rotated); k_new, v_new: device
 * fp32 [B][n_kv_heads][head_dim]; k_cache, v_cache: device fp16
 * [n_slots][n_kv_heads][cap][head_dim]; slots, positions: host int32 [B] (slots
 * distinct, 0 <= positions[b] < cap); out: device fp16 [B][n_heads*head_dim];
 * workspace: device memory of kd_attn_workspace_bytes(B, n_heads, head_dim, cap).
 * k_cache, v_cache and workspace must be 16-byte aligned and q 8-byte aligned
 * (KD_ERR_INVALID_ARG otherwise). */
kd_status kd_attn_append_decode(const float* q, const float* k_new, const float* v_new,
                                uint16_t* k_cache, uint16_t* v_cache, const int32_t* slots,
                                const int32_t* positions, int32_t B, int32_t n_heads,
                                int32_t n_kv_heads, int32_t head_dim, int32_t n_slots,
                                int32_t cap, uint16_t* out, void* workspace,
                                size_t workspace_bytes, kd_stream stream);

/* Wait for `stream`, then read the fault word of the last attention call:
 * `workspace` = the workspace that call was given, or NULL for the last
 * kd_attn_append_decode_noalloc call on the current device.  *flags_out = 0
 * when no bounded wait ran out; otherwise KD_ERR_DEVICE (that call's output is
 * not valid).  Each call clears its word when it starts. */
kd_status kd_attn_device_status(const void* workspace, int32_t* flags_out, kd_stream stream);

/* The Q8_0 KV row format (KD_FLAG_KV_Q8_0), for the isolated workloads: rows of
 * 128 values as 128 quant bytes u = q + 128 (uint8 [rows][128]) and 4 fp16 block
 * scales (uint16 bits [rows][4]), quantised as KD_FLAG_KV_Q8_0 states.
 * kd_kv_q8_quantize: src device fp32 [rows][128] -> quants, scales (device). */
kd_status kd_kv_q8_quantize(const float* src, int64_t rows, uint8_t* quants, uint16_t* scales, kd_stream stream);

/* kd_attn_append_decode over a Q8_0 cache of head_dim 128: the new rows (fp32,
 * k_new / v_new as for kd_attn_append_decode) are quantised into row pos_b of
 * slot_b, then every session attends keys 0..pos_b.  Caches:
 * [n_slots][n_kv_heads][cap] rows of quants ([..][128] uint8) and scales
 * ([..][4] fp16 bits); cap even.  Workspace: kd_attn_workspace_bytes(B, n_heads,
 * 128, cap).  All device buffers 16-byte aligned.  Other arguments and errors
 * as for kd_attn_append_decode. */
kd_status kd_attn_append_decode_q8(const float* q, const float* k_new, const float* v_new, uint8_t* k_quants,
                                   uint16_t* k_scales, uint8_t* v_quants, uint16_t* v_scales,
                                   const int32_t* slots, const int32_t* positions, int32_t B, int32_t n_heads,
                                   int32_t n_kv_heads, int32_t n_slots, int32_t cap, uint16_t* out,
                                   void* workspace, size_t workspace_bytes, kd_stream stream);

/* ------------------------------------------------------------------------
 * Allocation-free variant (no counterpart on the batched-decode pages: it
 * exists for callers, not for the method).
 *
 * kd_attn_append_decode_noalloc computes exactly what kd_attn_append_decode
 * computes, with the same kernels, but takes no workspace and allocates
 * nothing: no cudaMalloc/cudaFree, no allocating library routine, no
 * host-to-device copy (slots and positions are passed to the device as kernel
 * arguments).  It is meant for callers that cannot allocate device memory
 * where they decode -- e.g. code inside a memory pool or arena that owns the
 * whole GPU, or a hot path where an allocation's implicit device
 * synchronisation is not acceptable.
 *
 * Its scratch is one fixed device array of KD_ATTN_NOALLOC_SCRATCH_BYTES that
 * every GPU using this entry point holds from library load to process exit.
 * Requests whose partial results do not fit are refused with
 * KD_ERR_UNSUPPORTED: they need
 *   256 + B * n_heads * ceil(cap / 64) * (head_dim + 4) * 4  bytes
 * (e.g. B = 8, 32 heads of 128, cap up to 7936 positions).
 * All calls share the array, and it keeps the last call's contents (each call
 * rewrites what it reads, so no clearing is needed between calls): calls that
 * overlap on the GPU -- on different streams without ordering, or from
 * different threads -- race on it and must not be issued.
 * The first call on each device looks up the array's device address (once,
 * with that device current); make that first call before any stream capture
 * (a first call made during a capture is refused with KD_ERR_INVALID_ARG, and
 * a failed lookup is retried by the next call).
 * Arguments, layouts and errors as for kd_attn_append_decode; a device-side
 * fault (a bounded wait that ran out) is read with kd_attn_device_status(NULL). */
#define KD_ATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
kd_status kd_attn_append_decode_noalloc(const float* q, const float* k_new, const float* v_new,
                                        uint16_t* k_cache, uint16_t* v_cache,
                                        const int32_t* slots, const int32_t* positions,
                                        int32_t B, int32_t n_heads, int32_t n_kv_heads,
                                        int32_t head_dim, int32_t n_slots, int32_t cap,
                                        uint16_t* out, kd_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* KD_H_ */
