/*
 * llama_layer.h -- C ABI of the GB300 (sm_103a) forward pass of one
 * Llama-style decoder layer.
 *
 * The operator chain follows the page "Which ops-transformer operators one
 * Llama2-7B layer calls" (seekfood.cn/news/1207529), section "single-layer
 * operator call chain": x -> RMSNorm -> merged Q/K/V Linear -> RotaryEmbedding
 * -> Self-Attention (GQA) -> Attention Output Linear -> residual -> RMSNorm ->
 * merged Gate/Up Linear -> SiLU * up -> Down Linear -> residual.  Prefill and
 * decode take different attention kernels (same page, section "KV Cache and
 * the operators").  The KV cache is paged as on the page "ATB KV-cache paging,
 * quantisation, speculative decoding and communication overlap"
 * (hwcomputing.csdn.net), section "KV Cache memory wall": fixed-size blocks,
 * a block_table from logical to physical blocks, contextLens per request, and
 * ReshapeAndCache writing each step's K/V into its slot.
 *
 * Conventions shared by every call
 *  - All tensor pointers are DEVICE pointers, caller-owned, row-major, and
 *    16-byte aligned.  BF16 is IEEE bfloat16 (2 bytes); gains are float32.
 *  - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream).  No call allocates device memory, synchronises, or
 *    keeps a pointer after it returns, except ll_pack_weights (see there).
 *  - The return value reports what the host can check before launching
 *    (LL_OK or an LL_ERR_* code; nothing is launched on error).  Problems
 *    only the device can see (a block_table entry or slot out of range, a
 *    position beyond the RoPE table) are OR-ed as LL_DEV_* bits into
 *    `*status`, a caller-owned device int32 that the caller zeroes and reads
 *    after synchronising.  The offending row is skipped; kernels never trap.
 *  - Every bounded wait inside a kernel gives up after about two seconds,
 *    sets LL_DEV_TIMEOUT and lets the kernel finish.
 *  - The KV pool is two tensors, K and V, each BF16
 *    [num_blocks, n_kv_heads, block_size, head_dim] ("BNSD" inside a block, as
 *    the 910B layout on the paging page).  Slot s = block * block_size + offset.
 *  - block_table is int32 [batch, max_blocks]; entry j is the physical block
 *    holding positions j*block_size .. (j+1)*block_size-1 of that sequence.
 */
#ifndef LLAMA_LAYER_H
#define LLAMA_LAYER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* host-detectable errors (return values) */
#define LL_OK 0
#define LL_ERR_INVALID_ARG 1   /* null pointer, non-positive or inconsistent size */
#define LL_ERR_UNSUPPORTED 2   /* shape outside what the kernels implement */
#define LL_ERR_WORKSPACE 3     /* workspace missing or smaller than required */
#define LL_ERR_CUDA 4          /* a CUDA runtime/driver call failed */

/* device-detected problems (bits OR-ed into *status) */
#define LL_DEV_BAD_BLOCK 1     /* block_table entry < 0 or >= num_blocks where a block was needed */
#define LL_DEV_BAD_SLOT 2      /* slot_mapping entry >= num_blocks * block_size */
#define LL_DEV_BAD_POSITION 4  /* position < 0 or >= max_position, or context_len out of range */
#define LL_DEV_TIMEOUT 8       /* a bounded in-kernel wait gave up */

/* Layer shape.  head_dim must be 64 or 128; n_heads % n_kv_heads == 0;
 * n_heads / n_kv_heads <= 16; hidden and intermediate multiples of 16;
 * block_size a power of two in [16, 256]; max_position = rows of the RoPE
 * table (largest position + 1).
 * RoPE uses half-split pairs and angle pos * rope_theta^(-2i/head_dim). */
typedef struct {
    int32_t hidden;
    int32_t n_heads;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t intermediate;
    int32_t block_size;
    int32_t max_position;
    float rms_eps;
    float rope_theta;
} ll_config;

/* Canonical weights as a model stores them, all BF16 [out, in] row-major:
 * w_qkv [(n_heads + 2 n_kv_heads) head_dim, hidden], rows = Q heads, then K
 * heads, then V heads (the merged QKV MatMul of the chain page);
 * w_o [hidden, n_heads head_dim]; w_gate and w_up [intermediate, hidden];
 * w_down [hidden, intermediate]; g_attn and g_ffn float32 [hidden]. */
typedef struct {
    const void* w_qkv;
    const void* w_o;
    const void* w_gate;
    const void* w_up;
    const void* w_down;
    const float* g_attn;
    const float* g_ffn;
} ll_weights;

typedef struct {
    void* k;              /* BF16 [num_blocks, n_kv_heads, block_size, head_dim] */
    void* v;              /* same shape */
    int32_t num_blocks;
} ll_kv_pool;

/* An INT8 KV pool (paging page, section "KV Cache quantisation": per-token
 * granularity, each token's K and V with their own float32 scale).  Codes in the
 * layout of ll_kv_pool; one scale per token and KV head.  A cached row reads back
 * as code * scale. */
typedef struct {
    void* k;              /* int8 [num_blocks, n_kv_heads, block_size, head_dim] */
    void* v;              /* same shape */
    float* k_scale;       /* float32 [num_blocks, n_kv_heads, block_size] */
    float* v_scale;       /* same shape */
    int32_t num_blocks;
} ll_kv_pool_q8;

/* Human-readable name of an LL_ERR_* code (static string). */
const char* ll_strerror(int code);

/* Description of the last failure behind an LL_ERR_* return on the calling
 * thread (the failing step and CUDA's message), or "" if none.  Valid until
 * the thread's next library call. */
const char* ll_last_error(void);

/* Bytes of the packed-weight buffer for `cfg` (0 if cfg is invalid). */
size_t ll_packed_weights_size(const ll_config* cfg);

/* Lays out the weights the way the kernels read them, into the caller-owned
 * device buffer `packed` (ll_packed_weights_size bytes): Q/K head rows
 * reordered so that each RoPE pair is adjacent, gate and up rows interleaved
 * (the MergedMatMul(GateUp) of the chain page), the other weights copied, and
 * a float32 cos/sin table for max_position positions computed in float64.
 * The canonical weights may be freed once the stream has passed this call.
 * Setup-time call: it synchronises `stream` before returning. */
int ll_pack_weights(const ll_config* cfg, const ll_weights* w, void* packed, size_t packed_bytes,
                    void* stream);

/* Workspace bytes for layer calls of up to max_tokens tokens (prefill: batch *
 * seq_len; decode: batch) and block tables up to max_blocks wide. */
size_t ll_workspace_size(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks);

/* Checkpoints of the fused layer (page "ATB fused-operator matrix and KV-cache
 * management", section on the engineering limits of fusion granularity: besides
 * the step-by-step and fully fused execution modes it names a fused mode with
 * verification checkpoints at key nodes, so that a wrong result can be traced to
 * one step).  A layer call leaves the output of every kernel of its chain in the
 * workspace; these are their byte offsets from the workspace start, for a
 * workspace sized by ll_workspace_size(cfg, max_tokens, max_blocks).  After a call
 * over T tokens (and until the next call on the same workspace), row t < T of:
 *   x_hat  BF16    [T][hidden]           RMSNorm(x) * g_attn
 *   q      BF16    [T][n_heads*head_dim] q after RoPE, heads in order, element i of a
 *                                        head at i (RoPE pairs i, i + head_dim/2)
 *   o      BF16    [T][n_heads*head_dim] attention output
 *   h      float32 [T][hidden]           x + o W_o^T
 *   h_hat  BF16    [T][hidden]           RMSNorm(h) * g_ffn
 *   a      BF16    [T][intermediate]     SiLU(x_hat2 W_gate^T) * (x_hat2 W_up^T)
 * The new tokens' K and V are in the KV pool at their slots.  Host-only; no GPU
 * work.  Returns LL_ERR_INVALID_ARG for an invalid cfg or sizes. */
typedef struct {
    size_t x_hat, q, o, h, h_hat, a;
} ll_checkpoints;

int ll_workspace_checkpoints(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks,
                             ll_checkpoints* out);

/* Execution modes of a layer call (page "ATB fused-operator matrix and KV-cache
 * management", section on the engineering limits of fusion granularity, which
 * names a step-by-step mode, a fused mode and a fused mode with verification
 * checkpoints).  LL_MODE_FUSED is the fused chain of ll_layer_prefill and
 * ll_layer_decode_step, whose kernel outputs stay readable through
 * ll_workspace_checkpoints (the checkpointed mode needs nothing more).
 * LL_MODE_STEP_BY_STEP runs every operator of the chain as its own kernel and
 * keeps every intermediate: RMSNorm, the merged QKV Linear (float32 output),
 * RotaryEmbedding, the slot mapping, ReshapeAndCache, attention, the O Linear,
 * the residual add, RMSNorm, the merged gate/up Linear, SiLU * up, the down
 * Linear and the residual add.  Its element-wise arithmetic is the fused
 * epilogues', so the two modes compute the same values; it exists to locate a
 * wrong result by comparing one operator at a time.  It takes BF16 pools. */
#define LL_MODE_FUSED 0
#define LL_MODE_STEP_BY_STEP 1

/* Workspace bytes for calls in `mode` (LL_MODE_FUSED: ll_workspace_size). */
size_t ll_workspace_size_mode(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks, int32_t mode);

/* The step-by-step mode's extra intermediates, as byte offsets from the start of a
 * workspace sized by ll_workspace_size_mode(cfg, max_tokens, max_blocks,
 * LL_MODE_STEP_BY_STEP); the offsets of ll_workspace_checkpoints hold in that
 * workspace too.  After a step-by-step call over T tokens, row t < T of:
 *   qkv      float32 [T][(n_heads + 2 n_kv_heads) head_dim]  x_hat W_qkv^T before RoPE, in the
 *            packed column order: within each Q and K head column 2i holds element i and
 *            2i + 1 element i + head_dim/2; V heads in element order
 *   k, v     BF16    [T][n_kv_heads head_dim]   K after RoPE and V, element order
 *   slots    int32   [T]                        cache slot of each token (-1 if invalid)
 *   o_proj   float32 [T][hidden]                o W_o^T
 *   gate_up  float32 [T][2 intermediate]        h_hat W_gate^T and h_hat W_up^T, interleaved
 *                                               (column 2j gate j, 2j + 1 up j)
 *   down     float32 [T][hidden]                a W_down^T
 * Host-only; no GPU work. */
typedef struct {
    size_t qkv, k, v, slots, o_proj, gate_up, down;
} ll_step_checkpoints;

int ll_workspace_step_checkpoints(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks,
                                  ll_step_checkpoints* out);

/* Prefill: x BF16 [batch*seq_len, hidden], token-major; token t belongs to
 * sequence t / seq_len and sits at positions[t] (int32 [batch*seq_len]).
 * Writes every token's K and V (after RoPE on K) into the pool at
 * block_table[seq][pos / block_size], offset pos % block_size; then every
 * query at position p attends (causally, GQA) over cache positions 0..p of
 * its sequence, which therefore must already be cached below this call's
 * first position (chunked prefill).  Writes y BF16 [batch*seq_len, hidden];
 * y must not alias x.  The chain page's prefill path. */
int ll_layer_prefill(const ll_config* cfg, const void* packed, const void* x,
                     const int32_t* positions, int32_t batch, int32_t seq_len,
                     const ll_kv_pool* pool, const int32_t* block_table, int32_t max_blocks,
                     void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                     void* stream);

/* Decode step: x BF16 [batch, hidden], one new token per sequence.
 * context_lens (int32 [batch]) counts each sequence's cache INCLUDING the new
 * token, which is written at position context_lens[b] - 1; its query attends
 * over positions 0..context_lens[b]-1.  y BF16 [batch, hidden].  The chain
 * page's decode path (one-row query against the cached K/V). */
int ll_layer_decode_step(const ll_config* cfg, const void* packed, const void* x,
                         const ll_kv_pool* pool, const int32_t* block_table, int32_t max_blocks,
                         const int32_t* context_lens, int32_t batch, void* y, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream);

/* ll_layer_prefill and ll_layer_decode_step with an execution mode (LL_MODE_FUSED or
 * LL_MODE_STEP_BY_STEP; anything else is LL_ERR_INVALID_ARG).  Arguments as there; the
 * workspace comes from ll_workspace_size_mode for the same mode. */
int ll_layer_prefill_mode(const ll_config* cfg, const void* packed, const void* x, const int32_t* positions,
                          int32_t batch, int32_t seq_len, const ll_kv_pool* pool, const int32_t* block_table,
                          int32_t max_blocks, void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                          int32_t mode, void* stream);
int ll_layer_decode_step_mode(const ll_config* cfg, const void* packed, const void* x, const ll_kv_pool* pool,
                              const int32_t* block_table, int32_t max_blocks, const int32_t* context_lens,
                              int32_t batch, void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                              int32_t mode, void* stream);

/* ll_layer_decode_step over an INT8 pool: the new tokens' K and V (after RoPE,
 * BF16) are quantised into the pool as ll_reshape_and_cache_q8 does, and the
 * attention reads code * scale (ll_paged_attention_decode_q8).  head_dim 128;
 * workspace from ll_workspace_size; other arguments as ll_layer_decode_step.
 * (Prefill into an INT8 pool is not provided.) */
int ll_layer_decode_step_q8(const ll_config* cfg, const void* packed, const void* x, const ll_kv_pool_q8* pool,
                            const int32_t* block_table, int32_t max_blocks, const int32_t* context_lens,
                            int32_t batch, void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                            void* stream);

/* ReshapeAndCache (paging page, section "KV Cache memory wall",
 * ReshapeAndCacheOperation): k, v BF16 [tokens, n_kv_heads, head_dim];
 * slot_mapping int32 [tokens]; token t's rows go to
 * pool[slot / block_size, :, slot % block_size, :].  slot -1 skips the token;
 * slot >= num_blocks*block_size sets LL_DEV_BAD_SLOT and skips it.  Bit-exact
 * copy.  head_dim a multiple of 8. */
int ll_reshape_and_cache(const void* k, const void* v, const int32_t* slot_mapping, int32_t tokens,
                         int32_t n_kv_heads, int32_t head_dim, int32_t block_size,
                         const ll_kv_pool* pool, int32_t* status, void* stream);


/* ReshapeAndCache into an INT8 pool, quantising online: for token t and KV head h,
 * scale = max_i |row_i| / 127 and code_i = round-half-even(row_i / scale) in
 * float32 (IEEE division), clipped to [-127, 127]; a row of zeros gets scale 0
 * and codes 0.  Arguments and slot rules as ll_reshape_and_cache; head_dim a
 * multiple of 32, at most 256.  Codes and scales are bit-exact. */
int ll_reshape_and_cache_q8(const void* k, const void* v, const int32_t* slot_mapping, int32_t tokens,
                            int32_t n_kv_heads, int32_t head_dim, int32_t block_size,
                            const ll_kv_pool_q8* pool, int32_t* status, void* stream);

/* Workspace bytes for ll_paged_attention_decode. */
size_t ll_attention_workspace_size(int32_t batch, int32_t n_heads, int32_t head_dim,
                                   int32_t max_blocks, int32_t block_size);

/* Decode attention over the paged cache (chain page, section "KV Cache and
 * the operators", flash_attention_decode; paging page PagedAttentionOperation):
 * q BF16 [batch, n_heads, head_dim]; sequence b's query head h attends over
 * positions 0..context_lens[b]-1 of KV head h / (n_heads / n_kv_heads) with
 * softmax(q k^T * scale).  out BF16 [batch, n_heads, head_dim]; a sequence
 * with context length 0 gets zero rows.  head_dim 64 or 128, n_heads /
 * n_kv_heads <= 16, block_size a power of two in [16, 256]. */
int ll_paged_attention_decode(const void* q, const ll_kv_pool* pool, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* context_lens, int32_t batch,
                              int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                              int32_t block_size, float scale, void* out, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream);

/* ll_paged_attention_decode over an INT8 pool: the cached rows are code * scale
 * (paging page, section "KV Cache quantisation": dequantised as the cache block
 * is loaded).  head_dim 128; workspace sized by ll_attention_workspace_size; the
 * other arguments and limits as ll_paged_attention_decode. */
int ll_paged_attention_decode_q8(const void* q, const ll_kv_pool_q8* pool, const int32_t* block_table,
                                 int32_t max_blocks, const int32_t* context_lens, int32_t batch,
                                 int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t block_size, float scale, void* out, void* workspace,
                                 size_t workspace_bytes, int32_t* status, void* stream);

/* ll_paged_attention_decode for callers that cannot allocate device memory.
 * The pages have no counterpart of this call.  Some callers only own the
 * buffers they pass in: a plugin that receives input and output tensors from
 * a host framework with no hook for extra workspace, or code running where a
 * device allocation would synchronise the device or bypass the allocator that
 * owns the memory.  This variant takes the same arguments minus the workspace
 * and keeps the per-split partial results in a fixed device array inside the
 * library (32 MiB; every GPU that loads the library holds it until the
 * process exits).  It allocates nothing and calls no allocator.
 *  - Limit: with rows = batch * n_heads * ceil(max_blocks * block_size / 1024)
 *    (one per 1024-key split of every query head), the call needs
 *    rows * ((head_dim + 2) * 4 + 16) + 16 bytes of the array (per row the
 *    float32 partial output, its running max and sum, and a 16-byte entry of
 *    the splits' dispatch order; then a 16-byte pad);
 *    ll_attention_workspace_size gives the same figure rounded up to a
 *    multiple of 256.  Beyond 32 MiB it returns LL_ERR_UNSUPPORTED
 *    (ll_last_error gives the sizes) and launches nothing.
 *  - The first call on a device resolves the array's device address (this may
 *    load the library's device code); make that first call before any stream
 *    capture on the device.
 *  - All calls share the one array and each overwrites what it uses (nothing
 *    in it needs to start at zero): calls that may overlap on the GPU (other
 *    streams, other host threads) race on it and must be serialised.
 * Results equal ll_paged_attention_decode's for the same inputs. */
int ll_paged_attention_decode_noalloc(const void* q, const ll_kv_pool* pool,
                                      const int32_t* block_table, int32_t max_blocks,
                                      const int32_t* context_lens, int32_t batch, int32_t n_heads,
                                      int32_t n_kv_heads, int32_t head_dim, int32_t block_size,
                                      float scale, void* out, int32_t* status, void* stream);

/* Workspace bytes for ll_linear. */
size_t ll_linear_workspace_size(int32_t m, int32_t n, int32_t k);

/* Plain Linear y = x w^T (the chain page's Q/K/V, Output, Gate/Up and Down
 * Linear without their fused epilogues): x BF16 [m, k], w BF16 [n, k],
 * y BF16 [m, n], float32 accumulation.  n and k multiples of 16.  Runs the
 * same tensor-core GEMM the layer uses (m <= 256 takes the decode form). */
int ll_linear(const void* x, const void* w, void* y, int32_t m, int32_t n, int32_t k,
              void* workspace, size_t workspace_bytes, int32_t* status, void* stream);

/* Launch tracing, for measurement (off by default).  ll_trace_begin creates
 * 2 * capacity CUDA events on the current device; until ll_trace_end, each
 * kernel launch the library makes is bracketed by two of them, recorded on
 * the launch's stream, and its kernel name kept.  ll_trace_end returns the
 * number of launches recorded (at most capacity; later ones are not traced).
 * Once the stream has been synchronised, ll_trace_elapsed_ms(i) is launch i's
 * duration in milliseconds (-1 on error) and ll_trace_name(i) its kernel.
 * Process-wide state, not thread-safe.  This is a measuring aid the pages do
 * not describe (their profiler is the graph timeline of the ATB debugging
 * section). */
int ll_trace_begin(int32_t capacity);
int32_t ll_trace_end(void);
float ll_trace_elapsed_ms(int32_t i);
const char* ll_trace_name(int32_t i);

/* Self-test of the in-kernel failure detection (not a layer operation): one
 * block of 64 threads waits on an mbarrier that nothing completes, with a
 * limit of limit_us microseconds (1 .. 2,000,000).  Each wait gives up, sets
 * LL_DEV_TIMEOUT in *status and adds 1 to *out (device int32, caller-zeroed),
 * and the kernel finishes normally: the context stays usable. */
int ll_selftest_bounded_wait(int32_t limit_us, int32_t* status, int32_t* out, void* stream);

/* Number of streaming multiprocessors the library sizes its grids for
 * (queried once per device), or -1 without a device. */
int ll_device_sm_count(void);

/* Upper bound on the CTAs of the prefill attention, which is persistent: each
 * CTA (one per SM by default) runs a fixed list of (sequence, query head,
 * 128-query tile) items back to back.  n <= 0 restores one per SM.  A smaller
 * bound leaves SMs to other work on the device, and lets small problems run
 * several items per CTA.  Applies to launches made after the call, from any
 * thread.  Always returns LL_OK. */
int ll_set_prefill_attention_ctas(int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* LLAMA_LAYER_H */
