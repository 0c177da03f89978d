// Internal launcher interface between the C-ABI layer (api.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ll {

// Launches `kernel` with programmatic dependent launch (it may be scheduled while
// the previous kernel in the stream finishes; the kernel itself waits for that
// kernel with griddepcontrol.wait) and, when cluster_x > 1, as clusters of
// cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = grid;
    lc.blockDim = block;
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute at[2];
    unsigned n = 0;
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        at[n].id = cudaLaunchAttributeClusterDimension;
        at[n].val.clusterDim.x = cluster_x;
        at[n].val.clusterDim.y = 1;
        at[n].val.clusterDim.z = 1;
        ++n;
    }
    lc.attrs = at;
    lc.numAttrs = n;
    return cudaLaunchKernelEx(&lc, kernel, static_cast<Args&&>(args)...);
}

enum EpiKind : int {
    EPI_STORE = 0,   // out = acc (BF16 `out`, or float32 `out_f32`)
    EPI_RESID = 1,   // out = resid + acc (O projection, down projection); resid and out may be fp32
    EPI_SWIGLU = 2,  // out[j] = silu(acc[2j]) * acc[2j+1] (merged gate/up, rows interleaved)
    EPI_QKV = 3,     // RoPE on Q/K, Q -> q_out, K/V -> paged pool (merged QKV)
};

struct EpiParams {
    int kind;
    __nv_bfloat16* out;            // STORE / RESID / SWIGLU destination [tokens, ld_out]
    int ld_out;
    const __nv_bfloat16* resid;    // RESID: [tokens, n] BF16 residual, or
    const float* resid_f32;        //        [tokens, n] float32 residual (one of the two)
    float* out_f32;                // STORE / RESID: float32 destination instead of `out`
    // EPI_QKV
    __nv_bfloat16* q_out;          // [tokens, n_heads * head_dim]
    __nv_bfloat16* k_pool;         // the paged pool, or with kv_stage a staging buffer
    __nv_bfloat16* v_pool;         // [tokens, n_kv_heads, head_dim] (block_size then 1)
    int kv_stage;
    const int32_t* positions;      // prefill: position of each token (null in decode)
    const int32_t* context_lens;   // decode: position = context_lens[token] - 1
    const int32_t* block_table;
    int max_blocks;
    int seq_len;                   // tokens per sequence (decode: 1)
    int num_blocks;
    int block_size;
    int n_heads;
    int n_kv_heads;
    int head_dim;
    int max_position;
    const float2* rope_cs;         // [max_position][head_dim / 2] (cos, sin)
    int32_t* status;
};

struct GemmProblem {
    const __nv_bfloat16* act;      // [tokens, k]
    const __nv_bfloat16* w;        // [n, k]
    int tokens, n, k;
    EpiParams ep;
    float* partials;               // split-K scratch (swap form), may be null when splits == 1
    size_t partial_bytes;
    int32_t* counters;             // one per output tile, zero on entry, left zero on exit
    int counter_cap;
    bool w_static;                 // w is not written by any kernel that may still be running
                                   // (it may be read before the wait on the previous kernel)
};

// Scratch the GEMM may need for a problem of this shape (bytes of float
// partials, number of tile counters).
void gemm_scratch_need(int tokens, int n, int k, size_t* partial_bytes, int* counters);
size_t gemm_partial_bound_bytes(int max_tokens);   // bound over all calls of <= max_tokens tokens
int gemm_counter_bound(int n);          // counters needed for an output of n features

cudaError_t launch_gemm(const GemmProblem& p, cudaStream_t stream);

// Tensor map of a row-major BF16 matrix [rows, inner] read in boxes of
// box_rows x 64 elements with the 128-byte swizzle (the layout tcgen05 and
// the ldmatrix readers expect).  Records the reason and returns false on error.
bool make_tmap_bf16_sw128(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                          uint32_t box_rows);

// Tensor map of 128-byte rows of bytes [rows, 128] (an INT8 K/V pool with head_dim
// 128) read in boxes of box_rows full rows with the 128-byte swizzle.
bool make_tmap_u8_sw128(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t box_rows);

int device_sm_count();

// Sets function attribute `attr` of `kernel` to `value` on the current device, once per
// (device, kernel, attribute): function attributes belong to each device's context, so a
// process driving several GPUs configures each.  For the dynamic shared-memory size the
// largest value asked for so far stays set.  Thread-safe; records the failing step.
cudaError_t ensure_func_attr(const void* kernel, cudaFuncAttribute attr, int value, const char* what);

// Records why the current call failed (thread-local; read by ll_last_error).
void set_last_error(const char* where, const char* what);
void clear_last_error();
cudaError_t record(cudaError_t e, const char* where);

// Launch tracing hooks (no-ops unless ll_trace_begin is active).
void trace_before(const char* kernel, cudaStream_t stream);
void trace_after(cudaStream_t stream);

// RMSNorm: out[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps) * g) of a BF16 or a
// float32 input; also zeroes `zero_words` int32 words at `zero_ptr` (tile
// counters) when non-null.
cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const float* g, __nv_bfloat16* out, int tokens,
                           int hidden, float eps, int32_t* zero_ptr, int zero_words,
                           cudaStream_t stream);
cudaError_t launch_rmsnorm_f32(const float* x, const float* g, __nv_bfloat16* out, int tokens,
                               int hidden, float eps, cudaStream_t stream);

// ReshapeAndCache into an INT8 pool (one warp per token and KV head: absmax, float32
// scale = absmax / 127, round-half-even codes).  A token's slot comes from `slots`
// when non-null, else from its position (positions[t], or context_lens[t / seq_len] - 1
// when positions is null) through block_table (sequence t / seq_len).
cudaError_t launch_reshape_and_cache_q8(const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* slots,
                                        const int32_t* positions, const int32_t* context_lens,
                                        const int32_t* block_table, int max_blocks, int seq_len, int tokens,
                                        int n_kv_heads, int head_dim, int block_size, int8_t* k_pool,
                                        int8_t* v_pool, float* k_scale, float* v_scale, int num_blocks,
                                        int32_t* status, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const __nv_bfloat16* k, const __nv_bfloat16* v,
                                     const int32_t* slots, int tokens, int n_kv_heads, int head_dim,
                                     int block_size, __nv_bfloat16* k_pool, __nv_bfloat16* v_pool,
                                     int num_blocks, int32_t* status, cudaStream_t stream);

struct AttnPrefillArgs {
    const __nv_bfloat16* q;        // [tokens, n_heads, d]
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    const int32_t* positions;      // [tokens]
    const int32_t* block_table;
    int max_blocks, num_blocks, block_size;
    int batch, seq_len, n_heads, n_kv_heads, head_dim;
    float scale;
    __nv_bfloat16* out;            // [tokens, n_heads, d]
    int32_t* status;
};
cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t stream);
void set_prefill_attention_ctas(int n);   // 0: one CTA per SM

struct AttnDecodeArgs {
    const __nv_bfloat16* q;        // [batch, n_heads, d]
    const __nv_bfloat16* k_pool;
    const __nv_bfloat16* v_pool;
    const int32_t* context_lens;
    const int32_t* block_table;
    int max_blocks, num_blocks, block_size;
    int batch, n_heads, n_kv_heads, head_dim;
    float scale;
    __nv_bfloat16* out;            // [batch, n_heads, d]
    float* part_o;                 // scratch [batch, n_heads, max_splits, d]
    float* part_ml;                // scratch [batch, n_heads, max_splits, 2]
    int32_t* status;
    const int8_t* k_q8;            // INT8 pool codes (launch_attn_decode_q8) ...
    const int8_t* v_q8;
    const float* k_scale;          // ... and their scales [num_blocks, n_kv_heads, block_size]
    const float* v_scale;
    int4* order;                   // dispatch order of the split grid, in the scratch (set by the launcher)
};
int attn_decode_max_splits(int max_blocks, int block_size);
size_t attn_decode_scratch_bytes(int batch, int n_heads, int head_dim, int max_blocks,
                                 int block_size);
cudaError_t launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t stream);
// Decode attention over an INT8 pool (k_q8/v_q8 + scales; head_dim 128).
cudaError_t launch_attn_decode_q8(const AttnDecodeArgs& a, cudaStream_t stream);

// Step-by-step operators (each one kernel; arithmetic as in the fused epilogues).
// RotaryEmbedding of the merged QKV Linear output (float32, packed column order) into
// q, k (rotated) and v, BF16 [tokens][heads * head_dim] in element order.
cudaError_t launch_rope_split(const float* qkv, const int32_t* positions, const int32_t* context_lens, int seq_len,
                              int tokens, int n_heads, int n_kv_heads, int head_dim, int max_position,
                              const float2* rope_cs, __nv_bfloat16* q, __nv_bfloat16* k, __nv_bfloat16* v,
                              int32_t* status, cudaStream_t stream);
// Cache slot of each token from its position and the block table (-1 where invalid).
cudaError_t launch_slot_mapping(const int32_t* positions, const int32_t* context_lens, int seq_len, int tokens,
                                const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                int max_position, int32_t* slots, int32_t* status, cudaStream_t stream);
// a = bf16(silu(gate) * up) from the merged gate/up Linear output (float32, interleaved).
cudaError_t launch_swiglu(const float* gate_up, __nv_bfloat16* a, int tokens, int intermediate, cudaStream_t stream);
// out = resid + acc (float32 add) over n elements.
cudaError_t launch_residual_add(const __nv_bfloat16* resid, const float* acc, float* out, long long n,
                                cudaStream_t stream);
cudaError_t launch_residual_add(const float* resid, const float* acc, __nv_bfloat16* out, long long n,
                                cudaStream_t stream);

// Weight packing helpers.
cudaError_t launch_pack_rows(const __nv_bfloat16* src, __nv_bfloat16* dst, int rows, int cols,
                             int mode, int head_dim, int q_k_rows, cudaStream_t stream);
cudaError_t launch_interleave_rows(const __nv_bfloat16* a, const __nv_bfloat16* b,
                                   __nv_bfloat16* dst, int rows, int cols, cudaStream_t stream);
cudaError_t launch_rope_table(float2* cs, int max_position, int head_dim, double theta,
                              cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(int32_t* status, int32_t* out, uint64_t limit_ns,
                                         cudaStream_t stream);

}  // namespace ll
