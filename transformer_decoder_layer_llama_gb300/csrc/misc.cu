// Bandwidth-bound kernels of the decoder layer: RMSNorm, the standalone
// ReshapeAndCache scatter, and the setup-time weight packing / RoPE table.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace ll {

namespace {

constexpr int kNormThreads = 256;

// RMSNorm of one token row per CTA (chain page: "x -> RMSNorm"):
// out = bf16(x * r * g), r = 1 / sqrt(mean(x^2) + eps), sums in float32.
// The input row is BF16 (the layer input) or float32 (the residual stream
// after the attention block).  The row is read twice; the second read comes
// from L1/L2.
template <typename In>
struct RowIO;
template <>
struct RowIO<__nv_bfloat16> {
    LL_DEVINL static void load(const __nv_bfloat16* row, int i, float (&f)[8]) {
        uint4 u = reinterpret_cast<const uint4*>(row)[i];
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            f[2 * j] = bf16_lo(w[j]);
            f[2 * j + 1] = bf16_hi(w[j]);
        }
    }
};
template <>
struct RowIO<float> {
    LL_DEVINL static void load(const float* row, int i, float (&f)[8]) {
        float4 a = reinterpret_cast<const float4*>(row)[2 * i];
        float4 b = reinterpret_cast<const float4*>(row)[2 * i + 1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

// One row per CTA.  With NV > 0 each thread keeps its NV 8-element vectors of the row
// (and of the gains) in registers between the sum of squares and the scaling, so the
// row is read once; NV = 0 reads it twice (any width).  The gains live in the packed
// weights, which no kernel still running can be writing (packing synchronises its
// stream), so they load before the grid-dependency wait.
template <typename In, int NV>
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const In* __restrict__ x,
                                                               const float* __restrict__ g,
                                                               __nv_bfloat16* __restrict__ out,
                                                               int hidden, float eps,
                                                               int32_t* zero_ptr, int zero_words) {
    const int t = blockIdx.x;
    const int nv = hidden >> 3;
    const float4* g4 = reinterpret_cast<const float4*>(g);
    float4 ga[NV > 0 ? NV : 1], gb[NV > 0 ? NV : 1];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int i = threadIdx.x + k * blockDim.x;
        if (i < nv) {
            ga[k] = g4[2 * i];
            gb[k] = g4[2 * i + 1];
        }
    }
    pdl_wait();
    pdl_trigger();
    if (zero_ptr && t == 0)
        for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero_ptr[i] = 0;
    const In* xr = x + (size_t)t * hidden;
    float f[NV > 0 ? NV : 1][8];
    float ss = 0.f;
    if (NV > 0) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int i = threadIdx.x + k * blockDim.x;
            if (i < nv) {
                RowIO<In>::load(xr, i, f[k]);
#pragma unroll
                for (int j = 0; j < 8; ++j) ss += f[k][j] * f[k][j];
            }
        }
    } else {
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            RowIO<In>::load(xr, i, f[0]);
#pragma unroll
            for (int j = 0; j < 8; ++j) ss += f[0][j] * f[0][j];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    __shared__ float red[kNormThreads / 32];
    __shared__ float r_s;
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int i = 0; i < (int)(blockDim.x >> 5); ++i) s += red[i];
        r_s = 1.0f / sqrtf(s / (float)hidden + eps);
    }
    __syncthreads();
    const float r = r_s;
    uint4* orow = reinterpret_cast<uint4*>(out + (size_t)t * hidden);
    auto emit = [&](int i, const float (&v)[8], float4 a, float4 b) {
        uint4 o;
        o.x = pack_bf16x2(v[0] * r * a.x, v[1] * r * a.y);
        o.y = pack_bf16x2(v[2] * r * a.z, v[3] * r * a.w);
        o.z = pack_bf16x2(v[4] * r * b.x, v[5] * r * b.y);
        o.w = pack_bf16x2(v[6] * r * b.z, v[7] * r * b.w);
        orow[i] = o;
    };
    if (NV > 0) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int i = threadIdx.x + k * blockDim.x;
            if (i < nv) emit(i, f[k], ga[k], gb[k]);
        }
    } else {
        for (int i = threadIdx.x; i < nv; i += blockDim.x) {
            RowIO<In>::load(xr, i, f[0]);
            emit(i, f[0], g4[2 * i], g4[2 * i + 1]);
        }
    }
}

// Launches rmsnorm_kernel with the register-resident row when each thread holds at most
// four vectors (hidden <= 8192 at 256 threads).
template <typename In>
cudaError_t launch_rmsnorm_any(const In* x, const float* g, __nv_bfloat16* out, int tokens, int hidden,
                               float eps, int32_t* zero_ptr, int zero_words, cudaStream_t stream) {
    const int nv = hidden / 8;
    const int threads = std::min(kNormThreads, std::max(32, ((nv + 31) / 32) * 32));
    const int per = (nv + threads - 1) / threads;
    switch (per) {
        case 1:
            return launch_pdl(rmsnorm_kernel<In, 1>, dim3(tokens), dim3(threads), 0, stream, 1, x, g, out, hidden, eps,
                              zero_ptr, zero_words);
        case 2:
            return launch_pdl(rmsnorm_kernel<In, 2>, dim3(tokens), dim3(threads), 0, stream, 1, x, g, out, hidden, eps,
                              zero_ptr, zero_words);
        case 3:
        case 4:
            return launch_pdl(rmsnorm_kernel<In, 4>, dim3(tokens), dim3(threads), 0, stream, 1, x, g, out, hidden, eps,
                              zero_ptr, zero_words);
        default:
            return launch_pdl(rmsnorm_kernel<In, 0>, dim3(tokens), dim3(threads), 0, stream, 1, x, g, out, hidden, eps,
                              zero_ptr, zero_words);
    }
}

// ReshapeAndCache (paging page, ReshapeAndCacheOperation): one thread moves one
// 16-byte vector of K and the matching vector of V of one (token, head).
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                         const int32_t* __restrict__ slots, int tokens,
                                         int n_kv_heads, int vec_per_row, int block_size,
                                         uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                         long long num_slots, int32_t* status) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long per_tok = (long long)n_kv_heads * vec_per_row;
    if (idx >= per_tok * tokens) return;
    const int t = (int)(idx / per_tok);
    const int rem = (int)(idx - (long long)t * per_tok);
    const int h = rem / vec_per_row;
    const int c = rem - h * vec_per_row;
    const int slot = slots[t];
    if (slot < 0) return;
    if ((long long)slot >= num_slots) {
        if (h == 0 && c == 0) flag_status(status, LL_DEV_BAD_SLOT);
        return;
    }
    const long long blk = slot / block_size;
    const int off = slot - (int)blk * block_size;
    const size_t dst = (((size_t)blk * n_kv_heads + h) * block_size + off) * vec_per_row + c;
    k_pool[dst] = k[idx];
    v_pool[dst] = v[idx];
}

// ReshapeAndCache into an INT8 pool: one warp per (token, KV head) row of
// head_dim values, E = head_dim / 32 per lane.  scale = absmax / 127 and
// code = round-half-even(x / scale) in float32 with IEEE division (the same
// decisions as the reference quantiser); a zero row gets scale 0, codes 0.
template <int E>
__global__ void reshape_and_cache_q8_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                                            const int32_t* __restrict__ slots, const int32_t* __restrict__ positions,
                                            const int32_t* __restrict__ context_lens,
                                            const int32_t* __restrict__ block_table, int max_blocks, int seq_len,
                                            int tokens, int n_kv_heads, int block_size, int8_t* __restrict__ k_pool,
                                            int8_t* __restrict__ v_pool, float* __restrict__ k_scale,
                                            float* __restrict__ v_scale, int num_blocks, int32_t* status) {
    pdl_wait();
    pdl_trigger();
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= (long long)tokens * n_kv_heads) return;          // whole warps
    const int t = (int)(row / n_kv_heads), h = (int)(row - (long long)t * n_kv_heads);
    constexpr int D = 32 * E;
    long long slot;
    if (slots) {
        slot = slots[t];
    } else {
        const int seq = t / seq_len;
        const int pos = positions ? positions[t] : context_lens[seq] - 1;
        if (pos < 0 || pos / block_size >= max_blocks) {
            if (h == 0 && lane == 0) flag_status(status, LL_DEV_BAD_POSITION);
            return;
        }
        const int blk = block_table[(size_t)seq * max_blocks + pos / block_size];
        slot = blk < 0 ? (long long)num_blocks * block_size : (long long)blk * block_size + pos % block_size;
    }
    if (slot < 0) return;
    if (slot >= (long long)num_blocks * block_size) {
        if (h == 0 && lane == 0) flag_status(status, slots ? LL_DEV_BAD_SLOT : LL_DEV_BAD_BLOCK);
        return;
    }
    const long long blk = slot / block_size;
    const int off = (int)(slot - blk * block_size);
    const size_t srow = (size_t)row * D + lane * E;
    const size_t drow = (((size_t)blk * n_kv_heads + h) * block_size + off);
#pragma unroll
    for (int kv = 0; kv < 2; ++kv) {
        const __nv_bfloat16* src = (kv ? v : k) + srow;
        float x[E];
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) {
            x[i] = __bfloat162float(src[i]);
            amax = fmaxf(amax, fabsf(x[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float sc = __fdiv_rn(amax, 127.f);
        int8_t q[E];
#pragma unroll
        for (int i = 0; i < E; ++i) {
            int c = sc > 0.f ? __float2int_rn(__fdiv_rn(x[i], sc)) : 0;
            q[i] = (int8_t)min(127, max(-127, c));
        }
        int8_t* dst = (kv ? v_pool : k_pool) + drow * D + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) dst[i] = q[i];
        if (lane == 0) (kv ? v_scale : k_scale)[drow] = sc;
    }
}

// Packs rows of a [rows, cols] matrix.  mode 0: copy.  mode 1: the merged QKV
// weight, whose first q_k_rows rows (the Q and K heads) are reordered inside
// each head so that packed row 2i holds element i and row 2i+1 holds element
// i + head_dim/2 (the two halves RoPE rotates together).
__global__ void pack_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int rows,
                                 int vec_per_row, int mode, int head_dim, int q_k_rows) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)rows * vec_per_row) return;
    const int r = (int)(idx / vec_per_row);
    const int c = (int)(idx - (long long)r * vec_per_row);
    int sr = r;
    if (mode == 1 && r < q_k_rows) {
        const int head = r / head_dim;
        const int e = r - head * head_dim;
        sr = head * head_dim + ((e & 1) ? (e >> 1) + (head_dim >> 1) : (e >> 1));
    }
    dst[idx] = src[(size_t)sr * vec_per_row + c];
}

// Merged gate/up weight: packed row 2j = gate row j, row 2j+1 = up row j.
__global__ void interleave_rows_kernel(const uint4* __restrict__ a, const uint4* __restrict__ b,
                                       uint4* __restrict__ dst, int rows, int vec_per_row) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)2 * rows * vec_per_row) return;
    const int r = (int)(idx / vec_per_row);
    const int c = (int)(idx - (long long)r * vec_per_row);
    const uint4* src = (r & 1) ? b : a;
    dst[idx] = src[(size_t)(r >> 1) * vec_per_row + c];
}

// RoPE table: cs[pos][i] = (cos, sin)(pos * theta^(-2i/d)), evaluated in float64.
__global__ void rope_table_kernel(float2* cs, int max_position, int head_dim, double theta) {
    const int half = head_dim >> 1;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)max_position * half) return;
    const int pos = (int)(idx / half);
    const int i = (int)(idx - (long long)pos * half);
    const double inv_freq = pow(theta, -(2.0 * i) / (double)head_dim);
    const double ang = (double)pos * inv_freq;
    double s, c;
    sincos(ang, &s, &c);
    cs[idx] = make_float2((float)c, (float)s);
}

// Failure-detection self-test: every thread of the block waits on an mbarrier
// whose phase nothing ever completes, with a limit of limit_ns.  The bounded
// wait must give up, set LL_DEV_TIMEOUT and let the kernel finish; out[0]
// receives the number of threads that returned from the wait.
__global__ void bounded_wait_selftest_kernel(int32_t* status, int32_t* out, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_s;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);      // one arrival needed; none will come
        abort_s = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool done = mbar_wait_bounded(&bar, 0, &abort_s, status, limit_ns);
    if (!done) atomicAdd(out, 1);
}

// ---------------------------------------------------------------- step-by-step operators
// The element-wise operators of the chain as kernels of their own, for the step-by-step
// execution mode (page "ATB fused-operator matrix and KV-cache management", section on
// the engineering limits of fusion granularity).  Their arithmetic is the fused
// epilogues' (rope_rotate, silu_mul, float32 residual adds), so both modes compute the
// same values from the same Linear outputs.

// A token's position: positions[t], or context_lens[t / seq_len] - 1 when positions is null.
LL_DEVINL int token_position(const int32_t* positions, const int32_t* context_lens, int seq_len, int t) {
    return positions ? positions[t] : context_lens[t / seq_len] - 1;
}

// RotaryEmbedding on the merged QKV Linear output (float32 [tokens][nqkv], the packed
// column order: for Q and K heads column 2i holds element i and 2i + 1 element i + d/2,
// V heads in element order).  One thread per (token, head, pair); writes q and k rotated
// and v, each BF16 in element order ([tokens][heads * d]).  A token whose position is
// outside the RoPE table is flagged and skipped, as in the fused epilogue.
__global__ void rope_split_kernel(const float* __restrict__ qkv, const int32_t* __restrict__ positions,
                                  const int32_t* __restrict__ context_lens, int seq_len, int tokens, int n_heads,
                                  int n_kv_heads, int head_dim, int max_position, const float2* __restrict__ rope_cs,
                                  __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ k,
                                  __nv_bfloat16* __restrict__ v, int32_t* status) {
    const int half = head_dim >> 1;
    const int heads = n_heads + 2 * n_kv_heads;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)tokens * heads * half) return;
    const int t = (int)(idx / ((long long)heads * half));
    const int rem = (int)(idx - (long long)t * heads * half);
    const int head = rem / half, i = rem - head * half;
    const int pos = token_position(positions, context_lens, seq_len, t);
    if (pos < 0 || pos >= max_position) {
        if (head == 0 && i == 0) flag_status(status, LL_DEV_BAD_POSITION);
        return;
    }
    const float* row = qkv + (size_t)t * heads * head_dim + (size_t)head * head_dim;
    if (head >= n_heads + n_kv_heads) {           // V: two elements, unrotated
        const int hv = head - n_heads - n_kv_heads;
        __nv_bfloat16* dst = v + ((size_t)t * n_kv_heads + hv) * head_dim;
        dst[2 * i] = __float2bfloat16_rn(row[2 * i]);
        dst[2 * i + 1] = __float2bfloat16_rn(row[2 * i + 1]);
        return;
    }
    const float2 cs = rope_cs[(size_t)pos * half + i];
    const float2 r = rope_rotate(row[2 * i], row[2 * i + 1], cs.x, cs.y);
    __nv_bfloat16* dst = head < n_heads ? q + ((size_t)t * n_heads + head) * head_dim
                                        : k + ((size_t)t * n_kv_heads + (head - n_heads)) * head_dim;
    dst[i] = __float2bfloat16_rn(r.x);
    dst[i + half] = __float2bfloat16_rn(r.y);
}

// The cache slot of each token: block_table[seq][pos / block_size] * block_size + pos %
// block_size; -1 (and a status bit) where the position or its block is out of range.
__global__ void slot_mapping_kernel(const int32_t* __restrict__ positions, const int32_t* __restrict__ context_lens,
                                    int seq_len, int tokens, const int32_t* __restrict__ block_table, int max_blocks,
                                    int block_size, int num_blocks, int max_position, int32_t* __restrict__ slots,
                                    int32_t* status) {
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= tokens) return;
    const int pos = token_position(positions, context_lens, seq_len, t);
    int slot = -1;
    if (pos < 0 || pos >= max_position) {
        flag_status(status, LL_DEV_BAD_POSITION);
    } else if (pos / block_size >= max_blocks) {
        flag_status(status, LL_DEV_BAD_BLOCK);
    } else {
        const int blk = block_table[(size_t)(t / seq_len) * max_blocks + pos / block_size];
        if (blk < 0 || blk >= num_blocks)
            flag_status(status, LL_DEV_BAD_BLOCK);
        else
            slot = blk * block_size + pos % block_size;
    }
    slots[t] = slot;
}

// a[t][j] = bf16(silu(gu[t][2j]) * gu[t][2j + 1]) from the merged gate/up Linear output
// (float32, gate and up columns interleaved).
__global__ void swiglu_kernel(const float2* __restrict__ gu, __nv_bfloat16* __restrict__ a, long long n) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const float2 p = gu[idx];
    a[idx] = __float2bfloat16_rn(silu_mul(p.x, p.y));
}

// out = resid + acc elementwise (float32 add), resid BF16 or float32, out float32 or BF16.
template <typename In, typename Out>
__global__ void residual_add_kernel(const In* __restrict__ resid, const float* __restrict__ acc,
                                    Out* __restrict__ out, long long n) {
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const float r = static_cast<float>(resid[idx]);
    const float s = r + acc[idx];
    if constexpr (sizeof(Out) == 4)
        out[idx] = s;
    else
        out[idx] = __float2bfloat16_rn(s);
}

unsigned blocks_for(long long n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_rope_split(const float* qkv, const int32_t* positions, const int32_t* context_lens, int seq_len,
                              int tokens, int n_heads, int n_kv_heads, int head_dim, int max_position,
                              const float2* rope_cs, __nv_bfloat16* q, __nv_bfloat16* k, __nv_bfloat16* v,
                              int32_t* status, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const long long n = (long long)tokens * (n_heads + 2 * n_kv_heads) * (head_dim / 2);
    trace_before("rope", stream);
    rope_split_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(qkv, positions, context_lens, seq_len, tokens, n_heads,
                                                               n_kv_heads, head_dim, max_position, rope_cs, q, k, v,
                                                               status);
    trace_after(stream);
    return record(cudaGetLastError(), "rope_split launch");
}

cudaError_t launch_slot_mapping(const int32_t* positions, const int32_t* context_lens, int seq_len, int tokens,
                                const int32_t* block_table, int max_blocks, int block_size, int num_blocks,
                                int max_position, int32_t* slots, int32_t* status, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    trace_before("slot_mapping", stream);
    slot_mapping_kernel<<<blocks_for(tokens, 256), 256, 0, stream>>>(positions, context_lens, seq_len, tokens,
                                                                      block_table, max_blocks, block_size, num_blocks,
                                                                      max_position, slots, status);
    trace_after(stream);
    return record(cudaGetLastError(), "slot_mapping launch");
}

cudaError_t launch_swiglu(const float* gate_up, __nv_bfloat16* a, int tokens, int intermediate, cudaStream_t stream) {
    const long long n = (long long)tokens * intermediate;
    if (n <= 0) return cudaSuccess;
    trace_before("swiglu", stream);
    swiglu_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(reinterpret_cast<const float2*>(gate_up), a, n);
    trace_after(stream);
    return record(cudaGetLastError(), "swiglu launch");
}

cudaError_t launch_residual_add(const __nv_bfloat16* resid, const float* acc, float* out, long long n,
                                cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    trace_before("residual_add", stream);
    residual_add_kernel<__nv_bfloat16, float><<<blocks_for(n, 256), 256, 0, stream>>>(resid, acc, out, n);
    trace_after(stream);
    return record(cudaGetLastError(), "residual_add launch");
}

cudaError_t launch_residual_add(const float* resid, const float* acc, __nv_bfloat16* out, long long n,
                                cudaStream_t stream) {
    if (n <= 0) return cudaSuccess;
    trace_before("residual_add", stream);
    residual_add_kernel<float, __nv_bfloat16><<<blocks_for(n, 256), 256, 0, stream>>>(resid, acc, out, n);
    trace_after(stream);
    return record(cudaGetLastError(), "residual_add launch");
}

cudaError_t launch_rmsnorm(const __nv_bfloat16* x, const float* g, __nv_bfloat16* out, int tokens,
                           int hidden, float eps, int32_t* zero_ptr, int zero_words,
                           cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    trace_before("rmsnorm", stream);
    cudaError_t e = launch_rmsnorm_any(x, g, out, tokens, hidden, eps, zero_ptr, zero_words, stream);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "rmsnorm launch");
    return record(cudaGetLastError(), "rmsnorm launch");
}

cudaError_t launch_rmsnorm_f32(const float* x, const float* g, __nv_bfloat16* out, int tokens,
                               int hidden, float eps, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    trace_before("rmsnorm", stream);
    cudaError_t e = launch_rmsnorm_any(x, g, out, tokens, hidden, eps, (int32_t*)nullptr, 0, stream);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "rmsnorm_f32 launch");
    return record(cudaGetLastError(), "rmsnorm_f32 launch");
}

cudaError_t launch_reshape_and_cache(const __nv_bfloat16* k, const __nv_bfloat16* v,
                                     const int32_t* slots, int tokens, int n_kv_heads, int head_dim,
                                     int block_size, __nv_bfloat16* k_pool, __nv_bfloat16* v_pool,
                                     int num_blocks, int32_t* status, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const int vpr = head_dim / 8;
    const long long n = (long long)tokens * n_kv_heads * vpr;
    trace_before("reshape_and_cache", stream);
    reshape_and_cache_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), slots, tokens,
        n_kv_heads, vpr, block_size, reinterpret_cast<uint4*>(k_pool), reinterpret_cast<uint4*>(v_pool),
        (long long)num_blocks * block_size, status);
    trace_after(stream);
    return record(cudaGetLastError(), "reshape_and_cache launch");
}

cudaError_t launch_reshape_and_cache_q8(const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* slots,
                                        const int32_t* positions, const int32_t* context_lens,
                                        const int32_t* block_table, int max_blocks, int seq_len, int tokens,
                                        int n_kv_heads, int head_dim, int block_size, int8_t* k_pool,
                                        int8_t* v_pool, float* k_scale, float* v_scale, int num_blocks,
                                        int32_t* status, cudaStream_t stream) {
    if (tokens <= 0) return cudaSuccess;
    const long long threads = (long long)tokens * n_kv_heads * 32;
    trace_before("reshape_and_cache_q8", stream);
    cudaError_t e = cudaErrorInvalidValue;
#define LL_Q8_LAUNCH(E_)                                                                                    \
    e = launch_pdl(reshape_and_cache_q8_kernel<E_>, dim3(blocks_for(threads, 256)), dim3(256), 0, stream, 1, \
                   k, v, slots, positions, context_lens, block_table, max_blocks, seq_len, tokens,            \
                   n_kv_heads, block_size, k_pool, v_pool, k_scale, v_scale, num_blocks, status)
    switch (head_dim) {
        case 32: LL_Q8_LAUNCH(1); break;
        case 64: LL_Q8_LAUNCH(2); break;
        case 96: LL_Q8_LAUNCH(3); break;
        case 128: LL_Q8_LAUNCH(4); break;
        case 160: LL_Q8_LAUNCH(5); break;
        case 192: LL_Q8_LAUNCH(6); break;
        case 224: LL_Q8_LAUNCH(7); break;
        case 256: LL_Q8_LAUNCH(8); break;
        default: break;
    }
#undef LL_Q8_LAUNCH
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "reshape_and_cache_q8 launch");
    return record(cudaGetLastError(), "reshape_and_cache_q8 launch");
}

cudaError_t launch_pack_rows(const __nv_bfloat16* src, __nv_bfloat16* dst, int rows, int cols,
                             int mode, int head_dim, int q_k_rows, cudaStream_t stream) {
    const int vpr = cols / 8;
    const long long n = (long long)rows * vpr;
    pack_rows_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(reinterpret_cast<const uint4*>(src),
                                                             reinterpret_cast<uint4*>(dst), rows, vpr,
                                                             mode, head_dim, q_k_rows);
    return record(cudaGetLastError(), "pack_rows launch");
}

cudaError_t launch_interleave_rows(const __nv_bfloat16* a, const __nv_bfloat16* b,
                                   __nv_bfloat16* dst, int rows, int cols, cudaStream_t stream) {
    const int vpr = cols / 8;
    const long long n = 2LL * rows * vpr;
    interleave_rows_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(
        reinterpret_cast<const uint4*>(a), reinterpret_cast<const uint4*>(b),
        reinterpret_cast<uint4*>(dst), rows, vpr);
    return record(cudaGetLastError(), "interleave_rows launch");
}

cudaError_t launch_bounded_wait_selftest(int32_t* status, int32_t* out, uint64_t limit_ns,
                                         cudaStream_t stream) {
    trace_before("bounded_wait_selftest", stream);
    bounded_wait_selftest_kernel<<<1, 64, 0, stream>>>(status, out, limit_ns);
    trace_after(stream);
    return record(cudaGetLastError(), "bounded_wait_selftest launch");
}

cudaError_t launch_rope_table(float2* cs, int max_position, int head_dim, double theta,
                              cudaStream_t stream) {
    const long long n = (long long)max_position * (head_dim / 2);
    rope_table_kernel<<<blocks_for(n, 256), 256, 0, stream>>>(cs, max_position, head_dim, theta);
    return record(cudaGetLastError(), "rope_table launch");
}

}  // namespace ll
