// C ABI of the decoder layer (declared in include/llama_layer.h): host-side
// validation, packed-weight and workspace layouts, and the launch sequence of
// one layer call.  Every step of the layer runs in the library's kernels; this
// file only checks arguments, carves buffers and enqueues launches.
//
// Launch sequence of a layer call (one stream, in order):
//   rmsnorm(x, g_attn) -> x_hat
//   gemm[QKV]  x_hat * W_qkv^T, epilogue RoPE(Q,K) -> q, K/V -> paged pool
//   attention  prefill: flash attention over the pool; decode: split-context
//              flash-decoding plus the log-sum-exp combine
//   gemm[O]    o * W_o^T + x -> h
//   rmsnorm(h, g_ffn) -> h_hat
//   gemm[GU]   h_hat * [W_gate;W_up]^T, epilogue silu(gate) * up -> a
//   gemm[DOWN] a * W_down^T + h -> y
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/llama_layer.h"
#include "kernels.h"

using ll::EpiParams;
using ll::GemmProblem;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The decode attention loads K/V in boxes of min(block_size, 64) rows that must
// tile a 64-key span exactly and keep the 1024-byte swizzle alignment.
bool block_size_ok(int bs) { return bs >= 16 && bs <= 256 && (bs & (bs - 1)) == 0; }

bool config_ok(const ll_config* c) {
    if (!c) return false;
    if (c->hidden <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->intermediate <= 0 ||
        c->block_size <= 0 || c->max_position <= 0 || c->head_dim <= 0)
        return false;
    if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return false;
    return true;
}

int config_supported(const ll_config* c) {
    if (!config_ok(c)) return LL_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128) return LL_ERR_UNSUPPORTED;
    if (c->n_heads % c->n_kv_heads != 0) return LL_ERR_UNSUPPORTED;
    if (c->n_heads / c->n_kv_heads > 16) return LL_ERR_UNSUPPORTED;
    if (c->hidden % 16 != 0 || c->intermediate % 16 != 0) return LL_ERR_UNSUPPORTED;
    if (!block_size_ok(c->block_size)) return LL_ERR_UNSUPPORTED;
    return LL_OK;
}

struct PackedLayout {
    size_t qkv, o, gu, down, g_attn, g_ffn, rope, total;
};

PackedLayout packed_layout(const ll_config* c) {
    PackedLayout L{};
    const size_t H = c->hidden, I = c->intermediate, d = c->head_dim;
    const size_t nqkv = (size_t)(c->n_heads + 2 * c->n_kv_heads) * d;
    const size_t nq = (size_t)c->n_heads * d;
    size_t at = 0;
    L.qkv = at;    at = align_up(at + nqkv * H * 2);
    L.o = at;      at = align_up(at + H * nq * 2);
    L.gu = at;     at = align_up(at + 2 * I * H * 2);
    L.down = at;   at = align_up(at + H * I * 2);
    L.g_attn = at; at = align_up(at + H * 4);
    L.g_ffn = at;  at = align_up(at + H * 4);
    L.rope = at;   at = align_up(at + (size_t)c->max_position * (d / 2) * 8);
    L.total = at;
    return L;
}

struct Packed {
    const __nv_bfloat16 *qkv, *o, *gu, *down;
    const float *g_attn, *g_ffn;
    const float2* rope;
};

Packed packed_view(const ll_config* c, const void* base) {
    PackedLayout L = packed_layout(c);
    const uint8_t* b = static_cast<const uint8_t*>(base);
    Packed p;
    p.qkv = reinterpret_cast<const __nv_bfloat16*>(b + L.qkv);
    p.o = reinterpret_cast<const __nv_bfloat16*>(b + L.o);
    p.gu = reinterpret_cast<const __nv_bfloat16*>(b + L.gu);
    p.down = reinterpret_cast<const __nv_bfloat16*>(b + L.down);
    p.g_attn = reinterpret_cast<const float*>(b + L.g_attn);
    p.g_ffn = reinterpret_cast<const float*>(b + L.g_ffn);
    p.rope = reinterpret_cast<const float2*>(b + L.rope);
    return p;
}

// Workspace of a layer call over T tokens with block tables max_blocks wide.  The
// step-by-step mode appends its float32 Linear outputs and the slot mapping; its K and V
// after RoPE take the INT8 staging rows.
struct WsLayout {
    size_t xh, q, o, h, hh, a, kst, vst, partials, counters, attn, total;
    size_t qkv, slots, o_proj, gate_up, down;   // step-by-step only (0 otherwise)
    size_t partial_bytes;
    int counter_words;       // per GEMM
};

WsLayout ws_layout(const ll_config* c, int T, int max_blocks, int mode = LL_MODE_FUSED) {
    WsLayout L{};
    const size_t H = c->hidden, I = c->intermediate;
    const size_t nq = (size_t)c->n_heads * c->head_dim;
    const int nqkv = (c->n_heads + 2 * c->n_kv_heads) * c->head_dim;
    size_t at = 0;
    L.xh = at; at = align_up(at + (size_t)T * H * 2);
    L.q = at;  at = align_up(at + (size_t)T * nq * 2);
    L.o = at;  at = align_up(at + (size_t)T * nq * 2);
    L.h = at;  at = align_up(at + (size_t)T * H * 4);   // float32 residual stream
    L.hh = at; at = align_up(at + (size_t)T * H * 2);
    L.a = at;  at = align_up(at + (size_t)T * I * 2);
    // the new tokens' K and V before quantisation into an INT8 pool
    const size_t kv_row = (size_t)c->n_kv_heads * c->head_dim * 2;
    L.kst = at; at = align_up(at + (size_t)T * kv_row);
    L.vst = at; at = align_up(at + (size_t)T * kv_row);
    L.partial_bytes = ll::gemm_partial_bound_bytes(T);
    L.partials = at; at = align_up(at + L.partial_bytes);
    L.counter_words = std::max({ll::gemm_counter_bound(nqkv), ll::gemm_counter_bound((int)H),
                                ll::gemm_counter_bound(2 * (int)I)});
    L.counters = at; at = align_up(at + (size_t)4 * L.counter_words * 4);
    L.attn = at;
    at = align_up(at + ll::attn_decode_scratch_bytes(T, c->n_heads, c->head_dim, max_blocks,
                                                     c->block_size));
    if (mode == LL_MODE_STEP_BY_STEP) {
        L.qkv = at;     at = align_up(at + (size_t)T * nqkv * 4);
        L.slots = at;   at = align_up(at + (size_t)T * 4);
        L.o_proj = at;  at = align_up(at + (size_t)T * H * 4);
        L.gate_up = at; at = align_up(at + (size_t)T * 2 * I * 4);
        L.down = at;    at = align_up(at + (size_t)T * H * 4);
    }
    L.total = at;
    return L;
}

bool mode_ok(int mode) { return mode == LL_MODE_FUSED || mode == LL_MODE_STEP_BY_STEP; }

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? LL_OK : LL_ERR_CUDA; }

thread_local char g_last_error[512];

bool pool_ok(const ll_kv_pool* p) {
    return p && p->k && p->v && p->num_blocks > 0 && aligned16(p->k) && aligned16(p->v);
}

int run_layer(const ll_config* cfg, const void* packed, const void* x, const int32_t* positions,
              const int32_t* context_lens, int T, int seq_len, int batch, const ll_kv_pool* pool,
              const int32_t* block_table, int max_blocks, void* y, void* workspace,
              size_t workspace_bytes, int32_t* status, cudaStream_t stream, bool decode,
              const ll_kv_pool_q8* pq8 = nullptr) {
    WsLayout L = ws_layout(cfg, T, max_blocks);
    if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return LL_ERR_WORKSPACE;
    Packed P = packed_view(cfg, packed);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto* xh = reinterpret_cast<__nv_bfloat16*>(ws + L.xh);
    auto* q = reinterpret_cast<__nv_bfloat16*>(ws + L.q);
    auto* o = reinterpret_cast<__nv_bfloat16*>(ws + L.o);
    auto* h = reinterpret_cast<float*>(ws + L.h);
    auto* hh = reinterpret_cast<__nv_bfloat16*>(ws + L.hh);
    auto* a = reinterpret_cast<__nv_bfloat16*>(ws + L.a);
    auto* partials = reinterpret_cast<float*>(ws + L.partials);
    auto* counters = reinterpret_cast<int32_t*>(ws + L.counters);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    auto* yb = static_cast<__nv_bfloat16*>(y);
    const int H = cfg->hidden, I = cfg->intermediate, d = cfg->head_dim;
    const int nq = cfg->n_heads * d;
    const int nqkv = (cfg->n_heads + 2 * cfg->n_kv_heads) * d;

    cudaError_t e = ll::launch_rmsnorm(xb, P.g_attn, xh, T, H, cfg->rms_eps, counters,
                                       4 * L.counter_words, stream);
    if (e != cudaSuccess) return LL_ERR_CUDA;

    GemmProblem g{};
    g.w_static = true;                           // the packed weights
    g.partials = partials;
    g.partial_bytes = L.partial_bytes;
    g.counter_cap = L.counter_words;
    g.ep.status = status;

    // merged QKV + RoPE + ReshapeAndCache
    g.act = xh;
    g.w = P.qkv;
    g.tokens = T;
    g.n = nqkv;
    g.k = H;
    g.counters = counters;
    g.ep.kind = ll::EPI_QKV;
    g.ep.q_out = q;
    g.ep.positions = decode ? nullptr : positions;
    g.ep.context_lens = decode ? context_lens : nullptr;
    g.ep.block_table = block_table;
    g.ep.max_blocks = max_blocks;
    g.ep.seq_len = seq_len;
    if (pq8) {
        // K/V go to staging rows, then into the INT8 pool with their scales
        g.ep.kv_stage = 1;
        g.ep.k_pool = reinterpret_cast<__nv_bfloat16*>(ws + L.kst);
        g.ep.v_pool = reinterpret_cast<__nv_bfloat16*>(ws + L.vst);
        g.ep.num_blocks = pq8->num_blocks;
        g.ep.block_size = 1;
    } else {
        g.ep.k_pool = static_cast<__nv_bfloat16*>(pool->k);
        g.ep.v_pool = static_cast<__nv_bfloat16*>(pool->v);
        g.ep.num_blocks = pool->num_blocks;
        g.ep.block_size = cfg->block_size;
    }
    g.ep.n_heads = cfg->n_heads;
    g.ep.n_kv_heads = cfg->n_kv_heads;
    g.ep.head_dim = d;
    g.ep.max_position = cfg->max_position;
    g.ep.rope_cs = P.rope;
    if ((e = ll::launch_gemm(g, stream)) != cudaSuccess) return LL_ERR_CUDA;
    if (pq8 &&
        (e = ll::launch_reshape_and_cache_q8(g.ep.k_pool, g.ep.v_pool, nullptr, decode ? nullptr : positions,
                                             decode ? context_lens : nullptr, block_table, max_blocks, seq_len, T,
                                             cfg->n_kv_heads, d, cfg->block_size, static_cast<int8_t*>(pq8->k),
                                             static_cast<int8_t*>(pq8->v), pq8->k_scale, pq8->v_scale,
                                             pq8->num_blocks, status, stream)) != cudaSuccess)
        return LL_ERR_CUDA;

    // attention
    const float scale = 1.0f / std::sqrt((float)d);
    if (!decode) {
        ll::AttnPrefillArgs at{};
        at.q = q;
        at.k_pool = g.ep.k_pool;
        at.v_pool = g.ep.v_pool;
        at.positions = positions;
        at.block_table = block_table;
        at.max_blocks = max_blocks;
        at.num_blocks = pool->num_blocks;
        at.block_size = cfg->block_size;
        at.batch = batch;
        at.seq_len = seq_len;
        at.n_heads = cfg->n_heads;
        at.n_kv_heads = cfg->n_kv_heads;
        at.head_dim = d;
        at.scale = scale;
        at.out = o;
        at.status = status;
        if ((e = ll::launch_attn_prefill_tc(at, stream)) != cudaSuccess) return LL_ERR_CUDA;
    } else {
        ll::AttnDecodeArgs at{};
        at.q = q;
        if (pq8) {
            at.k_q8 = static_cast<const int8_t*>(pq8->k);
            at.v_q8 = static_cast<const int8_t*>(pq8->v);
            at.k_scale = pq8->k_scale;
            at.v_scale = pq8->v_scale;
        } else {
            at.k_pool = g.ep.k_pool;
            at.v_pool = g.ep.v_pool;
        }
        at.context_lens = context_lens;
        at.block_table = block_table;
        at.max_blocks = max_blocks;
        at.num_blocks = g.ep.num_blocks;
        at.block_size = cfg->block_size;
        at.batch = batch;
        at.n_heads = cfg->n_heads;
        at.n_kv_heads = cfg->n_kv_heads;
        at.head_dim = d;
        at.scale = scale;
        at.out = o;
        const size_t rows = (size_t)batch * cfg->n_heads *
                            ll::attn_decode_max_splits(max_blocks, cfg->block_size);
        at.part_o = reinterpret_cast<float*>(ws + L.attn);
        at.part_ml = at.part_o + rows * d;
        at.status = status;
        if ((e = pq8 ? ll::launch_attn_decode_q8(at, stream) : ll::launch_attn_decode(at, stream)) != cudaSuccess)
            return LL_ERR_CUDA;
    }

    // O projection + residual
    GemmProblem go = g;
    go.act = o;
    go.w = P.o;
    go.n = H;
    go.k = nq;
    go.counters = counters + L.counter_words;
    go.ep = EpiParams{};
    go.ep.kind = ll::EPI_RESID;
    go.ep.out_f32 = h;
    go.ep.ld_out = H;
    go.ep.resid = xb;
    go.ep.status = status;
    if ((e = ll::launch_gemm(go, stream)) != cudaSuccess) return LL_ERR_CUDA;

    if ((e = ll::launch_rmsnorm_f32(h, P.g_ffn, hh, T, H, cfg->rms_eps, stream)) != cudaSuccess)
        return LL_ERR_CUDA;

    // merged gate/up + SwiGLU
    GemmProblem gg = go;
    gg.act = hh;
    gg.w = P.gu;
    gg.n = 2 * I;
    gg.k = H;
    gg.counters = counters + 2 * L.counter_words;
    gg.ep = EpiParams{};
    gg.ep.kind = ll::EPI_SWIGLU;
    gg.ep.out = a;
    gg.ep.ld_out = I;
    gg.ep.status = status;
    if ((e = ll::launch_gemm(gg, stream)) != cudaSuccess) return LL_ERR_CUDA;

    // down + residual
    GemmProblem gd = go;
    gd.act = a;
    gd.w = P.down;
    gd.n = H;
    gd.k = I;
    gd.counters = counters + 3 * L.counter_words;
    gd.ep = EpiParams{};
    gd.ep.kind = ll::EPI_RESID;
    gd.ep.out = yb;
    gd.ep.ld_out = H;
    gd.ep.resid_f32 = h;
    gd.ep.status = status;
    if ((e = ll::launch_gemm(gd, stream)) != cudaSuccess) return LL_ERR_CUDA;
    return LL_OK;
}

// The same chain with every operator its own kernel and every intermediate kept in the
// workspace: RMSNorm -> QKV Linear (float32 out) -> RotaryEmbedding -> slot mapping ->
// ReshapeAndCache -> attention -> O Linear -> residual add -> RMSNorm -> gate/up Linear ->
// SiLU * up -> down Linear -> residual add.
int run_layer_step_by_step(const ll_config* cfg, const void* packed, const void* x, const int32_t* positions,
                           const int32_t* context_lens, int T, int seq_len, int batch, const ll_kv_pool* pool,
                           const int32_t* block_table, int max_blocks, void* y, void* workspace,
                           size_t workspace_bytes, int32_t* status, cudaStream_t stream, bool decode) {
    WsLayout L = ws_layout(cfg, T, max_blocks, LL_MODE_STEP_BY_STEP);
    if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return LL_ERR_WORKSPACE;
    Packed P = packed_view(cfg, packed);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto* xh = reinterpret_cast<__nv_bfloat16*>(ws + L.xh);
    auto* q = reinterpret_cast<__nv_bfloat16*>(ws + L.q);
    auto* o = reinterpret_cast<__nv_bfloat16*>(ws + L.o);
    auto* h = reinterpret_cast<float*>(ws + L.h);
    auto* hh = reinterpret_cast<__nv_bfloat16*>(ws + L.hh);
    auto* a = reinterpret_cast<__nv_bfloat16*>(ws + L.a);
    auto* k_rot = reinterpret_cast<__nv_bfloat16*>(ws + L.kst);
    auto* v_new = reinterpret_cast<__nv_bfloat16*>(ws + L.vst);
    auto* qkv = reinterpret_cast<float*>(ws + L.qkv);
    auto* slots = reinterpret_cast<int32_t*>(ws + L.slots);
    auto* o_proj = reinterpret_cast<float*>(ws + L.o_proj);
    auto* gate_up = reinterpret_cast<float*>(ws + L.gate_up);
    auto* down = reinterpret_cast<float*>(ws + L.down);
    auto* counters = reinterpret_cast<int32_t*>(ws + L.counters);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    const int H = cfg->hidden, I = cfg->intermediate, d = cfg->head_dim;
    const int nq = cfg->n_heads * d;
    const int nqkv = (cfg->n_heads + 2 * cfg->n_kv_heads) * d;
    const int32_t* pos = decode ? nullptr : positions;
    const int32_t* ctx = decode ? context_lens : nullptr;

    if (ll::launch_rmsnorm(xb, P.g_attn, xh, T, H, cfg->rms_eps, counters, 4 * L.counter_words, stream) !=
        cudaSuccess)
        return LL_ERR_CUDA;
    // a plain Linear: float32 output [T][n]
    auto linear = [&](const __nv_bfloat16* act, const __nv_bfloat16* w, int n, int k, float* out, int slot) {
        GemmProblem g{};
        g.w_static = true;
        g.partials = reinterpret_cast<float*>(ws + L.partials);
        g.partial_bytes = L.partial_bytes;
        g.counters = counters + slot * L.counter_words;
        g.counter_cap = L.counter_words;
        g.act = act;
        g.w = w;
        g.tokens = T;
        g.n = n;
        g.k = k;
        g.ep.kind = ll::EPI_STORE;
        g.ep.out_f32 = out;
        g.ep.ld_out = n;
        g.ep.status = status;
        return ll::launch_gemm(g, stream);
    };
    if (linear(xh, P.qkv, nqkv, H, qkv, 0) != cudaSuccess) return LL_ERR_CUDA;
    if (ll::launch_rope_split(qkv, pos, ctx, seq_len, T, cfg->n_heads, cfg->n_kv_heads, d, cfg->max_position,
                              P.rope, q, k_rot, v_new, status, stream) != cudaSuccess)
        return LL_ERR_CUDA;
    if (ll::launch_slot_mapping(pos, ctx, seq_len, T, block_table, max_blocks, cfg->block_size, pool->num_blocks,
                                cfg->max_position, slots, status, stream) != cudaSuccess)
        return LL_ERR_CUDA;
    if (ll::launch_reshape_and_cache(k_rot, v_new, slots, T, cfg->n_kv_heads, d, cfg->block_size,
                                     static_cast<__nv_bfloat16*>(pool->k), static_cast<__nv_bfloat16*>(pool->v),
                                     pool->num_blocks, status, stream) != cudaSuccess)
        return LL_ERR_CUDA;
    const float scale = 1.0f / std::sqrt((float)d);
    if (!decode) {
        ll::AttnPrefillArgs at{};
        at.q = q;
        at.k_pool = static_cast<const __nv_bfloat16*>(pool->k);
        at.v_pool = static_cast<const __nv_bfloat16*>(pool->v);
        at.positions = positions;
        at.block_table = block_table;
        at.max_blocks = max_blocks;
        at.num_blocks = pool->num_blocks;
        at.block_size = cfg->block_size;
        at.batch = batch;
        at.seq_len = seq_len;
        at.n_heads = cfg->n_heads;
        at.n_kv_heads = cfg->n_kv_heads;
        at.head_dim = d;
        at.scale = scale;
        at.out = o;
        at.status = status;
        if (ll::launch_attn_prefill_tc(at, stream) != cudaSuccess) return LL_ERR_CUDA;
    } else {
        ll::AttnDecodeArgs at{};
        at.q = q;
        at.k_pool = static_cast<const __nv_bfloat16*>(pool->k);
        at.v_pool = static_cast<const __nv_bfloat16*>(pool->v);
        at.context_lens = context_lens;
        at.block_table = block_table;
        at.max_blocks = max_blocks;
        at.num_blocks = pool->num_blocks;
        at.block_size = cfg->block_size;
        at.batch = batch;
        at.n_heads = cfg->n_heads;
        at.n_kv_heads = cfg->n_kv_heads;
        at.head_dim = d;
        at.scale = scale;
        at.out = o;
        const size_t rows = (size_t)batch * cfg->n_heads * ll::attn_decode_max_splits(max_blocks, cfg->block_size);
        at.part_o = reinterpret_cast<float*>(ws + L.attn);
        at.part_ml = at.part_o + rows * d;
        at.status = status;
        if (ll::launch_attn_decode(at, stream) != cudaSuccess) return LL_ERR_CUDA;
    }
    if (linear(o, P.o, H, nq, o_proj, 1) != cudaSuccess) return LL_ERR_CUDA;
    if (ll::launch_residual_add(xb, o_proj, h, (long long)T * H, stream) != cudaSuccess) return LL_ERR_CUDA;
    if (ll::launch_rmsnorm_f32(h, P.g_ffn, hh, T, H, cfg->rms_eps, stream) != cudaSuccess) return LL_ERR_CUDA;
    if (linear(hh, P.gu, 2 * I, H, gate_up, 2) != cudaSuccess) return LL_ERR_CUDA;
    if (ll::launch_swiglu(gate_up, a, T, I, stream) != cudaSuccess) return LL_ERR_CUDA;
    if (linear(a, P.down, H, I, down, 3) != cudaSuccess) return LL_ERR_CUDA;
    if (ll::launch_residual_add(h, down, static_cast<__nv_bfloat16*>(y), (long long)T * H, stream) != cudaSuccess)
        return LL_ERR_CUDA;
    return LL_OK;
}

}  // namespace

namespace ll {
namespace {
std::mutex g_attr_mu;
std::map<std::tuple<int, const void*, int>, int> g_attr_set;   // (device, kernel, attribute) -> value
}  // namespace

cudaError_t ensure_func_attr(const void* kernel, cudaFuncAttribute attr, int value, const char* what) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_attr_mu);
    const auto key = std::make_tuple(dev, kernel, (int)attr);
    auto it = g_attr_set.find(key);
    if (it != g_attr_set.end() &&
        (it->second == value || (attr == cudaFuncAttributeMaxDynamicSharedMemorySize && it->second >= value)))
        return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, attr, value);
    if (e != cudaSuccess) return record(e, what);
    g_attr_set[key] = value;
    return cudaSuccess;
}

void set_last_error(const char* where, const char* what) {
    snprintf(g_last_error, sizeof(g_last_error), "%s: %s", where, what);
}
void clear_last_error() { g_last_error[0] = 0; }
cudaError_t record(cudaError_t e, const char* where) {
    if (e != cudaSuccess) set_last_error(where, cudaGetErrorString(e));
    return e;
}

namespace {
struct Trace {
    bool on = false;
    int capacity = 0;
    int count = 0;
    std::vector<cudaEvent_t> ev;
    std::vector<const char*> names;
};
Trace g_trace;

void trace_free() {
    for (cudaEvent_t e : g_trace.ev) cudaEventDestroy(e);
    g_trace.ev.clear();
    g_trace.names.clear();
    g_trace.capacity = g_trace.count = 0;
}
}  // namespace

void trace_before(const char* kernel, cudaStream_t stream) {
    if (!g_trace.on || g_trace.count >= g_trace.capacity) return;
    g_trace.names[g_trace.count] = kernel;
    cudaEventRecord(g_trace.ev[2 * g_trace.count], stream);
}

void trace_after(cudaStream_t stream) {
    if (!g_trace.on || g_trace.count >= g_trace.capacity) return;
    cudaEventRecord(g_trace.ev[2 * g_trace.count + 1], stream);
    ++g_trace.count;
}
}  // namespace ll

extern "C" {

const char* ll_last_error(void) { return g_last_error; }

int ll_trace_begin(int32_t capacity) {
    ll::clear_last_error();
    if (capacity <= 0 || capacity > (1 << 20)) return LL_ERR_INVALID_ARG;
    ll::trace_free();
    ll::g_trace.ev.resize(2 * (size_t)capacity, nullptr);
    ll::g_trace.names.resize(capacity, "");
    for (auto& e : ll::g_trace.ev) {
        if (ll::record(cudaEventCreate(&e), "cudaEventCreate(trace)") != cudaSuccess) {
            e = nullptr;
            ll::trace_free();
            return LL_ERR_CUDA;
        }
    }
    ll::g_trace.capacity = capacity;
    ll::g_trace.count = 0;
    ll::g_trace.on = true;
    return LL_OK;
}

int32_t ll_trace_end(void) {
    ll::g_trace.on = false;
    return ll::g_trace.count;
}

float ll_trace_elapsed_ms(int32_t i) {
    if (i < 0 || i >= ll::g_trace.count) return -1.f;
    float ms = -1.f;
    if (cudaEventElapsedTime(&ms, ll::g_trace.ev[2 * i], ll::g_trace.ev[2 * i + 1]) != cudaSuccess)
        return -1.f;
    return ms;
}

const char* ll_trace_name(int32_t i) {
    if (i < 0 || i >= ll::g_trace.count) return "";
    return ll::g_trace.names[i];
}

const char* ll_strerror(int code) {
    switch (code) {
        case LL_OK: return "ok";
        case LL_ERR_INVALID_ARG: return "invalid argument";
        case LL_ERR_UNSUPPORTED: return "unsupported shape";
        case LL_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case LL_ERR_CUDA: return "CUDA call failed";
        default: return "unknown error";
    }
}

int ll_device_sm_count(void) { return ll::device_sm_count(); }

int ll_set_prefill_attention_ctas(int32_t n) {
    ll::set_prefill_attention_ctas(n);
    return LL_OK;
}

int ll_selftest_bounded_wait(int32_t limit_us, int32_t* status, int32_t* out, void* stream) {
    ll::clear_last_error();
    if (!status || !out || limit_us <= 0 || limit_us > 2000000) return LL_ERR_INVALID_ARG;
    return cuda_rc(ll::launch_bounded_wait_selftest(status, out, (uint64_t)limit_us * 1000ull,
                                                    static_cast<cudaStream_t>(stream)));
}

size_t ll_packed_weights_size(const ll_config* cfg) {
    if (config_supported(cfg) != LL_OK) return 0;
    return packed_layout(cfg).total;
}

int ll_pack_weights(const ll_config* cfg, const ll_weights* w, void* packed, size_t packed_bytes,
                    void* stream_) {
    ll::clear_last_error();
    int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    if (!w || !w->w_qkv || !w->w_o || !w->w_gate || !w->w_up || !w->w_down || !w->g_attn ||
        !w->g_ffn || !packed)
        return LL_ERR_INVALID_ARG;
    if (!aligned16(w->w_qkv) || !aligned16(w->w_o) || !aligned16(w->w_gate) ||
        !aligned16(w->w_up) || !aligned16(w->w_down) || !aligned16(packed))
        return LL_ERR_INVALID_ARG;
    PackedLayout L = packed_layout(cfg);
    if (packed_bytes < L.total) return LL_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    uint8_t* base = static_cast<uint8_t*>(packed);
    const int H = cfg->hidden, I = cfg->intermediate, d = cfg->head_dim;
    const int nqkv = (cfg->n_heads + 2 * cfg->n_kv_heads) * d;
    const int nq = cfg->n_heads * d;
    const int qk_rows = (cfg->n_heads + cfg->n_kv_heads) * d;
    cudaError_t e;
    if ((e = ll::launch_pack_rows(static_cast<const __nv_bfloat16*>(w->w_qkv),
                                  reinterpret_cast<__nv_bfloat16*>(base + L.qkv), nqkv, H, 1, d,
                                  qk_rows, s)) != cudaSuccess)
        return LL_ERR_CUDA;
    if ((e = ll::launch_pack_rows(static_cast<const __nv_bfloat16*>(w->w_o),
                                  reinterpret_cast<__nv_bfloat16*>(base + L.o), H, nq, 0, d, 0, s)) !=
        cudaSuccess)
        return LL_ERR_CUDA;
    if ((e = ll::launch_interleave_rows(static_cast<const __nv_bfloat16*>(w->w_gate),
                                        static_cast<const __nv_bfloat16*>(w->w_up),
                                        reinterpret_cast<__nv_bfloat16*>(base + L.gu), I, H, s)) !=
        cudaSuccess)
        return LL_ERR_CUDA;
    if ((e = ll::launch_pack_rows(static_cast<const __nv_bfloat16*>(w->w_down),
                                  reinterpret_cast<__nv_bfloat16*>(base + L.down), H, I, 0, d, 0,
                                  s)) != cudaSuccess)
        return LL_ERR_CUDA;
    if (ll::record(cudaMemcpyAsync(base + L.g_attn, w->g_attn, (size_t)H * 4,
                                   cudaMemcpyDeviceToDevice, s), "cudaMemcpyAsync(g_attn)") != cudaSuccess ||
        ll::record(cudaMemcpyAsync(base + L.g_ffn, w->g_ffn, (size_t)H * 4,
                                   cudaMemcpyDeviceToDevice, s), "cudaMemcpyAsync(g_ffn)") != cudaSuccess)
        return LL_ERR_CUDA;
    if ((e = ll::launch_rope_table(reinterpret_cast<float2*>(base + L.rope), cfg->max_position, d,
                                   (double)cfg->rope_theta, s)) != cudaSuccess)
        return LL_ERR_CUDA;
    return cuda_rc(ll::record(cudaStreamSynchronize(s), "cudaStreamSynchronize(pack)"));
}

size_t ll_workspace_size(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks) {
    if (config_supported(cfg) != LL_OK || max_tokens <= 0 || max_blocks <= 0) return 0;
    return ws_layout(cfg, max_tokens, max_blocks).total;
}

int ll_layer_prefill(const ll_config* cfg, const void* packed, const void* x,
                     const int32_t* positions, int32_t batch, int32_t seq_len,
                     const ll_kv_pool* pool, const int32_t* block_table, int32_t max_blocks,
                     void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                     void* stream) {
    ll::clear_last_error();
    int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    if (!packed || !x || !positions || !block_table || !y || !status || !pool_ok(pool))
        return LL_ERR_INVALID_ARG;
    if (batch <= 0 || seq_len <= 0 || max_blocks <= 0 || x == y) return LL_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(x) || !aligned16(y)) return LL_ERR_INVALID_ARG;
    if ((long long)batch * seq_len > (1 << 24)) return LL_ERR_UNSUPPORTED;
    return run_layer(cfg, packed, x, positions, nullptr, batch * seq_len, seq_len, batch, pool,
                     block_table, max_blocks, y, workspace, workspace_bytes, status,
                     static_cast<cudaStream_t>(stream), false);
}

int ll_layer_decode_step(const ll_config* cfg, const void* packed, const void* x,
                         const ll_kv_pool* pool, const int32_t* block_table, int32_t max_blocks,
                         const int32_t* context_lens, int32_t batch, void* y, void* workspace,
                         size_t workspace_bytes, int32_t* status, void* stream) {
    ll::clear_last_error();
    int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    if (!packed || !x || !context_lens || !block_table || !y || !status || !pool_ok(pool))
        return LL_ERR_INVALID_ARG;
    if (batch <= 0 || max_blocks <= 0 || x == y) return LL_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(x) || !aligned16(y)) return LL_ERR_INVALID_ARG;
    return run_layer(cfg, packed, x, nullptr, context_lens, batch, 1, batch, pool, block_table,
                     max_blocks, y, workspace, workspace_bytes, status,
                     static_cast<cudaStream_t>(stream), true);
}

int ll_reshape_and_cache(const void* k, const void* v, const int32_t* slot_mapping, int32_t tokens,
                         int32_t n_kv_heads, int32_t head_dim, int32_t block_size,
                         const ll_kv_pool* pool, int32_t* status, void* stream) {
    ll::clear_last_error();
    if (!k || !v || !slot_mapping || !status || !pool_ok(pool)) return LL_ERR_INVALID_ARG;
    if (tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return LL_ERR_INVALID_ARG;
    if (head_dim % 8 != 0) return LL_ERR_UNSUPPORTED;
    if (!aligned16(k) || !aligned16(v)) return LL_ERR_INVALID_ARG;
    return cuda_rc(ll::launch_reshape_and_cache(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), slot_mapping,
        tokens, n_kv_heads, head_dim, block_size, static_cast<__nv_bfloat16*>(pool->k),
        static_cast<__nv_bfloat16*>(pool->v), pool->num_blocks, status,
        static_cast<cudaStream_t>(stream)));
}

int ll_reshape_and_cache_q8(const void* k, const void* v, const int32_t* slot_mapping, int32_t tokens,
                            int32_t n_kv_heads, int32_t head_dim, int32_t block_size,
                            const ll_kv_pool_q8* pool, int32_t* status, void* stream) {
    ll::clear_last_error();
    if (!k || !v || !slot_mapping || !status || !pool || !pool->k || !pool->v || !pool->k_scale ||
        !pool->v_scale || pool->num_blocks <= 0)
        return LL_ERR_INVALID_ARG;
    if (tokens < 0 || n_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return LL_ERR_INVALID_ARG;
    if (head_dim % 32 != 0 || head_dim > 256) return LL_ERR_UNSUPPORTED;
    return cuda_rc(ll::launch_reshape_and_cache_q8(
        static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), slot_mapping, nullptr,
        nullptr, nullptr, 0, 1, tokens, n_kv_heads, head_dim, block_size, static_cast<int8_t*>(pool->k),
        static_cast<int8_t*>(pool->v), pool->k_scale, pool->v_scale, pool->num_blocks, status,
        static_cast<cudaStream_t>(stream)));
}

size_t ll_attention_workspace_size(int32_t batch, int32_t n_heads, int32_t head_dim,
                                   int32_t max_blocks, int32_t block_size) {
    if (batch <= 0 || n_heads <= 0 || head_dim <= 0 || max_blocks <= 0 || block_size <= 0) return 0;
    return align_up(ll::attn_decode_scratch_bytes(batch, n_heads, head_dim, max_blocks, block_size));
}

namespace {
bool pool_q8_ok(const ll_kv_pool_q8* p) {
    return p && p->k && p->v && p->k_scale && p->v_scale && p->num_blocks > 0 && aligned16(p->k) &&
           aligned16(p->v) && aligned16(p->k_scale) && aligned16(p->v_scale);
}
}  // namespace

int ll_paged_attention_decode_q8(const void* q, const ll_kv_pool_q8* pool, const int32_t* block_table,
                                 int32_t max_blocks, const int32_t* context_lens, int32_t batch,
                                 int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                                 int32_t block_size, float scale, void* out, void* workspace,
                                 size_t workspace_bytes, int32_t* status, void* stream) {
    ll::clear_last_error();
    if (!q || !block_table || !context_lens || !out || !status || !pool_q8_ok(pool)) return LL_ERR_INVALID_ARG;
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || max_blocks <= 0 || block_size <= 0)
        return LL_ERR_INVALID_ARG;
    if (head_dim != 128) return LL_ERR_UNSUPPORTED;
    if (n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > 16) return LL_ERR_UNSUPPORTED;
    if (!block_size_ok(block_size)) return LL_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out)) return LL_ERR_INVALID_ARG;
    const size_t need = ll_attention_workspace_size(batch, n_heads, head_dim, max_blocks, block_size);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LL_ERR_WORKSPACE;
    ll::AttnDecodeArgs at{};
    at.q = static_cast<const __nv_bfloat16*>(q);
    at.k_q8 = static_cast<const int8_t*>(pool->k);
    at.v_q8 = static_cast<const int8_t*>(pool->v);
    at.k_scale = pool->k_scale;
    at.v_scale = pool->v_scale;
    at.context_lens = context_lens;
    at.block_table = block_table;
    at.max_blocks = max_blocks;
    at.num_blocks = pool->num_blocks;
    at.block_size = block_size;
    at.batch = batch;
    at.n_heads = n_heads;
    at.n_kv_heads = n_kv_heads;
    at.head_dim = head_dim;
    at.scale = scale;
    at.out = static_cast<__nv_bfloat16*>(out);
    const size_t rows = (size_t)batch * n_heads * ll::attn_decode_max_splits(max_blocks, block_size);
    at.part_o = static_cast<float*>(workspace);
    at.part_ml = at.part_o + rows * head_dim;
    at.status = status;
    return cuda_rc(ll::launch_attn_decode_q8(at, static_cast<cudaStream_t>(stream)));
}

int ll_layer_decode_step_q8(const ll_config* cfg, const void* packed, const void* x, const ll_kv_pool_q8* pool,
                            const int32_t* block_table, int32_t max_blocks, const int32_t* context_lens,
                            int32_t batch, void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                            void* stream) {
    ll::clear_last_error();
    int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    if (cfg->head_dim != 128) return LL_ERR_UNSUPPORTED;
    if (!packed || !x || !context_lens || !block_table || !y || !status || !pool_q8_ok(pool))
        return LL_ERR_INVALID_ARG;
    if (batch <= 0 || max_blocks <= 0 || x == y) return LL_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(x) || !aligned16(y)) return LL_ERR_INVALID_ARG;
    return run_layer(cfg, packed, x, nullptr, context_lens, batch, 1, batch, nullptr, block_table, max_blocks, y,
                     workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream), true, pool);
}

int ll_paged_attention_decode(const void* q, const ll_kv_pool* pool, const int32_t* block_table,
                              int32_t max_blocks, const int32_t* context_lens, int32_t batch,
                              int32_t n_heads, int32_t n_kv_heads, int32_t head_dim,
                              int32_t block_size, float scale, void* out, void* workspace,
                              size_t workspace_bytes, int32_t* status, void* stream) {
    ll::clear_last_error();
    if (!q || !block_table || !context_lens || !out || !status || !pool_ok(pool))
        return LL_ERR_INVALID_ARG;
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || max_blocks <= 0 || block_size <= 0)
        return LL_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return LL_ERR_UNSUPPORTED;
    if (n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > 16) return LL_ERR_UNSUPPORTED;
    if (!block_size_ok(block_size)) return LL_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out)) return LL_ERR_INVALID_ARG;
    const size_t need = ll_attention_workspace_size(batch, n_heads, head_dim, max_blocks, block_size);
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LL_ERR_WORKSPACE;
    ll::AttnDecodeArgs at{};
    at.q = static_cast<const __nv_bfloat16*>(q);
    at.k_pool = static_cast<const __nv_bfloat16*>(pool->k);
    at.v_pool = static_cast<const __nv_bfloat16*>(pool->v);
    at.context_lens = context_lens;
    at.block_table = block_table;
    at.max_blocks = max_blocks;
    at.num_blocks = pool->num_blocks;
    at.block_size = block_size;
    at.batch = batch;
    at.n_heads = n_heads;
    at.n_kv_heads = n_kv_heads;
    at.head_dim = head_dim;
    at.scale = scale;
    at.out = static_cast<__nv_bfloat16*>(out);
    const size_t rows = (size_t)batch * n_heads * ll::attn_decode_max_splits(max_blocks, block_size);
    at.part_o = static_cast<float*>(workspace);
    at.part_ml = at.part_o + rows * head_dim;
    at.status = status;
    return cuda_rc(ll::launch_attn_decode(at, static_cast<cudaStream_t>(stream)));
}

int ll_workspace_checkpoints(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks,
                             ll_checkpoints* out) {
    ll::clear_last_error();
    if (!out || max_tokens <= 0 || max_blocks <= 0) return LL_ERR_INVALID_ARG;
    const int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    const WsLayout L = ws_layout(cfg, max_tokens, max_blocks);
    out->x_hat = L.xh;
    out->q = L.q;
    out->o = L.o;
    out->h = L.h;
    out->h_hat = L.hh;
    out->a = L.a;
    return LL_OK;
}

size_t ll_workspace_size_mode(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks, int32_t mode) {
    if (config_supported(cfg) != LL_OK || max_tokens <= 0 || max_blocks <= 0 || !mode_ok(mode)) return 0;
    return ws_layout(cfg, max_tokens, max_blocks, mode).total;
}

int ll_workspace_step_checkpoints(const ll_config* cfg, int32_t max_tokens, int32_t max_blocks,
                                  ll_step_checkpoints* out) {
    ll::clear_last_error();
    if (!out || max_tokens <= 0 || max_blocks <= 0) return LL_ERR_INVALID_ARG;
    const int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    const WsLayout L = ws_layout(cfg, max_tokens, max_blocks, LL_MODE_STEP_BY_STEP);
    out->qkv = L.qkv;
    out->k = L.kst;
    out->v = L.vst;
    out->slots = L.slots;
    out->o_proj = L.o_proj;
    out->gate_up = L.gate_up;
    out->down = L.down;
    return LL_OK;
}

int ll_layer_prefill_mode(const ll_config* cfg, const void* packed, const void* x, const int32_t* positions,
                          int32_t batch, int32_t seq_len, const ll_kv_pool* pool, const int32_t* block_table,
                          int32_t max_blocks, void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                          int32_t mode, void* stream) {
    if (!mode_ok(mode)) return LL_ERR_INVALID_ARG;
    if (mode == LL_MODE_FUSED)
        return ll_layer_prefill(cfg, packed, x, positions, batch, seq_len, pool, block_table, max_blocks, y,
                                workspace, workspace_bytes, status, stream);
    ll::clear_last_error();
    int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    if (!packed || !x || !positions || !block_table || !y || !status || !pool_ok(pool)) return LL_ERR_INVALID_ARG;
    if (batch <= 0 || seq_len <= 0 || max_blocks <= 0 || x == y) return LL_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(x) || !aligned16(y)) return LL_ERR_INVALID_ARG;
    if ((long long)batch * seq_len > (1 << 24)) return LL_ERR_UNSUPPORTED;
    return run_layer_step_by_step(cfg, packed, x, positions, nullptr, batch * seq_len, seq_len, batch, pool,
                                  block_table, max_blocks, y, workspace, workspace_bytes, status,
                                  static_cast<cudaStream_t>(stream), false);
}

int ll_layer_decode_step_mode(const ll_config* cfg, const void* packed, const void* x, const ll_kv_pool* pool,
                              const int32_t* block_table, int32_t max_blocks, const int32_t* context_lens,
                              int32_t batch, void* y, void* workspace, size_t workspace_bytes, int32_t* status,
                              int32_t mode, void* stream) {
    if (!mode_ok(mode)) return LL_ERR_INVALID_ARG;
    if (mode == LL_MODE_FUSED)
        return ll_layer_decode_step(cfg, packed, x, pool, block_table, max_blocks, context_lens, batch, y, workspace,
                                    workspace_bytes, status, stream);
    ll::clear_last_error();
    int rc = config_supported(cfg);
    if (rc != LL_OK) return rc;
    if (!packed || !x || !context_lens || !block_table || !y || !status || !pool_ok(pool))
        return LL_ERR_INVALID_ARG;
    if (batch <= 0 || max_blocks <= 0 || x == y) return LL_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(x) || !aligned16(y)) return LL_ERR_INVALID_ARG;
    return run_layer_step_by_step(cfg, packed, x, nullptr, context_lens, batch, 1, batch, pool, block_table,
                                  max_blocks, y, workspace, workspace_bytes, status, static_cast<cudaStream_t>(stream),
                                  true);
}

size_t ll_linear_workspace_size(int32_t m, int32_t n, int32_t k) {
    if (m <= 0 || n <= 0 || k <= 0) return 0;
    size_t pb = 0;
    int cw = 0;
    ll::gemm_scratch_need(m, n, k, &pb, &cw);
    return align_up(pb) + align_up((size_t)std::max(cw, 1) * 4);
}

int ll_linear(const void* x, const void* w, void* y, int32_t m, int32_t n, int32_t k,
              void* workspace, size_t workspace_bytes, int32_t* status, void* stream) {
    ll::clear_last_error();
    if (!x || !w || !y || !status) return LL_ERR_INVALID_ARG;
    if (m <= 0 || n <= 0 || k <= 0) return LL_ERR_INVALID_ARG;
    if (n % 16 != 0 || k % 16 != 0) return LL_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return LL_ERR_INVALID_ARG;
    size_t pb = 0;
    int cw = 0;
    ll::gemm_scratch_need(m, n, k, &pb, &cw);
    const size_t need = ll_linear_workspace_size(m, n, k);
    if (workspace_bytes < need || (need && !workspace) || (workspace && !aligned16(workspace)))
        return LL_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    GemmProblem g{};
    g.act = static_cast<const __nv_bfloat16*>(x);
    g.w = static_cast<const __nv_bfloat16*>(w);
    g.tokens = m;
    g.n = n;
    g.k = k;
    g.partials = pb ? reinterpret_cast<float*>(ws) : nullptr;
    g.partial_bytes = pb;
    g.counters = reinterpret_cast<int32_t*>(ws + align_up(pb));
    g.counter_cap = std::max(cw, 1);
    g.ep.kind = ll::EPI_STORE;
    g.ep.out = static_cast<__nv_bfloat16*>(y);
    g.ep.ld_out = n;
    g.ep.status = status;
    if (cw > 0 && ll::record(cudaMemsetAsync(g.counters, 0, (size_t)cw * 4, s),
                             "cudaMemsetAsync(counters)") != cudaSuccess)
        return LL_ERR_CUDA;
    return cuda_rc(ll::launch_gemm(g, s));
}

}  // extern "C"
