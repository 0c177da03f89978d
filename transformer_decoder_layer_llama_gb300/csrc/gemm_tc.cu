// Tensor-core GEMM of the decoder layer on sm_103a: D = A * B^T with BF16
// operands staged by TMA (128-byte swizzle) and float32 accumulators in
// TMEM, issued as tcgen05.mma kind::f16 by one thread.  Its epilogues fuse
// the element-wise steps that follow each Linear of the Llama2-7B operator
// chain (page "Which ops-transformer operators one Llama2-7B layer calls",
// section "single-layer operator call chain"): RoPE on the merged QKV output
// plus the ReshapeAndCache write of K/V into the paged pool, the residual add
// after the output and down projections, and SiLU(gate) * up after the merged
// gate/up projection.
//
// Two forms:
//  * token form (more than 256 tokens, prefill): 256 x 256 output tiles of
//    tokens x features on CTA pairs (tcgen05.mma.cta_group::2); persistent
//    pairs walk the tiles token-block-fastest so that pairs running together
//    share the weight tile in L2.
//  * weight form (<= 256 tokens: decode and short prefill chunks): A = weights
//    in 128-row blocks, B = the token rows (MMA N = tokens rounded up to 16,
//    so the weights are streamed exactly once).  Persistent stream-K
//    CTAs (one per SM) split the tiles x K blocks evenly; tiles split between
//    CTAs leave float32 partials in scratch, which a small fix-up kernel,
//    launched right behind, adds up before running the epilogue.
//
// Warp roles (192 threads): warp 0 issues TMA loads, warp 1 allocates TMEM
// and issues the MMAs, warps 2-5 drain TMEM (warp w reads TMEM lanes
// 32*(w%4) .. +31) and run the epilogue.  Two TMEM accumulators let the
// epilogue of one tile overlap the main loop of the next.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace ll {

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn();

constexpr int BM = 128;          // rows of the A block = MMA M
constexpr int BK = 64;           // K per pipeline stage: one 128-byte swizzle row of BF16
constexpr int UK = 16;           // K of one tcgen05.mma kind::f16
constexpr int MAX_STAGES = 8;
constexpr int kThreads = 192;
constexpr int kSwapMaxTokens = 256;

struct GemmArgs {
    EpiParams ep;
    int swap;
    int tokens, n, k;
    int bn;                  // MMA N
    int tiles_m;             // number of A blocks
    int tiles_n;             // number of B blocks
    int num_kb;
    int units;
    int stages;
    uint32_t stage_bytes;
    uint32_t a_bytes;
    uint32_t tmem_cols;
    int w_prefetch;          // weight form: weights may be loaded before the grid dependency wait
    float* partials;         // weight form: [CTAs][2][tokens][128] float32 partial tiles
};

struct TokenSlot {
    int pos;         // -1 if invalid
    long long kv_row;  // row index (blk * Hkv) * bs + off of head 0, or -1
};

LL_DEVINL TokenSlot token_slot(const EpiParams& ep, int t) {
    TokenSlot s{-1, -1};
    int pos = ep.positions ? ep.positions[t] : ep.context_lens[t] - 1;
    if (pos < 0 || pos >= ep.max_position) {
        flag_status(ep.status, LL_DEV_BAD_POSITION);
        return s;
    }
    s.pos = pos;
    if (ep.kv_stage) {                           // staging rows [token][kv head]
        s.kv_row = (long long)t * ep.n_kv_heads;
        return s;
    }
    int seq = t / ep.seq_len;
    int lb = pos / ep.block_size;
    if (lb >= ep.max_blocks) {
        flag_status(ep.status, LL_DEV_BAD_BLOCK);
        return s;
    }
    int blk = ep.block_table[(size_t)seq * ep.max_blocks + lb];
    if (blk < 0 || blk >= ep.num_blocks) {
        flag_status(ep.status, LL_DEV_BAD_BLOCK);
        return s;
    }
    s.kv_row = ((long long)blk * ep.n_kv_heads) * ep.block_size + (pos % ep.block_size);
    return s;
}

// ---------------------------------------------------------------- token-form epilogue
// One thread owns one token row t and 16 consecutive output features n0..n0+15.
LL_DEVINL void epi_token_chunk(const EpiParams& ep, int t, bool row_ok, int n0, int N,
                               const TokenSlot& ts, const float (&v)[16]) {
    if (!row_ok) return;
    switch (ep.kind) {
        case EPI_STORE: {
            if (ep.out_f32) {
                float4* dst = reinterpret_cast<float4*>(ep.out_f32 + (size_t)t * ep.ld_out + n0);
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                break;
            }
            uint4 o0, o1;
            o0.x = pack_bf16x2(v[0], v[1]);   o0.y = pack_bf16x2(v[2], v[3]);
            o0.z = pack_bf16x2(v[4], v[5]);   o0.w = pack_bf16x2(v[6], v[7]);
            o1.x = pack_bf16x2(v[8], v[9]);   o1.y = pack_bf16x2(v[10], v[11]);
            o1.z = pack_bf16x2(v[12], v[13]); o1.w = pack_bf16x2(v[14], v[15]);
            uint4* dst = reinterpret_cast<uint4*>(ep.out + (size_t)t * ep.ld_out + n0);
            dst[0] = o0;
            dst[1] = o1;
            break;
        }
        case EPI_RESID: {
            float r[16];
            if (ep.resid_f32) {
                const float4* rp = reinterpret_cast<const float4*>(ep.resid_f32 + (size_t)t * N + n0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float4 f = rp[j];
                    r[4 * j] = f.x; r[4 * j + 1] = f.y; r[4 * j + 2] = f.z; r[4 * j + 3] = f.w;
                }
            } else {
                const uint4* rp = reinterpret_cast<const uint4*>(ep.resid + (size_t)t * N + n0);
                uint4 r0 = rp[0], r1 = rp[1];
                uint32_t rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    r[2 * j] = bf16_lo(rr[j]);
                    r[2 * j + 1] = bf16_hi(rr[j]);
                }
            }
            if (ep.out_f32) {
                float4* dst = reinterpret_cast<float4*>(ep.out_f32 + (size_t)t * N + n0);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(r[4 * j] + v[4 * j], r[4 * j + 1] + v[4 * j + 1],
                                         r[4 * j + 2] + v[4 * j + 2], r[4 * j + 3] + v[4 * j + 3]);
            } else {
                uint32_t oo[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) oo[j] = pack_bf16x2(r[2 * j] + v[2 * j], r[2 * j + 1] + v[2 * j + 1]);
                uint4* dst = reinterpret_cast<uint4*>(ep.out + (size_t)t * ep.ld_out + n0);
                dst[0] = make_uint4(oo[0], oo[1], oo[2], oo[3]);
                dst[1] = make_uint4(oo[4], oo[5], oo[6], oo[7]);
            }
            break;
        }
        case EPI_SWIGLU: {
            float a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = silu_mul(v[2 * j], v[2 * j + 1]);
            uint4 o;
            o.x = pack_bf16x2(a[0], a[1]); o.y = pack_bf16x2(a[2], a[3]);
            o.z = pack_bf16x2(a[4], a[5]); o.w = pack_bf16x2(a[6], a[7]);
            *reinterpret_cast<uint4*>(ep.out + (size_t)t * ep.ld_out + (n0 >> 1)) = o;
            break;
        }
        case EPI_QKV: {
            const int d = ep.head_dim;
            const int nq = ep.n_heads * d;
            const int nk = ep.n_kv_heads * d;
            if (ts.pos < 0) return;
            int sec, head, e0;
            if (n0 < nq) { sec = 0; head = n0 / d; e0 = n0 - head * d; }
            else if (n0 < nq + nk) { sec = 1; head = (n0 - nq) / d; e0 = n0 - nq - head * d; }
            else { sec = 2; head = (n0 - nq - nk) / d; e0 = n0 - nq - nk - head * d; }
            __nv_bfloat16* base;
            if (sec == 0) {
                base = ep.q_out + (size_t)t * nq + (size_t)head * d;
            } else {
                if (ts.kv_row < 0) return;
                size_t row = (size_t)ts.kv_row + (size_t)head * ep.block_size;
                base = (sec == 1 ? ep.k_pool : ep.v_pool) + row * d;
            }
            if (sec == 2) {
                uint4 o0, o1;
                o0.x = pack_bf16x2(v[0], v[1]);   o0.y = pack_bf16x2(v[2], v[3]);
                o0.z = pack_bf16x2(v[4], v[5]);   o0.w = pack_bf16x2(v[6], v[7]);
                o1.x = pack_bf16x2(v[8], v[9]);   o1.y = pack_bf16x2(v[10], v[11]);
                o1.z = pack_bf16x2(v[12], v[13]); o1.w = pack_bf16x2(v[14], v[15]);
                reinterpret_cast<uint4*>(base + e0)[0] = o0;
                reinterpret_cast<uint4*>(base + e0)[1] = o1;
            } else {
                // packed feature e0 + 2j holds element i = e0/2 + j, e0 + 2j + 1 holds i + d/2
                const int i0 = e0 >> 1;
                const float4* cs4 = reinterpret_cast<const float4*>(
                    ep.rope_cs + (size_t)ts.pos * (d >> 1) + i0);
                float lo[8], hi[8];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    float4 c = cs4[jj];   // (cos, sin) of pairs i0+2jj and i0+2jj+1
                    int j = 2 * jj;
                    const float2 r0 = rope_rotate(v[2 * j], v[2 * j + 1], c.x, c.y);
                    const float2 r1 = rope_rotate(v[2 * j + 2], v[2 * j + 3], c.z, c.w);
                    lo[j] = r0.x;
                    hi[j] = r0.y;
                    lo[j + 1] = r1.x;
                    hi[j + 1] = r1.y;
                }
                uint4 a, b;
                a.x = pack_bf16x2(lo[0], lo[1]); a.y = pack_bf16x2(lo[2], lo[3]);
                a.z = pack_bf16x2(lo[4], lo[5]); a.w = pack_bf16x2(lo[6], lo[7]);
                b.x = pack_bf16x2(hi[0], hi[1]); b.y = pack_bf16x2(hi[2], hi[3]);
                b.z = pack_bf16x2(hi[4], hi[5]); b.w = pack_bf16x2(hi[6], hi[7]);
                *reinterpret_cast<uint4*>(base + i0) = a;
                *reinterpret_cast<uint4*>(base + (d >> 1) + i0) = b;
            }
            break;
        }
    }
}

// ---------------------------------------------------------------- weight-form epilogue
// One thread owns one output feature n (its TMEM lane) and up to 16
// consecutive tokens t0..t0+tcount-1.  All 32 lanes of the warp call this
// together (shuffles).  The shared-memory tables hold tokens tb, tb+1, ...:
// s_pos / s_row the tokens' positions and cache rows (EPI_QKV); cs_s their
// RoPE (cos, sin) rows, [token][head_dim / 2] (EPI_QKV), and rs the residual
// rows of n's 128-feature tile, [token][128] (EPI_RESID), each null to read
// them from global memory instead.
LL_DEVINL void epi_weight_chunk(const EpiParams& ep, int n, int N, int t0, int T,
                                const float (&v)[16], const int* s_pos, const long long* s_row,
                                const float2* cs_s, const uint8_t* rs, int tb, int tcount = 16) {
    const bool n_ok = n < N;
    T = min(T, t0 + tcount);   // this call covers tokens t0 .. min(T, t0 + tcount) - 1
    switch (ep.kind) {
        case EPI_STORE:
            if (n_ok)
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (t0 + j < T) {
                        if (ep.out_f32)
                            ep.out_f32[(size_t)(t0 + j) * ep.ld_out + n] = v[j];
                        else
                            ep.out[(size_t)(t0 + j) * ep.ld_out + n] = __float2bfloat16_rn(v[j]);
                    }
            break;
        case EPI_RESID:
            if (n_ok) {
                // All 16 residuals are at hand before the first store: from shared memory, or
                // requested together from global memory (raw predicated loads, converted after,
                // so that no load waits for the one before it).
                float rv[16];
                const int col = n % 128;
                if (rs) {
                    if (ep.resid_f32) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            rv[j] = reinterpret_cast<const float*>(rs)[(t0 + j - tb) * 128 + col];
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            rv[j] = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(rs)[(t0 + j - tb) * 128 + col]);
                    }
                } else if (ep.resid_f32) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        rv[j] = t0 + j < T ? __ldcg(ep.resid_f32 + (size_t)(t0 + j) * N + n) : 0.f;
                } else {
                    const unsigned short* rb = reinterpret_cast<const unsigned short*>(ep.resid);
                    unsigned short raw[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        raw[j] = t0 + j < T ? __ldcg(rb + (size_t)(t0 + j) * N + n) : (unsigned short)0;
#pragma unroll
                    for (int j = 0; j < 16; ++j) rv[j] = __uint_as_float((uint32_t)raw[j] << 16);
                }
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (t0 + j < T) {
                        const size_t at = (size_t)(t0 + j) * N + n;
                        if (ep.out_f32)
                            ep.out_f32[at] = rv[j] + v[j];
                        else
                            ep.out[(size_t)(t0 + j) * ep.ld_out + n] = __float2bfloat16_rn(rv[j] + v[j]);
                    }
            }
            break;
        case EPI_SWIGLU:
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
                if (n_ok && (n & 1) == 0 && t0 + j < T)
                    ep.out[(size_t)(t0 + j) * ep.ld_out + (n >> 1)] =
                        __float2bfloat16_rn(silu_mul(v[j], other));
            }
            break;
        case EPI_QKV: {
            const int d = ep.head_dim;
            const int nq = ep.n_heads * d;
            const int nk = ep.n_kv_heads * d;
            int sec, head, e;
            if (n < nq) { sec = 0; head = n / d; e = n - head * d; }
            else if (n < nq + nk) { sec = 1; head = (n - nq) / d; e = n - nq - head * d; }
            else { sec = 2; head = (n - nq - nk) / d; e = n - nq - nk - head * d; }
            const int pair = e >> 1;
            const int orig = (sec == 2) ? e : ((e & 1) ? pair + (d >> 1) : pair);
            float other[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) other[j] = __shfl_xor_sync(0xffffffffu, v[j], 1);
            if (!n_ok) break;
            int pj[16];
            long long rj[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                pj[j] = t0 + j < T ? s_pos[t0 + j - tb] : -1;
                rj[j] = t0 + j < T ? s_row[t0 + j - tb] : -1;
            }
            float2 csj[16];
            if (sec != 2) {
                if (cs_s) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) csj[j] = cs_s[(t0 + j - tb) * (d >> 1) + pair];
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        csj[j] = __ldg(ep.rope_cs + (size_t)max(pj[j], 0) * (d >> 1) + pair);
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (pj[j] < 0) continue;
                float val = v[j];
                if (sec != 2) {
                    // lane pair (even, odd) = head elements (i, i + d/2)
                    const float2 cs = csj[j];
                    val = (e & 1) ? rope_rotate(other[j], v[j], cs.x, cs.y).y : rope_rotate(v[j], other[j], cs.x, cs.y).x;
                }
                const __nv_bfloat16 bv = __float2bfloat16_rn(val);
                if (sec == 0) {
                    ep.q_out[(size_t)(t0 + j) * nq + (size_t)head * d + orig] = bv;
                } else if (rj[j] >= 0) {
                    const size_t row = (size_t)rj[j] + (size_t)head * ep.block_size;
                    (sec == 1 ? ep.k_pool : ep.v_pool)[row * d + orig] = bv;
                }
            }
            break;
        }
    }
}

// ---------------------------------------------------------------- token form
// A cluster of two CTAs computes 256 x bn output tiles (bn in [128, 256], chosen per
// shape so that the tiles fill the last wave of pairs; see pair_tile_n) with
// tcgen05.mma.cta_group::2: CTA r stages rows [128 r, 128 r + 128) of the tile's A
// block and rows [bn/2 r, bn/2 (r + 1)) of its B block, the even CTA issues the pair's
// MMAs, and each CTA's TMEM receives its 128 output rows.  Per k-block each CTA moves
// 16 KB + bn/2 x 128 bytes (32 KB, not 48 KB, at bn = 256) for the same MMA work,
// which relieves shared memory.  Both CTAs' TMA loads complete the even CTA's full
// barrier; the MMA commits arrive on both CTAs' barriers (multicast); both CTAs'
// epilogue threads release the even CTA's accumulator barrier.
//
// A stage holds two k-blocks (three stages of 60 KB instead of seven of 30 KB): the
// one thread that issues the MMAs then waits on a barrier once per 8 MMAs instead of
// once per 4, and the tensor pipe no longer idles behind those waits (measured on
// GB300, the 7B prefill layer's four GEMMs: 585 -> 508 us; the same pipeline with no
// operand loads at all ran 535 us with one k-block per stage, so the waits and not the
// operand traffic were the limit; three k-blocks per stage leave two stages and are
// slower).  The per-stage loops are unrolled: a rolled loop over one k-block per stage
// put enough instructions between the MMAs to cost 20%.
constexpr int kPairBN = 256;      // the widest tile; each of the two TMEM accumulators starts a multiple of it apart
constexpr int kPairKbs = 2;       // 64-wide K blocks per stage

__global__ void __launch_bounds__(kThreads, 1)
    gemm_token2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES];
    __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;
    int32_t* status = a.ep.status;
    // a.tiles_m counts 256-row tiles here; a tile has a.bn output columns
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 256);
        }
        mbar_init(&drain_bar, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(&tmem_base_s, a.tmem_cols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();                              // both CTAs' barriers exist before remote use
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = tmem_base_s;
    const uint32_t half_bytes = (uint32_t)BM * BK * 2;     // 16 KB: this CTA's A rows (its B rows follow)
    const uint32_t sub_bytes = half_bytes + (uint32_t)(a.bn >> 1) * BK * 2;   // one K block of A and B

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[MAX_STAGES];
            for (int s = 0; s < MAX_STAGES; ++s) issued[s] = 0;
            bool ok = true;
            for (int u = pair; u < a.units && ok; u += num_pairs) {
                const int m2 = u % a.tiles_m, nb = u / a.tiles_m;
                for (int kb0 = 0; kb0 < a.num_kb; kb0 += kPairKbs) {
                    const int cnt = min(kPairKbs, a.num_kb - kb0);
                    if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, &abort_s, status)) {
                        ok = false;
                        break;
                    }
                    // both CTAs' loads of this stage complete the even CTA's full barrier
                    if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2u * (uint32_t)cnt * sub_bytes);
                    const uint32_t fb = cluster_map(smem_u32(&full_bar[stage]), 0);
#pragma unroll
                    for (int j = 0; j < kPairKbs; ++j) {
                        if (j < cnt) {
                            uint8_t* sa = smem + (size_t)stage * a.stage_bytes + (size_t)j * sub_bytes;
                            tma_load_2d_pair(sa, &tmA, (kb0 + j) * BK, m2 * 256 + (int)rank * BM, fb);
                            tma_load_2d_pair(sa + half_bytes, &tmB, (kb0 + j) * BK,
                                             nb * a.bn + (int)rank * (a.bn >> 1), fb);
                        }
                    }
                    for (int s = 0; s < MAX_STAGES; ++s) issued[s] += (s == stage);
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (abort_s && leader) {
                volatile int never = 0;
                for (int s = 0; s < a.stages; ++s)
                    if (issued[s]) mbar_wait_bounded(&full_bar[s], (issued[s] - 1) & 1, &never, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = umma_idesc_bf16(2 * BM, a.bn);
            int stage = 0;
            uint32_t phase = 0;
            int local = 0;
            bool ok = true;
            const int nbuf = (int)(a.tmem_cols / kPairBN);   // two accumulators, at column 0 and 256
            // operand descriptors: stage 0's, advanced by the stage size (start address in
            // 16-byte units; every address stays below 256 KB, so no carry leaves the field)
            const uint64_t desc0 = umma_desc_sw128(smem_u32(smem));
            const uint64_t stage_step = a.stage_bytes >> 4, sub_step = sub_bytes >> 4, half_step = half_bytes >> 4;
            uint64_t dstage = desc0;
            for (int u = pair; u < a.units && ok; u += num_pairs, ++local) {
                const int buf = local % nbuf;
                const uint32_t accp = (uint32_t)(local / nbuf) & 1;
                if (!mbar_wait_bounded(&tempty_bar[buf], accp ^ 1, &abort_s, status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * kPairBN);
                uint32_t acc0 = 0;                       // the tile's first MMA overwrites
                for (int kb0 = 0; kb0 < a.num_kb; kb0 += kPairKbs) {
                    const int cnt = min(kPairKbs, a.num_kb - kb0);
                    if (!mbar_wait_bounded(&full_bar[stage], phase, &abort_s, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < kPairKbs; ++j) {
                        if (j < cnt) {
                            const uint64_t da = dstage + (uint64_t)j * sub_step;
                            const uint64_t db = da + half_step;
#pragma unroll
                            for (int kk = 0; kk < BK / UK; ++kk)
                                tc_mma_bf16_pair(d_tmem, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc,
                                                 (j == 0 && kk == 0) ? acc0 : 1u);
                        }
                    }
                    acc0 = 1;
                    tc_commit_pair_mc(&empty_bar[stage], 0x3);
                    dstage += stage_step;
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1;
                        dstage = desc0;
                    }
                }
                if (ok) tc_commit_pair_mc(&tfull_bar[buf], 0x3);
            }
            tc_commit_pair_mc(&drain_bar, 0x1);
            volatile int never = 0;
            mbar_wait_bounded(&drain_bar, 0, &never, status);
        }
        __syncwarp();
    } else {
        const int q = warp & 3;
        const int r = q * 32 + lane;             // TMEM lane = token row within this CTA's 128
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int local = 0;
        const int nbuf = (int)(a.tmem_cols / kPairBN);
        for (int u = pair; u < a.units; u += num_pairs, ++local) {
            const int m2 = u % a.tiles_m, nb = u / a.tiles_m;
            const int buf = local % nbuf;
            const uint32_t accp = (uint32_t)(local / nbuf) & 1;
            if (!mbar_wait_bounded(&tfull_bar[buf], accp, &abort_s, status)) break;
            tc_fence_after();
            const uint32_t taddr = tmem + lane_base + (uint32_t)(buf * kPairBN);
            const int t = m2 * 256 + (int)rank * BM + r;
            const bool row_ok = t < a.tokens;
            TokenSlot ts{-1, -1};
            if (a.ep.kind == EPI_QKV && row_ok) ts = token_slot(a.ep, t);
            for (int c = 0; c < a.bn; c += 16) {
                const int n0 = nb * a.bn + c;
                if (n0 >= a.n) break;
                float v[16];
                tmem_ld16(taddr + (uint32_t)c, v);
                epi_token_chunk(a.ep, t, row_ok, n0, a.n, ts, v);
            }
            tc_fence_before();
            // the accumulator is in registers (wait::ld done): release it without waiting
            // for this tile's output stores
            mbar_arrive_cluster_relaxed(cluster_map(smem_u32(&tempty_bar[buf]), 0));
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();                              // no remote arrival or load outstanding
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------- weight form
// Persistent stream-K over the weights.  The tiles_m x num_kb (128-feature
// tile, 64-wide K block) iterations are cut into one contiguous, equal share
// per CTA, so every SM streams the same number of weight bytes whatever the
// tile count.  A share crosses tile boundaries; the part of a tile that one
// CTA covers (a segment) accumulates in one of two TMEM buffers, so the
// epilogue of one segment overlaps the main loop of the next.  A segment that
// covers its whole tile runs the fused epilogue straight from TMEM; any other
// segment stores its float32 partial to scratch (slot 0 for the CTA's first
// segment, slot 1 for its last) and the fix-up kernel finishes the tile.  No
// CTA ever waits for another.  The CTA leaves room in its SM's shared memory
// for fix-up CTAs, which are placed beside it and wait for it to finish.

// First iteration of CTA c's share, and the CTA whose share holds iteration w.
LL_DEVINL int sk_begin(int c, int W, int P) { return (int)((long long)c * W / P); }
LL_DEVINL int sk_owner(int w, int W, int P) { return (int)(((long long)(w + 1) * P - 1) / W); }

constexpr int kMaxWeightCtas = 160;                   // scratch bound: CTAs of one launch
constexpr int kMinItersPerCta = 4;

// bar.red.and over the 128 epilogue threads (named barrier 1): every one of them
// learns whether all of them hold `v`.
LL_DEVINL bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_weight_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const GemmArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t full_bar[MAX_STAGES], empty_bar[MAX_STAGES];
    __shared__ uint64_t tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ int tok_pos_s[kSwapMaxTokens];        // EPI_QKV: per-token position
    __shared__ long long tok_row_s[kSwapMaxTokens];  // ... and pool row of KV head 0 (or -1)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int32_t* status = a.ep.status;
    const int P = (int)gridDim.x;
    const int cta = (int)blockIdx.x;
    const int nkb = a.num_kb;
    const int W = a.tiles_m * nkb;
    const int w0 = sk_begin(cta, W, P), w1 = sk_begin(cta + 1, W, P);

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 128);
        }
        mbar_init(&drain_bar, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_s, a.tmem_cols);
        tmem_relinquish();
    }
    // weights stream once: keep them from pushing the activations out of L2
    const uint64_t pol_w = l2_policy_evict_first();
    // Weights that no kernel still in flight can be writing (the layer's packed
    // weights) fill the first ring of stages before the wait for the previous
    // kernel, so their latency overlaps its tail; the activations come after it.
    const int n_pre = a.w_prefetch ? min(a.stages, w1 - w0) : 0;
    __syncthreads();                             // barriers initialised before the first load
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < n_pre; ++i) {
            const int w = w0 + i, tile = w / nkb, kb = w - tile * nkb;
            mbar_arrive_expect_tx(&full_bar[i], a.stage_bytes);
            tma_load_2d_hint(smem + (size_t)i * a.stage_bytes, &tmW, kb * BK, tile * BM, &full_bar[i], pol_w);
        }
    }
    pdl_wait();
    pdl_trigger();
    if (warp >= 2 && a.ep.kind == EPI_QKV) {
        // each token's position and cache row, once per CTA
        for (int t = threadIdx.x - 64; t < a.tokens; t += 128) {
            TokenSlot ts = token_slot(a.ep, t);
            tok_pos_s[t] = ts.pos;
            tok_row_s[t] = ts.kv_row;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued[MAX_STAGES];
            for (int s = 0; s < MAX_STAGES; ++s) issued[s] = 0;
            for (int w = w0; w < w1; ++w) {
                const int tile = w / nkb, kb = w - tile * nkb;
                uint8_t* sa = smem + (size_t)stage * a.stage_bytes;
                uint8_t* sb = sa + a.a_bytes;
                if (w - w0 < n_pre) {
                    // the weight half of this stage is already on its way
                    tma_load_2d(sb, &tmX, kb * BK, 0, &full_bar[stage]);
                } else {
                    if (!mbar_wait_bounded(&empty_bar[stage], phase ^ 1, &abort_s, status)) break;
                    mbar_arrive_expect_tx(&full_bar[stage], a.stage_bytes);
                    tma_load_2d_hint(sa, &tmW, kb * BK, tile * BM, &full_bar[stage], pol_w);
                    tma_load_2d(sb, &tmX, kb * BK, 0, &full_bar[stage]);
                }
                for (int s = 0; s < MAX_STAGES; ++s) issued[s] += (s == stage);
                if (++stage == a.stages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (abort_s) {
                volatile int never = 0;
                for (int s = 0; s < a.stages; ++s)
                    if (issued[s]) mbar_wait_bounded(&full_bar[s], (issued[s] - 1) & 1, &never, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_bf16(BM, a.bn);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int w = w0, seg = 0; w < w1 && ok; ++seg) {
                const int tile = w / nkb;
                const int ws = w, we = min(w1, (tile + 1) * nkb);
                const int buf = seg & 1;
                const uint32_t accp = (uint32_t)(seg >> 1) & 1;
                if (!mbar_wait_bounded(&tempty_bar[buf], accp ^ 1, &abort_s, status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(buf * a.bn);
                for (; w < we; ++w) {
                    if (!mbar_wait_bounded(&full_bar[stage], phase, &abort_s, status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * a.stage_bytes);
                    const uint32_t sb = sa + a.a_bytes;
                    const uint64_t da = umma_desc_sw128(sa);
                    const uint64_t db = umma_desc_sw128(sb);
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk)
                        tc_mma_bf16(d_tmem, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc,
                                    (w > ws || kk > 0) ? 1u : 0u);
                    tc_commit(&empty_bar[stage]);
                    if (++stage == a.stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (ok) tc_commit(&tfull_bar[buf]);
            }
            tc_commit(&drain_bar);
            volatile int never = 0;
            mbar_wait_bounded(&drain_bar, 0, &never, status);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps 2-5
        const int q = warp & 3;
        const int r = q * 32 + lane;             // TMEM lane = feature row of the tile
        const int T = a.tokens;
        const int et = threadIdx.x - 64;         // 0..127
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const int resid_esz = a.ep.resid_f32 ? 4 : 2;
        if (a.ep.kind == EPI_QKV) {
            // warm L2 with the RoPE rows of the tokens' positions
            const int half = a.ep.head_dim / 2;
            const int lines = half * 8 / 128;
            for (int i = et; i < T * lines; i += 128) {
                const int p = tok_pos_s[i / lines];
                if (p >= 0)
                    prefetch_l2(reinterpret_cast<const uint8_t*>(a.ep.rope_cs + (size_t)p * half) + (i % lines) * 128);
            }
        } else if (a.ep.kind == EPI_RESID) {
            // warm L2 with the residual rows of the tiles this CTA touches
            const int lines = BM * resid_esz / 128;
            const uint8_t* base = a.ep.resid_f32 ? reinterpret_cast<const uint8_t*>(a.ep.resid_f32)
                                                 : reinterpret_cast<const uint8_t*>(a.ep.resid);
            for (int tile = w0 / nkb; tile <= (w1 - 1) / nkb; ++tile)
                for (int i = et; i < T * lines; i += 128) {
                    const int n0 = tile * BM + (i % lines) * (128 / resid_esz);
                    if (n0 < a.n) prefetch_l2(base + ((size_t)(i / lines) * a.n + n0) * resid_esz);
                }
        }

        for (int w = w0, seg = 0; w < w1; ++seg) {
            const int tile = w / nkb;
            const int ws = w, we = min(w1, (tile + 1) * nkb);
            w = we;
            const int buf = seg & 1;
            const uint32_t accp = (uint32_t)(seg >> 1) & 1;
            const bool have = mbar_wait_bounded(&tfull_bar[buf], accp, &abort_s, status);
            if (!epi_all(have)) break;           // all 128 threads leave together
            tc_fence_after();
            const uint32_t taddr = tmem + lane_base + (uint32_t)(buf * a.bn);
            if (ws == tile * nkb && we == (tile + 1) * nkb) {
                const int n = tile * BM + r;
                for (int c = 0; c < a.bn; c += 16) {
                    float v[16];
                    tmem_ld16(taddr + (uint32_t)c, v);
                    epi_weight_chunk(a.ep, n, a.n, c, T, v, tok_pos_s, tok_row_s, nullptr, nullptr, 0);
                }
            } else {
                // a piece of the tile: the CTA's first segment goes to slot 0, its last to slot 1
                float* mine = a.partials + ((size_t)cta * 2 + (ws == w0 ? 0 : 1)) * T * BM;
                for (int c = 0; c < a.bn; c += 16) {
                    float v[16];
                    tmem_ld16(taddr + (uint32_t)c, v);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c + j < T) __stcg(mine + (size_t)(c + j) * BM + r, v[j]);
                }
            }
            tc_fence_before();
            mbar_arrive(&tempty_bar[buf]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

// ---------------------------------------------------------------- weight form: fix-up
// One CTA per (128-feature tile, 16 tokens) of a tile that the stream-K kernel
// split over several CTAs: adds their float32 partials in CTA order (the same
// sum whichever of them finished first: deterministic) and runs the fused
// epilogue.  Launched right behind the stream-K kernel (programmatic dependent
// launch): its CTAs take the SMs as the stream-K CTAs drain and start the
// moment the last one finishes.  Thread r owns feature r of the tile.
constexpr int kFixTokens = 16;

__global__ void __launch_bounds__(BM)
    gemm_weight_fixup_kernel(const GemmArgs a, int P) {
    __shared__ int tok_pos_s[kFixTokens];
    __shared__ long long tok_row_s[kFixTokens];
    __shared__ __align__(16) uint8_t side_s[kFixTokens * 64 * 8];   // RoPE rows or residual rows
    const int tile = blockIdx.x, t0 = blockIdx.y * kFixTokens;
    const int nkb = a.num_kb, W = a.tiles_m * nkb;
    const int c_first = sk_owner(tile * nkb, W, P), c_last = sk_owner((tile + 1) * nkb - 1, W, P);
    const int r = threadIdx.x;
    const int T = a.tokens;
    const int cnt = min(kFixTokens, T - t0);
    const bool split = c_first != c_last;        // else the stream-K kernel finished the tile
    // Before the wait on the stream-K kernel: everything that does not come from it (the
    // token table, RoPE rows and residual rows are inputs of the layer call, complete
    // before the kernel that launched the stream-K kernel finished waiting on its own
    // predecessor).
    const float2* cs_s = reinterpret_cast<const float2*>(side_s);
    const uint8_t* rs = nullptr;
    if (split && a.ep.kind == EPI_QKV) {
        if (r < cnt) {
            TokenSlot ts = token_slot(a.ep, t0 + r);
            tok_pos_s[r] = ts.pos;
            tok_row_s[r] = ts.kv_row;
        }
        __syncthreads();
        const int half = a.ep.head_dim / 2;
        float2* dst = reinterpret_cast<float2*>(side_s);
        for (int i = r; i < cnt * half; i += BM) {
            const int p = tok_pos_s[i / half];
            dst[i] = p >= 0 ? __ldg(a.ep.rope_cs + (size_t)p * half + i % half) : make_float2(0.f, 0.f);
        }
    } else if (split && a.ep.kind == EPI_RESID && tile * BM + r < a.n) {
        // residual rows t0.., features of this tile: [token][128], float32 or BF16
        const int n = tile * BM + r;
        for (int j = 0; j < cnt; ++j) {
            const size_t at = (size_t)(t0 + j) * a.n + n;
            if (a.ep.resid_f32)
                reinterpret_cast<float*>(side_s)[j * BM + r] = __ldg(a.ep.resid_f32 + at);
            else
                reinterpret_cast<__nv_bfloat16*>(side_s)[j * BM + r] = a.ep.resid[at];
        }
    }
    if (a.ep.kind == EPI_RESID) rs = side_s;
    pdl_wait();
    pdl_trigger();
    if (!split) return;
    __syncthreads();
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = 0.f;
    // the contributors in CTA order, up to four partials in flight at once
    for (int c0 = c_first; c0 <= c_last; c0 += 4) {
        float part[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int cc = min(c0 + u, c_last);
            const int slot = (sk_begin(cc, W, P) / nkb == tile) ? 0 : 1;
            const float* pp = a.partials + ((size_t)cc * 2 + slot) * T * BM + (size_t)t0 * BM + r;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                part[u][j] = (c0 + u <= c_last && j < cnt) ? __ldcg(pp + (size_t)j * BM) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + u <= c_last)
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += part[u][j];
    }
    epi_weight_chunk(a.ep, tile * BM + r, a.n, t0, T, v, tok_pos_s, tok_row_s, cs_s, rs, t0, cnt);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D BF16 tensor [rows, inner] row-major, box [box_rows, 64] with the 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
    return make_tmap_bf16_sw128(m, ptr, inner, rows, box_rows);
}

int ceil_div(int a, int b) { return (a + b - 1) / b; }

uint32_t pow2_at_least(uint32_t x) {
    uint32_t p = 32;
    while (p < x) p <<= 1;
    return p;
}

struct Plan {
    bool swap;
    int bn, tiles_m, tiles_n, num_kb, units, stages, ctas_per_sm;
    uint32_t stage_bytes, a_bytes, tmem_cols;
    size_t smem_bytes;
};

// Weight form: one persistent CTA per SM, but never fewer than kMinItersPerCta
// K blocks per CTA (tiny problems use fewer CTAs and fewer partial tiles).
int weight_ctas(int tiles, int num_kb, int sms) {
    const int W = tiles * num_kb;
    return std::max(1, std::min({sms, kMaxWeightCtas, (W + kMinItersPerCta - 1) / kMinItersPerCta}));
}

// Weight form up to 192 tokens (measured on GB300 at 128 and 192 tokens: QKV and
// gate/up projections of a 4096-wide layer 8-25% faster than one row of 256 x 256
// pair tiles, the narrow projections even), and for up to 256 tokens when the pair
// tiles would leave most SMs idle (fewer than one tile per four SMs); else pair
// tiles, which reuse both operands.
bool use_weight_form(int tokens, int n, int sms) {
    if (tokens <= 192) return true;
    if (tokens > kSwapMaxTokens) return false;
    return ceil_div(tokens, 2 * BM) * ceil_div(n, kPairBN) * 4 < sms;
}

// Output columns of a CTA-pair tile: the width in [128, 256] (a multiple of 16) whose tiles
// fill the pairs' waves best, by a model of the time (waves, rounded up) x (width + 16):
// the width stands for the MMA time of a tile, the 16 for the fixed cost of its A block
// and epilogue.  A 2048-token 7B layer then takes 224 (QKV, O, down: 5.8 and 2.0 waves
// instead of 5.05 and 1.7 at 256) and 240 (gate/up: 9.7 waves instead of 9.05).
// Measured on GB300 that layer's four GEMMs went only from 590 to 586 us: a pair streams
// its operands from L2 at about 11 TB/s over the grid, and narrower tiles re-read the
// token block more often, which takes back most of what the fuller waves give.  Small
// shapes gain the most (a 300-token call spreads over twice the pairs).
int pair_tile_n(int tokens, int n, int sms) {
    const int pairs = std::max(1, sms / 2);
    const long long mt = ceil_div(tokens, 2 * BM);
    int best = kPairBN;
    long long best_cost = -1;
    for (int bn = kPairBN; bn >= 128; bn -= 16) {
        const long long waves = (mt * ceil_div(n, bn) + pairs - 1) / pairs;
        const long long cost = waves * (bn + 16);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

Plan make_plan(int tokens, int n, int k, int sms) {
    Plan p{};
    p.swap = use_weight_form(tokens, n, sms);
    p.num_kb = ceil_div(k, BK);
    p.a_bytes = BM * BK * 2;
    if (!p.swap) {
        p.bn = kPairBN;
        p.tiles_m = ceil_div(tokens, BM);
        p.tiles_n = ceil_div(n, p.bn);
        p.stage_bytes = p.a_bytes + p.bn * BK * 2;
        p.stages = 4;
        p.ctas_per_sm = 1;
        p.units = p.tiles_m * p.tiles_n;
        p.tmem_cols = pow2_at_least(2u * (uint32_t)p.bn);
    } else {
        p.bn = std::max(16, ceil_div(tokens, 16) * 16);
        p.tiles_m = ceil_div(n, BM);
        p.tiles_n = 1;
        p.stage_bytes = p.a_bytes + p.bn * BK * 2;
        p.ctas_per_sm = 1;
        // at most ~200 KB, so that fix-up CTAs (< 10 KB) can wait beside the stream-K CTA
        p.stages = std::min(MAX_STAGES, (200 * 1024) / (int)p.stage_bytes);
        p.units = weight_ctas(p.tiles_m, p.num_kb, sms);
        p.tmem_cols = pow2_at_least(2u * (uint32_t)p.bn);   // two accumulators
    }
    p.smem_bytes = (size_t)p.stages * p.stage_bytes + 1024;
    return p;
}

}  // namespace

bool make_tmap_bf16_sw128(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows,
                          uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        set_last_error("cuTensorMapEncodeTiled", "driver entry point not found");
        return false;
    }
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[160];
        snprintf(msg, sizeof(msg), "CUresult %d (inner %llu, rows %llu, box %u x %u)", (int)r,
                 (unsigned long long)inner, (unsigned long long)rows, (unsigned)BK, box_rows);
        set_last_error("cuTensorMapEncodeTiled", msg);
        return false;
    }
    return true;
}

bool make_tmap_u8_sw128(CUtensorMap* m, const void* ptr, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        set_last_error("cuTensorMapEncodeTiled", "driver entry point not found");
        return false;
    }
    cuuint64_t dims[2] = {128, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {128, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[160];
        snprintf(msg, sizeof(msg), "CUresult %d (uint8 rows %llu, box 128 x %u)", (int)r, (unsigned long long)rows,
                 box_rows);
        set_last_error("cuTensorMapEncodeTiled", msg);
        return false;
    }
    return true;
}

int device_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

void gemm_scratch_need(int tokens, int n, int k, size_t* partial_bytes, int* counters) {
    (void)n;
    (void)k;
    *partial_bytes = tokens > kSwapMaxTokens ? 0 : gemm_partial_bound_bytes(tokens);  // token form: none
    *counters = 0;
}

// Two partial tiles [tokens][128] float32 per CTA (its first and its last
// segment), for any call of at most max_tokens tokens.
size_t gemm_partial_bound_bytes(int max_tokens) {
    return (size_t)kMaxWeightCtas * 2 * (size_t)std::min(max_tokens, kSwapMaxTokens) * BM * sizeof(float);
}

int gemm_counter_bound(int n) {
    (void)n;
    return 0;
}

cudaError_t launch_gemm(const GemmProblem& pr, cudaStream_t stream) {
    int sms = device_sm_count();
    if (sms <= 0) return record(cudaErrorNoDevice, "launch_gemm");
    Plan p = make_plan(pr.tokens, pr.n, pr.k, sms);
    GemmArgs a{};
    a.ep = pr.ep;
    a.swap = p.swap;
    a.tokens = pr.tokens;
    a.n = pr.n;
    a.k = pr.k;
    a.bn = p.bn;
    a.tiles_m = p.tiles_m;
    a.tiles_n = p.tiles_n;
    a.num_kb = p.num_kb;
    a.units = p.units;
    a.stages = p.stages;
    a.stage_bytes = p.stage_bytes;
    a.a_bytes = p.a_bytes;
    a.tmem_cols = p.tmem_cols;
    CUtensorMap tmA, tmB;
    bool ok;
    if (!p.swap) {
        ok = make_tmap(&tmA, pr.act, pr.k, pr.tokens, BM) && make_tmap(&tmB, pr.w, pr.k, pr.n, p.bn);
    } else {
        ok = make_tmap(&tmA, pr.w, pr.k, pr.n, BM) && make_tmap(&tmB, pr.act, pr.k, pr.tokens, p.bn);
    }
    if (!ok) return cudaErrorInvalidValue;
    if (!p.swap) {
        // CTA pairs: 256 x 256 tiles, each CTA stages 128 rows of A and of B per stage
        a.tiles_m = ceil_div(pr.tokens, 2 * BM);
        a.bn = pair_tile_n(pr.tokens, pr.n, sms);
        a.tiles_n = ceil_div(pr.n, a.bn);
        a.units = a.tiles_m * a.tiles_n;
        a.stage_bytes = (uint32_t)kPairKbs * (uint32_t)(BM + a.bn / 2) * BK * 2;
        a.stages = std::min(MAX_STAGES, (int)((227 * 1024 - 2048) / a.stage_bytes));
        // two 256-column accumulators per CTA (the epilogue of one tile overlaps the main
        // loop of the next); tcgen05.alloc.cta_group::2 is one allocation made jointly by
        // the pair, at the same TMEM address in both CTAs
        a.tmem_cols = 512;
        CUtensorMap tA2, tB2;
        if (!make_tmap(&tA2, pr.act, pr.k, pr.tokens, BM) ||
            !make_tmap(&tB2, pr.w, pr.k, pr.n, (uint32_t)(a.bn / 2)))
            return cudaErrorInvalidValue;
        const size_t smem = (size_t)a.stages * a.stage_bytes + 1024;
        {
            const cudaError_t e = ensure_func_attr((const void*)gemm_token2_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem,
                                                   "cudaFuncSetAttribute(gemm_token2_kernel)");
            if (e != cudaSuccess) return e;
        }
        const int pairs = std::min(a.units, sms / 2);
        trace_before("gemm_tc", stream);
        cudaError_t e = launch_pdl(gemm_token2_kernel, dim3((unsigned)(2 * pairs)), dim3(kThreads), smem,
                                   stream, 2, tA2, tB2, a);
        trace_after(stream);
        if (e != cudaSuccess) return record(e, "gemm_token2_kernel launch");
        return record(cudaGetLastError(), "gemm_token2_kernel launch");
    }
    {
        const cudaError_t e = ensure_func_attr((const void*)gemm_weight_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem_bytes,
                                               "cudaFuncSetAttribute(gemm_weight_kernel)");
        if (e != cudaSuccess) return e;
    }
    if (!pr.partials || pr.partial_bytes < (size_t)p.units * 2 * pr.tokens * BM * sizeof(float)) {
        set_last_error("launch_gemm", "weight form needs split-K scratch");
        return cudaErrorInvalidValue;
    }
    a.partials = pr.partials;
    a.w_prefetch = pr.w_static ? 1 : 0;
    trace_before("gemm_tc", stream);
    cudaError_t e = launch_pdl(gemm_weight_kernel, dim3((unsigned)p.units), dim3(kThreads), p.smem_bytes,
                               stream, 1, tmA, tmB, a);
    trace_after(stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return record(e, "gemm_weight_kernel launch");
    trace_before("gemm_fixup", stream);
    e = launch_pdl(gemm_weight_fixup_kernel, dim3((unsigned)p.tiles_m, (unsigned)ceil_div(pr.tokens, kFixTokens)),
                   dim3(BM), 0, stream, 1, a, p.units);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "gemm_weight_fixup_kernel launch");
    return record(cudaGetLastError(), "gemm_weight_fixup_kernel launch");
}

}  // namespace ll
