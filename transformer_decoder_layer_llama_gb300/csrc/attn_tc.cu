// Prefill flash attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA):
// the FlashAttention operator of the Llama2-7B operator chain (page "Which
// ops-transformer operators one Llama2-7B layer calls", sections "single-layer
// operator call chain" and "KV Cache and the operators": MatMul -> Softmax ->
// MatMul fused, the whole sequence in one kernel).
//
// One CTA = 128 queries of one sequence and one query head (GQA: KV head
// h / (Hq / Hkv)).  Keys come from the paged pool through block_table, 128 at
// a time, in causal order up to the tile's last query position.
//
// Warp roles (320 threads):
//  * warp 0, one lane: TMA.  Q once (two 64-column boxes), then per key tile K
//    and V as boxes of min(block_size, 128) rows x 64 columns at the physical
//    block's rows, each double-buffered, K loaded one tile ahead of V.
//  * warp 1, one lane: tcgen05.mma.  S_j = Q K_j^T (M 128, N 128, K = head_dim,
//    Q as an A operand in TMEM: the softmax warps copy it there from the TMA tile
//    once) into TMEM buffer j & 1; once the softmax has replaced S_j by P_j in that
//    buffer, O += P_j V_j with P as the A operand read from TMEM (two BF16 parts
//    hi + lo, two MMAs per 16 keys) and V an MN-major operand straight from the
//    TMA tile.  O accumulates in TMEM over all key tiles.
//  * warps 2-9: two threads per query row (warps w and w + 4 read the same
//    TMEM lane quarter), each with half of the tile's keys and half of the head
//    dims.  One pass over its half row of S (kept in registers), a row-max
//    exchange with its partner, P = exp2(s - m) written back over S in TMEM.
//    The exponent base m only moves when the row max grows by more than 2^8
//    (the running O in TMEM and the row sums are then rescaled once, after the
//    previous P V has finished); otherwise the softmax of tile j + 1 runs while
//    the tensor core does P_j V_j.  The row's O / l is written as BF16.
// Every mbarrier wait is bounded; a timeout sets LL_DEV_TIMEOUT and all roles
// unwind.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace ll {

namespace {

constexpr int kTcThreads = 320;   // TMA warp, MMA warp, 8 softmax warps
constexpr int kKT = 128;          // keys per tile
constexpr int kQT = 128;          // queries per CTA
constexpr int kMaxKeyTiles = 512; // key positions up to 65535 per call
constexpr float kLog2eTc = 1.4426950408889634f;

template <int D>
struct TcLayout {
    static constexpr uint32_t Q_BYTES = kQT * D * 2;        // [D/64][128 rows][128 B]
    static constexpr uint32_t KV_BYTES = kKT * D * 2;       // one K or V tile
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;      // 2 stages
    static constexpr uint32_t OFF_V = OFF_K + 2 * KV_BYTES; // 2 stages
    static constexpr uint32_t TOTAL = OFF_V + 2 * KV_BYTES;
    static constexpr uint32_t TMEM_S0 = 0, TMEM_S1 = 128, TMEM_O = 256;
    static constexpr uint32_t TMEM_Q = 384;   // Q as the A operand of S: D / 2 columns, two BF16 per column
    static constexpr uint32_t TMEM_COLS = 512;
};

// MN-major operand with the 128-byte swizzle (V as the B operand of P V):
// rows of 128 bytes hold 64 consecutive MN elements (head dims), 8 rows (keys)
// form a 1024-byte atom; the next 8 keys are 1024 bytes on (stride byte
// offset), the next 64 head dims are `mn_atom_stride` bytes on (leading byte
// offset).  Version 1, layout type 2 (128-byte swizzle).
LL_DEVINL uint64_t umma_desc_sw128_mn(uint32_t smem_addr, uint32_t mn_atom_stride) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_atom_stride >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= 1ull << 46;
    d |= 2ull << 61;
    return d;
}

// kind::f16 instruction descriptor, BF16 A (K-major) and B (MN-major when
// b_mn), float32 D: bit 16 = B transposed (MN-major).
__host__ __device__ constexpr uint32_t idesc_bf16_bmn(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// byte offset of 16-byte chunk c (8 BF16) of row r in a K-major 128-byte-
// swizzled tile [halves][rows][128 B] whose halves are `half_bytes` apart
LL_DEVINL uint32_t sw128_off(int r, int c, uint32_t half_bytes) {
    return (uint32_t)(c >> 3) * half_bytes + (uint32_t)r * 128u + ((uint32_t)((c & 7) ^ (r & 7)) << 4);
}

struct TcArgs {
    AttnPrefillArgs a;
    int box_rows;       // rows per K/V box = min(block_size, 128)
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const TcArgs args) {
    using L = TcLayout<D>;
    constexpr float kRescaleLog2 = 8.f;   // exponent base moves only when the max grows by > 2^8
    const AttnPrefillArgs& a = args.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    __shared__ uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2];
    __shared__ uint64_t s_full[2], p_full, pv_done[2], drain, q_tmem;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ int max_pos_s;
    __shared__ float red_max[2][2][kQT];      // [tile parity][key half][row]
    __shared__ float red_sum[2][kQT];         // [key half][row], at the end
    __shared__ uint32_t tile_ok_s[kMaxKeyTiles];   // per key tile: bit c = 16-key chunk c has a valid block

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // CTAs are dispatched x-fastest: every head's heaviest (latest) query tile first,
    // then the next heaviest, ... (longest-first keeps the SMs evenly loaded)
    const int b = blockIdx.z, h = blockIdx.x;
    const int mt = gridDim.y - 1 - blockIdx.y;
    const int G = a.n_heads / a.n_kv_heads;
    const int hk = h / G;
    const int row0 = mt * kQT;
    const size_t tok0 = (size_t)b * a.seq_len;
    const int32_t* table_row = a.block_table + (size_t)b * a.max_blocks;
    const int pos_cap = a.max_blocks * a.block_size;
    int32_t* status = a.status;

    if (threadIdx.x == 0) {
        mbar_init(&q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(&p_full, 256);
        mbar_init(&q_tmem, 256);
        mbar_init(&drain, 1);
        abort_s = 0;
        max_pos_s = -1;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_s, L::TMEM_COLS);
        tmem_relinquish();
    }
    pdl_wait();
    pdl_trigger();
    __syncthreads();
    // the tile's last query position (rows beyond the sequence or out of range count as -1)
    if (threadIdx.x < kQT) {
        int p = -1;
        if (row0 + (int)threadIdx.x < a.seq_len) p = a.positions[tok0 + row0 + threadIdx.x];
        if (p >= pos_cap) {
            flag_status(status, LL_DEV_BAD_POSITION);
            p = -1;
        }
        atomicMax(&max_pos_s, p);
    }
    for (int i = threadIdx.x; i < kMaxKeyTiles; i += blockDim.x) tile_ok_s[i] = 0;
    __syncthreads();
    {
        // which 16-key chunks of the tile's key range are backed by a valid block (bs >= 16)
        const int mp = max_pos_s;
        if (threadIdx.x == 0 && mp >= kMaxKeyTiles * kKT) flag_status(status, LL_DEV_BAD_POSITION);
        for (int i = threadIdx.x; i <= mp / 16 && i < kMaxKeyTiles * (kKT / 16); i += blockDim.x) {
            const int blk = table_row[(i * 16) / a.block_size];
            if (blk >= 0 && blk < a.num_blocks) atomicOr(&tile_ok_s[i / (kKT / 16)], 1u << (i % (kKT / 16)));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const int max_pos = max_pos_s;
    const int n_kt = max_pos < 0 ? 0 : min((max_pos + kKT) / kKT, kMaxKeyTiles);

    if (warp == 0) {
        if (lane == 0 && n_kt > 0) {
            // ------------------------------------------------ TMA producer
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            mbar_arrive_expect_tx(&q_full, L::Q_BYTES);
#pragma unroll
            for (int hh = 0; hh < D / 64; ++hh)
                tma_load_2d(smem + L::OFF_Q + hh * (kQT * 128), &tmQ, h * D + hh * 64,
                            (int)(tok0 + row0), &q_full);
            uint32_t issued[2][2] = {{0, 0}, {0, 0}};   // [K/V][stage]
            const int br = args.box_rows;
            // one K or V tile: boxes of br rows per valid block, both column halves
            auto load_tile = [&](int j, int kv) -> bool {
                const int p0 = j * kKT;
                const int st = j & 1;
                uint32_t bytes = 0;
                for (int p = p0; p < p0 + kKT && p <= max_pos; p += br) {
                    const int blk = table_row[p / a.block_size];
                    if (blk >= 0 && blk < a.num_blocks) bytes += (uint32_t)(D / 64) * br * 128u;
                }
                uint64_t* emp = kv ? &v_empty[st] : &k_empty[st];
                uint64_t* ful = kv ? &v_full[st] : &k_full[st];
                if (!mbar_wait_bounded(emp, ((uint32_t)(j >> 1) & 1u) ^ 1u, &abort_s, status)) return false;
                mbar_arrive_expect_tx(ful, bytes);
                uint8_t* dst = smem + (kv ? L::OFF_V : L::OFF_K) + st * L::KV_BYTES;
                for (int p = p0, sb = 0; p < p0 + kKT && p <= max_pos; p += br, ++sb) {
                    const int blk = table_row[p / a.block_size];
                    if (blk < 0 || blk >= a.num_blocks) {
                        if (kv == 0) flag_status(status, LL_DEV_BAD_BLOCK);
                        continue;
                    }
                    const int row = (blk * a.n_kv_heads + hk) * a.block_size + (p % a.block_size);
#pragma unroll
                    for (int hh = 0; hh < D / 64; ++hh)
                        tma_load_2d(dst + hh * (kKT * 128) + sb * br * 128, kv ? &tmV : &tmK, hh * 64,
                                    row, ful);
                }
                ++issued[kv][st];
                return true;
            };
            if (!load_tile(0, 0)) goto producer_done;
            for (int j = 0; j < n_kt; ++j) {
                if (j + 1 < n_kt && !load_tile(j + 1, 0)) goto producer_done;
                if (!load_tile(j, 1)) goto producer_done;
            }
        producer_done:
            if (abort_s) {
                volatile int never = 0;
                mbar_wait_bounded(&q_full, 0, &never, nullptr);
                for (int kv = 0; kv < 2; ++kv)
                    for (int st = 0; st < 2; ++st)
                        if (issued[kv][st])
                            mbar_wait_bounded(kv ? &v_full[st] : &k_full[st], (issued[kv][st] - 1) & 1u,
                                              &never, nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && n_kt > 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t id_s = umma_idesc_bf16(kQT, kKT);
            const uint32_t id_o = idesc_bf16_bmn(kQT, D);
            // Q sits in TMEM once the softmax warps have copied it there (S from an A operand
            // in TMEM: measured on GB300, M128 N128 MMAs with both operands in shared memory
            // take up to twice as long as with A in TMEM)
            bool ok = mbar_wait_bounded(&q_tmem, 0, &abort_s, status);
            tc_fence_after();
            // S_j = Q K_j^T into TMEM buffer j & 1 (after P_{j-2} V_{j-2} has read it)
            auto issue_s = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait_bounded(&k_full[st], (uint32_t)(j >> 1) & 1u, &abort_s, status)) return false;
                if (j >= 2 && !mbar_wait_bounded(&pv_done[st], (uint32_t)((j - 2) >> 1) & 1u, &abort_s, status))
                    return false;
                tc_fence_after();
                const uint32_t sk = smem_u32(smem + L::OFF_K + st * L::KV_BYTES);
                const uint32_t d_s = tmem + (st ? L::TMEM_S1 : L::TMEM_S0);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t offk = (uint32_t)(kk >> 2) * (kKT * 128) + (uint32_t)(kk & 3) * 32;
                    tc_mma_bf16_ts(d_s, tmem + L::TMEM_Q + (uint32_t)kk * 8u, umma_desc_sw128(sk + offk), id_s,
                                   kk > 0 ? 1u : 0u);
                }
                tc_commit(&s_full[st]);
                tc_commit(&k_empty[st]);
                return true;
            };
            // O += (P_hi + P_lo) V_j, P read from TMEM buffer j & 1
            auto issue_pv = [&](int j) -> bool {
                const int st = j & 1;
                if (!mbar_wait_bounded(&p_full, (uint32_t)j & 1u, &abort_s, status)) return false;
                if (!mbar_wait_bounded(&v_full[st], (uint32_t)(j >> 1) & 1u, &abort_s, status)) return false;
                tc_fence_after();
                const uint32_t sv = smem_u32(smem + L::OFF_V + st * L::KV_BYTES);
                const uint32_t pbuf = tmem + (st ? L::TMEM_S1 : L::TMEM_S0);
                const uint32_t d_o = tmem + L::TMEM_O;
#pragma unroll
                for (int kk = 0; kk < kKT / 16; ++kk) {
                    const uint64_t bv = umma_desc_sw128_mn(sv + (uint32_t)kk * 2048u, kKT * 128);
                    tc_mma_bf16_ts(d_o, pbuf + (uint32_t)kk * 8u, bv, id_o, (j > 0 || kk > 0) ? 1u : 0u);
                    tc_mma_bf16_ts(d_o, pbuf + 64u + (uint32_t)kk * 8u, bv, id_o, 1u);
                }
                tc_commit(&pv_done[st]);
                tc_commit(&v_empty[st]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < n_kt && ok; ++j) {
                if (j + 1 < n_kt) ok = issue_s(j + 1);
                if (ok) ok = issue_pv(j);
            }
            tc_commit(&drain);
            volatile int never = 0;
            mbar_wait_bounded(&drain, 0, &never, status);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------- softmax warps
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;             // 0: keys 0-63, dims 0..D/2-1; 1: the rest
        const int r = q4 * 32 + lane;                 // query row of the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        constexpr int HK = kKT / 2;                   // keys per half
        constexpr int HD = D / 2;                     // head dims per half
        int my_pos = -1;
        if (row0 + r < a.seq_len) my_pos = a.positions[tok0 + row0 + r];
        if (my_pos >= pos_cap) my_pos = -1;
        const float sl2 = a.scale * kLog2eTc;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        if (n_kt > 0) {
            // this thread's half of Q row r into TMEM (column c holds elements 2c, 2c + 1),
            // read from the 128-byte-swizzled TMA tile [D / 64][128 rows][128 B]
            const bool got_q = __all_sync(0xffffffffu, mbar_wait_bounded(&q_full, 0, &abort_s, status));
#pragma unroll
            for (int g = 0; g < HD / 32; ++g) {       // 32 elements (16 columns) at a time
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int e = half * HD + g * 32 + c * 8;   // first element of the 16-byte chunk
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (got_q)
                        x = *reinterpret_cast<const uint4*>(smem + L::OFF_Q + (e >> 6) * (kQT * 128) + r * 128 +
                                                            ((((e & 63) >> 3) ^ (r & 7)) << 4));
                    w[4 * c] = x.x;
                    w[4 * c + 1] = x.y;
                    w[4 * c + 2] = x.z;
                    w[4 * c + 3] = x.w;
                }
                tmem_st16(tmem + lane_base + L::TMEM_Q + (uint32_t)(half * HD / 2 + g * 16), w);
            }
            tc_fence_before();
            mbar_arrive(&q_tmem);
        }
        for (int j = 0; j < n_kt && ok; ++j) {
            const int st = j & 1;
            const uint32_t ph = (uint32_t)(j >> 1) & 1u;
            // A failed (timed-out) wait never skips the named barrier below: every softmax
            // thread reaches it each tile, and all leave the loop together after it.
            const bool got_s = __all_sync(0xffffffffu, mbar_wait_bounded(&s_full[st], ph, &abort_s, status));
            tc_fence_after();
            const uint32_t tbuf = tmem + lane_base + (st ? L::TMEM_S1 : L::TMEM_S0);
            const int kbase = j * kKT + half * HK;    // first key of this thread's half
            const uint32_t tile_ok = tile_ok_s[j];
            const uint32_t chunk_ok = (tile_ok >> (half * (HK / 16))) & ((1u << (HK / 16)) - 1u);
            // V rows of this tile that hold no key (past the tile's last position, or in an
            // invalid block) may be stale or uninitialised: zero them so 0 * V stays 0.  Thread
            // (row r, half) owns V row r's half of the head dims.
            {
                const int jb = j * kKT;
                const bool need = jb + kKT - 1 > max_pos || tile_ok != (1u << (kKT / 16)) - 1u;
                if (need && mbar_wait_bounded(&v_full[st], ph, &abort_s, status)) {
                    const int kr = jb + r;
                    const bool row_ok = kr <= max_pos && ((tile_ok >> (r >> 4)) & 1u);
                    if (!row_ok) {
                        uint8_t* vrow = smem + L::OFF_V + st * L::KV_BYTES;
#pragma unroll
                        for (int c = half * (HD / 8); c < (half + 1) * (HD / 8); ++c)
                            *reinterpret_cast<uint4*>(vrow + sw128_off(r, c, kKT * 128)) = make_uint4(0, 0, 0, 0);
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    }
                }
            }
            // one pass over the half row of S: raw scores in registers, masked (-inf) only
            // where this half touches the diagonal or an invalid block
            const bool full = chunk_ok == (1u << (HK / 16)) - 1u && kbase + HK - 1 <= my_pos;
            static_assert(HK == 64, "one 64-column TMEM load per half row");
            float sv[HK];
            if (got_s) {
                tmem_ld64(tbuf + (uint32_t)(half * HK), sv);   // the half row, one wait
            } else {
#pragma unroll
                for (int i = 0; i < HK; ++i) sv[i] = 0.f;
            }
            if (!full) {
#pragma unroll
                for (int i = 0; i < HK; ++i)
                    if (!(((chunk_ok >> (i >> 4)) & 1u) && kbase + i <= my_pos)) sv[i] = -INFINITY;
            }
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < HK; ++i) mx = fmaxf(mx, sv[i]);
            red_max[j & 1][half][r] = mx;
            asm volatile("bar.sync 2, 256;" ::: "memory");   // both halves have read S_j
            if (abort_s) { ok = false; break; }
            mx = fmaxf(mx, red_max[j & 1][half ^ 1][r]) * sl2;  // scale > 0: max commutes
            const float m_new = fmaxf(m_used, mx);
            const bool move = m_new > m_used + kRescaleLog2;  // false while the row has no key
            if (__any_sync(0xffffffffu, move)) {
                if (j > 0) {
                    // rescale the running O (this half's dims) once P_{j-1} V_{j-1} is in it
                    const bool got_pv = __all_sync(0xffffffffu,
                        mbar_wait_bounded(&pv_done[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, &abort_s, status));
                    tc_fence_after();
                    const float f = move ? exp2f(m_used - m_new) : 1.f;
                    const uint32_t to = tmem + lane_base + L::TMEM_O + (uint32_t)(half * HD);
#pragma unroll
                    for (int c = 0; c < HD && got_pv; c += 16) {
                        float v[16];
                        uint32_t w[16];
                        tmem_ld16(to + (uint32_t)c, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(v[i] * f);
                        tmem_st16(to + (uint32_t)c, w);
                    }
                }
                if (move) {
                    l *= exp2f(m_used - m_new);
                    m_used = m_new;
                }
            }
            const float base = (m_used == -INFINITY) ? 0.f : m_used;
            // P = exp2(s - base) as hi + lo BF16 parts, written over S in TMEM:
            // hi in columns [0, 64) and lo in [64, 128) of the buffer, two keys per column
            float rs = 0.f;
            {
                uint32_t hi[HK / 2], lo[HK / 2];
#pragma unroll
                for (int i = 0; i < HK / 2; ++i) {
                    const float p0 = ex2_approx(fmaf(sv[2 * i], sl2, -base));
                    const float p1 = ex2_approx(fmaf(sv[2 * i + 1], sl2, -base));
                    rs += p0 + p1;
                    split_bf16x2(p0, p1, hi[i], lo[i]);
                }
                // the half row's 32 hi and 32 lo columns, one wait
                const uint32_t col = (uint32_t)((half * HK) >> 1);
                tmem_st32x2(tbuf + col, hi, tbuf + 64u + col, lo);
            }
            l += rs;
            tc_fence_before();
            mbar_arrive(&p_full);
        }
        // row sum = both halves' sums (same exponent base)
        red_sum[half][r] = l;
        asm volatile("bar.sync 2, 256;" ::: "memory");
        l += red_sum[half ^ 1][r];
        if (ok && n_kt > 0)
            ok = mbar_wait_bounded(&pv_done[(n_kt - 1) & 1], (uint32_t)((n_kt - 1) >> 1) & 1u, &abort_s, status);
        ok = __all_sync(0xffffffffu, ok);   // the TMEM reads below are warp-collective
        // TMEM reads are warp-collective: every lane loads, only rows of the sequence store
        const bool row_valid = row0 + r < a.seq_len;
        if (ok || n_kt == 0) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(a.out + ((tok0 + row0 + r) * a.n_heads + h) * D + half * HD);
            const uint32_t to = tmem + lane_base + L::TMEM_O + (uint32_t)(half * HD);
#pragma unroll
            for (int c = 0; c < HD; c += 16) {
                float v[16];
                if (n_kt > 0) {
                    tmem_ld16(to + (uint32_t)c, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                }
                if (row_valid) {
#pragma unroll
                    for (int i = 0; i < 16; i += 8) {
                        uint4 o;
                        o.x = pack_bf16x2(v[i] * inv, v[i + 1] * inv);
                        o.y = pack_bf16x2(v[i + 2] * inv, v[i + 3] * inv);
                        o.z = pack_bf16x2(v[i + 4] * inv, v[i + 5] * inv);
                        o.w = pack_bf16x2(v[i + 6] * inv, v[i + 7] * inv);
                        dst[(c + i) >> 3] = o;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

template <int D>
cudaError_t prefill_tc_for(const AttnPrefillArgs& a, cudaStream_t stream) {
    using L = TcLayout<D>;
    const size_t smem = L::TOTAL + 1024;
    {
        const cudaError_t e = ensure_func_attr((const void*)attn_prefill_tc_kernel<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem,
                                               "cudaFuncSetAttribute(attn_prefill_tc_kernel)");
        if (e != cudaSuccess) return e;
    }
    TcArgs args{a, std::min(a.block_size, kKT)};
    CUtensorMap tmQ, tmK, tmV;
    const uint64_t tokens = (uint64_t)a.batch * a.seq_len;
    const uint64_t rows = (uint64_t)a.num_blocks * a.n_kv_heads * a.block_size;
    if (!make_tmap_bf16_sw128(&tmQ, a.q, (uint64_t)a.n_heads * D, tokens, kQT) ||
        !make_tmap_bf16_sw128(&tmK, a.k_pool, D, rows, (uint32_t)args.box_rows) ||
        !make_tmap_bf16_sw128(&tmV, a.v_pool, D, rows, (uint32_t)args.box_rows))
        return cudaErrorInvalidValue;
    dim3 grid(a.n_heads, (a.seq_len + kQT - 1) / kQT, a.batch);
    trace_before("attn_prefill", stream);
    cudaError_t e = launch_pdl(attn_prefill_tc_kernel<D>, grid, dim3(kTcThreads), smem, stream, 1, tmQ, tmK,
                               tmV, args);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "attn_prefill_tc_kernel launch");
    return record(cudaGetLastError(), "attn_prefill_tc_kernel launch");
}

}  // namespace

cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t stream) {
    if (a.batch <= 0 || a.seq_len <= 0) return cudaSuccess;
    if (a.head_dim == 128) return prefill_tc_for<128>(a, stream);
    if (a.head_dim == 64) return prefill_tc_for<64>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace ll
