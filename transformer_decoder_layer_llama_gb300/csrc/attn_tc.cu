// Prefill flash attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA):
// the FlashAttention operator of the Llama2-7B operator chain (page "Which
// ops-transformer operators one Llama2-7B layer calls", sections "single-layer
// operator call chain" and "KV Cache and the operators": MatMul -> Softmax ->
// MatMul fused, the whole sequence in one kernel).
//
// Work item = 128 queries of one sequence and one query head (GQA: KV head
// h / (Hq / Hkv)).  Keys come from the paged pool through block_table, 128 at
// a time, in causal order up to the tile's last query position.  The kernel is
// persistent: one CTA per SM takes a fixed list of items (see tc_item) and runs
// them back to back, so that the next item's metadata, Q and first K/V tiles
// load, and its first S is computed, while the current item's output is being
// written.  Measured on GB300 with one CTA per item: ~3 us from a CTA's start to
// its first S and ~2 us of tail per item, 3.4 items per SM on the 7B prefill;
// persistent, 2.8 us from an item's last P to the next item's first S, and the
// 7B prefill attention 70.0 -> 65.7 us.
//
// Warp roles (352 threads):
//  * warp 10: per item, up to two items ahead, the tile's last query position
//    and which 16-key chunks are backed by a valid block (metadata slot k & 1).
//  * warp 0, one lane: TMA.  Per item Q (two 64-column boxes), then per key
//    tile K and V as boxes of min(block_size, 128) rows x 64 columns at the
//    physical block's rows, each double-buffered, K loaded one tile ahead of V.
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
//    the tensor core does P_j V_j.  After an item's last tile they copy the
//    next item's Q into TMEM, load the row's O from TMEM and release it to the
//    next item's first P V, then write O / l as BF16.
// Every mbarrier wait is bounded; a timeout sets LL_DEV_TIMEOUT and all roles
// unwind.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace ll {

namespace {

constexpr int kTcThreads = 352;   // TMA warp, MMA warp, 8 softmax warps, metadata warp
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
    int n_mt;           // 128-query tiles per sequence
    int n_items;        // batch * n_mt * n_heads work items
};

// Work items are (sequence, query head, 128-query tile).  Item order: the latest query
// tiles (the most key tiles under the causal mask) first, query heads fastest, so that
// the query heads of one KV head run side by side.  CTA c of P takes items c, 2P-1-c,
// 2P+c, 4P-1-c, ... (rounds of P items, every other round reversed), which pairs heavy
// with light items; -1 past the end (a CTA's items are a prefix of its rounds).
LL_DEVINL int tc_item(int cta, int P, int k, int n_items) {
    const int idx = k * P + ((k & 1) ? P - 1 - cta : cta);
    return idx < n_items ? idx : -1;
}

struct TcItem {
    int b, h, row0;
};

LL_DEVINL TcItem tc_item_coords(const TcArgs& t, int idx) {
    const int bh = t.a.batch * t.a.n_heads;
    const int rank = idx / bh, rem = idx - rank * bh;
    TcItem it;
    it.b = rem / t.a.n_heads;
    it.h = rem - it.b * t.a.n_heads;
    it.row0 = (t.n_mt - 1 - rank) * kQT;
    return it;
}

// Named barrier 2 over the 256 softmax threads, with an OR of `pred` returned to every
// thread: all of them take the same branch after it (a plain barrier followed by a
// read of a flag that another role may set in between would not guarantee that).
LL_DEVINL bool softmax_bar_any(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n"
        " barrier.cta.red.or.pred q, 2, 256, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

// Bounded wait for a warp that runs ahead of the barrier's producers by a whole work
// item: it sleeps between polls instead of taking issue slots from the warps doing
// the work on its SM sub-partition.
LL_DEVINL bool mbar_wait_idle(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(500);
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            flag_status(status, LL_DEV_TIMEOUT);
            return false;
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const TcArgs args) {
    using L = TcLayout<D>;
    constexpr float kRescaleLog2 = 8.f;   // exponent base moves only when the max grows by > 2^8
    constexpr int kChunks = kKT / 16;     // 16-key chunks per key tile
    const AttnPrefillArgs& a = args.a;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    // per item (phase = the CTA's item count k & 1, or (k >> 1) & 1 for the two-slot pairs)
    __shared__ uint64_t meta_full[2], meta_empty[2], q_full, q_empty, q_tmem, qt_free, o_free;
    // per key tile, counted over all of the CTA's items
    // (P_j is signalled per S buffer: with one barrier for all tiles the softmax warps,
    // which may finish tiles j and j + 1 before the MMA thread looks for tile j's
    // completion (S_{j+1} is issued before P_j V_j), would make that phase parity alias)
    __shared__ uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], p_full[2], pv_done[2];
    __shared__ uint64_t drain;
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ int meta_pos_s[2];                   // per item slot: the tile's last query position
    __shared__ int pos_s[2][kQT];                   // per slot and row: its position (-1: none)
    __shared__ uint32_t tile_ok_s[2][kMaxKeyTiles]; // per slot and key tile: bit c = 16-key chunk c valid
    __shared__ float red_max[2][2][kQT];            // [tile parity][key half][row]
    __shared__ float red_sum[2][2][kQT];            // [item parity][key half][row]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int P = (int)gridDim.x, cta = (int)blockIdx.x;
    const int G = a.n_heads / a.n_kv_heads;
    const int pos_cap = a.max_blocks * a.block_size;
    int32_t* status = a.status;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&meta_full[i], 32);
            mbar_init(&meta_empty[i], 8);
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 256);
            mbar_init(&pv_done[i], 1);
        }
        mbar_init(&q_full, 1);
        mbar_init(&q_empty, 8);
        mbar_init(&q_tmem, 256);
        mbar_init(&qt_free, 1);
        mbar_init(&o_free, 256);
        mbar_init(&drain, 1);
        abort_s = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_s, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    pdl_wait();
    pdl_trigger();

    if (warp == 10) {
        // ---------------------------------------------------- metadata warp
        // Per item, up to two items ahead of the softmax warps (slot k & 1): the tile's
        // last query position and which 16-key chunks of its key tiles are backed by a
        // valid block.
        for (int k = 0;; ++k) {
            const int idx = tc_item(cta, P, k, args.n_items);
            if (idx < 0) break;
            const TcItem it = tc_item_coords(args, idx);
            const int slot = k & 1;
            const size_t tok0 = (size_t)it.b * a.seq_len;
            const int32_t* table_row = a.block_table + (size_t)it.b * a.max_blocks;
            if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait_idle(&meta_empty[slot], (uint32_t)((k - 2) >> 1) & 1u,
                                                                   &abort_s, status)))
                break;
            int mp = -1;   // rows beyond the sequence or out of range count as -1
            for (int i = lane; i < kQT; i += 32) {
                int p = -1;
                if (it.row0 + i < a.seq_len) {
                    p = a.positions[tok0 + it.row0 + i];
                    if (p >= pos_cap) {
                        flag_status(status, LL_DEV_BAD_POSITION);
                        p = -1;
                    }
                }
                pos_s[slot][i] = p;
                mp = max(mp, p);
            }
            mp = __reduce_max_sync(0xffffffffu, mp);
            if (lane == 0 && mp >= kMaxKeyTiles * kKT) flag_status(status, LL_DEV_BAD_POSITION);
            const int n_kt = mp < 0 ? 0 : min((mp + kKT) / kKT, kMaxKeyTiles);
            for (int c0 = 0; c0 < n_kt * kChunks; c0 += 32) {   // 32 chunks = 32 / kChunks tiles
                const int ci = c0 + lane;
                bool valid = false;
                if (ci < n_kt * kChunks && ci * 16 <= mp) {
                    const int blk = table_row[(ci * 16) / a.block_size];
                    valid = blk >= 0 && blk < a.num_blocks;
                }
                const uint32_t m = __ballot_sync(0xffffffffu, valid);
                if (lane < 32 / kChunks && c0 / kChunks + lane < n_kt)
                    tile_ok_s[slot][c0 / kChunks + lane] = (m >> (lane * kChunks)) & ((1u << kChunks) - 1u);
            }
            if (lane == 0) meta_pos_s[slot] = mp;
            __syncwarp();
            mbar_arrive(&meta_full[slot]);          // every lane releases its own writes
        }
        __syncwarp();
    } else if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            // Per item: Q (as soon as the softmax warps have copied the previous one out),
            // then, once the item's metadata is in, K one tile ahead of V.
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t issued[2][2] = {{0, 0}, {0, 0}};   // [K/V][stage] loads issued
            uint32_t q_issued = 0;
            int g = 0;                                  // the CTA's key tiles so far
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int idx = tc_item(cta, P, k, args.n_items);
                if (idx < 0) break;
                const TcItem it = tc_item_coords(args, idx);
                const size_t tok0 = (size_t)it.b * a.seq_len;
                const int32_t* table_row = a.block_table + (size_t)it.b * a.max_blocks;
                const int hk = it.h / G;
                if (k >= 1 && !mbar_wait_bounded(&q_empty, (uint32_t)(k - 1) & 1u, &abort_s, status)) break;
                mbar_arrive_expect_tx(&q_full, L::Q_BYTES);
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh)
                    tma_load_2d(smem + L::OFF_Q + hh * (kQT * 128), &tmQ, it.h * D + hh * 64,
                                (int)(tok0 + it.row0), &q_full);
                ++q_issued;
                if (!mbar_wait_bounded(&meta_full[k & 1], (uint32_t)(k >> 1) & 1u, &abort_s, status)) break;
                const int mp = meta_pos_s[k & 1];
                const int n_kt = mp < 0 ? 0 : min((mp + kKT) / kKT, kMaxKeyTiles);
                const int br = args.box_rows;
                // key tile j of this item (the CTA's tile g + j): boxes of br rows per valid
                // block, both column halves
                auto load_tile = [&](int j, int kv) -> bool {
                    const int gg = g + j;
                    const int p0 = j * kKT;
                    const int st = gg & 1;
                    uint32_t bytes = 0;
                    for (int p = p0; p < p0 + kKT && p <= mp; p += br) {
                        const int blk = table_row[p / a.block_size];
                        if (blk >= 0 && blk < a.num_blocks) bytes += (uint32_t)(D / 64) * br * 128u;
                    }
                    uint64_t* emp = kv ? &v_empty[st] : &k_empty[st];
                    uint64_t* ful = kv ? &v_full[st] : &k_full[st];
                    if (!mbar_wait_bounded(emp, ((uint32_t)(gg >> 1) & 1u) ^ 1u, &abort_s, status)) return false;
                    mbar_arrive_expect_tx(ful, bytes);
                    uint8_t* dst = smem + (kv ? L::OFF_V : L::OFF_K) + st * L::KV_BYTES;
                    for (int p = p0, sb = 0; p < p0 + kKT && p <= mp; p += br, ++sb) {
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
                if (n_kt > 0) {
                    ok = load_tile(0, 0);
                    for (int j = 0; j < n_kt && ok; ++j) {
                        if (j + 1 < n_kt) ok = load_tile(j + 1, 0);
                        if (ok) ok = load_tile(j, 1);
                    }
                }
                g += n_kt;
            }
            if (abort_s) {
                // wait (bounded) for the copies in flight before the CTA leaves
                volatile int never = 0;
                if (q_issued) mbar_wait_bounded(&q_full, (q_issued - 1) & 1u, &never, nullptr);
                for (int kv = 0; kv < 2; ++kv)
                    for (int st = 0; st < 2; ++st)
                        if (issued[kv][st])
                            mbar_wait_bounded(kv ? &v_full[st] : &k_full[st], (issued[kv][st] - 1) & 1u, &never,
                                              nullptr);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            const uint32_t id_s = umma_idesc_bf16(kQT, kKT);
            const uint32_t id_o = idesc_bf16_bmn(kQT, D);
            int g = 0;
            bool ok = true;
            for (int k = 0; ok; ++k) {
                const int idx = tc_item(cta, P, k, args.n_items);
                if (idx < 0) break;
                if (!mbar_wait_bounded(&meta_full[k & 1], (uint32_t)(k >> 1) & 1u, &abort_s, status)) break;
                const int mp = meta_pos_s[k & 1];
                const int n_kt = mp < 0 ? 0 : min((mp + kKT) / kKT, kMaxKeyTiles);
                // Q sits in TMEM once the softmax warps have copied it there (S from an A
                // operand in TMEM: measured on GB300, M128 N128 MMAs with both operands in
                // shared memory take up to twice as long as with A in TMEM)
                if (!mbar_wait_bounded(&q_tmem, (uint32_t)k & 1u, &abort_s, status)) break;
                tc_fence_after();
                // S = Q K^T for the item's key tile j into TMEM buffer (g + j) & 1, after the
                // P V two tiles back has read that buffer
                auto issue_s = [&](int j) -> bool {
                    const int gg = g + j;
                    const int st = gg & 1;
                    if (!mbar_wait_bounded(&k_full[st], (uint32_t)(gg >> 1) & 1u, &abort_s, status)) return false;
                    if (gg >= 2 &&
                        !mbar_wait_bounded(&pv_done[st], (uint32_t)((gg - 2) >> 1) & 1u, &abort_s, status))
                        return false;
                    tc_fence_after();
                    const uint32_t sk = smem_u32(smem + L::OFF_K + st * L::KV_BYTES);
                    const uint32_t d_s = tmem + (st ? L::TMEM_S1 : L::TMEM_S0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t offk = (uint32_t)(kk >> 2) * (kKT * 128) + (uint32_t)(kk & 3) * 32;
                        tc_mma_bf16_ts(d_s, tmem + L::TMEM_Q + (uint32_t)kk * 8u, umma_desc_sw128(sk + offk),
                                       id_s, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(&s_full[st]);
                    tc_commit(&k_empty[st]);
                    return true;
                };
                // O += (P_hi + P_lo) V for key tile j, P read from TMEM buffer (g + j) & 1; the
                // item's first product overwrites O once the previous item's output is out
                auto issue_pv = [&](int j) -> bool {
                    const int gg = g + j;
                    const int st = gg & 1;
                    if (!mbar_wait_bounded(&p_full[st], (uint32_t)(gg >> 1) & 1u, &abort_s, status)) return false;
                    if (!mbar_wait_bounded(&v_full[st], (uint32_t)(gg >> 1) & 1u, &abort_s, status)) return false;
                    if (j == 0 && k >= 1 &&
                        !mbar_wait_bounded(&o_free, (uint32_t)(k - 1) & 1u, &abort_s, status))
                        return false;
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
                // qt_free: the item's last S has read Q from TMEM (one commit per item)
                if (n_kt > 0) ok = issue_s(0);
                if (n_kt <= 1) tc_commit(&qt_free);
                for (int j = 0; j < n_kt && ok; ++j) {
                    if (j + 1 < n_kt) {
                        ok = issue_s(j + 1);
                        if (j + 2 == n_kt) tc_commit(&qt_free);
                    }
                    if (ok) ok = issue_pv(j);
                }
                g += n_kt;
            }
            tc_commit(&drain);
            volatile int never = 0;
            mbar_wait_bounded(&drain, 0, &never, status);
        }
        __syncwarp();
    } else if (warp >= 2) {
        // ---------------------------------------------------- softmax warps (2-9)
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;             // 0: keys 0-63, dims 0..D/2-1; 1: the rest
        const int r = q4 * 32 + lane;                 // query row of the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        constexpr int HK = kKT / 2;                   // keys per half
        constexpr int HD = D / 2;                     // head dims per half
        const float sl2 = a.scale * kLog2eTc;
        // This thread's half of Q row r of item kq into TMEM (column c holds elements 2c,
        // 2c + 1), read from the 128-byte-swizzled TMA tile [D / 64][128 rows][128 B],
        // once the previous item's last S has read the TMEM copy before it.
        auto copy_q = [&](int kq) {
            const bool got_q =
                __all_sync(0xffffffffu, mbar_wait_bounded(&q_full, (uint32_t)kq & 1u, &abort_s, status));
            if (kq >= 1)
                __all_sync(0xffffffffu, mbar_wait_bounded(&qt_free, (uint32_t)(kq - 1) & 1u, &abort_s, status));
            tc_fence_after();
#pragma unroll
            for (int g2 = 0; g2 < HD / 32; ++g2) {    // 32 elements (16 columns) at a time
                uint32_t w[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int e = half * HD + g2 * 32 + c * 8;   // first element of the 16-byte chunk
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (got_q)
                        x = *reinterpret_cast<const uint4*>(smem + L::OFF_Q + (e >> 6) * (kQT * 128) + r * 128 +
                                                            ((((e & 63) >> 3) ^ (r & 7)) << 4));
                    w[4 * c] = x.x;
                    w[4 * c + 1] = x.y;
                    w[4 * c + 2] = x.z;
                    w[4 * c + 3] = x.w;
                }
                tmem_st16(tmem + lane_base + L::TMEM_Q + (uint32_t)(half * HD / 2 + g2 * 16), w);
            }
            tc_fence_before();
            mbar_arrive(&q_tmem);
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty);     // this warp is done with the Q tile
        };
        int g = 0;
        if (tc_item(cta, P, 0, args.n_items) >= 0) copy_q(0);
        // Item pe_k's output, once its last P V (tile pe_glast) is done: row sum pe_l of this
        // half, row pe_row valid, written at pe_dst.  Returns true when all softmax threads
        // stop (a wait ran out somewhere).
        int pe_k = 0, pe_n = 0, pe_glast = 0;
        float pe_l = 0.f;
        bool pe_row = false;
        __nv_bfloat16* pe_dst = nullptr;
        auto epilogue = [&]() -> bool {
            red_sum[pe_k & 1][half][r] = pe_l;   // row sum = both halves' sums (same base)
            if (softmax_bar_any(abort_s != 0)) return true;
            const float lt = pe_l + red_sum[pe_k & 1][half ^ 1][r];
            bool ok = true;
            if (pe_n > 0)
                ok = mbar_wait_bounded(&pv_done[pe_glast & 1], (uint32_t)(pe_glast >> 1) & 1u, &abort_s, status);
            ok = __all_sync(0xffffffffu, ok);   // the TMEM reads below are warp-collective
            // this thread's half row of O into registers; O is then released to the next
            // item's first P V before the stores
            float ov[HD];
#pragma unroll
            for (int i = 0; i < HD; ++i) ov[i] = 0.f;
            if (ok && pe_n > 0) {
                tc_fence_after();
                const uint32_t to = tmem + lane_base + L::TMEM_O + (uint32_t)(half * HD);
                if constexpr (HD == 64) {
                    tmem_ld64(to, ov);
                } else {
#pragma unroll
                    for (int c = 0; c < HD; c += 16) {
                        float v[16];
                        tmem_ld16(to + (uint32_t)c, v);
#pragma unroll
                        for (int i = 0; i < 16; ++i) ov[c + i] = v[i];
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&o_free);
            if (ok && pe_row) {
                const float inv = lt > 0.f ? 1.f / lt : 0.f;
                uint4* dst = reinterpret_cast<uint4*>(pe_dst);
#pragma unroll
                for (int i = 0; i < HD; i += 8) {
                    uint4 o;
                    o.x = pack_bf16x2(ov[i] * inv, ov[i + 1] * inv);
                    o.y = pack_bf16x2(ov[i + 2] * inv, ov[i + 3] * inv);
                    o.z = pack_bf16x2(ov[i + 4] * inv, ov[i + 5] * inv);
                    o.w = pack_bf16x2(ov[i + 6] * inv, ov[i + 7] * inv);
                    dst[i >> 3] = o;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&meta_empty[pe_k & 1]);
            return false;
        };
        // Every exit from the item and tile loops follows softmax_bar_any, whose result
        // is the same in all 256 threads: the named barriers stay matched.
        bool stop = false;
        for (int k = 0; !stop; ++k) {
            const int idx = tc_item(cta, P, k, args.n_items);
            if (idx < 0) break;
            const TcItem it = tc_item_coords(args, idx);
            const int slot = k & 1;
            const size_t tok0 = (size_t)it.b * a.seq_len;
            const bool has_next = tc_item(cta, P, k + 1, args.n_items) >= 0;
            const bool got_meta = __all_sync(
                0xffffffffu, mbar_wait_bounded(&meta_full[slot], (uint32_t)(k >> 1) & 1u, &abort_s, status));
            if (softmax_bar_any(!got_meta || abort_s != 0)) break;
            const int max_pos = meta_pos_s[slot];
            const int n_kt = max_pos < 0 ? 0 : min((max_pos + kKT) / kKT, kMaxKeyTiles);
            const int my_pos = pos_s[slot][r];
            float m_used = -INFINITY, l = 0.f;
            for (int j = 0; j < n_kt; ++j) {
                const int gg = g + j;
                const int st = gg & 1;
                const uint32_t ph = (uint32_t)(gg >> 1) & 1u;
                const bool got_s = __all_sync(0xffffffffu, mbar_wait_bounded(&s_full[st], ph, &abort_s, status));
                tc_fence_after();
                const uint32_t tbuf = tmem + lane_base + (st ? L::TMEM_S1 : L::TMEM_S0);
                const int kbase = j * kKT + half * HK;    // first key of this thread's half
                const uint32_t tile_ok = tile_ok_s[slot][j];
                const uint32_t chunk_ok = (tile_ok >> (half * (HK / 16))) & ((1u << (HK / 16)) - 1u);
                // V rows of this tile that hold no key (past the tile's last position, or in an
                // invalid block) may be stale or uninitialised: zero them so 0 * V stays 0.
                // Thread (row r, half) owns V row r's half of the head dims.
                {
                    const int jb = j * kKT;
                    const bool need = jb + kKT - 1 > max_pos || tile_ok != (1u << kChunks) - 1u;
                    if (need && mbar_wait_bounded(&v_full[st], ph, &abort_s, status)) {
                        const int kr = jb + r;
                        const bool row_ok = kr <= max_pos && ((tile_ok >> (r >> 4)) & 1u);
                        if (!row_ok) {
                            uint8_t* vrow = smem + L::OFF_V + st * L::KV_BYTES;
#pragma unroll
                            for (int c = half * (HD / 8); c < (half + 1) * (HD / 8); ++c)
                                *reinterpret_cast<uint4*>(vrow + sw128_off(r, c, kKT * 128)) =
                                    make_uint4(0, 0, 0, 0);
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
                red_max[st][half][r] = mx;
                if (softmax_bar_any(abort_s != 0)) {   // both halves have read S
                    stop = true;
                    break;
                }
                mx = fmaxf(mx, red_max[st][half ^ 1][r]) * sl2;  // scale > 0: max commutes
                const float m_new = fmaxf(m_used, mx);
                const bool move = m_new > m_used + kRescaleLog2;  // false while the row has no key
                if (__any_sync(0xffffffffu, move)) {
                    if (j > 0) {
                        // rescale the running O (this half's dims) once the previous P V is in it
                        const bool got_pv = __all_sync(
                            0xffffffffu, mbar_wait_bounded(&pv_done[(gg - 1) & 1], (uint32_t)((gg - 1) >> 1) & 1u,
                                                           &abort_s, status));
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
                mbar_arrive(&p_full[st]);
            }
            if (stop) break;
            // the next item's Q now, so that its first S runs while this item's output is written
            if (has_next) copy_q(k + 1);
            pe_k = k;
            pe_n = n_kt;
            pe_glast = g + n_kt - 1;
            pe_l = l;
            pe_row = it.row0 + r < a.seq_len;
            pe_dst = a.out + ((tok0 + it.row0 + r) * a.n_heads + it.h) * D + half * HD;
            g += n_kt;
            if (epilogue()) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

std::atomic<int> g_prefill_ctas_cap{0};   // 0: one CTA per SM

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
    const int n_mt = (a.seq_len + kQT - 1) / kQT;
    const long long n_items = (long long)a.batch * n_mt * a.n_heads;
    if (n_items > (1LL << 30)) {
        set_last_error("attn_prefill", "too many (sequence, head, query tile) items");
        return cudaErrorInvalidValue;
    }
    const int sms = device_sm_count();
    if (sms <= 0) return record(cudaErrorNoDevice, "attn_prefill");
    TcArgs args{a, std::min(a.block_size, kKT), n_mt, (int)n_items};
    CUtensorMap tmQ, tmK, tmV;
    const uint64_t tokens = (uint64_t)a.batch * a.seq_len;
    const uint64_t rows = (uint64_t)a.num_blocks * a.n_kv_heads * a.block_size;
    if (!make_tmap_bf16_sw128(&tmQ, a.q, (uint64_t)a.n_heads * D, tokens, kQT) ||
        !make_tmap_bf16_sw128(&tmK, a.k_pool, D, rows, (uint32_t)args.box_rows) ||
        !make_tmap_bf16_sw128(&tmV, a.v_pool, D, rows, (uint32_t)args.box_rows))
        return cudaErrorInvalidValue;
    // persistent: one CTA per SM (160 KB of shared memory and all of TMEM each), or fewer
    const int cap = g_prefill_ctas_cap.load(std::memory_order_relaxed);
    const int ctas = (int)std::min<long long>(n_items, cap > 0 ? std::min(cap, sms) : sms);
    trace_before("attn_prefill", stream);
    cudaError_t e = launch_pdl(attn_prefill_tc_kernel<D>, dim3((unsigned)ctas), dim3(kTcThreads), smem, stream, 1,
                               tmQ, tmK, tmV, args);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "attn_prefill_tc_kernel launch");
    return record(cudaGetLastError(), "attn_prefill_tc_kernel launch");
}

}  // namespace

void set_prefill_attention_ctas(int n) { g_prefill_ctas_cap.store(n > 0 ? n : 0, std::memory_order_relaxed); }

cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t stream) {
    if (a.batch <= 0 || a.seq_len <= 0) return cudaSuccess;
    if (a.head_dim == 128) return prefill_tc_for<128>(a, stream);
    if (a.head_dim == 64) return prefill_tc_for<64>(a, stream);
    return cudaErrorInvalidValue;
}

}  // namespace ll
