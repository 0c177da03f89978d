// Decode attention over the paged KV cache: the flash_attention_decode
// variant of the Llama2-7B operator chain (page "Which ops-transformer
// operators one Llama2-7B layer calls", section "KV Cache and the operators":
// a one-row query per head against the cached K/V).  K/V are read through
// block_table from the pool [num_blocks, n_kv_heads, block_size, head_dim]
// (paging page, section "KV Cache memory wall"); the score matrix is never
// materialised and each query row keeps a running max / denominator (online
// softmax, exp2 with the scale folded into log2 e).  Query head h reads KV
// head h / (n_heads / n_kv_heads).  The probabilities P enter the P V product
// as two BF16 parts (hi + lo), so P keeps about 16 significant bits; V stays
// exact.  (The prefill variant lives in attn_tc.cu.)
//
// Decode: the context of each (sequence, KV head) is cut into 1024-key
// splits, one CTA each; a producer warp streams the split's K/V tiles from the
// paged pool with TMA into a 3-stage mbarrier ring; 4 consumer warps share
// the G = n_heads / n_kv_heads query rows of the group (padded to 16 MMA rows)
// and each takes 16 keys of every 64-key tile.  Warps merge in shared memory,
// splits merge in a second kernel through their log-sum-exp.
#include <algorithm>
#include <cfloat>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

// Scratch for ll_paged_attention_decode_noalloc: the per-split partial
// results of decode attention live in this fixed device array instead of a
// caller-provided workspace.  Every GPU that loads the library holds it until
// the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace ll {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kDecodeChunk = 1024;

// byte offset of 16-byte chunk c of row r in a [rows][D] BF16 tile whose
// chunks are XOR-swizzled by (r & 7)
template <int D>
LL_DEVINL uint32_t swz(int r, int c) {
    return (uint32_t)(r * (D * 2) + ((c ^ (r & 7)) << 4));
}

// ---------------------------------------------------------------- decode dispatch order
// Entry L of the order table is the work of the split kernel's CTA with linear index L
// (x fastest): {sequence, KV head, split, context length}, or sequence -1 for none.
// Every full 1024-key split comes first (they all take the same time), then each
// sequence's partial last split, longest first (in sequence order for batches above
// kOrderSortMax), so that the CTAs still running at the end of the grid are short ones.
constexpr int kOrderThreads = 1024;
constexpr int kOrderSortMax = 512;
constexpr int kOrderMaxBatch = 8192;    // shared memory: three ints per sequence

// exclusive prefix sum over the block (one value per thread) and the block total
LL_DEVINL long long block_exclusive_scan(long long v, long long* s_warp, long long& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) s_warp[lane] = w;         // inclusive prefix of the warp totals
    }
    __syncthreads();
    total = s_warp[nw - 1];
    return (warp ? s_warp[warp - 1] : 0) + x - v;
}

__global__ void __launch_bounds__(kOrderThreads) attn_decode_order_kernel(const AttnDecodeArgs a, int max_splits) {
    extern __shared__ int s_ord[];             // [batch] context, [batch] full-split prefix, [batch] partial slot -> sequence
    __shared__ long long s_warp[32];
    pdl_trigger();
    const int B = a.batch, Hkv = a.n_kv_heads;
    const int max_ctx = a.max_blocks * a.block_size;
    int* s_c = s_ord;
    int* s_f = s_ord + B;
    int* s_inv = s_ord + 2 * B;
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        int c = a.context_lens[b];
        if (c < 0 || c > max_ctx) {
            flag_status(a.status, LL_DEV_BAD_POSITION);
            c = min(max(c, 0), max_ctx);
        }
        s_c[b] = c;
    }
    __syncthreads();
    // per sequence: full splits (high 32 bits) and whether a partial split follows (low 32 bits),
    // summed over a contiguous chunk of sequences per thread, then scanned over the block
    const int per = (B + (int)blockDim.x - 1) / (int)blockDim.x;
    const int b0 = min(B, (int)threadIdx.x * per), b1 = min(B, b0 + per);
    long long mine = 0;
    for (int b = b0; b < b1; ++b)
        mine += ((long long)(s_c[b] / kDecodeChunk) << 32) + (s_c[b] % kDecodeChunk != 0);
    long long total;
    long long run = block_exclusive_scan(mine, s_warp, total);
    const bool sorted = B <= kOrderSortMax;
    for (int b = b0; b < b1; ++b) {
        s_f[b] = (int)(run >> 32);
        if (!sorted && s_c[b] % kDecodeChunk != 0) s_inv[(int)(run & 0xffffffffll)] = b;
        run += ((long long)(s_c[b] / kDecodeChunk) << 32) + (s_c[b] % kDecodeChunk != 0);
    }
    const int F = (int)(total >> 32), P = (int)(total & 0xffffffffll);
    if (sorted) {
        // slot of a partial split: its rank by decreasing length (ties by sequence)
        for (int b = threadIdx.x; b < B; b += blockDim.x) {
            const int pk = s_c[b] % kDecodeChunk;
            if (pk == 0) continue;
            int r = 0;
            for (int j = 0; j < B; ++j) {
                const int pj = s_c[j] % kDecodeChunk;
                r += (pj > pk) || (pj == pk && j < b);
            }
            s_inv[r] = b;
        }
    }
    __syncthreads();
    // one entry per thread and step, consecutive threads on consecutive entries: full split
    // f (in sequence order) of KV head hk at f * Hkv + hk, then the partial splits by slot
    const long long full_end = (long long)Hkv * F, used = (long long)Hkv * ((long long)F + P);
    const long long all = (long long)max_splits * Hkv * B;
    for (long long L = threadIdx.x; L < all; L += blockDim.x) {
        int4 e = make_int4(-1, 0, 0, 0);
        if (L < full_end) {
            const int f = (int)(L / Hkv), hk = (int)(L - (long long)f * Hkv);
            int lo = 0, hi = B - 1;                  // last sequence whose full splits start at or before f
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_f[mid] <= f) lo = mid; else hi = mid - 1;
            }
            e = make_int4(lo, hk, f - s_f[lo], s_c[lo]);
        } else if (L < used) {
            const long long q = L - full_end;
            const int r = (int)(q / Hkv), hk = (int)(q - (long long)r * Hkv);
            const int b = s_inv[r];
            e = make_int4(b, hk, s_c[b] / kDecodeChunk, s_c[b]);
        }
        a.order[L] = e;
    }
    // the split kernel waits for this grid only: keep it ordered after the kernel before
    pdl_wait();
}

// The work of this CTA of the split grid: from the dispatch order when there is one, else
// the grid position (split, KV head, sequence).  False: nothing to do.
struct DecodeWork {
    int b, hk, split, ctx;
};

LL_DEVINL bool decode_work(const AttnDecodeArgs& a, DecodeWork& w) {
    if (a.order) {
        const int4 e = a.order[blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)];
        w.b = e.x;
        w.hk = e.y;
        w.split = e.z;
        w.ctx = e.w;
        return e.x >= 0;
    }
    w.split = blockIdx.x;
    w.hk = blockIdx.y;
    w.b = blockIdx.z;
    int ctx = a.context_lens[w.b];
    if (ctx > a.max_blocks * a.block_size || ctx < 0) {
        if (threadIdx.x == 0 && w.split == 0 && w.hk == 0) flag_status(a.status, LL_DEV_BAD_POSITION);
        ctx = min(max(ctx, 0), a.max_blocks * a.block_size);
    }
    w.ctx = ctx;
    return true;
}

// ---------------------------------------------------------------- decode

// Column of the BF16 kernel's merge buffer [4 warps][16 rows][D] that holds head dim `col`
// of row r: bits 0, 3 and 4 XORed with the three low bits of r, so that a warp's
// accumulator stores (rows g and g + 8, columns 8 i + 2 cq + e) hit 32 distinct banks and
// a warp's row reads stay conflict-free.
LL_DEVINL int bf16_merge_col(int r, int col) {
    return col ^ (r & 1) ^ (((r >> 1) & 1) << 3) ^ (((r >> 2) & 1) << 4);
}

// Byte offset of 16-byte chunk c of row r in a K/V tile that TMA wrote with the
// 128-byte swizzle: the tile is [D/64 column halves][ROWS rows][128 bytes] and
// chunk (c & 7) of a row sits at position (c & 7) ^ (r & 7).
template <int ROWS>
LL_DEVINL uint32_t tswz(int r, int c) {
    return (uint32_t)((c >> 3) * (ROWS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// One CTA = one (sequence, KV head, 1024-key split).  Warp 4 is the producer:
// one lane loads each 64-key K and V tile of the split with TMA, as boxes of
// min(block_size, 64) rows x 64 columns taken straight from the paged pool at
// the block_table's physical block, into a 3-stage ring guarded by mbarriers.
// Warps 0-3 consume: each owns 16 keys of every tile, multiplies the group's
// query rows (padded to 16) with them on the tensor cores and keeps its own
// online-softmax state; the four merge in shared memory at the end.
template <int D>
__global__ void __launch_bounds__(160, 2)
    attn_decode_split_kernel(const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const AttnDecodeArgs a,
                             int max_splits) {
    constexpr int BN = 64, STAGES = 3, NCONS = 128;
    constexpr int TILE = BN * D * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sk = sbase;                       // [STAGES][TILE]
    uint8_t* sv = sk + STAGES * TILE;          // [STAGES][TILE]
    uint8_t* sq = sv + STAGES * TILE;          // [16][D], XOR-swizzled rows
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ int abort_s;

    const int G = a.n_heads / a.n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    DecodeWork wk;
    if (!decode_work(a, wk)) return;
    const int split = wk.split, hk = wk.hk, b = wk.b, ctx = wk.ctx;
    const int k_begin = split * kDecodeChunk;
    const int k_end = min(ctx, k_begin + kDecodeChunk);
    const size_t part_row = ((size_t)b * a.n_heads + (size_t)hk * G) * max_splits + split;
    if (k_begin >= k_end) {
        if (threadIdx.x < G) {
            float* ml = a.part_ml + 2 * (part_row + (size_t)threadIdx.x * max_splits);
            ml[0] = -INFINITY;
            ml[1] = 0.f;
        }
        return;
    }
    const int32_t* table_row = a.block_table + (size_t)b * a.max_blocks;
    const int n_kt = (k_end - k_begin + BN - 1) / BN;
    const int kt_rows = min(a.block_size, BN);

    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&full_bar[st], 1);
            mbar_init(&empty_bar[st], 4);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 4) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t issued = 0, parity = 0;    // per stage: a load was issued; parity of the loads issued
            for (int kt = 0; kt < n_kt; ++kt) {
                const int st = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait_bounded(&empty_bar[st], ph ^ 1u, &abort_s, a.status)) break;
                const int p0 = k_begin + kt * BN;
                uint32_t bytes = 0;
                for (int p = p0; p < p0 + BN && p < k_end; p += kt_rows) {
                    const int blk = table_row[p / a.block_size];
                    if (blk >= 0 && blk < a.num_blocks) bytes += 2u * (D / 64) * kt_rows * 128u;
                }
                mbar_arrive_expect_tx(&full_bar[st], bytes);
                for (int p = p0, sb = 0; p < p0 + BN && p < k_end; p += kt_rows, ++sb) {
                    const int blk = table_row[p / a.block_size];
                    if (blk < 0 || blk >= a.num_blocks) {
                        flag_status(a.status, LL_DEV_BAD_BLOCK);
                        continue;
                    }
                    const int row = (blk * a.n_kv_heads + hk) * a.block_size + (p % a.block_size);
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        const uint32_t off = (uint32_t)(st * TILE + h * (BN * 128) + sb * kt_rows * 128);
                        tma_load_2d(sk + off, &tmK, h * 64, row, &full_bar[st]);
                        tma_load_2d(sv + off, &tmV, h * 64, row, &full_bar[st]);
                    }
                }
                issued |= 1u << st;
                parity ^= 1u << st;
            }
            if (abort_s) {
                volatile int never = 0;
                for (int st = 0; st < STAGES; ++st)
                    if ((issued >> st) & 1u) mbar_wait_bounded(&full_bar[st], ((parity >> st) & 1u) ^ 1u, &never, nullptr);
            }
        }
        __syncwarp();
        return;
    }

    // ---------------------------------------------------- consumers (warps 0-3)
    {
        constexpr int CPR = D / 8;
        for (int i = threadIdx.x; i < 16 * CPR; i += NCONS) {
            const int r = i / CPR, c = i % CPR;
            const bool ok = r < G;
            const __nv_bfloat16* src = a.q + ((size_t)b * a.n_heads + hk * G + (ok ? r : 0)) * D + c * 8;
            cp_async16(sq + swz<D>(r, c), src, ok);
        }
        cp_async_commit();
        cp_async_wait<0>();
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    uint32_t qf[D / 16][4];
    {
        const uint32_t qb = smem_u32(sq);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) ldmatrix_x4(qf[ks], qb + swz<D>(lane & 15, ks * 2 + (lane >> 4)));
    }

    const float sl2 = a.scale * kLog2e;
    const int g = lane >> 2, cq = lane & 3;
    float acc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int kt = 0; kt < n_kt; ++kt) {
        const int st = kt % STAGES;
        const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
        if (!mbar_wait_bounded(&full_bar[st], ph, &abort_s, a.status)) break;
        uint8_t* kbp = sk + st * TILE;
        uint8_t* vbp = sv + st * TILE;
        // validity of this warp's 16 keys: inside the split and backed by a valid block
        const int pbase = k_begin + kt * BN + warp * 16;
        bool my_ok = false;
        if (lane < 16) {
            const int p = pbase + lane;
            if (p < k_end) {
                const int blk = table_row[p / a.block_size];
                my_ok = blk >= 0 && blk < a.num_blocks;
            }
        }
        const uint32_t okmask = __ballot_sync(0xffffffffu, my_ok) & 0xffffu;
        if (okmask != 0xffffu) {
            // rows that hold no valid key: zero their V so 0 * garbage cannot be NaN
            for (int i = lane; i < 16 * (D / 8); i += 32) {
                const int r = i / (D / 8), c = i % (D / 8);
                if (!((okmask >> r) & 1u))
                    *reinterpret_cast<uint4*>(vbp + tswz<BN>(warp * 16 + r, c)) = make_uint4(0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        }
        const uint32_t kb = smem_u32(kbp), vb = smem_u32(vbp);
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
            uint32_t bfr[4];
            const int r = warp * 16 + (lane & 7) + ((lane >> 4) << 3);
            const int c = ks * 2 + ((lane >> 3) & 1);
            ldmatrix_x4(bfr, kb + tswz<BN>(r, c));
            mma_bf16_16816(s[0], qf[ks], bfr[0], bfr[1]);
            mma_bf16_16816(s[1], qf[ks], bfr[2], bfr[3]);
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int kk = nt * 8 + 2 * cq;   // key index within the warp's 16
            const bool v0 = (okmask >> kk) & 1u, v1 = (okmask >> (kk + 1)) & 1u;
            s[nt][0] = v0 ? s[nt][0] * sl2 : -INFINITY;
            s[nt][1] = v1 ? s[nt][1] * sl2 : -INFINITY;
            s[nt][2] = v0 ? s[nt][2] * sl2 : -INFINITY;
            s[nt][3] = v1 ? s[nt][3] * sl2 : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
#pragma unroll
        for (int o = 1; o <= 2; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float base0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float base1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float al0 = exp2f(m0 - base0), al1 = exp2f(m1 - base1);
        m0 = mn0;
        m1 = mn1;
        uint32_t phi[4], plo[4];
        float rs0 = 0.f, rs1 = 0.f;
        {
            float p[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                p[nt][0] = exp2f(s[nt][0] - base0);
                p[nt][1] = exp2f(s[nt][1] - base0);
                p[nt][2] = exp2f(s[nt][2] - base1);
                p[nt][3] = exp2f(s[nt][3] - base1);
                rs0 += p[nt][0] + p[nt][1];
                rs1 += p[nt][2] + p[nt][3];
            }
            // P carried as hi + lo BF16 parts (about 16 bits)
            split_bf16x2(p[0][0], p[0][1], phi[0], plo[0]);
            split_bf16x2(p[0][2], p[0][3], phi[1], plo[1]);
            split_bf16x2(p[1][0], p[1][1], phi[2], plo[2]);
            split_bf16x2(p[1][2], p[1][3], phi[3], plo[3]);
        }
        l0 = l0 * al0 + rs0;
        l1 = l1 * al1 + rs1;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            acc[i][0] *= al0;
            acc[i][1] *= al0;
            acc[i][2] *= al1;
            acc[i][3] *= al1;
        }
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
            uint32_t bfr[4];
            const int r = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            const int c = dp * 2 + (lane >> 4);
            ldmatrix_x4_trans(bfr, vb + tswz<BN>(r, c));
            mma_bf16_16816(acc[2 * dp], phi, bfr[0], bfr[1]);
            mma_bf16_16816(acc[2 * dp + 1], phi, bfr[2], bfr[3]);
            mma_bf16_16816(acc[2 * dp], plo, bfr[0], bfr[1]);
            mma_bf16_16816(acc[2 * dp + 1], plo, bfr[2], bfr[3]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
    }
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }

    // merge the 4 consumer warps: [4][16] (m, l) and [4][16][D] acc, over the K ring
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float* s_ml = reinterpret_cast<float*>(sk);            // [4][16][2]
    float* s_acc = s_ml + 4 * 16 * 2;                      // [4][16][D]
    if (cq == 0) {
        s_ml[(warp * 16 + g) * 2 + 0] = m0;
        s_ml[(warp * 16 + g) * 2 + 1] = l0;
        s_ml[(warp * 16 + g + 8) * 2 + 0] = m1;
        s_ml[(warp * 16 + g + 8) * 2 + 1] = l1;
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
        const int col = i * 8 + 2 * cq;
        s_acc[(warp * 16 + g) * D + bf16_merge_col(g, col)] = acc[i][0];
        s_acc[(warp * 16 + g) * D + bf16_merge_col(g, col + 1)] = acc[i][1];
        s_acc[(warp * 16 + g + 8) * D + bf16_merge_col(g, col)] = acc[i][2];
        s_acc[(warp * 16 + g + 8) * D + bf16_merge_col(g, col + 1)] = acc[i][3];
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int i = threadIdx.x; i < G * D; i += NCONS) {
        const int r = i / D, col = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, s_ml[(w * 16 + r) * 2]);
        const float base = (M == -INFINITY) ? 0.f : M;
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float e = exp2f(s_ml[(w * 16 + r) * 2] - base);
            num += e * s_acc[(w * 16 + r) * D + bf16_merge_col(r, col)];
            den += e * s_ml[(w * 16 + r) * 2 + 1];
        }
        const size_t pr = part_row + (size_t)r * max_splits;
        a.part_o[pr * D + col] = den > 0.f ? num / den : 0.f;
        if (col == 0) {
            a.part_ml[2 * pr] = M;
            a.part_ml[2 * pr + 1] = den;
        }
    }
}

// Column of the INT8 kernel's merge buffer [4 warps][16 rows][128] that holds head dim `col`
// of row r: XOR-swizzled within each 32-column group, so that a warp's accumulator stores
// (8 dims 16 apart in 4 row pairs) hit 32 distinct banks and a warp's row reads stay
// conflict-free.
LL_DEVINL int q8_merge_col(int r, int col) {
    return col ^ (((col >> 5) & 3) << 1) ^ ((r >> 1) & 1) ^ (((r >> 2) & 1) << 3);
}

// ---------------------------------------------------------------- decode over an INT8 cache
// The same split / warp structure over an INT8 pool (head_dim 128; paging page,
// section "KV Cache quantisation": the cache block is dequantised as it is
// loaded).  The producer streams each 64-key tile's codes (128-byte rows, the
// 128-byte swizzle) with TMA and its K and V scales with bulk copies, all on
// the stage's barrier.  Each consumer warp owns 16 keys of every tile and runs
// both products transposed, so that its keys (then the head dims) fill the
// MMA's 16 rows and the group's query rows its 8 columns (NT column tiles for
// groups of 9 to 16): S^T = K Q^T and O^T = V^T P^T, the codes converted
// straight from shared memory into FP16 A fragments (exact: |code| <= 127).
// The S^T fragment of a lane holds two keys of two query columns; transposing
// its two 8x8 FP16 halves (movmatrix) gives the B fragment of P^T.  A key's K
// scale multiplies its score and its V scale its probability before P V, so
// dequantised values are never formed; the row sum stays the sum of the
// unscaled probabilities.  Q enters as FP16 (exact for BF16 values of FP16's
// range).  P times the V scale enters P V as two FP16 parts (hi + lo), with the
// exponent base set by the largest such weight so that the parts stay in FP16's
// normal range: one FP16 operand under the score's own base left 7e-3 of the 7B
// decode layer's outputs outside the per-element bound against the oracle (which
// reads the same codes exactly), and a CPU model of the layer puts this form at
// 6e-4, the same as exact probabilities.
// One column tile runs four CTAs per SM (94 registers); two run two (their
// accumulators take 64 registers).
template <int NT>
__global__ void __launch_bounds__(160, NT == 1 ? 4 : 2)
    attn_decode_split_q8_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                                const AttnDecodeArgs a, int max_splits) {
    constexpr int D = 128, BN = 64, STAGES = 3, NCONS = 128;
    constexpr int TILE = BN * D;                       // bytes of one INT8 K or V tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sbase = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sk = sbase;                               // [STAGES][TILE] codes
    uint8_t* sv = sk + STAGES * TILE;                  // [STAGES][TILE]
    float* ssc = reinterpret_cast<float*>(sv + STAGES * TILE);   // [STAGES][2][BN] K, V scales
    uint8_t* sq = reinterpret_cast<uint8_t*>(ssc + STAGES * 2 * BN);   // [16][D] FP16 q, swizzled rows
    __shared__ uint64_t full_bar[STAGES], empty_bar[STAGES];
    __shared__ unsigned long long valid_s[STAGES];     // per stage: bit k = key k of the tile is cached
    __shared__ int abort_s;

    const int G = a.n_heads / a.n_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    DecodeWork wk;
    if (!decode_work(a, wk)) return;
    const int split = wk.split, hk = wk.hk, b = wk.b, ctx = wk.ctx;
    const int k_begin = split * kDecodeChunk;
    const int k_end = min(ctx, k_begin + kDecodeChunk);
    const size_t part_row = ((size_t)b * a.n_heads + (size_t)hk * G) * max_splits + split;
    if (k_begin >= k_end) {
        if (threadIdx.x < G) {
            float* ml = a.part_ml + 2 * (part_row + (size_t)threadIdx.x * max_splits);
            ml[0] = -INFINITY;
            ml[1] = 0.f;
        }
        return;
    }
    const int32_t* table_row = a.block_table + (size_t)b * a.max_blocks;
    const int n_kt = (k_end - k_begin + BN - 1) / BN;
    const int kt_rows = min(a.block_size, BN);

    if (threadIdx.x == 0) {
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&full_bar[st], 1);
            mbar_init(&empty_bar[st], 4);
        }
        abort_s = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == 4) {
        // ------------------------------------------------ producer
        if (lane == 0) {
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            uint32_t issued = 0, parity = 0;    // per stage: a load was issued; parity of the loads issued
            for (int kt = 0; kt < n_kt; ++kt) {
                const int st = kt % STAGES;
                const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
                if (!mbar_wait_bounded(&empty_bar[st], ph ^ 1u, &abort_s, a.status)) break;
                const int p0 = k_begin + kt * BN;
                uint32_t bytes = 0;
                unsigned long long valid = 0;
                for (int p = p0, sb = 0; p < p0 + BN && p < k_end; p += kt_rows, ++sb) {
                    const int blk = table_row[p / a.block_size];
                    if (blk >= 0 && blk < a.num_blocks) {
                        bytes += 2u * kt_rows * (128u + 4u);
                        const int nk = min(kt_rows, k_end - p);
                        valid |= (nk == 64 ? ~0ull : ((1ull << nk) - 1ull)) << (sb * kt_rows);
                    }
                }
                valid_s[st] = valid;                       // released by the arrive below
                mbar_arrive_expect_tx(&full_bar[st], bytes);
                for (int p = p0, sb = 0; p < p0 + BN && p < k_end; p += kt_rows, ++sb) {
                    const int blk = table_row[p / a.block_size];
                    if (blk < 0 || blk >= a.num_blocks) {
                        flag_status(a.status, LL_DEV_BAD_BLOCK);
                        continue;
                    }
                    const size_t row = ((size_t)blk * a.n_kv_heads + hk) * a.block_size + (p % a.block_size);
                    const uint32_t off = (uint32_t)(st * TILE + sb * kt_rows * 128);
                    tma_load_2d(sk + off, &tmK, 0, (int)row, &full_bar[st]);
                    tma_load_2d(sv + off, &tmV, 0, (int)row, &full_bar[st]);
                    bulk_load(ssc + (st * 2 + 0) * BN + sb * kt_rows, a.k_scale + row, (uint32_t)kt_rows * 4u,
                              &full_bar[st]);
                    bulk_load(ssc + (st * 2 + 1) * BN + sb * kt_rows, a.v_scale + row, (uint32_t)kt_rows * 4u,
                              &full_bar[st]);
                }
                issued |= 1u << st;
                parity ^= 1u << st;
            }
            if (abort_s) {
                volatile int never = 0;
                for (int st = 0; st < STAGES; ++st)
                    if ((issued >> st) & 1u) mbar_wait_bounded(&full_bar[st], ((parity >> st) & 1u) ^ 1u, &never, nullptr);
            }
        }
        __syncwarp();
        return;
    }

    // ---------------------------------------------------- consumers (warps 0-3)
    for (int i = threadIdx.x; i < 16 * (D / 8); i += NCONS) {
        // q rows of the group (zero padding to 16 rows) as FP16
        const int r = i / (D / 8), c = i % (D / 8);
        uint4 o = make_uint4(0, 0, 0, 0);
        if (r < G) {
            const uint4 w = *reinterpret_cast<const uint4*>(a.q + ((size_t)b * a.n_heads + hk * G + r) * D + c * 8);
            o.x = pack_f16x2(bf16_lo(w.x), bf16_hi(w.x));
            o.y = pack_f16x2(bf16_lo(w.y), bf16_hi(w.y));
            o.z = pack_f16x2(bf16_lo(w.z), bf16_hi(w.z));
            o.w = pack_f16x2(bf16_lo(w.w), bf16_hi(w.w));
        }
        *reinterpret_cast<uint4*>(sq + swz<D>(r, c)) = o;
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    const float sl2 = a.scale * kLog2e;
    const int g = lane >> 2, cq = lane & 3;
    // B fragments of Q^T, column g of tile nt = query row 8 nt + g.  The head dims are permuted
    // alike in Q and K: MMA step ks gives k indices 2 cq + e and 2 cq + 8 + e (e = 0, 1) the
    // dims 32 cq + 4 ks + e and 32 cq + 4 ks + 2 + e, so that lane cq reads 32 consecutive
    // code bytes of each of its key rows.
    uint2 qf[NT][D / 16];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
            qf[nt][ks] = *reinterpret_cast<const uint2*>(sq + swz<D>(8 * nt + g, 4 * cq + (ks >> 1)) + (ks & 1) * 8);
    // O^T: row r of tile t is head dim 16 (r & 7) + 2 t + (r >> 3), column n of tile nt
    // query row 8 nt + n.  Per query column: running max m (the exponent base) and the lane's
    // part of the row sum l.
    float acc[NT][D / 16][4];
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int t = 0; t < D / 16; ++t) acc[nt][t][0] = acc[nt][t][1] = acc[nt][t][2] = acc[nt][t][3] = 0.f;
        m[nt][0] = m[nt][1] = -INFINITY;
        l[nt][0] = l[nt][1] = 0.f;
    }

    for (int kt = 0; kt < n_kt; ++kt) {
        const int st = kt % STAGES;
        const uint32_t ph = (uint32_t)(kt / STAGES) & 1u;
        if (!mbar_wait_bounded(&full_bar[st], ph, &abort_s, a.status)) break;
        // validity of this warp's 16 keys (inside the split and backed by a valid block), as
        // the producer found it
        const uint32_t okmask = (uint32_t)(valid_s[st] >> (warp * 16)) & 0xffffu;
        const uint8_t* ktile = sk + st * TILE;
        const uint8_t* vtile = sv + st * TILE;
        // S^T = K Q^T: A rows g and g + 8 are the warp's keys g and g + 8.  Keys without a
        // valid block hold stale (finite) codes; their scores are masked below.
        uint32_t kw[2][8];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int R = warp * 16 + j * 8 + g;
            const uint4 w0 = *reinterpret_cast<const uint4*>(ktile + R * 128 + (((2 * cq) ^ (R & 7)) << 4));
            const uint4 w1 = *reinterpret_cast<const uint4*>(ktile + R * 128 + (((2 * cq + 1) ^ (R & 7)) << 4));
            kw[j][0] = w0.x; kw[j][1] = w0.y; kw[j][2] = w0.z; kw[j][3] = w0.w;
            kw[j][4] = w1.x; kw[j][5] = w1.y; kw[j][6] = w1.z; kw[j][7] = w1.w;
        }
        float s[NT][4];
        {
            // two accumulators per column tile (even and odd steps) halve the MMA chain
            float sp[NT][2][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int h = 0; h < 2; ++h) sp[nt][h][0] = sp[nt][h][1] = sp[nt][h][2] = sp[nt][h][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t af[4];
                i8x4_to_f16x4(kw[0][ks], af[0], af[2]);
                i8x4_to_f16x4(kw[1][ks], af[1], af[3]);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_f16_16816(sp[nt][ks & 1], af, qf[nt][ks].x, qf[nt][ks].y);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 4; ++j) s[nt][j] = sp[nt][0][j] + sp[nt][1][j];
        }
        // lane: keys g (s[.][0..1]) and g + 8 (s[.][2..3]) of query columns 2 cq and 2 cq + 1
        const float* ksc = ssc + (st * 2 + 0) * BN + warp * 16;
        const float* vsc = ssc + (st * 2 + 1) * BN + warp * 16;
        const bool v0 = (okmask >> g) & 1u, v1 = (okmask >> (g + 8)) & 1u;
        const float f0 = sl2 * ksc[g], f1 = sl2 * ksc[g + 8];
        const float vs0 = v0 ? vsc[g] : 0.f, vs1 = v1 ? vsc[g + 8] : 0.f;
        // A key's weight in P V is its probability times its V scale, so the exponent base
        // follows the largest log2 weight: P times the V scale then stays below 2^8 and in FP16's
        // normal range down to 2^-14 of the largest weight (keys below that no longer matter).
        // Scales under 2^-40 count as 2^-40, which keeps P itself below 2^48.
        const float lv0 = fmaxf(lg2_approx(vs0), -40.f), lv1 = fmaxf(lg2_approx(vs1), -40.f);
        float mx[NT][2];
        bool grow = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            s[nt][0] = v0 ? s[nt][0] * f0 : -INFINITY;
            s[nt][1] = v0 ? s[nt][1] * f0 : -INFINITY;
            s[nt][2] = v1 ? s[nt][2] * f1 : -INFINITY;
            s[nt][3] = v1 ? s[nt][3] * f1 : -INFINITY;
            mx[nt][0] = fmaxf(s[nt][0] + lv0, s[nt][2] + lv1);
            mx[nt][1] = fmaxf(s[nt][1] + lv0, s[nt][3] + lv1);
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) {
                mx[nt][0] = fmaxf(mx[nt][0], __shfl_xor_sync(0xffffffffu, mx[nt][0], o));
                mx[nt][1] = fmaxf(mx[nt][1], __shfl_xor_sync(0xffffffffu, mx[nt][1], o));
            }
            grow = grow || mx[nt][0] > m[nt][0] + 8.f || mx[nt][1] > m[nt][1] + 8.f;
        }
        // The exponent base of a column moves only when its max grows by more than 2^8 (P times
        // the V scale then stays below 256); otherwise the running sums need no rescaling.
        if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float mn = mx[nt][e] > m[nt][e] + 8.f ? mx[nt][e] : m[nt][e];
                    const float al = mn == m[nt][e] ? 1.f : ex2_approx(m[nt][e] - mn);
                    l[nt][e] *= al;
#pragma unroll
                    for (int t = 0; t < D / 16; ++t) {
                        acc[nt][t][e] *= al;
                        acc[nt][t][e + 2] *= al;
                    }
                    m[nt][e] = mn;
                }
        }
        // P^T (each key's V scale riding on its probability) as the B fragments of O^T = V^T P^T,
        // in two FP16 parts (hi + lo, about 22 significant bits together)
        uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const float b0 = (m[nt][0] == -INFINITY) ? 0.f : m[nt][0];
            const float b1 = (m[nt][1] == -INFINITY) ? 0.f : m[nt][1];
            const float p00 = ex2_approx(s[nt][0] - b0), p01 = ex2_approx(s[nt][1] - b1);
            const float p10 = ex2_approx(s[nt][2] - b0), p11 = ex2_approx(s[nt][3] - b1);
            l[nt][0] += p00 + p10;
            l[nt][1] += p01 + p11;
            uint32_t h0, l0, h1, l1;
            split_f16x2(p00 * vs0, p01 * vs0, h0, l0);     // keys 0-7
            split_f16x2(p10 * vs1, p11 * vs1, h1, l1);     // keys 8-15
            pb[nt][0] = movmatrix_trans(h0);
            pb[nt][1] = movmatrix_trans(h1);
            pl[nt][0] = movmatrix_trans(l0);
            pl[nt][1] = movmatrix_trans(l1);
        }
        // O^T += V^T P^T: lane g reads one 16-byte chunk (dims 16 g .. 16 g + 15) of each of its
        // key rows 2 cq, 2 cq + 1, 2 cq + 8, 2 cq + 9 and byte-interleaves the rows of a key pair
        // into FP16 pairs: word i gives tile 2 i (dims 16 g + 4 i, + 1) and tile 2 i + 1 (+ 2, + 3).
        uint32_t vw[4][4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const int R = warp * 16 + 2 * cq + (q4 & 1) + (q4 >> 1) * 8;
            const uint4 w = *reinterpret_cast<const uint4*>(vtile + R * 128 + ((g ^ (R & 7)) << 4));
            vw[q4][0] = w.x; vw[q4][1] = w.y; vw[q4][2] = w.z; vw[q4][3] = w.w;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t x01, y01, x23, y23;
            asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(x01) : "r"(vw[0][i]), "r"(vw[1][i]));
            asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(y01) : "r"(vw[0][i]), "r"(vw[1][i]));
            asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(x23) : "r"(vw[2][i]), "r"(vw[3][i]));
            asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(y23) : "r"(vw[2][i]), "r"(vw[3][i]));
            uint32_t at0[4], at1[4];
            i8x4_to_f16x4(x01, at0[0], at0[1]);      // keys 2 cq, 2 cq + 1: dims 16 g + 4 i, + 1
            i8x4_to_f16x4(x23, at0[2], at0[3]);      // keys 2 cq + 8, 2 cq + 9
            i8x4_to_f16x4(y01, at1[0], at1[1]);      // dims 16 g + 4 i + 2, + 3
            i8x4_to_f16x4(y23, at1[2], at1[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                mma_f16_16816(acc[nt][2 * i], at0, pb[nt][0], pb[nt][1]);
                mma_f16_16816(acc[nt][2 * i + 1], at1, pb[nt][0], pb[nt][1]);
                mma_f16_16816(acc[nt][2 * i], at0, pl[nt][0], pl[nt][1]);
                mma_f16_16816(acc[nt][2 * i + 1], at1, pl[nt][0], pl[nt][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
            for (int o = 4; o <= 16; o <<= 1) l[nt][e] += __shfl_xor_sync(0xffffffffu, l[nt][e], o);

    // merge the 4 consumer warps: [4][16] (m, l) and [4][16][D] acc, over the code rings
    asm volatile("bar.sync 1, 128;" ::: "memory");
    float* s_ml = reinterpret_cast<float*>(sk);            // [4][16][2]
    float* s_acc = s_ml + 4 * 16 * 2;                      // [4][16][D]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        if (g == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = warp * 16 + 8 * nt + 2 * cq + e;
                s_ml[r * 2 + 0] = m[nt][e];
                s_ml[r * 2 + 1] = l[nt][e];
            }
        }
#pragma unroll
        for (int t = 0; t < D / 16; ++t)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int r = 8 * nt + 2 * cq + (j & 1);
                s_acc[(warp * 16 + r) * D + q8_merge_col(r, 16 * g + 2 * t + (j >> 1))] = acc[nt][t][j];
            }
    }
    asm volatile("bar.sync 1, 128;" ::: "memory");
    for (int i = threadIdx.x; i < G * D; i += NCONS) {
        const int r = i / D, col = i % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, s_ml[(w * 16 + r) * 2]);
        const float base = (M == -INFINITY) ? 0.f : M;
        float num = 0.f, den = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const float e = exp2f(s_ml[(w * 16 + r) * 2] - base);
            num += e * s_acc[(w * 16 + r) * D + q8_merge_col(r, col)];
            den += e * s_ml[(w * 16 + r) * 2 + 1];
        }
        const size_t pr = part_row + (size_t)r * max_splits;
        a.part_o[pr * D + col] = den > 0.f ? num / den : 0.f;
        if (col == 0) {
            a.part_ml[2 * pr] = M;
            a.part_ml[2 * pr + 1] = den;
        }
    }
}

// out[b][h] = sum_s 2^(m_s - M) l_s o_s / sum_s 2^(m_s - M) l_s over the splits of (b, h)
__global__ void attn_decode_combine_kernel(const AttnDecodeArgs a, int max_splits) {
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y;
    const int D = a.head_dim;
    int ctx = min(max(a.context_lens[b], 0), a.max_blocks * a.block_size);
    const int ns = min(max_splits, (ctx + kDecodeChunk - 1) / kDecodeChunk);
    const size_t base_row = ((size_t)b * a.n_heads + h) * max_splits;
    float M = -INFINITY;
    for (int s = 0; s < ns; ++s) M = fmaxf(M, a.part_ml[2 * (base_row + s)]);
    const float mb = (M == -INFINITY) ? 0.f : M;
    for (int col = threadIdx.x; col < D; col += blockDim.x) {
        float num = 0.f, den = 0.f;
        for (int s = 0; s < ns; ++s) {
            const float ms = a.part_ml[2 * (base_row + s)];
            const float w = exp2f(ms - mb) * a.part_ml[2 * (base_row + s) + 1];
            num += w * a.part_o[(base_row + s) * D + col];
            den += w;
        }
        a.out[((size_t)b * a.n_heads + h) * D + col] = __float2bfloat16_rn(den > 0.f ? num / den : 0.f);
    }
}

// The dispatch order table sits in the scratch after the split partials (16-byte entries).
int4* order_table(const AttnDecodeArgs& a, int max_splits) {
    const size_t rows = (size_t)a.batch * a.n_heads * max_splits;
    const uintptr_t p = reinterpret_cast<uintptr_t>(a.part_ml + 2 * rows);
    return reinterpret_cast<int4*>((p + 15) & ~uintptr_t(15));
}

// Launches the order kernel and points a.order at its table.  The table pays where the
// grid's tail is long next to the one more kernel it puts between the QKV epilogue and the
// split kernel: INT8 caches (short CTAs, four per SM) and BF16 contexts of 8 or more splits
// (measured on GB300: 70B decode step 1.5-2% faster; with at most 4-5 splits per sequence,
// the 7B decode and the 32-layer continuous batching, 2-4% slower).  Otherwise, and for
// batches beyond what it sorts in shared memory, a.order is null and the split CTAs work in
// grid order.
constexpr int kOrderMinSplitsBf16 = 8;

cudaError_t launch_order(AttnDecodeArgs& a, int max_splits, bool int8_cache, cudaStream_t stream) {
    if (a.batch > kOrderMaxBatch || (!int8_cache && max_splits < kOrderMinSplitsBf16)) {
        a.order = nullptr;
        return cudaSuccess;
    }
    {
        const cudaError_t e = ensure_func_attr((const void*)attn_decode_order_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)(3 * kOrderMaxBatch * sizeof(int)),
                                               "cudaFuncSetAttribute(attn_decode_order_kernel)");
        if (e != cudaSuccess) return e;
    }
    a.order = order_table(a, max_splits);
    trace_before("attn_decode_order", stream);
    cudaError_t e = launch_pdl(attn_decode_order_kernel, dim3(1), dim3(kOrderThreads), 3 * (size_t)a.batch * sizeof(int),
                               stream, 1, a, max_splits);
    trace_after(stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? cudaSuccess : record(e, "attn_decode_order_kernel launch");
}

template <int D>
cudaError_t decode_for(const AttnDecodeArgs& args, cudaStream_t stream) {
    AttnDecodeArgs a = args;
    const int max_splits = attn_decode_max_splits(a.max_blocks, a.block_size);
    {
        const cudaError_t eo = launch_order(a, max_splits, false, stream);
        if (eo != cudaSuccess) return eo;
    }
    const size_t smem = (size_t)2 * 3 * (64 * D * 2) + 16 * D * 2 + 1024;
    {
        const cudaError_t e = ensure_func_attr((const void*)attn_decode_split_kernel<D>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem,
                                               "cudaFuncSetAttribute(attn_decode_split_kernel)");
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)a.num_blocks * a.n_kv_heads * a.block_size;
    const uint32_t box_rows = (uint32_t)std::min(a.block_size, 64);
    if (!make_tmap_bf16_sw128(&tmK, a.k_pool, D, rows, box_rows) ||
        !make_tmap_bf16_sw128(&tmV, a.v_pool, D, rows, box_rows))
        return cudaErrorInvalidValue;
    dim3 grid(max_splits, a.n_kv_heads, a.batch);
    trace_before("attn_decode_split", stream);
    cudaError_t e = launch_pdl(attn_decode_split_kernel<D>, grid, dim3(160), smem, stream, 1, tmK, tmV, a,
                               max_splits);
    trace_after(stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return record(e, "attn_decode_split_kernel launch");
    trace_before("attn_decode_combine", stream);
    e = launch_pdl(attn_decode_combine_kernel, dim3(a.n_heads, a.batch), dim3(D), 0, stream, 1, a,
                   max_splits);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "attn_decode_combine_kernel launch");
    return record(cudaGetLastError(), "attn_decode_combine_kernel launch");
}

template <int NT>
cudaError_t decode_q8_for(const AttnDecodeArgs& args, cudaStream_t stream) {
    AttnDecodeArgs a = args;
    constexpr int D = 128, BN = 64, STAGES = 3;
    const int max_splits = attn_decode_max_splits(a.max_blocks, a.block_size);
    {
        const cudaError_t eo = launch_order(a, max_splits, true, stream);
        if (eo != cudaSuccess) return eo;
    }
    const size_t smem = (size_t)STAGES * 2 * BN * D + STAGES * 2 * BN * 4 + 16 * D * 2 + 1024;
    {
        cudaError_t e = ensure_func_attr((const void*)attn_decode_split_q8_kernel<NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem,
                                         "cudaFuncSetAttribute(attn_decode_split_q8_kernel)");
        if (e != cudaSuccess) return e;
        // four CTAs of 56 KB per SM need the whole shared-memory carveout
        e = ensure_func_attr((const void*)attn_decode_split_q8_kernel<NT>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared,
                             "cudaFuncSetAttribute(attn_decode_split_q8_kernel carveout)");
        if (e != cudaSuccess) return e;
    }
    CUtensorMap tmK, tmV;
    const uint64_t rows = (uint64_t)a.num_blocks * a.n_kv_heads * a.block_size;
    const uint32_t box_rows = (uint32_t)std::min(a.block_size, BN);
    if (!make_tmap_u8_sw128(&tmK, a.k_q8, rows, box_rows) || !make_tmap_u8_sw128(&tmV, a.v_q8, rows, box_rows))
        return cudaErrorInvalidValue;
    dim3 grid(max_splits, a.n_kv_heads, a.batch);
    trace_before("attn_decode_split", stream);
    cudaError_t e = launch_pdl(attn_decode_split_q8_kernel<NT>, grid, dim3(160), smem, stream, 1, tmK, tmV, a,
                               max_splits);
    trace_after(stream);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return record(e, "attn_decode_split_q8_kernel launch");
    trace_before("attn_decode_combine", stream);
    e = launch_pdl(attn_decode_combine_kernel, dim3(a.n_heads, a.batch), dim3(D), 0, stream, 1, a, max_splits);
    trace_after(stream);
    if (e != cudaSuccess) return record(e, "attn_decode_combine_kernel launch");
    return record(cudaGetLastError(), "attn_decode_combine_kernel launch");
}

}  // namespace

int attn_decode_max_splits(int max_blocks, int block_size) {
    const long long max_ctx = (long long)max_blocks * block_size;
    return (int)std::max<long long>(1, (max_ctx + kDecodeChunk - 1) / kDecodeChunk);
}

size_t attn_decode_scratch_bytes(int batch, int n_heads, int head_dim, int max_blocks,
                                 int block_size) {
    // per split row: the partial output and (m, l); then the dispatch order (one 16-byte entry
    // per CTA of the split grid, at most one per row) behind a 16-byte alignment pad
    const size_t rows = (size_t)batch * n_heads * attn_decode_max_splits(max_blocks, block_size);
    return rows * head_dim * sizeof(float) + rows * 2 * sizeof(float) + 16 + rows * sizeof(int4);
}

cudaError_t launch_attn_decode_q8(const AttnDecodeArgs& a, cudaStream_t stream) {
    if (a.batch <= 0) return cudaSuccess;
    if (a.head_dim != 128 || a.n_kv_heads <= 0 || a.n_heads % a.n_kv_heads != 0) return cudaErrorInvalidValue;
    const int G = a.n_heads / a.n_kv_heads;
    if (G <= 8) return decode_q8_for<1>(a, stream);
    if (G <= 16) return decode_q8_for<2>(a, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_decode(const AttnDecodeArgs& a, cudaStream_t stream) {
    if (a.batch <= 0) return cudaSuccess;
    if (a.head_dim == 128) return decode_for<128>(a, stream);
    if (a.head_dim == 64) return decode_for<64>(a, stream);
    return cudaErrorInvalidValue;
}

namespace {
// Device address of g_noalloc_scratch, resolved once per device.  In host
// code the array's name is only a host-side stand-in, never a device address.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

cudaError_t noalloc_scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record(e, "cudaGetDevice(noalloc)");
    if (dev < 0 || dev >= kMaxDevices) {
        set_last_error("ll_paged_attention_decode_noalloc", "device index beyond 63");
        return cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return record(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return cudaSuccess;
}
}  // namespace

}  // namespace ll

extern "C" int ll_paged_attention_decode_noalloc(const void* q, const ll_kv_pool* pool,
                                                 const int32_t* block_table, int32_t max_blocks,
                                                 const int32_t* context_lens, int32_t batch,
                                                 int32_t n_heads, int32_t n_kv_heads,
                                                 int32_t head_dim, int32_t block_size, float scale,
                                                 void* out, int32_t* status, void* stream) {
    ll::clear_last_error();
    if (!q || !block_table || !context_lens || !out || !status || !pool || !pool->k || !pool->v ||
        pool->num_blocks <= 0)
        return LL_ERR_INVALID_ARG;
    if (batch <= 0 || n_heads <= 0 || n_kv_heads <= 0 || max_blocks <= 0 || block_size <= 0)
        return LL_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return LL_ERR_UNSUPPORTED;
    if (n_heads % n_kv_heads != 0 || n_heads / n_kv_heads > 16) return LL_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 256 || (block_size & (block_size - 1)) != 0)
        return LL_ERR_UNSUPPORTED;
    if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
          reinterpret_cast<uintptr_t>(pool->k) | reinterpret_cast<uintptr_t>(pool->v)) & 15u) != 0)
        return LL_ERR_INVALID_ARG;
    const size_t need = ll::attn_decode_scratch_bytes(batch, n_heads, head_dim, max_blocks, block_size);
    if (need > kNoAllocScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof(msg), "needs %zu bytes of scratch, the fixed array holds %zu", need,
                 kNoAllocScratchBytes);
        ll::set_last_error("ll_paged_attention_decode_noalloc", msg);
        return LL_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    if (ll::noalloc_scratch_address(&scratch) != cudaSuccess) return LL_ERR_CUDA;
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
    at.part_o = static_cast<float*>(scratch);
    at.part_ml = at.part_o + rows * head_dim;
    at.status = status;
    return ll::launch_attn_decode(at, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LL_OK
                                                                                          : LL_ERR_CUDA;
}
