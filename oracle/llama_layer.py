"""CPU oracle of one Llama-style decoder layer -- TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct numpy float64 restatement of what the layer
computes.  Only the tests, `__graft_entry__.smoke()` and the CPU-baseline /
reference legs of `bench.py` may import it; the product path never does.  It
shares no code with the CUDA library and imports nothing from the package.

Sources (web pages on Ascend Transformer Boost; cited by page and section):

* [chain]   "Which ops-transformer operators one Llama2-7B layer calls"
            (seekfood.cn/news/1207529), section "single-layer operator call
            chain": x -> RMSNorm -> Q/K/V Linear -> RotaryEmbedding ->
            Self-Attention (GQA) -> Attention Output Linear -> residual ->
            RMSNorm -> Gate/Up Linear -> SiLU -> Down Linear -> residual; and
            section "KV Cache and the operators": prefill runs the whole
            sequence through FlashAttention, decode has a one-row query
            Q [1, heads, 1, dim] against K/V [1, kv_heads, seq, dim] read from
            the cache.
* [paging]  "ATB KV-cache paging, quantisation, speculative decoding and
            communication overlap" (hwcomputing.csdn.net), section "KV Cache
            memory wall": cache bytes = 2 x L x s x b x d x sizeof(dtype);
            fixed-size blocks, a block_table mapping logical to physical
            blocks, contextLens; ReshapeAndCacheOperation writes the step's
            K/V into the paged cache (BNSD layout on 910B).
* [kvfuse]  "ATB fused-operator matrix and KV-cache management"
            (agent.csdn.net), section "KVCache management": per-request cache
            [batch, num_heads, seq_len, head_dim]; decode reads the cache,
            computes the new K/V, updates the cache in place, then attends
            over the whole cache.
* [layer]   "ATB: whole decoder-layer fusion" (ai6s.net), section "operator
            fusion graph of a decoder layer": QKV projection as one MatMul,
            then RoPE, then attention, softmax, times V, O projection.

Readings where the pages are silent (the same in the CUDA path):
* RMSNorm: y = x / sqrt(mean(x^2) + eps) * g (g fp32, eps 1e-5).
* RoPE: half-split pairing (element i with i + d/2), angle pos * theta^(-2i/d).
* GQA: query head h uses KV head floor(h / (Hq / Hkv)).
* Attention scale 1/sqrt(d); a query at position p sees cache positions 0..p
  of its own sequence (causal); no bias anywhere (Llama).
* SwiGLU: a = silu(x W_gate^T) * (x W_up^T), silu(z) = z / (1 + e^-z).
* Storage precision ("bf16" mode, the default).  The pages name no precision
  for the intermediates.  Reading: every tensor that feeds a MatMul is BF16
  (the BF16 tensor cores take nothing else): the normalised input, q after
  RoPE, the attention output, the normalised h and the SwiGLU output; k/v
  after RoPE are BF16 because the KV cache holds BF16.  Each is computed
  exactly (float64) and then rounded once to the nearest BF16 (ties to even).
  The residual stream h = x + o W_o^T feeds no MatMul, so it is not rounded
  (it stays float32 on the GPU).  The final y is returned unrounded.  "exact"
  mode rounds nothing (pools then hold float64) and serves the invariant pins.

Two forms of the same layer are implemented: "opbyop" materialises every
intermediate of the unfused chain; "streaming" computes RMSNorm with the
deferred row scale (diag(r) (x*g) W^T), and attention by blockwise online
softmax over the cache pages in block-table order with the context split in
chunks merged through their log-sum-exp.  In exact mode the two agree to
rounding (pinned in tests).

Pools: a K pool and a V pool, each [num_blocks, n_kv_heads, block_size,
head_dim].  A uint16 pool holds BF16 bit patterns; a float64 pool holds exact
values.  block_table[b, j] is the physical block of logical block j of
sequence b (-1 = unused); slot = block * block_size + offset.  A QuantPool holds
INT8 codes with one float32 scale per token and head (see quantize_int8_rows).

Every function here is pinned in tests/test_oracle.py against closed forms, invariants,
library routines or the figures the pages print.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# BF16 as a storage format: rounding and bit patterns
# --------------------------------------------------------------------------

_DROP = np.uint64((1 << 45) - 1)   # float64 keeps 52 mantissa bits, BF16 keeps 7: drop 45
_HALF_M1 = np.uint64((1 << 44) - 1)  # half of the dropped unit, minus one


def bf16_round(x):
    """Nearest BF16 value (ties to even) of float64 data, returned as float64.

    Rounds the float64 bit pattern directly to 7 stored mantissa bits, so there
    is no double rounding through float32.  Valid for the normal range, which
    is all this layer produces; NaN/Inf are not expected.
    """
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    b = a.view(np.uint64)
    lsb = (b >> np.uint64(45)) & np.uint64(1)
    r = (b + _HALF_M1 + lsb) & ~_DROP
    return r.view(np.float64)


def bf16_bits(x):
    """uint16 BF16 bit pattern of float64 values that are already BF16-exact."""
    f32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_value(bits):
    """float64 value of uint16 BF16 bit patterns."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _identity(x):
    return np.asarray(x, dtype=np.float64)


def _rounder(storage: str):
    if storage == "bf16":
        return bf16_round
    if storage == "exact":
        return _identity
    raise ValueError(storage)


# --------------------------------------------------------------------------
# Operators of the chain [chain]
# --------------------------------------------------------------------------

def rmsnorm(x, g, eps):
    """RMSNorm of each row: x / sqrt(mean(x^2) + eps), times the gain g. [chain]"""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rms_scale(x, eps):
    """The per-row factor r = 1/sqrt(mean(x^2)+eps) alone (the streaming form's deferred scale)."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)


def rope(u, pos, theta):
    """Rotary embedding of head vectors u[..., T, heads, d] at positions pos[T].

    Half-split pairing: element i is rotated with element i + d/2 by the angle
    pos * theta^(-2i/d), i < d/2.  [chain] "RotaryEmbedding"; pairing and
    frequencies are this oracle's reading (the page gives neither).
    """
    u = np.asarray(u, dtype=np.float64)
    d = u.shape[-1]
    half = d // 2
    inv_freq = theta ** (-(2.0 * np.arange(half)) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]   # [T, d/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    u1, u2 = u[..., :half], u[..., half:]
    return np.concatenate([u1 * c - u2 * s, u2 * c + u1 * s], axis=-1)


def softmax(s, axis=-1):
    """exp(s - max) / sum exp(s - max) along `axis`; -inf entries get weight 0."""
    s = np.asarray(s, dtype=np.float64)
    m = np.max(s, axis=axis, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=axis, keepdims=True)


def silu(z):
    """silu(z) = z / (1 + e^-z)."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def attention_head(q, K, V, q_pos, k_pos, scale):
    """softmax(q K^T * scale, causal by position) V for one head.

    q [nq, d]; K, V [nk, d]; key j is visible to query i iff k_pos[j] <= q_pos[i].
    [chain] FlashAttention = MatMul -> Softmax -> MatMul.
    """
    s = (np.asarray(q, np.float64) @ np.asarray(K, np.float64).T) * scale
    mask = np.asarray(k_pos)[None, :] > np.asarray(q_pos)[:, None]
    s = np.where(mask, -np.inf, s)
    return softmax(s, axis=-1) @ np.asarray(V, np.float64)


def attention_head_streaming(q, K, V, q_pos, k_pos, scale, chunk, n_splits=1):
    """Same result as attention_head, computed the way a fused kernel does.

    Keys are visited in chunks of `chunk`; each chunk updates a running max m,
    running denominator l and unnormalised output acc (online softmax).  The
    key range is first cut into `n_splits` contiguous parts that are reduced
    independently and merged through their log-sum-exp:
    o = sum_i e^(m_i - M) acc_i / sum_i e^(m_i - M) l_i.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    nq, d = q.shape
    nk = K.shape[0]
    bounds = np.linspace(0, nk, n_splits + 1).round().astype(int)
    parts = []
    for si in range(n_splits):
        m = np.full(nq, -np.inf)
        l = np.zeros(nq)
        acc = np.zeros((nq, V.shape[1]))
        for j0 in range(bounds[si], bounds[si + 1], chunk):
            j1 = min(j0 + chunk, bounds[si + 1])
            s = (q @ K[j0:j1].T) * scale
            s = np.where(np.asarray(k_pos[j0:j1])[None, :] > np.asarray(q_pos)[:, None], -np.inf, s)
            m_new = np.maximum(m, np.max(s, axis=1))
            safe = np.where(np.isfinite(m_new), m_new, 0.0)
            p = np.exp(s - safe[:, None])
            alpha = np.where(np.isfinite(m), np.exp(m - safe), 0.0)
            l = alpha * l + p.sum(axis=1)
            acc = alpha[:, None] * acc + p @ V[j0:j1]
            m = m_new
        parts.append((m, l, acc))
    M = np.max(np.stack([p[0] for p in parts]), axis=0)
    safeM = np.where(np.isfinite(M), M, 0.0)
    num = np.zeros((nq, V.shape[1]))
    den = np.zeros(nq)
    for m, l, acc in parts:
        w = np.where(np.isfinite(m), np.exp(m - safeM), 0.0)
        num += w[:, None] * acc
        den += w * l
    return num / den[:, None]


# --------------------------------------------------------------------------
# Paged KV cache [paging], [kvfuse]
# --------------------------------------------------------------------------

def kv_cache_bytes(n_layers, seq_len, batch, width, elem_bytes):
    """KV-cache size 2 * L * s * b * d * sizeof(dtype) [paging] (d = the K/V row width)."""
    return 2 * n_layers * seq_len * batch * width * elem_bytes


def slot_of(block_table, b, pos, block_size):
    """Cache slot of position `pos` of sequence b: block_table[b, pos // bs] * bs + pos % bs."""
    blk = int(block_table[b][pos // block_size])
    if blk < 0:
        raise IndexError(f"sequence {b} has no block for position {pos}")
    return blk * block_size + pos % block_size


def quantize_int8_rows(x):
    """INT8 codes and float32 scales of the rows of x (last axis) [paging] section
    "KV Cache quantisation": per-token granularity, each token's K (or V) vector
    with its own float32 scale.  Reading (symmetric, absmax): scale = max|x| / 127,
    code = round-half-even(x / scale) clipped to [-127, 127]; a row of zeros has
    scale 0 and codes 0.  The codes are integers decided by floating point, so they
    are computed in float32, the kernel's precision, with IEEE division."""
    xf = np.asarray(x, np.float32)
    amax = np.abs(xf).max(axis=-1)
    scale = (amax / np.float32(127.0)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    codes = np.rint(xf / safe[..., None]).astype(np.float32)
    codes = np.clip(codes, -127, 127)
    codes[scale == 0] = 0
    return codes.astype(np.int8), scale


class QuantPool:
    """An INT8 KV pool: codes int8 [num_blocks, heads, block_size, d] and float32
    scales [num_blocks, heads, block_size] (one per token and head); a row reads
    back as codes * scale."""

    def __init__(self, codes, scales):
        self.codes = codes
        self.scales = scales
        self.shape = codes.shape
        self.dtype = np.int8


def _pool_store(pool, blk, off, vals):
    if isinstance(pool, QuantPool):
        codes, scale = quantize_int8_rows(vals)        # vals [heads, d]: one scale per head
        pool.codes[blk, :, off, :] = codes
        pool.scales[blk, :, off] = scale
    elif pool.dtype == np.uint16:
        pool[blk, :, off, :] = bf16_bits(bf16_round(vals))
    else:
        pool[blk, :, off, :] = vals


def _pool_load(pool, blks, n):
    """Contiguous [heads, n, d] float64 view of the first n positions held in blocks `blks`."""
    bs = pool.shape[2]
    used = [int(bk) for bk in blks[: -(-n // bs)]]
    if isinstance(pool, QuantPool):
        codes = np.concatenate([pool.codes[bk] for bk in used], axis=1)[:, :n, :]
        scales = np.concatenate([pool.scales[bk] for bk in used], axis=1)[:, :n]
        return codes.astype(np.float64) * scales.astype(np.float64)[:, :, None]
    raw = np.concatenate([pool[bk] for bk in used], axis=1)[:, :n, :]
    return bf16_value(raw) if pool.dtype == np.uint16 else np.asarray(raw, np.float64)


def reshape_and_cache(k, v, slot_mapping, k_pool, v_pool):
    """Scatter each token's K/V rows ([T, Hkv, d]) into its pool slot, in place.

    slot_mapping[t] = block * block_size + offset; -1 skips the token.  A K/V
    row of head h lands at pool[block, h, offset, :].  [paging]
    ReshapeAndCacheOperation.  A uint16 pool receives BF16 bit patterns.
    """
    bs = k_pool.shape[2]
    for t, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        blk, off = divmod(int(slot), bs)
        _pool_store(k_pool, blk, off, np.asarray(k[t], np.float64))
        _pool_store(v_pool, blk, off, np.asarray(v[t], np.float64))


def gather_cache(pool, block_table_row, n):
    """The contiguous cache [heads, n, d] of one sequence, read through its block table [kvfuse]."""
    return _pool_load(pool, np.asarray(block_table_row), n)


def paged_attention_decode(q, k_pool, v_pool, block_table, context_lens, scale):
    """Decode attention: for every sequence b the one-row query q[b] ([B, Hq, d])
    attends over positions 0..context_lens[b]-1 of its paged cache.  [chain]
    decode variant.  Returns float64 [B, Hq, d]."""
    q = np.asarray(q, np.float64)
    B, Hq, d = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    out = np.zeros_like(q)
    for b in range(B):
        n = int(context_lens[b])
        K = gather_cache(k_pool, block_table[b], n)
        V = gather_cache(v_pool, block_table[b], n)
        kp = np.arange(n)
        for h in range(Hq):
            out[b, h] = attention_head(q[b, h][None, :], K[h // G], V[h // G], [n - 1], kp, scale)[0]
    return out


# --------------------------------------------------------------------------
# The layer [chain], [layer], [kvfuse]
# --------------------------------------------------------------------------

def layer_forward(dims, W, x, positions, seq_of_token, k_pool, v_pool, block_table,
                  storage="bf16", form="opbyop", attn_chunk=64, attn_splits=1, want=None):
    """One decoder layer over T tokens; updates the pools in place and returns y [T, H].

    dims: object with hidden, n_heads, n_kv_heads, head_dim, intermediate,
      block_size, rms_eps, rope_theta.
    W: dict of float64 (or BF16-exact) arrays: w_qkv [(Hq+2Hkv)d, H] rows
      [Q heads; K heads; V heads], w_o [H, Hq d], w_gate, w_up [I, H],
      w_down [H, I], g_attn, g_ffn [H].
    x [T, H]; positions[T]; seq_of_token[T] (the sequence each token belongs to).
    Every token's K/V is written to the cache at its position first; then each
    query at position p attends over cache positions 0..p of its sequence.
    want: optional dict that receives the intermediates by name: xh, qkv (before RoPE), q, k,
      v (after RoPE; v as cached), o, o_proj (o W_o^T), h, hh, gate, up, a, down (a W_down^T),
      slots.
    """
    rnd = _rounder(storage)
    H, Hq, Hkv, d = dims.hidden, dims.n_heads, dims.n_kv_heads, dims.head_dim
    G = Hq // Hkv
    T = x.shape[0]
    x = np.asarray(x, np.float64)
    positions = np.asarray(positions).astype(np.int64)
    seq_of_token = np.asarray(seq_of_token).astype(np.int64)
    w = {k: np.asarray(v, np.float64) for k, v in W.items()}

    # 1-2. RMSNorm, merged QKV projection
    if form == "opbyop":
        xh = rnd(rmsnorm(x, w["g_attn"], dims.rms_eps))
        qkv = xh @ w["w_qkv"].T
    elif form == "streaming":
        # deferred row scale: rmsnorm(x) W^T = diag(r) ((x * g) W^T)
        r = rms_scale(x, dims.rms_eps)
        xh = rnd((x * w["g_attn"]) * r[:, None])
        qkv = xh @ w["w_qkv"].T if storage == "bf16" else ((x * w["g_attn"]) @ w["w_qkv"].T) * r[:, None]
    else:
        raise ValueError(form)
    q = qkv[:, : Hq * d].reshape(T, Hq, d)
    k = qkv[:, Hq * d: (Hq + Hkv) * d].reshape(T, Hkv, d)
    v = qkv[:, (Hq + Hkv) * d:].reshape(T, Hkv, d)

    # 3. RoPE on q and k
    q = rnd(rope(q, positions, dims.rope_theta))
    k = rnd(rope(k, positions, dims.rope_theta))
    v = rnd(v)

    # 4. ReshapeAndCache: append this call's K/V at their positions
    bs = dims.block_size
    slots = [slot_of(block_table, int(b), int(p), bs) for b, p in zip(seq_of_token, positions)]
    reshape_and_cache(k, v, slots, k_pool, v_pool)

    # 5. attention over the cache, per sequence and query head
    scale = 1.0 / math.sqrt(d)
    o = np.zeros((T, Hq, d))
    for b in np.unique(seq_of_token):
        rows = np.nonzero(seq_of_token == b)[0]
        n = int(positions[rows].max()) + 1
        K = gather_cache(k_pool, block_table[b], n)
        V = gather_cache(v_pool, block_table[b], n)
        kp = np.arange(n)
        qp = positions[rows]
        for h in range(Hq):
            if form == "opbyop":
                o[rows, h] = attention_head(q[rows, h], K[h // G], V[h // G], qp, kp, scale)
            else:
                o[rows, h] = attention_head_streaming(q[rows, h], K[h // G], V[h // G], qp, kp,
                                                      scale, attn_chunk, attn_splits)
    o = rnd(o)

    # 6. O projection + residual (the residual stream is not a MatMul operand: not rounded)
    o_proj = o.reshape(T, Hq * d) @ w["w_o"].T
    h1 = x + o_proj

    # 7-8. RMSNorm, merged gate/up projection, SwiGLU
    if form == "opbyop":
        hh = rnd(rmsnorm(h1, w["g_ffn"], dims.rms_eps))
        gate = hh @ w["w_gate"].T
        up = hh @ w["w_up"].T
    else:
        r2 = rms_scale(h1, dims.rms_eps)
        if storage == "bf16":
            hh = rnd((h1 * w["g_ffn"]) * r2[:, None])
            gate, up = hh @ w["w_gate"].T, hh @ w["w_up"].T
        else:
            hg = h1 * w["g_ffn"]
            gate, up = (hg @ w["w_gate"].T) * r2[:, None], (hg @ w["w_up"].T) * r2[:, None]
    a = rnd(silu(gate) * up)

    # 9. down projection + residual
    down = a @ w["w_down"].T
    y = h1 + down
    if want is not None:
        want.update(xh=xh, qkv=qkv, q=q, k=k, v=v, o=o, o_proj=o_proj, h=h1,
                    hh=hh if form == "opbyop" or storage == "bf16" else None,
                    gate=gate, up=up, a=a, down=down, slots=np.asarray(slots))
    return y


def layer_prefill(dims, W, x, positions, batch, seq_len, k_pool, v_pool, block_table, **kw):
    """Prefill: x holds `batch` sequences of `seq_len` tokens, token-major; token t
    belongs to sequence t // seq_len and sits at positions[t].  [chain] prefill path."""
    seq = np.repeat(np.arange(batch), seq_len)
    return layer_forward(dims, W, x, positions, seq, k_pool, v_pool, block_table, **kw)


def layer_decode_step(dims, W, x, k_pool, v_pool, block_table, context_lens, **kw):
    """Decode: one new token per sequence (x [B, H]); context_lens[b] counts the cache
    including this token, which is appended at position context_lens[b] - 1.  [chain]
    decode path, [paging] contextLens, [kvfuse] read-update-attend."""
    ctx = np.asarray(context_lens).astype(np.int64)
    return layer_forward(dims, W, x, ctx - 1, np.arange(len(ctx)), k_pool, v_pool, block_table, **kw)
