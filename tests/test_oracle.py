"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Each test checks a closed form, an invariant, a library routine, a value the
pages print, or a special case that reduces to a hand-checkable result, so a
plausible slip in the oracle (a dropped term, a wrong sign or index, a
transposed operand) fails at least one of them.
"""
import math
import os
import types

import numpy as np
import pytest
import scipy.special
import torch

from oracle import llama_layer as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def dims(**kw):
    base = dict(hidden=8, n_heads=2, n_kv_heads=1, head_dim=4, intermediate=8, block_size=2,
                rms_eps=0.0, rope_theta=10000.0)
    base.update(kw)
    return types.SimpleNamespace(**base)


# ---------------------------------------------------------------- BF16 storage

def test_bf16_round_matches_torch_rne():
    rng = np.random.default_rng(0)
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(x32.astype(np.float64)), ref)


def test_bf16_round_ties_and_no_double_rounding():
    one = 1.0
    assert O.bf16_round(np.array([one + 2.0 ** -8]))[0] == 1.0               # tie -> even (down)
    assert O.bf16_round(np.array([one + 3 * 2.0 ** -8]))[0] == one + 2.0 ** -6  # tie -> even (up)
    # just above a tie: float32 would first round to the tie, then to even (1.0)
    assert O.bf16_round(np.array([one + 2.0 ** -8 + 2.0 ** -40]))[0] == one + 2.0 ** -7
    assert O.bf16_round(np.array([-(one + 2.0 ** -8 + 2.0 ** -40)]))[0] == -(one + 2.0 ** -7)


def test_bf16_bits_known_patterns():
    vals = np.array([1.0, -2.0, 0.5, 3.0, -1024.0])
    assert O.bf16_bits(vals).tolist() == [0x3F80, 0xC000, 0x3F00, 0x4040, 0xC480]
    np.testing.assert_array_equal(O.bf16_value(O.bf16_bits(vals)), vals)


# ---------------------------------------------------------------- RMSNorm

def test_rmsnorm_hand_case_and_unit_rms():
    x = np.array([[3.0, 4.0]])                 # mean(x^2) = 12.5
    y = O.rmsnorm(x, np.ones(2), 0.0)
    np.testing.assert_allclose(y, x / math.sqrt(12.5), rtol=0, atol=1e-15)
    eps = 0.5
    y = O.rmsnorm(x, np.ones(2), eps)
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2)), math.sqrt(12.5 / (12.5 + eps)), rtol=1e-15)
    g = np.array([2.0, -1.0])
    np.testing.assert_allclose(O.rmsnorm(x, g, 0.0), x / math.sqrt(12.5) * g, rtol=1e-15)


def test_rmsnorm_unit_rms_random_and_scale_invariant():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 64)) * 7
    y = O.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.rmsnorm(3.5 * x, np.ones(64), 0.0), y, rtol=1e-13)
    np.testing.assert_allclose(O.rms_scale(x, 1e-5), 1 / np.sqrt(np.mean(x * x, 1) + 1e-5), rtol=1e-15)


# ---------------------------------------------------------------- RoPE

def test_rope_pairing_and_frequencies_by_hand():
    d = 4
    e0 = np.zeros((1, 1, d)); e0[0, 0, 0] = 1.0
    e1 = np.zeros((1, 1, d)); e1[0, 0, 1] = 1.0
    r0 = O.rope(e0, np.array([1]), 10000.0)[0, 0]
    np.testing.assert_allclose(r0, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    r1 = O.rope(e1, np.array([1]), 10000.0)[0, 0]          # theta^(-2/4) = 0.01
    np.testing.assert_allclose(r1, [0, math.cos(0.01), 0, math.sin(0.01)], atol=1e-15)
    e2 = np.zeros((1, 1, d)); e2[0, 0, 2] = 1.0             # second half rotates the other way
    np.testing.assert_allclose(O.rope(e2, np.array([1]), 10000.0)[0, 0],
                               [-math.sin(1), 0, math.cos(1), 0], atol=1e-15)


def test_rope_norm_identity_and_relative_position():
    rng = np.random.default_rng(2)
    u = rng.standard_normal((6, 3, 128))
    pos = np.array([0, 1, 17, 511, 4095, 32767])
    r = O.rope(u, pos, 10000.0)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(u, axis=-1), rtol=1e-13)
    np.testing.assert_array_equal(r[0], u[0])                # position 0 is the identity
    q = rng.standard_normal((1, 1, 64)); k = rng.standard_normal((1, 1, 64))
    dots = []
    for p1, p2 in [(5, 2), (103, 100), (40003, 40000)]:
        dots.append(float(np.sum(O.rope(q, np.array([p1]), 1e4) * O.rope(k, np.array([p2]), 1e4))))
    np.testing.assert_allclose(dots, dots[0], rtol=1e-9)


# ---------------------------------------------------------------- softmax / attention

def test_softmax_rows_sum_to_one_and_match_scipy():
    rng = np.random.default_rng(3)
    s = rng.standard_normal((7, 33)) * 10
    p = O.softmax(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    np.testing.assert_allclose(p, scipy.special.softmax(s, axis=1), rtol=1e-13, atol=1e-300)
    assert O.softmax(np.array([[0.0, -np.inf]]))[0, 1] == 0.0
    np.testing.assert_allclose(O.silu(np.array([0.0, 1.0, -2.0])),
                               [0.0, 1 / (1 + math.exp(-1)), -2 / (1 + math.exp(2))], rtol=1e-15)


def test_attention_closed_forms():
    rng = np.random.default_rng(4)
    d = 16
    q = rng.standard_normal((1, d))
    K = rng.standard_normal((1, d)); V = rng.standard_normal((1, d))
    np.testing.assert_allclose(O.attention_head(q, K, V, [0], [0], 0.25), V, rtol=1e-15)
    K = np.repeat(rng.standard_normal((1, d)), 5, axis=0); V = rng.standard_normal((5, d))
    np.testing.assert_allclose(O.attention_head(q, K, V, [9], np.arange(5), 0.25),
                               V.mean(axis=0, keepdims=True), rtol=1e-13)
    # two keys: weight of key 0 is the logistic of the score difference
    K = rng.standard_normal((2, d)); V = rng.standard_normal((2, d))
    s = (q @ K.T)[0] * 0.3
    w0 = 1 / (1 + math.exp(s[1] - s[0]))
    np.testing.assert_allclose(O.attention_head(q, K, V, [1], [0, 1], 0.3)[0],
                               w0 * V[0] + (1 - w0) * V[1], rtol=1e-13)
    # causal: a query at position 0 sees only key 0
    np.testing.assert_allclose(O.attention_head(q, K, V, [0], [0, 1], 0.3)[0], V[0], rtol=1e-15)


@pytest.mark.parametrize("chunk,splits", [(1, 1), (16, 1), (7, 3), (64, 5), (1000, 2)])
def test_streaming_attention_equals_direct(chunk, splits):
    rng = np.random.default_rng(5)
    nq, nk, d = 9, 70, 32
    q = rng.standard_normal((nq, d)) * 3
    K = rng.standard_normal((nk, d)); V = rng.standard_normal((nk, d))
    qp = np.array([0, 5, 6, 30, 31, 50, 60, 68, 69]); kp = np.arange(nk)
    ref = O.attention_head(q, K, V, qp, kp, 1 / math.sqrt(d))
    got = O.attention_head_streaming(q, K, V, qp, kp, 1 / math.sqrt(d), chunk, splits)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- paged cache

def test_kv_cache_size_formula_matches_printed_examples():
    with open(os.path.join(GOLDEN, "kv_cache_sizes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert rows
    for L, s, b, d, e, gb, tol in rows:
        got = O.kv_cache_bytes(int(L), int(s), int(b), int(d), int(e)) / 1e9
        assert abs(got - float(gb)) < float(tol), (got, gb)
    assert O.kv_cache_bytes(80, 4096, 4, 8192, 2) == 4 * O.kv_cache_bytes(80, 4096, 1, 8192, 2)
    assert O.kv_cache_bytes(80, 32768, 1, 8192, 2) == 8 * O.kv_cache_bytes(80, 4096, 1, 8192, 2)
    # GQA: the cache holds n_kv_heads * head_dim per token, 8x less for 8 of 64 heads
    assert O.kv_cache_bytes(80, 4096, 1, 8 * 128, 2) * 8 == O.kv_cache_bytes(80, 4096, 1, 8192, 2)


def test_reshape_and_cache_is_an_exact_placement():
    rng = np.random.default_rng(6)
    nb, Hkv, bs, d, T = 6, 2, 4, 8, 10
    kp = np.full((nb, Hkv, bs, d), 0xC480, np.uint16)    # BF16 -1024 sentinel
    vp = kp.copy()
    k = O.bf16_round(rng.standard_normal((T, Hkv, d))); v = O.bf16_round(rng.standard_normal((T, Hkv, d)))
    slots = rng.permutation(nb * bs)[:T]
    slots[3] = -1
    O.reshape_and_cache(k, v, slots, kp, vp)
    written = set()
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), bs)
        written.add((blk, off))
        np.testing.assert_array_equal(O.bf16_value(kp[blk, :, off, :]), k[t])
        np.testing.assert_array_equal(O.bf16_value(vp[blk, :, off, :]), v[t])
    for blk in range(nb):
        for off in range(bs):
            if (blk, off) not in written:
                assert (kp[blk, :, off, :] == 0xC480).all() and (vp[blk, :, off, :] == 0xC480).all()
    assert len(written) == T - 1


def test_shuffled_block_table_equals_contiguous_cache():
    rng = np.random.default_rng(7)
    B, Hq, Hkv, d, bs = 3, 4, 2, 16, 4
    ctx = np.array([1, 9, 12])
    nblk = [-(-c // bs) for c in ctx]
    total = sum(nblk)
    Kc = [rng.standard_normal((Hkv, c, d)) for c in ctx]
    Vc = [rng.standard_normal((Hkv, c, d)) for c in ctx]
    q = rng.standard_normal((B, Hq, d))

    def build(perm):
        kp = np.zeros((total, Hkv, bs, d)); vp = np.zeros_like(kp)
        table = -np.ones((B, max(nblk)), np.int64)
        at = 0
        for b in range(B):
            table[b, :nblk[b]] = perm[at:at + nblk[b]]
            for p in range(ctx[b]):
                blk = table[b, p // bs]
                kp[blk, :, p % bs] = Kc[b][:, p]; vp[blk, :, p % bs] = Vc[b][:, p]
            at += nblk[b]
        return O.paged_attention_decode(q, kp, vp, table, ctx, 1 / math.sqrt(d))

    a = build(np.arange(total))
    b = build(rng.permutation(total))
    np.testing.assert_array_equal(a, b)
    for bi in range(B):      # and each equals attention over the contiguous cache
        for h in range(Hq):
            ref = O.attention_head(q[bi, h][None], Kc[bi][h // 2], Vc[bi][h // 2], [ctx[bi] - 1],
                                   np.arange(ctx[bi]), 1 / math.sqrt(d))[0]
            np.testing.assert_allclose(a[bi, h], ref, rtol=1e-14)


# ---------------------------------------------------------------- whole layer

def _rand_layer(dm, seed, w_std=0.3):
    rng = np.random.default_rng(seed)
    H, I, Hq, Hkv, d = dm.hidden, dm.intermediate, dm.n_heads, dm.n_kv_heads, dm.head_dim
    W = dict(w_qkv=rng.standard_normal(((Hq + 2 * Hkv) * d, H)) * w_std,
             w_o=rng.standard_normal((H, Hq * d)) * w_std,
             w_gate=rng.standard_normal((I, H)) * w_std, w_up=rng.standard_normal((I, H)) * w_std,
             w_down=rng.standard_normal((H, I)) * w_std,
             g_attn=1 + 0.1 * rng.standard_normal(H), g_ffn=1 + 0.1 * rng.standard_normal(H))
    return W, rng


def _pools(dm, nb, exact=True):
    shape = (nb, dm.n_kv_heads, dm.block_size, dm.head_dim)
    if exact:
        return np.zeros(shape), np.zeros(shape)
    return np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)


def test_layer_residual_and_o_projection_orientation():
    # H = Hq*d = 8, one token at position 0: attention returns v; W_o is a cyclic shift,
    # gate/up are zero so the FFN adds nothing: y_i = x_i + o_{(i+1) mod 8}.
    dm = dims()
    H = 8
    x = np.array([[1.0, -2.0, 3.0, 0.5, -1.5, 2.5, 0.25, -0.75]])
    W = dict(w_qkv=np.zeros((16, H)), w_o=np.zeros((H, H)), w_gate=np.zeros((8, H)),
             w_up=np.zeros((8, H)), w_down=np.ones((H, 8)), g_attn=np.ones(H), g_ffn=np.ones(H))
    W["w_qkv"][12:16, 0:4] = np.eye(4)       # V head (rows after 2 Q heads + 1 K head) = x_hat[0:4]
    for i in range(H):
        W["w_o"][i, (i + 1) % H] = 1.0
    kp, vp = _pools(dm, 2)
    y = O.layer_prefill(dm, W, x, [0], 1, 1, kp, vp, np.array([[1, 0]]), storage="exact")
    xh = x[0] / math.sqrt(np.mean(x[0] ** 2))
    o = np.concatenate([xh[:4], xh[:4]])     # both query heads read KV head 0
    np.testing.assert_allclose(y[0], x[0] + np.roll(o, -1), rtol=1e-14, atol=1e-15)
    # the token's K/V landed at block_table[0][0] = physical block 1, offset 0
    np.testing.assert_allclose(vp[1, 0, 0], xh[:4], rtol=1e-15)


def test_layer_swiglu_and_down_by_hand():
    dm = dims()
    H = 8
    rng = np.random.default_rng(8)
    x = rng.standard_normal((1, H))
    W = dict(w_qkv=np.zeros((16, H)), w_o=np.zeros((H, H)), w_gate=np.eye(8) * 2.0,
             w_up=np.eye(8)[::-1].copy(), w_down=np.zeros((H, 8)), g_attn=np.ones(H), g_ffn=np.ones(H))
    for i in range(H):
        W["w_down"][i, (3 * i) % 8] = 1.0
    kp, vp = _pools(dm, 2)
    y = O.layer_prefill(dm, W, x, [0], 1, 1, kp, vp, np.array([[0, 1]]), storage="exact")
    hh = x[0] / math.sqrt(np.mean(x[0] ** 2))
    a = [2 * hh[j] / (1 + math.exp(-2 * hh[j])) * hh[7 - j] for j in range(8)]
    want = [x[0, i] + a[(3 * i) % 8] for i in range(8)]
    np.testing.assert_allclose(y[0], want, rtol=1e-13)


def test_layer_gqa_grouping_is_consecutive():
    dm = dims(hidden=8, n_heads=4, n_kv_heads=2, head_dim=2)
    H = 8
    x = np.ones((1, H))
    W = dict(w_qkv=np.zeros(((4 + 4) * 2, H)), w_o=np.eye(H), w_gate=np.zeros((8, H)),
             w_up=np.zeros((8, H)), w_down=np.zeros((H, 8)), g_attn=np.ones(H), g_ffn=np.ones(H))
    W["w_qkv"][12:14, :] = 1.0 / 8      # V of KV head 0: both elements = mean(x_hat) = 1
    W["w_qkv"][14:16, :] = 2.0 / 8      # V of KV head 1: 2
    kp, vp = _pools(dm, 1)
    y = O.layer_prefill(dm, W, x, [0], 1, 1, kp, vp, np.array([[0]]), storage="exact")
    np.testing.assert_allclose(y[0] - 1.0, [1, 1, 1, 1, 2, 2, 2, 2], rtol=1e-14)


def test_layer_causality_and_v_not_rotated():
    dm = dims(hidden=16, n_heads=2, n_kv_heads=2, head_dim=8, intermediate=24, block_size=4)
    W, rng = _rand_layer(dm, 9)
    x = rng.standard_normal((3, 16))
    ys = []
    for theta in (10000.0, 123.0):
        kp, vp = _pools(dm, 2)
        d2 = dims(**{**vars(dm), "rope_theta": theta})
        ys.append(O.layer_prefill(d2, W, x[:1], [0], 1, 1, kp, vp, np.array([[1, 0]]), storage="exact"))
    np.testing.assert_array_equal(ys[0], ys[1])     # single token: RoPE cannot reach v
    # the first token's output does not depend on later tokens
    kp, vp = _pools(dm, 2)
    y3 = O.layer_prefill(dm, W, x, [0, 1, 2], 1, 3, kp, vp, np.array([[1, 0]]), storage="exact")
    np.testing.assert_allclose(y3[0], ys[0][0], rtol=1e-13)
    kp, vp = _pools(dm, 2)
    d2 = dims(**{**vars(dm), "rope_theta": 123.0})
    y3b = O.layer_prefill(d2, W, x, [0, 1, 2], 1, 3, kp, vp, np.array([[1, 0]]), storage="exact")
    assert np.abs(y3b[2] - y3[2]).max() > 1e-6      # ... but later tokens do see RoPE


def test_layer_relative_position_invariance():
    dm = dims(hidden=16, n_heads=4, n_kv_heads=2, head_dim=4, intermediate=20, block_size=4)
    W, rng = _rand_layer(dm, 10)
    x = rng.standard_normal((5, 16))
    # the same 5 tokens at positions 0..4 and (after 3 other cache entries) 3..7: with
    # zero V/K for the earlier entries it differs, so instead compare positions 0..4
    # against a copy whose block table is shifted -- placement must not matter.
    kp, vp = _pools(dm, 4)
    a = O.layer_prefill(dm, W, x, np.arange(5), 1, 5, kp, vp, np.array([[0, 1]]), storage="exact")
    kp, vp = _pools(dm, 4)
    b = O.layer_prefill(dm, W, x, np.arange(5), 1, 5, kp, vp, np.array([[3, 2]]), storage="exact")
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("splits", [1, 3])
def test_layer_opbyop_equals_streaming(splits):
    dm = dims(hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=40, block_size=4,
              rms_eps=1e-5)
    W, rng = _rand_layer(dm, 11)
    x = rng.standard_normal((2 * 11, 32))
    table = np.array([[5, 0, 2], [1, 4, 3]])
    outs = []
    for form in ("opbyop", "streaming"):
        kp, vp = _pools(dm, 6)
        outs.append(O.layer_prefill(dm, W, x, np.tile(np.arange(11), 2), 2, 11, kp, vp, table,
                                    storage="exact", form=form, attn_chunk=3, attn_splits=splits))
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-12, atol=1e-12)


def test_decode_after_prefill_equals_longer_prefill():
    dm = dims(hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=40, block_size=4,
              rms_eps=1e-5)
    W, rng = _rand_layer(dm, 12)
    S = 9
    x = rng.standard_normal((S + 1, 32))
    table = np.array([[2, 0, 1]])
    kp, vp = _pools(dm, 3)
    O.layer_prefill(dm, W, x[:S], np.arange(S), 1, S, kp, vp, table, storage="exact")
    y_dec = O.layer_decode_step(dm, W, x[S:], kp, vp, table, [S + 1], storage="exact")
    kp2, vp2 = _pools(dm, 3)
    y_full = O.layer_prefill(dm, W, x, np.arange(S + 1), 1, S + 1, kp2, vp2, table, storage="exact")
    np.testing.assert_allclose(y_dec[0], y_full[S], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(kp, kp2, rtol=1e-13, atol=1e-15)


def test_bf16_storage_mode_rounds_the_cache():
    dm = dims(hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=40, block_size=4,
              rms_eps=1e-5)
    W, rng = _rand_layer(dm, 13)
    x = O.bf16_round(rng.standard_normal((6, 32)))
    kp, vp = _pools(dm, 2, exact=False)
    want = {}
    y = O.layer_prefill(dm, W, x, np.arange(6), 1, 6, kp, vp, np.array([[1, 0]]), want=want)
    kpe, vpe = _pools(dm, 2)
    ye = O.layer_prefill(dm, W, x, np.arange(6), 1, 6, kpe, vpe, np.array([[1, 0]]), storage="exact")
    np.testing.assert_array_equal(O.bf16_value(kp[1, :, 0]), want["k"][0])
    np.testing.assert_allclose(O.bf16_value(kp), kpe, rtol=0.02, atol=0.02)
    np.testing.assert_allclose(y, ye, rtol=0.02, atol=0.02 * np.abs(ye).max())


def _on_bf16_grid(a):
    """Elementwise: is the value a BF16 number (round-tripping through torch's BF16 keeps it)?"""
    a = np.asarray(a, np.float64)
    back = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    return back == a


@pytest.mark.parametrize("mode", ["prefill", "decode"])
def test_bf16_storage_mode_rounding_points(mode):
    """Which intermediates the BF16 storage mode rounds, pinned by value: every MatMul
    operand (x_hat, q, k, v, o, h_hat, a) comes back as BF16 numbers, the float32 residual
    stream h and the output y do not (their exact values are off the BF16 grid), and each
    rounded stage is the nearest BF16 of the exact stage value computed from the stage
    before it (so no tensor is rounded twice, or rounded and then moved).  Adding or
    dropping one rounding in the layer fails here."""
    dm = dims(hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, intermediate=40, block_size=4, rms_eps=1e-5)
    W, rng = _rand_layer(dm, 15)
    W = {k: (O.bf16_round(v) if k.startswith("w_") else v) for k, v in W.items()}
    x = O.bf16_round(rng.standard_normal((7, 32)))
    table = np.array([[1, 0]])
    kp, vp = _pools(dm, 2, exact=False)
    want = {}
    if mode == "prefill":
        y = O.layer_prefill(dm, W, x, np.arange(7), 1, 7, kp, vp, table, want=want)
    else:
        O.layer_prefill(dm, W, x[:6], np.arange(6), 1, 6, kp, vp, table)
        y = O.layer_decode_step(dm, W, x[6:], kp, vp, table, [7], want=want)
    for name in ("xh", "q", "k", "v", "o", "hh", "a"):
        assert _on_bf16_grid(want[name]).all(), f"{name} is not a BF16 tensor"
    for name, t in (("h", want["h"]), ("y", y)):
        assert _on_bf16_grid(t).mean() < 0.2, f"{name} looks rounded to BF16"
    # each rounded stage against torch's BF16 rounding of the exact value from the stage before
    nearest = lambda t: torch.from_numpy(np.ascontiguousarray(t, np.float64)).to(torch.bfloat16).double().numpy()
    T = want["xh"].shape[0]
    xr = x[6:] if mode == "decode" else x
    ms = np.mean(xr * xr, axis=1, keepdims=True)
    np.testing.assert_array_equal(want["xh"], nearest(xr / np.sqrt(ms + dm.rms_eps) * W["g_attn"]))
    qkv = want["xh"] @ W["w_qkv"].T
    np.testing.assert_array_equal(want["v"], nearest(qkv[:, 48:].reshape(T, 2, 8)))
    h = xr + want["o"].reshape(T, -1) @ W["w_o"].T
    np.testing.assert_array_equal(want["h"], h)
    ms2 = np.mean(h * h, axis=1, keepdims=True)
    np.testing.assert_array_equal(want["hh"], nearest(h / np.sqrt(ms2 + dm.rms_eps) * W["g_ffn"]))
    g, u = want["hh"] @ W["w_gate"].T, want["hh"] @ W["w_up"].T
    np.testing.assert_array_equal(want["a"], nearest(g / (1 + np.exp(-g)) * u))
    np.testing.assert_array_equal(y, h + want["a"] @ W["w_down"].T)


def test_layer_two_token_attention_by_hand():
    # H = Hq*d = 8 (2 heads of d=4, one KV head), W_o = I, FFN zero: y = x + o.  Token 1
    # (position 1) attends to keys 0 and 1 with weight logistic(s0 - s1) on key 0, where
    # s_j = <rope(q_1, 1), rope(k_j, j)> / sqrt(d).
    dm = dims()
    H, d = 8, 4
    rng = np.random.default_rng(14)
    x = rng.standard_normal((2, H))
    W = dict(w_qkv=rng.standard_normal((16, H)) * 0.5, w_o=np.eye(H), w_gate=np.zeros((8, H)),
             w_up=np.zeros((8, H)), w_down=np.zeros((H, 8)), g_attn=np.ones(H), g_ffn=np.ones(H))
    kp, vp = _pools(dm, 2)
    y = O.layer_prefill(dm, W, x, [0, 1], 1, 2, kp, vp, np.array([[0, 1]]), storage="exact")
    xh = x / np.sqrt(np.mean(x ** 2, axis=1, keepdims=True))
    qkv = xh @ W["w_qkv"].T
    k = [O.rope(qkv[j, 8:12].reshape(1, 1, d), np.array([j]), 1e4)[0, 0] for j in range(2)]
    v = [qkv[j, 12:16] for j in range(2)]
    o = []
    for h in range(2):
        qh = O.rope(qkv[1, 4 * h:4 * h + 4].reshape(1, 1, d), np.array([1]), 1e4)[0, 0]
        s0, s1 = qh @ k[0] / 2.0, qh @ k[1] / 2.0
        w0 = 1 / (1 + math.exp(s1 - s0))
        o.append(w0 * v[0] + (1 - w0) * v[1])
    np.testing.assert_allclose(y[1], x[1] + np.concatenate(o), rtol=1e-13)
    np.testing.assert_allclose(y[0], x[0] + np.concatenate([v[0], v[0]]), rtol=1e-13)


# ---------------------------------------------------------------- INT8 KV cache

def test_int8_quantizer_is_a_uniform_quantizer_within_half_a_step():
    rng = np.random.default_rng(5)
    x = (rng.normal(size=(64, 128)) * rng.uniform(0.01, 20, size=(64, 1))).astype(np.float32)
    codes, scale = O.quantize_int8_rows(x)
    assert codes.dtype == np.int8 and scale.dtype == np.float32
    assert codes.min() >= -127 and codes.max() <= 127
    # textbook round-to-nearest bound: every value within half a step of its code
    err = np.abs(x.astype(np.float64) - codes.astype(np.float64) * scale[:, None])
    assert (err <= 0.5 * scale[:, None].astype(np.float64) * (1 + 1e-6)).all()
    # the largest magnitude of each row sits on the end of the code range, with its sign
    i = np.abs(x).argmax(axis=1)
    assert (codes[np.arange(64), i] == np.sign(x[np.arange(64), i]) * 127).all()
    # a step is max|x| / 127
    np.testing.assert_allclose(scale, np.abs(x).max(axis=1) / 127, rtol=1e-7)


def test_int8_quantizer_zero_row_and_exact_grid():
    codes, scale = O.quantize_int8_rows(np.zeros((2, 16), np.float32))
    assert scale.tolist() == [0.0, 0.0] and not codes.any()
    # values already on the grid k * 2^-3 with max 127 * 2^-3 come back exactly
    k = np.arange(-127, 129, 16)[:16].astype(np.float32)
    k[0] = -127
    codes, scale = O.quantize_int8_rows((k * 0.125)[None, :])
    assert scale[0] == np.float32(0.125) and (codes[0] == k).all()


def test_int8_paged_attention_reduces_to_exact_attention_on_grid_values():
    """K/V rows that are integers times a power of two (with a max of 127 steps) quantize
    losslessly, so attention through an INT8 pool equals attention through an exact pool."""
    rng = np.random.default_rng(9)
    nb, Hkv, bs, d, B, Hq = 6, 2, 4, 8, 2, 4
    step = 2.0 ** rng.integers(-6, -2, size=(nb, Hkv, bs))
    ints = rng.integers(-126, 127, size=(nb, Hkv, bs, d)).astype(np.float64)
    ints[..., 0] = 127                              # every row's max is exactly 127 steps
    vals = ints * step[..., None]
    exact_k, exact_v = vals.copy(), vals[::-1].copy()
    qk = O.QuantPool(np.zeros((nb, Hkv, bs, d), np.int8), np.zeros((nb, Hkv, bs), np.float32))
    qv = O.QuantPool(np.zeros((nb, Hkv, bs, d), np.int8), np.zeros((nb, Hkv, bs), np.float32))
    slots = np.arange(nb * bs)
    O.reshape_and_cache(exact_k.transpose(0, 2, 1, 3).reshape(-1, Hkv, d),
                        exact_v.transpose(0, 2, 1, 3).reshape(-1, Hkv, d), slots, qk, qv)
    table = np.array([[3, 0, 5], [1, 4, 2]])
    ctx = np.array([11, 9])
    q = rng.normal(size=(B, Hq, d))
    got = O.paged_attention_decode(q, qk, qv, table, ctx, 0.35)
    ref = O.paged_attention_decode(q, exact_k, exact_v, table, ctx, 0.35)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # and off the grid the cached rows read back within half a step
    x = rng.normal(size=(5, Hkv, d))
    O.reshape_and_cache(x, x, [0, 1, 2, 3, 4], qk, qv)
    back = O.gather_cache(qk, [0, 1, 2], 5).transpose(1, 0, 2)
    codes, scale = O.quantize_int8_rows(x)
    assert (np.abs(back - x) <= 0.5 * scale[..., None] * (1 + 1e-6) + 1e-7).all()
