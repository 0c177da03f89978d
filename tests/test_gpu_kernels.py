"""GPU parity of each C-ABI entry point against the CPU oracle, on small and
ragged shapes that still span several tiles."""
import math

import numpy as np
import pytest
import torch

from oracle import llama_layer as O
from tests.helpers import assert_close, bits, f64
from transformer_decoder_layer_llama_gb300 import synth

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from transformer_decoder_layer_llama_gb300 import api
DEV = "cuda"


# ---------------------------------------------------------------- Linear (the tensor-core GEMM)

@pytest.mark.parametrize("m,n,k", [
    (1, 128, 64), (2, 512, 256), (16, 1376, 688), (64, 4096, 4096), (33, 11008, 4096),
    (64, 4096, 11008),                                   # weight form, split K
    (64, 128, 4096), (48, 256, 8192),                    # 16-32 CTAs share one tile
    (200, 1376, 688), (256, 4096, 4096),                 # weight form up to 256 tokens
    (129, 12288, 512),                                   # weight form, wide output
    (232, 12288, 512),                                   # few tokens, wide output: CTA pairs, ragged
    (65, 256, 128), (128, 512, 256), (300, 1376, 688), (2048, 4096, 4096), (257, 12288, 4096),
    (5, 12304, 512), (16, 38912, 256),                   # weight form, several tiles per CTA: split, whole
    (16, 40144, 256), (3, 24400, 320),                   # ... a ragged last tile (80 and 80 rows)
    (520, 2048, 1040), (257, 640, 80),                   # CTA pairs: 17 K blocks (a half last stage), a ragged K block
])
def test_linear_matches_float64_matmul(m, n, k):
    x = synth.normal_bf16((m, k), 1.0, seed=m * 7 + 1, tag="x")
    w = synth.normal_bf16((n, k), 0.02, seed=n * 3 + k, tag="w")
    y = api.linear(x.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    ref = f64(x) @ f64(w).T
    # BF16 output rounding (2^-9 relative) plus float32 accumulation order
    assert_close(f64(y), ref, f"linear {m}x{n}x{k}", atol=2e-3, rtol=8e-3)


def test_linear_twice_same_buffers_is_repeatable():
    x = synth.normal_bf16((64, 4096), 1.0, seed=1, tag="x").to(DEV)
    w = synth.normal_bf16((4096, 4096), 0.02, seed=2, tag="w").to(DEV)
    ws = torch.empty(api.lib.ll_linear_workspace_size(64, 4096, 4096), dtype=torch.uint8, device=DEV)
    y1 = api.linear(x, w, workspace=ws)
    y2 = api.linear(x, w, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


# ---------------------------------------------------------------- ReshapeAndCache

@pytest.mark.parametrize("T,Hkv,d,bs,nb", [(37, 2, 64, 16, 8), (300, 8, 128, 128, 5), (1, 32, 128, 128, 2)])
def test_reshape_and_cache_bit_exact(T, Hkv, d, bs, nb):
    dims = synth.LayerDims(Hkv * d, Hkv, Hkv, d, 64, bs)
    k = synth.normal_bf16((T, Hkv, d), 1.0, seed=T, tag="k")
    v = synth.normal_bf16((T, Hkv, d), 1.0, seed=T, tag="v")
    slots = synth.make_slot_mapping(T, nb * bs, seed=T + 3, n_skip=min(3, T - 1))
    kp, vp = synth.make_pool(nb, dims, 0, fill="sentinel")
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    st = api.reshape_and_cache(k.to(DEV), v.to(DEV), slots.to(DEV), kpd, vpd)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ko, vo = bits(kp), bits(vp)
    O.reshape_and_cache(f64(k), f64(v), slots.numpy(), ko, vo)
    np.testing.assert_array_equal(bits(kpd), ko)
    np.testing.assert_array_equal(bits(vpd), vo)


def test_reshape_and_cache_flags_out_of_range_slot():
    dims = synth.LayerDims(128, 2, 2, 64, 64, 16)
    k = synth.normal_bf16((4, 2, 64), 1.0, seed=1)
    slots = torch.tensor([0, 5, 10_000, -1], dtype=torch.int32)
    kp, vp = synth.make_pool(4, dims, 0, fill="sentinel")
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    st = api.reshape_and_cache(k.to(DEV), k.to(DEV), slots.to(DEV), kpd, vpd)
    torch.cuda.synchronize()
    assert int(st.item()) == api.LL_DEV_BAD_SLOT
    ko, vo = bits(kp), bits(vp)
    O.reshape_and_cache(f64(k), f64(k), [0, 5, -1, -1], ko, vo)   # the bad one is skipped
    np.testing.assert_array_equal(bits(kpd), ko)


# ---------------------------------------------------------------- paged decode attention

@pytest.mark.parametrize("B,Hq,Hkv,d,bs,ctx_lo,ctx_hi", [
    (2, 4, 2, 64, 16, 1, 80),           # tiny GQA layer shape
    (5, 8, 8, 128, 128, 1, 300),        # MHA, ragged
    (3, 16, 2, 128, 128, 900, 3100),    # GQA 8, several 1024-key splits
    (4, 4, 4, 64, 32, 1023, 1026),      # split boundaries
    (2, 16, 1, 128, 128, 1, 700),       # GQA 16, one KV head
])
def test_paged_attention_decode(B, Hq, Hkv, d, bs, ctx_lo, ctx_hi):
    dims = synth.LayerDims(Hq * d, Hq, Hkv, d, 64, bs)
    ctx = synth.make_context_lens(B, ctx_lo, ctx_hi, seed=B * 11)
    ctx[0] = ctx_lo
    table, nb = synth.make_block_table(ctx.tolist(), bs, seed=B * 13, extra_blocks=3)
    kp, vp = synth.make_pool(nb, dims, seed=B * 17)
    q = synth.normal_bf16((B, Hq, d), 1.0, seed=B, tag="q")
    scale = 1 / math.sqrt(d)
    out = api.paged_attention_decode(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), ctx.to(DEV), scale)
    torch.cuda.synchronize()
    ref = O.paged_attention_decode(f64(q), bits(kp), bits(vp), table.numpy(), ctx.numpy(), scale)
    assert_close(f64(out), ref, "paged_attention_decode")


@pytest.mark.parametrize("B,Hq,Hkv,d,bs,ctx_hi", [
    (40, 8, 2, 64, 16, 3100),           # full splits first, then the partial ones by length
    (520, 2, 1, 64, 32, 60),            # beyond the sorted batch: partial splits in sequence order
])
def test_paged_attention_decode_dispatch_order(B, Hq, Hkv, d, bs, ctx_hi):
    """Many sequences with contexts on, next to and away from the 1024-key split
    boundaries, empty ones (their output rows are zero) and two of 9 splits (long enough
    for the split grid to run in its dispatch order)."""
    dims = synth.LayerDims(Hq * d, Hq, Hkv, d, 64, bs)
    ctx = synth.make_context_lens(B, 1, ctx_hi, seed=B * 31)
    ctx[:9] = torch.tensor([0, 1024, 2048, 1023, 1025, 0, 1, 8200, 9216], dtype=torch.int32)
    table, nb = synth.make_block_table(ctx.tolist(), bs, seed=B * 37, extra_blocks=3)
    kp, vp = synth.make_pool(nb, dims, seed=B * 41)
    q = synth.normal_bf16((B, Hq, d), 1.0, seed=B + 3, tag="q")
    scale = 1 / math.sqrt(d)
    status = api.new_status()
    out = api.paged_attention_decode(q.to(DEV), kp.to(DEV), vp.to(DEV), table.to(DEV), ctx.to(DEV), scale,
                                     status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = f64(out)
    live = ctx.numpy() > 0
    assert (got[~live] == 0).all()
    ref = O.paged_attention_decode(f64(q)[live], bits(kp), bits(vp), table.numpy()[live], ctx.numpy()[live], scale)
    assert_close(got[live], ref, "paged_attention_decode, many sequences")


# ---------------------------------------------------------------- whole layer, tiny GQA workload

def _tiny_setup(seed=1, S=None, B=None, steps=8):
    wl = synth.WORKLOADS["tiny_gqa"]
    d = wl.dims
    B = B or wl.batch
    S = S or wl.prefill_len
    W = synth.make_weights(d, wl.w_std, seed=seed)
    table, nb = synth.make_block_table([S + steps] * B, d.block_size, seed=seed + 3, extra_blocks=3)
    kp, vp = synth.make_pool(nb, d, seed=seed + 4, fill="sentinel")
    cfg = api.make_config(d, max_position=S + steps + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    Wn = {k: f64(v) for k, v in W.items()}
    return wl, d, B, S, W, Wn, table, kp, vp, cfg, packed


def test_tiny_layer_prefill_then_decode_steps():
    wl, d, B, S, W, Wn, table, kp, vp, cfg, packed = _tiny_setup()
    x = synth.make_x(B * S, d.hidden, seed=21)
    pos = synth.prefill_positions(B, S)
    kpd, vpd, td = kp.to(DEV), vp.to(DEV), table.to(DEV)
    status = api.new_status()
    y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kpd, vpd, td, status=status)
    torch.cuda.synchronize()
    ko, vo = bits(kp), bits(vp)
    want = {}
    y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy(), want=want)
    assert int(status.item()) == 0
    assert_close(f64(y), y_ref, "prefill y")
    # the same slots were written (others keep the sentinel), values within BF16 tolerance
    kg, vg = bits(kpd), bits(vpd)
    sentinel = 0xC480
    np.testing.assert_array_equal(kg == sentinel, ko == sentinel)
    assert_close(O.bf16_value(kg), O.bf16_value(ko), "K cache")
    assert_close(O.bf16_value(vg), O.bf16_value(vo), "V cache")
    for step in range(wl.decode_steps):
        xd = synth.make_x(B, d.hidden, seed=100 + step)
        ctx = torch.full((B,), S + step + 1, dtype=torch.int32)
        yd = api.layer_decode_step(cfg, packed, xd.to(DEV), kpd, vpd, td, ctx.to(DEV), status=status)
        torch.cuda.synchronize()
        yd_ref = O.layer_decode_step(d, Wn, f64(xd), ko, vo, table.numpy(), ctx.numpy())
        assert int(status.item()) == 0
        assert_close(f64(yd), yd_ref, f"decode step {step}")


@pytest.mark.parametrize("B,S", [(3, 17), (1, 130), (2, 1), (1, 200), (2, 300)])
def test_tiny_layer_ragged_prefill(B, S):
    wl, d, B, S, W, Wn, table, kp, vp, cfg, packed = _tiny_setup(seed=5, S=S, B=B, steps=0)
    x = synth.make_x(B * S, d.hidden, seed=31)
    pos = synth.prefill_positions(B, S)
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kpd, vpd, table.to(DEV))
    torch.cuda.synchronize()
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy())
    assert_close(f64(y), y_ref, f"prefill B{B} S{S}")


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("ctas", [1, 3, 7])
def test_prefill_attention_several_items_per_cta(head_dim, ctas):
    """The persistent prefill attention with its CTAs capped, so that each runs several
    (sequence, head, query tile) items back to back: ragged last query tiles, a chunk
    appended after a cached prefix (items of one and two key tiles with rows to mask).
    Against the oracle, and bit for bit against the default one-CTA-per-SM launch."""
    d = synth.DIMS_TINY if head_dim == 64 else synth.LayerDims(512, 4, 2, 128, 1024, 16)
    B, S, extra = 3, 300, 70
    W = synth.make_weights(d, 0.02, seed=131)
    Wn = {k: f64(v) for k, v in W.items()}
    table, nb = synth.make_block_table([S + extra] * B, d.block_size, seed=132, extra_blocks=3)
    kp, vp = synth.make_pool(nb, d, seed=133, fill="sentinel")
    cfg = api.make_config(d, max_position=S + extra + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    td = table.to(DEV)

    def run(cap):
        kpd, vpd = kp.to(DEV), vp.to(DEV)
        status = api.new_status()
        api.set_prefill_attention_ctas(cap)
        try:
            ys = []
            for start, n, seed in ((0, S, 134), (S, extra, 135)):
                x = synth.make_x(B * n, d.hidden, seed=seed)
                pos = synth.prefill_positions(B, n, start=start)
                ys.append(api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, n, kpd, vpd, td,
                                            status=status))
            torch.cuda.synchronize()
        finally:
            api.set_prefill_attention_ctas(0)
        assert int(status.item()) == 0
        return ys

    got, full = run(ctas), run(0)
    for g_, f_ in zip(got, full):
        assert torch.equal(g_, f_), "the result depends on how items are spread over CTAs"
    ko, vo = bits(kp), bits(vp)
    for (start, n, seed), y in zip(((0, S, 134), (S, extra, 135)), got):
        x = synth.make_x(B * n, d.hidden, seed=seed)
        pos = synth.prefill_positions(B, n, start=start)
        y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, n, ko, vo, table.numpy())
        assert_close(f64(y), y_ref, f"prefill from {start}, {n} tokens, {ctas} CTAs")


@pytest.mark.parametrize("ctas", [1, 0])
def test_prefill_attention_item_without_valid_positions(ctas):
    """A sequence whose positions are all out of range gives work items with no key tile:
    with one CTA they sit between the other sequences' items in its list.  The position
    error is flagged, nothing waits out its limit, and the other sequences match the oracle."""
    wl = synth.WORKLOADS["tiny_gqa"]
    d = wl.dims
    B, S = 3, 100
    W = synth.make_weights(d, wl.w_std, seed=141)
    Wn = {k: f64(v) for k, v in W.items()}
    table, nb = synth.make_block_table([S] * B, d.block_size, seed=142, extra_blocks=3)
    kp, vp = synth.make_pool(nb, d, seed=143, fill="sentinel")
    cfg = api.make_config(d, max_position=S + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    x = synth.make_x(B * S, d.hidden, seed=144)
    pos = synth.prefill_positions(B, S)
    pos[S:2 * S] = 10_000                      # sequence 1: beyond the cache and the RoPE table
    status = api.new_status()
    api.set_prefill_attention_ctas(ctas)
    try:
        y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kp.to(DEV), vp.to(DEV),
                              table.to(DEV), status=status)
        torch.cuda.synchronize()
    finally:
        api.set_prefill_attention_ctas(0)
    st = int(status.item())
    assert st & api.LL_DEV_BAD_POSITION and not st & api.LL_DEV_TIMEOUT, st
    keep = np.r_[0:S, 2 * S:3 * S]
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, Wn, f64(x)[keep], pos.numpy()[keep], 2, S, ko, vo, table.numpy()[[0, 2]])
    assert_close(f64(y)[keep], y_ref, "sequences 0 and 2")


@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (16, 1)])
def test_prefill_attention_wide_query_groups(Hq, Hkv):
    """Prefill layers whose KV heads serve 8 and 16 query heads (head_dim 128), with the
    CTAs capped so that the query heads of one KV head share a CTA's item list."""
    d = synth.LayerDims(Hq * 64, Hq, Hkv, 128, 512, 16)
    B, S = 2, 200
    W = synth.make_weights(d, 0.02, seed=171)
    Wn = {k: f64(v) for k, v in W.items()}
    table, nb = synth.make_block_table([S] * B, d.block_size, seed=172, extra_blocks=2)
    kp, vp = synth.make_pool(nb, d, seed=173, fill="sentinel")
    cfg = api.make_config(d, max_position=S + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    x = synth.make_x(B * S, d.hidden, seed=174)
    pos = synth.prefill_positions(B, S)
    status = api.new_status()
    api.set_prefill_attention_ctas(4)
    try:
        y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kp.to(DEV), vp.to(DEV),
                              table.to(DEV), status=status)
        torch.cuda.synchronize()
    finally:
        api.set_prefill_attention_ctas(0)
    assert int(status.item()) == 0
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy())
    assert_close(f64(y), y_ref, f"prefill, {Hq} query heads over {Hkv} KV heads")


@pytest.mark.parametrize("bs", [32, 64, 256])
def test_prefill_attention_block_sizes(bs):
    """Paged prefill attention with KV blocks of 32, 64 and 256 positions (a 256-position
    block spans two 128-key tiles; smaller ones fill a tile from several boxes), with
    the CTAs capped so that each runs several items.  Against the oracle."""
    d = synth.LayerDims(256, 4, 2, 64, 688, bs)
    B, S = 2, 300
    W = synth.make_weights(d, 0.02, seed=151)
    Wn = {k: f64(v) for k, v in W.items()}
    table, nb = synth.make_block_table([S] * B, bs, seed=152, extra_blocks=2)
    kp, vp = synth.make_pool(nb, d, seed=153, fill="sentinel")
    cfg = api.make_config(d, max_position=S + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    x = synth.make_x(B * S, d.hidden, seed=154)
    pos = synth.prefill_positions(B, S)
    status = api.new_status()
    api.set_prefill_attention_ctas(5)
    try:
        y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kp.to(DEV), vp.to(DEV),
                              table.to(DEV), status=status)
        torch.cuda.synchronize()
    finally:
        api.set_prefill_attention_ctas(0)
    assert int(status.item()) == 0
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy())
    assert_close(f64(y), y_ref, f"prefill with {bs}-position blocks")


def test_prefill_attention_long_cached_context():
    """A 64-token chunk appended at positions 60000..60063 over a cached prefix of N(0, 1)
    K/V: each work item runs 469 key tiles (the metadata warp marks 3752 valid 16-key
    chunks per item).  Against the oracle."""
    d = synth.DIMS_TINY
    start, n = 60_000, 64
    W = synth.make_weights(d, 0.02, seed=161)
    Wn = {k: f64(v) for k, v in W.items()}
    table, nb = synth.make_block_table([start + n], d.block_size, seed=162, extra_blocks=2)
    kp, vp = synth.make_pool(nb, d, seed=163)
    cfg = api.make_config(d, max_position=start + n + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    x = synth.make_x(n, d.hidden, seed=164)
    pos = synth.prefill_positions(1, n, start=start)
    status = api.new_status()
    y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), 1, n, kp.to(DEV), vp.to(DEV), table.to(DEV),
                          status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), 1, n, ko, vo, table.numpy())
    assert_close(f64(y), y_ref, "64 tokens after a 60000-position prefix")


def test_chunked_prefill_attends_to_cached_prefix():
    wl, d, B, S, W, Wn, table, kp, vp, cfg, packed = _tiny_setup(seed=7, S=64, B=2, steps=40)
    kpd, vpd, td = kp.to(DEV), vp.to(DEV), table.to(DEV)
    ko, vo = bits(kp), bits(vp)
    for start, n in ((0, 64), (64, 40)):
        x = synth.make_x(B * n, d.hidden, seed=41 + start)
        pos = synth.prefill_positions(B, n, start=start)
        y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, n, kpd, vpd, td)
        torch.cuda.synchronize()
        y_ref = O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, n, ko, vo, table.numpy())
        assert_close(f64(y), y_ref, f"chunk at {start}")


def test_bad_block_table_sets_status_without_fault():
    wl, d, B, S, W, Wn, table, kp, vp, cfg, packed = _tiny_setup(seed=9, S=32, B=2, steps=1)
    bad = table.clone()
    bad[1, 0] = 10_000        # beyond the pool
    bad[0, 1] = -1            # a hole inside the context
    x = synth.make_x(B * 32, d.hidden, seed=51)
    pos = synth.prefill_positions(B, 32)
    status = api.new_status()
    y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, 32, kp.to(DEV), vp.to(DEV),
                          bad.to(DEV), status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & api.LL_DEV_BAD_BLOCK
    assert torch.isfinite(y.float()).all()


def test_decode_step_is_bitwise_repeatable():
    """The weight-form GEMMs split K over CTAs and add the float32 partials in a fixed
    order whichever CTA finishes last, so repeating a step reproduces every bit (the
    K/V rows it appends are rewritten with the same values)."""
    wl, d, B, S, W, Wn, table, kp, vp, cfg, packed = _tiny_setup(seed=11, S=40, B=2, steps=2)
    kpd, vpd, td = kp.to(DEV), vp.to(DEV), table.to(DEV)
    ctx = torch.full((B,), S + 1, dtype=torch.int32, device=DEV)
    xd = synth.make_x(B, d.hidden, seed=61).to(DEV)
    status = api.new_status()
    y1 = api.layer_decode_step(cfg, packed, xd, kpd, vpd, td, ctx, status=status).clone()
    y2 = api.layer_decode_step(cfg, packed, xd, kpd, vpd, td, ctx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("m,n,k", [(64, 12288, 4096), (7, 22016, 4096), (64, 4096, 11008), (200, 4096, 4096)])
def test_weight_form_linear_repeatable(m, n, k):
    x = synth.normal_bf16((m, k), 1.0, seed=k + m, tag="x").to(DEV)
    w = synth.normal_bf16((n, k), 0.02, seed=n, tag="w").to(DEV)
    y1 = api.linear(x, w)
    y2 = api.linear(x, w)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    idx = torch.arange(0, n, 997)
    ref = f64(x.cpu()) @ f64(w.cpu()[idx]).T
    assert_close(f64(y1.cpu()[:, idx]), ref, f"linear {m}x{n}x{k} sampled", atol=2e-3, rtol=8e-3)


@pytest.mark.parametrize("ctx0,q_len", [((17, 130, 64), 4), ((1, 255, 40), 3), ((300, 5), 16)])
def test_multi_token_decode_over_ragged_cached_contexts(ctx0, q_len):
    """Several new tokens per request appended after cached contexts of different lengths
    (a prefill chunk per request at its own position offset): each token attends to its
    request's cached prefix plus the new tokens up to itself."""
    B = len(ctx0)
    wl = synth.WORKLOADS["tiny_gqa"]
    d = wl.dims
    W = synth.make_weights(d, wl.w_std, seed=71)
    lens = [c + q_len for c in ctx0]
    table, nb = synth.make_block_table(lens, d.block_size, seed=72, extra_blocks=3)
    kp, vp = synth.make_pool(nb, d, seed=73)            # the cached prefix: N(0, 1) K/V
    cfg = api.make_config(d, max_position=max(lens) + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    x = synth.make_x(B * q_len, d.hidden, seed=74)
    pos = torch.cat([torch.arange(c, c + q_len, dtype=torch.int32) for c in ctx0])
    kpd, vpd = kp.to(DEV), vp.to(DEV)
    status = api.new_status()
    y = api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, q_len, kpd, vpd, table.to(DEV), status=status)
    torch.cuda.synchronize()
    ko, vo = bits(kp), bits(vp)
    y_ref = O.layer_prefill(d, {k: f64(v) for k, v in W.items()}, f64(x), pos.numpy(), B, q_len, ko, vo,
                            table.numpy())
    assert int(status.item()) == 0
    assert_close(f64(y), y_ref, f"multi-token decode {ctx0} + {q_len}")
    np.testing.assert_array_equal(bits(kpd) == bits(kp), ko == bits(kp))   # only the new slots changed


@pytest.mark.parametrize("mode", ["prefill", "decode"])
def test_checkpoints_match_oracle_stage_by_stage(mode):
    """Each kernel output the fused layer leaves in its workspace (x_hat, q after RoPE,
    attention o, residual h, h_hat, SwiGLU a) against the oracle's value of that stage,
    so that a wrong layer output can be traced to one kernel."""
    wl, d, B, S, W, Wn, table, kp, vp, cfg, packed = _tiny_setup(seed=81, S=40, B=2, steps=1)
    kpd, vpd, td = kp.to(DEV), vp.to(DEV), table.to(DEV)
    ko, vo = bits(kp), bits(vp)
    want = {}
    if mode == "prefill":
        T = B * S
        x = synth.make_x(T, d.hidden, seed=82)
        pos = synth.prefill_positions(B, S)
        ws = api.new_workspace(cfg, T, table.shape[1])
        api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kpd, vpd, td, workspace=ws)
        O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy(), want=want)
    else:
        # a prefill fills the cache, then one decode step is checked stage by stage
        x = synth.make_x(B * S, d.hidden, seed=83)
        pos = synth.prefill_positions(B, S)
        api.layer_prefill(cfg, packed, x.to(DEV), pos.to(DEV), B, S, kpd, vpd, td)
        O.layer_prefill(d, Wn, f64(x), pos.numpy(), B, S, ko, vo, table.numpy())
        T = B
        xd = synth.make_x(B, d.hidden, seed=84)
        ctx = torch.full((B,), S + 1, dtype=torch.int32)
        ws = api.new_workspace(cfg, T, table.shape[1])
        api.layer_decode_step(cfg, packed, xd.to(DEV), kpd, vpd, td, ctx.to(DEV), workspace=ws)
        O.layer_decode_step(d, Wn, f64(xd), ko, vo, table.numpy(), ctx.numpy(), want=want)
    torch.cuda.synchronize()
    cp = api.checkpoints(cfg, ws, T, table.shape[1], T)
    for name, ref in (("x_hat", want["xh"]), ("q", want["q"].reshape(T, -1)), ("o", want["o"].reshape(T, -1)),
                      ("h", want["h"]), ("h_hat", want["hh"]), ("a", want["a"])):
        assert_close(f64(cp[name]), ref, f"{mode} checkpoint {name}")


# ---------------------------------------------------------------- INT8 KV cache

@pytest.mark.parametrize("T,Hkv,d,bs,nb", [(37, 2, 64, 16, 8), (300, 8, 128, 128, 5), (5, 4, 128, 32, 3)])
def test_reshape_and_cache_q8_bit_exact(T, Hkv, d, bs, nb):
    g = torch.Generator().manual_seed(T * 7 + d)
    # rows of very different magnitudes, one all-zero row, one row with a single non-zero
    mag = torch.exp(torch.randn(T, Hkv, 1, generator=g) * 3)
    k = (torch.randn(T, Hkv, d, generator=g) * mag).to(torch.bfloat16)
    v = (torch.randn(T, Hkv, d, generator=g) * mag).to(torch.bfloat16)
    k[0, 0] = 0
    v[min(1, T - 1), Hkv - 1] = 0
    v[min(1, T - 1), Hkv - 1, 3] = -2.5
    slots = synth.make_slot_mapping(T, nb * bs, seed=T + 11, n_skip=min(2, T - 1))
    pool = api.PoolQ8.empty(nb, Hkv, bs, d)
    st = api.reshape_and_cache_q8(k.to(DEV), v.to(DEV), slots.to(DEV), pool)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qk = O.QuantPool(np.zeros((nb, Hkv, bs, d), np.int8), np.zeros((nb, Hkv, bs), np.float32))
    qv = O.QuantPool(np.zeros((nb, Hkv, bs, d), np.int8), np.zeros((nb, Hkv, bs), np.float32))
    O.reshape_and_cache(f64(k), f64(v), slots.numpy(), qk, qv)
    np.testing.assert_array_equal(pool.k.cpu().numpy(), qk.codes)
    np.testing.assert_array_equal(pool.v.cpu().numpy(), qv.codes)
    np.testing.assert_array_equal(pool.k_scale.cpu().numpy().view(np.uint32), qk.scales.view(np.uint32))
    np.testing.assert_array_equal(pool.v_scale.cpu().numpy().view(np.uint32), qv.scales.view(np.uint32))


def _random_q8_pool(nb, Hkv, bs, d, seed):
    g = torch.Generator().manual_seed(seed)
    codes = lambda: torch.randint(-127, 128, (nb, Hkv, bs, d), generator=g, dtype=torch.int32).to(torch.int8)
    scales = lambda: (torch.rand(nb, Hkv, bs, generator=g) * 0.03 + 0.001).float()
    return codes(), codes(), scales(), scales()


@pytest.mark.parametrize("B,Hq,Hkv,bs,ctx_lo,ctx_hi", [
    (5, 8, 8, 128, 1, 300),             # MHA, ragged
    (3, 16, 2, 128, 900, 3100),         # GQA 8, several 1024-key splits
    (4, 4, 4, 32, 1023, 1026),          # split boundaries, 32-row blocks
    (2, 8, 1, 16, 1, 90),               # 16-row blocks, one KV head
    (3, 12, 3, 128, 1, 700),            # GQA 4: half the query columns padding
    (2, 16, 1, 64, 500, 2100),          # GQA 16: two query column tiles
    (40, 8, 1, 16, 1, 2100),            # many sequences: the sorted dispatch order
])
def test_paged_attention_decode_q8(B, Hq, Hkv, bs, ctx_lo, ctx_hi):
    d = 128
    ctx = synth.make_context_lens(B, ctx_lo, ctx_hi, seed=B * 19)
    ctx[0] = ctx_lo
    table, nb = synth.make_block_table(ctx.tolist(), bs, seed=B * 23, extra_blocks=3)
    kc, vc, ks, vs = _random_q8_pool(nb, Hkv, bs, d, seed=B * 29)
    q = synth.normal_bf16((B, Hq, d), 1.0, seed=B + 5, tag="q")
    pool = api.PoolQ8(kc.to(DEV), vc.to(DEV), ks.to(DEV), vs.to(DEV))
    scale = 1 / math.sqrt(d)
    out = api.paged_attention_decode_q8(q.to(DEV), pool, table.to(DEV), ctx.to(DEV), scale)
    torch.cuda.synchronize()
    ref = O.paged_attention_decode(f64(q), O.QuantPool(kc.numpy(), ks.numpy()), O.QuantPool(vc.numpy(), vs.numpy()),
                                   table.numpy(), ctx.numpy(), scale)
    assert_close(f64(out), ref, "paged_attention_decode_q8")


def test_paged_attention_decode_q8_bad_block_is_flagged_and_finite():
    B, Hq, Hkv, bs, d = 2, 4, 2, 16, 128
    ctx = torch.tensor([40, 33], dtype=torch.int32)
    table, nb = synth.make_block_table(ctx.tolist(), bs, seed=3, extra_blocks=2)
    table[1, 1] = 10_000                     # beyond the pool: its keys are left out
    kc, vc, ks, vs = _random_q8_pool(nb, Hkv, bs, d, seed=7)
    ks[:] = float("inf")                     # stale scales must never reach P
    ks[table[0, :3].long()] = 0.01
    ks[table[1, [0, 2]].long()] = 0.01
    pool = api.PoolQ8(kc.to(DEV), vc.to(DEV), ks.to(DEV), vs.to(DEV))
    q = synth.normal_bf16((B, Hq, d), 1.0, seed=9, tag="q")
    status = api.new_status()
    out = api.paged_attention_decode_q8(q.to(DEV), pool, table.to(DEV), ctx.to(DEV), 0.09, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & api.LL_DEV_BAD_BLOCK
    assert torch.isfinite(out.float()).all()


def test_layer_decode_steps_over_int8_cache():
    """Decode steps of a GQA layer (head_dim 128) over a pre-filled INT8 pool: each step
    quantises the new token's K/V into the pool and attends over code * scale."""
    d = synth.LayerDims(512, 4, 2, 128, 1024, 16)
    B, steps = 3, 4
    W = synth.make_weights(d, 0.02, seed=91)
    Wn = {k: f64(v) for k, v in W.items()}
    ctx0 = synth.make_context_lens(B, 20, 140, seed=92)
    table, nb = synth.make_block_table((ctx0 + steps).tolist(), d.block_size, seed=93, extra_blocks=2)
    kc, vc, ks, vs = _random_q8_pool(nb, d.n_kv_heads, d.block_size, d.head_dim, seed=94)
    pool = api.PoolQ8(kc.to(DEV), vc.to(DEV), ks.to(DEV), vs.to(DEV))
    qk, qv = O.QuantPool(kc.numpy().copy(), ks.numpy().copy()), O.QuantPool(vc.numpy().copy(), vs.numpy().copy())
    cfg = api.make_config(d, max_position=int(ctx0.max()) + steps + 1)
    packed = api.pack_weights(cfg, {k: v.to(DEV) for k, v in W.items()})
    td = table.to(DEV)
    status = api.new_status()
    for step in range(steps):
        ctx = (ctx0 + step + 1).to(torch.int32)
        x = synth.make_x(B, d.hidden, seed=95 + step)
        y = api.layer_decode_step_q8(cfg, packed, x.to(DEV), pool, td, ctx.to(DEV), status=status)
        torch.cuda.synchronize()
        y_ref = O.layer_decode_step(d, Wn, f64(x), qk, qv, table.numpy(), ctx.numpy())
        assert int(status.item()) == 0
        assert_close(f64(y), y_ref, f"INT8-cache decode step {step}")
    # the appended rows: codes within one step of the oracle's (its K/V may round the other
    # way in a last bit), scales within a few parts in a thousand
    gk, gs = pool.k.cpu().numpy(), pool.k_scale.cpu().numpy()
    assert np.abs(gk.astype(np.int32) - qk.codes.astype(np.int32)).max() <= 1
    np.testing.assert_allclose(gs, qk.scales, rtol=5e-3)
