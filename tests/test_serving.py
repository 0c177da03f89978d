"""Continuous batching: the host block allocator and scheduler (CPU), and a tiny
multi-layer stack driven through admissions and retirements against the oracle (GPU)."""
import numpy as np
import pytest
import torch

from oracle import llama_layer as O
from tests.helpers import assert_close, bits, f64
from transformer_decoder_layer_llama_gb300 import synth
from transformer_decoder_layer_llama_gb300.serving import BlockAllocator, Scheduler


def test_allocator_lifo_and_double_free():
    a = BlockAllocator(10, seed=1)
    x = a.alloc(3)
    assert len(set(x)) == 3 and a.free_count() == 7
    a.free([x[1]])
    assert a.alloc(1) == [x[1]]            # last freed, first reused
    with pytest.raises(ValueError):
        a.free([x[0], x[0]])
    with pytest.raises(MemoryError):
        a.alloc(100)


def _replay(n_slots, bs, ctx0, budgets_seed, steps, prompt, bmax, nb, seed):
    """Independent re-simulation of the policy: LIFO free list from the same seeded
    permutation, budgets from the same seeded stream, retire -> free -> admit, then one
    appended token per slot with a new block at each block boundary."""
    free = torch.randperm(nb, generator=torch.Generator().manual_seed(seed)).tolist()
    rng = np.random.default_rng(budgets_seed)
    reqs = []
    for c in ctx0:
        n = -(-c // bs)
        blocks = [free.pop() for _ in range(n)]
        reqs.append([c, int(rng.integers(1, bmax + 1)), blocks])
    history = []
    for _ in range(steps):
        for s in range(n_slots):
            if reqs[s][1] > 0:
                continue
            free.extend(reqs[s][2])
            blocks = [free.pop() for _ in range(-(-prompt // bs))]
            reqs[s] = [prompt, int(rng.integers(1, bmax + 1)), blocks]
        for r in reqs:
            if r[0] % bs == 0 and r[0] // bs >= len(r[2]):
                r[2].append(free.pop())
            r[0] += 1
            r[1] -= 1
        history.append([(r[0], list(r[2])) for r in reqs])
    return history


def test_scheduler_matches_independent_replay_and_invariants():
    n_slots, bs, steps, prompt, bmax, nb = 6, 16, 40, 24, 5, 200
    ctx0 = [5, 16, 17, 40, 63, 1]
    alloc = BlockAllocator(nb, seed=3)
    sch = Scheduler(n_slots, bs, 16, alloc, seed=9, budget_max=bmax, prompt_len=prompt)
    for s, c in enumerate(ctx0):
        sch.start_resident(s, c)
    expect = _replay(n_slots, bs, ctx0, 9, steps, prompt, bmax, nb, 3)
    admitted_total = 0
    for step in range(steps):
        admitted_total += len(sch.retire_and_admit())
        ctx = sch.grow_for_decode()
        live = [b for r in sch.slots for b in r.blocks]
        assert len(live) == len(set(live))                       # no block shared
        assert len(live) + alloc.free_count() == nb              # nothing leaked
        for s, r in enumerate(sch.slots):
            assert ctx[s] == r.ctx and -(-r.ctx // bs) == len(r.blocks)
            row = sch.table[s]
            assert list(row[:len(r.blocks)]) == r.blocks and (row[len(r.blocks):] == -1).all()
        assert [(r.ctx, r.blocks) for r in sch.slots] == expect[step]
    assert admitted_total > n_slots          # requests did retire and get replaced


@pytest.mark.gpu
def test_tiny_stack_continuous_batching_matches_oracle():
    """Steps 0-1 decode eagerly, steps 2-5 replay a captured CUDA graph; requests retire
    (budgets <= 3) and new ones are prefilled on the way."""
    from transformer_decoder_layer_llama_gb300 import api
    from transformer_decoder_layer_llama_gb300.serving import StackEngine
    d = synth.DIMS_TINY
    L, n_slots, prompt, steps, bmax = 2, 4, 16, 6, 3
    ctx0 = [8, 20, 33, 40]
    max_blocks = 8
    nb = 64
    Ws = [synth.make_weights(d, 0.02, seed=100 + l) for l in range(L)]
    cfg = api.make_config(d, max_position=max_blocks * d.block_size)
    packed = [api.pack_weights(cfg, {k: v.cuda() for k, v in W.items()}) for W in Ws]
    pools_cpu = [synth.make_pool(nb, d, seed=200 + l) for l in range(L)]
    pools = [(k.cuda(), v.cuda()) for k, v in pools_cpu]
    opools = [(bits(k), bits(v)) for k, v in pools_cpu]
    Wn = [{k: f64(v) for k, v in W.items()} for W in Ws]
    alloc = BlockAllocator(nb, seed=5)
    sch = Scheduler(n_slots, d.block_size, max_blocks, alloc, seed=6, budget_max=bmax, prompt_len=prompt)
    for s, c in enumerate(ctx0):
        sch.start_resident(s, c)
    eng = StackEngine(api, [cfg] * L, packed, pools, n_slots, max_blocks, n_slots * prompt)
    stream = torch.cuda.Stream()            # graph capture needs a non-default stream
    torch.cuda.set_stream(stream)
    for step in range(steps):
        admitted = sch.retire_and_admit()
        if admitted:
            xp = synth.make_x(len(admitted) * prompt, d.hidden, seed=300 + step)
            pos = synth.prefill_positions(len(admitted), prompt)
            sub = torch.from_numpy(sch.table[admitted].copy())
            eng.pf_x[:len(xp)].copy_(xp)
            eng.pf_pos[:len(pos)].copy_(pos)
            eng.pf_table[:len(admitted)].copy_(sub)
            yp = eng.prefill(len(admitted), prompt, stream)
            xo = f64(xp)
            for l in range(L):
                y = O.layer_prefill(d, Wn[l], xo, pos.numpy(), len(admitted), prompt, *opools[l], sub.numpy())
                xo = O.bf16_round(y) if l < L - 1 else y
            torch.cuda.synchronize()
            assert_close(f64(yp), xo, f"step {step} prefill")
        ctx = sch.grow_for_decode()
        xd = synth.make_x(n_slots, d.hidden, seed=400 + step)
        eng.table.copy_(torch.from_numpy(sch.table))
        eng.ctx.copy_(torch.from_numpy(ctx))
        eng.x.copy_(xd)
        if step == 2:
            eng.capture_decode(stream)   # later steps replay the all-layer decode as a CUDA graph
        yd = eng.decode(stream)
        xo = f64(xd)
        for l in range(L):
            y = O.layer_decode_step(d, Wn[l], xo, *opools[l], sch.table.copy(), ctx)
            xo = O.bf16_round(y) if l < L - 1 else y
        torch.cuda.synchronize()
        assert int(eng.status.item()) == 0
        assert_close(f64(yd), xo, f"step {step} decode")
    torch.cuda.set_stream(torch.cuda.default_stream())
