"""GPU parity of the 32-layer continuous-batching workload at its full size:
Llama-2-7B-shaped layers, 64 slots with resident contexts ~U[128, 4096],
128-token blocks, decode budgets ~U[1, 256], admitted requests prefilled with
256 tokens (page "Which ops-transformer operators one Llama2-7B layer calls",
section "single-layer operator call chain": the stack is the service time;
page "ATB KV-cache paging, quantisation, speculative decoding and communication
overlap", section "KV Cache memory wall": blocks handed out and returned).

The first two steps, as the benchmark runs them (the scheduler, one batched
prefill per layer for the admitted requests, the all-layer decode eagerly in
step 0 and replayed from a captured CUDA graph in step 1), against the oracle
chaining its own 32 layers from the same seeded inputs.  The scheduler seed is
one whose first step retires two requests, so step 1 admits and prefills.

Then every layer of both steps teacher-forced: each GPU layer call gets the
oracle's own input for that layer (rounded to BF16 as the stack passes it on)
over a pool that started from the same seeded contents, and its output is held
to the single-layer limits.

Weights, pools and inputs are drawn by torch's seeded generators (weights and
pools on the device, for speed); the oracle gets host copies of those draws,
never a value the library computed.
"""
import numpy as np
import pytest
import torch

from oracle import llama_layer as O
from tests.helpers import bits, f64, outside_stats
from transformer_decoder_layer_llama_gb300 import synth
from transformer_decoder_layer_llama_gb300.serving import BlockAllocator, Scheduler

pytestmark = pytest.mark.gpu

DEV = "cuda"
L, N_SLOTS, PROMPT, STEPS = 32, 64, 256, 2
SCHED_SEED = 5            # two requests with a decode budget of 1: step 1 admits two

# Limits (fraction of elements outside 1e-2 + 1e-2 |oracle|, worst multiple of the bound),
# set just above what GB300 measures.
# 32 chained layers: each layer's rounding differences feed the next, and the random-init
# stack amplifies them, so the per-element bound is no measure here.  The chained check
# takes each token row's relative error ||y_gpu - y_oracle|| / ||y_oracle|| instead (a slot
# run with a wrong table, context or input would be off by order one); the oracle itself
# shows the amplification: moving 1% of the elements of the first layer's input by one
# BF16 unit moves its 32-layer output by 2.9% per row.  GB300 against the oracle: 2.7%
# (decode, median; 3.3% worst row) and 3.3% (prefill; 3.8% worst row).
CHAIN_ROW_REL_LIMIT = 0.05
# One teacher-forced decode layer: GB300 worst over the 64 layer calls 1.3e-4 / 1.73x.
DECODE_LAYER_LIMIT = (2e-4, 2.0)
# One teacher-forced 2 x 256-token prefill layer.  A short prefill averages its attention
# over fewer keys, so o is larger and its BF16 roundings move h further: on GB300 a 7B
# prefill layer of 2 x 256 tokens leaves 5.6e-3 of its outputs outside the bound (2048
# tokens: 2.6e-3), the CPU model of a correct float32-accumulating BF16 implementation
# 2.9e-3 (tests/tolerance_model.py's arithmetic at that shape); every stage before the
# SwiGLU output is clean.  Worst over the 32 layer calls: 6.0e-3 / 2.40x.
PREFILL_LAYER_LIMIT = (8e-3, 3.0)


def _setup():
    from transformer_decoder_layer_llama_gb300 import api
    d = synth.DIMS_7B
    ctx0 = synth.make_context_lens(N_SLOTS, 128, 4096, seed=501).tolist()
    max_ctx = max(max(ctx0), PROMPT) + STEPS + 1
    max_blocks = -(-max_ctx // d.block_size) + 1
    nb = sum(-(-(max(c, PROMPT) + STEPS + 1) // d.block_size) + 1 for c in ctx0) + 2 * N_SLOTS
    cfg = api.make_config(d, max_blocks * d.block_size)
    packed = []
    for l in range(L):
        W = synth.make_weights(d, 0.02, seed=600 + l, device=DEV)
        packed.append(api.pack_weights(cfg, W))
        del W
    pools = [synth.make_pool(nb, d, seed=700 + l, device=DEV) for l in range(L)]
    return api, d, ctx0, max_blocks, nb, cfg, packed, pools


def _refill(pools, d, nb):
    for l, (k, v) in enumerate(pools):
        k0, v0 = synth.make_pool(nb, d, seed=700 + l, device=DEV)
        k.copy_(k0)
        v.copy_(v0)


def test_stack_first_two_steps_and_teacher_forced_layers():
    from transformer_decoder_layer_llama_gb300.serving import StackEngine
    api, d, ctx0, max_blocks, nb, cfg, packed, pools = _setup()
    alloc = BlockAllocator(nb, seed=502)
    sch = Scheduler(N_SLOTS, d.block_size, max_blocks, alloc, seed=SCHED_SEED, budget_max=256, prompt_len=PROMPT)
    for s, c in enumerate(ctx0):
        sch.start_resident(s, c)
    eng = StackEngine(api, [cfg] * L, packed, pools, N_SLOTS, max_blocks, N_SLOTS * PROMPT)
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    steps = []
    try:
        for step in range(STEPS):
            admitted = sch.retire_and_admit()
            rec = {"admitted": admitted, "yp": None}
            if admitted:
                n = len(admitted)
                rec["xp"] = synth.make_x(n * PROMPT, d.hidden, seed=520 + step)
                rec["pos"] = synth.prefill_positions(n, PROMPT)
                rec["sub"] = sch.table[admitted].copy()
                eng.pf_x[:n * PROMPT].copy_(rec["xp"])
                eng.pf_pos[:n * PROMPT].copy_(rec["pos"])
                eng.pf_table[:n].copy_(torch.from_numpy(rec["sub"]))
                rec["yp"] = eng.prefill(n, PROMPT, stream).clone()
            rec["ctx"] = sch.grow_for_decode()
            rec["table"] = sch.table.copy()
            rec["x"] = synth.make_x(N_SLOTS, d.hidden, seed=510 + step)
            eng.table.copy_(torch.from_numpy(rec["table"]))
            eng.ctx.copy_(torch.from_numpy(rec["ctx"]))
            eng.x.copy_(rec["x"])
            if step == 1:
                eng.capture_decode(stream)   # the benchmark's graph-replayed decode
            rec["yd"] = eng.decode(stream).clone()
            steps.append(rec)
        torch.cuda.synchronize()
        assert int(eng.status.item()) == 0
        assert not steps[0]["admitted"] and len(steps[1]["admitted"]) == 2

        # teacher-forced pass over pools refilled with the same draws, layer by layer beside the oracle
        _refill(pools, d, nb)
        ws = api.new_workspace(cfg, N_SLOTS * PROMPT, max_blocks)
        status = api.new_status()
        xo_dec = [f64(r["x"]) for r in steps]
        xo_pf = {i: f64(r["xp"]) for i, r in enumerate(steps) if r["admitted"]}
        rng = np.random.default_rng(503)
        xo_pert = xo_dec[0].copy()
        hit = rng.random(xo_pert.shape) < 0.01
        ulp = 2.0 ** (np.floor(np.log2(np.abs(xo_pert) + 1e-30)) - 7)
        xo_pert[hit] += np.where(rng.random(int(hit.sum())) < 0.5, -1.0, 1.0) * ulp[hit]
        worst_layer = {}
        for l in range(L):
            W = synth.make_weights(d, 0.02, seed=600 + l, device=DEV)
            Wn = {k: f64(v) for k, v in W.items()}
            del W
            k0, v0 = synth.make_pool(nb, d, seed=700 + l, device=DEV)
            ko, vo = bits(k0), bits(v0)
            del k0, v0
            kd, vd = pools[l]
            # the oracle's sensitivity: step 0 again from a perturbed input, on its own pool copy
            xo_pert = O.layer_decode_step(d, Wn, xo_pert, ko.copy(), vo.copy(), steps[0]["table"], steps[0]["ctx"])
            xo_pert = O.bf16_round(xo_pert) if l < L - 1 else xo_pert
            for i, r in enumerate(steps):
                if r["admitted"]:
                    n = len(r["admitted"])
                    yp_ref = O.layer_prefill(d, Wn, xo_pf[i], r["pos"].numpy(), n, PROMPT, ko, vo, r["sub"])
                    yp = api.layer_prefill(cfg, packed[l], torch.from_numpy(xo_pf[i]).to(torch.bfloat16).to(DEV),
                                           r["pos"].to(DEV), n, PROMPT, kd, vd, torch.from_numpy(r["sub"]).to(DEV),
                                           workspace=ws, status=status)
                    torch.cuda.synchronize()
                    worst_layer[(l, i, "prefill")] = outside_stats(f64(yp), yp_ref)
                    xo_pf[i] = O.bf16_round(yp_ref) if l < L - 1 else yp_ref
                yd_ref = O.layer_decode_step(d, Wn, xo_dec[i], ko, vo, r["table"], r["ctx"])
                yd = api.layer_decode_step(cfg, packed[l], torch.from_numpy(xo_dec[i]).to(torch.bfloat16).to(DEV),
                                           kd, vd, torch.from_numpy(r["table"]).to(DEV),
                                           torch.from_numpy(r["ctx"]).to(DEV), workspace=ws, status=status)
                torch.cuda.synchronize()
                worst_layer[(l, i, "decode")] = outside_stats(f64(yd), yd_ref)
                xo_dec[i] = O.bf16_round(yd_ref) if l < L - 1 else yd_ref
        assert int(status.item()) == 0
        for kind, limit in (("decode", DECODE_LAYER_LIMIT), ("prefill", PREFILL_LAYER_LIMIT)):
            st = {k: v for k, v in worst_layer.items() if k[2] == kind}
            frac = max(v[0] for v in st.values())
            ratio = max(v[1] for v in st.values())
            print(f"teacher-forced {kind} layers ({len(st)}): worst fraction outside {frac:.2e}, "
                  f"worst multiple {ratio:.2f}x, mean fraction {np.mean([v[0] for v in st.values()]):.2e}")
        for (l, i, kind), (frac, ratio, _) in sorted(worst_layer.items()):
            max_frac, max_ratio = DECODE_LAYER_LIMIT if kind == "decode" else PREFILL_LAYER_LIMIT
            assert frac <= max_frac and ratio <= max_ratio, (
                f"layer {l} step {i} {kind} (teacher-forced): {frac:.2e} outside, {ratio:.2f}x the bound")

        # the chained outputs of the engine run against the oracle's own 32-layer chain
        row_rel = lambda got, ref: np.linalg.norm(got - ref, axis=1) / np.linalg.norm(ref, axis=1)
        pert = row_rel(xo_pert, xo_dec[0])
        print(f"oracle: 1% of the first layer's input moved by one BF16 unit moves the 32-layer output by "
              f"{np.median(pert):.2e} per row (median), {pert.max():.2e} (max)")
        chained = []
        for i, r in enumerate(steps):
            if r["admitted"]:
                chained.append((f"32-layer prefill step {i}", f64(r["yp"]), xo_pf[i]))
            chained.append((f"32-layer decode step {i}", f64(r["yd"]), xo_dec[i]))
        for name, got, ref in chained:
            frac, worst, rms = outside_stats(got, ref)
            rr = row_rel(got, ref)
            print(f"{name}: row relative error median {np.median(rr):.2e}, max {rr.max():.2e}; "
                  f"{frac:.2e} of elements outside the per-element bound")
        for name, got, ref in chained:
            assert np.isfinite(got).all(), name
            rr = row_rel(got, ref)
            assert rr.max() <= CHAIN_ROW_REL_LIMIT, f"{name}: a row is {rr.max():.2e} off (limit {CHAIN_ROW_REL_LIMIT})"
    finally:
        torch.cuda.set_stream(torch.cuda.default_stream())
