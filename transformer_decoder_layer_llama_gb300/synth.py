"""Seeded synthetic inputs for the Llama-style decoder layer.

This module only draws random numbers and lays them out; it holds none of the
layer's arithmetic.  Both the CUDA path and the CPU oracle are fed from here,
so the two sides see identical bytes.  Every tensor is drawn on the CPU with a
`torch.Generator` seeded by the caller.

Shapes and distributions follow the workloads the decoder-layer pages discuss:
a Llama2-7B layer (hidden 4096, 32 heads x 128, FFN 11008; page "Which
ops-transformer operators one Llama2-7B layer calls", section "single-layer
operator chain"), a 70B-shaped GQA layer (hidden 8192, 80 layers; page "ATB
KV-cache paging...", section "the KV-cache memory wall"), and a tiny GQA layer
for exhaustive checks.  Weights are BF16 ~ N(0, w_std^2), RMSNorm gains are
fp32 ~ 1 + N(0, 0.1^2), activations and pre-filled cache contents are BF16 ~
N(0, 1), context lengths are uniform integers and block tables are seeded
random permutations of the pool's blocks.
"""
from __future__ import annotations

import dataclasses
import zlib

import torch

BF16 = torch.bfloat16


@dataclasses.dataclass(frozen=True)
class LayerDims:
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    block_size: int
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def qkv_rows(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: LayerDims
    w_std: float
    batch: int
    prefill_len: int = 0      # tokens per sequence in a prefill call (0: decode workload)
    decode_steps: int = 0     # decode steps that follow the prefill (tiny workload)
    ctx_lo: int = 0           # decode: context_lens ~ U[ctx_lo, ctx_hi] (inclusive)
    ctx_hi: int = 0
    layers: int = 1
    steps: int = 0            # continuous batching: steps measured
    new_prefill: int = 0      # continuous batching: prompt length of a newly admitted request


DIMS_TINY = LayerDims(256, 4, 2, 64, 688, 16)
DIMS_7B = LayerDims(4096, 32, 32, 128, 11008, 128)
DIMS_70B = LayerDims(8192, 64, 8, 128, 28672, 128)

WORKLOADS = {
    "tiny_gqa": Workload("tiny_gqa", DIMS_TINY, 0.02, batch=2, prefill_len=64, decode_steps=8),
    "llama2_7b_prefill": Workload("llama2_7b_prefill", DIMS_7B, 0.02, batch=1, prefill_len=2048),
    "llama2_7b_decode": Workload("llama2_7b_decode", DIMS_7B, 0.02, batch=64, ctx_lo=512, ctx_hi=4096),
    "llama70b_gqa_decode": Workload("llama70b_gqa_decode", DIMS_70B, 0.01, batch=16,
                                    ctx_lo=4096, ctx_hi=32768),
    "llama2_7b_stack_cb": Workload("llama2_7b_stack_cb", DIMS_7B, 0.02, batch=64, ctx_lo=128,
                                   ctx_hi=4096, layers=32, steps=256, new_prefill=256),
}


def _gen(seed: int, tag: str, device=None) -> torch.Generator:
    """Generator of stream `tag` for a user seed (on the CPU, or on `device`).  Different
    tags give independent streams for the same seed (the seed is hashed with the tag), so
    two tensors can never be drawn from one stream by accident (e.g. an input equal to a
    scaled weight row).  A device generator draws other numbers than the CPU one for the
    same seed; each is reproducible on its own."""
    g = torch.Generator(device=device) if device is not None else torch.Generator()
    g.manual_seed(zlib.crc32(f"{tag}:{int(seed)}".encode()) * 2654435761 % (1 << 63))
    return g


def normal_bf16(shape, std: float, seed: int, tag: str = "normal", device=None) -> torch.Tensor:
    """BF16 tensor of N(0, std^2) draws (drawn in fp32, rounded to nearest BF16), on the
    CPU or, with `device`, drawn there by its own generator (for large inputs)."""
    t = torch.randn(*shape, generator=_gen(seed, tag, device), dtype=torch.float32,
                    device=device if device is not None else "cpu")
    if std != 1.0:
        t.mul_(std)
    return t.to(BF16)


def make_weights(d: LayerDims, w_std: float, seed: int, device=None) -> dict:
    """Canonical layer weights, all `[out, in]` row-major (drawn on `device` if given).

    w_qkv rows are [Q heads; K heads; V heads], each head `head_dim` rows.
    Gate and up are separate `[I, H]` matrices; w_down is `[H, I]`.
    """
    H, I = d.hidden, d.intermediate
    dev = device if device is not None else "cpu"
    gain = lambda tag: 1.0 + 0.1 * torch.randn(H, generator=_gen(seed, tag, device), dtype=torch.float32, device=dev)
    return {
        "w_qkv": normal_bf16((d.qkv_rows, H), w_std, seed, "w_qkv", device),
        "w_o": normal_bf16((H, d.n_heads * d.head_dim), w_std, seed, "w_o", device),
        "w_gate": normal_bf16((I, H), w_std, seed, "w_gate", device),
        "w_up": normal_bf16((I, H), w_std, seed, "w_up", device),
        "w_down": normal_bf16((H, I), w_std, seed, "w_down", device),
        "g_attn": gain("g_attn"),
        "g_ffn": gain("g_ffn"),
    }


def make_x(tokens: int, hidden: int, seed: int) -> torch.Tensor:
    return normal_bf16((tokens, hidden), 1.0, seed, "x")


def make_context_lens(batch: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    return torch.randint(lo, hi + 1, (batch,), generator=_gen(seed, "context_lens"), dtype=torch.int32)


def blocks_needed(tokens: int, block_size: int) -> int:
    return -(-int(tokens) // block_size)


def make_block_table(seq_tokens, block_size: int, seed: int, extra_blocks: int = 0,
                     width: int | None = None):
    """Shuffled, non-contiguous block table.

    seq_tokens[b] = cache capacity (tokens) sequence b needs.  Returns
    (block_table int32 [B, width] with -1 in unused entries, num_blocks) where
    num_blocks = sum of blocks needed + extra_blocks, and the physical ids come
    from one seeded random permutation of range(num_blocks).
    """
    need = [blocks_needed(t, block_size) for t in seq_tokens]
    num_blocks = sum(need) + int(extra_blocks)
    w = max(need) if width is None else int(width)
    perm = torch.randperm(num_blocks, generator=_gen(seed, "block_table")).to(torch.int32)
    table = torch.full((len(need), max(w, 1)), -1, dtype=torch.int32)
    at = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[at:at + n]
        at += n
    return table, num_blocks


def make_pool(num_blocks: int, d: LayerDims, seed: int, fill: str = "normal", device=None):
    """(k_pool, v_pool), each BF16 `[num_blocks, n_kv_heads, block_size, head_dim]`.

    fill="normal": N(0,1) draws (a pre-filled cache; drawn on `device` if given).
    fill="sentinel": every element is the BF16 value -1024.0, so untouched slots can be
    recognised.
    """
    shape = (num_blocks, d.n_kv_heads, d.block_size, d.head_dim)
    if fill == "normal":
        return normal_bf16(shape, 1.0, seed, "k_pool", device), normal_bf16(shape, 1.0, seed, "v_pool", device)
    if fill == "sentinel":
        return (torch.full(shape, -1024.0, dtype=BF16), torch.full(shape, -1024.0, dtype=BF16))
    raise ValueError(fill)


def make_pool_q8(num_blocks: int, d: LayerDims, seed: int):
    """A pre-filled INT8 pool: (k_codes, v_codes, k_scales, v_scales); codes int8
    `[num_blocks, n_kv_heads, block_size, head_dim]` uniform on -127..127, scales float32
    `[num_blocks, n_kv_heads, block_size]` uniform on [0.001, 0.031) (dequantised cache
    values of order 1, like the BF16 pools' N(0, 1))."""
    shape = (num_blocks, d.n_kv_heads, d.block_size, d.head_dim)
    codes = lambda tag: torch.randint(-127, 128, shape, generator=_gen(seed, tag), dtype=torch.int8)
    scales = lambda tag: torch.rand(shape[:3], generator=_gen(seed, tag), dtype=torch.float32) * 0.03 + 0.001
    return codes("k_codes"), codes("v_codes"), scales("k_scales"), scales("v_scales")


def prefill_positions(batch: int, seq_len: int, start: int = 0) -> torch.Tensor:
    """Positions start..start+seq_len-1 for each of `batch` sequences, token-major [B*S]."""
    return (torch.arange(seq_len, dtype=torch.int32) + start).repeat(batch)


def make_slot_mapping(tokens: int, num_slots: int, seed: int, n_skip: int = 0) -> torch.Tensor:
    """Distinct random destination slots for `tokens` tokens, drawn from range(num_slots);
    `n_skip` of them (at seeded random positions) are -1, meaning "write nothing"."""
    g = _gen(seed, "slot_mapping")
    slots = torch.randperm(num_slots, generator=g)[:tokens].to(torch.int32)
    if n_skip:
        idx = torch.randperm(tokens, generator=g)[:n_skip]
        slots[idx] = -1
    return slots


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("dataclasses", "torch")]
