"""Continuous batching over a stack of decoder layers on one GPU.

Host-side logic from the pages, driving the C-ABI layer calls:

* paged KV-cache management (page "ATB KV-cache paging, quantisation,
  speculative decoding and communication overlap", section "KV Cache memory
  wall"): fixed-size blocks handed out on demand from a free list, a
  block_table per request mapping its logical blocks to physical ones, blocks
  of a finished request returned to the free list at once and reused in any
  order;
* the continuous-batching scheduler (page "ATB: whole decoder-layer fusion",
  section "graph execution engine"): a running set of requests, each step
  allocating what every request needs (a KV slot) and recycling a finished
  request's resources immediately to admit a new one.

One block table serves every layer: layer l keeps its own K/V pool, indexed by
the same physical block ids.  Each step first prefills the newly admitted
requests (all layers, one batched prefill call per layer), then runs one decode
step for every slot through all layers (one decode call per layer; this part
can be captured once as a CUDA graph and replayed with the tables updated in
place).  Every computation runs in the library's kernels; this module only
moves indices.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import synth


class BlockAllocator:
    """LIFO free list of physical KV blocks (seeded initial order)."""

    def __init__(self, num_blocks: int, seed: int):
        g = torch.Generator()
        g.manual_seed(int(seed))
        self.num_blocks = int(num_blocks)
        self._free = torch.randperm(self.num_blocks, generator=g).tolist()
        self._used = set()

    def free_count(self) -> int:
        return len(self._free)

    def alloc(self, n: int) -> list:
        if n > len(self._free):
            raise MemoryError(f"KV pool exhausted: need {n} blocks, {len(self._free)} free")
        out = [self._free.pop() for _ in range(n)]
        self._used.update(out)
        return out

    def free(self, blocks) -> None:
        for b in blocks:
            if b not in self._used:
                raise ValueError(f"block {b} freed twice or never allocated")
            self._used.remove(b)
            self._free.append(b)


@dataclasses.dataclass
class Request:
    rid: int
    ctx: int              # tokens in the cache
    budget: int           # decode tokens still to produce
    blocks: list


class Scheduler:
    """Slots, budgets and the block table (host side, numpy)."""

    def __init__(self, n_slots: int, block_size: int, max_blocks: int, allocator: BlockAllocator,
                 seed: int, budget_max: int = 256, prompt_len: int = 256):
        self.n_slots, self.bs, self.max_blocks = n_slots, block_size, max_blocks
        self.alloc = allocator
        self.prompt_len, self.budget_max = prompt_len, budget_max
        self.rng = np.random.default_rng(seed)
        self.table = np.full((n_slots, max_blocks), -1, np.int32)
        self.slots: list = [None] * n_slots
        self.next_rid = 0

    def _new_budget(self) -> int:
        return int(self.rng.integers(1, self.budget_max + 1))

    def _set_blocks(self, slot: int, blocks: list) -> None:
        if len(blocks) > self.max_blocks:
            raise ValueError("request outgrew the block table width")
        self.table[slot, :] = -1
        self.table[slot, :len(blocks)] = blocks

    def start_resident(self, slot: int, ctx: int) -> Request:
        """A request whose first `ctx` tokens are already cached (pre-filled pool)."""
        blocks = self.alloc.alloc(-(-ctx // self.bs))
        r = Request(self.next_rid, ctx, self._new_budget(), blocks)
        self.next_rid += 1
        self.slots[slot] = r
        self._set_blocks(slot, blocks)
        return r

    def retire_and_admit(self) -> list:
        """Frees every finished request's blocks and admits a new request in its slot.
        Returns the slots that need a prefill of `prompt_len` tokens this step."""
        admitted = []
        for s, r in enumerate(self.slots):
            if r is not None and r.budget > 0:
                continue
            if r is not None:
                self.alloc.free(r.blocks)
            blocks = self.alloc.alloc(-(-self.prompt_len // self.bs))
            nr = Request(self.next_rid, self.prompt_len, self._new_budget(), blocks)
            self.next_rid += 1
            self.slots[s] = nr
            self._set_blocks(s, blocks)
            admitted.append(s)
        return admitted

    def grow_for_decode(self) -> np.ndarray:
        """Every slot appends one token: a block is added when the new position starts one.
        Returns context_lens (int32) including the appended token."""
        ctx = np.empty(self.n_slots, np.int32)
        for s, r in enumerate(self.slots):
            pos = r.ctx                       # position of the appended token
            if pos % self.bs == 0 and pos // self.bs >= len(r.blocks):
                r.blocks += self.alloc.alloc(1)
                self._set_blocks(s, r.blocks)
            r.ctx += 1
            r.budget -= 1
            ctx[s] = r.ctx
        return ctx


class StackEngine:
    """The GPU side: L layers (packed weights, K/V pools) and device copies of the tables."""

    def __init__(self, api, cfgs, packed, pools, n_slots, max_blocks, max_prefill_tokens,
                 device="cuda"):
        self.api = api
        self.cfgs, self.packed, self.pools = cfgs, packed, pools
        self.n_slots = n_slots
        cfg = cfgs[0]
        self.H = cfg.hidden
        self.table = torch.full((n_slots, max_blocks), -1, dtype=torch.int32, device=device)
        self.ctx = torch.zeros(n_slots, dtype=torch.int32, device=device)
        self.ws = api.new_workspace(cfg, max(n_slots, max_prefill_tokens), max_blocks, device)
        self.status = api.new_status(device)
        self.x = torch.zeros(n_slots, self.H, dtype=torch.bfloat16, device=device)
        self.bufs = [torch.empty(n_slots, self.H, dtype=torch.bfloat16, device=device) for _ in range(2)]
        self.pf_x = torch.empty(max_prefill_tokens, self.H, dtype=torch.bfloat16, device=device)
        self.pf_bufs = [torch.empty(max_prefill_tokens, self.H, dtype=torch.bfloat16, device=device)
                        for _ in range(2)]
        self.pf_pos = torch.empty(max_prefill_tokens, dtype=torch.int32, device=device)
        self.pf_table = torch.full((n_slots, max_blocks), -1, dtype=torch.int32, device=device)
        self.graph = None
        self.y = None

    def prefill(self, n_req, prompt_len, stream):
        """All layers over the n_req requests whose rows are in pf_table[:n_req] and whose
        inputs are in pf_x[:n_req * prompt_len]."""
        T = n_req * prompt_len
        src = self.pf_x[:T]
        for l in range(len(self.cfgs)):
            dst = self.pf_bufs[l & 1][:T]
            k, v = self.pools[l]
            self.api.layer_prefill(self.cfgs[l], self.packed[l], src, self.pf_pos[:T], n_req, prompt_len,
                                   k, v, self.pf_table[:n_req], y=dst, workspace=self.ws,
                                   status=self.status, stream=stream)
            src = dst
        return src

    def _decode_layers(self, stream):
        src = self.x
        for l in range(len(self.cfgs)):
            dst = self.bufs[l & 1]
            k, v = self.pools[l]
            self.api.layer_decode_step(self.cfgs[l], self.packed[l], src, k, v, self.table, self.ctx,
                                       y=dst, workspace=self.ws, status=self.status, stream=stream)
            src = dst
        return src

    def capture_decode(self, stream):
        """Records the all-layer decode step once as a CUDA graph (replayed by decode())."""
        with torch.cuda.stream(stream):
            self.y = self._decode_layers(stream)      # warm-up outside the capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            self.y = self._decode_layers(stream)
        self.graph = g

    def decode(self, stream):
        if self.graph is not None:
            with torch.cuda.stream(stream):
                self.graph.replay()
            return self.y
        self.y = self._decode_layers(stream)
        return self.y


def kv_blocks_needed(ctx_hi: int, n_slots: int, steps: int, prompt_len: int, block_size: int) -> int:
    """A pool size that covers the resident contexts, their growth over `steps` steps and
    the admitted requests' prompts, with head room for block rounding."""
    per_slot = -(-(ctx_hi + steps + prompt_len) // block_size) + 2
    return n_slots * per_slot


__all__ = ["BlockAllocator", "Request", "Scheduler", "StackEngine", "kv_blocks_needed"]
