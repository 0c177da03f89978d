"""ctypes binding of libllamalayer.so (include/llama_layer.h), names as in the C ABI.

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, then their device pointers go to the library; every step of the
layer runs in the library's CUDA kernels.  Importing this module loads the
library and fails loudly if it has not been built (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

LL_OK = 0
LL_ERR_INVALID_ARG = 1
LL_ERR_UNSUPPORTED = 2
LL_ERR_WORKSPACE = 3
LL_ERR_CUDA = 4

LL_MODE_FUSED = 0
LL_MODE_STEP_BY_STEP = 1

LL_DEV_BAD_BLOCK = 1
LL_DEV_BAD_SLOT = 2
LL_DEV_BAD_POSITION = 4
LL_DEV_TIMEOUT = 8

EXPORTED = [
    "ll_strerror", "ll_last_error", "ll_packed_weights_size", "ll_pack_weights", "ll_workspace_size",
    "ll_layer_prefill", "ll_layer_decode_step", "ll_reshape_and_cache",
    "ll_attention_workspace_size", "ll_paged_attention_decode", "ll_linear_workspace_size",
    "ll_linear", "ll_device_sm_count", "ll_trace_begin", "ll_trace_end", "ll_trace_elapsed_ms",
    "ll_trace_name", "ll_paged_attention_decode_noalloc", "ll_selftest_bounded_wait",
    "ll_workspace_checkpoints", "ll_reshape_and_cache_q8", "ll_paged_attention_decode_q8",
    "ll_layer_decode_step_q8", "ll_workspace_size_mode", "ll_workspace_step_checkpoints",
    "ll_layer_prefill_mode", "ll_layer_decode_step_mode", "ll_set_prefill_attention_ctas",
]


class ll_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("intermediate", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_position", ctypes.c_int32), ("rms_eps", ctypes.c_float),
                ("rope_theta", ctypes.c_float)]


class ll_weights(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w_gate", ctypes.c_void_p),
                ("w_up", ctypes.c_void_p), ("w_down", ctypes.c_void_p),
                ("g_attn", ctypes.c_void_p), ("g_ffn", ctypes.c_void_p)]


class ll_kv_pool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("num_blocks", ctypes.c_int32)]


class ll_kv_pool_q8(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("num_blocks", ctypes.c_int32)]


class ll_checkpoints(ctypes.Structure):
    _fields_ = [("x_hat", ctypes.c_size_t), ("q", ctypes.c_size_t), ("o", ctypes.c_size_t),
                ("h", ctypes.c_size_t), ("h_hat", ctypes.c_size_t), ("a", ctypes.c_size_t)]


class ll_step_checkpoints(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("qkv", "k", "v", "slots", "o_proj", "gate_up", "down")]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    cfgp = ctypes.POINTER(ll_config)
    poolp = ctypes.POINTER(ll_kv_pool)
    sig = {
        "ll_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "ll_last_error": (ctypes.c_char_p, []),
        "ll_packed_weights_size": (S, [cfgp]),
        "ll_pack_weights": (ctypes.c_int, [cfgp, ctypes.POINTER(ll_weights), P, S, P]),
        "ll_workspace_size": (S, [cfgp, I32, I32]),
        "ll_layer_prefill": (ctypes.c_int, [cfgp, P, P, P, I32, I32, poolp, P, I32, P, P, S, P, P]),
        "ll_layer_decode_step": (ctypes.c_int, [cfgp, P, P, poolp, P, I32, P, I32, P, P, S, P, P]),
        "ll_reshape_and_cache": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, poolp, P, P]),
        "ll_attention_workspace_size": (S, [I32, I32, I32, I32, I32]),
        "ll_paged_attention_decode": (ctypes.c_int, [P, poolp, P, I32, P, I32, I32, I32, I32, I32,
                                                     ctypes.c_float, P, P, S, P, P]),
        "ll_paged_attention_decode_noalloc": (ctypes.c_int, [P, poolp, P, I32, P, I32, I32, I32, I32,
                                                             I32, ctypes.c_float, P, P, P]),
        "ll_linear_workspace_size": (S, [I32, I32, I32]),
        "ll_linear": (ctypes.c_int, [P, P, P, I32, I32, I32, P, S, P, P]),
        "ll_device_sm_count": (ctypes.c_int, []),
        "ll_set_prefill_attention_ctas": (ctypes.c_int, [I32]),
        "ll_trace_begin": (ctypes.c_int, [I32]),
        "ll_trace_end": (I32, []),
        "ll_trace_elapsed_ms": (ctypes.c_float, [I32]),
        "ll_trace_name": (ctypes.c_char_p, [I32]),
        "ll_selftest_bounded_wait": (ctypes.c_int, [I32, P, P, P]),
        "ll_workspace_checkpoints": (ctypes.c_int, [cfgp, I32, I32, ctypes.POINTER(ll_checkpoints)]),
        "ll_reshape_and_cache_q8": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, ctypes.POINTER(ll_kv_pool_q8),
                                                   P, P]),
        "ll_paged_attention_decode_q8": (ctypes.c_int, [P, ctypes.POINTER(ll_kv_pool_q8), P, I32, P, I32, I32, I32,
                                                        I32, I32, ctypes.c_float, P, P, S, P, P]),
        "ll_layer_decode_step_q8": (ctypes.c_int, [cfgp, P, P, ctypes.POINTER(ll_kv_pool_q8), P, I32, P, I32, P, P,
                                                   S, P, P]),
        "ll_workspace_size_mode": (S, [cfgp, I32, I32, I32]),
        "ll_workspace_step_checkpoints": (ctypes.c_int, [cfgp, I32, I32, ctypes.POINTER(ll_step_checkpoints)]),
        "ll_layer_prefill_mode": (ctypes.c_int, [cfgp, P, P, P, I32, I32, poolp, P, I32, P, P, S, P, I32, P]),
        "ll_layer_decode_step_mode": (ctypes.c_int, [cfgp, P, P, poolp, P, I32, P, I32, P, P, S, P, I32, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class LayerError(RuntimeError):
    def __init__(self, name, code):
        detail = lib.ll_last_error().decode()
        super().__init__(f"{name}: {lib.ll_strerror(code).decode()} (code {code})"
                         + (f" -- {detail}" if detail else ""))
        self.code = code


def _check(name, rc):
    if rc != LL_OK:
        raise LayerError(name, rc)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, device=True, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must live on the GPU")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def make_config(dims, max_position: int) -> ll_config:
    """ll_config from any object with the layer's dimension attributes."""
    return ll_config(dims.hidden, dims.n_heads, dims.n_kv_heads, dims.head_dim, dims.intermediate,
                     dims.block_size, int(max_position), float(dims.rms_eps), float(dims.rope_theta))


def new_status(device=None):
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def packed_weights_size(cfg: ll_config) -> int:
    return lib.ll_packed_weights_size(ctypes.byref(cfg))


def pack_weights(cfg: ll_config, W: dict, stream=None) -> torch.Tensor:
    """Packs canonical weights (dict of CUDA tensors, see include/llama_layer.h) into a new
    uint8 CUDA buffer and returns it."""
    H, I, d = cfg.hidden, cfg.intermediate, cfg.head_dim
    _need(W["w_qkv"], "w_qkv", torch.bfloat16, shape=((cfg.n_heads + 2 * cfg.n_kv_heads) * d, H))
    _need(W["w_o"], "w_o", torch.bfloat16, shape=(H, cfg.n_heads * d))
    _need(W["w_gate"], "w_gate", torch.bfloat16, shape=(I, H))
    _need(W["w_up"], "w_up", torch.bfloat16, shape=(I, H))
    _need(W["w_down"], "w_down", torch.bfloat16, shape=(H, I))
    _need(W["g_attn"], "g_attn", torch.float32, shape=(H,))
    _need(W["g_ffn"], "g_ffn", torch.float32, shape=(H,))
    n = packed_weights_size(cfg)
    if n == 0:
        raise LayerError("ll_packed_weights_size", LL_ERR_UNSUPPORTED)
    packed = torch.empty(n, dtype=torch.uint8, device=W["w_qkv"].device)
    w = ll_weights(W["w_qkv"].data_ptr(), W["w_o"].data_ptr(), W["w_gate"].data_ptr(),
                   W["w_up"].data_ptr(), W["w_down"].data_ptr(), W["g_attn"].data_ptr(),
                   W["g_ffn"].data_ptr())
    _check("ll_pack_weights", lib.ll_pack_weights(ctypes.byref(cfg), ctypes.byref(w), _ptr(packed),
                                                  n, _stream(stream)))
    return packed


def workspace_size(cfg: ll_config, max_tokens: int, max_blocks: int, mode: int = LL_MODE_FUSED) -> int:
    if mode == LL_MODE_FUSED:
        return lib.ll_workspace_size(ctypes.byref(cfg), int(max_tokens), int(max_blocks))
    return lib.ll_workspace_size_mode(ctypes.byref(cfg), int(max_tokens), int(max_blocks), int(mode))


def new_workspace(cfg, max_tokens, max_blocks, device=None, mode=LL_MODE_FUSED):
    n = workspace_size(cfg, max_tokens, max_blocks, mode)
    if n == 0:
        raise LayerError("ll_workspace_size", LL_ERR_INVALID_ARG)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def checkpoints(cfg: ll_config, workspace: torch.Tensor, max_tokens: int, max_blocks: int, tokens: int) -> dict:
    """Views into `workspace` (allocated by new_workspace(cfg, max_tokens, max_blocks)) of the
    intermediates the last layer call over `tokens` tokens left there: x_hat, q, o, h_hat, a
    (BF16) and h (float32), each [tokens, features].  Read them after the call has finished
    on its stream; the next call on the workspace overwrites them."""
    out = ll_checkpoints()
    rc = lib.ll_workspace_checkpoints(ctypes.byref(cfg), int(max_tokens), int(max_blocks), ctypes.byref(out))
    if rc != 0:
        raise LayerError("ll_workspace_checkpoints", rc)
    if not 0 < tokens <= max_tokens:
        raise ValueError("tokens must be in 1..max_tokens")
    nq = cfg.n_heads * cfg.head_dim
    shapes = {"x_hat": (cfg.hidden, torch.bfloat16), "q": (nq, torch.bfloat16), "o": (nq, torch.bfloat16),
              "h": (cfg.hidden, torch.float32), "h_hat": (cfg.hidden, torch.bfloat16),
              "a": (cfg.intermediate, torch.bfloat16)}
    views = {}
    for name, (width, dt) in shapes.items():
        off = getattr(out, name)
        nbytes = tokens * width * torch.finfo(dt).bits // 8
        views[name] = workspace[off:off + nbytes].view(dt).view(tokens, width)
    return views


def step_checkpoints(cfg: ll_config, workspace: torch.Tensor, max_tokens: int, max_blocks: int,
                     tokens: int) -> dict:
    """Views into a step-by-step workspace (new_workspace(..., mode=LL_MODE_STEP_BY_STEP)) of
    the intermediates that mode adds, after a call over `tokens` tokens: qkv (float32, packed
    column order), k, v (BF16), slots (int32), o_proj, gate_up (interleaved), down (float32)."""
    out = ll_step_checkpoints()
    rc = lib.ll_workspace_step_checkpoints(ctypes.byref(cfg), int(max_tokens), int(max_blocks), ctypes.byref(out))
    if rc != 0:
        raise LayerError("ll_workspace_step_checkpoints", rc)
    if not 0 < tokens <= max_tokens:
        raise ValueError("tokens must be in 1..max_tokens")
    nqkv = (cfg.n_heads + 2 * cfg.n_kv_heads) * cfg.head_dim
    nkv = cfg.n_kv_heads * cfg.head_dim
    shapes = {"qkv": ((nqkv,), torch.float32), "k": ((nkv,), torch.bfloat16), "v": ((nkv,), torch.bfloat16),
              "slots": ((), torch.int32), "o_proj": ((cfg.hidden,), torch.float32),
              "gate_up": ((2 * cfg.intermediate,), torch.float32), "down": ((cfg.hidden,), torch.float32)}
    views = {}
    for name, (width, dt) in shapes.items():
        off = getattr(out, name)
        count = tokens * (width[0] if width else 1)
        nbytes = count * (torch.finfo(dt).bits if dt.is_floating_point else torch.iinfo(dt).bits) // 8
        views[name] = workspace[off:off + nbytes].view(dt).view(tokens, *width)
    return views


def _pool(k_pool, v_pool):
    _need(k_pool, "k_pool", torch.bfloat16)
    _need(v_pool, "v_pool", torch.bfloat16)
    if k_pool.shape != v_pool.shape or k_pool.dim() != 4:
        raise ValueError("k_pool and v_pool must both be [num_blocks, n_kv_heads, block_size, head_dim]")
    return ll_kv_pool(k_pool.data_ptr(), v_pool.data_ptr(), k_pool.shape[0])


def layer_prefill(cfg, packed, x, positions, batch, seq_len, k_pool, v_pool, block_table,
                  y=None, workspace=None, status=None, stream=None, mode=LL_MODE_FUSED):
    """ll_layer_prefill (ll_layer_prefill_mode for another mode).  Returns y (BF16
    [batch*seq_len, hidden])."""
    T = int(batch) * int(seq_len)
    _need(x, "x", torch.bfloat16, shape=(T, cfg.hidden))
    _need(positions, "positions", torch.int32, shape=(T,))
    _need(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] < batch:
        raise ValueError("block_table must be [batch, max_blocks]")
    pool = _pool(k_pool, v_pool)
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = new_workspace(cfg, T, block_table.shape[1], x.device, mode)
    if status is None:
        status = new_status(x.device)
    args = (ctypes.byref(cfg), _ptr(packed), _ptr(x), _ptr(positions), int(batch), int(seq_len),
            ctypes.byref(pool), _ptr(block_table), block_table.shape[1], _ptr(y), _ptr(workspace),
            workspace.numel(), _ptr(status))
    if mode == LL_MODE_FUSED:
        _check("ll_layer_prefill", lib.ll_layer_prefill(*args, _stream(stream)))
    else:
        _check("ll_layer_prefill_mode", lib.ll_layer_prefill_mode(*args, int(mode), _stream(stream)))
    return y


def layer_decode_step(cfg, packed, x, k_pool, v_pool, block_table, context_lens, y=None,
                      workspace=None, status=None, stream=None, mode=LL_MODE_FUSED):
    """ll_layer_decode_step (ll_layer_decode_step_mode for another mode).  Returns y (BF16
    [batch, hidden])."""
    B = x.shape[0]
    _need(x, "x", torch.bfloat16, shape=(B, cfg.hidden))
    _need(context_lens, "context_lens", torch.int32, shape=(B,))
    _need(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] < B:
        raise ValueError("block_table must be [batch, max_blocks]")
    pool = _pool(k_pool, v_pool)
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = new_workspace(cfg, B, block_table.shape[1], x.device, mode)
    if status is None:
        status = new_status(x.device)
    args = (ctypes.byref(cfg), _ptr(packed), _ptr(x), ctypes.byref(pool), _ptr(block_table),
            block_table.shape[1], _ptr(context_lens), B, _ptr(y), _ptr(workspace), workspace.numel(),
            _ptr(status))
    if mode == LL_MODE_FUSED:
        _check("ll_layer_decode_step", lib.ll_layer_decode_step(*args, _stream(stream)))
    else:
        _check("ll_layer_decode_step_mode", lib.ll_layer_decode_step_mode(*args, int(mode), _stream(stream)))
    return y


def layer_decode_step_q8(cfg, packed, x, pool, block_table, context_lens, y=None, workspace=None, status=None,
                         stream=None):
    """ll_layer_decode_step_q8 over an INT8 pool (PoolQ8).  Returns y (BF16 [batch, hidden])."""
    B = x.shape[0]
    _need(x, "x", torch.bfloat16, shape=(B, cfg.hidden))
    _need(context_lens, "context_lens", torch.int32, shape=(B,))
    _need(block_table, "block_table", torch.int32)
    if block_table.dim() != 2 or block_table.shape[0] < B:
        raise ValueError("block_table must be [batch, max_blocks]")
    cp = pool.c()
    if y is None:
        y = torch.empty_like(x)
    if workspace is None:
        workspace = new_workspace(cfg, B, block_table.shape[1], x.device)
    if status is None:
        status = new_status(x.device)
    _check("ll_layer_decode_step_q8", lib.ll_layer_decode_step_q8(
        ctypes.byref(cfg), _ptr(packed), _ptr(x), ctypes.byref(cp), _ptr(block_table), block_table.shape[1],
        _ptr(context_lens), B, _ptr(y), _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)))
    return y


def reshape_and_cache(k, v, slot_mapping, k_pool, v_pool, status=None, stream=None):
    """ll_reshape_and_cache: k, v BF16 [tokens, n_kv_heads, head_dim]."""
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16, shape=tuple(k.shape))
    T, Hkv, d = k.shape
    _need(slot_mapping, "slot_mapping", torch.int32, shape=(T,))
    pool = _pool(k_pool, v_pool)
    if status is None:
        status = new_status(k.device)
    _check("ll_reshape_and_cache", lib.ll_reshape_and_cache(
        _ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, d, k_pool.shape[2], ctypes.byref(pool),
        _ptr(status), _stream(stream)))
    return status


class PoolQ8:
    """An INT8 KV pool on the GPU: codes k, v int8 [num_blocks, n_kv_heads, block_size,
    head_dim] and float32 scales k_scale, v_scale [num_blocks, n_kv_heads, block_size]."""

    def __init__(self, k, v, k_scale, v_scale):
        _need(k, "k codes", torch.int8)
        _need(v, "v codes", torch.int8, shape=tuple(k.shape))
        _need(k_scale, "k_scale", torch.float32, shape=tuple(k.shape[:3]))
        _need(v_scale, "v_scale", torch.float32, shape=tuple(k.shape[:3]))
        self.k, self.v, self.k_scale, self.v_scale = k, v, k_scale, v_scale

    @classmethod
    def empty(cls, num_blocks, n_kv_heads, block_size, head_dim, device="cuda"):
        shape = (num_blocks, n_kv_heads, block_size, head_dim)
        return cls(torch.zeros(shape, dtype=torch.int8, device=device),
                   torch.zeros(shape, dtype=torch.int8, device=device),
                   torch.zeros(shape[:3], dtype=torch.float32, device=device),
                   torch.zeros(shape[:3], dtype=torch.float32, device=device))

    @property
    def block_size(self):
        return self.k.shape[2]

    def c(self):
        return ll_kv_pool_q8(self.k.data_ptr(), self.v.data_ptr(), self.k_scale.data_ptr(),
                             self.v_scale.data_ptr(), self.k.shape[0])


def reshape_and_cache_q8(k, v, slot_mapping, pool: PoolQ8, status=None, stream=None):
    """ll_reshape_and_cache_q8: k, v BF16 [tokens, n_kv_heads, head_dim] quantised into pool."""
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16, shape=tuple(k.shape))
    T, Hkv, d = k.shape
    _need(slot_mapping, "slot_mapping", torch.int32, shape=(T,))
    cp = pool.c()
    if status is None:
        status = new_status(k.device)
    _check("ll_reshape_and_cache_q8", lib.ll_reshape_and_cache_q8(
        _ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, d, pool.block_size, ctypes.byref(cp),
        _ptr(status), _stream(stream)))
    return status


def paged_attention_decode_q8(q, pool: PoolQ8, block_table, context_lens, scale, out=None, workspace=None,
                              status=None, stream=None):
    """ll_paged_attention_decode_q8: q BF16 [batch, n_heads, 128] over an INT8 pool."""
    _need(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32, shape=(B,))
    Hkv, bs = pool.k.shape[1], pool.block_size
    mb = block_table.shape[1]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(max(attention_workspace_size(B, Hq, d, mb, bs), 16), dtype=torch.uint8,
                                device=q.device)
    if status is None:
        status = new_status(q.device)
    cp = pool.c()
    _check("ll_paged_attention_decode_q8", lib.ll_paged_attention_decode_q8(
        _ptr(q), ctypes.byref(cp), _ptr(block_table), mb, _ptr(context_lens), B, Hq, Hkv, d, bs,
        float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _ptr(status), _stream(stream)))
    return out


def attention_workspace_size(batch, n_heads, head_dim, max_blocks, block_size):
    return lib.ll_attention_workspace_size(batch, n_heads, head_dim, max_blocks, block_size)


def paged_attention_decode(q, k_pool, v_pool, block_table, context_lens, scale, out=None,
                           workspace=None, status=None, stream=None):
    """ll_paged_attention_decode: q BF16 [batch, n_heads, head_dim]."""
    _need(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32, shape=(B,))
    pool = _pool(k_pool, v_pool)
    bs = k_pool.shape[2]
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        n = attention_workspace_size(B, Hq, d, block_table.shape[1], bs)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device)
    if status is None:
        status = new_status(q.device)
    _check("ll_paged_attention_decode", lib.ll_paged_attention_decode(
        _ptr(q), ctypes.byref(pool), _ptr(block_table), block_table.shape[1], _ptr(context_lens), B,
        Hq, k_pool.shape[1], d, bs, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
        _ptr(status), _stream(stream)))
    return out


def paged_attention_decode_noalloc(q, k_pool, v_pool, block_table, context_lens, scale, out=None,
                                   status=None, stream=None):
    """ll_paged_attention_decode_noalloc: as paged_attention_decode, but the library keeps
    the split partials in its own fixed device array, so no workspace is passed or made."""
    _need(q, "q", torch.bfloat16)
    B, Hq, d = q.shape
    _need(block_table, "block_table", torch.int32)
    _need(context_lens, "context_lens", torch.int32, shape=(B,))
    pool = _pool(k_pool, v_pool)
    if out is None:
        out = torch.empty_like(q)
    if status is None:
        status = new_status(q.device)
    _check("ll_paged_attention_decode_noalloc", lib.ll_paged_attention_decode_noalloc(
        _ptr(q), ctypes.byref(pool), _ptr(block_table), block_table.shape[1], _ptr(context_lens), B,
        Hq, k_pool.shape[1], d, k_pool.shape[2], float(scale), _ptr(out), _ptr(status),
        _stream(stream)))
    return out


def set_prefill_attention_ctas(n: int) -> None:
    """ll_set_prefill_attention_ctas: bound on the persistent prefill attention's CTAs
    (n <= 0: one per SM)."""
    lib.ll_set_prefill_attention_ctas(int(n))


def linear(x, w, y=None, workspace=None, status=None, stream=None):
    """ll_linear: y = x w^T, x BF16 [m, k], w BF16 [n, k]."""
    _need(x, "x", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    m, k = x.shape
    n = w.shape[0]
    if w.shape[1] != k:
        raise ValueError("w must be [n, k]")
    if y is None:
        y = torch.empty(m, n, dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(lib.ll_linear_workspace_size(m, n, k), dtype=torch.uint8,
                                device=x.device)
    if status is None:
        status = new_status(x.device)
    _check("ll_linear", lib.ll_linear(_ptr(x), _ptr(w), _ptr(y), m, n, k, _ptr(workspace),
                                      workspace.numel(), _ptr(status), _stream(stream)))
    return y


class trace:
    """Context manager over ll_trace_begin/ll_trace_end: records every kernel launch the
    library makes inside the block.  After the stream is synchronised, `launches()`
    returns [(kernel name, milliseconds), ...] in launch order."""

    def __init__(self, capacity=4096):
        self.capacity = capacity
        self.count = 0

    def __enter__(self):
        _check("ll_trace_begin", lib.ll_trace_begin(self.capacity))
        return self

    def __exit__(self, *exc):
        self.count = lib.ll_trace_end()
        return False

    def launches(self):
        return [(lib.ll_trace_name(i).decode(), lib.ll_trace_elapsed_ms(i)) for i in range(self.count)]
