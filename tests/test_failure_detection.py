"""Failure detection without a GPU fault: a bounded in-kernel wait that nothing
completes must time out, report LL_DEV_TIMEOUT through the status word and let
the kernel finish, after which the context keeps working."""
import ctypes
import time

import pytest
import torch

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from transformer_decoder_layer_llama_gb300 import api


def test_bounded_wait_times_out_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    rc = api.lib.ll_selftest_bounded_wait(20000, ctypes.c_void_p(status.data_ptr()),
                                          ctypes.c_void_p(out.data_ptr()),
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == api.LL_OK
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 10.0
    assert int(status.item()) == api.LL_DEV_TIMEOUT
    assert int(out.item()) == 64              # every waiting thread gave up and returned
    # the context is intact: ordinary work still runs and is right
    x = torch.ones(64, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(128, 256, dtype=torch.bfloat16, device="cuda")
    y = api.linear(x, w)
    torch.cuda.synchronize()
    assert float(y.float().mean()) == 256.0


def test_selftest_rejects_bad_limits():
    null = ctypes.c_void_p(0)
    assert api.lib.ll_selftest_bounded_wait(0, null, null, null) == api.LL_ERR_INVALID_ARG
