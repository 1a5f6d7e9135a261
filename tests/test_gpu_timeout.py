"""The kernels' failure path, run on purpose without a fault: every wait in
the split kernels is bounded and, when it expires, sets STATUS_TIMEOUT and
returns ("The Launch Wrapper", section The Design Decision: Three Modes of
Operation: a failure must leave the service able to fall back).  The
library's self-test entry point runs that same bounded wait on a barrier
nothing arrives on, with a short limit; the tests check that it returns
after about the limit, that the status bit is set, and that the context
then serves normal calls that match the oracle."""
import ctypes
import time

import pytest
import torch

from speculative_decode_mla_paged_gb300 import api, build
from speculative_decode_mla_paged_gb300 import workloads as W


def _lib():
    build.build()
    return api.load_library()


def test_wait_probe_rejects_bad_arguments_on_the_host():
    lib = _lib()
    A = ctypes.c_void_p(0x100000)
    assert lib.verify_attn_check_wait_timeout(10**6, None, 256, None) == -1           # null workspace
    assert lib.verify_attn_check_wait_timeout(10**6, ctypes.c_void_p(0x100010), 256, None) == -2
    assert lib.verify_attn_check_wait_timeout(10**6, A, 255, None) == -4              # under 256 bytes
    assert lib.verify_attn_check_wait_timeout(999, A, 256, None) == -3                # limit below 1 us
    assert lib.verify_attn_check_wait_timeout(10**9 + 1, A, 256, None) == -3          # above 1 s


@pytest.mark.gpu
@pytest.mark.parametrize("limit_ms", [2, 30])
def test_bounded_wait_expires_sets_timeout_and_the_next_call_is_correct(limit_ms):
    from gpu_helpers import as_rows, assert_parity, oracle_rows, run

    api.init()
    ws = torch.full((256,), 0xFF, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    api.check_wait_timeout(limit_ms * 1_000_000, ws)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    status = api.read_status(ws)
    assert status == api.STATUS_TIMEOUT, f"status {status:#x}"     # cleared, then only the timeout bit
    assert limit_ms / 1e3 <= elapsed < limit_ms / 1e3 + 2.0, elapsed
    # the context is usable: a normal call on both cluster shapes matches the oracle
    inp = W.make_inputs([900, 300], [24, 8], 8, 4096, seed=93)
    out, st = run(inp, num_splits=3)
    assert st == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"call after a {limit_ms} ms timeout")
