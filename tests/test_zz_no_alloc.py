"""verify_attn_run_static: the entry point for callers that cannot allocate.

Engines that reserve nearly all GPU memory for their KV pool, plug-in hosts
that give a library no allocator, and paths where an allocation would
synchronise the device cannot hand verify_attn_run a workspace.  For them
the library carries a fixed 32 MiB scratch array and this entry point uses
it.  These tests call it through the C ABI and compare it with the
workspace entry point.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decode_mla_paged_gb300 import api, build
from speculative_decode_mla_paged_gb300 import workloads as W

_p, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
STATIC_ARGS = [_p, _i64, _i64, _p, _i64, _p, _p, _p, _p, _p, _p, ctypes.c_float, _p, _i64, _i64,
               _i32, _i32, _i32, _i32, _p]
SCRATCH_LIMIT = 32 << 20


def _static_fn():
    build.build()
    lib = api.load_library()
    fn = lib.verify_attn_run_static
    fn.argtypes = STATIC_ARGS
    fn.restype = _i32
    return fn


def _call_static(fn, d, inp, out, max_q, splits, stream):
    v = lambda t: ctypes.c_void_p(t.data_ptr() if t.numel() else 0)
    return fn(v(d["q"]), d["q"].stride(0), d["q"].stride(1), v(d["kv_pool"]), d["kv_pool"].shape[0],
              v(d["qo_indptr"]), v(d["kv_indptr"]), v(d["kv_indices"]), v(d["out_cache_loc"]),
              v(d["custom_mask"]), v(d["mask_indptr"]), inp.sm_scale, v(out), out.stride(0),
              out.stride(1), inp.batch, max_q, inp.num_heads, splits, ctypes.c_void_p(stream))


def test_static_rejects_capacities_beyond_its_scratch():
    """Capacities needing more than the static array fail before any launch."""
    fn = _static_fn()
    A = 0x100000
    need = api.load_library().verify_attn_workspace_size(64, 64, 64, 8)
    assert need > SCRATCH_LIMIT
    rc = fn(A, 64 * 576, 576, A, 4096, A, A, A, A, A, A, 0.07, A, 64 * 512, 512, 64, 64, 64, 8, 0)
    assert rc == -9
    assert "32 MiB" in api.status_string(-9)


@pytest.mark.gpu
def test_static_matches_workspace_entry_point_on_two_calls():
    from gpu_helpers import as_rows, assert_parity, device_inputs

    fn = _static_fn()
    api.init()
    stream = torch.cuda.current_stream().cuda_stream
    cases = [(W.make_inputs([300, 41, 7], [16, 9, 4], 8, pool_size=2048, seed=40, q_scale=2.0), 16, 6),
             (W.make_inputs([1000], [5], 8, pool_size=2048, seed=41), 8, 3)]
    for k, (inp, max_q, splits) in enumerate(cases):
        d = device_inputs(inp)
        shape = (inp.total_q, inp.num_heads, 512)
        ref = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        got = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        runner = api.VerifyAttention(inp.batch, max_q, inp.num_heads, splits)
        runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
               d["custom_mask"], d["mask_indptr"], inp.sm_scale, ref)
        rc = _call_static(fn, d, inp, got, max_q, splits, stream)
        assert rc == 0, api.status_string(rc)
        torch.cuda.synchronize()
        assert_parity(as_rows(got), as_rows(ref), f"static call {k}")
