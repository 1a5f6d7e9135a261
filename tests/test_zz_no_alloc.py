"""verify_attn_run_static: the entry point for callers that cannot allocate.

Engines that reserve nearly all GPU memory for their KV pool, plug-in hosts
that give a library no allocator, and paths where an allocation would
synchronise the device cannot hand verify_attn_run a workspace.  For them
the library carries a fixed 32 MiB scratch array and this entry point uses
it; verify_attn_static_status_word gives them the device address of that
array's status word.  These tests call both through the C ABI: two calls in
a row against the oracle and against the workspace entry point, the status
word after each, and a bad slot that a static-path caller must be able to
see.  The file is named to be collected last.
"""
import ctypes

import pytest
import torch

from speculative_decode_mla_paged_gb300 import api, build
from speculative_decode_mla_paged_gb300 import workloads as W

_p, _i64, _i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
STATIC_ARGS = [_p, _i64, _i64, _p, _i64, _p, _p, _p, _p, _p, _p, ctypes.c_float, _p, _i64, _i64,
               _i32, _i32, _i32, _i32, _p]
SCRATCH_LIMIT = 32 << 20


def _lib():
    build.build()
    lib = api.load_library()
    lib.verify_attn_run_static.argtypes = STATIC_ARGS
    lib.verify_attn_run_static.restype = _i32
    lib.verify_attn_static_status_word.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
    lib.verify_attn_static_status_word.restype = _i32
    return lib


def _call_static(lib, d, inp, out, max_q, splits, stream):
    v = lambda t: ctypes.c_void_p(t.data_ptr() if t.numel() else 0)
    return lib.verify_attn_run_static(
        v(d["q"]), d["q"].stride(0), d["q"].stride(1), v(d["kv_pool"]), d["kv_pool"].shape[0],
        v(d["qo_indptr"]), v(d["kv_indptr"]), v(d["kv_indices"]), v(d["out_cache_loc"]),
        v(d["custom_mask"]), v(d["mask_indptr"]), inp.sm_scale, v(out), out.stride(0), out.stride(1),
        inp.batch, max_q, inp.num_heads, splits, ctypes.c_void_p(stream))


def _status_word(lib):
    """The static path's status word, read on the current stream (a view of
    the library's device memory through __cuda_array_interface__, no copy
    into memory the test owns until .item())."""
    ptr = ctypes.c_void_p()
    rc = lib.verify_attn_static_status_word(ctypes.byref(ptr))
    assert rc == 0, api.status_string(rc)
    assert ptr.value and ptr.value % 256 == 0

    class _Word:
        __cuda_array_interface__ = {"shape": (1,), "typestr": "<i4", "data": (ptr.value, False),
                                    "strides": None, "version": 2}

    return int(torch.as_tensor(_Word(), device="cuda").item()) & 0xFFFFFFFF


def test_static_rejects_capacities_beyond_its_scratch():
    """Capacities needing more than the static array fail before any launch."""
    lib = _lib()
    A = 0x100000
    need = lib.verify_attn_workspace_size(64, 64, 64, 8)
    assert need > SCRATCH_LIMIT
    rc = lib.verify_attn_run_static(A, 64 * 576, 576, A, 4096, A, A, A, A, A, A, 0.07, A, 64 * 512, 512,
                                    64, 64, 64, 8, 0)
    assert rc == -9
    assert "32 MiB" in api.status_string(-9)


def test_static_status_word_rejects_a_null_out_pointer():
    assert _lib().verify_attn_static_status_word(None) == -1


@pytest.mark.gpu
def test_static_matches_oracle_and_workspace_entry_point_on_two_calls():
    from gpu_helpers import as_rows, assert_parity, device_inputs, oracle_rows

    lib = _lib()
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
        rc = _call_static(lib, d, inp, got, max_q, splits, stream)
        assert rc == 0, api.status_string(rc)
        assert _status_word(lib) == 0, f"static call {k}: status word set"
        torch.cuda.synchronize()
        assert_parity(as_rows(got), oracle_rows(inp), f"static call {k} vs oracle")
        assert_parity(as_rows(got), as_rows(ref), f"static call {k} vs verify_attn_run")


@pytest.mark.gpu
def test_static_caller_sees_a_bad_slot_then_a_clean_call():
    """A slot outside the pool sets VA_STATUS_BAD_SLOT in the static path's
    status word, where its caller can read it; the next good call clears it."""
    from gpu_helpers import as_rows, assert_parity, device_inputs, oracle_rows

    lib = _lib()
    api.init()
    stream = torch.cuda.current_stream().cuda_stream
    good = W.make_inputs([200, 30], [8, 4], 4, pool_size=1024, seed=42)
    bad = W.make_inputs([200, 30], [8, 4], 4, pool_size=1024, seed=42)
    bad.kv_indices = bad.kv_indices.copy()
    bad.kv_indices[17] = bad.pool_size + 5
    for inp, want in ((bad, api.STATUS_BAD_SLOT), (good, 0)):
        d = device_inputs(inp)
        out = torch.zeros(inp.total_q, inp.num_heads, 512, dtype=torch.bfloat16, device="cuda")
        rc = _call_static(lib, d, inp, out, 8, 3, stream)
        assert rc == 0, api.status_string(rc)
        status = _status_word(lib)
        assert status & api.STATUS_BAD_SLOT == want, f"status {status:#x}"
        if want == 0:
            torch.cuda.synchronize()
            assert_parity(as_rows(out), oracle_rows(inp), "good call after a bad one")
