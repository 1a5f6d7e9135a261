"""GPU tests of the validate mode: the production kernel cross-checked
against the CUDA-core kernel on the same live buffers ("The Launch Wrapper",
section The Design Decision: Three Modes of Operation)."""
import numpy as np
import pytest
import torch

from speculative_decode_mla_paged_gb300 import api
from speculative_decode_mla_paged_gb300 import workloads as W

from gpu_helpers import META

pytestmark = pytest.mark.gpu


def _call(runner, inp, d, out):
    return runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
                  d["custom_mask"], d["mask_indptr"], inp.sm_scale, out)


def _dev(inp):
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).cuda() for k in META}
    d["q"], d["kv_pool"] = inp.q.cuda(), inp.kv_pool.cuda()
    return d


@pytest.mark.parametrize("name", ["short", "mid", "chain", "decode"])
def test_validate_mode_agrees(name):
    inp = W.make_config_inputs(name, device="cuda")
    d = _dev(inp)
    out = torch.empty((inp.total_q, inp.num_heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 8, validate=True)
    _call(runner, inp, d, out)
    rec = runner.last_validation
    assert rec is not None and rec["against"] == "simt"
    assert rec["ok"], rec


def test_validate_mode_from_environment(monkeypatch):
    monkeypatch.setenv("VERIFY_ATTN_VALIDATE", "1")
    inp = W.make_config_inputs("tiny", device="cpu")
    d = _dev(inp)
    out = torch.empty((inp.total_q, inp.num_heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 2)
    assert runner.validate
    _call(runner, inp, d, out)
    assert runner.last_validation["ok"]


def test_validate_mode_flags_a_mismatch():
    """The check compares the output the caller received with a fresh run of
    the other kernel: an output that no kernel produced must be flagged."""
    inp = W.make_config_inputs("tiny", device="cpu")
    d = _dev(inp)
    out = torch.empty((inp.total_q, inp.num_heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 2, validate=False)
    _call(runner, inp, d, out)
    out += 1.0
    with pytest.warns(UserWarning):
        runner._cross_check(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                            d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], inp.sm_scale, out, None)
    assert not runner.last_validation["ok"]


def test_validate_mode_on_a_stream_that_is_not_current():
    """With an explicit stream both kernels and the comparison run on it, so
    the check reads finished outputs."""
    inp = W.make_config_inputs("mid", device="cuda")
    d = _dev(inp)
    out = torch.empty((inp.total_q, inp.num_heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 8, validate=True)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
           d["custom_mask"], d["mask_indptr"], inp.sm_scale, out, stream=side)
    rec = runner.last_validation
    assert rec["ok"], rec
    torch.cuda.current_stream().wait_stream(side)
    assert runner.status() == 0
