"""Every output row of every full-size workload against the oracle.

The five workloads (tiny, short, mid, long, ragged) and the three extra ones
(chain verify, decode, a defragmented pool) at their full sizes, each run the
way the benchmark runs it: one call of the production path captured in a
CUDA graph and replayed after an L2 flush, at every split count the
benchmark chooses among (the grid simulation's four best candidates; the
benchmark keeps whichever it times fastest).  Each replay's whole output is
compared with the oracle's, element by element, under the parity bar
|got - ref| <= 1e-2 + 1e-2 |ref| ("The Cutover", section The Decision to Cut
Over: the new kernel matches the trusted path before it takes the traffic).
The oracle computes each workload once (about a minute in total on a
16-core host).
"""
import copy

import numpy as np
import pytest
import torch

from speculative_decode_mla_paged_gb300 import api, tuning
from speculative_decode_mla_paged_gb300 import workloads as W

from gpu_helpers import as_rows, assert_parity, device_inputs, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _init():
    api.init()


@pytest.mark.parametrize("name", W.CONFIG_ORDER + W.EXTRA_CONFIG_ORDER)
def test_every_row_at_full_size_as_bench_replays(name):
    inp = W.make_config_inputs(name, device="cuda")
    d = device_inputs(inp)
    host = copy.copy(inp)
    host.q, host.kv_pool = inp.q.cpu(), inp.kv_pool.cpu()
    ref = oracle_rows(host)                               # every row, [total_q * H, 512]
    assert ref.shape == (inp.total_q * inp.num_heads, 512)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    cands = tuning.ranked_num_splits(inp.prefix_lens, inp.draft_lens, inp.num_heads, k=4)
    for splits in cands:
        runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, splits)
        out = torch.full((inp.total_q, inp.num_heads, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
                       d["custom_mask"], d["mask_indptr"], inp.sm_scale, out)
        flush.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert runner.status() == 0, f"{name}/{splits}: status {runner.status():#x}"
        got = as_rows(out)
        assert np.all(np.isfinite(got)), f"{name}/{splits}: non-finite output"
        assert_parity(got, ref, f"{name}/graph replay/{splits} splits, every row")
        del g, runner, out
