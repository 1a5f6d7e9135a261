"""GPU tests of the KV save ("The Launch Wrapper", section The KV Cache
Ordering Insight) through the C ABI: the save alone against the oracle's
definition (bit-exact), invalid slots, and the save fused in front of the
attention (verify_attn_save_and_run), eager and under graph capture."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decode_mla_paged_gb300 import api
from speculative_decode_mla_paged_gb300 import workloads as W

from gpu_helpers import META, as_rows, assert_parity, oracle_rows

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _new_rows(n, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((n, W.LATENT_DIM), generator=g) * 2.0).to(torch.bfloat16)


def test_save_kv_bit_exact():
    inp = W.make_config_inputs("short", device="cpu")
    pool_dev = inp.kv_pool.cuda()
    kv_new = _new_rows(inp.total_q, 11)
    loc = torch.from_numpy(inp.out_cache_loc).cuda()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.save_kv(kv_new.cuda(), loc, pool_dev, ws)
    torch.cuda.synchronize()
    want = oracle.save_kv(_bits(inp.kv_pool), inp.out_cache_loc, _bits(kv_new))
    assert api.read_status(ws) == 0
    assert np.array_equal(_bits(pool_dev), want)


def test_save_kv_strided_rows():
    inp = W.make_config_inputs("tiny", device="cpu")
    pool_dev = inp.kv_pool.cuda()
    wide = _new_rows(inp.total_q * 2, 12).reshape(inp.total_q, 2 * W.LATENT_DIM)
    kv_new = wide.cuda()[:, W.LATENT_DIM:]            # row stride 1152 elements
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.save_kv(kv_new, torch.from_numpy(inp.out_cache_loc).cuda(), pool_dev, ws)
    want = oracle.save_kv(_bits(inp.kv_pool), inp.out_cache_loc, _bits(wide[:, W.LATENT_DIM:].contiguous()))
    assert np.array_equal(_bits(pool_dev), want)


def test_save_kv_skips_invalid_slots():
    inp = W.make_config_inputs("tiny", device="cpu")
    pool_dev = inp.kv_pool.cuda()
    kv_new = _new_rows(inp.total_q, 13)
    loc = inp.out_cache_loc.copy()
    loc[2] = inp.pool_size            # outside the pool
    loc[5] = -3
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.save_kv(kv_new.cuda(), torch.from_numpy(loc).cuda(), pool_dev, ws)
    assert api.read_status(ws) & api.STATUS_BAD_SLOT
    keep = np.array([i for i in range(inp.total_q) if i not in (2, 5)])
    want = oracle.save_kv(_bits(inp.kv_pool), loc[keep], _bits(kv_new)[keep])
    assert np.array_equal(_bits(pool_dev), want)


def test_save_kv_empty_is_a_no_op():
    pool = torch.zeros((16, W.LATENT_DIM), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    api.save_kv(torch.zeros((0, W.LATENT_DIM), dtype=torch.bfloat16, device="cuda"),
                torch.zeros(0, dtype=torch.int64, device="cuda"), pool, ws)
    assert api.read_status(ws) == 0 and int(pool.abs().sum()) == 0


@pytest.mark.parametrize("name", ["tiny", "short"])
def test_save_and_run_matches_oracle_on_updated_pool(name):
    inp = W.make_config_inputs(name, device="cpu")
    kv_new = _new_rows(inp.total_q, 21)
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).cuda() for k in META}
    q, pool = inp.q.cuda(), inp.kv_pool.cuda()
    out = torch.full((inp.total_q, inp.num_heads, W.V_DIM), float("nan"), dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 4)
    runner(q, pool, d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"], d["custom_mask"],
           d["mask_indptr"], inp.sm_scale, out, kv_new=kv_new.cuda())
    torch.cuda.synchronize()
    assert runner.status() == 0
    new_bits = oracle.save_kv(_bits(inp.kv_pool), inp.out_cache_loc, _bits(kv_new))
    assert np.array_equal(_bits(pool), new_bits)
    inp.kv_pool = torch.from_numpy(new_bits.view(np.int16)).view(torch.bfloat16)
    assert_parity(as_rows(out), oracle_rows(inp), f"save+run {name}")


def test_save_and_run_graph_replay_sees_new_rows():
    """One captured graph (save + split + combine) replayed with different
    draft rows: every replay attends over the rows it saved."""
    inp = W.make_config_inputs("tiny", device="cpu")
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).cuda() for k in META}
    q, pool = inp.q.cuda(), inp.kv_pool.cuda()
    kv_new = torch.zeros((inp.total_q, W.LATENT_DIM), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((inp.total_q, inp.num_heads, W.V_DIM), dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 2)
    s = torch.cuda.Stream()
    call = lambda: runner(q, pool, d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
                          d["custom_mask"], d["mask_indptr"], inp.sm_scale, out, stream=s, kv_new=kv_new)
    with torch.cuda.stream(s):
        call()                                           # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for seed in (31, 32):
        rows = _new_rows(inp.total_q, seed)
        kv_new.copy_(rows)
        g.replay()
        torch.cuda.synchronize()
        assert runner.status() == 0
        host = inp
        new_bits = oracle.save_kv(_bits(inp.kv_pool), inp.out_cache_loc, _bits(rows))
        assert np.array_equal(_bits(pool), new_bits)
        ref_inp = W.make_config_inputs("tiny", device="cpu")
        ref_inp.kv_pool = torch.from_numpy(new_bits.view(np.int16)).view(torch.bfloat16)
        assert_parity(as_rows(out), oracle_rows(ref_inp), f"graph replay {seed}")
