"""Shared helpers for the GPU tests: move seeded inputs to the device, run the
library through its C ABI, and compare with the oracle under the parity bar
|got - ref| <= 1e-2 + 1e-2 * |ref| (per element)."""
import numpy as np
import torch

import oracle
from speculative_decode_mla_paged_gb300 import api

META = ("qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask", "mask_indptr")
ATOL = 1e-2
RTOL = 1e-2


def device_inputs(inp, dev="cuda"):
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).to(dev) for k in META}
    d["q"] = inp.q.to(dev)
    d["kv_pool"] = inp.kv_pool.to(dev)
    return d


def run(inp, impl="tc", num_splits=4, max_q=None, d=None, out=None):
    """Returns (out bf16 on device, status word)."""
    d = d if d is not None else device_inputs(inp)
    max_q = max_q if max_q is not None else max(1, inp.max_q_per_req)
    q = d["q"]
    runner = api.VerifyAttention(max(inp.batch, 1), max_q, inp.num_heads, num_splits, impl=impl)
    if out is None:
        out = torch.full((q.shape[0], q.shape[1], 512), float("nan"), dtype=torch.bfloat16, device=q.device)
    runner(q, d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
           d["custom_mask"], d["mask_indptr"], inp.sm_scale, out)
    torch.cuda.synchronize()
    return out, runner.status()


def as_rows(out):
    return out.float().cpu().numpy().astype(np.float64).reshape(-1, 512)


def assert_parity(got_rows, ref_rows, what=""):
    assert got_rows.shape == ref_rows.shape
    assert np.all(np.isfinite(got_rows)), f"{what}: non-finite outputs"
    excess = np.abs(got_rows - ref_rows) - (ATOL + RTOL * np.abs(ref_rows))
    worst = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= 0, (f"{what}: parity fails at row {worst[0]} col {worst[1]}: got "
                               f"{got_rows[worst]:.6f} ref {ref_rows[worst]:.6f}")


def sample_rows(inp, n_random=32, seed=0):
    """First and last row of every request plus random rows."""
    H = inp.num_heads
    rows = set()
    for b in range(inp.batch):
        t0, t1 = int(inp.qo_indptr[b]), int(inp.qo_indptr[b + 1])
        if t1 > t0:
            rows.update([t0 * H, t1 * H - 1])
    total = inp.total_q * H
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, total, size=min(n_random, total)).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def oracle_rows(inp, rows=None):
    out, _ = oracle.run(inp, rows=rows)
    return out
