"""Launch-shape planning (host-side arithmetic only; no attention math).

The split kernels run a static grid of units (key split x row tile x
request); ``num_splits`` is a host capacity that fixes it ("The Capture-Safe
Kernel", Decision 3).  These helpers pick it for a known workload by
simulating how the units fill the GPU.
"""
from __future__ import annotations

import heapq
import math
from typing import Sequence

NUM_SMS = 152                  # GB300: 2 dies x 76 SMs
TC_CLUSTERS = 36               # 4-CTA clusters of the tensor-core kernel resident at once on a GB300
                               # (a cluster stays inside one GPC: 144 of the 152 SMs)
TC_CLUSTERS_ONE_TILE = 76      # 2-CTA clusters resident at once (the shape used when T * H <= 128)
TC_TILE_ROWS = 128             # rows per row tile of the tensor-core kernel
KEY_ALIGN = 128                # must match the library's split chunk rule
MIN_CHUNK = 256
CANDIDATES = tuple(range(1, 65)) + (72, 80, 96, 108, 128, 144, 160, 192, 256)


def split_chunk(n: int, num_splits: int) -> int:
    """Keys per split: max(ceil(n / S), 256) rounded up to 128 (the library's rule)."""
    c = max(-(-n // num_splits), MIN_CHUNK)
    return -(-c // KEY_ALIGN) * KEY_ALIGN


def splits_used(n: int, num_splits: int) -> int:
    return 0 if n <= 0 else -(-n // split_chunk(n, num_splits))


def simulate(prefix_lens: Sequence[int], draft_lens: Sequence[int], num_heads: int, num_splits: int,
             kernel: str = "tc") -> float:
    """Estimated time of one call in units of one key tile of a unit.

    Units are dispatched in grid order (row group fastest, then split, then
    request) onto the concurrent slots (tensor-core kernel: 36 four-CTA
    clusters of 256 rows, or 76 two-CTA clusters of 128 rows when every
    request has T * H <= 128, 128-key tiles; CUDA-core kernel: 304 CTAs of 16
    rows, 32-key tiles); each costs its key tiles plus a fixed start-up (query
    load, pipeline fill, partial write).  The combine's workspace traffic is
    added on top.
    """
    max_q = max(draft_lens) if len(draft_lens) else 0
    if kernel == "simt":
        rows, slots, overhead, tile_keys, tile_cost, tile_s = 16, 2 * NUM_SMS, 2.0, 32, 1.0, 0.5e-6
    elif max_q * num_heads <= TC_TILE_ROWS:
        rows, slots, overhead, tile_keys, tile_cost, tile_s = TC_TILE_ROWS, TC_CLUSTERS_ONE_TILE, 4.0, 128, 1.0, 2.5e-6
    else:
        rows, slots, overhead, tile_keys, tile_cost, tile_s = 2 * TC_TILE_ROWS, TC_CLUSTERS, 4.0, 128, 1.0, 2.5e-6
    max_tiles = math.ceil(max_q * num_heads / rows)
    free = [0.0] * slots
    heapq.heapify(free)
    finish = 0.0
    total_rows_splits = 0
    for l, t in zip(prefix_lens, draft_lens):
        n = int(l) + int(t)
        r_tiles = math.ceil(int(t) * num_heads / rows)
        used = splits_used(n, num_splits)
        chunk = split_chunk(n, num_splits) if n > 0 else 0
        total_rows_splits += int(t) * num_heads * used
        for s in range(num_splits):
            keys = max(0, min(n, (s + 1) * chunk) - s * chunk) if s < used else 0
            for rt in range(max_tiles):
                cost = (overhead + tile_cost * math.ceil(keys / tile_keys)) if (rt < r_tiles and keys) else 0.05
                t0 = heapq.heappop(free)
                heapq.heappush(free, t0 + cost)
                finish = max(finish, t0 + cost)
    # combine: each used split's fp32 partial row (2 KB) written then read at ~6.8 TB/s
    combine = total_rows_splits * 2048 * 2 / 6.8e12 / tile_s
    return finish + combine


def _candidates(prefix_lens: Sequence[int], draft_lens: Sequence[int]):
    """Split counts worth simulating: every candidate up to the point where a
    larger count no longer changes the longest request's chunk."""
    n_max = max(int(l) + int(t) for l, t in zip(prefix_lens, draft_lens))
    for s in CANDIDATES:
        if s > 1 and split_chunk(n_max, s) == split_chunk(n_max, s - 1) and s > n_max // MIN_CHUNK + 1:
            break
        yield s


def plan_num_splits(prefix_lens: Sequence[int], draft_lens: Sequence[int], num_heads: int,
                    kernel: str = "tc") -> int:
    """The candidate split count with the smallest simulated time."""
    best, best_s = None, 1
    for s in _candidates(prefix_lens, draft_lens):
        cost = simulate(prefix_lens, draft_lens, num_heads, s, kernel)
        if best is None or cost < best * 0.98:
            best, best_s = cost, s
    return best_s


def ranked_num_splits(prefix_lens: Sequence[int], draft_lens: Sequence[int], num_heads: int, k: int = 4,
                      kernel: str = "tc") -> list:
    """The k candidate split counts with the smallest simulated times, best
    first (the planner's pick leads).  The simulation tracks measured times
    closely for calls of one cluster shape; when a call runs both shapes the
    two grids interleave in ways it does not model, so these are candidates
    to time (``api.tune_num_splits``), not an answer."""
    costs = sorted((simulate(prefix_lens, draft_lens, num_heads, s, kernel), s)
                   for s in _candidates(prefix_lens, draft_lens))
    plan = plan_num_splits(prefix_lens, draft_lens, num_heads, kernel)
    out = [plan] + [s for _, s in costs if s != plan]
    return out[:max(1, k)]


def default_num_splits(batch: int, max_q_per_req: int, num_heads: int, max_keys: int,
                       kernel: str = "tc") -> int:
    """Split count for a uniform batch of `batch` requests of max_keys keys each."""
    return plan_num_splits([max_keys - max_q_per_req] * max(1, batch), [max_q_per_req] * max(1, batch),
                           num_heads, kernel)
