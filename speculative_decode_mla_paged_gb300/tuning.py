"""Launch-shape defaults (host-side arithmetic only)."""
from __future__ import annotations

import math

NUM_SMS = 152          # GB300: 2 dies x 76 SMs


def default_num_splits(batch: int, max_q_per_req: int, num_heads: int, max_keys: int,
                       kernel: str = "tc") -> int:
    """Split count so the static grid covers about two waves of the 152 SMs.

    The grid is num_splits x row_tiles x batch; each split of a request needs
    enough keys (>= 256) to amortise loading its query tile.
    """
    rows_per_cta, ctas_per_sm = (16, 2) if kernel == "simt" else (128, 1)
    row_tiles = max(1, math.ceil(max_q_per_req * num_heads / rows_per_cta)) * max(1, batch)
    splits = math.ceil(2 * NUM_SMS * ctas_per_sm / row_tiles)
    splits = min(splits, max(1, max_keys // 256), 256)
    return max(1, splits)
