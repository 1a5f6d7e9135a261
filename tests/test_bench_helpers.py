"""Host-side helpers of bench.py: the kernel-source key of the profile table,
the launch count per call, and the traffic lookup."""
import types

import bench


def test_code_text_ignores_comments_and_whitespace_only():
    a = '// header\nint f(int x) {  /* block\n comment */ return x + 1; }\nconst char *s = "a // b";\n'
    b = 'int f(int x){return x+1;}  // trailing\nconst char *s = "a // b";'
    c = 'int f(int x){return x+2;}\nconst char *s = "a // b";'
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
    assert '"a // b"' in bench.code_text(a)          # string contents are code


def test_kernel_hash_is_stable_and_keys_the_table():
    h = bench.kernel_hash("tc")
    assert len(h) == 12 and int(h, 16) >= 0
    assert bench.kernel_hash("tc") == h
    # the table either holds this exact source or yields no traffic figure
    t = bench.profiled_traffic("tc", "ragged")
    assert t is None or t > 0
    assert bench.profiled_traffic("tc", "no-such-workload") is None


def test_launches_per_call():
    cfg = lambda max_q, heads: types.SimpleNamespace(max_q_per_req=max_q, num_heads=heads)
    assert bench.launches_per_call(cfg(64, 8), "tc") == 3       # both cluster shapes + combine
    assert bench.launches_per_call(cfg(16, 8), "tc") == 2       # 2-CTA shape alone + combine
    assert bench.launches_per_call(cfg(1, 16), "tc") == 2
    assert bench.launches_per_call(cfg(64, 256), "tc") == 2     # every request above one tile
    assert bench.launches_per_call(cfg(64, 8), "simt") == 2


def test_ranked_num_splits_leads_with_the_plan():
    import numpy as np

    from speculative_decode_mla_paged_gb300 import tuning, workloads as W

    for name in ("ragged", "long", "decode", "short"):
        cfg = W.CONFIGS[name]
        prefix, drafts = W.draw_lengths(cfg, np.random.Generator(np.random.PCG64(cfg.seed + 7919)))
        r = tuning.ranked_num_splits(prefix, drafts, cfg.num_heads, k=4)
        assert r[0] == tuning.plan_num_splits(prefix, drafts, cfg.num_heads)
        assert 1 <= len(r) <= 4 and len(set(r)) == len(r)
