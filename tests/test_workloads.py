"""CPU tests of the seeded input generator: tree shapes, slot assignment,
packed ancestor masks, bf16 rounding, the configuration table and the work
counts, each checked against an independent construction or a hand count."""
import math

import numpy as np
import pytest
import torch

from speculative_decode_mla_paged_gb300 import workloads as W


def _dense_masks(inp):
    """Per request, the bool [T, N] visibility matrix unpacked from the packed mask."""
    bits = np.unpackbits(inp.custom_mask, bitorder="little")
    out = []
    for b in range(inp.batch):
        t, l = int(inp.draft_lens[b]), int(inp.prefix_lens[b])
        lo = int(inp.mask_indptr[b])
        out.append(bits[lo: lo + t * (l + t)].reshape(t, l + t).astype(bool))
    return out


def test_random_tree_parents_point_to_the_root_or_earlier_drafts():
    rng = np.random.Generator(np.random.PCG64(3))
    for t in (1, 2, 8, 64):
        p = W.random_tree(rng, t)
        assert p.shape == (t,)
        assert all(-1 <= p[i] <= i - 1 for i in range(t))
    # every choice of {root} U [0, i-1] occurs
    assert {int(W.random_tree(rng, 4)[3]) for _ in range(400)} == {-1, 0, 1, 2}


def test_ancestors_or_self_hand_example():
    # root -> 0 -> 1 and root -> 2 -> 3
    vis = W.ancestors_or_self(np.array([-1, 0, -1, 2]))
    expect = np.array([[1, 0, 0, 0], [1, 1, 0, 0], [0, 0, 1, 0], [0, 0, 1, 1]], dtype=bool)
    assert (vis == expect).all()
    assert (W.ancestors_or_self(W.chain_tree(5)) == np.tril(np.ones((5, 5), dtype=bool))).all()


def test_make_inputs_metadata_follows_the_recipe():
    inp = W.make_inputs([37, 0, 300], [5, 3, 9], 4, 1024, seed=11)
    assert list(inp.kv_indptr) == [0, 37, 37, 337]
    assert list(inp.qo_indptr) == [0, 5, 8, 17]
    assert inp.kv_indices.dtype == np.int32 and inp.out_cache_loc.dtype == np.int64
    slots = np.concatenate([inp.kv_indices.astype(np.int64), inp.out_cache_loc])
    assert len(np.unique(slots)) == len(slots)          # every token owns its own slot
    assert slots.min() >= 0 and slots.max() < inp.pool_size
    assert list(np.diff(inp.mask_indptr)) == [5 * 42, 3 * 3, 9 * 309]
    for b, m in enumerate(_dense_masks(inp)):
        l = int(inp.prefix_lens[b])
        assert m[:, :l].all()                            # the whole prefix is visible
        assert (m[:, l:] == W.ancestors_or_self(inp.parents[b])).all()
    assert inp.q.shape == (17, 4, 576) and inp.q.dtype == torch.bfloat16
    assert inp.kv_pool.shape == (1024, 576) and inp.kv_pool.dtype == torch.bfloat16


def test_pack_tree_masks_equals_bitwise_packing():
    """The packed-form builder (all ones, then clear the invisible bits)
    agrees with packing the dense matrices one bit at a time, with a custom
    prefix part and rows that start inside a byte."""
    rng = np.random.Generator(np.random.PCG64(5))
    prefix = [3, 0, 17]
    parents = [W.random_tree(rng, t) for t in (5, 2, 7)]
    pre = [rng.random((len(p), l)) < 0.5 for l, p in zip(prefix, parents)]
    packed, indptr = W.pack_tree_masks(prefix, parents, lambda b, t, l: pre[b])
    dense = [np.concatenate([pre[b], W.ancestors_or_self(p)], axis=1) for b, p in enumerate(parents)]
    flat = np.concatenate([d.reshape(-1) for d in dense])
    ref = np.zeros((len(flat) + 7) // 8, dtype=np.uint8)
    for n, v in enumerate(flat):                         # bit n: byte n >> 3, position n & 7
        if v:
            ref[n >> 3] |= 1 << (n & 7)
    assert (packed == ref).all()
    assert list(indptr) == [0, 40, 44, 212]
    p2, i2 = W.pack_mask(dense)
    assert (p2 == ref).all() and (i2 == indptr).all()


def test_bf16_rounding_matches_torch():
    rng = np.random.Generator(np.random.PCG64(9))
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1.0, -0.0, 0.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 65504.0, 1e-30], np.float32)])
    ours = W.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (ours == ref).all()
    # the two ties round to even: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    assert W.bf16_bits_to_f32(ours[-4:-2]).tolist() == [1.0, 1 + 2 ** -6]
    assert np.allclose(W.bf16_bits_to_f32(ours), x, rtol=2 ** -8, atol=0)


def test_configuration_table():
    rows = {  # name: (B, prefix lengths, draft lengths, H, pool, seed, q scale)
        "tiny": (1, [256], [8], 8, 4096, 0, 1.0),
        "short": (1, [5760], [16], 8, 65536, 1, 1.0),
        "mid": (4, [23040] * 4, [32] * 4, 8, 131072, 2, 1.0),
        "long": (1, [92160], [64], 64, 131072, 3, 3.0),
    }
    for name, row in rows.items():
        c = W.CONFIGS[name]
        assert (c.batch, list(c.prefix_lens), list(c.draft_lens), c.num_heads, c.pool_size, c.seed,
                c.q_scale) == row, name
        assert c.sm_scale == 1 / math.sqrt(192)
    c = W.CONFIGS["ragged"]
    assert (c.batch, c.num_heads, c.pool_size, c.seed) == (8, 8, 1_500_000, 4)
    prefix, drafts = W.draw_lengths(c, np.random.Generator(np.random.PCG64(c.seed + 7919)))
    assert len(prefix) == 8 and prefix[0] == 185000 and ((prefix >= 1024) & (prefix <= 185000)).all()
    assert len(drafts) == 8 and set(drafts.tolist()) <= {16, 32, 64}
    assert prefix.sum() + drafts.sum() <= c.pool_size
    d = W.CONFIGS["decode"]
    prefix, drafts = W.draw_lengths(d, np.random.Generator(np.random.PCG64(d.seed + 7919)))
    assert len(prefix) == 32 and prefix[0] == 32768 and ((prefix >= 1024) & (prefix <= 32768)).all()
    assert (drafts == 1).all() and d.num_heads == 16


def test_ragged_prefix_lengths_are_log_uniform():
    c = W.CONFIGS["ragged"]
    rng = np.random.Generator(np.random.PCG64(1))
    logs = np.concatenate([np.log(W.draw_lengths(c, rng)[0][1:]) for _ in range(300)])
    u = (logs - math.log(1024)) / (math.log(185000) - math.log(1024))
    # uniform on [0, 1]: mean 1/2, variance 1/12 (2100 draws; bounds ~5 sigma)
    assert abs(u.mean() - 0.5) < 0.03 and abs(u.var() - 1 / 12) < 0.01


@pytest.mark.parametrize("slots", ["random", "contiguous", "runs:16"])
def test_slot_layouts(slots):
    order = W.slot_order(np.random.Generator(np.random.PCG64(2)), 1000, 300, slots)
    assert sorted(order.tolist()) == list(range(1000))   # a permutation of the pool
    if slots == "contiguous":
        assert (np.diff(order[:300]) == 1).all()          # the used keys form one run
    elif slots == "runs:16":
        # runs of 16 consecutive slots (the last one 8), each starting at a multiple of 16
        for i in range(len(order)):
            if order[i] % 16:
                assert i > 0 and order[i - 1] == order[i] - 1


def test_work_counts():
    inp = W.make_inputs([40, 7], [6, 3], 5, 512, seed=4)
    pairs = sum(int(m.sum()) for m in _dense_masks(inp)) * 5
    expect = sum(int(t) * int(l) + int(W.ancestors_or_self(p).sum())
                 for l, t, p in zip(inp.prefix_lens, inp.draft_lens, inp.parents))
    assert inp.visible_pairs() == pairs == expect * 5
    assert inp.algorithmic_flops() == 2 * (576 + 512) * pairs
    # B = 1, L = 2, T = 1, H = 1 by hand: 3 KV rows (3456 B), q (1152), out
    # (1024), 2 prefix indices (8), 1 draft slot (8), 3 mask bits (1 byte),
    # indptrs 2 x (4 + 4 + 8) (32)
    assert W.make_inputs([2], [1], 1, 16, seed=0).algorithmic_bytes() == 5681
