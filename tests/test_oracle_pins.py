"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test names the mistake class it is there to catch.  All run on the CPU.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from speculative_decode_mla_paged_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(W.to_bf16_bits(np.asarray(x, np.float32)).view(np.int16)).view(torch.bfloat16)


def _f64(t: torch.Tensor) -> np.ndarray:
    return t.float().double().numpy()


def _visible_closure(parents):
    """Ancestor-or-self sets by dynamic programming over the parent list
    (independent of the generator's walk-up loop)."""
    sets = []
    for i, p in enumerate(parents):
        sets.append((set(sets[p]) if p >= 0 else set()) | {i})
    return sets


def _dense_request(inp, b, prefix_vis=None):
    """Gather request b's keys/values/mask densely, straight from the slot lists."""
    l0, l1 = int(inp.kv_indptr[b]), int(inp.kv_indptr[b + 1])
    t0, t1 = int(inp.qo_indptr[b]), int(inp.qo_indptr[b + 1])
    slots = list(inp.kv_indices[l0:l1]) + list(inp.out_cache_loc[t0:t1])
    pool = inp.kv_pool.float().double()
    keys = pool[torch.tensor(np.asarray(slots, dtype=np.int64))] if slots else pool[:0]
    L, T = l1 - l0, t1 - t0
    vis = np.zeros((T, L + T), dtype=bool)
    vis[:, :L] = True if prefix_vis is None else prefix_vis
    for i, s in enumerate(_visible_closure(list(inp.parents[b]))):
        for j in s:
            vis[i, L + j] = True
    return keys, torch.from_numpy(vis)


def _sdpa_reference(inp, prefix_vis=None):
    """torch SDPA (float64, explicit boolean mask) per request -> [total_q*H, 512]."""
    outs = []
    for b in range(inp.batch):
        t0, t1 = int(inp.qo_indptr[b]), int(inp.qo_indptr[b + 1])
        if t1 == t0:
            continue
        keys, vis = _dense_request(inp, b, None if prefix_vis is None else prefix_vis[b])
        q = inp.q[t0:t1].float().double().transpose(0, 1)           # [H, T, 576]
        k = keys.unsqueeze(0).expand(inp.num_heads, -1, -1)          # [H, N, 576]
        v = keys[:, :512].unsqueeze(0).expand(inp.num_heads, -1, -1)
        o = F.scaled_dot_product_attention(q, k, v, attn_mask=vis.unsqueeze(0), scale=inp.sm_scale)
        outs.append(o.transpose(0, 1).reshape(-1, 512))
    return torch.cat(outs).numpy()


# ---------------------------------------------------------------- mask layout

def _read_fixture():
    fx = {}
    with open(os.path.join(GOLDEN, "packed_mask_two_requests.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            fx[key] = vals
    return fx


def test_mask_fixture_packing():
    """Generator packs the hand-derived fixture bit for bit (bit order, row-major, no padding)."""
    fx = _read_fixture()
    parents = [np.array([int(v) for v in fx["parents0"]]), np.array([int(v) for v in fx["parents1"]])]
    packed, indptr = W.pack_tree_masks([int(v) for v in fx["prefix_lens"]], parents)
    assert [int(v) for v in indptr] == [int(v) for v in fx["mask_indptr"]]
    assert bytes(packed) == bytes(int(v, 16) for v in fx["bytes"])


def test_mask_fixture_oracle_decode():
    """Oracle decodes the fixture's raw bytes into the fixture's visible sets.

    q = 0 gives every visible key the same weight; key j of each request has a
    one-hot V on dim j, so out[d] = 1/|visible| exactly on the visible keys.
    Catches a wrong bit order, a transposed mask, or a wrong mask offset.
    """
    fx = _read_fixture()
    prefix = [int(v) for v in fx["prefix_lens"]]
    drafts = [len(fx["parents0"]), len(fx["parents1"])]
    H = 2
    pool = np.zeros((16, 576), np.float32)
    kv_indices, ocl, slot = [], [], 0
    for b in range(2):
        for j in range(prefix[b] + drafts[b]):
            pool[slot, j] = 1.0
            (kv_indices if j < prefix[b] else ocl).append(slot)
            slot += 1
    qo = np.array([0, drafts[0], drafts[0] + drafts[1]], np.int32)
    kvp = np.array([0, prefix[0], prefix[0] + prefix[1]], np.int32)
    mask = np.array([int(v, 16) for v in fx["bytes"]], np.uint8)
    mip = np.array([int(v) for v in fx["mask_indptr"]], np.int64)
    q = np.zeros((sum(drafts), H, 576), np.float32)
    out, lse = oracle.verify_attn(_bf16(q), _bf16(pool), qo, kvp, np.array(kv_indices, np.int32),
                                  np.array(ocl, np.int64), mask, mip, W.SM_SCALE, H)
    expect_sets = [[set(map(int, s.split(","))) for s in fx["visible0"]],
                   [set(map(int, s.split(","))) for s in fx["visible1"]]]
    row = 0
    for b in range(2):
        for i in range(drafts[b]):
            vis = expect_sets[b][i]
            for h in range(H):
                expect = np.zeros(512)
                for j in vis:
                    expect[j] = 1.0 / len(vis)
                np.testing.assert_allclose(out[row], expect, rtol=0, atol=1e-15)
                assert lse[row] == pytest.approx(np.log(len(vis)), abs=1e-15)
                row += 1


# ---------------------------------------------------------------- library routine pins

@pytest.mark.parametrize("seed", [0, 1])
def test_matches_sdpa_on_ragged_batch(seed):
    """Whole definition vs torch SDPA (float64) on a ragged batch with random prefix masks.

    Catches: dropped RoPE dims, wrong scale or sign, wrong slot / indptr
    indexing, V taken from the wrong dims, wrong mask column order.
    """
    rng = np.random.default_rng(100 + seed)
    prefix = [0, 5, 37, 64]
    drafts = [3, 4, 9, 1]
    pvis = [rng.random((t, l)) < 0.6 for l, t in zip(prefix, drafts)]
    inp = W.make_inputs(prefix, drafts, num_heads=3, pool_size=256, seed=seed, q_scale=2.0,
                        extra_prefix_mask=lambda b, t, l: pvis[b])
    ref = _sdpa_reference(inp, prefix_vis=pvis)
    out, _ = oracle.run(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_chain_tree_is_causal_attention():
    """A chain tree (parent[i] = i-1) is standard causal attention: the drafts are
    positions L..L+T-1 of one sequence.  Reference: SDPA with is_causal over the
    whole sequence, last T rows.  Catches a transposed or shifted draft mask."""
    L, T, H = 21, 7, 2
    inp = W.make_inputs([L], [T], num_heads=H, pool_size=64, seed=5, tree="chain")
    slots = list(inp.kv_indices) + list(inp.out_cache_loc)
    seq = inp.kv_pool.float().double()[torch.tensor(np.asarray(slots, np.int64))]   # [N, 576]
    qfull = torch.randn(L + T, H, 576, dtype=torch.float64)
    qfull[L:] = inp.q.float().double()
    o = F.scaled_dot_product_attention(qfull.transpose(0, 1), seq.expand(H, -1, -1),
                                       seq[:, :512].expand(H, -1, -1), is_causal=True,
                                       scale=inp.sm_scale)
    ref = o.transpose(0, 1)[L:].reshape(-1, 512).numpy()
    out, _ = oracle.run(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_all_ones_mask_is_full_attention():
    """Every bit set: plain (unmasked) SDPA over prefix + drafts."""
    L, T, H = 30, 5, 2
    full = lambda b, t, l: np.ones((t, l), bool)
    inp = W.make_inputs([L], [T], num_heads=H, pool_size=64, seed=6, tree="star",
                        extra_prefix_mask=full)
    nbits = int(inp.mask_indptr[-1])
    inp.custom_mask = np.packbits(np.ones(nbits, np.uint8), bitorder="little")
    slots = list(inp.kv_indices) + list(inp.out_cache_loc)
    seq = inp.kv_pool.float().double()[torch.tensor(np.asarray(slots, np.int64))]
    q = inp.q.float().double().transpose(0, 1)
    o = F.scaled_dot_product_attention(q, seq.expand(H, -1, -1), seq[:, :512].expand(H, -1, -1),
                                       scale=inp.sm_scale)
    ref = o.transpose(0, 1).reshape(-1, 512).numpy()
    out, _ = oracle.run(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_single_visible_key_returns_its_v_exactly():
    """One visible key: weight exactly 1, out = pool[slot, :512] bit for bit, lse = its score."""
    L, T, H = 40, 6, 4
    inp = W.make_inputs([L], [T], num_heads=H, pool_size=128, seed=7)
    N = L + T
    rng = np.random.default_rng(7)
    pick = rng.integers(0, N, size=T)
    bits = np.zeros((T, N), bool)
    bits[np.arange(T), pick] = True
    inp.custom_mask = np.packbits(bits.reshape(-1).astype(np.uint8), bitorder="little")
    out, lse = oracle.run(inp)
    pool = inp.kv_pool.float().double().numpy()
    slots = np.concatenate([inp.kv_indices, inp.out_cache_loc]).astype(np.int64)
    q = inp.q.float().double().numpy()
    for i in range(T):
        slot = slots[pick[i]]
        for h in range(H):
            r = i * H + h
            assert np.array_equal(out[r], pool[slot, :512])
            s = inp.sm_scale * float(np.dot(q[i, h], pool[slot]))
            assert lse[r] == pytest.approx(s, rel=1e-13, abs=1e-13)


def test_two_keys_differing_only_in_rope_dims():
    """Two visible keys whose scores differ only through the 64 RoPE dims (512..575).

    Closed form: weights are the logistic of the scaled score difference.
    Catches a score that drops the RoPE part, a wrong sm_scale, or V taken
    from dims other than 0..511."""
    H, sc = 1, W.SM_SCALE
    pool = np.zeros((4, 576), np.float32)
    pool[1, 540] = 2.0; pool[1, 3] = 1.0; pool[1, 575] = 5.0   # key 0 (slot 1); dim 575 is not V
    pool[2, 7] = 1.0                                           # key 1 (slot 2, draft)
    q = np.zeros((1, H, 576), np.float32); q[0, 0, 540] = 1.5; q[0, 0, 575] = 0.25
    qo = np.array([0, 1], np.int32); kvp = np.array([0, 1], np.int32)
    mask = np.packbits(np.array([1, 1], np.uint8), bitorder="little")
    out, lse = oracle.verify_attn(_bf16(q), _bf16(pool), qo, kvp, np.array([1], np.int32),
                                  np.array([2], np.int64), mask, np.array([0, 2], np.int64), sc, H)
    s0 = sc * (1.5 * 2.0 + 0.25 * 5.0)
    w0 = 1.0 / (1.0 + np.exp(-s0))
    expect = np.zeros(512); expect[3] = w0; expect[7] = 1 - w0
    np.testing.assert_allclose(out[0], expect, rtol=1e-14, atol=1e-15)
    assert lse[0] == pytest.approx(np.log(np.exp(s0) + 1.0), rel=1e-14)


def test_zero_query_gives_mean_of_visible_values():
    """q = 0: uniform weights, out = mean of the visible V rows."""
    L, T, H = 17, 5, 2
    inp = W.make_inputs([L], [T], num_heads=H, pool_size=64, seed=8)
    inp.q = torch.zeros_like(inp.q)
    out, lse = oracle.run(inp)
    pool = inp.kv_pool.float().double().numpy()
    sets = _visible_closure(list(inp.parents[0]))
    for i in range(T):
        slots = list(inp.kv_indices) + [int(inp.out_cache_loc[j]) for j in sorted(sets[i])]
        mean = pool[slots, :512].mean(axis=0)
        for h in range(H):
            np.testing.assert_allclose(out[i * H + h], mean, rtol=1e-13, atol=1e-14)
            assert lse[i * H + h] == pytest.approx(np.log(len(slots)), rel=1e-14)


# ---------------------------------------------------------------- invariances

def test_pool_permutation_invariance():
    """Permute pool rows by pi and map every slot through pi: bit-identical output."""
    inp = W.make_inputs([50, 9], [6, 3], num_heads=3, pool_size=128, seed=9)
    out0, lse0 = oracle.run(inp)
    pi = np.random.default_rng(9).permutation(inp.pool_size)
    newpool = torch.empty_like(inp.kv_pool)
    newpool[torch.from_numpy(pi)] = inp.kv_pool
    inp.kv_pool = newpool
    inp.kv_indices = pi[inp.kv_indices].astype(np.int32)
    inp.out_cache_loc = pi[inp.out_cache_loc].astype(np.int64)
    out1, lse1 = oracle.run(inp)
    assert np.array_equal(out0, out1) and np.array_equal(lse0, lse1)


@pytest.mark.parametrize("splits", [1, 2, 7, 64, 200])
def test_split_count_independence(splits):
    """Split + log-sum-exp combine equals the direct definition (up to rounding)."""
    inp = W.make_inputs([120, 3, 0], [8, 5, 2], num_heads=2, pool_size=256, seed=10, q_scale=3.0)
    out0, lse0 = oracle.run(inp)
    out1, lse1 = oracle.run(inp, num_splits=splits)
    np.testing.assert_allclose(out1, out0, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse1, lse0, rtol=1e-13, atol=1e-13)


def test_batch_packing_independence():
    """A request gives bit-identical rows alone and packed between other requests."""
    big = W.make_inputs([11, 40, 7], [3, 6, 2], num_heads=2, pool_size=128, seed=11)
    out_all, _ = oracle.run(big)
    b = 1
    l0, l1 = big.kv_indptr[b], big.kv_indptr[b + 1]
    t0, t1 = big.qo_indptr[b], big.qo_indptr[b + 1]
    m0, m1 = int(big.mask_indptr[b]), int(big.mask_indptr[b + 1])
    bits = np.unpackbits(big.custom_mask, bitorder="little")[m0:m1]
    out_one, _ = oracle.verify_attn(
        big.q[t0:t1], big.kv_pool, np.array([0, t1 - t0], np.int32), np.array([0, l1 - l0], np.int32),
        big.kv_indices[l0:l1], big.out_cache_loc[t0:t1], np.packbits(bits, bitorder="little"),
        np.array([0, m1 - m0], np.int64), big.sm_scale, big.num_heads)
    H = big.num_heads
    assert np.array_equal(out_all[t0 * H:t1 * H], out_one)


def test_head_permutation_equivariance():
    inp = W.make_inputs([33], [4], num_heads=5, pool_size=64, seed=12)
    out0, _ = oracle.run(inp)
    perm = np.array([3, 0, 4, 1, 2])
    inp.q = inp.q[:, torch.from_numpy(perm)].contiguous()
    out1, _ = oracle.run(inp)
    T, H = 4, 5
    assert np.array_equal(out1.reshape(T, H, 512), out0.reshape(T, H, 512)[:, perm])


# ---------------------------------------------------------------- degenerate cases

def test_row_with_no_visible_key_is_zero():
    inp = W.make_inputs([10], [3], num_heads=2, pool_size=32, seed=13)
    bits = np.unpackbits(inp.custom_mask, bitorder="little")[: int(inp.mask_indptr[-1])].copy()
    bits[13:26] = 0                       # row 1 (N = 13) sees nothing
    inp.custom_mask = np.packbits(bits, bitorder="little")
    out, lse = oracle.run(inp)
    assert np.all(out[2:4] == 0) and np.all(np.isneginf(lse[2:4]))
    assert np.all(np.isfinite(lse[[0, 1, 4, 5]]))


def test_empty_prefix_and_empty_requests():
    """L_b = 0 (drafts only) and T_b = 0 requests next to normal ones."""
    inp = W.make_inputs([0, 25, 9], [4, 0, 2], num_heads=2, pool_size=64, seed=14)
    ref = _sdpa_reference(inp)
    out, _ = oracle.run(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12)


def test_bad_slot_and_bad_mask_indptr_are_errors():
    inp = W.make_inputs([10], [2], num_heads=1, pool_size=16, seed=15)
    bad = inp.kv_indices.copy(); bad[3] = 16
    with pytest.raises(ValueError, match="slot"):
        oracle.verify_attn(inp.q, inp.kv_pool, inp.qo_indptr, inp.kv_indptr, bad, inp.out_cache_loc,
                           inp.custom_mask, inp.mask_indptr, inp.sm_scale, 1)
    with pytest.raises(ValueError, match="mask_indptr"):
        oracle.verify_attn(inp.q, inp.kv_pool, inp.qo_indptr, inp.kv_indptr, inp.kv_indices,
                           inp.out_cache_loc, inp.custom_mask, inp.mask_indptr + np.array([0, 1]),
                           inp.sm_scale, 1)


def test_save_kv_oracle_replaces_exactly_the_named_rows():
    """The KV save definition: named rows replaced, every other row untouched,
    invalid or repeated slots rejected."""
    rng = np.random.default_rng(3)
    pool = rng.integers(0, 1 << 16, size=(50, 576), dtype=np.uint16)
    loc = np.array([7, 0, 49, 23], dtype=np.int64)
    new = rng.integers(0, 1 << 16, size=(4, 576), dtype=np.uint16)
    pool0 = pool.copy()
    got = oracle.save_kv(pool, loc, new)
    for i, s in enumerate(loc):
        assert np.array_equal(got[s], new[i])
    others = np.setdiff1d(np.arange(50), loc)
    assert np.array_equal(got[others], pool[others])
    assert np.array_equal(pool, pool0)                   # the input is not modified in place
    with pytest.raises(ValueError):
        oracle.save_kv(pool, np.array([1, 1]), new[:2])
    with pytest.raises(ValueError):
        oracle.save_kv(pool, np.array([50]), new[:1])


def test_thread_count_does_not_change_results():
    """Rows are independent: one thread and all threads give bit-identical
    outputs (the bench times the oracle both ways)."""
    inp = W.make_inputs([300, 40, 0], [8, 5, 3], num_heads=4, pool_size=512, seed=12)
    n = oracle.num_threads()
    try:
        oracle.set_num_threads(1)
        assert oracle.num_threads() == 1
        out1, lse1 = oracle.run(inp)
    finally:
        oracle.set_num_threads(n)
    outn, lsen = oracle.run(inp)
    assert np.array_equal(out1, outn) and np.array_equal(lse1, lsen)
