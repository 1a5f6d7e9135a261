"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle."""

import copy
import numpy as np
import pytest
import torch

from speculative_decode_mla_paged_gb300 import api
from speculative_decode_mla_paged_gb300 import workloads as W

from gpu_helpers import as_rows, assert_parity, device_inputs, oracle_rows, run, sample_rows

pytestmark = pytest.mark.gpu
IMPLS = ["tc", "simt"]


@pytest.fixture(scope="module", autouse=True)
def _init():
    api.init()


# ---------------------------------------------------------------- the five workloads

@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name,splits", [("tiny", 1), ("tiny", 4), ("tiny", 64), ("short", 8)])
def test_small_configs_every_row(name, splits, impl):
    inp = W.make_config_inputs(name, device="cpu")
    out, status = run(inp, impl=impl, num_splits=splits)
    assert status == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"{name}/{impl}/{splits}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name,splits", [("mid", 16), ("long", 8), ("ragged", 64)])
def test_large_configs_sampled_rows(name, splits, impl):
    """Full-size launch; the oracle checks sampled rows (first/last row of each
    request plus random ones)."""
    inp = W.make_config_inputs(name, device="cuda")
    out, status = run(inp, impl=impl, num_splits=splits)
    assert status == 0
    got = as_rows(out)
    assert np.all(np.isfinite(got))
    inp_host = inp
    inp_host.q, inp_host.kv_pool = inp.q.cpu(), inp.kv_pool.cpu()
    rows = sample_rows(inp_host, n_random=40, seed=hash(name) % 1000)
    assert_parity(got[rows], oracle_rows(inp_host, rows), f"{name}/{impl}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", ["chain", "decode", "contig"])
def test_extra_workloads(name, impl):
    """Chain verify (linear draft), plain decode (T = 1) and a defragmented
    pool (contiguous slots: the tensor-core kernel's plain-tile fast path) on
    the same kernels: sampled rows against the oracle, all rows finite."""
    inp = W.make_config_inputs(name, device="cuda")
    out, status = run(inp, impl=impl, num_splits=9)
    assert status == 0
    got = as_rows(out)
    assert np.all(np.isfinite(got))
    inp.q, inp.kv_pool = inp.q.cpu(), inp.kv_pool.cpu()
    rows = sample_rows(inp, n_random=48, seed=7)
    assert_parity(got[rows], oracle_rows(inp, rows), f"{name}/{impl}")


@pytest.mark.parametrize("slots", ["runs:64", "runs:37", "runs:200", "contiguous"])
@pytest.mark.parametrize("drafts", [(32, 16, 8), (16, 8, 4)], ids=["two_row_tiles", "one_row_tile"])
def test_contiguous_runs_every_row(slots, drafts):
    """Pools cut into runs of consecutive slots: units whose keys are all
    consecutive take plain TMA tiles, the others gathers; with T * H up to
    256 (4-CTA clusters) and up to 128 (2-CTA clusters); every output row
    against the oracle."""
    inp = W.make_inputs([3000, 1500, 700], list(drafts), 8, 65536, seed=41, slots=slots)
    out, status = run(inp, impl="tc", num_splits=3)
    assert status == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"tc/{slots}/{drafts}")


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("sm_scale,q_scale", [(-0.3, 1.0), (0.0, 1.0), (2.5, 1.0), (W.SM_SCALE, 8.0)])
def test_softmax_scale_and_range(sm_scale, q_scale, impl):
    """Negative, zero and large softmax scales (the tensor-core kernel folds a
    negative scale into Q's signs; a zero scale gives uniform weights over the
    visible keys) and a wide score range (many online rescales): every row
    against the oracle."""
    inp = W.make_inputs([1500, 600], [24, 8], 8, 8192, seed=53, q_scale=q_scale, sm_scale=sm_scale)
    out, status = run(inp, impl=impl, num_splits=2)
    assert status == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"{impl}/scale={sm_scale}/q={q_scale}")


def _rising_score_inputs(seed):
    """Scores that climb about 47 (log2 units) every 128 keys: Q's last 64
    dims are 1 and key j's are 7 j / 128, so the score gains 64 * 7 * scale
    * log2(e) ~ 47 per 128 keys over a random part of spread ~2.4."""
    inp = W.make_inputs([1500, 600], [24, 8], 8, 8192, seed=seed)
    q, pool = inp.q.clone(), inp.kv_pool.clone()
    q[:, :, 512:] = 1.0
    for b in range(inp.batch):
        slots = np.concatenate([inp.kv_indices[inp.kv_indptr[b]:inp.kv_indptr[b + 1]],
                                inp.out_cache_loc[inp.qo_indptr[b]:inp.qo_indptr[b + 1]]])
        ramp = torch.tensor(7.0 * np.arange(len(slots)) / 128.0, dtype=torch.float32)
        pool[torch.from_numpy(slots.astype(np.int64)), 512:] = ramp[:, None].to(torch.bfloat16)
    inp.q, inp.kv_pool = q, pool
    return inp


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("splits", [1, 2])
def test_rising_scores_rescale_on_every_tile(splits, impl):
    """Every 128-key window's row maximum exceeds the previous window's by
    more than 32 (log2 units) in every row, so the tensor-core kernel's lazy
    maximum must rescale O on every tile: every row against the oracle."""
    inp = _rising_score_inputs(seed=54)
    L, T0 = int(inp.prefix_lens[0]), int(inp.draft_lens[0])
    s = (inp.q[:T0].double().reshape(-1, 576).numpy()
         @ inp.kv_pool[torch.from_numpy(inp.kv_indices[:L].astype(np.int64))].double().numpy().T)
    s *= inp.sm_scale * np.log2(np.e)
    win = s[:, : (L // 128) * 128].reshape(s.shape[0], -1, 128).max(axis=2)
    assert np.diff(win, axis=1).min() > 32.0, "inputs do not force a rescale per tile"
    out, status = run(inp, impl=impl, num_splits=splits)
    assert status == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"{impl}/rising scores/{splits} splits")


def test_large_config_kernels_agree_on_every_row():
    """At full size every row of the tensor-core path matches the CUDA-core
    path within the same bar (the oracle covers the sampled rows above)."""
    inp = W.make_config_inputs("mid", device="cuda")
    d = device_inputs(inp)
    a, _ = run(inp, impl="tc", num_splits=16, d=d)
    b, _ = run(inp, impl="simt", num_splits=5, d=d)
    assert_parity(as_rows(a), as_rows(b), "tc vs simt on mid")


# ---------------------------------------------------------------- edge cases

RAGGED_CASES = {
    # prefix lengths, draft lengths, heads
    "mixed": ([0, 1, 63, 64, 65, 200], [1, 3, 7, 2, 16, 5], 8),
    "odd_heads": ([37, 130], [5, 9], 3),
    "one_head_one_token": ([500], [1], 1),
    "empty_requests": ([10, 0, 77, 5], [0, 4, 0, 2], 4),
    "drafts_only": ([0, 0], [6, 11], 8),
    "many_rows": ([300], [64], 16),
    "wide_heads": ([300, 50, 0], [3, 2, 4], 160),   # H > 128: one token's heads span row tiles
}


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("case", sorted(RAGGED_CASES))
@pytest.mark.parametrize("splits", [1, 3, 256])
def test_ragged_edge_cases(case, splits, impl):
    prefix, drafts, H = RAGGED_CASES[case]
    inp = W.make_inputs(prefix, drafts, H, pool_size=2048, seed=len(prefix) + splits, q_scale=2.0)
    out, status = run(inp, impl=impl, num_splits=splits, max_q=max(drafts) + 3)
    assert status == 0
    if inp.total_q:
        assert_parity(as_rows(out), oracle_rows(inp), f"{case}/{impl}/{splits}")


@pytest.mark.parametrize("impl", IMPLS)
def test_random_prefix_bits_and_blind_rows(impl):
    """Prefix bits are read, not assumed: random prefix masks, plus one draft
    row that sees nothing at all (zeros)."""
    prefix, drafts, H = [150, 70], [6, 4], 4
    rng = np.random.default_rng(3)
    pv = [rng.random((t, l)) < 0.5 for l, t in zip(prefix, drafts)]
    inp = W.make_inputs(prefix, drafts, H, pool_size=512, seed=3,
                        extra_prefix_mask=lambda b, t, l: pv[b])
    bits = np.unpackbits(inp.custom_mask, bitorder="little")[: int(inp.mask_indptr[-1])].copy()
    N0 = prefix[0] + drafts[0]
    bits[2 * N0:3 * N0] = 0                      # request 0, draft 2 sees nothing
    inp.custom_mask = np.packbits(bits, bitorder="little")
    out, status = run(inp, impl=impl, num_splits=3)
    assert status == 0
    got, ref = as_rows(out), oracle_rows(inp)
    assert np.all(got[2 * H:3 * H] == 0)
    assert_parity(got, ref, f"random prefix/{impl}")


@pytest.mark.parametrize("offset", [1, 3, 7])
@pytest.mark.parametrize("impl", IMPLS)
def test_mask_at_unaligned_address(impl, offset):
    """The custom mask passed as a view that starts `offset` bytes into its
    buffer, with random prefix bits (every row's bit offset differs): the
    kernels read it in aligned words and shift it into place."""
    prefix, drafts, H = [300, 77, 5], [9, 4, 2], 4
    rng = np.random.default_rng(offset)
    pv = [rng.random((t, l)) < 0.6 for l, t in zip(prefix, drafts)]
    inp = W.make_inputs(prefix, drafts, H, pool_size=1024, seed=30 + offset,
                        extra_prefix_mask=lambda b, t, l: pv[b])
    d = device_inputs(inp)
    n = d["custom_mask"].numel()
    buf = torch.full((n + 16,), 0xA5, dtype=torch.uint8, device="cuda")
    buf[offset:offset + n] = d["custom_mask"]
    d["custom_mask"] = buf[offset:offset + n]
    out, status = run(inp, impl=impl, num_splits=3, d=d)
    assert status == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"mask at +{offset}/{impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_strided_q_and_out(impl):
    """q and out as views with padded token/head strides (no .contiguous())."""
    inp = W.make_inputs([90, 33], [7, 3], 4, pool_size=512, seed=21)
    d = device_inputs(inp)
    big_q = torch.zeros(inp.total_q, 6, 584, dtype=torch.bfloat16, device="cuda")
    big_q[:, 1:5, 8:584] = d["q"]
    d["q"] = big_q[:, 1:5, 8:584]
    big_out = torch.full((inp.total_q, 5, 520), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big_out[:, :4, 8:520]
    run(inp, impl=impl, num_splits=2, d=d, out=out)
    assert_parity(as_rows(out.contiguous()), oracle_rows(inp), f"strided/{impl}")
    assert torch.all(big_out[:, 4] == 7.0) and torch.all(big_out[:, :, :8] == 7.0)


@pytest.mark.parametrize("impl", IMPLS)
def test_unused_pool_rows_are_never_read(impl):
    """Every pool row no request names is NaN: any stray read poisons the output."""
    inp = W.make_inputs([120, 64, 1], [8, 16, 3], 8, pool_size=1024, seed=22)
    used = np.concatenate([inp.kv_indices.astype(np.int64), inp.out_cache_loc])
    poison = np.ones(inp.pool_size, bool); poison[used] = False
    inp.kv_pool[torch.from_numpy(poison)] = float("nan")
    out, status = run(inp, impl=impl, num_splits=5)
    assert status == 0
    assert_parity(as_rows(out), oracle_rows(inp), f"poisoned pool/{impl}")


@pytest.mark.parametrize("impl", IMPLS)
def test_bad_slot_sets_status_without_fault(impl):
    inp = W.make_inputs([40], [4], 2, pool_size=128, seed=23)
    inp.kv_indices = inp.kv_indices.copy()
    inp.kv_indices[5] = inp.pool_size + 1000
    out, status = run(inp, impl=impl, num_splits=2)
    assert status & api.STATUS_BAD_SLOT
    assert np.all(np.isfinite(as_rows(out)))


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("drafts", [(12, 3), (40, 20)], ids=["one_row_tile", "two_row_tiles"])
def test_bad_slots_across_many_tiles_are_skipped(drafts, impl):
    """Slots outside the pool at scattered key positions of a 25-tile unit
    (one split, so the per-tile valid-key bits wrap their ring many times):
    the call sets VA_STATUS_BAD_SLOT and every row equals the oracle run on
    the same inputs with those keys hidden from every row (the kernels skip
    a key whose slot is invalid)."""
    prefix, H = [3100, 700], 8
    inp = W.make_inputs(prefix, list(drafts), H, pool_size=8192, seed=27)
    rng = np.random.default_rng(27)
    bad = {0: np.sort(rng.choice(prefix[0], 40, replace=False)), 1: np.array([0, 127, 128, 699])}
    bits = np.unpackbits(inp.custom_mask, bitorder="little")[: int(inp.mask_indptr[-1])].copy()
    kv_bad = inp.kv_indices.copy()
    for b, keys in bad.items():
        n = prefix[b] + drafts[b]
        rows = bits[int(inp.mask_indptr[b]): int(inp.mask_indptr[b + 1])].reshape(drafts[b], n)
        rows[:, keys] = 0                       # the reference: these keys hidden from every row
        kv_bad[inp.kv_indptr[b] + keys] = inp.pool_size + 7 + keys
    ref_inp = copy.copy(inp)
    ref_inp.custom_mask = np.packbits(bits, bitorder="little")
    ref = oracle_rows(ref_inp)                  # valid slots, hidden keys
    inp.kv_indices = kv_bad                     # the kernels see the invalid slots, full mask
    out, status = run(inp, impl=impl, num_splits=1)
    assert status & api.STATUS_BAD_SLOT
    assert_parity(as_rows(out), ref, f"bad slots/{impl}/{drafts}")


@pytest.mark.parametrize("impl", IMPLS)
def test_too_many_drafts_sets_meta_status(impl):
    inp = W.make_inputs([40, 12], [4, 6], 2, pool_size=128, seed=24)
    _, status = run(inp, impl=impl, num_splits=2, max_q=5)
    assert status & api.STATUS_BAD_META


# ---------------------------------------------------------------- bit-exact decode

@pytest.mark.parametrize("impl", IMPLS)
def test_slot_decode_bit_exact(impl):
    """Each pool row's V encodes its slot id in small integers (exact in bf16);
    each draft row sees exactly one key, so the output must be that row's V
    bit for bit.  Checks slot resolution through kv_indices / out_cache_loc."""
    prefix, drafts, H = [700, 90, 3], [9, 5, 12], 4
    inp = W.make_inputs(prefix, drafts, H, pool_size=4096, seed=25)
    slots = np.arange(inp.pool_size)
    code = np.stack([((slots >> k) & 1) * 2 - 1 + (k % 3) for k in range(12)], axis=1).astype(np.float32)
    pool = np.zeros((inp.pool_size, 576), np.float32)
    pool[:, :12] = code
    pool[:, 12] = (slots % 251).astype(np.float32)
    inp.kv_pool = torch.from_numpy(W.to_bf16_bits(pool).view(np.int16)).view(torch.bfloat16)
    rng = np.random.default_rng(25)
    rows_bits, picks = [], []
    for l, t in zip(prefix, drafts):
        n = l + t
        pick = rng.integers(0, n, size=t)
        m = np.zeros((t, n), bool); m[np.arange(t), pick] = True
        rows_bits.append(m); picks.append(pick)
    inp.custom_mask, inp.mask_indptr = W.pack_mask(rows_bits)
    out, status = run(inp, impl=impl, num_splits=7)
    assert status == 0
    got = out.view(torch.int16).cpu().numpy().reshape(inp.total_q, H, 512)
    poolbits = W.to_bf16_bits(pool)[:, :512].view(np.int16)
    t = 0
    for b, (l, n_t) in enumerate(zip(prefix, drafts)):
        for i in range(n_t):
            j = int(picks[b][i])
            slot = inp.kv_indices[inp.kv_indptr[b] + j] if j < l else inp.out_cache_loc[inp.qo_indptr[b] + j - l]
            for h in range(H):
                assert np.array_equal(got[t, h], poolbits[slot]), f"request {b} draft {i} head {h}"
            t += 1


@pytest.mark.parametrize("impl", IMPLS)
def test_mask_decode_bit_exact(impl):
    """q = 0 gives every visible key equal weight; key j's V is one-hot on dim
    j, so out[row, j] != 0 exactly when the mask lets row see key j.  The
    recovered bit matrix must equal the packed mask bit for bit."""
    prefix, drafts, H = [230, 41], [20, 33], 2
    rng = np.random.default_rng(26)
    pv = [rng.random((t, l)) < 0.7 for l, t in zip(prefix, drafts)]
    inp = W.make_inputs(prefix, drafts, H, pool_size=1024, seed=26,
                        extra_prefix_mask=lambda b, t, l: pv[b])
    pool = np.zeros((inp.pool_size, 576), np.float32)
    for b, (l, t) in enumerate(zip(prefix, drafts)):
        for j in range(l + t):
            slot = inp.kv_indices[inp.kv_indptr[b] + j] if j < l else inp.out_cache_loc[inp.qo_indptr[b] + j - l]
            pool[slot, j] = 1.0
    inp.kv_pool = torch.from_numpy(W.to_bf16_bits(pool).view(np.int16)).view(torch.bfloat16)
    inp.q = torch.zeros_like(inp.q)
    out, status = run(inp, impl=impl, num_splits=4)
    assert status == 0
    got = out.float().cpu().numpy().reshape(inp.total_q, H, 512)
    bits = np.unpackbits(inp.custom_mask, bitorder="little")
    t = 0
    for b, (l, n_t) in enumerate(zip(prefix, drafts)):
        n = l + n_t
        for i in range(n_t):
            want = bits[int(inp.mask_indptr[b]) + i * n: int(inp.mask_indptr[b]) + (i + 1) * n].astype(bool)
            for h in range(H):
                assert np.array_equal(got[t, h, :n] != 0, want), f"request {b} draft {i}"
                assert np.all(got[t, h, n:] == 0)
            t += 1


# ---------------------------------------------------------------- CUDA graph capture / replay

@pytest.mark.parametrize("max_q", [16, 32], ids=["one_row_tile", "two_row_tiles"])
@pytest.mark.parametrize("impl", IMPLS)
def test_graph_capture_and_replay_with_new_contents(impl, max_q):
    """Capture one call, then rewrite the *contents* of the static buffers
    (new trees, new slots, new prefix lengths, new q) and replay: each replay
    must match the oracle on the new inputs ("The Capture-Safe Kernel",
    Decision 6: no replay hook, the kernel reads the static buffers).  With
    H = 8, max_q 16 launches the tensor-core kernel's 2-CTA cluster shape and
    max_q 32 its 4-CTA shape."""
    B, H, splits, pool_size = 3, 8, 8, 8192
    cap_kv, cap_bits = 3 * 1500, 3 * max_q * (1500 + max_q)
    pool = W.make_inputs([1], [1], H, pool_size=pool_size, seed=30).kv_pool.cuda()
    st = {
        "q": torch.zeros(B * max_q, H, 576, dtype=torch.bfloat16, device="cuda"),
        "qo_indptr": torch.zeros(B + 1, dtype=torch.int32, device="cuda"),
        "kv_indptr": torch.zeros(B + 1, dtype=torch.int32, device="cuda"),
        "kv_indices": torch.zeros(cap_kv, dtype=torch.int32, device="cuda"),
        "out_cache_loc": torch.zeros(B * max_q, dtype=torch.int64, device="cuda"),
        "custom_mask": torch.zeros(cap_bits // 8 + 1, dtype=torch.uint8, device="cuda"),
        "mask_indptr": torch.zeros(B + 1, dtype=torch.int64, device="cuda"),
    }
    out = torch.zeros(B * max_q, H, 512, dtype=torch.bfloat16, device="cuda")
    runner = api.VerifyAttention(B, max_q, H, splits, impl=impl)

    def fill(inp):
        for k in ("qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask", "mask_indptr"):
            src = torch.from_numpy(np.ascontiguousarray(getattr(inp, k))).cuda()
            st[k][: src.numel()].copy_(src)
        st["q"].zero_()
        st["q"][: inp.total_q].copy_(inp.q.cuda())

    def call():
        runner(st["q"], pool, st["qo_indptr"], st["kv_indptr"], st["kv_indices"], st["out_cache_loc"],
               st["custom_mask"], st["mask_indptr"], W.SM_SCALE, out)

    first = W.make_inputs([1000, 10, 400], [max_q, 3, 9], H, pool_size=pool_size, seed=31)
    first.kv_pool = pool.cpu()
    fill(first)
    call()                                   # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.synchronize()
    for seed, prefix, drafts in [(32, [1500, 700, 1], [5, max_q, 2]), (33, [3, 1400, 1499], [max_q, 1, 16]),
                                 (34, [0, 0, 1200], [2, 2, 2])]:
        inp = W.make_inputs(prefix, drafts, H, pool_size=pool_size, seed=seed)
        inp.kv_pool = pool.cpu()
        fill(inp)
        g.replay()
        torch.cuda.synchronize()
        got = as_rows(out)[: inp.total_q * H]
        assert_parity(got, oracle_rows(inp), f"replay seed {seed}/{impl}")


def test_profiled_call_times_every_graph_replay():
    """The library's phase events time a direct call and, recorded inside a
    captured graph (external event records), each replay: start <= split
    start <= split end <= combine end, all readable, and the output still
    matches the oracle."""
    inp = W.make_inputs([1200, 300], [24, 8], 8, 8192, seed=61)
    d = device_inputs(inp)
    runner = api.VerifyAttention(inp.batch, inp.max_q_per_req, inp.num_heads, 4)
    out = torch.zeros(inp.total_q, inp.num_heads, 512, dtype=torch.bfloat16, device="cuda")
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    def call():
        runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
               d["custom_mask"], d["mask_indptr"], inp.sm_scale, out, events=ev)

    call()                                   # a direct profiled call first
    torch.cuda.synchronize()
    t = [ev[0].elapsed_time(e) for e in ev]
    assert t[0] == 0 and 0 <= t[1] <= t[2] <= t[3] < 1000.0, t
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        t = [ev[0].elapsed_time(e) for e in ev]
        assert t[0] == 0 and 0 <= t[1] <= t[2] <= t[3] < 1000.0, t
        assert_parity(as_rows(out), oracle_rows(inp), "profiled replay")
    assert runner.status() == 0


def test_concurrent_mixed_calls_from_two_threads():
    """Two host threads, each with its own workspace and stream, issue mixed
    calls (both cluster shapes, each forking to its thread's second stream)
    at the same time; every output matches the oracle."""
    import threading

    cases = [W.make_inputs([900, 200, 40], [24, 8, 16], 8, 8192, seed=81),
             W.make_inputs([300, 1200], [8, 32], 8, 8192, seed=82)]
    refs = [oracle_rows(c) for c in cases]
    devs = [device_inputs(c) for c in cases]
    torch.cuda.synchronize()                  # inputs copied before other streams read them
    errors = []

    def worker(k):
        try:
            c, d = cases[k], devs[k]
            runner = api.VerifyAttention(c.batch, c.max_q_per_req, c.num_heads, 4)
            s = torch.cuda.Stream()
            out = torch.zeros(c.total_q, c.num_heads, 512, dtype=torch.bfloat16, device="cuda")
            for _ in range(20):
                with torch.cuda.stream(s):
                    out.zero_()
                    runner(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                           d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], c.sm_scale, out)
                s.synchronize()
                assert runner.status() == 0
                assert_parity(as_rows(out), refs[k], f"thread {k}")
        except Exception as e:          # reported in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_concurrent_captures_of_mixed_calls_from_two_threads():
    """Two host threads capture a mixed call (both cluster shapes, so both
    fork to a second stream) into CUDA graphs at the same time; each thread's
    call forks to its own second stream, so neither capture invalidates the
    other, and every replay matches the oracle."""
    import threading

    cases = [W.make_inputs([900, 200, 40], [24, 8, 16], 8, 8192, seed=83),
             W.make_inputs([300, 1200], [8, 32], 8, 8192, seed=84)]
    refs = [oracle_rows(c) for c in cases]
    devs = [device_inputs(c) for c in cases]
    torch.cuda.synchronize()
    both_capturing = threading.Barrier(2, timeout=60)
    errors = []

    def worker(k):
        try:
            c, d = cases[k], devs[k]
            runner = api.VerifyAttention(c.batch, c.max_q_per_req, c.num_heads, 4)   # this thread's second stream
            s = torch.cuda.Stream()
            out = torch.zeros(c.total_q, c.num_heads, 512, dtype=torch.bfloat16, device="cuda")
            args = (d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"], d["out_cache_loc"],
                    d["custom_mask"], d["mask_indptr"], c.sm_scale, out)
            with torch.cuda.stream(s):
                runner(*args)                  # warm-up outside the capture
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                runner(*args)
                both_capturing.wait()          # the other thread's capture is open too
            for _ in range(3):
                with torch.cuda.stream(s):
                    out.zero_()
                    g.replay()
                s.synchronize()
                assert runner.status() == 0
                assert_parity(as_rows(out), refs[k], f"thread {k}")
        except Exception as e:          # reported in the main thread
            both_capturing.abort()
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors


def test_tune_num_splits_returns_a_candidate_and_a_correct_call():
    """api.tune_num_splits times each candidate as graph replays of the real
    (here mixed-shape) call and returns one of them; the output it leaves
    matches the oracle, and a runner at the chosen count agrees."""
    from speculative_decode_mla_paged_gb300 import tuning

    inp = W.make_inputs([2500, 700, 90], [24, 8, 16], 8, 8192, seed=91)
    d = device_inputs(inp)
    out = torch.zeros(inp.total_q, inp.num_heads, 512, dtype=torch.bfloat16, device="cuda")
    cands = tuning.ranked_num_splits(inp.prefix_lens, inp.draft_lens, inp.num_heads, k=3)
    s = api.tune_num_splits(d["q"], d["kv_pool"], d["qo_indptr"], d["kv_indptr"], d["kv_indices"],
                            d["out_cache_loc"], d["custom_mask"], d["mask_indptr"], inp.sm_scale, out,
                            inp.max_q_per_req, cands, replays=2, flush_bytes=8 << 20)
    assert s in cands
    ref = oracle_rows(inp)
    assert_parity(as_rows(out), ref, "after tuning")
    got, status = run(inp, num_splits=s)
    assert status == 0
    assert_parity(as_rows(got), ref, f"tuned {s} splits")
