"""Seeded synthetic inputs for tree-verify attention over a paged MLA latent pool.

This module only *draws inputs*; it holds none of the attention arithmetic, so
both the CUDA path and the CPU oracle can be fed from it without sharing any
of the method's code.

Workload shapes follow the pages' serving scenario (Kimi K2.6 with a DDTree
drafter on SGLang, "The Integration Chasm", section Context: 185k-token
context; "The Cutover", section Decision to Cut Over: 5.7k / 23k / 91k
contexts) and the five synthetic configurations this library is measured on:

* latent rows are 576 wide (512 no-PE + 64 RoPE dims), V is the first 512
  dims of the same row, sm_scale = 1/sqrt(192);
* page_size = 1: every token owns one pool slot; a request's prefix slots
  are named by ``kv_indices[kv_indptr[b]:kv_indptr[b+1]]`` and its draft
  tokens' own slots by ``out_cache_loc[qo_indptr[b]:qo_indptr[b+1]]``
  ("The Capture-Safe Kernel", Decision 1 and Decision 2);
* each request's draft tree has ``parent[i]`` uniform in {root} U [0, i-1];
  draft token i sees every prefix key and its own ancestors-or-self among the
  drafts (the tree mask, "The Launch Wrapper", section Input);
* the mask is packed bits: request b's ``T_b x N_b`` visibility matrix,
  row-major, starts at *bit* ``mask_indptr[b]``; bit n lives in byte ``n>>3``
  at position ``n&7`` (least-significant bit first).

Floating-point inputs are drawn N(0,1) (q times a per-config scale) and
rounded to bf16.  Small configurations draw them on the host with numpy's
PCG64; the big pools (up to 1.5 M rows x 576) are drawn on the GPU with a
seeded torch generator, because the host fill of 1.7 GB is minutes on slow
hosts.  Either way the bytes the GPU consumes are the bytes the oracle reads
(the oracle receives a host copy).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np
import torch

LATENT_DIM = 576          # 512 no-PE + 64 RoPE dims per latent row
V_DIM = 512               # V = first 512 dims of the same row
SM_SCALE = 1.0 / math.sqrt(192.0)


@dataclasses.dataclass(frozen=True)
class VerifyConfig:
    """One synthetic tree-verify workload."""
    name: str
    prefix_lens: Optional[Sequence[int]]      # None -> drawn (ragged config)
    draft_lens: Optional[Sequence[int]]       # None -> drawn from draft_choices
    num_heads: int
    pool_size: int
    seed: int
    q_scale: float = 1.0
    batch: int = 1
    ragged_prefix_range: Optional[tuple] = None  # (lo, hi) log-uniform, request 0 fixed at hi
    draft_choices: Optional[Sequence[int]] = None
    sm_scale: float = SM_SCALE
    tree: str = "random"                      # draft tree shape: "random", "chain" or "star"
    slots: str = "random"                     # pool slot layout: "random", "contiguous" or "runs:<k>"
    description: str = ""


# The five measured workloads.  Seeds: 0 for the tiny case, 1..4 for the rest
# in order.
CONFIGS = {
    "tiny": VerifyConfig(
        name="tiny", prefix_lens=[256], draft_lens=[8], num_heads=8, pool_size=4096, seed=0,
        description="B=1, prefix 256, T=8 random tree, H=8, pool 4096"),
    "short": VerifyConfig(
        name="short", prefix_lens=[5760], draft_lens=[16], num_heads=8, pool_size=65536, seed=1,
        description="B=1, prefix 5760, T=16 random tree, H=8, pool 65536"),
    "mid": VerifyConfig(
        name="mid", prefix_lens=[23040] * 4, draft_lens=[32] * 4, num_heads=8, pool_size=131072,
        seed=2, batch=4,
        description="B=4, prefix 23040 each, T=32 random trees, H=8, shared shuffled pool 131072"),
    "long": VerifyConfig(
        name="long", prefix_lens=[92160], draft_lens=[64], num_heads=64, pool_size=131072, seed=3,
        q_scale=3.0,
        description="B=1, prefix 92160, T=64 random tree, H=64, q ~ 3*N(0,1), pool 131072"),
    "ragged": VerifyConfig(
        name="ragged", prefix_lens=None, draft_lens=None, num_heads=8, pool_size=1_500_000, seed=4,
        batch=8, ragged_prefix_range=(1024, 185000), draft_choices=(16, 32, 64),
        description="B=8, prefix log-uniform [1024,185000] with request 0 at 185000, "
                    "T in {16,32,64}, H=8, pool 1.5M"),
}
CONFIG_ORDER = ["tiny", "short", "mid", "long", "ragged"]

# Second workloads on the same kernels (degenerate masks): a linear draft
# (chain verify) and plain decode (one new token per request).
CONFIGS["chain"] = VerifyConfig(
    name="chain", prefix_lens=[23040] * 4, draft_lens=[32] * 4, num_heads=8, pool_size=131072, seed=5,
    batch=4, tree="chain",
    description="B=4, prefix 23040 each, T=32 linear draft (chain verify), H=8, pool 131072")
CONFIGS["decode"] = VerifyConfig(
    name="decode", prefix_lens=None, draft_lens=[1] * 32, num_heads=16, pool_size=1_000_000, seed=6,
    batch=32, ragged_prefix_range=(1024, 32768),
    description="B=32, prefix log-uniform [1024,32768] with request 0 at 32768, T=1 (decode), H=16, "
                "pool 1M")
CONFIGS["contig"] = VerifyConfig(
    name="contig", prefix_lens=[23040] * 4, draft_lens=[32] * 4, num_heads=8, pool_size=131072, seed=7,
    batch=4, slots="contiguous",
    description="B=4, prefix 23040 each, T=32 random trees, H=8, pool 131072, contiguous slots "
                "(defragmented pool)")
EXTRA_CONFIG_ORDER = ["chain", "decode", "contig"]


@dataclasses.dataclass
class VerifyInputs:
    """Host-side metadata (numpy) plus float inputs (torch, host or device)."""
    cfg_name: str
    batch: int
    num_heads: int
    pool_size: int
    sm_scale: float
    prefix_lens: np.ndarray      # [B] int64
    draft_lens: np.ndarray       # [B] int64
    parents: List[np.ndarray]    # per request, int64 [T_b], -1 = root
    qo_indptr: np.ndarray        # [B+1] int32
    kv_indptr: np.ndarray        # [B+1] int32
    kv_indices: np.ndarray       # [sum L_b] int32
    out_cache_loc: np.ndarray    # [sum T_b] int64
    custom_mask: np.ndarray      # packed bits, uint8
    mask_indptr: np.ndarray      # [B+1] int64, in bits
    q: torch.Tensor              # [sum T_b, H, 576] bf16
    kv_pool: torch.Tensor        # [pool_size, 576] bf16

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def max_q_per_req(self) -> int:
        return int(self.draft_lens.max()) if self.batch else 0

    def visible_pairs(self) -> int:
        """Number of visible (row, key) pairs, counted from the packed mask."""
        bits = np.unpackbits(self.custom_mask, bitorder="little")
        return int(bits[: int(self.mask_indptr[-1])].sum()) * self.num_heads

    def algorithmic_bytes(self) -> int:
        """Each KV row once + q + out + indices + mask + indptrs (qo_indptr and
        kv_indptr int32, mask_indptr int64)."""
        n_keys = int(self.kv_indptr[-1]) + int(self.qo_indptr[-1])
        rows = self.total_q * self.num_heads
        return (n_keys * LATENT_DIM * 2 + rows * LATENT_DIM * 2 + rows * V_DIM * 2
                + int(self.kv_indptr[-1]) * 4 + self.total_q * 8
                + (int(self.mask_indptr[-1]) + 7) // 8 + (self.batch + 1) * (4 + 4 + 8))

    def algorithmic_flops(self) -> int:
        """2*(576+512) flops per visible (row, key) pair."""
        return 2 * (LATENT_DIM + V_DIM) * self.visible_pairs()


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def random_tree(rng: np.random.Generator, t: int) -> np.ndarray:
    """parent[i] uniform over {-1 (root)} U [0, i-1]."""
    return np.array([rng.integers(-1, i) for i in range(t)], dtype=np.int64)


def chain_tree(t: int) -> np.ndarray:
    return np.arange(-1, t - 1, dtype=np.int64)


def ancestors_or_self(parents: np.ndarray) -> np.ndarray:
    """Dense bool [T, T]: entry (i, j) is True iff draft j is i or an ancestor of i."""
    t = len(parents)
    vis = np.zeros((t, t), dtype=bool)
    for i in range(t):
        j = i
        while j >= 0:
            vis[i, j] = True
            j = int(parents[j])
    return vis


def pack_mask(rows: List[np.ndarray]) -> tuple:
    """Pack per-request bool [T_b, N_b] matrices back to back, LSB-first."""
    sizes = [int(r.size) for r in rows]
    indptr = np.zeros(len(rows) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(sizes)
    flat = np.concatenate([r.reshape(-1) for r in rows]) if rows else np.zeros(0, bool)
    packed = np.packbits(flat.astype(np.uint8), bitorder="little")
    return packed, indptr


def pack_tree_masks(prefix_lens, parents_list, extra_prefix_mask=None) -> tuple:
    """Packed masks for tree-verify: all prefix bits 1, draft bits = ancestor-or-self.

    Built directly in packed form (all-ones then clear the invisible draft
    bits) so 100M-bit masks are cheap.  ``extra_prefix_mask(b, T_b, L_b)`` may
    return a bool [T_b, L_b] to replace the all-ones prefix part (tests use it
    to make the kernel read real prefix bits).
    """
    sizes = [len(p) * (int(l) + len(p)) for l, p in zip(prefix_lens, parents_list)]
    indptr = np.zeros(len(sizes) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(sizes)
    nbits = int(indptr[-1])
    packed = np.full((nbits + 7) // 8, 0xFF, dtype=np.uint8)
    if nbits % 8:
        packed[-1] = np.uint8((1 << (nbits % 8)) - 1)
    for b, (l, p) in enumerate(zip(prefix_lens, parents_list)):
        t, l = len(p), int(l)
        n = l + t
        vis = ancestors_or_self(p)
        if extra_prefix_mask is not None:
            pre = extra_prefix_mask(b, t, l)
            full = np.concatenate([pre, vis], axis=1)
            ii, jj = np.nonzero(~full)
        else:
            ii, jj = np.nonzero(~vis)
            jj = jj + l
        pos = indptr[b] + ii.astype(np.int64) * n + jj.astype(np.int64)
        np.bitwise_and.at(packed, pos >> 3, ~(np.uint8(1) << (pos & 7).astype(np.uint8)))
    return packed, indptr


def draw_lengths(cfg: VerifyConfig, rng: np.random.Generator):
    if cfg.prefix_lens is not None:
        prefix = np.asarray(cfg.prefix_lens, dtype=np.int64)
    else:
        lo, hi = cfg.ragged_prefix_range
        u = rng.uniform(math.log(lo), math.log(hi), size=cfg.batch - 1)
        prefix = np.concatenate([[hi], np.floor(np.exp(u)).astype(np.int64)]).astype(np.int64)
    if cfg.draft_lens is not None:
        drafts = np.asarray(cfg.draft_lens, dtype=np.int64)
    else:
        drafts = rng.choice(np.asarray(cfg.draft_choices, dtype=np.int64), size=cfg.batch)
    return prefix, drafts


def _float_inputs(shape_q, pool_shape, q_scale, seed, device, rng):
    """q and pool in bf16: numpy PCG64 on the host, or a seeded torch generator on cuda."""
    dev = torch.device(device)
    if dev.type == "cuda":
        g = torch.Generator(device=dev)
        g.manual_seed(1_000_003 * seed + 17)
        q = (torch.randn(shape_q, generator=g, device=dev, dtype=torch.float32) * q_scale).to(torch.bfloat16)
        pool = torch.empty(pool_shape, device=dev, dtype=torch.bfloat16)
        rows_per = 1 << 18
        for r0 in range(0, pool_shape[0], rows_per):
            r1 = min(pool_shape[0], r0 + rows_per)
            pool[r0:r1] = torch.randn((r1 - r0, pool_shape[1]), generator=g, device=dev,
                                      dtype=torch.float32).to(torch.bfloat16)
        return q, pool
    qf = rng.standard_normal(shape_q, dtype=np.float32) * np.float32(q_scale)
    pf = rng.standard_normal(pool_shape, dtype=np.float32)
    q = torch.from_numpy(to_bf16_bits(qf).view(np.int16)).view(torch.bfloat16)
    pool = torch.from_numpy(to_bf16_bits(pf).view(np.int16)).view(torch.bfloat16)
    return q.reshape(shape_q), pool.reshape(pool_shape)


def slot_order(rng: np.random.Generator, pool_size: int, n_keys: int, slots: str) -> np.ndarray:
    """The pool slots handed out in request order (prefix, then drafts).

    "random": a random permutation of the pool (a fragmented pool);
    "contiguous": one run starting at a random offset (a defragmented pool:
    every request's keys sit in consecutive slots); "runs:<k>": the pool cut
    into runs of k consecutive slots, the runs shuffled (partly fragmented).
    """
    if slots == "random":
        return rng.permutation(pool_size).astype(np.int64)
    if slots == "contiguous":
        off = int(rng.integers(0, pool_size - n_keys + 1))
        return (off + np.arange(pool_size, dtype=np.int64)) % pool_size
    if slots.startswith("runs:"):
        k = int(slots.split(":")[1])
        starts = np.arange(0, pool_size, k, dtype=np.int64)
        rng.shuffle(starts)
        return np.concatenate([np.arange(s0, min(s0 + k, pool_size), dtype=np.int64) for s0 in starts])
    raise ValueError(slots)


def make_inputs(prefix_lens, draft_lens, num_heads, pool_size, seed, *, q_scale=1.0,
                sm_scale=SM_SCALE, device="cpu", parents=None, tree="random",
                extra_prefix_mask=None, cfg_name="custom", slots="random") -> VerifyInputs:
    """Draw one ragged batch.

    tree: "random" (parent uniform over root and earlier drafts), "chain"
    (parent[i] = i-1), or "star" (every draft hangs off the root).
    slots: pool slot layout (see ``slot_order``).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    prefix_lens = np.asarray(prefix_lens, dtype=np.int64)
    draft_lens = np.asarray(draft_lens, dtype=np.int64)
    bsz = len(prefix_lens)
    if parents is None:
        if tree == "random":
            parents = [random_tree(rng, int(t)) for t in draft_lens]
        elif tree == "chain":
            parents = [chain_tree(int(t)) for t in draft_lens]
        elif tree == "star":
            parents = [np.full(int(t), -1, dtype=np.int64) for t in draft_lens]
        else:
            raise ValueError(tree)
    n_keys = int(prefix_lens.sum() + draft_lens.sum())
    if n_keys > pool_size:
        raise ValueError(f"pool of {pool_size} slots cannot hold {n_keys} tokens")
    perm = slot_order(rng, pool_size, n_keys, slots)
    kv_idx, ocl = [], []
    off = 0
    for b in range(bsz):
        l, t = int(prefix_lens[b]), int(draft_lens[b])
        kv_idx.append(perm[off:off + l]); off += l
        ocl.append(perm[off:off + t]); off += t
    kv_indices = (np.concatenate(kv_idx) if bsz else np.zeros(0, np.int64)).astype(np.int32)
    out_cache_loc = (np.concatenate(ocl) if bsz else np.zeros(0, np.int64)).astype(np.int64)
    qo_indptr = np.zeros(bsz + 1, dtype=np.int32); qo_indptr[1:] = np.cumsum(draft_lens)
    kv_indptr = np.zeros(bsz + 1, dtype=np.int32); kv_indptr[1:] = np.cumsum(prefix_lens)
    custom_mask, mask_indptr = pack_tree_masks(prefix_lens, parents, extra_prefix_mask)
    total_q = int(qo_indptr[-1])
    q, pool = _float_inputs((total_q, num_heads, LATENT_DIM), (pool_size, LATENT_DIM), q_scale,
                            seed, device, rng)
    return VerifyInputs(cfg_name=cfg_name, batch=bsz, num_heads=num_heads, pool_size=pool_size,
                        sm_scale=float(sm_scale), prefix_lens=prefix_lens, draft_lens=draft_lens,
                        parents=parents, qo_indptr=qo_indptr, kv_indptr=kv_indptr,
                        kv_indices=kv_indices, out_cache_loc=out_cache_loc,
                        custom_mask=custom_mask, mask_indptr=mask_indptr, q=q, kv_pool=pool)


def make_config_inputs(name: str, device="cpu") -> VerifyInputs:
    cfg = CONFIGS[name]
    rng = np.random.Generator(np.random.PCG64(cfg.seed + 7919))
    prefix, drafts = draw_lengths(cfg, rng)
    return make_inputs(prefix, drafts, cfg.num_heads, cfg.pool_size, cfg.seed,
                       q_scale=cfg.q_scale, sm_scale=cfg.sm_scale, device=device, tree=cfg.tree, cfg_name=name,
                       slots=cfg.slots)
