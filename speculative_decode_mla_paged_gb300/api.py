"""Python binding of libverify_attn (ctypes; argument marshalling only).

Every step of the computation runs in the library's CUDA kernels.  This
module turns torch tensors into device pointers, strides and the current
stream, and maps the C status codes to exceptions.  There is no fallback:
if the library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
import warnings
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libverify_attn.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "verify_attn.h")

LATENT_DIM = 576
V_DIM = 512
MAX_SPLITS = 256
STATUS_BAD_SLOT = 0x1
STATUS_BAD_META = 0x2
STATUS_TIMEOUT = 0x4

_lock = threading.Lock()
_lib = None

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int
_RUN_ARGS = [_p, _i64, _i64, _p, _i64, _p, _p, _p, _p, _p, _p, ctypes.c_float, _p, _i64, _i64,
             _i32, _i32, _i32, _i32, _p, ctypes.c_size_t, _p]


class VerifyAttnError(RuntimeError):
    pass


def load_library():
    """Load libverify_attn.so (built by ``build.py``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise VerifyAttnError(
                    f"{LIB_PATH} is missing: build it with `python -m speculative_decode_mla_paged_gb300.build`")
            lib = ctypes.CDLL(LIB_PATH)
            lib.verify_attn_workspace_size.argtypes = [_i32, _i32, _i32, _i32]
            lib.verify_attn_workspace_size.restype = ctypes.c_size_t
            lib.verify_attn_init.argtypes = []
            lib.verify_attn_init.restype = _i32
            for name in ("verify_attn_run", "verify_attn_run_simt"):
                fn = getattr(lib, name)
                fn.argtypes = _RUN_ARGS
                fn.restype = _i32
            lib.verify_attn_run_profiled.argtypes = [_i32, _p] + _RUN_ARGS
            lib.verify_attn_run_profiled.restype = _i32
            lib.verify_attn_save_kv.argtypes = [_p, _i64, _p, _i64, _p, _i64, _p, ctypes.c_size_t, _p]
            lib.verify_attn_save_kv.restype = _i32
            lib.verify_attn_save_and_run.argtypes = [_p, _i64] + _RUN_ARGS
            lib.verify_attn_save_and_run.restype = _i32
            lib.verify_attn_check_wait_timeout.argtypes = [ctypes.c_uint64, _p, ctypes.c_size_t, _p]
            lib.verify_attn_check_wait_timeout.restype = _i32
            lib.verify_attn_status_string.argtypes = [_i32]
            lib.verify_attn_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def header_symbols():
    """Names of the functions include/verify_attn.h declares."""
    text = open(HEADER).read()
    return re.findall(r"VERIFY_ATTN_API\s+[\w\s\*]+?\b(verify_attn_\w+)\s*\(", text)


def status_string(code: int) -> str:
    return load_library().verify_attn_status_string(int(code)).decode()


def workspace_size(batch: int, max_q_per_req: int, num_heads: int, num_splits: int) -> int:
    n = int(load_library().verify_attn_workspace_size(batch, max_q_per_req, num_heads, num_splits))
    if n == 0:
        raise VerifyAttnError("invalid capacities for the workspace")
    return n


def init() -> None:
    rc = load_library().verify_attn_init()
    if rc != 0:
        raise VerifyAttnError(f"verify_attn_init: {status_string(rc)}")


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr() if t is not None and t.numel() else 0)


def _check_dev(name, t, dtype):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def verify_attn(q: torch.Tensor, kv_pool: torch.Tensor, qo_indptr: torch.Tensor,
                kv_indptr: torch.Tensor, kv_indices: torch.Tensor, out_cache_loc: torch.Tensor,
                custom_mask: torch.Tensor, mask_indptr: torch.Tensor, sm_scale: float, *,
                out: torch.Tensor, workspace: torch.Tensor, max_q_per_req: int, num_splits: int,
                impl: str = "tc", stream: Optional[torch.cuda.Stream] = None,
                events=None, kv_new: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Tree-verify attention into ``out`` ([sum T_b, H, 512] bf16).

    Tensors are used in place (no copies): q [sum T_b, H, 576] bf16 with a
    contiguous last dim, kv_pool [pool, 576] bf16 contiguous, int32
    qo_indptr/kv_indptr/kv_indices, int64 out_cache_loc/mask_indptr, uint8
    packed custom_mask, uint8 workspace of at least ``workspace_size(...)``.
    ``impl``: "tc" (production) or "simt" (CUDA-core cross-check).
    ``events``: optional four torch.cuda.Event objects recorded at the start
    of the call, before the split kernel, between it and the combine, and
    after the combine.
    ``kv_new``: optional [sum T_b, 576] bf16 rows of the draft tokens; when
    given, the library first writes them into ``kv_pool`` at
    ``out_cache_loc`` (the KV save) and the attention reads them
    (verify_attn_save_and_run; production kernel only, no events).
    """
    lib = load_library()
    _check_dev("q", q, torch.bfloat16)
    _check_dev("kv_pool", kv_pool, torch.bfloat16)
    _check_dev("out", out, torch.bfloat16)
    for name, t, dt in (("qo_indptr", qo_indptr, torch.int32), ("kv_indptr", kv_indptr, torch.int32),
                        ("kv_indices", kv_indices, torch.int32), ("out_cache_loc", out_cache_loc, torch.int64),
                        ("custom_mask", custom_mask, torch.uint8), ("mask_indptr", mask_indptr, torch.int64),
                        ("workspace", workspace, torch.uint8)):
        _check_dev(name, t, dt)
    if q.dim() != 3 or q.shape[2] != LATENT_DIM or q.stride(2) != 1:
        raise ValueError("q must be [tokens, heads, 576] with a contiguous last dim")
    if out.dim() != 3 or out.shape[2] != V_DIM or out.stride(2) != 1 or out.shape[:2] != q.shape[:2]:
        raise ValueError("out must be [tokens, heads, 512] with a contiguous last dim")
    if kv_pool.dim() != 2 or kv_pool.shape[1] != LATENT_DIM or not kv_pool.is_contiguous():
        raise ValueError("kv_pool must be a contiguous [pool_size, 576] tensor")
    for name, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr), ("kv_indices", kv_indices),
                    ("out_cache_loc", out_cache_loc), ("custom_mask", custom_mask),
                    ("mask_indptr", mask_indptr), ("workspace", workspace)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    batch = qo_indptr.numel() - 1
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    if impl not in ("tc", "simt"):
        raise ValueError(f"unknown impl {impl!r}")
    if kv_new is not None:
        _check_dev("kv_new", kv_new, torch.bfloat16)
        if kv_new.dim() != 2 or kv_new.shape[1] != LATENT_DIM or kv_new.stride(1) != 1 or kv_new.shape[0] < q.shape[0]:
            raise ValueError("kv_new must be [>= tokens, 576] with a contiguous last dim")
        if impl != "tc" or events is not None:
            raise ValueError("kv_new runs with the production kernel and without events")
        fn = lambda *a: lib.verify_attn_save_and_run(_ptr(kv_new), kv_new.stride(0), *a)
    elif events is not None:
        for e in events:                 # torch creates the CUDA event lazily, on first record
            if e is not None and not e.cuda_event:
                e.record(s)
        ev = (ctypes.c_void_p * 4)(*[e.cuda_event if e is not None else 0 for e in events])
        fn = lambda *a: lib.verify_attn_run_profiled(0 if impl == "tc" else 1, ev, *a)
    else:
        fn = lib.verify_attn_run if impl == "tc" else lib.verify_attn_run_simt
    rc = fn(_ptr(q), q.stride(0), q.stride(1), _ptr(kv_pool), kv_pool.shape[0], _ptr(qo_indptr),
            _ptr(kv_indptr), _ptr(kv_indices), _ptr(out_cache_loc), _ptr(custom_mask),
            _ptr(mask_indptr), float(sm_scale), _ptr(out), out.stride(0), out.stride(1), batch,
            int(max_q_per_req), q.shape[1], int(num_splits), _ptr(workspace),
            workspace.numel(), ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise VerifyAttnError(f"verify_attn_run: {status_string(rc)} ({rc})")
    return out


def save_kv(kv_new: torch.Tensor, out_cache_loc: torch.Tensor, kv_pool: torch.Tensor, workspace: torch.Tensor,
            stream: Optional[torch.cuda.Stream] = None) -> None:
    """The KV save alone: kv_pool[out_cache_loc[i]] = kv_new[i] (in place).
    ``workspace``: a uint8 CUDA tensor of at least 256 bytes; its status word
    reports slots outside the pool (``read_status``)."""
    lib = load_library()
    _check_dev("kv_new", kv_new, torch.bfloat16)
    _check_dev("kv_pool", kv_pool, torch.bfloat16)
    _check_dev("out_cache_loc", out_cache_loc, torch.int64)
    _check_dev("workspace", workspace, torch.uint8)
    if kv_new.dim() != 2 or kv_new.shape[1] != LATENT_DIM or kv_new.stride(1) != 1:
        raise ValueError("kv_new must be [tokens, 576] with a contiguous last dim")
    if kv_pool.dim() != 2 or kv_pool.shape[1] != LATENT_DIM or not kv_pool.is_contiguous():
        raise ValueError("kv_pool must be a contiguous [pool_size, 576] tensor")
    if not out_cache_loc.is_contiguous() or out_cache_loc.numel() != kv_new.shape[0]:
        raise ValueError("out_cache_loc must be contiguous with one slot per kv_new row")
    s = stream if stream is not None else torch.cuda.current_stream(kv_pool.device)
    rc = lib.verify_attn_save_kv(_ptr(kv_new), kv_new.stride(0), _ptr(out_cache_loc), kv_new.shape[0],
                                 _ptr(kv_pool), kv_pool.shape[0], _ptr(workspace), workspace.numel(),
                                 ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise VerifyAttnError(f"verify_attn_save_kv: {status_string(rc)} ({rc})")


def check_wait_timeout(limit_ns: int, workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Launch the failure-path self-test (verify_attn_check_wait_timeout):
    one warp runs the split kernels' bounded wait on a barrier nothing
    arrives on, gives up after ``limit_ns`` and sets STATUS_TIMEOUT in the
    status word of ``workspace`` (a uint8 CUDA tensor of at least 256
    bytes; read it with ``read_status`` after the stream's work is done)."""
    _check_dev("workspace", workspace, torch.uint8)
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    rc = load_library().verify_attn_check_wait_timeout(int(limit_ns), _ptr(workspace), workspace.numel(),
                                                        ctypes.c_void_p(s.cuda_stream))
    if rc != 0:
        raise VerifyAttnError(f"verify_attn_check_wait_timeout: {status_string(rc)} ({rc})")


def read_status(workspace: torch.Tensor) -> int:
    """The device status word (byte 0 of the workspace); synchronises the device."""
    return int(workspace[:4].view(torch.int32).item()) & 0xFFFFFFFF


def tune_num_splits(q: torch.Tensor, kv_pool: torch.Tensor, qo_indptr: torch.Tensor, kv_indptr: torch.Tensor,
                    kv_indices: torch.Tensor, out_cache_loc: torch.Tensor, custom_mask: torch.Tensor,
                    mask_indptr: torch.Tensor, sm_scale: float, out: torch.Tensor, max_q_per_req: int,
                    candidates, impl: str = "tc", replays: int = 6, flush_bytes: int = 256 << 20) -> int:
    """The fastest of `candidates` (split counts) for this call, timed as a
    serving loop runs it: one call captured in a CUDA graph and replayed,
    L2 flushed (a `flush_bytes` write) before each replay, CUDA events around
    it; the median of `replays` after one warm-up replay.  Allocates a
    workspace per candidate and the flush buffer, so run it once per
    workload shape, outside any capture; `out` is overwritten."""
    num_heads = q.shape[1]
    batch = qo_indptr.numel() - 1
    flush = torch.empty(flush_bytes, dtype=torch.uint8, device=q.device)
    best, best_s = None, None
    for s in candidates:
        run = VerifyAttention(batch, max_q_per_req, num_heads, int(s), device=q.device, impl=impl)
        args = (q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask, mask_indptr, sm_scale, out)
        run(*args)
        torch.cuda.synchronize(q.device)
        graph, stream = torch.cuda.CUDAGraph(), torch.cuda.Stream(q.device)
        with torch.cuda.stream(stream):
            with torch.cuda.graph(graph, stream=stream):
                run(*args)
        torch.cuda.synchronize(q.device)
        times = []
        for k in range(replays + 1):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            graph.replay()
            e1.record()
            e1.synchronize()
            if k > 0:
                times.append(e0.elapsed_time(e1))
        if run.status() != 0:
            raise VerifyAttnError(f"tune_num_splits: device status {run.status():#x} with {s} splits")
        t = sorted(times)[len(times) // 2]
        if best is None or t < best:
            best, best_s = t, int(s)
        del graph, run
    return best_s


class VerifyAttention:
    """Holds a workspace sized for fixed capacities and runs the call.

    Allocate once (before any CUDA-graph capture), then call repeatedly --
    "The Capture-Safe Kernel", Decision 4 (workspace as a caller tensor) and
    Decision 3 (grid fixed by host capacities).

    Validate mode (``validate=True``, or the environment variable
    VERIFY_ATTN_VALIDATE=1): every call also runs the other kernel ("simt"
    for "tc" and the reverse) on the same live buffers into a scratch
    output, compares the two (|a - b| <= atol + rtol |b| per element), keeps
    the figures in ``last_validation`` and warns on a mismatch; the caller
    still receives the primary kernel's output.  This is the offline analogue
    of the pages' validate mode ("The Launch Wrapper", section The Design
    Decision: Three Modes of Operation).  It synchronises, so it is for eager
    runs, not for graph capture.
    """

    def __init__(self, batch: int, max_q_per_req: int, num_heads: int, num_splits: int,
                 device="cuda", impl: str = "tc", validate: Optional[bool] = None,
                 atol: float = 1e-2, rtol: float = 1e-2):
        self.batch, self.max_q_per_req = batch, max_q_per_req
        self.num_heads, self.num_splits, self.impl = num_heads, num_splits, impl
        if validate is None:
            validate = os.environ.get("VERIFY_ATTN_VALIDATE", "0") == "1"
        self.validate, self.atol, self.rtol = bool(validate), float(atol), float(rtol)
        self.last_validation = None
        init()
        self.workspace = torch.empty(workspace_size(batch, max_q_per_req, num_heads, num_splits),
                                     dtype=torch.uint8, device=device)
        self._check_ws = None

    def __call__(self, q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                 mask_indptr, sm_scale, out, stream=None, events=None, kv_new=None):
        if qo_indptr.numel() - 1 > self.batch:
            raise ValueError("batch exceeds the workspace capacity")
        res = verify_attn(q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                          mask_indptr, sm_scale, out=out, workspace=self.workspace,
                          max_q_per_req=self.max_q_per_req, num_splits=self.num_splits,
                          impl=self.impl, stream=stream, events=events, kv_new=kv_new)
        if self.validate:
            self._cross_check(q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                              mask_indptr, sm_scale, out, stream)
        return res

    def _cross_check(self, q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                     mask_indptr, sm_scale, out, stream):
        if self._check_ws is None:
            self._check_ws = torch.empty_like(self.workspace)
        other = "simt" if self.impl == "tc" else "tc"
        # The comparison runs on the stream both kernels ran on, so its reads
        # (and the synchronising .item() calls) come after them.
        s = stream if stream is not None else torch.cuda.current_stream(out.device)
        with torch.cuda.stream(s):
            ref = torch.empty_like(out)
            verify_attn(q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask, mask_indptr,
                        sm_scale, out=ref, workspace=self._check_ws, max_q_per_req=self.max_q_per_req,
                        num_splits=self.num_splits, impl=other, stream=s)
            a, b = out.float(), ref.float()
            diff = (a - b).abs()
            excess = diff - (self.atol + self.rtol * b.abs())
            rec = {"against": other, "max_abs_diff": float(diff.max()) if diff.numel() else 0.0,
                   "max_excess": float(excess.max()) if excess.numel() else float("-inf"),
                   "status": read_status(self.workspace), "check_status": read_status(self._check_ws)}
        rec["ok"] = bool(rec["max_excess"] <= 0 and rec["status"] == 0 and rec["check_status"] == 0)
        self.last_validation = rec
        if not rec["ok"]:
            warnings.warn(f"verify-attn validate: {self.impl} vs {other}: {rec}")

    def status(self) -> int:
        return read_status(self.workspace)
