"""C-ABI checks that need no GPU: the library loads, exports every declared
symbol, sizes workspaces, and rejects bad host arguments before any CUDA call."""
import ctypes
import math
import re

import pytest

from speculative_decode_mla_paged_gb300 import api, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return api.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = api.header_symbols()
    assert set(names) >= {"verify_attn_workspace_size", "verify_attn_init", "verify_attn_run",
                          "verify_attn_run_simt", "verify_attn_status_string"}
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/verify_attn.h but not exported"


def test_workspace_size_layout(lib):
    # 256-B header + fp32 partials + lse rounded to 256 B
    rows = 2 * 16 * 8
    expect = 256 + 4 * rows * 512 * 4 + math.ceil(4 * rows * 4 / 256) * 256
    assert api.workspace_size(2, 16, 8, 4) == expect
    assert lib.verify_attn_workspace_size(1, 8, 0, 4) == 0
    assert lib.verify_attn_workspace_size(1, 8, 8, 0) == 0
    assert lib.verify_attn_workspace_size(1, 8, 8, 257) == 0


def _header_text():
    return open(api.HEADER).read()


def test_status_strings(lib):
    codes = {name: int(v) for name, v in re.findall(r"\b(VA_ERR_\w+)\s*=\s*(-\d+)", _header_text())}
    assert len(codes) >= 9 and sorted(codes.values()) == list(range(-len(codes), 0))
    for code in [0] + list(codes.values()):
        assert api.status_string(code) != "unknown status"
    assert api.status_string(-99) == "unknown status"


def test_binding_constants_match_the_header():
    defs = {k: int(v, 0) for k, v in re.findall(r"#define\s+(\w+)\s+(0x[0-9a-fA-F]+|\d+)u?\b", _header_text())}
    assert defs["VERIFY_ATTN_LATENT_DIM"] == api.LATENT_DIM == 576
    assert defs["VERIFY_ATTN_V_DIM"] == api.V_DIM == 512
    assert defs["VERIFY_ATTN_MAX_SPLITS"] == api.MAX_SPLITS
    assert defs["VA_STATUS_BAD_SLOT"] == api.STATUS_BAD_SLOT
    assert defs["VA_STATUS_BAD_META"] == api.STATUS_BAD_META
    assert defs["VA_STATUS_TIMEOUT"] == api.STATUS_TIMEOUT
    assert (defs["VERIFY_ATTN_IMPL_TC"], defs["VERIFY_ATTN_IMPL_SIMT"]) == (0, 1)


A = 0x100000  # a fake, well-aligned device address: never dereferenced on the host path


def _call(lib, **over):
    args = dict(q=A, qst=8 * 576, qsh=576, pool=A, pool_size=4096, qo=A, kvp=A, kvi=A, ocl=A,
                mask=A, mip=A, scale=0.07, out=A, ost=8 * 512, osh=512, batch=1, maxq=8, heads=8,
                splits=4, ws=A, ws_bytes=1 << 30, stream=0)
    args.update(over)
    v = lambda x: ctypes.c_void_p(x)
    return lib.verify_attn_run(v(args["q"]), args["qst"], args["qsh"], v(args["pool"]), args["pool_size"],
                               v(args["qo"]), v(args["kvp"]), v(args["kvi"]), v(args["ocl"]),
                               v(args["mask"]), v(args["mip"]), args["scale"], v(args["out"]),
                               args["ost"], args["osh"], args["batch"], args["maxq"], args["heads"],
                               args["splits"], v(args["ws"]), args["ws_bytes"], v(args["stream"]))


@pytest.mark.parametrize("over,code", [
    (dict(q=0), -1), (dict(pool=0), -1), (dict(qo=0), -1), (dict(mask=0), -1), (dict(ws=0), -1),
    (dict(out=0), -1), (dict(mip=0), -1),
    (dict(q=A + 8), -2), (dict(out=A + 4), -2), (dict(ws=A + 128), -2), (dict(qst=8 * 576 + 4), -2),
    (dict(osh=513), -2),
    (dict(heads=0), -3), (dict(batch=-1), -3), (dict(pool_size=0), -3),
    (dict(ws_bytes=1000), -4),
    (dict(splits=0), -5), (dict(splits=257), -5),
    (dict(scale=float("nan")), -7), (dict(scale=float("inf")), -7),
])
def test_bad_host_arguments_are_rejected(lib, over, code):
    assert _call(lib, **over) == code


def test_valid_arguments_without_gpu_report_device_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert _call(lib) == -8
