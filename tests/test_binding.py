"""CPU tests of the Python binding: it fails loudly instead of computing
anywhere but the library's CUDA kernels -- a missing library, tensors that
are not on a CUDA device, wrong dtypes or shapes, and a machine without an
sm_103 GPU all raise."""
import numpy as np
import pytest
import torch

from speculative_decode_mla_paged_gb300 import api, build
from speculative_decode_mla_paged_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _cpu_args(inp):
    meta = {k: torch.from_numpy(np.ascontiguousarray(getattr(inp, k)))
            for k in ("qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask", "mask_indptr")}
    out = torch.empty(inp.total_q, inp.num_heads, W.V_DIM, dtype=torch.bfloat16)
    ws = torch.empty(1 << 16, dtype=torch.uint8)
    args = (inp.q, inp.kv_pool, meta["qo_indptr"], meta["kv_indptr"], meta["kv_indices"], meta["out_cache_loc"],
            meta["custom_mask"], meta["mask_indptr"], inp.sm_scale)
    return args, out, ws


def test_missing_library_raises(tmp_path, monkeypatch):
    monkeypatch.setattr(api, "_lib", None)
    monkeypatch.setattr(api, "LIB_PATH", str(tmp_path / "libverify_attn.so"))
    with pytest.raises(api.VerifyAttnError, match="missing"):
        api.load_library()
    inp = W.make_config_inputs("tiny")
    args, out, ws = _cpu_args(inp)
    with pytest.raises(api.VerifyAttnError):
        api.verify_attn(*args, out=out, workspace=ws, max_q_per_req=8, num_splits=2)


def test_host_tensors_are_rejected_not_computed():
    inp = W.make_config_inputs("tiny")
    args, out, ws = _cpu_args(inp)
    before = out.clone()
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.verify_attn(*args, out=out, workspace=ws, max_q_per_req=8, num_splits=2)
    assert torch.equal(out.view(torch.int16), before.view(torch.int16))   # nothing was written


@pytest.mark.parametrize("name,dtype", [("q", torch.float32), ("kv_indices", torch.int64),
                                        ("out_cache_loc", torch.int32), ("mask_indptr", torch.int32)])
def test_wrong_dtypes_are_rejected(name, dtype):
    inp = W.make_config_inputs("tiny")
    args, out, ws = _cpu_args(inp)
    names = ["q", "kv_pool", "qo_indptr", "kv_indptr", "kv_indices", "out_cache_loc", "custom_mask",
             "mask_indptr", "sm_scale"]
    args = list(args)
    i = names.index(name)
    args[i] = args[i].to(dtype)
    before = out.clone()
    # q is checked first, so its dtype error shows on any machine; the others
    # are refused too (on a machine without a GPU already as host tensors)
    with pytest.raises(TypeError if name == "q" else (TypeError, ValueError)):
        api.verify_attn(*args, out=out, workspace=ws, max_q_per_req=8, num_splits=2)
    assert torch.equal(out.view(torch.int16), before.view(torch.int16))


def test_invalid_capacities_raise():
    with pytest.raises(api.VerifyAttnError):
        api.workspace_size(1, 8, 8, 0)
    with pytest.raises(api.VerifyAttnError):
        api.workspace_size(1, 8, 0, 4)


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_no_gpu_means_an_error_not_a_fallback():
    with pytest.raises(api.VerifyAttnError, match="sm_103"):
        api.init()
    with pytest.raises(api.VerifyAttnError):
        api.VerifyAttention(1, 8, 8, 2, device="cpu")
