"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake (a textual
substitution, always in bounds), builds it into a temporary library and runs
the pin suite against it in a child process.  The pins must fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "verify_attn_oracle.c")

MUTATIONS = {
    "drop_rope_dims": ("for (int d = 0; d < ORACLE_D; ++d)\n            dot +=",
                       "for (int d = 0; d < ORACLE_DV; ++d)\n            dot +="),
    "msb_first_bits": ("(mask[bit >> 3] >> (bit & 7)) & 1", "(mask[bit >> 3] >> (7 - (bit & 7))) & 1"),
    "v_from_wrong_dims": ("out[d] += w * bf16_to_double(vrow[d]);", "out[d] += w * bf16_to_double(vrow[d + 64]);"),
    "no_sm_scale": ("double s = a->sm_scale * dot;", "double s = dot;"),
    "ignore_mask_indptr": ("a->mask_indptr[b] + i * N + j", "i * N + j"),
    "softmax_sign": ("double w = exp(scores[j - k0] - m);", "double w = exp(m - scores[j - k0]);"),
    "mask_row_stride_prefix_len": ("a->mask_indptr[b] + i * N + j", "a->mask_indptr[b] + i * L + j"),
    "draft_slot_without_request_offset": ("return a->out_cache_loc[a->qo_indptr[b] + (j - L)];",
                                          "return a->out_cache_loc[j - L];"),
    "q_head_stride_dropped": ("+ (int64_t)h * a->q_stride_head;", "+ (int64_t)h * 0;"),
    "max_not_subtracted": ("double w = exp(scores[j - k0] - m);", "double w = exp(scores[j - k0]);"),
    "lse_in_log2": ("*lse_out = m + log(z);", "*lse_out = m + log2(z);"),
    "splits_averaged_equally": ("double w = exp(plse[s] - mx);", "double w = 1.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(lib), str(mutated), "-lm"],
                   check=True, capture_output=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"
