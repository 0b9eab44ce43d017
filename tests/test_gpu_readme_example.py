"""The usage example in README.md runs as written and its merged output for
one request matches the oracle."""

import os
import re

import numpy as np
import pytest
import torch

import oracle
from parity_utils import TOL_LSE, TOL_OUT, bits, max_abs

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example():
    from paged_decode_attention_attn_gb300 import build
    build.build()
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    env = {}
    torch.manual_seed(0)
    exec(compile(code, "README.md", "exec"), env)
    torch.cuda.synchronize()
    merged, merged_lse = env["merged"], env["merged_lse"]
    assert torch.isfinite(merged).all() and torch.isfinite(merged_lse).all()
    r = 0
    L, D, Hkv = env["L"], env["D"], env["Hkv"]
    ref = oracle.decode_layer(bits(env["q"][r]), bits(env["pool"]), env["table"][r].cpu().numpy(), L,
                              [tuple(x) for x in env["tiles"][r]], 1 / 16, Hkv, D,
                              new_row_bits=bits(env["new_rows"][r]))
    assert max_abs(merged[r].double().cpu().numpy(), ref["out"]) <= TOL_OUT
    assert max_abs(merged_lse[r].double().cpu().numpy(), ref["lse"]) <= TOL_LSE
