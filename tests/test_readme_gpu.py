"""The README's single-request example runs as written and matches the oracle."""
import os
import re

import pytest
import torch

from oracle import verify_request
from parity_util import assert_within_tolerance

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example() -> str:
    text = open(os.path.join(ROOT, "README.md")).read()
    section = text[text.index("## Python usage"):]
    m = re.search(r"```python\n(.*?)```", section, re.S)
    assert m, "no python block under 'Python usage'"
    return m.group(1)


def test_example_is_found_on_the_cpu():
    code = _example()
    assert "ddtree_verify_mla(" in code and "ddtree_verify_mla_check" in code
    compile(code, "README.md", "exec")


@pytest.mark.gpu
def test_readme_example_matches_oracle():
    torch.manual_seed(0)
    ns = {}
    exec(compile(_example(), "README.md", "exec"), ns)
    P, T = ns["P"], ns["T"]
    O_ref, L_ref = verify_request(ns["q_latent"].cpu(), ns["q_rope"].cpu(), ns["kv_pool"].cpu(),
                                  ns["kv_indices"].cpu(), P, ns["tree_parent"].tolist(), 192 ** -0.5)
    assert_within_tolerance(ns["out"], ns["lse"], O_ref, L_ref, "README example")
