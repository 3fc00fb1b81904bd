"""The Python example in README.md runs as written and computes what the
README says: the partition puts rank r's tokens in q_local[r], and the
gradient return is the ordered binary32 sum of the writers' rows."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_example_runs_and_is_right(cpt, cuda_device):
    with open(README) as f:
        blocks = re.findall(r"```python\n(.*?)```", f.read(), flags=re.S)
    assert len(blocks) == 1
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    torch.cuda.synchronize()
    P, S = env["P"], env["S"]
    plan = env["plan"]
    l2g = torch.empty(S, dtype=torch.int32, device="cuda")
    cpt.cpt_index_map(plan, l2g, None)
    idx = l2g.long()
    assert torch.equal(env["q_local"].view(S, 20, 128), env["q"].index_select(0, idx))
    w = env["dk_writers"]
    acc = w[0].index_select(0, idx).float()
    for k in range(1, P):
        acc = acc + w[k].index_select(0, idx).float()
    assert torch.equal(acc.bfloat16().view(torch.int16), env["dk_owner"].view(S, 20, 128).view(torch.int16))
