"""The README's Python example runs as written and its step matches the
separate calls (tag check, then append + attention) on the same inputs."""
import os
import re

import pytest
import torch

import fp8_quantised_paged_kv_gb300 as kvq

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example_code():
    text = open(os.path.join(ROOT, "README.md")).read()
    section = text[text.index("## Using it from Python"):]
    return re.search(r"```python\n(.*?)```", section, re.S).group(1)


def test_readme_example_runs_and_matches_separate_calls():
    torch.manual_seed(0)
    env = {}
    exec(compile(_example_code(), "README.md", "exec"), env)
    torch.cuda.synchronize()
    assert int(env["abort"].sum()) == 0
    # the same step as separate calls on a copy of the cache as it was before the step: the
    # new token is the only thing the step wrote, so write it back out and redo it
    desc, B, Hq = env["desc"], env["B"], env["Hq"]
    k2, v2 = env["k_cache"].clone(), env["v_cache"].clone()
    out2 = torch.empty_like(env["out"])
    ab2 = torch.empty_like(env["abort"])
    kvq.kvq_tag_check(env["block_table"], env["expected"], env["seq_lens"], env["ps"],
                      env["page_tags"], ab2)
    kvq.kvq_decode_attn_append(desc, env["q"], k2, v2, env["k_scale"], env["v_scale"],
                               env["block_table"], env["seq_lens"], 1 / env["math"].sqrt(env["D"]),
                               ab2, env["k_new"], env["v_new"], out2,
                               kvq.workspace_for(desc, B, Hq, env["maxp"]))
    torch.cuda.synchronize()
    assert torch.equal(ab2, env["abort"])
    assert torch.equal(out2.view(torch.int16), env["out"].view(torch.int16))
    assert torch.isfinite(env["out"].float()).all()
