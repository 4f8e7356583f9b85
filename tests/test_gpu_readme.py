"""The usage example of README.md runs as written on the GPU (one pass, then a loop driven by a
caller's denoiser hook)."""
import re
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parents[1]


@pytest.mark.gpu
def test_readme_usage_example_runs():
    text = (ROOT / "README.md").read_text()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)
    torch.cuda.synchronize()
    out, res, dg = ns["out"], ns["res"], ns["dg"]
    assert int(out["status"][0]) == 0 and int(res["status"][0]) == 0
    fields = dg.state_fields(res["state"])
    assert 1 <= int(fields["passes"][0]) <= 48 and int(fields["done"][0]) == 1
    V = ns["V"]
    assert int(res["canvas"].min()) >= 0 and int(res["canvas"].max()) < V
