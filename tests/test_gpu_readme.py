"""The README's Python example runs as written on a GPU, and its device
status check sees a failure flagged by a kernel (a bare "cuda" names the
current device, as the tensors' own "cuda:0" does)."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def test_readme_example_runs():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    # the example's outputs are written and finite
    for name in ("z", "o", "dres", "dypre"):
        for x in scope[name]:
            assert torch.isfinite(x.float()).all(), name


def test_status_word_is_the_same_for_cuda_and_cuda0():
    from sp_boundary_norm_gb300 import binding as sp
    assert sp.device_status("cuda") is sp.device_status(torch.device("cuda", 0))
    sp.device_status("cuda:0").fill_(6)
    with pytest.raises(sp.SpError):
        sp.check_device_status("cuda")
    sp.check_device_status(torch.device("cuda:0"))   # reset by the check above
