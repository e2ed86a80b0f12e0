"""The Python example in README.md runs as written (needs a GB300), and its
outputs agree with the calls' documented shapes and with the oracle's
fake-quantized values."""
import os
import re

import numpy as np
import pytest
import torch

import oracle
from gpu_common import as_oracle_input, assert_eq, bits

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def readme_example() -> str:
    with open(os.path.join(ROOT, "README.md")) as f:
        text = f.read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert len(blocks) == 1
    return blocks[0]


def test_readme_example_runs():
    ns = {}
    torch.manual_seed(0)
    exec(compile(readme_example(), "README.md", "exec"), ns)
    torch.cuda.synchronize()
    x, xhat, mask, rq, cq = ns["x"], ns["xhat"], ns["mask"], ns["rq"], ns["cq"]
    assert xhat.shape == x.shape and xhat.dtype == torch.bfloat16
    assert rq.codes.shape == (4096, 2048) and cq.codes.shape == (4096, 2048)
    assert ns["dx"].shape == x.shape
    assert ns["gq"].codes.shape == (4096, 2048) and ns["gqt"].codes.shape == (4096, 2048)
    c, err = ns["c"], ns["err"]
    assert c.shape == (4096, 2048) and c.dtype == torch.bfloat16
    assert int(err.item()) == 0
    # the fake-quantized values of a few rows against the oracle
    xo = as_oracle_input(x)
    ref = oracle.quantize(xo[:64], oracle.NVFP4, want_xhat=True,
                          amax_in=float(np.abs(xo).max()))["row"]
    assert_eq("xhat", bits(xhat[:64]), oracle.f32_to_bf16_bits(ref["xhat"]))
    assert np.isfinite(c.float().cpu().numpy()).all()
