"""fq_osci_update_noalloc (the OsciReset step for callers that cannot
allocate device memory, which keeps its scratch in a static device array)
must give the same results as fq_osci_update with a caller workspace, on two
calls in a row, so that scratch left over from the first call cannot leak
into the second.  Runs through the C ABI; collected last on purpose."""
import numpy as np
import pytest
import torch

from fp4_quantization_aware_fq_gb300 import fq
from fp4_quantization_aware_fq_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _state(shapes, cfg):
    master = [W.normal(s, 0.02, seed=60 + i).to(DEV) for i, s in enumerate(shapes)]
    return {
        "master": master,
        "dq": [torch.zeros_like(m) for m in master],
        "dm": [torch.zeros_like(m) for m in master],
        "prev": [fq.fq_quantize(m, cfg)[0] for m in master],
        "next": [fq.alloc_qtensor(*m.shape, cfg.format, DEV) for m in master],
        "xhat": [torch.empty(m.shape, dtype=torch.bfloat16, device=DEV) for m in master],
        "mask": [torch.zeros(((m.numel() + 7) // 8 + 15) // 16 * 16, dtype=torch.uint8,
                             device=DEV) for m in master],
    }


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_noalloc_update_matches_workspace_update_twice():
    shapes = [(64, 256), (128, 128), (32, 512)]
    cfg = fq.Config(fq.NVFP4, fq.RNE)
    ref = _state(shapes, cfg)
    new = _state(shapes, cfg)
    ws = torch.empty(fq.fq_osci_workspace_size(len(shapes)), dtype=torch.uint8, device=DEV)
    for t in (1, 2):
        deltas = [W.master_update(s, t, std=3e-3).to(DEV) for s in shapes]
        c = fq.Config(fq.NVFP4, fq.RNE, 0, t)
        fq.fq_osci_update(c, ref["master"], deltas, ref["dq"], ref["dm"], ref["prev"],
                          ref["next"], xhat=ref["xhat"], mask=ref["mask"], ws=ws)
        fq.fq_osci_update_noalloc(c, new["master"], deltas, new["dq"], new["dm"], new["prev"],
                                  new["next"], xhat=new["xhat"], mask=new["mask"])
        torch.cuda.synchronize()
        for i in range(len(shapes)):
            for k in ("master", "dq", "dm", "xhat", "mask"):
                assert _same(ref[k][i], new[k][i]), (t, i, k)
            for f in ("codes", "scales"):
                assert _same(getattr(ref["next"][i], f), getattr(new["next"][i], f)), (t, i, f)
            # NVFP4 writes only element 0 of its tensor-scale buffer
            assert _same(ref["next"][i].tscale[:1], new["next"][i].tscale[:1]), (t, i, "tscale")
        for st in (ref, new):
            st["prev"], st["next"] = st["next"], st["prev"]
    # the tensor scale of every tensor moved away from its initial value
    assert not np.isnan(ref["prev"][0].tscale[0].item())


def test_noalloc_rejects_more_tensors_than_its_scratch_holds():
    cfg = fq.Config(fq.NVFP4)
    m = [torch.zeros((16, 16), device=DEV)] * 65
    q = [fq.alloc_qtensor(16, 16, fq.NVFP4, DEV)] * 65
    with pytest.raises(fq.FqError) as e:
        fq.fq_osci_update_noalloc(cfg, m, m, m, m, q, q)
    assert e.value.status == 4  # FQ_ERR_WORKSPACE
