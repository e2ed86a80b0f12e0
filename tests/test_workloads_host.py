"""The seeded input generators draw what their recipes state (CPU, small
shapes of the same recipes): shapes, dtypes, distributions, outlier structure,
and identical bits for identical seeds."""
import math

import torch

from fp4_quantization_aware_fq_gb300 import workloads as W


def test_same_seed_same_bits():
    a = W.mxfp4_weight(shape=(64, 256), seed=1)
    b = W.mxfp4_weight(shape=(64, 256), seed=1)
    c = W.mxfp4_weight(shape=(64, 256), seed=2)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_nvfp4_small_is_standard_normal_fp32():
    x = W.nvfp4_small(shape=(256, 1024))
    assert x.dtype == torch.float32 and x.shape == (256, 1024)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_mxfp4_weight_has_a_thousandth_of_entries_scaled_by_100():
    x = W.mxfp4_weight(shape=(512, 512)).float()
    n = x.numel()
    k = n // 1000
    big = x.abs() > 0.15                              # 7.5 sigma of N(0, 0.02)
    # the scaled entries ~ N(0, 2): about 94% of them exceed 0.15
    assert 0.85 * k <= int(big.sum()) <= k
    assert abs(float(x[~big].std()) - 0.02) < 0.001


def test_nvfp4_act_has_its_outlier_columns():
    x = W.nvfp4_act(shape=(256, 512), n_outlier_cols=8).float()
    col_std = x.std(0)
    assert int((col_std > 10).sum()) == 8
    assert abs(float(col_std[col_std < 10].mean()) - 1.0) < 0.05


def test_channel_act_shares_its_channels_across_batches():
    a = W.channel_act(shape=(128, 512), seed=500, n_outlier_cols=16).float()
    b = W.channel_act(shape=(128, 512), seed=501, n_outlier_cols=16).float()
    ca = set(torch.nonzero(a.std(0) > 10).flatten().tolist())
    cb = set(torch.nonzero(b.std(0) > 10).flatten().tolist())
    want = set(W.outlier_channels(512, 16, 5).tolist())
    assert ca == cb == want
    assert not torch.equal(a, b)


def test_grad_2level_is_laplace():
    x = W.grad_2level(shape=(512, 1024), scale=1e-3)
    assert x.dtype == torch.bfloat16
    x = x.double()
    a = x.abs()
    assert abs(float(a.mean()) / 1e-3 - 1.0) < 0.02               # E|x| = b
    assert abs(float(a.median()) / (math.log(2) * 1e-3) - 1.0) < 0.02
    assert abs(float(x.mean())) < 2e-5


def test_qad_logits_teacher_and_student():
    zt, zs = W.qad_logits(shape=(64, 4096))
    assert zt.dtype == zs.dtype == torch.bfloat16
    assert abs(float(zt.float().std()) - 3.0) < 0.05
    assert abs(float((zs.float() - zt.float()).std()) - 0.3) < 0.02


def test_moe_weights_alternate_up_and_down_matrices():
    ws = W.moe_weights(experts=2, up_shape=(32, 64), down_shape=(64, 32))
    assert [tuple(w.shape) for w in ws] == [(32, 64), (64, 32)] * 2
    assert all(w.dtype == torch.bfloat16 for w in ws)
    allw = torch.cat([w.float().flatten() for w in ws])
    assert abs(float(allw.std()) - 0.02) < 0.002
    d1, d2 = W.master_update((64, 64), 1), W.master_update((64, 64), 2)
    assert d1.dtype == torch.float32 and not torch.equal(d1, d2)
    assert abs(float(d1.std()) - 1e-4) < 1e-5
