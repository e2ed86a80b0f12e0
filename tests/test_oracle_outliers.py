"""Pins for the oracle's static outlier retention ("Resumo Técnico:
TetraJet-v2", §2C) on the CPU: numpy reductions and sorts for the calibration
statistic and the channel choice, torch's float8_e4m3fn cast for the FP8
codes of the retained channels, and the effect the page describes (retained
outlier channels stop inflating the FP4 block scales of their rows)."""
import numpy as np
import torch

import oracle
from fp4_quantization_aware_fq_gb300 import workloads as W

RNG = np.random.default_rng(2024)


def _act(rows=96, cols=256, seed=0):
    return oracle.bf16_bits_to_f32(W.bf16_bits(
        W.nvfp4_act(shape=(rows, cols), seed=seed, n_outlier_cols=5))).reshape(rows, cols)


def test_channel_amax_is_running_column_max():
    a, b = _act(seed=1), _act(seed=2)
    got = oracle.channel_amax(b, oracle.channel_amax(a))
    want = np.maximum(np.abs(a).max(axis=0), np.abs(b).max(axis=0))
    assert np.array_equal(got, want)


def test_select_is_topk_with_low_index_ties():
    amax_c = RNG.uniform(0, 1, 300).astype(np.float32)
    amax_c[[10, 20, 30]] = 5.0                     # a three-way tie at the top
    amax_c[[40, 41]] = 4.0
    for k in (0, 1, 2, 4, 30, 300):
        sel = oracle.select_channels(amax_c, k)
        order = np.lexsort((np.arange(300), -amax_c.astype(np.float64)))
        want = np.sort(order[:k])
        assert np.array_equal(sel["idx"], want), k
        bits = np.unpackbits(sel["bitmap"].view(np.uint8), bitorder="little")[:300]
        assert np.array_equal(np.flatnonzero(bits), want)
        assert np.array_equal(sel["fp8_scale"], (amax_c[want] / np.float32(448)).astype(np.float32))
    assert list(oracle.select_channels(amax_c, 2)["idx"]) == [10, 20]


def test_retained_channels_are_fp8_e4m3():
    x = _act(seed=3)
    sel = oracle.select_channels(oracle.channel_amax(x), 12)
    out = oracle.quantize_outliers(x, sel["idx"], sel["fp8_scale"], oracle.NVFP4)
    s = sel["fp8_scale"].astype(np.float32)
    r = np.where(s == 0, np.float32(0), np.float32(1) / s).astype(np.float32)
    y = (x[:, sel["idx"]] * r).astype(np.float32)
    t = torch.from_numpy(np.clip(y, -448, 448)).to(torch.float8_e4m3fn)
    assert np.array_equal(out["fp8"], t.view(torch.uint8).numpy())
    dec = (t.to(torch.float32).numpy() * s).astype(np.float32)
    assert np.array_equal(out["xhat"][:, sel["idx"]], dec)


def test_fp4_part_is_the_tensor_without_retained_channels():
    x = _act(seed=4)
    sel = oracle.select_channels(oracle.channel_amax(x), 8)
    for fmt in (oracle.NVFP4, oracle.MXFP4, oracle.NVFP4_2LEVEL):
        out = oracle.quantize_outliers(x, sel["idx"], sel["fp8_scale"], fmt)
        xz = x.copy()
        xz[:, sel["idx"]] = 0.0
        ref = oracle.quantize(xz, fmt, want_xhat=True)["row"]
        assert np.array_equal(out["codes"], ref["codes"])
        assert np.array_equal(out["scales"], ref["scales"])
        keep = np.ones(x.shape[1], bool)
        keep[sel["idx"]] = False
        assert np.array_equal(out["xhat"][:, keep], ref["xhat"][:, keep])


def test_retention_shrinks_block_scales_and_error():
    x = _act(rows=128, cols=512, seed=5)
    sel = oracle.select_channels(oracle.channel_amax(x), 5)     # the 5 planted outlier channels
    plain = oracle.quantize(x, oracle.MXFP4, want_xhat=True)["row"]
    split = oracle.quantize_outliers(x, sel["idx"], sel["fp8_scale"], oracle.MXFP4)
    blocks = np.unique(sel["idx"] // 32)
    assert (split["scales"][:, blocks] <= plain["scales"][:, blocks]).all()
    assert (split["scales"][:, blocks] < plain["scales"][:, blocks]).mean() > 0.9
    err_plain = np.mean((plain["xhat"] - x) ** 2)
    err_split = np.mean((split["xhat"] - x) ** 2)
    assert err_split < 0.5 * err_plain
