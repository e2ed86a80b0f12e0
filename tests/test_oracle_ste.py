"""Pins for the oracle's straight-through-estimator backward (CPU only).

The STE lets the gradient through the quantize/dequantize operator and
zeroes it where the forward clipped ("Como o Treinamento com Quantização
Detecta e Recupera Precisão em Inferência de Baixa Precisão", "Detalhes
técnicos"): dx = dy where the mask bit of the element is 1, else +0.  The
mask layout is bit e % 8 of byte e / 8 for flat element e.

The expected dx is built here from numpy alone (``np.unpackbits`` with
little bit order and ``np.where`` on the raw bit patterns), which shares no
step with the oracle's word-and-shift loop; a hand-worked case and the E2
golden block (the saturating element gets no gradient) pin the meaning of
the bit.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _numpy_ste(dy_bits: np.ndarray, mask_words: np.ndarray) -> np.ndarray:
    n = dy_bits.size
    keep = np.unpackbits(mask_words.view(np.uint8), bitorder="little")[:n].astype(bool)
    return np.where(keep, dy_bits, dy_bits.dtype.type(0))


@pytest.mark.parametrize("itemsize", [2, 4])
@pytest.mark.parametrize("n", [8, 40, 1000, 4096 + 24])
def test_ste_backward_matches_numpy_bit_order(itemsize, n):
    rng = np.random.default_rng(1000 * itemsize + n)
    dt = np.uint16 if itemsize == 2 else np.uint32
    dy = rng.integers(0, np.iinfo(dt).max, size=n, dtype=dt, endpoint=True)
    # the last word is partial whenever n % 32 != 0
    mask = rng.integers(0, 2 ** 32, size=(n + 31) // 32, dtype=np.uint32)
    got = oracle.ste_backward(dy, mask)
    assert got.dtype == dy.dtype
    assert np.array_equal(got, _numpy_ste(dy, mask))


@pytest.mark.parametrize("itemsize", [2, 4])
def test_ste_backward_passes_bits_verbatim(itemsize):
    # special patterns pass unchanged where kept (no float arithmetic on dy):
    # -0, +inf, -inf, a NaN payload, the smallest subnormal, the largest finite
    if itemsize == 2:
        dy = np.array([0x8000, 0x7F80, 0xFF80, 0x7FC1, 0x0001, 0x7F7F, 0x3F80, 0xBF80],
                      dtype=np.uint16)
    else:
        dy = np.array([0x80000000, 0x7F800000, 0xFF800000, 0x7FC00123, 0x00000001,
                       0x7F7FFFFF, 0x3F800000, 0xBF800000], dtype=np.uint32)
    all_on = oracle.ste_backward(dy, np.array([0xFFFFFFFF], dtype=np.uint32))
    assert np.array_equal(all_on, dy)
    all_off = oracle.ste_backward(dy, np.array([0], dtype=np.uint32))
    assert np.array_equal(all_off, np.zeros_like(dy))   # +0, not -0, where dropped


def test_ste_backward_hand_worked():
    # mask word 0x00000005: elements 0 and 2 keep their gradient; elements 1
    # and 3..7 are clipped.  Element 32 sits in word 1, bit 0 (0x00000001).
    dy = np.arange(1, 41, dtype=np.uint32) * np.uint32(0x01010101)
    mask = np.array([0x00000005, 0x00000001], dtype=np.uint32)
    got = oracle.ste_backward(dy, mask)
    want = np.zeros_like(dy)
    want[[0, 2, 32]] = dy[[0, 2, 32]]
    assert np.array_equal(got, want)


def test_ste_backward_of_the_clipped_golden_block():
    # E2: [7, 1 x 15] under s_eff = 1.125 -- element 0 saturates (|7| > 6.75)
    # and its gradient is dropped; the other 15 pass.
    with open(os.path.join(GOLDEN, "nvfp4_block_e2.json")) as f:
        g = json.load(f)
    x = np.array(g["x"], dtype=np.float32).reshape(g["rows"], g["cols"])
    q = oracle.quantize(x, oracle.NVFP4, want_mask=True)["row"]
    assert int(q["mask"][0]) == g["mask_word0"]
    dy = np.full(g["cols"], 0x3F80, dtype=np.uint16)    # BF16 1.0 everywhere
    dx = oracle.ste_backward(dy, q["mask"])
    assert dx[0] == 0 and np.all(dx[1:16] == 0x3F80)
