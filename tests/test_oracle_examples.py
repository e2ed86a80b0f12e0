"""Hand-worked examples (tests/golden/*.json) checked against the oracle (CPU)."""
import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _nibbles(codes, n):
    codes = codes.reshape(-1)
    out = []
    for e in range(n):
        out.append(int(codes[e // 2] >> (4 * (e % 2))) & 0xF)
    return out


def test_nvfp4_block_e1():
    g = _load("nvfp4_block_e1.json")
    x = np.array(g["x"], dtype=np.float32).reshape(g["rows"], g["cols"])
    r = oracle.quantize(x, oracle.NVFP4, want_xhat=True, want_mask=True)["row"]
    assert _nibbles(r["codes"], 32) == g["codes_nibbles"]
    assert list(r["codes"].reshape(-1)[:8]) == g["packed_bytes_block0"]
    assert list(r["scales"].reshape(-1)) == g["scales"]
    assert float(r["tscale"][0]) == g["tscale"]
    xh = r["xhat"].reshape(-1)
    assert list(xh[:16]) == g["xhat_block0"]
    assert np.signbit(xh[7])  # -0.1 quantizes to -0
    assert float(xh[16]) == g["xhat_first_of_block1"]
    assert int(r["mask"][0]) == g["mask_word0"]


def test_nvfp4_block_e2():
    g = _load("nvfp4_block_e2.json")
    x = np.array(g["x"], dtype=np.float32).reshape(g["rows"], g["cols"])
    r = oracle.quantize(x, oracle.NVFP4, want_xhat=True, want_mask=True)["row"]
    assert list(r["scales"].reshape(-1)) == g["scales"]
    assert _nibbles(r["codes"], 16) == g["codes_nibbles_block0"]
    assert list(r["xhat"].reshape(-1)[:16]) == g["xhat_block0"]
    assert int(r["mask"][0]) == g["mask_word0"]


def test_mxfp4_block_e3():
    g = _load("mxfp4_block_e3.json")
    x = np.array(g["x"], dtype=np.float32).reshape(g["rows"], g["cols"])
    r = oracle.quantize(x, oracle.MXFP4, want_xhat=True, want_mask=True)["row"]
    assert list(r["scales"].reshape(-1)) == g["scales"]
    assert _nibbles(r["codes"], 3) == g["codes_nibbles_first3"]
    assert list(r["xhat"].reshape(-1)[:3]) == g["xhat_first3"]
    m = int(r["mask"][0])
    assert [(m >> i) & 1 for i in range(3)] == g["mask_first3"]


def test_osci_flip_e4():
    g = _load("osci_flip_e4.json")
    w0 = np.zeros((g["rows"], g["cols"]), dtype=np.float32)
    for k, v in g["w0"].items():
        w0[0, int(k)] = v
    st = oracle.OsciState(w0, oracle.NVFP4)
    watched_codes = []
    for t in range(1, g["steps"] + 1):
        d = np.zeros_like(w0)
        d[0, 1] = g["delta_watched"] if t % 2 == 1 else -g["delta_watched"]
        d[0, 2] = g["delta_control"]
        out = st.step(d, offset=t)
        watched_codes.append(int(st.codes[0, 0] >> 4) & 0xF)
        # the tensor scale never moves (2688 is untouched)
        assert float(st.tscale[0]) == 1.0
        assert float(out["xhat"][0, 1]) == (0.5 if t % 2 == 1 else 0.0)
    assert watched_codes == [1, 0] * (g["steps"] // 2)
    assert float(st.dist_q[0, 1]) == g["expected_dist_q_watched"]
    assert abs(float(st.dist_m[0, 1]) - g["expected_dist_m_watched_approx"]) < 1e-5
    assert float(st.dist_q[0, 2]) == g["expected_dist_q_control"]
    assert float(st.dist_q[0, 0]) == 0.0 and float(st.dist_m[0, 0]) == 0.0
    n = st.reset(g["threshold"])
    assert n == g["expected_resets"]
    assert float(st.master[0, 1]) == g["expected_master_watched_after_reset"]
    assert abs(float(st.master[0, 2]) - 0.11) < 1e-6  # control weight untouched
    assert float(st.master[0, 0]) == 6.0 and float(st.master[0, 16]) == 2688.0
    assert not st.dist_q.any() and not st.dist_m.any()


def test_nvfp4_2level_e5():
    g = _load("nvfp4_2level_e5.json")
    x = np.zeros((g["rows"], g["cols"]), dtype=np.float32)
    for k, v in g["x_nonzero"].items():
        x[0, int(k)] = v
    r = oracle.quantize(x, oracle.NVFP4_2LEVEL, want_xhat=True, want_mask=True)["row"]
    assert list(r["tscale"].reshape(-1)) == g["tscale"]
    assert list(r["scales"].reshape(-1)) == g["scales"]
    want = [0] * g["cols"]
    for k, v in g["codes_nonzero"].items():
        want[int(k)] = v
    assert _nibbles(r["codes"], g["cols"]) == want
    xh = r["xhat"].reshape(-1)
    want_xh = np.zeros(g["cols"], np.float32)
    for k, v in g["xhat_nonzero"].items():
        want_xh[int(k)] = v
    assert np.array_equal(xh.view(np.uint32), want_xh.view(np.uint32))   # zeros are +0
    assert list(r["mask"].reshape(-1)) == g["mask_words"]

