"""The seeded input generators (CPU): the same seed gives the same bytes,
different seeds differ, the shapes and value recipes are the configs' own
(bf16 N(0,1) activations with 1% x20 outliers for prefill, gamma = 1 +
N(0, 0.1), E4M3 codes without the NaN codes, per-channel scales in
U(0.5, 2) * 1e-3), and the generators hold none of the method's arithmetic."""
import os
import re

import numpy as np

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _f32(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def test_same_seed_same_bytes_other_seed_differs():
    a, b, c = workloads.decode_fused(seed=0, n=256), workloads.decode_fused(seed=0, n=256), \
        workloads.decode_fused(seed=1, n=256)
    for k in ("x", "gamma", "B", "sb"):
        assert np.array_equal(a[k], b[k]), k
        assert not np.array_equal(a[k], c[k]), k


def test_decode_fused_recipe():
    d = workloads.decode_fused(seed=0)
    assert d["x"].shape == (32, 5120) and d["x"].dtype == np.uint16
    assert d["B"].shape == (10240, 5120) and d["B"].dtype == np.uint8
    assert d["sb"].shape == (10240,) and d["sb"].dtype == np.float32
    x = _f32(d["x"])
    assert abs(float(x.mean())) < 0.02 and abs(float(x.std()) - 1.0) < 0.02
    gm = _f32(d["gamma"])
    assert abs(float(gm.mean()) - 1.0) < 0.01 and abs(float(gm.std()) - 0.1) < 0.01
    assert not np.any((d["B"] & 0x7F) == 0x7F)                   # no NaN codes
    assert len(np.unique(d["B"])) == 254                          # every other code occurs
    assert d["sb"].min() >= 0.5e-3 and d["sb"].max() <= 2e-3
    assert d["eps"] == 1e-6 and d["s_a"] == np.float32(1 / 56)


def test_prefill_outliers():
    d = workloads.prefill(seed=0, m=256, n=8)
    x = np.abs(_f32(d["x"]))
    frac = float(np.mean(x > 6.0))                               # N(0,1) beyond 6 sigma: ~2e-9
    assert 0.005 < frac < 0.015                                   # the 1% scaled by 20
    w = _f32(d["w"])
    assert abs(float(w.std()) - 0.02) < 0.002


def test_layer_shapes_and_step_bytes():
    s = workloads.LayerShapes()
    assert (s.qkv, s.o, s.gate_up, s.down) == ((10240, 5120), (5120, 8192), (34816, 5120), (5120, 17408))
    per_layer = sum(n * k for (n, k) in (s.qkv, s.o, s.gate_up, s.down))
    assert per_layer == 361_758_720
    assert workloads.STEP_LAYERS * per_layer == 23_152_558_080


def test_generators_hold_no_method_arithmetic():
    """The shared input module neither imports the oracle nor the library,
    and has no quantiser or GEMM of its own."""
    text = open(os.path.join(ROOT, "workloads.py")).read()
    assert not re.search(r"^\s*(from|import)\s+(oracle|fp8_w8a8_scaled_gb300)\b", text, flags=re.M)
    for word in ("448", "amax", "rsqrt", "matmul", "@"):
        assert word not in re.sub(r"(#.*|\"\"\".*?\"\"\")", "", text, flags=re.S), word
