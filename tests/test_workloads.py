"""Host logic of the synthetic workloads: counted work under the causal mask and
the key/value head count of grouped-query workloads."""
import importlib.util
import os

import numpy as np
import pytest

from bf16_forward_attention_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (256, 256), (300, 300), (129, 1000), (700, 200),
                                   (1, 4096), (4096, 1)])
def test_causal_visible_pairs_brute_force(Sq, Sk):
    w = inputs.Workload("c", "bhsd", 1, 1, Sq, Sk, causal=True)
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    assert w.visible_pairs == int((j <= i + (Sk - Sq)).sum())
    assert w.flops == 4 * 128 * w.visible_pairs


def test_unmasked_flops_unchanged():
    w = inputs.WORKLOADS["self8k"]
    assert w.flops == 4 * 2 * 16 * 8192 * 8192 * 128


def test_gqa_shapes():
    w = inputs.Workload("g", "bshd", 1, 8, 64, 96, hkv=2, seed=5)
    q, k, v = inputs.make_qkv(w)
    assert tuple(q.shape) == (1, 64, 8, 128)
    assert tuple(k.shape) == tuple(v.shape) == (1, 96, 2, 128)
    # Without grouping, the key/value draws are those of the plain workload.
    _, k1, _ = inputs.make_qkv(w.scaled(hkv=0))
    assert tuple(k1.shape) == (1, 96, 8, 128)


def test_io_bytes_closed_forms():
    # Q and O: B*H*Sq*d each; K and V: B*Hkv*Sk*d each; 2 bytes per element.
    assert inputs.WORKLOADS["self8k"].io_bytes == 4 * 2 * 16 * 8192 * 128 * 2
    assert inputs.WORKLOADS["gqa8k"].io_bytes == (2 * 2 * 16 * 8192 + 2 * 2 * 4 * 8192) * 128 * 2
    w = inputs.WORKLOADS["varlen16"]
    tokens = sum(n for n, _ in w.seqlens)
    assert w.io_bytes == 4 * tokens * 16 * 128 * 2


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


PEAKS = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0, "hbm_gbs": 8000.0}


@pytest.mark.parametrize("name,bound", [("short77", "hbm"), ("tiny", "hbm"),
                                        ("self8k", "tensor"), ("cross4k32k", "tensor"),
                                        ("causal8k", "tensor")])
def test_roofline_bound_follows_intensity(name, bound):
    bench = _bench()
    w = inputs.WORKLOADS[name]
    got, achieved, peak, unit = bench.roofline_of(w.flops, w.io_bytes, 1e-3, PEAKS, False)
    assert got == bound
    if bound == "hbm":
        assert (peak, unit) == (8000.0, "GB/s")
        assert achieved == pytest.approx(w.io_bytes / 1e-3 / 1e9)
    else:
        assert (peak, unit) == (2000.0, "TFLOP/s")
        assert achieved == pytest.approx(w.flops / 1e-3 / 1e12)


def test_roofline_ridge_and_sustained_peak():
    bench = _bench()
    # The ridge is 2000e12 / 8000e9 = 250 flop per byte (225 with the sustained peak).
    assert bench.roofline_of(249e9, 1e9, 1.0, PEAKS, False)[0] == "hbm"
    assert bench.roofline_of(251e9, 1e9, 1.0, PEAKS, False)[0] == "tensor"
    assert bench.roofline_of(240e9, 1e9, 1.0, PEAKS, True)[:3] == ("tensor", 0.24, 1800.0)
