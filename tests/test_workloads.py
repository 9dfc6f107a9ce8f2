"""Host logic of the synthetic workloads: counted work under the causal mask and
the key/value head count of grouped-query workloads."""
import numpy as np
import pytest

from bf16_forward_attention_gb300 import inputs


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
