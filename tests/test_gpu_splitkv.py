"""Split-KV (key range split over CTAs, fp32 partials merged by a second kernel)
against the fp64 oracle, on a GB300: same numerics bar as the fused path."""
import json

import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_fp64, attention_rows_fp64, bf16_bits_to_f64, to_bhsd

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _run(q, k, v, layout, mode, splits, scale=None):
    out = attn.attn_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), num_splits=splits, layout=layout,
                                rounding=mode, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    return out


@pytest.mark.parametrize("layout,B,H,Sq,Sk,splits", [
    ("bhsd", 1, 2, 256, 256, 2),
    ("bshd", 1, 2, 100, 1000, 3),
    ("bhsd", 2, 1, 300, 2049, 8),
    ("bshd", 1, 3, 1, 4096, 32),
    ("bhsd", 1, 1, 129, 130, 2),
])
@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
def test_split_parity(layout, B, H, Sq, Sk, splits, mode):
    w = inputs.Workload("split", layout, B, H, Sq, Sk, seed=500 + Sq + Sk + splits)
    q, k, v = inputs.make_qkv(w)
    out = _run(q, k, v, layout, mode, splits)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout)
    assert_parity(compare(bits_of(out), exact, mode))


def test_split_deterministic_and_close_to_fused():
    w = inputs.Workload("det", "bshd", 1, 4, 300, 3000, seed=501)
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    a = attn.attn_fwd_splitkv(q, k, v, num_splits=5, layout="bshd")
    b = attn.attn_fwd_splitkv(q, k, v, num_splits=5, layout="bshd")
    f = attn.attn_fwd(q, k, v, layout="bshd")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    from oracle import ulp_distance
    assert (ulp_distance(bits_of(a), bits_of(f)) <= 2).mean() > 0.999


def test_split_with_specials_and_empty_split():
    w = inputs.Workload("spec", "bhsd", 1, 2, 260, 600, seed=502)
    q, k, v = inputs.make_qkv(w)
    q[0, 0, 5, 17] = float("nan")           # NaN row
    k[0, 1, 500, 40] = float("inf")          # +Inf key in the last split
    q[0, 0, 0, 9] = 1.0
    k[0, 0, :256, 9] = float("-inf")         # row 0 of head 0: whole first split -Inf
    for mode in inputs.ROUNDINGS:
        out = _run(q, k, v, "bhsd", mode, 3)
        exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), "bhsd")
        stats = compare(bits_of(out), exact, mode)
        assert_parity(stats)
        assert stats["n_nonfinite"] > 128


def test_split_negative_scale():
    w = inputs.Workload("neg", "bhsd", 1, 2, 200, 700, seed=503)
    q, k, v = inputs.make_qkv(w)
    out = _run(q, k, v, "bhsd", "rtne", 4, scale=-0.09)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), -0.09, "bhsd")
    assert_parity(compare(bits_of(out), exact, "rtne"))


def test_split_long_keys_sampled():
    # Decode-like: few query rows, 128K keys, automatic split count.
    w = inputs.Workload("declike", "bshd", 1, 8, 256, 131072, seed=504)
    q, k, v = inputs.make_qkv(w)
    splits = attn.splitkv_num_splits(1, 8, 256, 131072)
    assert splits > 1
    out = _run(q, k, v, "bshd", "rtna", splits)
    qb, kb, vb = (to_bhsd(t.view(torch.int16).numpy(), "bshd") for t in (q, k, v))
    ob = to_bhsd(bits_of(out), "bshd")
    rows = np.array([0, 1, 127, 128, 200, 255])
    got, exact = [], []
    for h in range(8):
        exact.append(attention_rows_fp64(bf16_bits_to_f64(qb[0, h]), bf16_bits_to_f64(kb[0, h]),
                                         bf16_bits_to_f64(vb[0, h]), inputs.default_scale(), rows))
        got.append(ob[0, h, rows])
    stats = compare(np.concatenate(got), np.concatenate(exact), "rtna")
    print("\nPARITY split128k rtna: " + json.dumps(stats))
    assert_parity(stats)
