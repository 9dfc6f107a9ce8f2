"""Causal mask (bottom-right aligned) and grouped-query heads through attn_fwd_ex,
against the fp64 oracle on a GB300."""
import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_fp64

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _qkv(layout, B, Hq, Hkv, Sq, Sk, seed, std=1.0):
    w = inputs.Workload("ex", layout, B, Hq, Sq, Sk, seed=seed, qk_std=std)
    q, _, _ = inputs.make_qkv(w)
    wk = inputs.Workload("ex", layout, B, Hkv, Sq, Sk, seed=seed + 1, qk_std=std)
    _, k, v = inputs.make_qkv(wk)
    return q, k, v


@pytest.mark.parametrize("layout,B,Hq,Hkv,Sq,Sk,causal", [
    ("bhsd", 1, 2, 2, 256, 256, True),
    ("bshd", 1, 2, 2, 300, 300, True),
    ("bhsd", 2, 2, 2, 129, 1000, True),     # Sq < Sk: every row sees the early keys
    ("bshd", 1, 1, 1, 700, 200, True),      # Sq > Sk: the first 500 rows see no key
    ("bhsd", 1, 8, 2, 333, 777, False),
    ("bshd", 2, 6, 3, 257, 257, True),
    ("bhsd", 1, 4, 1, 1, 4096, True),
])
@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
def test_ex_parity(layout, B, Hq, Hkv, Sq, Sk, causal, mode):
    q, k, v = _qkv(layout, B, Hq, Hkv, Sq, Sk, seed=900 + Sq + Sk + Hq)
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, layout=layout,
                           rounding=mode)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout,
                           causal=causal)
    # Causal rows near the start see few keys, so outputs reach magnitude ~4.
    assert_parity(compare(bits_of(out), exact, mode), excess=causal)


def test_ex_non_causal_equals_attn_fwd_bitwise():
    q, k, v = (t.cuda() for t in _qkv("bhsd", 1, 3, 3, 300, 500, seed=950))
    a = attn.attn_fwd(q, k, v)
    b = attn.attn_fwd_ex(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_gqa_equals_repeated_heads_bitwise():
    q, k, v = (t.cuda() for t in _qkv("bshd", 1, 8, 2, 300, 600, seed=951))
    a = attn.attn_fwd_ex(q, k, v, layout="bshd", causal=True)
    kr = k.repeat_interleave(4, dim=2).contiguous()
    vr = v.repeat_interleave(4, dim=2).contiguous()
    b = attn.attn_fwd_ex(q, kr, vr, layout="bshd", causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_causal_wide_logits_and_negative_scale():
    q, k, v = _qkv("bhsd", 1, 2, 1, 400, 400, seed=952, std=8.0)
    for scale in (inputs.default_scale(), -0.05):
        out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=scale)
        torch.cuda.synchronize()
        exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), scale, "bhsd", causal=True)
        assert_parity(compare(bits_of(out), exact, "rtz"), max_abs_err=None)


def test_causal_zero_scale_is_mean_of_visible_rows():
    # scale 0: every visible logit is 0, so each row is the mean of its visible V rows.
    q, k, v = _qkv("bshd", 1, 2, 2, 300, 420, seed=953)
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=True, layout="bshd", scale=0.0)
    torch.cuda.synchronize()
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), 0.0, "bshd", causal=True)
    assert_parity(compare(bits_of(out), exact, "rtne"), excess=True)
