"""The debug flavour of the library (-DATTN_DEBUG=1): its bounds and protocol
checks stay silent on every entry point and the results equal the release build
bit for bit; its self-test raises exactly the debug status, which reading clears."""
import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _libraries():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    build.build(debug=True)
    attn.load_library(debug=False)
    attn.load_library(debug=True)


def _both(monkeypatch, fn):
    """fn() through the release library, then through the debug library; the
    debug run must leave its status clean."""
    monkeypatch.setenv("ATTN_FWD_DEBUG", "0")
    a = fn()
    torch.cuda.synchronize()
    monkeypatch.setenv("ATTN_FWD_DEBUG", "1")
    b = fn()
    torch.cuda.synchronize()
    assert attn.load_library(debug=True).attn_fwd_last_error() == attn.ATTN_OK
    monkeypatch.setenv("ATTN_FWD_DEBUG", "0")
    return a, b


def _qkv(layout, B, Hq, Hkv, Sq, Sk, seed):
    q, _, _ = inputs.make_qkv(inputs.Workload("d", layout, B, Hq, Sq, Sk, seed=seed))
    _, k, v = inputs.make_qkv(inputs.Workload("d", layout, B, Hkv, Sq, Sk, seed=seed + 1))
    return q.cuda(), k.cuda(), v.cuda()


def _same(a, b):
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("layout,Sq,Sk", [("bhsd", 300, 517), ("bshd", 129, 4000), ("bshd", 1, 1)])
def test_base_and_causal_gqa(monkeypatch, layout, Sq, Sk):
    q, k, v = _qkv(layout, 2, 4, 2, Sq, Sk, seed=1400 + Sq)
    _same(*_both(monkeypatch, lambda: attn.attn_fwd_ex(q, k, v, layout=layout)))
    _same(*_both(monkeypatch, lambda: attn.attn_fwd_ex(q, k, v, causal=True, layout=layout)))


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_persistent_short_keys(monkeypatch, layout):
    # 2 x 96 heads x 2 query-tile pairs = 384 items (more than the SMs) over 3 key
    # tiles: the persistent variant, one CTA per SM looping over items.
    q, k, v = _qkv(layout, 2, 96, 96, 500, 300, seed=1405)
    _same(*_both(monkeypatch, lambda: attn.attn_fwd(q, k, v, layout=layout)))


def test_split_kv(monkeypatch):
    q, k, v = _qkv("bhsd", 1, 2, 2, 256, 5000, seed=1410)
    _same(*_both(monkeypatch, lambda: attn.attn_fwd_splitkv(q, k, v, num_splits=5)))


def test_varlen(monkeypatch):
    w = inputs.Workload("d", "thd", 4, 2, 300, 300, seed=1420,
                        seqlens=((5, 7), (300, 200), (0, 3), (129, 0)))
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    cq, ck = (torch.from_numpy(a).cuda() for a in w.cu_seqlens)
    _same(*_both(monkeypatch, lambda: attn.attn_fwd_varlen(q, k, v, cq, ck, 300, causal=True)))


def test_selftest_reports_the_debug_status():
    dbg = attn.load_library(debug=True)
    q, k, v = _qkv("bhsd", 1, 2, 2, 256, 256, seed=1430)
    out = torch.empty_like(q)
    st = dbg.attn_fwd_debug_selftest(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), 0, 1,
                                     2, 256, 256, 128, inputs.default_scale(), 0,
                                     torch.cuda.current_stream().cuda_stream)
    assert st == attn.ATTN_OK
    torch.cuda.synchronize()
    assert dbg.attn_fwd_last_error() == attn.ATTN_ERR_DEBUG_CHECK
    assert dbg.attn_fwd_last_error() == attn.ATTN_OK  # reading cleared it
    # The launch itself computed normally (the poison performs no bad access).
    ref = attn.attn_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
