"""Packed variable-length batches through attn_fwd_varlen, against the fp64 oracle
on a GB300."""
import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_varlen_fp64

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _batch(lq, lk, Hq, Hkv, seed):
    w = inputs.Workload("vl", "thd", len(lq), Hq, max(lq), max(lk), seed=seed, hkv=Hkv,
                        seqlens=tuple(zip(lq, lk)))
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    return q, k, v, cq, ck


def _run(q, k, v, cq, ck, causal, mode="rtne", max_sq=None, scale=None):
    cqd = torch.from_numpy(cq).cuda()
    ckd = torch.from_numpy(ck).cuda()
    max_sq = int(np.diff(cq).max()) if max_sq is None else max_sq
    out = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), cqd, ckd, max(1, max_sq),
                               causal=causal, rounding=mode, scale=scale)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("lq,lk,Hq,Hkv", [
    ([1, 127, 128, 129, 300, 513], [1, 127, 128, 129, 300, 513], 2, 2),
    ([5, 400, 0, 260], [700, 3, 9, 128], 4, 2),
    ([10, 20, 257], [0, 30, 1], 2, 1),        # a sequence with no keys: NaN rows
])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
def test_varlen_parity(lq, lk, Hq, Hkv, causal, mode):
    q, k, v, cq, ck = _batch(lq, lk, Hq, Hkv, seed=1000 + sum(lq) + Hq)
    out = _run(q, k, v, cq, ck, causal, mode)
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    exact = attention_varlen_fp64(f64_of(q), f64_of(k), f64_of(v), cq, ck,
                                  inputs.default_scale(), causal=causal)
    # Short causal rows and short sequences give outputs up to magnitude ~4.
    assert_parity(compare(bits_of(out), exact, mode), excess=True)


@pytest.mark.parametrize("causal", [False, True])
def test_equal_lengths_equal_batched_call_bitwise(causal):
    B, S, H = 3, 300, 2
    q, k, v, cq, ck = _batch([S] * B, [S] * B, H, H, seed=1100)
    got = _run(q, k, v, cq, ck, causal)
    # The same tokens as a BSHD batch (B, S, H, d).
    qb, kb, vb = (t.reshape(B, S, H, 128).cuda() for t in (q, k, v))
    want = attn.attn_fwd_ex(qb, kb, vb, causal=causal, layout="bshd")
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16).reshape(-1), want.view(torch.int16).reshape(-1))


def test_loose_max_seqlen_bound_changes_nothing():
    q, k, v, cq, ck = _batch([70, 300, 129], [90, 310, 129], 2, 2, seed=1101)
    a = _run(q, k, v, cq, ck, True)
    b = _run(q, k, v, cq, ck, True, max_sq=int(cq[-1]))
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_invalid_offsets_are_reported_and_cleared():
    q, k, v, cq, ck = _batch([100, 100, 100], [100, 100, 100], 1, 1, seed=1102)
    bad_q = np.array([0, 100, 50, 300], dtype=np.int32)    # a negative length
    _run(q, k, v, bad_q, ck, False, max_sq=300)
    assert attn.attn_fwd_last_error() == attn.ATTN_ERR_SEQLENS
    past_end = np.array([0, 100, 200, 400], dtype=np.int32)  # runs past total_q
    _run(q, k, v, past_end, ck, False, max_sq=200)
    assert attn.attn_fwd_last_error() == attn.ATTN_ERR_SEQLENS
    too_long = np.array([0, 250, 280, 300], dtype=np.int32)  # longer than max_seqlen_q
    _run(q, k, v, too_long, ck, False, max_sq=100)
    assert attn.attn_fwd_last_error() == attn.ATTN_ERR_SEQLENS
    # The status was cleared by reading it; a valid call is clean and correct.
    out = _run(q, k, v, cq, ck, False)
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    exact = attention_varlen_fp64(f64_of(q), f64_of(k), f64_of(v), cq, ck, inputs.default_scale())
    assert_parity(compare(bits_of(out), exact, "rtne"))


def test_varlen_wide_logits_negative_and_zero_scale():
    w = inputs.Workload("vl", "thd", 3, 2, 400, 500, seed=1103, qk_std=8.0,
                        seqlens=((400, 500), (33, 7), (130, 130)))
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    for scale in (inputs.default_scale(), -0.05, 0.0):
        out = _run(q, k, v, cq, ck, True, "rtz", scale=scale)
        exact = attention_varlen_fp64(f64_of(q), f64_of(k), f64_of(v), cq, ck, scale, causal=True)
        assert_parity(compare(bits_of(out), exact, "rtz"), max_abs_err=None)
