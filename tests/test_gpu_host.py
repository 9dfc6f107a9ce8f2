"""attn_fwd_host: host buffers in, host buffer out, copies overlapped with the
kernels in chunks. The chunks are sub-problems of the same kernel, so the result
must equal attn_fwd_ex on the device bit for bit."""
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


def _qkv(layout, B, Hq, Hkv, Sq, Sk, seed):
    q, _, _ = inputs.make_qkv(inputs.Workload("h", layout, B, Hq, Sq, Sk, seed=seed))
    _, k, v = inputs.make_qkv(inputs.Workload("h", layout, B, Hkv, Sq, Sk, seed=seed + 1))
    return q, k, v


# Shapes large enough that the planner cuts several chunks (>= 512 CTAs of 256
# query rows x one head):
# - BSHD runs of key/value heads of one entry (strided on the host, packed on the
#   device), with grouped heads and causal;
# - BSHD row chunks of one entry (a single key/value head), also causal with
#   Sq > Sk, where the first chunk must take every row that sees no key;
# - BSHD batch runs;
# - BHSD head runs with grouped heads.
# The 3- and 7-entry shapes ask for 8 chunks with fewer entries: the planner
# must stay within its 8 chunks.
@pytest.mark.parametrize("layout,B,Hq,Hkv,Sq,Sk,causal", [
    ("bshd", 1, 16, 16, 8192, 3000, False),
    ("bshd", 1, 16, 4, 8192, 5000, True),
    ("bshd", 1, 16, 16, 8200, 700, True),      # Sq > Sk: the first 7500 rows see no key
    ("bshd", 1, 16, 1, 8200, 700, True),       # one key/value head: row chunks
    ("bshd", 3, 32, 32, 5632, 512, False),     # 2 head runs per entry, 6 chunks
    ("bshd", 3, 32, 1, 5632, 512, True),       # 2 row chunks per entry
    ("bshd", 7, 16, 16, 4864, 300, False),     # one chunk per entry
    ("bshd", 4, 8, 8, 2304, 2304, True),
    ("bhsd", 2, 16, 8, 4096, 1000, False),
    ("bhsd", 3, 12, 3, 2500, 2600, True),
])
def test_host_equals_device_call_bitwise(layout, B, Hq, Hkv, Sq, Sk, causal):
    q, k, v = _qkv(layout, B, Hq, Hkv, Sq, Sk, seed=1200 + Sq + Hq)
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    got = attn.attn_fwd_host(qp, kp, vp, causal=causal, layout=layout)
    want = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, layout=layout)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    assert torch.equal(got.view(torch.int16), want.cpu().view(torch.int16))


def test_host_small_problem_against_oracle_pageable_memory():
    # Pageable (not pinned) host memory: the copies serialise but the result holds.
    q, k, v = _qkv("bhsd", 1, 4, 2, 300, 500, seed=1300)
    out = torch.zeros(q.shape, dtype=torch.bfloat16)
    attn.attn_fwd_host(q, k, v, causal=True, layout="bhsd", rounding="rtz", out=out)
    torch.cuda.synchronize()
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), "bhsd",
                           causal=True)
    assert_parity(compare(bits_of(out), exact, "rtz"), excess=True)


def test_host_calls_on_two_streams_with_two_workspaces():
    q, k, v = (t.pin_memory() for t in _qkv("bshd", 2, 16, 16, 4096, 4096, seed=1301))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        a = attn.attn_fwd_host(q, k, v, layout="bshd", rounding="rtne")
    with torch.cuda.stream(s2):
        b = attn.attn_fwd_host(q, k, v, layout="bshd", rounding="rtz")
    torch.cuda.synchronize()
    want_a = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), layout="bshd", rounding="rtne").cpu()
    want_b = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), layout="bshd", rounding="rtz").cpu()
    assert torch.equal(a.view(torch.int16), want_a.view(torch.int16))
    assert torch.equal(b.view(torch.int16), want_b.view(torch.int16))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_host_equals_device_call_bitwise(causal):
    # Enough sequences and rows for several chunks of whole sequences, with a
    # sequence without queries and one without keys among them.
    lens = ((700, 900), (0, 5), (2048, 2048), (300, 0), (4096, 3000), (129, 129), (1500, 1600),
            (4000, 4100))
    w = inputs.Workload("vh", "thd", len(lens), 16, 4096, 4100, seed=1310, hkv=4, seqlens=lens)
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    got = attn.attn_fwd_varlen_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                    torch.from_numpy(cq), torch.from_numpy(ck), causal=causal)
    want = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cq).cuda(),
                                torch.from_numpy(ck).cuda(), 4096, causal=causal)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    assert torch.equal(got.view(torch.int16), want.cpu().view(torch.int16))


def test_varlen_host_trailing_sequences_without_queries():
    # 2048 CTAs ask for 8 chunks, reached at the last sequence with queries; the
    # sequences after it (no queries) join the last chunk.
    lens = ((4096, 4096),) * 8 + ((0, 300), (0, 10))
    w = inputs.Workload("vh", "thd", len(lens), 16, 4096, 4096, seed=1312, hkv=16, seqlens=lens)
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    got = attn.attn_fwd_varlen_host(q.pin_memory(), k.pin_memory(), v.pin_memory(),
                                    torch.from_numpy(cq), torch.from_numpy(ck))
    want = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cq).cuda(),
                                torch.from_numpy(ck).cuda(), 4096)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    assert torch.equal(got.view(torch.int16), want.cpu().view(torch.int16))


def test_varlen_host_rejects_bad_offsets_before_running():
    w = inputs.Workload("vh", "thd", 2, 2, 100, 100, seed=1311, seqlens=((100, 100), (100, 100)))
    q, k, v = inputs.make_qkv(w)
    for cq in ([0, 210, 200], [0, 100, 150], [1, 100, 200]):  # decreasing, short, not from 0
        with pytest.raises(attn.AttnError) as e:
            attn.attn_fwd_varlen_host(q, k, v, torch.tensor(cq, dtype=torch.int32),
                                      torch.tensor([0, 100, 200], dtype=torch.int32))
        assert e.value.status in (attn.ATTN_ERR_SEQLENS, attn.ATTN_ERR_INVALID_ARG)
