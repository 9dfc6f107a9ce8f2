"""The follow-on workloads at their full sizes, called exactly as the benchmark
calls them, compared with the fp64 oracle on sampled rows: causal8k (causal
mask), gqa8k (grouped-query heads), varlen16 (packed variable-length batch) and
decode32k (split-KV)."""
import json

import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_rows_fp64, bf16_bits_to_f64, to_bhsd

from _parity import assert_parity, bits_of, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _rows(S, rng, n, extra=()):
    fixed = {0, 1, 2, 127, 128, 129, 255, 256, S // 2, S - 129, S - 2, S - 1, *extra}
    return np.array(sorted({r for r in fixed if 0 <= r < S} | set(rng.integers(0, S, n).tolist())))


@pytest.mark.parametrize("name", ["causal8k", "gqa8k", "decode32k"])
def test_fixed_shape_followon_sampled(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    if w.splitkv:
        s = attn.splitkv_num_splits(w.B, w.H, w.Sq, w.Sk)
        assert s > 1
        out = attn.attn_fwd_splitkv(qd, kd, vd, num_splits=s, layout=w.layout)
    else:
        out = attn.attn_fwd_ex(qd, kd, vd, causal=w.causal, layout=w.layout)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    rng = np.random.default_rng(w.seed)
    qb, kb, vb = (to_bhsd(t.view(torch.int16).numpy(), w.layout) for t in (q, k, v))
    ob = to_bhsd(bits_of(out), w.layout)
    group = w.H // w.kv_heads
    got, exact = [], []
    for b in range(w.B):
        for h in range(w.H):
            rows = _rows(w.Sq, rng, max(4, 256 // (w.B * w.H)))
            exact.append(attention_rows_fp64(bf16_bits_to_f64(qb[b, h]),
                                             bf16_bits_to_f64(kb[b, h // group]),
                                             bf16_bits_to_f64(vb[b, h // group]),
                                             inputs.default_scale(), rows, causal=w.causal))
            got.append(ob[b, h, rows])
    stats = compare(np.concatenate(got), np.concatenate(exact), w.roundings[0])
    print(f"\nPARITY {name}: " + json.dumps(stats))
    assert_parity(stats, excess=w.causal)


def test_varlen16_sampled():
    w = inputs.WORKLOADS["varlen16"]
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    out = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cq).cuda(),
                               torch.from_numpy(ck).cuda(), max(a for a, _ in w.seqlens),
                               causal=w.causal)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    rng = np.random.default_rng(w.seed)
    qn, kn, vn = (t.view(torch.int16).numpy() for t in (q, k, v))
    on = bits_of(out)
    got, exact = [], []
    for b in range(w.B):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        for h in range(0, w.H, 5):
            rows = _rows(q1 - q0, rng, 8)
            exact.append(attention_rows_fp64(bf16_bits_to_f64(qn[q0:q1, h]),
                                             bf16_bits_to_f64(kn[k0:k1, h]),
                                             bf16_bits_to_f64(vn[k0:k1, h]),
                                             inputs.default_scale(), rows, causal=w.causal))
            got.append(on[q0 + rows, h])
    stats = compare(np.concatenate(got), np.concatenate(exact), w.roundings[0])
    print("\nPARITY varlen16: " + json.dumps(stats))
    assert_parity(stats)
