"""The index arithmetic at the far ends of the sizes, on a GB300, against the fp64
oracle on sampled rows:
- one item of a million keys (7813 key tiles, the last holding 64 keys): one CTA,
  the pair variant (ATTN_FLAG_SPLIT_TAIL) and a 64-way key split;
- 40,000 (batch, head) items of one ragged key tile each (the short persistent
  variant), the last query tile of each holding 2 rows;
- 3050 items of 18 key tiles (one CTA per item: 20 full waves and a tail of 10),
  with and without the tail split.
Inputs are unit normals from a seeded torch generator, rounded to bf16."""
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


def _normal(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _f64(t):
    return bf16_bits_to_f64(t.view(torch.int16).numpy())


def _check_heads(out, q, k, v, layout, heads, rows, group=1):
    """Oracle rows of the given (b, h) heads against `out` (same layout as q)."""
    qb, kb, vb = (to_bhsd(t.view(torch.int16).numpy(), layout) for t in (q, k, v))
    ob = to_bhsd(bits_of(out), layout)
    got, exact = [], []
    for b, h in heads:
        exact.append(attention_rows_fp64(bf16_bits_to_f64(qb[b, h]),
                                         bf16_bits_to_f64(kb[b, h // group]),
                                         bf16_bits_to_f64(vb[b, h // group]),
                                         inputs.default_scale(), rows))
        got.append(ob[b, h, rows])
    return compare(np.concatenate(got), np.concatenate(exact), "rtne")


def test_a_million_keys():
    Sq, Sk = 300, 1_000_000
    q = _normal((1, 1, Sq, 128), 3001)
    k = _normal((1, 1, Sk, 128), 3002)
    v = _normal((1, 1, Sk, 128), 3003)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    one = attn.attn_fwd(qd, kd, vd)
    assert attn.split_tail_items(1, 1, Sq, Sk) == 2
    pair = attn.attn_fwd_ex(qd, kd, vd, split_tail=True)
    split = attn.attn_fwd_splitkv(qd, kd, vd, num_splits=64)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    # Every other row (both query tiles, their edges included): 19,200 outputs, so
    # that the 99.9%-within-1-ULP rule is a real statistic at this length.
    rows = np.unique(np.concatenate([np.arange(0, Sq, 2), [127, 129, 255, 299]]))
    qf, kf, vf = _f64(q[0, 0]), _f64(k[0, 0]), _f64(v[0, 0])
    scale = inputs.default_scale()
    exact = np.concatenate([attention_rows_fp64(qf, kf, vf, scale, rows[i:i + 50])
                            for i in range(0, len(rows), 50)])
    for out in (one, pair, split):
        # Averages over a million keys are small (|O| ~ 1e-3): tight absolute error.
        assert_parity(compare(bits_of(out)[0, 0, rows], exact, "rtne"), max_abs_err=1e-4)


def test_forty_thousand_short_items():
    # BSHD, 2 x 20000 heads, 130 queries (one query-tile pair, the second tile
    # holding 2 rows), 100 keys: the short persistent variant over 40,000 items.
    B, H, Sq, Sk = 2, 20000, 130, 100
    q = _normal((B, Sq, H, 128), 3011)
    k = _normal((B, Sk, H, 128), 3012)
    v = _normal((B, Sk, H, 128), 3013)
    out = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), layout="bshd")
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    rng = np.random.default_rng(3014)
    heads = [(0, 0), (1, H - 1), (0, H - 1), (1, 0)] + [
        (int(b), int(h)) for b, h in zip(rng.integers(0, B, 24), rng.integers(0, H, 24))]
    # Few keys per row: outputs reach magnitude ~2, where 1 ULP exceeds 8e-3.
    assert_parity(_check_heads(out.cpu(), q, k, v, "bshd", heads, np.arange(Sq)), excess=True)


@pytest.mark.parametrize("split_tail", [False, True])
def test_three_thousand_items_with_a_tail(split_tail):
    # BHSD, 3050 heads of one query-tile pair and 18 key tiles: 20 full waves of
    # one CTA per item and a tail of 10 items (on pairs with the flag).
    B, H, Sq, Sk = 1, 3050, 256, 2200
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    q = _normal((B, H, Sq, 128), 3021)
    k = _normal((B, H, Sk, 128), 3022)
    v = _normal((B, H, Sk, 128), 3023)
    if split_tail:
        assert attn.split_tail_items(B, H, Sq, Sk) == H % sms
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), split_tail=split_tail)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    rng = np.random.default_rng(3024)
    heads = [(0, 0), (0, H - 1), (0, H - 2), (0, H - H % sms)] + [
        (0, int(h)) for h in rng.integers(0, H, 12)]
    rows = np.array([0, 1, 127, 128, 129, 200, 254, 255])
    assert_parity(_check_heads(out.cpu(), q, k, v, "bhsd", heads, rows))
