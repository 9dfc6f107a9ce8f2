"""The pair variant against the fp64 oracle and against the split-key path, on a GB300.

With ATTN_FLAG_SPLIT_TAIL (``split_tail=True``), a whole-range call (no mask)
whose last wave is partial runs the items of that
wave as 2-CTA clusters when they fit on the GPU at once and the key range has at
least 8 tiles (more than 16 when there are more items than SMs: up to 16, such
calls take the persistent variant). Each CTA of a cluster takes one half of the
item's key tiles; the second sends its unnormalised rows, running max and row sum
to the first through distributed shared memory, and the first merges and stores. The halves and the
merge are those of ``attn_fwd_splitkv`` with two splits (same tile ranges, same
operations in the same order), so the outputs of the tail items must equal that
path bit for bit; the items of the full waves must equal a call that has no tail.
Without the flag, a slice of the heads gives the same bits as the whole call.
"""
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


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _qkv(layout, B, Hq, Hkv, Sq, Sk, seed, std=1.0):
    w = inputs.Workload("pair", layout, B, Hq, Sq, Sk, seed=seed, qk_std=std)
    q, _, _ = inputs.make_qkv(w)
    wk = inputs.Workload("pair", layout, B, Hkv, Sq, Sk, seed=seed + 1, qk_std=std)
    _, k, v = inputs.make_qkv(wk)
    return q, k, v


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


# Fewer items (batch x head x pair of 128-row query tiles) than fit as clusters at
# once, at least 8 key tiles: the whole call is one partial wave of pairs.
# split_tail_items() says which path the call takes on this device.
SHAPES = [
    ("bhsd", 1, 4, 500, 3000),   # 24 key tiles, the last holds 56 keys; query tail
    ("bshd", 2, 3, 256, 1024),   # 8 full key tiles: 4 per half
    ("bhsd", 1, 2, 100, 1025),   # 9 key tiles: 5 and 4, the second half ends in 1 key
    ("bshd", 1, 8, 1000, 4097),  # 33 key tiles, 32 items
    ("bhsd", 1, 1, 1, 1100),     # one query row
]


@pytest.mark.parametrize("layout,B,H,Sq,Sk", SHAPES)
def test_pair_equals_two_way_split_bitwise(layout, B, H, Sq, Sk):
    n_items = B * H * ((Sq + 255) // 256)
    assert attn.split_tail_items(B, H, Sq, Sk) == n_items  # every item runs on a pair
    q, k, v = (t.cuda() for t in _qkv(layout, B, H, H, Sq, Sk, seed=1500 + Sq + Sk))
    exact = attention_fp64(f64_of(q.cpu()), f64_of(k.cpu()), f64_of(v.cpu()),
                           inputs.default_scale(), layout)
    for mode in inputs.ROUNDINGS:
        out = attn.attn_fwd_ex(q, k, v, layout=layout, rounding=mode, split_tail=True)
        split = attn.attn_fwd_splitkv(q, k, v, num_splits=2, layout=layout, rounding=mode)
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        assert _same_bits(out, split)
        assert_parity(compare(bits_of(out), exact, mode))


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_pair_tail_after_full_waves(layout):
    # One item per head (256 queries): the first `sms` heads form one full wave
    # of single CTAs, the remaining 5 run as pairs (17 key tiles, the last holding
    # 52 keys).
    sms = _sms()
    H, Sq, Sk = sms + 5, 256, 2100
    assert attn.split_tail_items(1, H, Sq, Sk) == 5
    q, k, v = _qkv(layout, 1, H, H, Sq, Sk, seed=1600)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    head = (lambda t, a, b: t[:, a:b]) if layout == "bhsd" else (lambda t, a, b: t[:, :, a:b])
    whole = attn.attn_fwd_ex(qd, kd, vd, layout=layout, split_tail=True)
    full = attn.attn_fwd(*(head(t, 0, sms).contiguous() for t in (qd, kd, vd)), layout=layout)
    tail = attn.attn_fwd_splitkv(*(head(t, sms, H).contiguous() for t in (qd, kd, vd)),
                                 num_splits=2, layout=layout)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    assert _same_bits(head(whole, 0, sms).contiguous(), full)
    assert _same_bits(head(whole, sms, H).contiguous(), tail)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout)
    assert_parity(compare(bits_of(whole), exact, "rtne"))


def test_pair_grouped_heads():
    # Grouped-query heads (8 key/value heads) through attn_fwd_ex: a tail of at
    # most 8 items after the full wave.
    sms = _sms()
    Hkv = 8
    H = Hkv * ((sms + Hkv) // Hkv)
    assert 0 < H - sms <= 8
    assert attn.split_tail_items(1, H, 200, 2200) == H - sms
    layout, Sq, Sk = "bshd", 200, 2200
    q, k, v = _qkv(layout, 1, H, Hkv, Sq, Sk, seed=1700)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout)
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), layout=layout, rounding="rtz",
                           split_tail=True)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    assert_parity(compare(bits_of(out), exact, "rtz"))


def test_pair_specials_and_negative_scale():
    # NaN in a query row; +Inf and -Inf key elements, one in each half of the key
    # range; wide logits; a negative scale.
    layout, B, H, Sq, Sk = "bhsd", 1, 6, 300, 2100
    assert attn.split_tail_items(B, H, Sq, Sk) == 12
    q, k, v = _qkv(layout, B, H, H, Sq, Sk, seed=1800, std=8.0)
    qb, kb = q.view(torch.int16), k.view(torch.int16)
    qb[0, 1, 200, 3] = 0x7FC0    # row 200 of head 1 is NaN
    kb[0, 2, 100, 9] = 0x7F80    # +Inf key element in the first half of head 2
    kb[0, 4, 2050, 0] = -0x80    # -Inf (0xFF80) in the second half of head 4
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for scale in (inputs.default_scale(), -0.04):
        exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), scale, layout)
        for mode in inputs.ROUNDINGS:
            out = attn.attn_fwd_ex(qd, kd, vd, layout=layout, rounding=mode, scale=scale,
                                   split_tail=True)
            split = attn.attn_fwd_splitkv(qd, kd, vd, num_splits=2, layout=layout,
                                          rounding=mode, scale=scale)
            torch.cuda.synchronize()
            assert attn.attn_fwd_last_error() == attn.ATTN_OK
            assert _same_bits(out, split)
            assert_parity(compare(bits_of(out), exact, mode), max_abs_err=None)


def test_pair_reruns_are_bit_identical():
    assert attn.split_tail_items(1, 16, 512, 5000) == 32
    q, k, v = (t.cuda() for t in _qkv("bshd", 1, 16, 16, 512, 5000, seed=1900))
    a = attn.attn_fwd_ex(q, k, v, layout="bshd", split_tail=True)
    b = attn.attn_fwd_ex(q, k, v, layout="bshd", split_tail=True)
    torch.cuda.synchronize()
    assert _same_bits(a, b)


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_without_the_flag_a_slice_gives_the_same_bits(layout):
    # The shape of the tail test, without the flag: every head's output is the
    # same whether it is computed in the whole call or in a call of its own slice.
    sms = _sms()
    H, Sq, Sk = sms + 5, 256, 2100
    q, k, v = (t.cuda() for t in _qkv(layout, 1, H, H, Sq, Sk, seed=2000))
    head = (lambda t, a, b: t[:, a:b]) if layout == "bhsd" else (lambda t, a, b: t[:, :, a:b])
    whole = attn.attn_fwd(q, k, v, layout=layout)
    ex = attn.attn_fwd_ex(q, k, v, layout=layout)
    parts = [attn.attn_fwd(*(head(t, a, b).contiguous() for t in (q, k, v)), layout=layout)
             for a, b in ((0, 3), (3, sms), (sms, H))]
    torch.cuda.synchronize()
    assert _same_bits(whole, ex)
    for (a, b), part in zip(((0, 3), (3, sms), (sms, H)), parts):
        assert _same_bits(head(whole, a, b).contiguous(), part)


def test_split_tail_items_where_the_flag_changes_nothing():
    sms = _sms()
    assert attn.split_tail_items(1, sms + 5, 256, 2000) == 0  # 16 key tiles, more items than SMs
    assert attn.split_tail_items(1, 4, 256, 896) == 0         # 7 key tiles
    assert attn.split_tail_items(1, 2 * sms, 256, 4000) == 0  # no partial wave
    assert attn.split_tail_items(1, sms - 1, 256, 4000) == 0  # a wave too large for pairs
    assert attn.split_tail_items(1, 4, 256, 1024) == 4        # 8 key tiles: one wave of pairs


def test_split_tail_full_size_cross4k32k():
    # The workload whose last wave the flag halves: 512 items, the last 56 of them
    # (from head 28, query pair 8 on) on pairs. Those items must equal the
    # full-size 2-way split and every other item the default call, bit for bit;
    # sampled rows (most of them from the tail heads) go against the oracle.
    import numpy as np
    from oracle import attention_rows_fp64, bf16_bits_to_f64, to_bhsd

    w = inputs.WORKLOADS["cross4k32k"]
    n_qp = (w.Sq + 255) // 256
    n_items = w.B * w.H * n_qp
    n_tail = attn.split_tail_items(w.B, w.H, w.Sq, w.Sk)
    assert 0 < n_tail < n_items
    q, k, v = inputs.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    tail = attn.attn_fwd_ex(qd, kd, vd, layout=w.layout, split_tail=True)
    plain = attn.attn_fwd(qd, kd, vd, layout=w.layout)
    split = attn.attn_fwd_splitkv(qd, kd, vd, num_splits=2, layout=w.layout)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    tb, pb, sb = (to_bhsd(bits_of(t), w.layout) for t in (tail, plain, split))
    # Item of (b, h, row): pair + (b * H + h) * n_qp, rows of a pair 256 apart.
    item = ((np.arange(w.B)[:, None, None] * w.H + np.arange(w.H)[None, :, None]) * n_qp
            + (np.arange(w.Sq)[None, None, :] // 256))
    in_tail = item >= n_items - n_tail
    assert (tb[in_tail] == sb[in_tail]).all()
    assert (tb[~in_tail] == pb[~in_tail]).all()
    rng = np.random.default_rng(w.seed)
    qb, kb, vb = (to_bhsd(t.view(torch.int16).numpy(), w.layout) for t in (q, k, v))
    got, exact = [], []
    for h in list(range(w.H - 5, w.H)) + [0, w.H // 2]:
        rows = np.unique(np.concatenate([[0, 255, 256, 2047, 2048, w.Sq - 1],
                                         rng.integers(0, w.Sq, 24)]))
        exact.append(attention_rows_fp64(bf16_bits_to_f64(qb[0, h]), bf16_bits_to_f64(kb[0, h]),
                                         bf16_bits_to_f64(vb[0, h]), inputs.default_scale(), rows))
        got.append(tb[0, h, rows])
    assert_parity(compare(np.concatenate(got), np.concatenate(exact), w.roundings[0]))
