"""Parity of the persistent short-key-range path against the fp64 oracle, on a GB300.

Whole-range problems with at most 16 key tiles and more work items (batch x
head x pair of 128-row query tiles) than the GPU has SMs run one CTA per SM, each
looping over its items with the barrier phases carried from one item to the next
and the output stored through its own staging buffer. Every shape below takes
that path; those whose items have at most 4 key tiles ending in a ragged one
take one of its short forms (one tile, or 2 to 4), which keep the partial in
TMEM until the epilogue and S in registers between the two softmax passes, and
stop the P V MMAs and the exp pass at the last 16-key chunk holding a key.
Whole tensors are compared, in both layouts and all rounding modes,
with ragged query and key lengths, grouped-query heads, a NaN query, an infinite
key and a negative scale. Reruns must be bit-identical.
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


def _items(B, H, Sq):
    return B * H * ((Sq + 255) // 256)


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _qkv(layout, B, Hq, Hkv, Sq, Sk, seed, std=1.0):
    w = inputs.Workload("p", layout, B, Hq, Sq, Sk, seed=seed, qk_std=std)
    q, _, _ = inputs.make_qkv(w)
    wk = inputs.Workload("p", layout, B, Hkv, Sq, Sk, seed=seed + 1, qk_std=std)
    _, k, v = inputs.make_qkv(wk)
    return q, k, v


SHAPES = [
    ("bshd", 2, 40, 40, 700, 77),     # one masked key tile, query tail of 188 rows
    ("bhsd", 1, 160, 160, 300, 512),  # four full key tiles
    ("bshd", 1, 200, 200, 129, 130),  # two key tiles, the second holds 2 keys
    ("bhsd", 3, 64, 64, 1000, 1),     # a single key
    ("bshd", 1, 96, 8, 520, 200),     # grouped-query heads, 12 per key/value head
    ("bhsd", 1, 170, 170, 256, 2000), # 16 key tiles (the last holds 80 keys): 4 fold intervals
]


@pytest.mark.parametrize("layout,B,Hq,Hkv,Sq,Sk", SHAPES)
def test_persistent_parity(layout, B, Hq, Hkv, Sq, Sk):
    assert _items(B, Hq, Sq) > _sms() and (Sk + 127) // 128 <= 16  # takes the persistent path
    q, k, v = _qkv(layout, B, Hq, Hkv, Sq, Sk, seed=1200 + Sq + Sk + Hq)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for mode in inputs.ROUNDINGS:
        out = attn.attn_fwd_ex(qd, kd, vd, layout=layout, rounding=mode)
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        # Few keys per row: outputs reach magnitude ~2, where 1 ULP exceeds 8e-3.
        assert_parity(compare(bits_of(out), exact, mode), excess=True)
    again = attn.attn_fwd_ex(qd, kd, vd, layout=layout, rounding=inputs.ROUNDINGS[-1])
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), out.view(torch.int16))


def test_persistent_specials_and_negative_scale():
    layout, B, H, Sq, Sk = "bhsd", 1, 180, 260, 140
    q, k, v = _qkv(layout, B, H, H, Sq, Sk, seed=1300, std=8.0)
    qb, kb = q.view(torch.int16), k.view(torch.int16)
    qb[0, 7, 100, 5] = 0x7FC0  # NaN query element: row 100 of head 7 is NaN
    kb[0, 11, 3, 9] = 0x7F80  # +Inf key element in head 11
    for scale in (inputs.default_scale(), -0.04):
        exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), scale, layout)
        for mode in inputs.ROUNDINGS:  # every mode writes NaN as the one pattern 0x7FC0
            out = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), layout=layout, rounding=mode,
                                scale=scale)
            torch.cuda.synchronize()
            assert attn.attn_fwd_last_error() == attn.ATTN_OK
            assert_parity(compare(bits_of(out), exact, mode), max_abs_err=None)


@pytest.mark.parametrize("Sk", [300, 77, 17])
def test_persistent_equals_one_cta_per_item_bitwise(Sk):
    # Splitting the heads into calls of at most as many items as SMs keeps each
    # call on one CTA per item; results must match the persistent call bit for bit.
    # 77 and 17 keys (one ragged key tile) take the one-tile short form, 300 keys
    # (3 tiles, the last of 44 keys) the 2-to-4-tile short form.
    layout, B, H, Sq = "bhsd", 1, 240, 256
    q, k, v = (t.cuda() for t in _qkv(layout, B, H, H, Sq, Sk, seed=1400 + Sk))
    whole = attn.attn_fwd(q, k, v, layout=layout)
    step = min(H, _sms())
    parts = [attn.attn_fwd(q[:, h:h + step].contiguous(), k[:, h:h + step].contiguous(),
                           v[:, h:h + step].contiguous(), layout=layout)
             for h in range(0, H, step)]
    torch.cuda.synchronize()
    assert _items(B, H, Sq) > _sms() >= _items(B, step, Sq)
    assert torch.equal(whole.view(torch.int16), torch.cat(parts, dim=1).view(torch.int16))


def test_persistent_sign_bit_nans_come_out_canonical():
    # NaNs with the sign bit set, in V (0xFFC1) and in Q (0xFFFF), on the persistent
    # path: every NaN output must be the one pattern 0x7FC0 in every mode.
    layout, B, H, Sq, Sk = "bhsd", 1, 180, 260, 140
    assert _items(B, H, Sq) > _sms()
    q, k, v = _qkv(layout, B, H, H, Sq, Sk, seed=1310)
    q.view(torch.int16)[0, 9, 100, 17] = -1          # 0xFFFF: row 100 of head 9 is NaN
    v.view(torch.int16)[0, 5, 17, 33] = -63          # 0xFFC1: column 33 of head 5 is NaN
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout)
    for mode in inputs.ROUNDINGS:
        out = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), layout=layout, rounding=mode)
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        got = bits_of(out)
        assert (got[0, 9, 100] == 0x7FC0).all() and (got[0, 5, :, 33] == 0x7FC0).all()
        stats = compare(got, exact, mode)
        assert stats["n_nonfinite"] == 128 + Sq  # different heads: no overlap
        assert_parity(stats, excess=True)
