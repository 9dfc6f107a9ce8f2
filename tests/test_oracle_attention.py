"""Pins for the oracle's attention core (CPU only).

The oracle is checked against things other than itself:
  * a library routine: torch's scaled_dot_product_attention in float64 on CPU;
  * closed forms: constant V, Q = 0, scale = 0, one key, two keys (a logistic
    weight), -Inf logits, NaN and +Inf propagation;
  * invariants: joint permutation of K/V rows, BSHD vs BHSD, weights summing to 1;
  * planted mistakes: a few plausible bugs, planted in a copy of the oracle here
    on the CPU, must each fail one of the pins above.
Sources: snilld.dk article "Open source attention-kernel i HIP slaar AITER v3 paa
MI300X", sections "Hvordan kernen arbejder" (softmax(QK^T/sqrt(d))V) and
"Hvad er udgivet" (layouts, lengths, cross-attention).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import attention_fp64, attention_rows_fp64, round_bf16

from bf16_forward_attention_gb300 import inputs


def _rand(shape, seed, std=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape) * std
    # bf16-exact values, like the real inputs
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def _sdpa(q, k, v, scale):
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale).numpy()


@pytest.mark.parametrize("B,H,Sq,Sk,d", [(1, 1, 1, 1, 128), (2, 3, 17, 29, 128),
                                         (1, 2, 130, 7, 128), (1, 1, 5, 300, 64)])
def test_matches_torch_sdpa(B, H, Sq, Sk, d):
    q, k, v = _rand((B, H, Sq, d), 1), _rand((B, H, Sk, d), 2), _rand((B, H, Sk, d), 3)
    scale = inputs.default_scale(d)
    got = attention_fp64(q, k, v, scale)
    want = _sdpa(q, k, v, float(np.float32(scale)))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_wide_logits_match_sdpa():
    q, k = _rand((1, 2, 9, 128), 4, 8.0), _rand((1, 2, 33, 128), 5, 8.0)
    v = _rand((1, 2, 33, 128), 6)
    scale = inputs.default_scale()
    np.testing.assert_allclose(attention_fp64(q, k, v, scale),
                               _sdpa(q, k, v, float(np.float32(scale))), rtol=1e-11, atol=1e-12)


def test_constant_v_gives_v():
    q, k = _rand((1, 2, 11, 128), 7), _rand((1, 2, 13, 128), 8)
    c = _rand((128,), 9)
    v = np.broadcast_to(c, (1, 2, 13, 128)).copy()
    o = attention_fp64(q, k, v, 0.088)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=1e-14, atol=0)
    for mode in ("rtne", "rtna"):  # the fp64 result is within 1e-14 of a bf16 value
        assert (round_bf16(o, mode) == round_bf16(np.broadcast_to(c, o.shape), mode)).all()


def test_zero_q_and_zero_scale_give_mean():
    k, v = _rand((1, 1, 19, 128), 10), _rand((1, 1, 19, 128), 11)
    mean = v.mean(axis=2, keepdims=True)
    o = attention_fp64(np.zeros((1, 1, 4, 128)), k, v, 0.5)
    np.testing.assert_allclose(o, np.broadcast_to(mean, o.shape), rtol=1e-13, atol=1e-15)
    o = attention_fp64(_rand((1, 1, 4, 128), 12), k, v, 0.0)
    np.testing.assert_allclose(o, np.broadcast_to(mean, o.shape), rtol=1e-13, atol=1e-15)


def test_single_key_gives_v0():
    q, k, v = _rand((1, 1, 6, 128), 13), _rand((1, 1, 1, 128), 14), _rand((1, 1, 1, 128), 15)
    o = attention_fp64(q, k, v, 0.3)
    assert (o == np.broadcast_to(v, o.shape)).all()


def test_two_keys_logistic_closed_form():
    # s0 - s1 = scale * q.(k0 - k1); the weight of key 0 is 1 / (1 + exp(-(s0 - s1))).
    rng = np.random.default_rng(16)
    for _ in range(20):
        q, k, v = _rand((1, 1, 1, 128), rng.integers(1e9)), _rand((1, 1, 2, 128), rng.integers(1e9)), \
            _rand((1, 1, 2, 128), rng.integers(1e9))
        scale = float(np.float32(rng.uniform(-0.3, 0.3)))
        ds = scale * math.fsum(q[0, 0, 0] * (k[0, 0, 0] - k[0, 0, 1]))
        w0 = 1.0 / (1.0 + math.exp(-ds))
        want = w0 * v[0, 0, 0] + (1.0 - w0) * v[0, 0, 1]
        np.testing.assert_allclose(attention_fp64(q, k, v, scale)[0, 0, 0], want,
                                   rtol=1e-12, atol=1e-14)


def test_weights_sum_to_one():
    # With V = identity rows, O_i is the softmax row itself.
    Sk = 40
    q, k = _rand((1, 1, 8, 128), 17), _rand((1, 1, Sk, 128), 18)
    v = np.zeros((1, 1, Sk, 128))
    v[0, 0, np.arange(Sk), np.arange(Sk)] = 1.0
    o = attention_fp64(q, k, v, inputs.default_scale())
    np.testing.assert_allclose(o.sum(axis=-1), 1.0, rtol=0, atol=1e-15)
    assert (o[..., Sk:] == 0).all() and (o[..., :Sk] > 0).all()


def test_joint_kv_permutation_invariance():
    q, k, v = _rand((1, 2, 10, 128), 19), _rand((1, 2, 50, 128), 20), _rand((1, 2, 50, 128), 21)
    perm = np.random.default_rng(22).permutation(50)
    a = attention_fp64(q, k, v, 0.09)
    b = attention_fp64(q, k[:, :, perm], v[:, :, perm], 0.09)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-15)


def test_layouts_agree():
    q, k, v = _rand((2, 3, 9, 128), 23), _rand((2, 3, 14, 128), 24), _rand((2, 3, 14, 128), 25)
    a = attention_fp64(q, k, v, 0.1, "bhsd")
    t = lambda x: np.ascontiguousarray(np.swapaxes(x, 1, 2))
    b = attention_fp64(t(q), t(k), t(v), 0.1, "bshd")
    assert (t(a) == b).all()


def test_rows_subset_matches_full():
    q, k, v = _rand((1, 1, 37, 128), 26), _rand((1, 1, 41, 128), 27), _rand((1, 1, 41, 128), 28)
    full = attention_fp64(q, k, v, 0.1)[0, 0]
    rows = [0, 5, 36]
    sub = attention_rows_fp64(q[0, 0], k[0, 0], v[0, 0], 0.1, rows)
    assert (sub == full[rows]).all()


def test_nan_in_q_row_gives_nan_row_only():
    q, k, v = _rand((1, 1, 6, 128), 29), _rand((1, 1, 9, 128), 30), _rand((1, 1, 9, 128), 31)
    q[0, 0, 2, 77] = np.nan
    o = attention_fp64(q, k, v, 0.1)
    assert np.isnan(o[0, 0, 2]).all()
    assert np.isfinite(np.delete(o[0, 0], 2, axis=0)).all()


def test_inf_in_k_closed_form():
    # One +Inf at K[j, c]: s_ij = +Inf if q_ic > 0 (row NaN: Inf - Inf), NaN if q_ic = 0
    # (0 * Inf), -Inf if q_ic < 0 (key j gets weight exp(-Inf) = 0).
    q, k, v = _rand((1, 1, 64, 128), 32), _rand((1, 1, 9, 128), 33), _rand((1, 1, 9, 128), 34)
    j, c = 4, 50
    q[0, 0, :3, c] = [0.0, -0.0, 1.0]
    q[0, 0, 3, c] = -2.0
    k[0, 0, j, c] = np.inf
    o = attention_fp64(q, k, v, 0.1)[0, 0]
    nan_rows = q[0, 0, :, c] >= 0
    assert np.isnan(o[nan_rows]).all()
    assert np.isfinite(o[~nan_rows]).all()
    keep = [i for i in range(9) if i != j]
    ref = attention_fp64(q[:, :, ~nan_rows], k[:, :, keep], v[:, :, keep], 0.1)[0, 0]
    np.testing.assert_allclose(o[~nan_rows], ref, rtol=1e-13, atol=1e-15)


def test_all_minus_inf_row_is_nan():
    q = np.ones((1, 1, 1, 128))
    k = np.full((1, 1, 3, 128), -np.inf)
    v = _rand((1, 1, 3, 128), 35)
    assert np.isnan(attention_fp64(q, k, v, 0.1)).all()


def test_generator_is_deterministic_and_shaped():
    w = inputs.WORKLOADS["tiny"].scaled(Sq=5, Sk=7, H=1)
    a = inputs.make_qkv(w)
    b = inputs.make_qkv(w)
    assert all(torch.equal(x.view(torch.int16), y.view(torch.int16)) for x, y in zip(a, b))
    assert a[0].shape == (1, 1, 5, 128) and a[1].shape == (1, 1, 7, 128)
    s = inputs.normal_f32(1, 0, 200000)
    assert abs(s.mean()) < 0.01 and abs(s.std() - 1) < 0.01
    u = inputs.uniform_f32(1, 1, 200000, -1, 1)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.01


# --- planted mistakes: each must be caught by a pin above -----------------------

def _mutant(kind):
    def rows(q, k, v, scale, rows=None, causal=False):
        scale_d = float(np.float32(scale))
        if rows is not None:
            q = q[np.asarray(rows)]
        if kind == "no_scale":
            s = q @ k.T
        elif kind == "transposed_v":
            s = (q @ k.T) * scale_d
        else:
            s = (q @ k.T) * scale_d
        m = np.max(s, axis=1, keepdims=True)
        p = np.exp(s - m)
        l = np.sum(p, axis=1, keepdims=True)
        if kind == "no_normalise":
            return p @ v
        if kind == "wrong_axis":
            return (p / p.sum(axis=0, keepdims=True)) @ v
        if kind == "transposed_v":
            vv = v.T if v.shape[0] == v.shape[1] else v[::-1]
            return p @ vv / l
        return p @ v / l
    return rows


@pytest.mark.parametrize("kind", ["no_scale", "no_normalise", "wrong_axis", "transposed_v"])
def test_planted_mistakes_are_caught(kind, monkeypatch):
    import oracle.attention as oa
    monkeypatch.setattr(oa, "attention_rows_fp64", _mutant(kind))
    q, k, v = _rand((1, 1, 17, 128), 36), _rand((1, 1, 29, 128), 37), _rand((1, 1, 29, 128), 38)
    scale = inputs.default_scale()
    got = oa.attention_fp64(q, k, v, scale)
    want = _sdpa(q, k, v, float(np.float32(scale)))
    assert not np.allclose(got, want, rtol=1e-12, atol=1e-13)


# --- follow-on steps: causal mask (bottom-right aligned) and grouped-query heads --

def _sdpa_mask(q, k, v, scale, mask):
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(a)) for a in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.from_numpy(mask), scale=scale).numpy()


@pytest.mark.parametrize("Sq,Sk", [(7, 7), (5, 12), (130, 300)])
def test_causal_matches_sdpa_with_explicit_mask(Sq, Sk):
    q, k, v = _rand((1, 2, Sq, 128), 40), _rand((1, 2, Sk, 128), 41), _rand((1, 2, Sk, 128), 42)
    scale = inputs.default_scale()
    allowed = np.arange(Sk)[None, :] <= np.arange(Sq)[:, None] + (Sk - Sq)
    got = attention_fp64(q, k, v, scale, causal=True)
    want = _sdpa_mask(q, k, v, float(np.float32(scale)), allowed)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_causal_closed_forms():
    q, k, v = _rand((1, 1, 6, 128), 43), _rand((1, 1, 6, 128), 44), _rand((1, 1, 6, 128), 45)
    o = attention_fp64(q, k, v, 0.1, causal=True)
    assert (o[0, 0, 0] == v[0, 0, 0]).all()           # first query sees only key 0
    full = attention_fp64(q, k, v, 0.1)
    np.testing.assert_allclose(o[0, 0, -1], full[0, 0, -1], rtol=1e-14)  # last sees all
    # more queries than keys: the first Sq - Sk rows see no key and are NaN
    o = attention_fp64(_rand((1, 1, 9, 128), 46), k[:, :, :4], v[:, :, :4], 0.1, causal=True)
    assert np.isnan(o[0, 0, :5]).all() and np.isfinite(o[0, 0, 5:]).all()
    assert (o[0, 0, 5] == v[0, 0, 0]).all()


def test_gqa_equals_repeated_heads_and_sdpa():
    q = _rand((2, 6, 11, 128), 47)
    k, v = _rand((2, 2, 13, 128), 48), _rand((2, 2, 13, 128), 49)
    got = attention_fp64(q, k, v, 0.09)
    rep = attention_fp64(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.09)
    assert (got == rep).all()
    qt, kt, vt = (torch.from_numpy(a) for a in (q, k, v))
    want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=float(np.float32(0.09)),
                                                            enable_gqa=True).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):
        attention_fp64(q, k[:, :1].repeat(4, axis=1), v[:, :1].repeat(4, axis=1), 0.1)


# --- follow-on step: variable-length batches (packed tokens, cu_seqlens) ---------

def _packed(lengths, H, seed):
    total = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return _rand((total, H, 128), seed), cu


def _block_mask(cq, ck, causal):
    """Allowed (query, key) pairs of the packed batch, built position by position."""
    tq, tk = int(cq[-1]), int(ck[-1])
    allowed = np.zeros((tq, tk), dtype=bool)
    for b in range(len(cq) - 1):
        for i in range(cq[b], cq[b + 1]):
            for j in range(ck[b], ck[b + 1]):
                li, lj = i - cq[b], j - ck[b]
                lq, lk = cq[b + 1] - cq[b], ck[b + 1] - ck[b]
                allowed[i, j] = (not causal) or lj <= li + (lk - lq)
    return allowed


_VL_Q, _VL_K = [5, 1, 17, 9], [7, 3, 17, 2]


def _varlen_pin(fn, causal):
    """Compares fn (an attention_varlen_fp64) with torch SDPA over the whole packed
    batch under an explicit block-diagonal mask; returns (matches, unseen rows)."""
    q, cq = _packed(_VL_Q, 4, 60)
    k, ck = _packed(_VL_K, 2, 61)
    v, _ = _packed(_VL_K, 2, 62)
    scale = inputs.default_scale()
    got = fn(q, k, v, cq, ck, scale, causal=causal)
    allowed = _block_mask(cq, ck, causal)
    # The packed batch as one (1, H, T, d) problem; K/V heads repeated for the
    # query heads that share them.
    qt = np.swapaxes(q, 0, 1)[None]
    kt = np.repeat(np.swapaxes(k, 0, 1)[None], 2, axis=1)
    vt = np.repeat(np.swapaxes(v, 0, 1)[None], 2, axis=1)
    want = np.swapaxes(_sdpa_mask(qt, kt, vt, float(np.float32(scale)), allowed)[0], 0, 1)
    seen = allowed.any(axis=1)
    ok = (np.allclose(got[seen], want[seen], rtol=1e-12, atol=1e-13)
          and bool(np.isnan(got[~seen]).all()))
    return ok, int((~seen).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_sdpa_with_block_diagonal_mask(causal):
    ok, unseen = _varlen_pin(oracle.attention_varlen_fp64, causal)
    assert ok
    # Causal: the last sequence has 9 queries and 2 keys, so its first 7 rows see
    # no key and are NaN.
    assert unseen == (7 if causal else 0)


def _mutant_varlen(kind):
    real = oracle.attention_fp64

    def fn(q, k, v, cq, ck, scale, causal=False):
        out = np.empty(q.shape)
        for b in range(len(cq) - 1):
            q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
            if kind == "key_offset_from_q":
                k0, k1 = int(cq[b]), int(cq[b]) + (k1 - k0)
            if kind == "key_off_by_one":
                k1 = min(k1 + 1, k.shape[0])
            if q1 == q0:
                continue
            if k1 <= k0:
                out[q0:q1] = np.nan
                continue
            kk, vv = k[None, k0:k1], v[None, k0:k1]
            if kind == "top_left_causal" and causal:
                # causal aligned at the top left: query i sees keys 0..i
                lq, lk = q1 - q0, k1 - k0
                o = real(q[None, q0:q1], kk, vv, scale, layout="bshd")[0]
                for i in range(lq):
                    n = min(i + 1, lk)
                    o[i] = real(q[None, q0 + i:q0 + i + 1], kk[:, :n], vv[:, :n], scale,
                                layout="bshd")[0][0]
                out[q0:q1] = o
                continue
            out[q0:q1] = real(q[None, q0:q1], kk, vv, scale, layout="bshd", causal=causal)[0]
        return out
    return fn


@pytest.mark.parametrize("kind", ["key_offset_from_q", "key_off_by_one", "top_left_causal"])
def test_varlen_planted_mistakes_are_caught(kind):
    assert not _varlen_pin(_mutant_varlen(kind), causal=True)[0]
    assert _varlen_pin(_mutant_varlen("none"), causal=True)[0]


def test_varlen_sequence_order_does_not_matter():
    lq, lk = [3, 8, 5], [4, 8, 6]
    q, cq = _packed(lq, 2, 63)
    k, ck = _packed(lk, 2, 64)
    v, _ = _packed(lk, 2, 65)
    got = oracle.attention_varlen_fp64(q, k, v, cq, ck, 0.1, causal=True)
    order = [2, 0, 1]
    def perm(x, cu):
        return np.concatenate([x[cu[b]:cu[b + 1]] for b in order])
    cq2 = np.concatenate([[0], np.cumsum([lq[b] for b in order])])
    ck2 = np.concatenate([[0], np.cumsum([lk[b] for b in order])])
    got2 = oracle.attention_varlen_fp64(perm(q, cq), perm(k, ck), perm(v, ck), cq2, ck2, 0.1,
                                        causal=True)
    assert (perm(got, cq) == got2).all()


def test_varlen_empty_sequences():
    q, cq = _packed([0, 4, 3], 1, 66)
    k, ck = _packed([5, 0, 2], 1, 67)
    v, _ = _packed([5, 0, 2], 1, 68)
    got = oracle.attention_varlen_fp64(q, k, v, cq, ck, 0.1)
    assert np.isnan(got[0:4]).all()          # sequence 1 has queries but no keys
    # sequence 2 alone is ordinary attention of its 3 rows over its 2 keys
    want = _sdpa(q[None, 4:7].swapaxes(1, 2), k[None, 5:7].swapaxes(1, 2),
                 v[None, 5:7].swapaxes(1, 2), float(np.float32(0.1)))
    np.testing.assert_allclose(got[4:7], want[0].swapaxes(0, 1), rtol=1e-12, atol=1e-13)
    with pytest.raises(ValueError):
        oracle.attention_varlen_fp64(q, k, v, [0, 4, 3, 7], ck, 0.1)


def test_causal_hidden_keys_take_no_part_even_with_nonfinite_v():
    q, k, v = _rand((1, 1, 6, 128), 80), _rand((1, 1, 6, 128), 81), _rand((1, 1, 6, 128), 82)
    v_bad = v.copy()
    v_bad[0, 0, 4, 7] = np.nan      # key 4: seen by rows 4 and 5 only
    v_bad[0, 0, 5, 9] = np.inf      # key 5: seen by row 5 only
    got = attention_fp64(q, k, v_bad, 0.1, causal=True)
    clean = attention_fp64(q, k, v, 0.1, causal=True)
    # Rows 0..3 see neither key: the clean result (up to summation order).
    np.testing.assert_allclose(got[0, 0, :4], clean[0, 0, :4], rtol=1e-13, atol=1e-15)
    # Row i equals the unmasked definition over keys 0..i (the row's own truncated
    # problem); non-finite positions exactly.
    for i in range(6):
        want = attention_rows_fp64(q[0, 0], k[0, 0, :i + 1], v_bad[0, 0, :i + 1], 0.1, [i])[0]
        np.testing.assert_allclose(got[0, 0, i], want, rtol=1e-13, atol=1e-15)
    assert np.isnan(got[0, 0, 4:, 7]).all()
    assert got[0, 0, 5, 9] == np.inf and np.isfinite(got[0, 0, 4, 9])


def test_varlen_other_sequences_nonfinite_v_takes_no_part():
    # Each sequence attends only within itself: NaN and infinities in another
    # sequence's V leave its rows exactly as if that sequence were alone, and a
    # sequence's own visible non-finite V shows in its rows.
    cq, ck = [0, 3, 7], [0, 5, 9]
    q, k, v = _rand((7, 2, 128), 90), _rand((9, 2, 128), 91), _rand((9, 2, 128), 92)
    v_bad = v.copy()
    v_bad[6, 0, 3] = np.nan        # sequence 1, key 1, head 0
    v_bad[8, 1, 4] = -np.inf       # sequence 1, key 3, head 1
    v_bad[0, 0, 5] = np.inf        # sequence 0, key 0, head 0
    for causal in (False, True):
        got = oracle.attention_varlen_fp64(q, k, v_bad, cq, ck, 0.1, causal=causal)
        for b in range(2):
            for h in range(2):
                sq = cq[b + 1] - cq[b]
                want = oracle.attention_rows_fp64(q[cq[b]:cq[b + 1], h], k[ck[b]:ck[b + 1], h],
                                                  v_bad[ck[b]:ck[b + 1], h], 0.1, np.arange(sq),
                                                  causal=causal)
                np.testing.assert_allclose(got[cq[b]:cq[b + 1], h], want, rtol=1e-13, atol=1e-15)
        # Sequence 0 holds none of sequence 1's values; sequence 1 none of sequence 0's.
        assert np.isfinite(got[0:3, 0, 3]).all() and np.isfinite(got[0:3, 1, 4]).all()
        assert np.isfinite(got[3:7, 0, 5]).all()
    got = oracle.attention_varlen_fp64(q, k, v_bad, cq, ck, 0.1)
    assert np.isnan(got[3:7, 0, 3]).all() and (got[3:7, 1, 4] == -np.inf).all()
    assert (got[0:3, 0, 5] == np.inf).all()
