"""Parity of the CUDA path (through the C ABI) against the fp64 oracle, on a GB300.

Small shapes are compared element by element over whole tensors: they span several
query/key tiles and ragged tails in both layouts and all three rounding modes.
The five full-size synthetic workloads run in the same launch configuration as
the benchmark and are compared on sampled rows (the first and last rows of tiles
plus random rows), with the NaN/Inf pattern of the stress case checked over the
whole tensor against its closed form.
"""
import json

import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_fp64, attention_rows_fp64, nonfinite_bits, round_bf16, to_bhsd

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _gpu(q, k, v, layout, mode, scale=None):
    out = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), layout=layout, rounding=mode, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    return out


def _full_check(w, mode, scale=None, max_abs_err=8e-3):
    q, k, v = inputs.make_qkv(w)
    sc = inputs.default_scale() if scale is None else scale
    out = _gpu(q, k, v, w.layout, mode, sc)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), sc, w.layout)
    stats = compare(bits_of(out), exact, mode)
    assert_parity(stats, max_abs_err)
    return stats


SMALL = [
    ("bhsd", 1, 2, 256, 256),
    ("bshd", 1, 3, 1, 1),
    ("bhsd", 2, 1, 2, 129),
    ("bshd", 1, 2, 127, 128),
    ("bhsd", 1, 1, 129, 255),
    ("bshd", 2, 2, 300, 257),
    ("bhsd", 1, 2, 513, 1000),
    ("bshd", 1, 1, 384, 4096),
    ("bhsd", 1, 3, 700, 130),
]


@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
@pytest.mark.parametrize("layout,B,H,Sq,Sk", SMALL)
def test_small_shapes(layout, B, H, Sq, Sk, mode):
    w = inputs.Workload("small", layout, B, H, Sq, Sk, seed=1000 + Sq * 7 + Sk)
    _full_check(w, mode)


@pytest.mark.parametrize("scale", [0.0, -0.0883883, 0.5, 1e-3])
def test_other_scales(scale):
    w = inputs.Workload("scales", "bhsd", 1, 2, 200, 333, seed=77)
    _full_check(w, "rtne", scale=scale, max_abs_err=2e-2 if scale == 0.5 else 8e-3)


@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
def test_wide_logits_uniform_v(mode):
    w = inputs.Workload("wide", "bshd", 1, 2, 300, 600, qk_std=8.0, v_dist="uniform", seed=78)
    _full_check(w, mode, max_abs_err=None)


def test_nan_and_inf_propagation():
    w = inputs.Workload("spec", "bhsd", 1, 2, 260, 300, seed=79)
    q, k, v = inputs.make_qkv(w)
    q[0, 0, 5, 17] = float("nan")
    k[0, 1, 200, 40] = float("inf")
    q[0, 1, 0:4, 40] = torch.tensor([0.0, -0.0, 1.0, -1.0], dtype=torch.bfloat16)
    k[0, 0, 299, 3] = float("-inf")  # last key of the ragged tail tile
    for mode in inputs.ROUNDINGS:
        out = _gpu(q, k, v, "bhsd", mode)
        exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), "bhsd")
        stats = compare(bits_of(out), exact, mode)
        assert_parity(stats)
        assert stats["n_nonfinite"] > 128


def test_minus_inf_keys_fill_a_whole_tile():
    # Every key of the first key tile has logit -Inf for row 0: the running max stays
    # -Inf through that tile and the weights must still come out as exactly 0.
    w = inputs.Workload("minf", "bhsd", 1, 1, 4, 300, seed=80)
    q, k, v = inputs.make_qkv(w)
    q[0, 0, 0, 9] = 1.0
    k[0, 0, :128, 9] = float("-inf")
    out = _gpu(q, k, v, "bhsd", "rtne")
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), "bhsd")
    assert_parity(compare(bits_of(out), exact, "rtne"))


def test_deterministic_reruns():
    w = inputs.Workload("det", "bshd", 1, 4, 1000, 3000, seed=81)
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    a = attn.attn_fwd(q, k, v, layout="bshd")
    b = attn.attn_fwd(q, k, v, layout="bshd")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_layouts_agree_bitwise():
    w = inputs.Workload("lay", "bhsd", 2, 3, 333, 444, seed=82)
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    a = attn.attn_fwd(q, k, v, layout="bhsd")
    t = lambda x: x.transpose(1, 2).contiguous()
    b = attn.attn_fwd(t(q), t(k), t(v), layout="bshd")
    torch.cuda.synchronize()
    assert torch.equal(t(a).view(torch.int16), b.view(torch.int16))


def test_out_argument_and_stream():
    w = inputs.Workload("st", "bhsd", 1, 1, 130, 140, seed=83)
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    out = torch.full_like(q, float("nan"))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r = attn.attn_fwd(q, k, v, out=out)
    s.synchronize()
    assert r.data_ptr() == out.data_ptr() and not torch.isnan(out).any()


# ---------------------------------------------------------------- full size

def _sample_rows(Sq, rng, n_random):
    fixed = {0, 1, 127, 128, 129, 255, 256, Sq // 2, Sq - 129, Sq - 128, Sq - 2, Sq - 1}
    rows = {r for r in fixed if 0 <= r < Sq} | set(rng.integers(0, Sq, n_random).tolist())
    return np.array(sorted(rows))


def _closed_form_nonfinite_rows(w, q):
    """Rows that must be NaN in the stress workload: the Q row holding a NaN, and in
    the head holding K[j, c'] = +Inf every row i with scale * Q[i, c'] >= 0
    (s_ij is then +Inf or NaN, so exp(s - max) is NaN)."""
    qb = to_bhsd(q.view(torch.int16).numpy(), w.layout)
    mask = np.zeros((w.B, w.H, w.Sq), dtype=bool)
    for b, (h, i, _c), (h2, _j, c2) in inputs.special_positions(w):
        mask[b, h, i] = True
        col = qb[b, h2, :, c2].astype(np.uint16)
        is_nan = (col & 0x7FFF) > 0x7F80
        negative = (col & 0x8000) != 0
        mask[b, h2] |= is_nan | ~negative  # q >= 0 (incl. -0) or NaN
    return mask


@pytest.mark.parametrize("name", ["self8k", "cross4k32k", "long128k", "stress16381", "short77"])
def test_full_size_sampled(name):
    w = inputs.WORKLOADS[name]
    q, k, v = inputs.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    scale = inputs.default_scale()
    rng = np.random.default_rng(w.seed)
    qb, kb, vb = (to_bhsd(t.view(torch.int16).numpy(), w.layout) for t in (q, k, v))
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    n_rand = max(4, 512 // len(heads))
    plan = []
    for b, h in heads:
        rows = _sample_rows(w.Sq, rng, n_rand)
        if w.specials:
            for bb, (hq, iq, _), (hk, _j, _c) in inputs.special_positions(w):
                if bb == b and hq == h:
                    rows = np.union1d(rows, [iq])
        plan.append((b, h, rows))
    exact = []
    from oracle import bf16_bits_to_f64
    for b, h, rows in plan:
        kh, vh = bf16_bits_to_f64(kb[b, h]), bf16_bits_to_f64(vb[b, h])
        exact.append(attention_rows_fp64(bf16_bits_to_f64(qb[b, h]), kh, vh, scale, rows))
    exact = np.concatenate(exact)
    for mode in w.roundings:
        out = attn.attn_fwd(qd, kd, vd, layout=w.layout, rounding=mode)
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        ob = to_bhsd(bits_of(out), w.layout)
        got = np.concatenate([ob[b, h, rows] for b, h, rows in plan])
        stats = compare(got, exact, mode)
        print(f"\nPARITY {name} {mode}: " + json.dumps(stats))
        assert_parity(stats, 8e-3 if w.qk_std == 1.0 else None)
        if w.specials:
            mask = _closed_form_nonfinite_rows(w, q)
            nan_rows = ((ob & 0x7FFF) > 0x7F80).all(axis=-1)
            finite_rows = ((ob & 0x7F80) != 0x7F80).all(axis=-1)
            assert (nan_rows == mask).all()
            assert (finite_rows == ~mask).all()
    if name == "self8k":
        again = attn.attn_fwd(qd, kd, vd, layout=w.layout, rounding=w.roundings[-1])
        torch.cuda.synchronize()
        assert torch.equal(again.view(torch.int16), out.view(torch.int16))


def _v_specials(layout, causal, plant):
    w = inputs.Workload("vs", layout, 1, 2, 300, 300, seed=90)
    q, k, v = inputs.make_qkv(w)
    vb = v.view(torch.int16).numpy()  # bf16 bit patterns, in place
    for (h, j, c, bits) in plant:
        vb[index_of_layout(layout, 0, h, j, c)] = np.uint16(bits).view(np.int16)
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, layout=layout)
    torch.cuda.synchronize()
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout,
                           causal=causal)
    return bits_of(out), exact


def index_of_layout(layout, b, h, s, c):
    return (b, h, s, c) if layout == "bhsd" else (b, s, h, c)


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
def test_nan_in_v_propagates_exactly(layout):
    got, exact = _v_specials(layout, False, [(0, 17, 5, 0x7FC0), (1, 299, 100, 0xFFC1)])
    stats = compare(got, exact, "rtne")
    assert stats["n_nonfinite"] == 2 * 300
    assert_parity(stats)


def test_nan_in_v_at_a_key_every_causal_row_sees():
    got, exact = _v_specials("bhsd", True, [(0, 0, 3, 0x7FC0)])
    stats = compare(got, exact, "rtne")
    assert stats["n_nonfinite"] == 300
    assert_parity(stats, excess=True)


def test_inf_in_v_positions():
    # +-Inf in V: the exact output is +-Inf in that column (p > 0 times Inf). The
    # kernel's two-term P meets it as P_hi*Inf + P_lo*Inf, where P_lo <= 0 or 0
    # gives Inf - Inf or 0 * Inf = NaN: the positions are exact, the pattern may be
    # the NaN instead of the Inf (a documented deviation).
    got, exact = _v_specials("bshd", False, [(0, 40, 8, 0x7F80), (1, 200, 77, 0xFF80)])
    want = round_bf16(exact, "rtne")
    nf_w, nf_g = nonfinite_bits(want), nonfinite_bits(got)
    assert nf_w.sum() == 2 * 300 and (nf_w == nf_g).all()
    ok = (got[nf_w] == want[nf_w]) | (got[nf_w] == 0x7FC0)
    assert ok.all()
    finite = ~nf_w
    fin_stats = compare(np.where(finite, got, 0).astype(np.uint16), np.where(finite, exact, 0.0),
                        "rtne")
    assert_parity(fin_stats)

