"""The oracle against a 50-digit evaluation of the definition, on tiny inputs (CPU).

Each output is O[i,c] = sum_j p_ij V[j,c] / sum_j p_ij with p_ij = exp(s_ij - max_j s_ij)
and s_ij = scale * sum_c Q[i,c] K[j,c] (snilld.dk article "Open source attention-kernel
i HIP slaar AITER v3 paa MI300X", section "Hvordan kernen arbejder": softmax(QK^T/sqrt(d))V).
Here it is evaluated in mpmath at 50 significant digits from the exact bf16 input values
(every bf16 is a short binary fraction). No numpy routine and no fp64 step is shared with
the oracle. The oracle's fp64 result must agree to 1e-13, and its bf16 rounding in each mode
must equal the rounding of the high-precision value.
"""
import numpy as np
import pytest
import torch

from oracle import attention_fp64, round_bf16

mpmath = pytest.importorskip("mpmath")


def _bf16_values(shape, seed, std):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy((rng.standard_normal(shape) * std).astype(np.float32))
    return x.to(torch.bfloat16).to(torch.float64).numpy()  # exact bf16 values in float64


def _attention_mp(q, k, v, scale):
    """(Sq, d), (Sk, d), (Sk, d) -> (Sq, d) list of mpf, by the definition."""
    mp = mpmath.mp
    sc = mp.mpf(scale)
    kq = [[mp.mpf(float(x)) for x in row] for row in k]
    vq = [[mp.mpf(float(x)) for x in row] for row in v]
    out = []
    for row in q:
        qr = [mp.mpf(float(x)) for x in row]
        s = [sc * mp.fsum(a * b for a, b in zip(qr, kr)) for kr in kq]
        m = max(s)
        p = [mp.exp(x - m) for x in s]
        den = mp.fsum(p)
        out.append([mp.fsum(pj * vr[c] for pj, vr in zip(p, vq)) / den for c in range(len(vq[0]))])
    return out


@pytest.mark.parametrize("Sq,Sk,d,std,scale", [
    (1, 1, 128, 1.0, 128 ** -0.5),
    (3, 5, 128, 1.0, 128 ** -0.5),
    (8, 8, 128, 1.0, 128 ** -0.5),
    (4, 7, 128, 8.0, 128 ** -0.5),   # wide logits: the max subtraction carries the result
    (5, 6, 64, 1.0, -0.3),           # negative scale: the largest weight is the smallest dot
    (2, 8, 32, 1.0, 0.0),            # zero scale: the column mean of V
])
def test_oracle_matches_50_digit_definition(Sq, Sk, d, std, scale):
    mpmath.mp.dps = 50
    seed = 7000 + 100 * Sq + Sk + d
    q = _bf16_values((1, 1, Sq, d), seed, std)
    k = _bf16_values((1, 1, Sk, d), seed + 1, std)
    v = _bf16_values((1, 1, Sk, d), seed + 2, 1.0)
    scale_f = float(np.float32(scale))  # both sides use the fp32 scale, widened
    got = attention_fp64(q, k, v, scale_f, "bhsd")[0, 0]
    exact = _attention_mp(q[0, 0], k[0, 0], v[0, 0], scale_f)
    ref = np.array([[float(x) for x in row] for row in exact])
    assert np.abs(got - ref).max() <= 1e-13
    for mode in ("rtne", "rtna", "rtz"):
        assert np.array_equal(round_bf16(got, mode), round_bf16(ref, mode)), mode


def test_grouped_heads_match_50_digit_definition():
    # Two query heads share one key/value head (grouped-query attention).
    mpmath.mp.dps = 50
    q = _bf16_values((1, 2, 3, 32), 7100, 1.0)
    k = _bf16_values((1, 1, 4, 32), 7101, 1.0)
    v = _bf16_values((1, 1, 4, 32), 7102, 1.0)
    scale = float(np.float32(32 ** -0.5))
    got = attention_fp64(q, k, v, scale, "bhsd")[0]
    for h in range(2):
        ref = np.array([[float(x) for x in row] for row in _attention_mp(q[0, h], k[0, 0], v[0, 0],
                                                                          scale)])
        assert np.abs(got[h] - ref).max() <= 1e-13


def _mutant(kind):
    """A copy of the oracle's row routine with one plausible mistake planted."""
    def rows(q, k, v, scale, rows=None, causal=False):
        scale_d = float(np.float32(scale))
        if rows is not None:
            q = q[np.asarray(rows)]
        if kind == "fp32_logits":  # products summed in fp32 instead of fp64
            s = (q.astype(np.float32) @ k.T.astype(np.float32)).astype(np.float64) * scale_d
        elif kind == "no_scale":
            s = q @ k.T
        else:
            s = (q @ k.T) * scale_d
        p = np.exp(s - np.max(s, axis=1, keepdims=True))
        if kind == "wrong_axis":
            return (p / p.sum(axis=0, keepdims=True)) @ v
        return p @ v / np.sum(p, axis=1, keepdims=True)
    return rows


@pytest.mark.parametrize("kind", ["fp32_logits", "no_scale", "wrong_axis"])
def test_planted_mistakes_fail_the_50_digit_pin(kind, monkeypatch):
    import oracle.attention as oa
    monkeypatch.setattr(oa, "attention_rows_fp64", _mutant(kind))
    mpmath.mp.dps = 50
    q = _bf16_values((1, 1, 6, 128), 7200, 1.0)
    k = _bf16_values((1, 1, 8, 128), 7201, 1.0)
    v = _bf16_values((1, 1, 8, 128), 7202, 1.0)
    scale = float(np.float32(128 ** -0.5))
    got = oa.attention_fp64(q, k, v, scale, "bhsd")[0, 0]
    ref = np.array([[float(x) for x in row] for row in _attention_mp(q[0, 0], k[0, 0], v[0, 0],
                                                                      scale)])
    assert np.abs(got - ref).max() > 1e-13
