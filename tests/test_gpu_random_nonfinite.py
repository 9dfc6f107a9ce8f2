"""Seeded random configurations with NaN and infinities planted in Q, K and V, against
the fp64 oracle: the causal mask, grouped heads and packed variable-length batches,
where some planted values sit at keys that some rows do not see.

Every NaN or infinity of the oracle must appear at the same position, and nowhere
else; NaN is the one pattern 0x7FC0. An infinity that a row sees through a key tile
without hidden keys may come out as NaN (the kernel's documented deviation for
+-Inf in V), so an expected +-Inf accepts 0x7FC0 too. Finite outputs meet the
usual bar. Planted K values never share a key with a planted V value: a key whose
logit is -Inf has weight 0, and 0 * Inf is NaN in the oracle, a case the kernel
does not single out inside the tiles it checks."""
import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_fp64, attention_varlen_fp64, nonfinite_bits, round_bf16

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu

SPECIALS = [0x7FC0, 0xFFC1, 0x7F80, 0xFF80]
LENGTHS = [1, 31, 127, 128, 129, 200, 255, 256, 257, 383, 511, 640]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _set(t, idx, bits):
    t.view(torch.int16)[idx] = int(np.uint16(bits).view(np.int16))


def _check(got, exact, mode):
    want = round_bf16(exact, mode)
    nf_w, nf_g = nonfinite_bits(want), nonfinite_bits(got)
    assert (nf_w == nf_g).all(), np.argwhere(nf_w != nf_g)[:8]
    inf_w = (want == 0x7F80) | (want == 0xFF80)
    ok = (got == want) | (inf_w & (got == 0x7FC0))
    assert ok[nf_w].all(), np.argwhere(nf_w & ~ok)[:8]
    fin = ~nf_w
    stats = compare(np.where(fin, got, 0).astype(np.uint16), np.where(fin, exact, 0.0), mode)
    assert_parity(stats, excess=True)


def _plants(rng, n_keys_of, n):
    """n (tensor, key-or-row index, column, bits) plants; K plants avoid V's keys."""
    out, v_keys = [], set()
    for _ in range(n):
        which = str(rng.choice(["v", "v", "v", "v", "k", "q"]))
        out.append([which, None, int(rng.integers(0, 128)), int(rng.choice(SPECIALS))])
    for p in out:
        if p[0] == "v":
            p[1] = int(rng.integers(0, n_keys_of("v")))
            v_keys.add(p[1])
    for p in out:
        if p[0] == "k":
            free = [j for j in range(n_keys_of("k")) if j not in v_keys]
            p[1] = int(rng.choice(free)) if free else None
        elif p[0] == "q":
            p[1] = int(rng.integers(0, n_keys_of("q")))
    return [p for p in out if p[1] is not None]


@pytest.mark.parametrize("i", range(24))
def test_random_nonfinite_fixed_length(i):
    rng = np.random.default_rng(20260200 + i)
    hkv = int(rng.choice([1, 2]))
    layout = str(rng.choice(["bhsd", "bshd"]))
    B, Hq = int(rng.integers(1, 3)), hkv * int(rng.choice([1, 2]))
    Sq, Sk = int(rng.choice(LENGTHS)), int(rng.choice(LENGTHS))
    causal = bool(rng.random() < 0.7)
    mode = str(rng.choice(inputs.ROUNDINGS))
    q, _, _ = inputs.make_qkv(inputs.Workload("rn", layout, B, Hq, Sq, Sk, seed=40000 + i))
    _, k, v = inputs.make_qkv(inputs.Workload("rn", layout, B, hkv, Sq, Sk, seed=40500 + i))

    def idx(b, h, s, c):
        return (b, h, s, c) if layout == "bhsd" else (b, s, h, c)

    lens = {"q": B * Sq, "k": B * Sk, "v": B * Sk}
    for which, flat, c, bits in _plants(rng, lambda t: lens[t], int(rng.integers(1, 7))):
        S = Sq if which == "q" else Sk
        b, s = divmod(flat, S)
        h = int(rng.integers(0, Hq if which == "q" else hkv))
        _set({"q": q, "k": k, "v": v}[which], idx(b, h, s, c), bits)
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=causal, layout=layout,
                           rounding=mode)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout,
                           causal=causal)
    _check(bits_of(out), exact, mode)


@pytest.mark.parametrize("i", range(12))
def test_random_nonfinite_varlen(i):
    rng = np.random.default_rng(20260300 + i)
    nseq = int(rng.integers(2, 5))
    lq = [int(rng.choice([0, 5, 100, 128, 200, 300])) for _ in range(nseq)]
    lk = [int(rng.choice([1, 77, 128, 129, 250, 400])) for _ in range(nseq)]
    if sum(lq) == 0:
        lq[0] = 50
    causal = bool(rng.random() < 0.5)
    mode = str(rng.choice(inputs.ROUNDINGS))
    Hq, Hkv = 2, int(rng.choice([1, 2]))
    w = inputs.Workload("rnv", "thd", nseq, Hq, max(lq), max(lk), seed=41000 + i, hkv=Hkv,
                        seqlens=tuple(zip(lq, lk)))
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    lens = {"q": int(cq[-1]), "k": int(ck[-1]), "v": int(ck[-1])}
    for which, tok, c, bits in _plants(rng, lambda t: lens[t], int(rng.integers(1, 7))):
        h = int(rng.integers(0, Hq if which == "q" else Hkv))
        _set({"q": q, "k": k, "v": v}[which], (tok, h, c), bits)
    out = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cq).cuda(),
                               torch.from_numpy(ck).cuda(), max(1, max(lq)), causal=causal,
                               rounding=mode)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    exact = attention_varlen_fp64(f64_of(q), f64_of(k), f64_of(v), cq, ck,
                                  inputs.default_scale(), causal=causal)
    _check(bits_of(out), exact, mode)
