"""Non-finite values in V at keys that some rows do not see, on a GB300.

Under the causal mask and at the end of a sequence of a packed batch, a row's
hidden keys take no part in its output: a NaN or an infinity in V at such a key
must not reach that row, while every row that sees the key gets it (NaN stays
NaN; an infinity times the key's positive weight is that infinity). The kernel
meets these keys inside the key tiles it computes for the diagonal and for the
sequence end; the tests plant non-finite V values there and compare positions
and bits with the fp64 oracle, which evaluates each row over its visible keys.

NaN must come out as the one pattern 0x7FC0 everywhere the oracle has NaN. An
infinity that a row sees through a key tile without hidden keys passes through
the tensor pipe's two-term product, which can turn it into NaN (the kernel's
documented deviation for +-Inf in V): there the test accepts 0x7FC0 for the
oracle's +-Inf, and everywhere the positions must match exactly.
"""
import numpy as np
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
from oracle import attention_fp64, attention_varlen_fp64, nonfinite_bits, round_bf16

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu

NAN, NNAN, PINF, NINF = 0x7FC0, 0xFFC1, 0x7F80, 0xFF80


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _plant(t, idx, bits):
    t.view(torch.int16)[idx] = int(np.uint16(bits).view(np.int16))


def _check(got, exact, mode, inf_may_be_nan=None):
    """Positions exact; NaN bits exact; where inf_may_be_nan (a boolean mask of
    the output) is set, an expected +-Inf may come out as 0x7FC0."""
    want = round_bf16(exact, mode)
    nf_w, nf_g = nonfinite_bits(want), nonfinite_bits(got)
    assert (nf_w == nf_g).all(), np.argwhere(nf_w != nf_g)[:10]
    same = got == want
    if inf_may_be_nan is not None:
        same |= inf_may_be_nan & (got == NAN) & ((want == PINF) | (want == NINF))
    assert same[nf_w].all(), np.argwhere(nf_w & ~same)[:10]
    fin = ~nf_w
    fin_stats = compare(np.where(fin, got, 0).astype(np.uint16), np.where(fin, exact, 0.0), mode)
    assert_parity(fin_stats, excess=True)
    return want


@pytest.mark.parametrize("layout", ["bhsd", "bshd"])
@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
def test_causal_hidden_keys_keep_nonfinite_v_out(layout, mode):
    B, H, S = 1, 2, 300
    w = inputs.Workload("nfv", layout, B, H, S, S, seed=95)
    q, k, v = inputs.make_qkv(w)
    at = (lambda h, s, c: (0, h, s, c)) if layout == "bhsd" else (lambda h, s, c: (0, s, h, c))
    # Head 0: NaNs of both signs and infinities at keys inside the first CTA's
    # diagonal tiles (rows 0..255) and in the second CTA's (rows 256..299).
    plants = [(0, 40, 3, NAN), (0, 200, 9, NNAN), (0, 131, 64, PINF), (0, 255, 127, NINF),
              (0, 299, 5, PINF), (0, 260, 70, NAN),
              # Head 1: +Inf and -Inf at two keys of one column (rows that see
              # both get NaN), and a NaN at the very first key (every row sees it).
              (1, 100, 20, PINF), (1, 180, 20, NINF), (1, 0, 100, NNAN)]
    for h, s, c, bits in plants:
        _plant(v, at(h, s, c), bits)
    out = attn.attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), causal=True, layout=layout, rounding=mode)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    got = bits_of(out)
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout,
                           causal=True)
    # Rows 256..299 see keys 0..255 through key tiles without hidden keys.
    late = np.arange(S) >= 256
    may = np.broadcast_to(late[None, None, :, None] if layout == "bhsd"
                          else late[None, :, None, None], got.shape)
    want = _check(got, exact, mode, may)
    # Spot checks straight from the definition (head 0, bottom-right aligned mask).
    g = got[0, 0] if layout == "bhsd" else got[0, :, 0]
    assert (g[:40, 3] != NAN).all() and (g[40:, 3] == NAN).all()
    assert (g[:200, 9] != NAN).all() and (g[200:, 9] == NAN).all()
    assert not nonfinite_bits(g[:131, 64]).any()
    assert (g[131:256, 64] == PINF).all()          # seen through a masked tile: exact +Inf
    assert (g[255:256, 127] == NINF).all() and (g[:255, 127] != NINF).all()
    assert g[299, 5] == PINF and (g[:299, 5] != PINF).all()
    assert (g[:260, 70] != NAN).all() and (g[260:, 70] == NAN).all()
    g1 = got[0, 1] if layout == "bhsd" else got[0, :, 1]
    assert (g1[180:256, 20] == NAN).all() and (g1[100:180, 20] == PINF).all()
    assert (g1[:, 100] == NAN).all()
    assert int(nonfinite_bits(want).sum()) == int(nonfinite_bits(got).sum())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mode", inputs.ROUNDINGS)
def test_varlen_next_sequence_keys_keep_nonfinite_v_out(causal, mode):
    # Sequence 0 ends inside a key tile that runs on into sequence 1's keys;
    # sequence 1 ends inside a tile that runs into sequence 2's. Non-finite V at
    # those following keys must stay in their own sequence.
    lq, lk, Hq, Hkv = [150, 200, 90], [150, 300, 77], 2, 1
    w = inputs.Workload("nfv_vl", "thd", len(lq), Hq, max(lq), max(lk), seed=97, hkv=Hkv,
                        seqlens=tuple(zip(lq, lk)))
    q, k, v = inputs.make_qkv(w)
    cq, ck = w.cu_seqlens
    # (global key token, column, bits)
    plants = [(int(ck[1]) + 10, 3, NAN), (int(ck[1]) + 40, 7, NNAN), (int(ck[1]) + 100, 8, PINF),
              (int(ck[2]) + 2, 11, NINF), (int(ck[2]) + 76, 12, NAN), (int(ck[1]) - 1, 13, NAN),
              (int(ck[2]) - 1, 14, PINF)]
    for tok, c, bits in plants:
        _plant(v, (tok, 0, c), bits)
    out = attn.attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cq).cuda(),
                               torch.from_numpy(ck).cuda(), max(lq), causal=causal, rounding=mode)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    got = bits_of(out)
    exact = attention_varlen_fp64(f64_of(q), f64_of(k), f64_of(v), cq, ck, inputs.default_scale(),
                                  causal=causal)
    # Sequence 1's keys past its first tile are seen by its rows through tiles
    # without hidden keys only where the tile holds no key of another sequence.
    _check(got, exact, mode, np.ones(got.shape, dtype=bool))
    # Sequence 0 gets none of sequence 1's values.
    s0 = got[:lq[0]]
    assert not (nonfinite_bits(s0[:, :, 3]) | nonfinite_bits(s0[:, :, 7]) |
                nonfinite_bits(s0[:, :, 8])).any()
