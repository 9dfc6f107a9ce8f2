"""The chunk plans of the host-buffer entry points (csrc/host_plan.h), built with
the host C++ compiler and checked by simulating their copies on tagged tensors:
no GPU is needed.

Every (token, head) row of d = 128 bf16 is 256 bytes, and every offset, width and
pitch of a plan is a whole number of rows. A tagged tensor holds, for each row,
its global (batch, head, position) index; uploading the Q and K/V spans of the
chunks, in chunk order, into device arrays and then reading each chunk's
sub-tensors at its device offsets, in the caller's layout with the chunk's own
sizes, must give back exactly the rows of the whole problem that the chunk
stands for: a block of batch entries x heads x query rows, with the matching
key/value heads, keys from position 0, the causal alignment of the whole
problem, and K/V that are on the device before the chunk runs. Downloading the
output spans must write every host output row exactly once, from the device row
that holds it."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bf16_forward_attention_gb300", "csrc")
ROW = 256  # bytes per (token, head) row
MAX_CHUNKS = 8
CTAS_PER_CHUNK = 256

DRIVER = r"""
#include <cstdio>
#include <iostream>
#include <string>
#include <vector>
#include "host_plan.h"

static void put(const attn_plan::CopyArgs& a) {
  std::printf(" %lld %lld %lld %lld %lld %lld", (long long)a.dst, (long long)a.dpitch,
              (long long)a.src, (long long)a.spitch, (long long)a.width, (long long)a.rows);
}

int main() {
  std::string kind;
  while (std::cin >> kind) {
    if (kind == "d") {
      long long layout, B, Hq, Hkv, Sq, Sk, causal;
      std::cin >> layout >> B >> Hq >> Hkv >> Sq >> Sk >> causal;
      const auto chunks = attn_plan::plan(int(layout), B, Hq, Hkv, Sq, Sk, causal != 0);
      std::printf("%zu\n", chunks.size());
      for (const auto& c : chunks) {
        std::printf("%lld %lld %lld %lld %lld", (long long)c.B, (long long)c.Hq,
                    (long long)c.Hkv, (long long)c.Sq, (long long)c.Sk);
        for (const auto* s : {&c.q, &c.kv})
          std::printf(" %lld %lld %lld %lld %lld", (long long)s->host, (long long)s->dev,
                      (long long)s->width, (long long)s->rows, (long long)s->pitch);
        put(attn_plan::copy_args(c.q, true));
        put(attn_plan::copy_args(c.q, false));
        put(attn_plan::copy_args(c.kv, true));
        std::printf("\n");
      }
    } else {
      long long B, Hq;
      std::cin >> B >> Hq;
      std::vector<int32_t> cq(B + 1);
      for (auto& x : cq) { long long t; std::cin >> t; x = int32_t(t); }
      const auto chunks = attn_plan::plan_varlen(cq.data(), B, Hq);
      std::printf("%zu\n", chunks.size());
      for (const auto& c : chunks)
        std::printf("%lld %lld %lld\n", (long long)c.b0, (long long)c.b1, (long long)c.max_sq);
    }
    std::fflush(stdout);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    d = tmp_path_factory.mktemp("plan")
    src = d / "plan_driver.cpp"
    src.write_text(DRIVER)
    exe = d / "plan_driver"
    subprocess.run([cxx, "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC, str(src), "-o", str(exe)],
                   check=True)
    return str(exe)


def _run(exe, cases):
    """Plans for `cases` (tuples for the driver's input lines), one list per case."""
    text = "".join(" ".join(str(x) for x in c) + "\n" for c in cases)
    r = subprocess.run([exe], input=text, capture_output=True, text=True, check=True)
    lines = r.stdout.split("\n")
    out, i = [], 0
    for _ in cases:
        n = int(lines[i])
        out.append([[int(x) for x in lines[i + 1 + j].split()] for j in range(n)])
        i += 1 + n
    return out


def _rows_index(layout, B, H, S):
    """Row index of (b, h, s) in a dense (B, H, S) tensor of the layout, as [B, H, S]."""
    b = np.arange(B)[:, None, None]
    h = np.arange(H)[None, :, None]
    s = np.arange(S)[None, None, :]
    return (b * H + h) * S + s if layout == 0 else (b * S + s) * H + h


def _tags(layout, B, H, S):
    """A tagged host tensor: tag[row] = (b, h, s) of that row, as an (n, 3) array."""
    t = np.empty((B * H * S, 3), dtype=np.int64)
    idx = _rows_index(layout, B, H, S)
    t[idx, 0] = np.arange(B)[:, None, None]
    t[idx, 1] = np.arange(H)[None, :, None]
    t[idx, 2] = np.arange(S)[None, None, :]
    return t


def _copy(dst, dst_count, src, args):
    """A (2-D) copy in rows: `args` = dst, dpitch, src, spitch, width, rows (bytes)."""
    d0, dp, s0, sp, w, n = args
    for x in (d0, dp, s0, sp, w):
        assert x % ROW == 0
    if n == 0:
        return
    r = np.arange(n)[:, None]
    k = np.arange(w // ROW)[None, :]
    di = (d0 // ROW + r * (dp // ROW) + k).ravel()
    si = (s0 // ROW + r * (sp // ROW) + k).ravel()
    assert di.min() >= 0 and di.max() < len(dst), "copy outside the destination tensor"
    assert si.min() >= 0 and si.max() < len(src), "copy outside the source tensor"
    dst[di] = src[si]
    np.add.at(dst_count, di, 1)


def _check_dense(layout, B, Hq, Hkv, Sq, Sk, causal, chunks):
    group = Hq // Hkv
    want = min(max(B * Hq * -(-Sq // 256) // CTAS_PER_CHUNK, 1), MAX_CHUNKS)
    assert 1 <= len(chunks) <= MAX_CHUNKS
    if layout == 0:  # runs of key/value heads over all entries
        assert len(chunks) == min(want, B * Hkv)
        assert all(c[0] == 1 for c in chunks)
    if layout == 0:
        # (B, H, S, d) is the same memory as (1, B*H, S, d): heads are flat (b, h).
        B, Hq, Hkv = 1, B * Hq, B * Hkv
    hq, hkv = _tags(layout, B, Hq, Sq), _tags(layout, B, Hkv, Sk)
    dq, dkv = np.full_like(hq, -1), np.full_like(hkv, -1)
    nq, nkv = np.zeros(len(hq), np.int64), np.zeros(len(hkv), np.int64)
    ho, no = np.full_like(hq, -1), np.zeros(len(hq), np.int64)
    for c in chunks:
        cB, cHq, cHkv, cSq, cSk = c[:5]
        q_span, kv_span = c[5:10], c[10:15]
        q_up, q_down, kv_up = c[15:21], c[21:27], c[27:33]
        assert min(cB, cHq, cHkv, cSq, cSk) >= 1
        assert cHq == cHkv * group
        assert q_span[1] % ROW == 0 and kv_span[1] % ROW == 0  # 16-byte aligned device bases
        # The Q span is exactly the chunk's Q; the K/V span (when it copies) holds
        # at least the chunk's K/V.
        assert q_span[2] * q_span[3] == cB * cHq * cSq * ROW
        if kv_span[3]:
            assert kv_span[2] * kv_span[3] >= cB * cHkv * cSk * ROW
        _copy(dq, nq, hq, q_up)
        _copy(dkv, nkv, hkv, kv_up)
        # The chunk's sub-tensors, read where its kernel reads them.
        iq = q_span[1] // ROW + _rows_index(layout, cB, cHq, cSq)
        ik = kv_span[1] // ROW + _rows_index(layout, cB, cHkv, cSk)
        assert iq.max() < len(dq) and ik.max() < len(dkv)
        tq, tk = dq[iq], dkv[ik]
        assert (tq >= 0).all(), "a chunk reads Q rows not uploaded before it"
        assert (tk >= 0).all(), "a chunk reads K/V rows not uploaded before it"
        b0, h0, s0 = tq[0, 0, 0]
        want_q = np.stack(np.broadcast_arrays(b0 + np.arange(cB)[:, None, None],
                                              h0 + np.arange(cHq)[None, :, None],
                                              s0 + np.arange(cSq)[None, None, :]), axis=-1)
        assert (tq == want_q).all(), "a chunk's Q is not a block of the whole problem"
        assert h0 % group == 0
        want_k = np.stack(np.broadcast_arrays(b0 + np.arange(cB)[:, None, None],
                                              h0 // group + np.arange(cHkv)[None, :, None],
                                              np.arange(cSk)[None, None, :]), axis=-1)
        assert (tk == want_k).all(), "a chunk's K/V do not belong to its query heads"
        # Causal: row s' of the chunk sees keys up to s' + cSk - cSq, as row s0 + s'
        # of the whole problem does (keys up to s0 + s' + Sk - Sq); no row of a
        # chunk sees fewer than one key unless it sees none in the whole problem.
        if causal:
            assert cSk - cSq == s0 + Sk - Sq
            assert cSk <= Sk
        else:
            assert cSk == Sk
        # The kernel writes O where Q sits; the download brings it back.
        _copy(ho, no, dq, q_down)
    assert (nq == 1).all() and (nkv == 1).all(), "device rows written other than once"
    assert (no == 1).all(), "host output rows written other than once"
    assert (ho == hq).all(), "an output row lands in the wrong place"


DENSE_EDGES = [
    # layout, B, Hq, Hkv, Sq, Sk, causal
    (1, 2, 16, 16, 8192, 8192, 0),   # the 8K self-attention shape: runs of heads
    (1, 2, 16, 4, 8192, 8192, 1),    # grouped heads, causal
    (1, 1, 32, 32, 16384, 16384, 0),  # one entry: 8 runs of 4 heads
    (1, 1, 32, 1, 4096, 4096, 1),    # single K/V head: runs of rows
    (1, 1, 64, 1, 2049, 300, 1),     # rows that see no key merge into the first chunk
    (1, 3, 32, 1, 8192, 8192, 1),    # B = 3: 2 row runs per entry, not 3
    (1, 7, 32, 8, 2048, 2048, 0),    # B = 7: one run per entry
    (1, 5, 12, 3, 4096, 77, 0),
    (0, 1, 8, 8, 16384, 16384, 0),
    (0, 4, 24, 24, 4096, 4096, 1),
    (0, 1, 6, 2, 8192, 100, 0),
    (1, 1, 1, 1, 1, 1, 0),
    (1, 1, 1, 1, 1, 1, 1),
    (0, 9, 3, 3, 300, 17, 1),
    (1, 2, 64, 64, 3000, 1, 1),      # causal with one key: rows 0..Sq-2 see none
]


def test_dense_plans_on_edge_shapes(driver):
    plans = _run(driver, [("d",) + c for c in DENSE_EDGES])
    for c, p in zip(DENSE_EDGES, plans):
        _check_dense(*c, p)
    counts = {c: len(p) for c, p in zip(DENSE_EDGES, plans)}
    # Split where the work allows, at most 8 chunks.
    assert counts[DENSE_EDGES[0]] == 4
    assert counts[DENSE_EDGES[2]] == 8
    assert counts[DENSE_EDGES[3]] == 2
    assert counts[DENSE_EDGES[5]] == 6
    assert counts[DENSE_EDGES[6]] == 7


def test_dense_plans_on_random_shapes(driver):
    rng = np.random.default_rng(4242)
    heads = [(1, 1), (2, 1), (4, 1), (3, 3), (8, 8), (8, 2), (12, 3), (16, 4), (32, 8), (40, 1),
             (64, 64)]
    cases = []
    while len(cases) < 400:
        Hq, Hkv = heads[rng.integers(len(heads))]
        B = int(rng.choice([1, 1, 2, 3, 5, 7, 8, 9, 13]))
        Sq = int(rng.choice([1, 100, 255, 256, 257, 700, 2048, 2049, 4096, 5000, 8192]))
        Sk = int(rng.choice([1, 17, 300, 2048, 4097]))
        if B * Hq * Sq > 600_000 or B * Hkv * Sk > 600_000:
            continue
        cases.append((int(rng.integers(2)), B, Hq, Hkv, Sq, Sk, int(rng.integers(2))))
    for c, p in zip(cases, _run(driver, [("d",) + c for c in cases])):
        _check_dense(*c, p)


def _check_varlen(B, Hq, cq, chunks):
    sq = np.diff(cq)
    total = int((Hq * -(-sq // 256)).sum())
    want = min(max(total // CTAS_PER_CHUNK, 1), MAX_CHUNKS)
    assert 1 <= len(chunks) <= want
    assert chunks[0][0] == 0 and chunks[-1][1] == B
    for (a0, a1, m), nxt in zip(chunks, chunks[1:] + [None]):
        assert a1 > a0
        assert m == int(sq[a0:a1].max())
        if nxt is not None:
            assert nxt[0] == a1


def test_varlen_plans(driver):
    rng = np.random.default_rng(4343)
    cases = []
    for B in (1, 2, 3, 7, 16, 40, 200):
        for Hq in (1, 8, 32):
            for kind in range(3):
                if kind == 0:
                    lens = rng.integers(1, 9000, B)
                elif kind == 1:
                    lens = rng.integers(0, 3, B) * rng.integers(1, 4000, B)  # some empty
                else:
                    lens = np.full(B, 8192)
                    lens[-1] = 0  # a trailing sequence without queries
                cases.append((B, Hq, np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)))
    plans = _run(driver, [("v", B, Hq, *cq.tolist()) for B, Hq, cq in cases])
    for (B, Hq, cq), p in zip(cases, plans):
        _check_varlen(B, Hq, cq, p)
    # Equal sequences, enough of them: exactly the wanted number of chunks.
    p = _run(driver, [("v", 16, 32, *range(0, 16 * 8192 + 1, 8192))])[0]
    assert len(p) == 8 and all(b1 - b0 == 2 for b0, b1, _ in p)
