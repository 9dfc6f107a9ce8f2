"""attn_fwd_splitkv_noalloc: split-KV whose workspace is the library's fixed device
scratch array, for callers that cannot allocate device memory when they need
attention (a framework pool that owns all allocations, a serving loop that must
not call cudaMalloc/cudaFree after start-up). Called through the C ABI and
compared bit for bit with attn_fwd_splitkv (caller-provided workspace, same
split count) on two calls in a row, since every call reuses the same scratch,
after another problem has left its own contents there, and against the fp64
oracle. This file is collected last."""
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs
import numpy as np

from oracle import attention_fp64

from _parity import assert_parity, bits_of, compare, f64_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _noalloc(q, k, v, out, layout, splits, mode=0):
    B, H, Sq, D = attn._dims(q, layout)
    Sk = attn._dims(k, layout)[2]
    return attn.attn_fwd_splitkv_noalloc_raw(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), attn.LAYOUTS[layout], B, H, Sq,
        Sk, D, inputs.default_scale(), mode, splits, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("layout,B,H,Sq,Sk,splits", [
    ("bshd", 1, 8, 256, 32768, None),   # decode-like; split count from the helper
    ("bhsd", 2, 3, 300, 2049, 7),
])
def test_noalloc_matches_workspace_entry_point_twice(layout, B, H, Sq, Sk, splits):
    w = inputs.Workload("noalloc", layout, B, H, Sq, Sk, seed=700 + Sk)
    q, k, v = (t.cuda() for t in inputs.make_qkv(w))
    if splits is None:
        splits = attn.splitkv_num_splits(B, H, Sq, Sk)
    assert splits > 1
    ref = attn.attn_fwd_splitkv(q, k, v, num_splits=splits, layout=layout)
    torch.cuda.synchronize()
    want = bits_of(ref)
    # The same kernels with the same split count run in a fixed order, so the
    # two entry points must agree bit for bit.
    for _ in range(2):  # the second call runs over the first call's scratch contents
        out = torch.full_like(q, float("nan"))
        assert _noalloc(q, k, v, out, layout, splits) == attn.ATTN_OK
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        assert np.array_equal(bits_of(out), want)
    # And both against the fp64 oracle, element by element.
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), layout)
    assert_parity(compare(want, exact, "rtne"), excess=Sk < 4096)


def test_noalloc_scratch_left_by_another_problem():
    # Problem A, then problem B (other inputs, more splits, more heads: it writes
    # scratch that A's layout reads) on the same stream, then A again: the stale
    # contents B left must not leak into A's result.
    layout = "bhsd"
    wa = inputs.Workload("noalloc_a", layout, 1, 4, 260, 3000, seed=811)
    wb = inputs.Workload("noalloc_b", layout, 1, 6, 500, 4100, seed=812)
    qa, ka, va = (t.cuda() for t in inputs.make_qkv(wa))
    qb, kb, vb = (t.cuda() for t in inputs.make_qkv(wb))
    sa, sb = 3, 11
    need_b = attn.splitkv_workspace_bytes(1, 6, 500, 4100, sb)
    assert attn.splitkv_workspace_bytes(1, 4, 260, 3000, sa) < need_b <= 32 << 20
    want_a = bits_of(attn.attn_fwd_splitkv(qa, ka, va, num_splits=sa, layout=layout))
    want_b = bits_of(attn.attn_fwd_splitkv(qb, kb, vb, num_splits=sb, layout=layout))
    outs = []
    for (q, k, v, s) in [(qa, ka, va, sa), (qb, kb, vb, sb), (qa, ka, va, sa)]:
        out = torch.full_like(q, float("nan"))
        assert _noalloc(q, k, v, out, layout, s) == attn.ATTN_OK
        outs.append(out)
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    assert np.array_equal(bits_of(outs[0]), want_a)
    assert np.array_equal(bits_of(outs[1]), want_b)
    assert np.array_equal(bits_of(outs[2]), want_a)


def test_noalloc_rejects_problems_beyond_the_scratch():
    # Real buffers of the stated sizes; the call must refuse before launching.
    B, H, Sq, Sk, splits = 1, 16, 2048, 4096, 32
    assert attn.splitkv_workspace_bytes(B, H, Sq, Sk, splits) > 32 << 20
    q = torch.zeros(B, H, Sq, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, H, Sk, 128, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    out = torch.full_like(q, 3.0)
    assert _noalloc(q, k, v, out, "bhsd", splits) == attn.ATTN_ERR_SCRATCH
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
