"""The launches are plain kernel launches on the caller's stream, so a CUDA graph
can capture them: replaying the graph on new inputs gives the same bits as
calling directly."""
import pytest
import torch

import bf16_forward_attention_gb300 as attn
from bf16_forward_attention_gb300 import build, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    build.build()
    attn.load_library()


def _qkv(seed, Sq=300, Sk=2000, Hq=4, Hkv=2):
    q, _, _ = inputs.make_qkv(inputs.Workload("g", "bshd", 2, Hq, Sq, Sk, seed=seed))
    _, k, v = inputs.make_qkv(inputs.Workload("g", "bshd", 2, Hkv, Sq, Sk, seed=seed + 1))
    return q.cuda(), k.cuda(), v.cuda()


def test_graph_replay_equals_direct_calls():
    q, k, v = _qkv(1500)
    out_ex = torch.empty_like(q)
    qs, ks, vs = (t.clone() for t in (q, k, v))
    s = 4
    ws = torch.empty(attn.splitkv_workspace_bytes(2, 4, 300, 2000, s), dtype=torch.uint8,
                     device="cuda")
    ks_full = ks.repeat_interleave(2, dim=2).contiguous()
    vs_full = vs.repeat_interleave(2, dim=2).contiguous()
    out_split = torch.empty_like(q)

    def step():
        attn.attn_fwd_ex(qs, ks, vs, causal=True, layout="bshd", out=out_ex)
        attn.attn_fwd_splitkv(qs, ks_full, vs_full, num_splits=s, layout="bshd", out=out_split,
                              workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (library setup, tensor-map encoder)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (1510, 1520):
        q2, k2, v2 = _qkv(seed)
        qs.copy_(q2)
        ks.copy_(k2)
        vs.copy_(v2)
        ks_full.copy_(k2.repeat_interleave(2, dim=2))
        vs_full.copy_(v2.repeat_interleave(2, dim=2))
        graph.replay()
        torch.cuda.synchronize()
        want_ex = attn.attn_fwd_ex(q2, k2, v2, causal=True, layout="bshd")
        want_split = attn.attn_fwd_splitkv(q2, k2.repeat_interleave(2, dim=2).contiguous(),
                                           v2.repeat_interleave(2, dim=2).contiguous(),
                                           num_splits=s, layout="bshd")
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        assert torch.equal(out_ex.view(torch.int16), want_ex.view(torch.int16))
        assert torch.equal(out_split.view(torch.int16), want_split.view(torch.int16))


def test_graph_replay_of_the_tail_split():
    # ATTN_FLAG_SPLIT_TAIL: the full waves, then the tail items as 2-CTA clusters
    # launched as a programmatic dependent of the full waves; and a call that is
    # all pairs (one launch). Both captured in one graph and replayed.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    shapes = [(sms + 5, 256, 2100), (4, 256, 2100)]
    assert [attn.split_tail_items(1, h, sq, sk) for h, sq, sk in shapes] == [5, 4]

    def make(seed):
        out = []
        for i, (h, sq, sk) in enumerate(shapes):
            q, k, v = inputs.make_qkv(inputs.Workload("gt", "bhsd", 1, h, sq, sk, seed=seed + i))
            out.append((q.cuda(), k.cuda(), v.cuda()))
        return out

    bufs = [tuple(t.clone() for t in qkv) for qkv in make(1600)]
    outs = [torch.empty_like(qkv[0]) for qkv in bufs]

    def step():
        for (q, k, v), o in zip(bufs, outs):
            attn.attn_fwd_ex(q, k, v, layout="bhsd", out=o, split_tail=True)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (1610, 1620):
        fresh = make(seed)
        for dst, src in zip(bufs, fresh):
            for d, s_ in zip(dst, src):
                d.copy_(s_)
        graph.replay()
        torch.cuda.synchronize()
        wants = [attn.attn_fwd_ex(q, k, v, layout="bhsd", split_tail=True) for q, k, v in fresh]
        torch.cuda.synchronize()
        assert attn.attn_fwd_last_error() == attn.ATTN_OK
        for o, want in zip(outs, wants):
            assert torch.equal(o.view(torch.int16), want.view(torch.int16))
