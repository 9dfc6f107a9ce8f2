"""Failure detection on the GPU without a fault: a launch whose own device-side
wait runs out (one internal signal withheld, 20 ms limit) must stop cleanly,
report ATTN_ERR_TIMEOUT through attn_fwd_last_error, leave the output alone and
leave the context usable for the next call."""
import time

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


# Sk = 1000 (8 key tiles, 2 items) with the tail split runs the pair variant:
# both CTAs of each cluster give up, skip the exchange and meet at the end.
@pytest.mark.parametrize("Sk,flags", [(200, 0), (1000, 0), (1000, attn.ATTN_FLAG_SPLIT_TAIL)])
def test_withheld_signal_times_out_cleanly(Sk, flags):
    w = inputs.Workload("fail", "bhsd", 1, 2, 256, Sk, seed=90)
    q, k, v = inputs.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.full_like(qd, 7.0)
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    stream = torch.cuda.current_stream().cuda_stream
    t0 = time.time()
    st = attn.attn_fwd_timeout_selftest_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                            out.data_ptr(), 0, 1, 2, 256, Sk, 128,
                                            inputs.default_scale(), 0, stream, 20_000_000, flags)
    assert st == attn.ATTN_OK
    torch.cuda.synchronize()
    assert time.time() - t0 < 10.0
    assert attn.attn_fwd_last_error() == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_fwd_last_error() == attn.ATTN_OK  # reading clears it
    assert bool((out == 7.0).all())                    # nothing was stored

    # The context still works: a normal call right after is correct.
    res = attn.attn_fwd(qd, kd, vd, layout="bhsd")
    torch.cuda.synchronize()
    assert attn.attn_fwd_last_error() == attn.ATTN_OK
    exact = attention_fp64(f64_of(q), f64_of(k), f64_of(v), inputs.default_scale(), "bhsd")
    assert_parity(compare(bits_of(res), exact, "rtne"))
