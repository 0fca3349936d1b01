"""The failure path of the tensor-core combine kernel, run on the GPU.

Every wait of the kernel is bounded.  The caller can hand the call a device
ready flag (the producer's completion flag of the page's flag handshake) and
a wait limit.  Here the flag stays zero -- nothing ever raises it -- so every
CTA's wait for it runs out after the short limit: the kernel must record
MLA_ERR_TIMEOUT in the device error word, drain the weight copies it started,
free its TMEM and return.  The host reads and clears the status, and the next
call must be exact against the oracle.  No wait here is endless: the limit
ends it.
"""
import numpy as np
import pytest
import torch

from parity_util import CANARY, compare, oracle_problem, run_gpu, seg_mask

pytestmark = pytest.mark.gpu

TC = 2


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def _call(inp, out, wait_ns, tile, flag=None):
    import mla_decode_attention_lse_gb300 as m

    m.mla_combine_uv(inp["o"], inp["lse"], inp["q"], inp["spr"], inp["w_v"], inp["w_fmt"],
                     inp["gate"], out, w_scale=inp["w_scale"], kernel=TC, tile_tokens=tile,
                     wait_ns=wait_ns, ready_flag=flag)


def _problem(w_fmt):
    from mla_decode_attention_lse_gb300 import synth

    return synth.custom(S=512, H=12, P=4, q=1, spr=4, w_fmt=w_fmt, neg_inf_frac=0.05, seed=40 + w_fmt,
                        device="cuda")


@pytest.mark.parametrize("w_fmt,tile", [(0, 32), (1, 32), (1, 16), (0, 8)])
def test_flag_never_raised_times_out_then_recovers(lib, orc, w_fmt, tile):
    import mla_decode_attention_lse_gb300 as m

    inp = _problem(w_fmt)
    out = torch.empty(inp["S_out"], inp["H"] * 128, dtype=torch.bfloat16, device="cuda")
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    ref = oracle_problem(orc, inp).full()
    for attempt in range(2):
        flag.zero_()
        _call(inp, out, 2_000_000, tile, flag)  # 2 ms; nothing raises the flag
        assert m.mla_combine_uv_status(stream) == m.MLA_ERR_TIMEOUT
        assert m.mla_combine_uv_status(stream) == m.MLA_OK  # cleared by the read
        # the kernel returned and freed its TMEM: the next calls allocate it
        # again and are exact, with the flag raised and without one
        flag.fill_(1)
        _call(inp, out, 0, tile, flag)
        assert m.mla_combine_uv_status(stream) == m.MLA_OK
        got = out.cpu().view(torch.int16).numpy().view(np.uint16)
        compare(got, ref, seg_mask(inp), f"flag raised, attempt {attempt}")
        gpu, canary = run_gpu(inp, kernel=TC, tile=tile)
        assert np.all(canary == CANARY)
        compare(gpu, ref, seg_mask(inp), f"after a timeout, attempt {attempt}")


@pytest.mark.parametrize("w_fmt,tile", [(0, 32), (1, 16)])
def test_short_wait_limit_is_safe(lib, orc, w_fmt, tile):
    """A 1 ns limit on the waits for the W_UV MMAs: the hardware's suspending
    wait usually covers an MMA that is about to land, so a call may finish
    normally; either way it returns a defined status, and the next default
    call is exact."""
    import mla_decode_attention_lse_gb300 as m

    inp = _problem(w_fmt)
    out = torch.empty(inp["S_out"], inp["H"] * 128, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    ref = oracle_problem(orc, inp).full()
    for _ in range(4):
        _call(inp, out, 1, tile)
        assert m.mla_combine_uv_status(stream) in (m.MLA_OK, m.MLA_ERR_TIMEOUT)
        assert m.mla_combine_uv_status(stream) == m.MLA_OK
    gpu, canary = run_gpu(inp, kernel=TC, tile=tile)
    assert np.all(canary == CANARY)
    compare(gpu, ref, seg_mask(inp), "after 1 ns limits")


def test_flag_needs_the_tensor_core_kernel(lib):
    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    inp = synth.custom(S=16, H=2, P=2, q=1, spr=2, w_fmt=0, seed=3, device="cuda")
    out = torch.empty(16, 256, dtype=torch.bfloat16, device="cuda")
    flag = torch.ones(1, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MlaError) as e:
        m.mla_combine_uv(inp["o"], inp["lse"], 1, 2, inp["w_v"], 0, inp["gate"], out, kernel=1,
                         ready_flag=flag)
    assert e.value.status == m.MLA_ERR_KERNEL


def test_negative_wait_limit_is_rejected(lib):
    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    inp = synth.custom(S=16, H=2, P=2, q=1, spr=2, w_fmt=0, seed=3, device="cuda")
    out = torch.empty(16, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MlaError) as e:
        _call(inp, out, -5, 16)
    assert e.value.status == m.MLA_ERR_SHAPE
