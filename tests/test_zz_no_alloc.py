"""The allocation-free decode step (mla_attn_combine_uv_noalloc) on the GPU.

Some callers cannot allocate device memory at the point where they run the
decode step -- a serving engine that gave nearly all free device memory to its
KV cache at start-up, or a decode loop that cannot afford the device-wide
synchronisation an allocation can cause.  For them the library keeps the
step's scratch in a fixed device buffer of its own.  This file checks, through
the C ABI, that such a call gives the same core rows as mla_attn_combine_uv
with caller-owned scratch (within the stage's tolerance), twice in a row and
after a call of another shape has left its data in the shared buffer; and
that a problem too big for the buffer is refused with MLA_ERR_SCRATCH.

Its name makes pytest collect it last, so a run that stops at the first
failure has run every other test before it.  It also runs alone in a fresh
process (the first call there does the buffer's set-up).
"""
import math

import pytest
import torch

from parity_util import compare, to_np16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def _small(seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    B, q, H, spr, Lmax = 5, 3, 5, 5, 150
    S = B * q
    qv = torch.randn((S, H, 576), generator=g, device="cuda").to(torch.bfloat16)
    kv = torch.randn((B, Lmax, 576), generator=g, device="cuda").to(torch.bfloat16)
    kv_len = torch.tensor([150, 9, 64, 0, 149], dtype=torch.int32, device="cuda")
    w_v = (torch.randn((H, 128, 512), generator=g, device="cuda") / math.sqrt(512)).to(torch.bfloat16)
    gate = torch.sigmoid(torch.randn((S, H * 128), generator=g, device="cuda")).to(torch.bfloat16)
    return dict(qv=qv, kv=kv, kv_len=kv_len, q=q, spr=spr, scale=1 / math.sqrt(192), B=B, H=H, w_v=w_v, gate=gate)


def _decode_step():
    from mla_decode_attention_lse_gb300 import synth

    a = synth.make_attn("attn_splitkv", device="cuda")
    return dict(qv=a["qv"], kv=a["kv"], kv_len=a["kv_len"], q=a["q"], spr=a["spr"], scale=a["scale"], B=a["B"],
                H=a["H"], w_v=a["w_v"], gate=a["gate"])


def _with_caller_scratch(inp):
    import mla_decode_attention_lse_gb300 as m

    B, q, H, spr = inp["B"], inp["q"], inp["H"], inp["spr"]
    S = B * q
    po = torch.empty((spr, S, H, 512), dtype=torch.bfloat16, device="cuda")
    pl = torch.empty((spr, S, H), dtype=torch.float32, device="cuda")
    ws = torch.zeros(m.mla_attn_combine_uv_workspace_words(B, q), dtype=torch.int32, device="cuda")
    out = torch.empty((S, H * 128), dtype=torch.bfloat16, device="cuda")
    m.mla_attn_combine_uv(inp["qv"], inp["kv"], inp["kv_len"], q, spr, inp["scale"], po, pl, inp["w_v"],
                          inp["gate"], out, ws)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    return to_np16(out)


def _without_allocation(inp):
    import mla_decode_attention_lse_gb300 as m

    S, H = inp["B"] * inp["q"], inp["H"]
    out = torch.empty((S, H * 128), dtype=torch.bfloat16, device="cuda")
    m.mla_attn_combine_uv_noalloc(inp["qv"], inp["kv"], inp["kv_len"], inp["q"], inp["spr"], inp["scale"],
                                  inp["w_v"], inp["gate"], out)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    return to_np16(out)


def test_no_alloc_step_matches_the_step_with_caller_scratch(lib):
    big = _decode_step()
    ref_big = _with_caller_scratch(big)
    for call in range(2):  # two calls in a row on the shared buffer
        got = _without_allocation(big)
        compare(got, ref_big, None, f"decode step without allocation, call {call}")
    small = _small(7)
    ref_small = _with_caller_scratch(small)
    for call in range(2):  # another shape, over the decode step's leftovers
        got = _without_allocation(small)
        compare(got, ref_small, None, f"small step without allocation, call {call}")
    got = _without_allocation(big)
    compare(got, ref_big, None, "decode step again")


def test_no_alloc_step_refuses_a_problem_bigger_than_its_buffer(lib):
    import mla_decode_attention_lse_gb300 as m

    # a batch whose partials (32 splits x 4096 tokens x 16 heads) need ~2 GB
    B, q, H, spr = 1024, 4, 16, 32
    qv = torch.empty((B * q, H, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((B, 16, 576), dtype=torch.bfloat16, device="cuda")
    kv_len = torch.zeros(B, dtype=torch.int32, device="cuda")
    w_v = torch.zeros((H, 128, 512), dtype=torch.bfloat16, device="cuda")
    gate = torch.zeros((B * q, H * 128), dtype=torch.bfloat16, device="cuda")
    out = torch.full((B * q, H * 128), 3, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MlaError) as e:
        m.mla_attn_combine_uv_noalloc(qv, kv, kv_len, q, spr, 0.07, w_v, gate, out)
    assert e.value.status == m.MLA_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.all(out == 3)  # nothing was launched
