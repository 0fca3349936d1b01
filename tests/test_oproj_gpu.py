"""GPU parity of the downstream o_proj shard (mla_o_proj: out = core W^T, the
linear layer that takes the core rows of the vLLM page "vllm.models.kimi_k3.
amd.specialized_decode.mono.attention.mla_back") against the oracle, through
the C ABI.  Tolerance: |gpu - oracle| <= 1e-2 + 1e-2 |oracle| element-wise
(fp32 tensor-core accumulation against double, one bf16 rounding each)."""
import numpy as np
import pytest
import torch

from parity_util import CANARY, bits_to_f32, to_np16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def run(x, w, out_pad=0):
    import mla_decode_attention_lse_gb300 as m

    S, Nout = x.shape[0], w.shape[0]
    big = torch.empty((S, Nout + out_pad), dtype=torch.int16, device="cuda").fill_(CANARY).view(torch.bfloat16)
    out = big[:, :Nout]
    m.mla_o_proj(x, w, out)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    if out_pad:
        assert np.all(to_np16(big[:, Nout:]) == CANARY)  # the padding is untouched
    return out


def check(got, ref, what):
    g, r = bits_to_f32(to_np16(got)), bits_to_f32(ref)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output (an element left unwritten)"
    d = np.abs(g - r)
    bad = d > 1e-2 + 1e-2 * np.abs(r)
    assert not bad.any(), f"{what}: {bad.sum()} out of tolerance, max {d.max()}"


@pytest.mark.parametrize("S,K,Nout", [(1, 64, 64), (5, 128, 192), (64, 1536, 256), (100, 256, 128),
                                      (130, 192, 64), (300, 128, 128), (64, 1536, 7168),
                                      (64, 256, 10240)])  # 160 units: CTAs that run two
def test_oproj_matches_oracle(lib, orc, S, K, Nout):
    g = torch.Generator(device="cuda")
    g.manual_seed(S * 7 + K)
    x = torch.randn((S, K), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((Nout, K), generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    out = run(x, w, out_pad=8 if Nout < 1000 else 0)
    check(out, orc.o_proj(to_np16(x), to_np16(w)), f"S={S} K={K} Nout={Nout}")


def test_oproj_unaligned_output(lib, orc):
    # out's rows start 2 bytes past a 16-byte boundary (base offset by one
    # element, row stride Nout + 8): the output tile is copied element by
    # element; the columns around out stay untouched
    import mla_decode_attention_lse_gb300 as m

    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    S, K, Nout = 70, 256, 192
    x = torch.randn((S, K), generator=g, device="cuda").to(torch.bfloat16)
    w = (torch.randn((Nout, K), generator=g, device="cuda") / K ** 0.5).to(torch.bfloat16)
    big = torch.empty((S, Nout + 9), dtype=torch.int16, device="cuda").fill_(CANARY).view(torch.bfloat16)
    out = big[:, 1:Nout + 1]
    m.mla_o_proj(x, w, out)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    assert np.all(to_np16(big[:, :1]) == CANARY) and np.all(to_np16(big[:, Nout + 1:]) == CANARY)
    check(out, orc.o_proj(to_np16(x), to_np16(w)), "unaligned output")


def test_oproj_strided_rows(lib, orc):
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    xb = torch.randn((40, 200), generator=g, device="cuda").to(torch.bfloat16)
    wb = torch.randn((128, 136), generator=g, device="cuda").to(torch.bfloat16)
    x, w = xb[:, :128], wb[:, :128]
    out = run(x, w, out_pad=3)
    check(out, orc.o_proj(to_np16(x), to_np16(w)), "strided")


def test_attention_combine_oproj_chain(lib, orc):
    # attention -> combine -> o_proj on the GPU against the oracle's chain
    import math

    import mla_decode_attention_lse_gb300 as m
    from parity_util import run_gpu

    from test_attn_gpu import oracle as attn_oracle, problem, run_attn

    inp = problem(2, 2, 4, 3, 200, [200, 50], seed=21)
    o, lse = run_attn(inp)
    o_ref, lse_ref = attn_oracle(orc, inp)
    S, H = inp["B"] * inp["q"], inp["H"]
    g = torch.Generator(device="cuda")
    g.manual_seed(8)
    w_v = (torch.randn((H, 128, 512), generator=g, device="cuda") / math.sqrt(512)).to(torch.bfloat16)
    gate = torch.sigmoid(torch.randn((S, H * 128), generator=g, device="cuda")).to(torch.bfloat16)
    w_o = (torch.randn((256, H * 128), generator=g, device="cuda") / math.sqrt(H * 128)).to(torch.bfloat16)
    core, _ = run_gpu(dict(o=o, lse=lse, q=inp["q"], spr=inp["spr"], w_v=w_v, w_fmt=0, w_scale=None, gate=gate,
                           S=S, S_out=S, H=H, P=inp["spr"]), kernel=0)
    core_t = torch.from_numpy(core.view(np.int16)).view(torch.bfloat16).cuda()
    out = run(core_t.contiguous(), w_o)
    core_ref = orc.Problem(o_ref, lse_ref, inp["q"], inp["spr"], to_np16(w_v), None, 0, to_np16(gate)).full()
    check(out, orc.o_proj(core_ref, to_np16(w_o)), "attention -> combine -> o_proj")


def test_oproj_errors(lib):
    import ctypes

    import mla_decode_attention_lse_gb300 as m

    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((64, 100), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((4, 64), dtype=torch.bfloat16, device="cuda")
    a = m.make_oproj_args(x, w, out)  # K = 100: not a multiple of 64
    assert m.load_library().mla_o_proj(ctypes.byref(a), None) == m.MLA_ERR_SHAPE
