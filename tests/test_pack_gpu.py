"""GPU parity of the DCP producer side (mla_dcp_pack, the page's stage_push)
against the oracle: the packed rows and LSE bit for bit, and pack -> combine
against oracle pack -> oracle combine within the stage's tolerance."""
import numpy as np
import pytest
import torch

from parity_util import CANARY, compare, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def bits16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def gpu_pack(inp, dst=None, o_all=None):
    import mla_decode_attention_lse_gb300 as m

    o_all = inp["o_all"] if o_all is None else o_all
    R, S, H = inp["R"], inp["S"], inp["H"]
    dst = inp["dst"] if dst is None else dst
    # canary-filled outputs: every element must be written
    cmb_o = torch.full((R, S, H, 512), 0, dtype=torch.int16, device="cuda").fill_(CANARY).view(torch.bfloat16)
    cmb_lse = torch.full((R, S, H), 1234.5, dtype=torch.float32, device="cuda")
    m.mla_dcp_pack(o_all, inp["lse_all"], inp["seq_lens"], inp["qsl"], inp["q"], dst, cmb_o, cmb_lse)
    torch.cuda.synchronize()
    return cmb_o, cmb_lse


def oracle_pack(orc, inp, dst=None, o_all=None):
    o_all = inp["o_all"] if o_all is None else o_all
    dst = inp["dst"] if dst is None else dst
    o = o_all.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    return orc.dcp_pack(o, inp["lse_all"].cpu().numpy(), inp["seq_lens"].cpu().numpy(),
                        inp["qsl"].cpu().numpy(), inp["q"], dst)


def small(R, S, H, q, live, empty_frac=0.2, seed=0, w_fmt=1):
    from mla_decode_attention_lse_gb300 import synth

    wl = synth.DcpWorkload("t", R=R, S=S, live=live, H=H, q=q, w_fmt=w_fmt, empty_frac=empty_frac, seed=seed)
    return synth.make_dcp(wl, device="cuda")


def check_pack(orc, inp, dst=None, o_all=None):
    cmb_o, cmb_lse = gpu_pack(inp, dst, o_all)
    ref_o, ref_lse = oracle_pack(orc, inp, dst, o_all)
    assert np.array_equal(bits16(cmb_o), ref_o)
    assert np.array_equal(cmb_lse.cpu().numpy().view(np.uint32), ref_lse.view(np.uint32))
    return cmb_o, cmb_lse


@pytest.mark.parametrize("dst", [0, 5, 7])
def test_dcp8_pack_bit_exact(lib, orc, dst):
    from mla_decode_attention_lse_gb300 import synth

    inp = synth.make_dcp("dcp8_mxfp4", device="cuda")
    check_pack(orc, inp, dst)


@pytest.mark.parametrize("R,S,H,q,live", [(1, 4, 3, 1, 4), (2, 6, 3, 2, 5), (3, 33, 2, 3, 30), (4, 1, 1, 1, 0)])
def test_small_packs_bit_exact(lib, orc, R, S, H, q, live):
    inp = small(R, S, H, q, live, seed=R * 100 + S)
    for dst in range(R):
        check_pack(orc, inp, dst)


def test_strided_partials_and_nan_lse(lib, orc):
    # o_all as a view into a wider buffer (extra heads, token stride padded),
    # and a NaN with a payload in a live LSE: copied bit for bit
    inp = small(3, 8, 2, 2, 7, seed=3)
    R, S, RH = 3, 8, 6
    big = torch.zeros(R, S + 1, RH + 3, 512, dtype=torch.bfloat16, device="cuda")
    big[:, :S, 1:RH + 1] = inp["o_all"]
    view = big[:, :S, 1:RH + 1]
    assert not view.is_contiguous()
    lse_bits = inp["lse_all"].view(torch.int32)
    lse_bits[1, 2, 3] = 0x7FC01234
    inp["seq_lens"][1, 1] = 5  # keep that row live
    for dst in range(R):
        check_pack(orc, inp, dst, o_all=view)


@pytest.mark.parametrize("kernel", [0, 2, 3])
def test_pack_then_combine(lib, orc, kernel):
    # destination rank 2 of the DCP8 workload, combined by the library and by
    # the oracle from their own packs
    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    inp = synth.make_dcp("dcp8_mxfp4", device="cuda")
    cmb_o, cmb_lse = gpu_pack(inp, dst=2)
    R, S, H = inp["R"], inp["S"], inp["H"]
    cinp = dict(o=cmb_o, lse=cmb_lse, q=inp["q"], spr=R, w_v=inp["w_v"], w_fmt=inp["w_fmt"],
                w_scale=inp["w_scale"], gate=inp["gate"], S=S, S_out=S, H=H, P=R)
    gpu, canary = run_gpu(cinp, kernel=kernel, tile=16 if kernel == 3 else 0)
    assert np.all(canary == CANARY)
    ref_o, ref_lse = oracle_pack(orc, inp, dst=2)
    ws = None if inp["w_scale"] is None else inp["w_scale"].cpu().numpy()
    ref = orc.Problem(ref_o, ref_lse, inp["q"], R, inp["w_v"].cpu().numpy(), ws, inp["w_fmt"],
                      bits16(inp["gate"])).full()
    # rows past the batch (qsl) and tokens every rank holds nothing of are exactly 0
    zero = np.zeros(ref.shape, bool)
    dead = np.all(np.isneginf(ref_lse), axis=0)  # [S, H]
    for h in range(H):
        zero[dead[:, h], h * 128:(h + 1) * 128] = True
    assert dead[inp["live"]:].all()
    compare(gpu, ref, zero, f"pack -> combine, kernel {kernel}")


def test_pack_errors(lib):
    import mla_decode_attention_lse_gb300 as m

    inp = small(2, 4, 2, 2, 4)
    cmb_o = torch.empty(2, 4, 2, 512, dtype=torch.bfloat16, device="cuda")
    cmb_lse = torch.empty(2, 4, 2, dtype=torch.float32, device="cuda")
    with pytest.raises(m.MlaError) as e:  # no such destination
        m.mla_dcp_pack(inp["o_all"], inp["lse_all"], inp["seq_lens"], inp["qsl"], 2, 2, cmb_o, cmb_lse)
    assert e.value.status == m.MLA_ERR_SHAPE
    flat = torch.empty(2 * 4 * 2 * 512 + 1, dtype=torch.bfloat16, device="cuda")
    odd = flat[1:].view(2, 4, 2, 512)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(m.MlaError) as e:
        m.mla_dcp_pack(inp["o_all"], inp["lse_all"], inp["seq_lens"], inp["qsl"], 2, 0, odd, cmb_lse)
    assert e.value.status == m.MLA_ERR_ALIGN
