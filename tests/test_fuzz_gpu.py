"""Seeded fuzzing of the C ABI on the GPU against the oracle: random sizes,
split layouts, W_V formats, kernel choices, strided views and dead / NaN
partials; every output element checked (tolerance as in the parity tests),
rows the definition zeroes exactly zero, rows past S_out untouched.  And the
DCP pack on random shapes, bit for bit."""
import numpy as np
import pytest
import torch

from parity_util import CANARY, compare, oracle_problem, run_gpu, seg_mask

pytestmark = pytest.mark.gpu

SIMT, TC, KS = 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def draw_case(rng):
    """One random problem description."""
    layout = rng.choice(["pass", "compact", "request_major"])
    q = int(rng.choice([1, 2, 3]))
    requests = int(rng.integers(1, 24))
    S = requests * q
    H = int(rng.integers(1, 6))
    if layout == "pass":
        P, spr = 1, 0
    elif layout == "compact":
        spr = int(rng.integers(2, 17))
        P = spr
    else:
        spr = int(rng.integers(2, 9))
        P = requests * spr
    S_out = S + int(rng.integers(0, 5))
    w_fmt = int(rng.integers(0, 2))
    n = 1 if layout == "pass" else spr
    kernels = [0, SIMT, TC] + ([KS] if n <= 16 else [])
    kernel = int(rng.choice(kernels))
    tile = int(rng.choice([0, 16, 32])) if kernel == TC and n <= 16 else (16 if kernel in (TC, KS) else 0)
    return dict(layout=layout, q=q, S=S, S_out=S_out, H=H, P=P, spr=spr, w_fmt=w_fmt, kernel=kernel, tile=tile,
                neg_inf=float(rng.choice([0.0, 0.1, 0.4])), nan=float(rng.choice([0.0, 0.05])),
                strided=bool(rng.integers(0, 2)), seed=int(rng.integers(0, 1 << 30)))


def make_case(c):
    from mla_decode_attention_lse_gb300 import synth

    inp = synth.custom(S=c["S"], S_out=c["S_out"], H=c["H"], P=c["P"], q=c["q"], spr=c["spr"], w_fmt=c["w_fmt"],
                       seed=c["seed"], device="cuda", neg_inf_frac=0.0 if c["layout"] == "pass" else c["neg_inf"],
                       nan_frac=0.0 if c["layout"] == "pass" else c["nan"], lse_unused=c["layout"] == "pass")
    if c["strided"]:
        # o as a slice of a wider tensor (extra heads, padded token stride)
        P, S, H = c["P"], c["S"], c["H"]
        big = torch.full((P, S + 1, H + 2, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        big[:, :S, 1:H + 1] = inp["o"]
        inp["o"] = big[:, :S, 1:H + 1]
    if inp["lse"] is not None:
        # dead partials' rows poisoned: they must never be read
        dead = ~torch.isfinite(inp["lse"])
        inp["o"][dead] = float("nan")
    return inp


@pytest.mark.parametrize("case", range(40))
def test_fuzz_combine(lib, orc, case):
    rng = np.random.default_rng(1000 + case)
    c = draw_case(rng)
    inp = make_case(c)
    gpu, canary = run_gpu(inp, kernel=c["kernel"], tile=c["tile"])
    assert np.all(canary == CANARY), c
    ref = oracle_problem(orc, inp).full()
    compare(gpu, ref, seg_mask(inp), f"fuzz {case}: {c}")


@pytest.mark.parametrize("case", range(16))
def test_fuzz_combine_eight_token_tiles(lib, orc, case):
    # the half-row instance (two warps per token) on random problems
    rng = np.random.default_rng(3000 + case)
    c = draw_case(rng)  # at most 16 partials per token
    c["kernel"], c["tile"] = TC, 8
    inp = make_case(c)
    gpu, canary = run_gpu(inp, kernel=TC, tile=8)
    assert np.all(canary == CANARY), c
    ref = oracle_problem(orc, inp).full()
    compare(gpu, ref, seg_mask(inp), f"fuzz 8-token tiles {case}: {c}")


@pytest.mark.parametrize("case", range(12))
def test_fuzz_pack(lib, orc, case):
    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    rng = np.random.default_rng(2000 + case)
    R, H, q = int(rng.integers(1, 9)), int(rng.integers(1, 13)), int(rng.choice([1, 2, 4]))
    S = int(rng.integers(0, 20)) * q
    live = int(rng.integers(0, S + 1))
    wl = synth.DcpWorkload("fuzz", R=R, S=S, live=live, H=H, q=q, w_fmt=1, empty_frac=float(rng.choice([0, 0.3])),
                           seed=int(rng.integers(0, 1 << 30)))
    d = synth.make_dcp(wl, device="cuda")
    dst = int(rng.integers(0, R))
    cmb_o = torch.full((R, S, H, 512), 0, dtype=torch.int16, device="cuda").fill_(CANARY).view(torch.bfloat16)
    cmb_lse = torch.full((R, S, H), 7.0, dtype=torch.float32, device="cuda")
    m.mla_dcp_pack(d["o_all"], d["lse_all"], d["seq_lens"], d["qsl"], q, dst, cmb_o, cmb_lse)
    torch.cuda.synchronize()
    ref_o, ref_lse = orc.dcp_pack(d["o_all"].cpu().view(torch.int16).numpy().view(np.uint16),
                                  d["lse_all"].cpu().numpy(), d["seq_lens"].cpu().numpy(), d["qsl"].cpu().numpy(),
                                  q, dst)
    assert np.array_equal(cmb_o.cpu().view(torch.int16).numpy().view(np.uint16), ref_o)
    assert np.array_equal(cmb_lse.cpu().numpy().view(np.uint32), ref_lse.view(np.uint32))
