"""GPU parity of the partial producer (mla_attn_split_kv: split-KV MLA decode
attention, the M1c producer named on the vLLM page "vllm.models.kimi_k3.amd.
specialized_decode.mono.attention.mla_back") against the oracle, through the
C ABI.

Tolerance: o (bf16) |gpu - oracle| <= 1e-2 + 1e-2 |oracle| element-wise (the
stage's bar; the kernel's softmax weights enter the latent sum as bf16, the
oracle works in double); lse |gpu - oracle| <= 1e-3 + 1e-4 |oracle| (fp32
tensor-core scores, hardware exp2 / log2).  A split the token sees nothing
of is exact: lse -inf and o 0.  Every output element is written (canary
check)."""
import math

import numpy as np
import pytest
import torch

from parity_util import CANARY, bits_to_f32, compare, run_gpu, to_np16

pytestmark = pytest.mark.gpu

D, K = 512, 576


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def problem(B, q, H, spr, Lmax, lens, seed=0, kv_pad=0, q_pad=0):
    """Random inputs; cached rows past a request's length are NaN. kv_pad /
    q_pad widen the row strides (strided views)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    S = B * q
    qbig = torch.randn((S, H + q_pad, K), generator=g, device="cuda").to(torch.bfloat16)
    qv = qbig[:, :H]
    kvbig = torch.randn((B, Lmax, K + kv_pad), generator=g, device="cuda").to(torch.bfloat16)
    kv = kvbig[:, :, :K]
    kv_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for b, L in enumerate(lens):
        kv[b, L:] = float("nan")
    return dict(qv=qv, kv=kv, kv_len=kv_len, q=q, spr=spr, scale=1 / math.sqrt(192), B=B, H=H, Lmax=Lmax)


def run_attn(inp, kernel=0):
    import mla_decode_attention_lse_gb300 as m

    S = inp["B"] * inp["q"]
    o = torch.empty((inp["spr"], S, inp["H"], D), dtype=torch.int16, device="cuda").fill_(CANARY)
    o = o.view(torch.bfloat16)
    lse = torch.full((inp["spr"], S, inp["H"]), 1234.5, dtype=torch.float32, device="cuda")
    m.mla_attn_split_kv(inp["qv"], inp["kv"], inp["kv_len"], inp["q"], inp["spr"], inp["scale"], o, lse,
                        kernel=kernel)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    return o, lse


def oracle(orc, inp, reqs=None):
    q = inp["q"]
    qv, kv, kv_len = inp["qv"], inp["kv"], inp["kv_len"]
    if reqs is not None:  # a subset of the requests, as a smaller batch
        idx = torch.tensor(reqs, device=qv.device)
        rows = (idx[:, None] * q + torch.arange(q, device=qv.device)[None]).reshape(-1)
        qv, kv, kv_len = qv[rows], kv[idx], kv_len[idx]
    return orc.mla_attn_split(to_np16(qv), to_np16(kv), kv_len.cpu().numpy(), q, inp["spr"], inp["scale"])


def check(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    og = bits_to_f32(to_np16(o_gpu))
    orf = bits_to_f32(o_ref)
    lg = lse_gpu.cpu().numpy()
    dead = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), dead), f"{what}: -inf pattern"
    assert np.all(og[dead] == 0), f"{what}: empty split not zero"
    live = ~dead
    err = np.abs(lg[live] - lse_ref[live])
    assert np.all(err <= 1e-3 + 1e-4 * np.abs(lse_ref[live])), f"{what}: lse max err {err.max()}"
    assert np.all(np.isfinite(og)), f"{what}: non-finite o (or an element left unwritten)"
    d = np.abs(og - orf)
    bad = d > 1e-2 + 1e-2 * np.abs(orf)
    assert not bad.any(), f"{what}: {bad.sum()} o elements out of tolerance, max {d.max()}"


@pytest.mark.parametrize("B,q,H,spr,Lmax,lens", [
    (3, 1, 12, 4, 300, [300, 129, 5]),            # N = 16, all heads in one CTA; an empty split
    (4, 2, 3, 3, 260, [128, 256, 1, 0]),          # q = 2 causal; kv_len 0: every split empty
    (2, 4, 16, 2, 200, [200, 77]),                # q H = 64: two head groups of 8 (N = 32)
    (2, 3, 5, 2, 64, [64, 9]),                    # q G = 15 (one padded row)
    (1, 1, 1, 1, 1000, [1000]),                   # one split of 8 tiles: the slot rings wrap
    (6, 1, 12, 1, 257, [127, 128, 129, 255, 256, 257]),  # tile boundaries
])
@pytest.mark.parametrize("kernel", [1, 2])  # one CTA per item; a 2-CTA cluster per item
def test_attn_matches_oracle(lib, orc, B, q, H, spr, Lmax, lens, kernel):
    inp = problem(B, q, H, spr, Lmax, lens, seed=B * 100 + q)
    o, lse = run_attn(inp, kernel)
    o_ref, lse_ref = oracle(orc, inp)
    check(o, lse, o_ref, lse_ref, f"kernel {kernel}: B={B} q={q} H={H} spr={spr} lens={lens}")


@pytest.mark.parametrize("kernel", [1, 2])
def test_attn_strided_views(lib, orc, kernel):
    inp = problem(3, 2, 6, 3, 150, [150, 64, 3], seed=7, kv_pad=64, q_pad=2)
    assert not inp["qv"].is_contiguous() and not inp["kv"].is_contiguous()
    o, lse = run_attn(inp, kernel)
    o_ref, lse_ref = oracle(orc, inp)
    check(o, lse, o_ref, lse_ref, f"strided, kernel {kernel}")


@pytest.mark.parametrize("kernel", [1, 2])
def test_attn_full_workload_sampled(lib, orc, kernel):
    # the bench's decode step (64 requests x 12 heads, 16 splits, up to 4096
    # cached positions), checked on a sample of requests
    from mla_decode_attention_lse_gb300 import synth

    inp = synth.make_attn("attn_splitkv", device="cuda")
    o, lse = run_attn(inp, kernel)
    lens = inp["kv_len"].cpu().numpy()
    reqs = [int(np.argmax(lens)), int(np.argmin(lens)), 0, 17, 63]
    o_ref, lse_ref = oracle(orc, inp, reqs)
    q = inp["q"]
    rows = [b * q + i for b in reqs for i in range(q)]
    check(o[:, rows], lse[:, rows], o_ref, lse_ref, "attn_splitkv sample")


def test_attn_then_combine(lib, orc):
    # producer -> combine on the GPU against oracle producer -> oracle combine
    inp = problem(4, 2, 3, 4, 300, [300, 37, 2, 180], seed=11)
    o, lse = run_attn(inp)
    o_ref, lse_ref = oracle(orc, inp)
    S, H = inp["B"] * inp["q"], inp["H"]
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    w_v = (torch.randn((H, 128, D), generator=g, device="cuda") / math.sqrt(D)).to(torch.bfloat16)
    gate = torch.sigmoid(torch.randn((S, H * 128), generator=g, device="cuda")).to(torch.bfloat16)
    cinp = dict(o=o, lse=lse, q=inp["q"], spr=inp["spr"], w_v=w_v, w_fmt=0, w_scale=None, gate=gate, S=S, S_out=S,
                H=H, P=inp["spr"])
    gpu, canary = run_gpu(cinp, kernel=0)
    assert np.all(canary == CANARY)
    ref = orc.Problem(o_ref, lse_ref, inp["q"], inp["spr"], to_np16(w_v), None, 0, to_np16(gate)).full()
    zero = np.zeros(ref.shape, bool)
    dead = np.all(np.isneginf(lse_ref), axis=0)  # [S, H]: the token sees nothing at all
    for h in range(H):
        zero[dead[:, h], h * 128:(h + 1) * 128] = True
    compare(gpu, ref, zero, "attention -> combine")


def test_attn_kv_len_out_of_range_is_reported(lib, orc):
    import mla_decode_attention_lse_gb300 as m

    inp = problem(2, 1, 2, 2, 64, [64, 10], seed=3)
    inp["kv_len"][1] = 65  # past Lmax: clamped to Lmax, reported
    S = inp["B"] * inp["q"]
    o = torch.empty((2, S, 2, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, S, 2), dtype=torch.float32, device="cuda")
    m.mla_attn_split_kv(inp["qv"], inp["kv"], inp["kv_len"], 1, 2, inp["scale"], o, lse)
    assert m.mla_combine_uv_status() == m.MLA_ERR_DATA
    assert m.mla_combine_uv_status() == m.MLA_OK  # read and cleared


def test_attn_errors(lib):
    import mla_decode_attention_lse_gb300 as m

    inp = problem(2, 1, 2, 2, 64, [64, 10])
    S = 2
    o = torch.empty((2, S, 2, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, S, 2), dtype=torch.float32, device="cuda")
    import ctypes

    a = m.make_attn_args(inp["qv"], inp["kv"], inp["kv_len"], 33, 2, 0.1, o, lse)  # q > 32
    assert m.load_library().mla_attn_split_kv(ctypes.byref(a), None) == m.MLA_ERR_SHAPE
    a = m.make_attn_args(inp["qv"], inp["kv"], inp["kv_len"], 1, 2, 0.1, o, lse, kernel=3)
    assert m.load_library().mla_attn_split_kv(ctypes.byref(a), None) == m.MLA_ERR_KERNEL
    flat = torch.empty(2 * 64 * K + 8, dtype=torch.bfloat16, device="cuda")
    odd = flat[1:1 + 2 * 64 * K].view(2, 64, K)  # 2-byte offset
    with pytest.raises(m.MlaError) as e:
        m.mla_attn_split_kv(inp["qv"], odd, inp["kv_len"], 1, 2, 0.1, o, lse)
    assert e.value.status == m.MLA_ERR_ALIGN


@pytest.mark.parametrize("case", range(24))
def test_attn_fuzz(lib, orc, case):
    # seeded random shapes: queries per request, heads (one or several head
    # groups), splits, lengths (empty, short, tile edges, long), strided views
    rng = np.random.default_rng(3000 + case)
    q = int(rng.choice([1, 1, 2, 3, 4, 8]))
    H = int(rng.integers(1, 25))
    B = int(rng.integers(1, 6))
    spr = int(rng.choice([1, 2, 3, 5, 16, 20]))
    Lmax = int(rng.choice([16, 64, 129, 300, 700]))
    lens = [int(rng.choice([0, 1, q, int(rng.integers(1, Lmax + 1)), Lmax])) for _ in range(B)]
    lens = [min(L, Lmax) for L in lens]
    inp = problem(B, q, H, spr, Lmax, lens, seed=case, kv_pad=int(rng.choice([0, 8, 64])),
                  q_pad=int(rng.choice([0, 1])))
    kernel = 1 + case % 2  # both kernels
    o, lse = run_attn(inp, kernel)
    o_ref, lse_ref = oracle(orc, inp)
    check(o, lse, o_ref, lse_ref, f"fuzz {case} (kernel {kernel}): B={B} q={q} H={H} spr={spr} Lmax={Lmax} lens={lens}")
