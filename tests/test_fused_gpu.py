"""GPU parity of the decode step in one launch (mla_attn_combine_uv: the split-KV
attention and the combine of its partials, as the vLLM page
"vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back" pairs
M1c's partials with the combine) against the oracle chain -- the oracle's
attention, then the oracle's combine on its partials -- through the C ABI.

The fused launch's combine units compute every output exactly as
mla_combine_uv does on the same partials (same weights, same merge, same GEMM
shape), so its core is compared bit for bit with mla_combine_uv run on the
partials the launch wrote.  (Its attention tiles hold 128 positions; the
standalone attention with up to 16 query rows tiles by 64, so the two
attentions' partials agree within rounding, not bit for bit: both are checked
against the oracle.)  Tolerances as the stage's: core |gpu - oracle| <= 1e-2 +
1e-2 |oracle|; tokens that see nothing are exactly zero; rows S .. S_out - 1
are zero; the workspace is zero again after every call.
"""
import math

import numpy as np
import pytest
import torch

from parity_util import CANARY, compare, to_np16

pytestmark = pytest.mark.gpu

D = 512


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def problem(B, q, H, spr, Lmax, lens, seed=0, S_out=None):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    S = B * q
    qv = torch.randn((S, H, 576), generator=g, device="cuda").to(torch.bfloat16)
    kv = torch.randn((B, Lmax, 576), generator=g, device="cuda").to(torch.bfloat16)
    kv_len = torch.tensor(lens, dtype=torch.int32, device="cuda")
    for b, L in enumerate(lens):
        kv[b, L:] = float("nan")  # never read
    w_v = (torch.randn((H, 128, D), generator=g, device="cuda") / math.sqrt(D)).to(torch.bfloat16)
    gate = torch.sigmoid(torch.randn((S, H * 128), generator=g, device="cuda")).to(torch.bfloat16)
    return dict(qv=qv, kv=kv, kv_len=kv_len, q=q, spr=spr, scale=1 / math.sqrt(192), B=B, H=H, Lmax=Lmax,
                w_v=w_v, gate=gate, S=S, S_out=S if S_out is None else S_out)


def run_fused(inp, ws=None, extra_rows=2):
    import mla_decode_attention_lse_gb300 as m

    B, q, H, spr, S, S_out = (inp[k] for k in ("B", "q", "H", "spr", "S", "S_out"))
    part_o = torch.empty((spr, S, H, D), dtype=torch.bfloat16, device="cuda")
    part_lse = torch.empty((spr, S, H), dtype=torch.float32, device="cuda")
    buf = torch.full((S_out + extra_rows, H * 128), CANARY, dtype=torch.int16, device="cuda")
    out = buf[:S_out].view(torch.bfloat16)
    if ws is None:
        ws = torch.zeros(m.mla_attn_combine_uv_workspace_words(B, q), dtype=torch.int32, device="cuda")
    m.mla_attn_combine_uv(inp["qv"], inp["kv"], inp["kv_len"], q, spr, inp["scale"], part_o, part_lse, inp["w_v"],
                          inp["gate"], out, ws)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    assert int(ws.abs().sum()) == 0, "workspace not left zero"
    full = buf.cpu().numpy().view(np.uint16)
    return full[:S_out], full[S_out:], part_o, part_lse


def combine_of(inp, po, pl):
    """mla_combine_uv (8-token tiles, as the fused launch's combine units) on
    given partials; returns core bits [S_out, H*128]."""
    import mla_decode_attention_lse_gb300 as m

    S_out, H = inp["S_out"], inp["H"]
    out = torch.empty((S_out, H * 128), dtype=torch.bfloat16, device="cuda")
    m.mla_combine_uv(po, pl, inp["q"], inp["spr"], inp["w_v"], 0, inp["gate"], out, tile_tokens=8)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    return to_np16(out)


def run_unfused(inp):
    import mla_decode_attention_lse_gb300 as m

    B, q, H, spr, S, S_out = (inp[k] for k in ("B", "q", "H", "spr", "S", "S_out"))
    o = torch.empty((spr, S, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((spr, S, H), dtype=torch.float32, device="cuda")
    out = torch.empty((S_out, H * 128), dtype=torch.bfloat16, device="cuda")
    # one CTA per item, the attention kernel the fused launch runs
    m.mla_attn_split_kv(inp["qv"], inp["kv"], inp["kv_len"], q, spr, inp["scale"], o, lse, kernel=1)
    m.mla_combine_uv(o, lse, q, spr, inp["w_v"], 0, inp["gate"], out, tile_tokens=8)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    return to_np16(out), o, lse


def oracle_chain(orc, inp, reqs=None):
    """The oracle's attention on the (selected) requests, then its combine."""
    q, H = inp["q"], inp["H"]
    qv, kv, kv_len, gate = inp["qv"], inp["kv"], inp["kv_len"], inp["gate"]
    if reqs is not None:
        idx = torch.tensor(reqs, device=qv.device)
        rows = (idx[:, None] * q + torch.arange(q, device=qv.device)[None]).reshape(-1)
        qv, kv, kv_len, gate = qv[rows], kv[idx], kv_len[idx], gate[rows]
    o_ref, lse_ref = orc.mla_attn_split(to_np16(qv), to_np16(kv), kv_len.cpu().numpy(), q, inp["spr"], inp["scale"])
    ref = orc.Problem(o_ref, lse_ref, q, inp["spr"], to_np16(inp["w_v"]), None, 0, to_np16(gate)).full()
    dead = np.all(np.isneginf(lse_ref), axis=0)  # [S, H]: the token sees nothing at all
    zero = np.zeros(ref.shape, bool)
    for h in range(H):
        zero[dead[:, h], h * 128:(h + 1) * 128] = True
    return ref, zero


CASES = [
    (3, 1, 12, 4, 300, [300, 129, 5], None),              # N = 16, all heads in one CTA; an empty split
    (4, 2, 3, 3, 260, [128, 256, 1, 0], 11),              # q = 2; kv_len 0: the token sees nothing; padded rows
    (2, 4, 16, 2, 200, [200, 77], None),                  # two head groups (N = 32): two items per split
    (5, 3, 5, 5, 150, [150, 9, 64, 0, 149], None),         # q = 3: requests straddle the 8-token tiles
    (1, 1, 1, 1, 1000, [1000], 4),                        # one split of 8 tiles; one head
    (20, 1, 12, 32, 512, list(range(40, 512, 24))[:20], None),  # 32 splits: every lane of the merge
    (17, 1, 12, 16, 700, [700 - 37 * i for i in range(17)], 20),  # a ragged last tile (17 tokens)
]


@pytest.mark.parametrize("B,q,H,spr,Lmax,lens,S_out", CASES)
def test_fused_matches_oracle_chain_and_unfused(lib, orc, B, q, H, spr, Lmax, lens, S_out):
    inp = problem(B, q, H, spr, Lmax, lens, seed=B * 10 + q + spr, S_out=S_out)
    got, canary, po, pl = run_fused(inp)
    assert np.all(canary == CANARY), "wrote past S_out"
    ref, zero = oracle_chain(orc, inp)
    S = inp["S"]
    compare(got[:S], ref, zero, f"fused B={B} q={q} H={H} spr={spr}")
    assert np.all(got[S:] == 0), "rows past S not zero"
    # the combine units: the same bits as mla_combine_uv on the launch's own partials
    assert np.array_equal(got, combine_of(inp, po, pl)), "core differs from mla_combine_uv on the same partials"
    # the two calls in sequence (the standalone attention's tiling) against the oracle too
    unf, o, lse = run_unfused(inp)
    compare(unf[:S], ref, zero, f"two calls B={B} q={q} H={H} spr={spr}")


def test_fused_decode_step_full_size(lib, orc):
    """The decode step the bench times (64 requests x 12 heads, 16 splits, up
    to 4096 cached positions, 10% short requests): bit for bit against the two
    calls, and against the oracle chain on sampled requests (short ones
    included); two calls in a row on one workspace agree."""
    from mla_decode_attention_lse_gb300 import synth

    a = synth.make_attn("attn_splitkv", device="cuda")
    inp = dict(qv=a["qv"], kv=a["kv"], kv_len=a["kv_len"], q=a["q"], spr=a["spr"], scale=a["scale"], B=a["B"],
               H=a["H"], Lmax=a["kv"].shape[1], w_v=a["w_v"], gate=a["gate"], S=a["B"] * a["q"],
               S_out=a["B"] * a["q"])
    import mla_decode_attention_lse_gb300 as m

    ws = torch.zeros(m.mla_attn_combine_uv_workspace_words(inp["B"], inp["q"]), dtype=torch.int32, device="cuda")
    got, canary, po, pl = run_fused(inp, ws)
    got2, _, _, _ = run_fused(inp, ws)
    assert np.array_equal(got, got2), "two calls differ"
    assert np.array_equal(got, combine_of(inp, po, pl)), "core differs from mla_combine_uv on the same partials"
    lens = a["kv_len"].cpu().numpy()
    short = [int(i) for i in np.nonzero(lens <= 64)[0][:2]]
    reqs = sorted(set([0, 17, 63] + short))
    ref, zero = oracle_chain(orc, inp, reqs)
    q = inp["q"]
    rows = [b * q + i for b in reqs for i in range(q)]
    compare(got[rows], ref, zero, "decode step, sampled requests")


def test_fused_empty_batch_and_errors(lib):
    import mla_decode_attention_lse_gb300 as m

    # B = 0: only the padded rows, zeroed
    H = 2
    out = torch.full((5, H * 128), 7, dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(2, dtype=torch.int32, device="cuda")
    qv = torch.empty((0, H, 576), dtype=torch.bfloat16, device="cuda")
    kv = torch.empty((0, 16, 576), dtype=torch.bfloat16, device="cuda")
    kv_len = torch.empty((0,), dtype=torch.int32, device="cuda")
    po = torch.empty((2, 0, H, D), dtype=torch.bfloat16, device="cuda")
    pl = torch.empty((2, 0, H), dtype=torch.float32, device="cuda")
    w_v = torch.zeros((H, 128, D), dtype=torch.bfloat16, device="cuda")
    gate = torch.empty((0, H * 128), dtype=torch.bfloat16, device="cuda")
    m.mla_attn_combine_uv(qv, kv, kv_len, 1, 2, 0.1, po, pl, w_v, gate, out, ws)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
    # a workspace too small for the batch is refused before anything runs
    inp = problem(9, 1, 2, 2, 64, [64] * 9, seed=1)
    small = torch.zeros(2, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MlaError) as e:
        run_fused(inp, small)
    assert e.value.status == m.MLA_ERR_SHAPE


def run_fused_oproj(inp, n_out, seed=5, ws=None, ypad=8, yoff=0):
    """The decode step with the o_proj shard in the same launch; returns (y,
    the canary columns around y, core, W_o).  y is columns yoff .. yoff + n_out
    of a canary-filled buffer of yoff + n_out + ypad columns."""
    import mla_decode_attention_lse_gb300 as m

    B, q, H, spr, S, S_out = (inp[k] for k in ("B", "q", "H", "spr", "S", "S_out"))
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    w_o = (torch.randn((n_out, H * 128), generator=g, device="cuda") / math.sqrt(H * 128)).to(torch.bfloat16)
    part_o = torch.empty((spr, S, H, D), dtype=torch.bfloat16, device="cuda")
    part_lse = torch.empty((spr, S, H), dtype=torch.float32, device="cuda")
    out = torch.empty((S_out, H * 128), dtype=torch.bfloat16, device="cuda")
    ybuf = torch.full((S, yoff + n_out + ypad), CANARY, dtype=torch.int16, device="cuda")
    y = ybuf[:, yoff:yoff + n_out].view(torch.bfloat16)
    if ws is None:
        ws = torch.zeros(m.mla_attn_combine_uv_workspace_words(B, q), dtype=torch.int32, device="cuda")
    m.mla_attn_combine_uv(inp["qv"], inp["kv"], inp["kv_len"], q, spr, inp["scale"], part_o, part_lse, inp["w_v"],
                          inp["gate"], out, ws, w_o=w_o, y=y)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status() == m.MLA_OK
    assert int(ws.abs().sum()) == 0, "workspace not left zero"
    full = ybuf.cpu().numpy().view(np.uint16)
    canary = np.concatenate([full[:, :yoff], full[:, yoff + n_out:]], axis=1)
    return full[:, yoff:yoff + n_out], canary, out, w_o


OPROJ_CASES = [
    (3, 1, 12, 4, 300, [300, 129, 5], 128),           # S = 3, K = 1536
    (4, 2, 3, 3, 260, [128, 256, 1, 0], 64),          # q = 2, a token that sees nothing, K = 384
    (40, 2, 2, 3, 200, [200 - 4 * i for i in range(40)], 192),  # S = 80: two 64-token tiles
    (3, 2, 12, 2, 300, [300, 150, 7], 128),           # 24 query rows: the one-CTA-per-SM instance (N = 32)
]


@pytest.mark.parametrize("B,q,H,spr,Lmax,lens,n_out", OPROJ_CASES)
def test_fused_with_oproj(lib, orc, B, q, H, spr, Lmax, lens, n_out):
    """o_proj in the same launch: y bit for bit as mla_o_proj on the launch's
    own core rows, and against the oracle chain (attention -> combine ->
    o_proj) at the stage's tolerance; the core rows as without o_proj."""
    import mla_decode_attention_lse_gb300 as m

    inp = problem(B, q, H, spr, Lmax, lens, seed=B * 3 + n_out)
    y, canary, core, w_o = run_fused_oproj(inp, n_out)
    assert np.all(canary == CANARY), "wrote past n_out"
    S = inp["S"]
    # core as the launch without o_proj gives it
    got, _, _, _ = run_fused(inp, extra_rows=0)
    assert np.array_equal(to_np16(core), got), "core differs from the launch without o_proj"
    # y as mla_o_proj on the same core rows
    y2 = torch.empty((S, n_out), dtype=torch.bfloat16, device="cuda")
    m.mla_o_proj(core[:S].contiguous(), w_o, y2)
    torch.cuda.synchronize()
    assert np.array_equal(y, to_np16(y2)), "y differs from mla_o_proj on the same core"
    # against the oracle chain
    ref_core, _ = oracle_chain(orc, inp)
    ref = orc.o_proj(ref_core, to_np16(w_o))
    g32 = (y.astype(np.uint32) << 16).view(np.float32)
    r32 = (ref.astype(np.uint32) << 16).view(np.float32) if ref.dtype == np.uint16 else ref
    assert np.all(np.isfinite(g32))
    d = np.abs(g32 - r32)
    bad = d > 1e-2 + 1e-2 * np.abs(r32)
    assert not bad.any(), f"o_proj in the launch: {bad.sum()} out of tolerance, max {d.max()}"


def test_fused_with_oproj_unaligned_y(lib):
    """y whose rows do not start on 16-byte boundaries (its base 2 bytes past
    one, its row stride n_out + 4): the shard's tile is copied out element by
    element, with the same bits as mla_o_proj and nothing written around y."""
    import mla_decode_attention_lse_gb300 as m

    inp = problem(3, 2, 12, 2, 300, [300, 150, 7], seed=77)
    n_out = 128
    y, canary, core, w_o = run_fused_oproj(inp, n_out, ypad=3, yoff=1)
    assert np.all(canary == CANARY), "wrote outside y"
    S = inp["S"]
    y2 = torch.empty((S, n_out), dtype=torch.bfloat16, device="cuda")
    m.mla_o_proj(core[:S].contiguous(), w_o, y2)
    torch.cuda.synchronize()
    assert np.array_equal(y, to_np16(y2)), "y differs from mla_o_proj on the same core"


def test_fused_with_oproj_decode_step(lib, orc):
    """The bench's decode step (64 requests x 12 heads, 16 splits) with the
    7168-output o_proj shard in the same launch: bit for bit as the launch
    without it followed by mla_o_proj; two calls in a row agree."""
    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    a = synth.make_attn("attn_splitkv", device="cuda")
    inp = dict(qv=a["qv"], kv=a["kv"], kv_len=a["kv_len"], q=a["q"], spr=a["spr"], scale=a["scale"], B=a["B"],
               H=a["H"], Lmax=a["kv"].shape[1], w_v=a["w_v"], gate=a["gate"], S=a["B"] * a["q"],
               S_out=a["B"] * a["q"])
    ws = torch.zeros(m.mla_attn_combine_uv_workspace_words(inp["B"], inp["q"]), dtype=torch.int32, device="cuda")
    y, canary, core, w_o = run_fused_oproj(inp, 7168, ws=ws)
    y_again, _, _, _ = run_fused_oproj(inp, 7168, ws=ws)
    assert np.array_equal(y, y_again), "two calls differ"
    assert np.all(canary == CANARY)
    got, _, _, _ = run_fused(inp, ws)
    assert np.array_equal(to_np16(core), got)
    y2 = torch.empty((inp["S"], 7168), dtype=torch.bfloat16, device="cuda")
    m.mla_o_proj(core.contiguous(), w_o, y2)
    torch.cuda.synchronize()
    assert np.array_equal(y, to_np16(y2))


def test_fused_oproj_argument_errors(lib):
    import mla_decode_attention_lse_gb300 as m

    inp = problem(2, 1, 2, 2, 64, [64, 10], seed=3)
    S, H = inp["S"], inp["H"]
    part_o = torch.empty((2, S, H, D), dtype=torch.bfloat16, device="cuda")
    part_lse = torch.empty((2, S, H), dtype=torch.float32, device="cuda")
    out = torch.empty((S, H * 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(m.mla_attn_combine_uv_workspace_words(2, 1), dtype=torch.int32, device="cuda")
    w_o = torch.zeros((96, H * 128), dtype=torch.bfloat16, device="cuda")  # 96 outputs: not a multiple of 64
    y = torch.zeros((S, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MlaError) as e:
        m.mla_attn_combine_uv(inp["qv"], inp["kv"], inp["kv_len"], 1, 2, inp["scale"], part_o, part_lse, inp["w_v"],
                              inp["gate"], out, ws, w_o=w_o, y=y)
    assert e.value.status == m.MLA_ERR_SHAPE
    # a workspace of the previous size (2 + tiles words) is refused
    small = torch.zeros(m.mla_attn_combine_uv_workspace_words(2, 1) - 1, dtype=torch.int32, device="cuda")
    with pytest.raises(m.MlaError) as e:
        m.mla_attn_combine_uv(inp["qv"], inp["kv"], inp["kv_len"], 1, 2, inp["scale"], part_o, part_lse, inp["w_v"],
                              inp["gate"], out, small)
    assert e.value.status == m.MLA_ERR_SHAPE


@pytest.mark.parametrize("case", range(16))
def test_fused_fuzz(lib, orc, case):
    """Seeded random decode steps through the one-launch path: requests,
    queries per request, heads (both tilings: up to 16 query rows and more),
    splits, lengths (empty, one position, tile edges, long), padded output
    rows, and (every other case) the o_proj shard in the launch.  core against
    the oracle chain and bit for bit against mla_combine_uv on the launch's own
    partials; y bit for bit against mla_o_proj on the same core rows."""
    import mla_decode_attention_lse_gb300 as m

    rng = np.random.default_rng(5000 + case)
    q = int(rng.choice([1, 1, 2, 3, 4]))
    H = int(rng.integers(1, 17))
    B = int(rng.integers(1, 7))
    spr = int(rng.choice([1, 2, 3, 5, 16, 32]))
    Lmax = int(rng.choice([16, 64, 65, 129, 300, 700]))
    lens = [min(int(rng.choice([0, 1, q, 63, 64, 65, int(rng.integers(1, Lmax + 1)), Lmax])), Lmax) for _ in range(B)]
    S = B * q
    S_out = S + int(rng.choice([0, 0, 3]))
    inp = problem(B, q, H, spr, Lmax, lens, seed=700 + case, S_out=S_out)
    what = f"fuzz {case}: B={B} q={q} H={H} spr={spr} Lmax={Lmax} lens={lens} S_out={S_out}"
    got, canary, po, pl = run_fused(inp)
    assert np.all(canary == CANARY), what
    ref, zero = oracle_chain(orc, inp)
    compare(got[:S], ref, zero, what)
    assert np.all(got[S:] == 0), what
    assert np.array_equal(got, combine_of(inp, po, pl)), what
    if case % 2:
        n_out = 64 * int(rng.integers(1, 4))
        y, ycan, core, w_o = run_fused_oproj(inp, n_out, seed=case)
        assert np.all(ycan == CANARY), what
        assert np.array_equal(to_np16(core), got), what
        y2 = torch.empty((S, n_out), dtype=torch.bfloat16, device="cuda")
        m.mla_o_proj(core[:S].contiguous(), w_o, y2)
        torch.cuda.synchronize()
        assert np.array_equal(y, to_np16(y2)), what
