"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Every workload of the synthetic recipe, both kernels where they apply, and
the edge cases the method has.  Tolerance |gpu - oracle| <= 1e-2 + 1e-2 *
|oracle| element-wise (both W_V formats); rows the definition zeroes must be
exactly zero; rows past S_out must be untouched.
"""
import numpy as np
import pytest
import torch

from parity_util import (CANARY, bits_to_f32, compare, dead_rows, host_inputs, oracle_problem,
                         run_gpu, seg_mask, to_np16)

pytestmark = pytest.mark.gpu

SIMT, TC, KS = 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from mla_decode_attention_lse_gb300 import build, load_library

    build.build()
    return load_library()


def synth():
    from mla_decode_attention_lse_gb300 import synth as s

    return s


def check_full(orc, inp, kernel, tile=0, what=""):
    gpu, canary = run_gpu(inp, kernel=kernel, tile=tile)
    ref = oracle_problem(orc, inp).full()
    assert np.all(canary == CANARY), f"{what}: wrote past S_out"
    return compare(gpu, ref, seg_mask(inp), what)


# ---- the recipe's workloads at full size ---------------------------------

CASES = [
    ("tiny_split", 0, 0), ("tiny_split", SIMT, 0), ("tiny_split", TC, 16),
    ("nosplit", SIMT, 0), ("nosplit", TC, 16), ("nosplit", TC, 32),
    ("splitkv", 0, 0), ("splitkv", SIMT, 0), ("splitkv", TC, 32),
    ("splitkv_rm", 0, 0), ("splitkv_rm", SIMT, 0),
    ("stacked_mxfp4", 0, 0), ("stacked_mxfp4", SIMT, 0), ("stacked_mxfp4", TC, 16),
    ("stacked_mxfp4", TC, 32),
    ("tiny_split", KS, 0), ("nosplit", KS, 0), ("splitkv", KS, 0), ("splitkv_rm", KS, 0),
    ("stacked_mxfp4", KS, 0),
    # 8-token tiles (two warps per token, half a row each): the automatic
    # choice for the bf16 split-KV decode steps, on request elsewhere
    ("nosplit", 0, 0), ("tiny_split", TC, 8), ("nosplit", TC, 8), ("splitkv", TC, 8), ("splitkv", TC, 16),
    ("splitkv_rm", TC, 8), ("stacked_mxfp4", TC, 8),
]


@pytest.mark.parametrize("name,kernel,tile", CASES)
def test_workload_full_parity(lib, orc, name, kernel, tile):
    inp = synth().make(name, device="cuda")
    check_full(orc, inp, kernel, tile, f"{name}/k{kernel}/t{tile}")


@pytest.mark.parametrize("w_fmt", [0, 1])
def test_stacked_both_weight_formats(lib, orc, w_fmt):
    inp = synth().make("stacked_mxfp4", device="cuda", w_fmt=w_fmt)
    check_full(orc, inp, 0, 0, f"stacked w_fmt={w_fmt}")


@pytest.mark.parametrize("name", ["mtp", "mtp_mxfp4"])
def test_large_batch_sampled_parity(lib, orc, name):
    """The large multi-token batch in the launch configuration the bench times
    (automatic kernel choice): sampled (t, h) rows against the oracle, plus
    whole-output properties."""
    s = synth()
    inp = s.make(name, device="cuda")
    gpu, canary = run_gpu(inp)
    assert np.all(canary == CANARY)
    host = host_inputs(inp)
    pr = oracle_problem(orc, inp, host)
    rng = np.random.default_rng(123)
    S, H = inp["S"], inp["H"]
    ts = np.concatenate([rng.integers(0, S, 1500), [0, S - 1, S // 2]])
    hs = np.concatenate([rng.integers(0, H, 1500), [0, H - 1, H // 2]])
    dr = dead_rows(inp)
    # every dead row is sampled too
    dts, dhs = np.nonzero(dr)
    ts = np.concatenate([ts, dts[:50]])
    hs = np.concatenate([hs, dhs[:50]])
    ref = pr.rows(ts, hs)
    got = np.stack([gpu[t, h * 128:(h + 1) * 128] for t, h in zip(ts, hs)])
    zmask = np.zeros_like(got, bool)
    zmask[dr[ts, hs]] = True
    compare(got, ref, zmask, name)
    g = bits_to_f32(gpu)
    assert not np.isnan(g).any()
    # all dead rows are exactly zero at full size, live rows are not
    for t, h in zip(dts, dhs):
        assert np.all(g[t, h * 128:(h + 1) * 128] == 0)
    live = ~dr
    assert np.count_nonzero(np.any(g.reshape(S, H, 128) != 0, axis=-1)[live]) == live.sum()


# ---- edge cases ---------------------------------------------------------------

def custom(**kw):
    return synth().custom(device="cuda", **kw)


@pytest.mark.parametrize("kernel", [SIMT, TC, KS])
@pytest.mark.parametrize("S,S_out", [(1, 1), (17, 20), (33, 33), (47, 64)])
def test_ragged_token_counts(lib, orc, kernel, S, S_out):
    inp = custom(S=S, S_out=S_out, H=3, P=3, q=1, spr=3, w_fmt=0, neg_inf_frac=0.2, seed=S)
    check_full(orc, inp, kernel, 16, f"S={S}")


@pytest.mark.parametrize("kernel", [SIMT, TC])
def test_empty_batch_zeroes_padding(lib, orc, kernel):
    inp = custom(S=0, S_out=5, H=2, P=2, q=1, spr=2, w_fmt=0)
    gpu, canary = run_gpu(inp, kernel=kernel)
    assert np.all(gpu == 0) and np.all(canary == CANARY)


@pytest.mark.parametrize("kernel", [SIMT, TC, KS])
def test_request_major_with_q3(lib, orc, kernel):
    # 6 requests x q=3, 5 splits each -> P = 30, request-major
    inp = custom(S=18, H=2, P=30, q=3, spr=5, w_fmt=1, neg_inf_frac=0.15, nan_frac=0.05, seed=5)
    check_full(orc, inp, kernel, 16, "rm q3")


@pytest.mark.parametrize("w_fmt", [0, 1])
def test_17_to_32_partials_on_tensor_cores(lib, orc, w_fmt):
    # one token per warp (16-token tiles); 20 partials, 25% dead
    inp = custom(S=40, H=3, P=20, q=1, spr=20, w_fmt=w_fmt, neg_inf_frac=0.25, seed=12 + w_fmt)
    check_full(orc, inp, TC, 0, f"P=20 w_fmt={w_fmt}")


def test_more_than_32_partials_on_cuda_cores(lib, orc):
    inp = custom(S=8, H=2, P=40, q=1, spr=40, w_fmt=0, neg_inf_frac=0.3, seed=6)
    check_full(orc, inp, SIMT, 0, "P=40")
    import mla_decode_attention_lse_gb300 as m

    with pytest.raises(m.MlaError) as e:
        run_gpu(inp, kernel=TC)
    assert e.value.status == m.MLA_ERR_KERNEL


@pytest.mark.parametrize("kernel,tile", [(SIMT, 16), (TC, 16), (TC, 32), (KS, 16)])
@pytest.mark.parametrize("w_fmt", [0, 1])
def test_all_dead_rows_and_planted_nan(lib, orc, kernel, tile, w_fmt):
    # tile 32 with 4 partials is the two-batch unit whose first unit's both
    # batches are loaded before the weights are known (MXFP4): dead rows are
    # loaded there and must still never reach the merge
    inp = custom(S=32 if tile == 16 else 96, H=4, P=4, q=1, spr=4, w_fmt=w_fmt, dead_rows=10,
                 neg_inf_frac=0.3, seed=7)
    # plant NaN and Inf in the o rows of dead partials: they must never be read
    lse, o = inp["lse"], inp["o"]
    dead = ~torch.isfinite(lse)
    o[dead] = float("nan")
    o[:, :, :, 5][dead] = float("inf")
    check_full(orc, inp, kernel, tile, f"planted NaN, tile {tile}")


@pytest.mark.parametrize("kernel", [SIMT, TC, KS])
def test_strided_views(lib, orc, kernel):
    s = synth()
    base = s.custom(S=40, H=6, P=3, q=1, spr=3, w_fmt=0, seed=8, device="cuda")
    # o as a head slice of a wider tensor, tokens strided; lse permuted view
    big = torch.randn(3, 40, 10, 512, device="cuda").to(torch.bfloat16)
    big[:, :, 2:8] = base["o"]
    lse_big = torch.randn(40, 6, 3, device="cuda")
    lse_big.copy_(base["lse"].permute(1, 2, 0))
    wbig = torch.zeros(6, 256, 512, dtype=torch.bfloat16, device="cuda")
    wbig[:, ::2] = base["w_v"]
    inp = dict(base, o=big[:, :, 2:8], lse=lse_big.permute(2, 0, 1), w_v=wbig[:, ::2])
    assert not inp["o"].is_contiguous() and inp["w_v"].stride(1) == 1024
    check_full(orc, inp, kernel, 16, "strided")


@pytest.mark.parametrize("kernel", [SIMT, TC, KS])
def test_passthrough_mxfp4_with_inf_latent(lib, orc, kernel):
    # P == 1: the o row is the latent; an Inf in it makes its block's scale NaN
    inp = custom(S=16, H=2, P=1, q=1, spr=0, w_fmt=1, lse_unused=True, seed=9)
    inp["o"][0, 3, 1, 70] = float("inf")
    check_full(orc, inp, kernel, 16, "inf latent")


def test_head_changes_inside_a_cta(lib, orc):
    # more units than SMs with 16-token tiles: CTAs walk across head boundaries
    for w_fmt in (0, 1):
        inp = custom(S=400, H=12, P=2, q=1, spr=2, w_fmt=w_fmt, neg_inf_frac=0.05, seed=10 + w_fmt)
        check_full(orc, inp, TC, 16, f"head changes w_fmt={w_fmt}")


def test_two_calls_two_streams(lib, orc):
    inp = synth().make("stacked_mxfp4", device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    a, _ = run_gpu(inp, stream=s1)
    b, _ = run_gpu(inp, stream=s2)
    assert np.array_equal(a, b)  # deterministic


def test_cluster_kernel_two_streams(lib, orc):
    # rank-ordered sums: the cluster kernel is deterministic across streams
    inp = synth().make("splitkv", device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    a, _ = run_gpu(inp, stream=s1, kernel=KS)
    b, _ = run_gpu(inp, stream=s2, kernel=KS)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("w_fmt", [0, 1])
def test_wide_offsets_take_the_64_bit_path(lib, orc, w_fmt):
    # an lse view whose partial stride is 2^32 elements (a 16 GiB allocation,
    # touched only at the viewed entries): the plan must drop 32-bit address
    # arithmetic, and that kernel instance must match the oracle too
    import mla_decode_attention_lse_gb300 as m

    base = custom(S=40, H=3, P=2, q=1, spr=2, w_fmt=w_fmt, neg_inf_frac=0.1, seed=20 + w_fmt)
    big = torch.empty((1 << 32) + 40 * 3, dtype=torch.float32, device="cuda")
    try:
        lse = big.as_strided((2, 40, 3), (1 << 32, 3, 1))
        lse.copy_(base["lse"])
        inp = dict(base, lse=lse)
        out = torch.empty(40, 3 * 128, dtype=torch.bfloat16, device="cuda")
        args = m.make_args(inp["o"], lse, 1, 2, inp["w_v"], w_fmt, inp["gate"], out, inp["w_scale"])
        assert m.mla_combine_uv_plan(args)["offsets32"] == 0
        ref = oracle_problem(orc, dict(inp, lse=lse.contiguous())).full()
        for kernel in (SIMT, TC, KS):
            gpu, canary = run_gpu(inp, kernel=kernel, tile=16)
            assert np.all(canary == CANARY)
            compare(gpu, ref, seg_mask(inp), f"64-bit offsets, kernel {kernel}")
    finally:
        del big
        torch.cuda.empty_cache()


# ---- 8-token tiles: two warps per token, each merging half of the row ------

@pytest.mark.parametrize("w_fmt", [0, 1])
@pytest.mark.parametrize("S,S_out,P,q,spr", [
    (1, 1, 3, 1, 3),        # one token
    (7, 9, 7, 1, 7),        # one batch per unit, padded rows
    (9, 9, 16, 1, 16),      # two batches per unit, a ragged second tile
    (47, 50, 1, 1, 0),      # passthrough
    (18, 18, 30, 3, 5),     # request-major, q = 3
    (24, 26, 24, 1, 24),    # three batches per unit
    (40, 40, 32, 1, 32),    # 32 partials: four batches per unit
])
def test_eight_token_tiles(lib, orc, w_fmt, S, S_out, P, q, spr):
    pas = P == 1
    inp = custom(S=S, S_out=S_out, H=3, P=P, q=q, spr=spr, w_fmt=w_fmt, neg_inf_frac=0.0 if pas else 0.2,
                 nan_frac=0.0 if pas else 0.05, lse_unused=pas, seed=100 + S + P + w_fmt)
    if not pas:  # dead partials' rows poisoned: they must never be read
        inp["o"][~torch.isfinite(inp["lse"])] = float("nan")
    check_full(orc, inp, TC, 8, f"8-token tiles S={S} P={P} w_fmt={w_fmt}")


@pytest.mark.parametrize("w_fmt", [0, 1])
def test_eight_token_tiles_dead_rows_strided_heads(lib, orc, w_fmt):
    s = synth()
    # all-dead rows with NaN planted in the dead partials
    inp = custom(S=32, H=4, P=4, q=1, spr=4, w_fmt=w_fmt, dead_rows=10, neg_inf_frac=0.3, seed=70 + w_fmt)
    inp["o"][~torch.isfinite(inp["lse"])] = float("nan")
    check_full(orc, inp, TC, 8, "8-token tiles, planted NaN")
    # strided o / lse / W_V views
    base = s.custom(S=40, H=6, P=3, q=1, spr=3, w_fmt=0, seed=80, device="cuda")
    big = torch.randn(3, 40, 10, 512, device="cuda").to(torch.bfloat16)
    big[:, :, 2:8] = base["o"]
    lse_big = torch.randn(40, 6, 3, device="cuda")
    lse_big.copy_(base["lse"].permute(1, 2, 0))
    wbig = torch.zeros(6, 256, 512, dtype=torch.bfloat16, device="cuda")
    wbig[:, ::2] = base["w_v"]
    inp = dict(base, o=big[:, :, 2:8], lse=lse_big.permute(2, 0, 1), w_v=wbig[:, ::2])
    check_full(orc, inp, TC, 8, "8-token tiles, strided")
    # more units than SMs: CTAs walk across head boundaries
    inp = custom(S=400, H=12, P=2, q=1, spr=2, w_fmt=w_fmt, neg_inf_frac=0.05, seed=90 + w_fmt)
    check_full(orc, inp, TC, 8, f"8-token tiles, head changes w_fmt={w_fmt}")
    # an Inf latent in the passthrough (its MX block's scale is NaN)
    inp = custom(S=16, H=2, P=1, q=1, spr=0, w_fmt=w_fmt, lse_unused=True, seed=95)
    inp["o"][0, 3, 1, 300] = float("inf")
    check_full(orc, inp, TC, 8, "8-token tiles, inf latent")


# ---- runtime tiles: the 32-token kernel with 17..31 tokens per unit ----------

@pytest.mark.parametrize("w_fmt", [0, 1])
@pytest.mark.parametrize("tile,S,S_out,P,q,spr", [
    (22, 256, 264, 8, 1, 8),    # the stacked decode batch's automatic tile
    (17, 40, 41, 4, 1, 4),      # two batches per unit (the blind second batch with MXFP4)
    (31, 95, 95, 16, 1, 16),    # a ragged last unit
    (20, 47, 50, 1, 1, 0),      # passthrough
    (24, 18, 18, 30, 3, 5),     # request-major, q = 3, one unit
])
def test_runtime_token_tiles(lib, orc, w_fmt, tile, S, S_out, P, q, spr):
    pas = P == 1
    inp = custom(S=S, S_out=S_out, H=3, P=P, q=q, spr=spr, w_fmt=w_fmt, neg_inf_frac=0.0 if pas else 0.2,
                 nan_frac=0.0 if pas else 0.05, lse_unused=pas, dead_rows=0 if pas else 4,
                 seed=200 + tile + S + w_fmt)
    if not pas:  # dead partials' rows poisoned: they must never be read
        inp["o"][~torch.isfinite(inp["lse"])] = float("nan")
    check_full(orc, inp, TC, tile, f"tile {tile} S={S} P={P} w_fmt={w_fmt}")


@pytest.mark.parametrize("w_fmt,S", [(0, 700), (1, 400)])
def test_runtime_tiles_head_changes(lib, orc, w_fmt, S):
    # more units than SMs: CTAs walk across head boundaries with 20-token units.
    # (MXFP4 on fewer rows: its E2M1 codes follow the latents exactly, and the
    # kernel's hardware exp2 / reciprocal for the weights can move a latent
    # one bf16 ulp across an E2M1 rounding midpoint, a flip that exceeded the
    # bound once in 1.07 M outputs of 700 x 12 rows)
    inp = custom(S=S, H=12, P=4, q=1, spr=4, w_fmt=w_fmt, neg_inf_frac=0.05, seed=300 + w_fmt)
    check_full(orc, inp, TC, 20, f"tile 20, head changes, w_fmt={w_fmt}")


# ---- CUDA cores for small batches: one CTA per (head, 16 V rows) ------------

@pytest.mark.parametrize("w_fmt", [0, 1])
@pytest.mark.parametrize("S,S_out,H,P,q,spr", [
    (1, 1, 2, 3, 1, 3),       # one token
    (3, 5, 12, 1, 1, 0),      # passthrough, padded rows
    (8, 8, 12, 16, 1, 16),    # a split-KV decode batch of 8 tokens
    (16, 20, 4, 32, 1, 32),   # 16 tokens (the layout's limit), 32 partials
    (12, 12, 3, 24, 2, 4),    # request-major, q = 2
])
def test_small_batch_cuda_cores(lib, orc, w_fmt, S, S_out, H, P, q, spr):
    import mla_decode_attention_lse_gb300 as m

    pas = P == 1
    inp = custom(S=S, S_out=S_out, H=H, P=P, q=q, spr=spr, w_fmt=w_fmt, neg_inf_frac=0.0 if pas else 0.2,
                 nan_frac=0.0 if pas else 0.05, lse_unused=pas, dead_rows=0 if pas else min(2, S),
                 seed=400 + S + P + w_fmt)
    if not pas:  # dead partials' rows poisoned: they must never be read
        inp["o"][~torch.isfinite(inp["lse"])] = float("nan")
    a = m.make_args(inp["o"], inp["lse"], inp["q"], inp["spr"], inp["w_v"], w_fmt, inp["gate"],
                    torch.empty(S_out, H * 128, dtype=torch.bfloat16, device="cuda"), inp["w_scale"], kernel=SIMT)
    plan = m.mla_combine_uv_plan(a)
    assert (plan["grid"], plan["tile_tokens"]) == (H * 8, S)  # the small-batch layout
    check_full(orc, inp, SIMT, 0, f"small-batch CUDA cores S={S} P={P} w_fmt={w_fmt}")
