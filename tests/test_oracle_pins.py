"""Pins for the CPU oracle: checks against what the page and the mathematics
fix, independent of the oracle's own code (no GPU).

Subject: the vLLM page
"vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
(sane, combine_ranks, combine_splits, stage_combine, stage_uv).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

D, V, BLK = 512, 128, 32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---- helpers (input formatting only) ------------------------------------

def to_bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def dummy_weights(H, rng):
    w = to_bf16_bits(rng.standard_normal((H, V, D)) / math.sqrt(D))
    gate = to_bf16_bits(1 / (1 + np.exp(-rng.standard_normal((1, H * V)))))
    return w, gate


def problem(orc, o_f32=None, lse=None, q=1, spr=0, H=None, w=None, gate=None, S_out=None,
            o_bits=None, w_fmt=0, w_scale=None, rng=None):
    rng = rng or np.random.default_rng(0)
    o = o_bits if o_bits is not None else to_bf16_bits(o_f32)
    P, S, Hh, _ = o.shape
    if w is None:
        w, g1 = dummy_weights(Hh, rng)
        gate = np.repeat(g1, S, axis=0) if gate is None else gate
    if gate is None:
        gate = to_bf16_bits(np.full((S, Hh * V), 0.5))
    lse = None if lse is None else np.ascontiguousarray(lse, np.float32)
    return orc.Problem(o, lse, q, spr, w, w_scale, w_fmt, np.ascontiguousarray(gate), S_out)


# ---- scalar formats -------------------------------------------------------

def test_bf16_round_matches_torch_rne(orc):
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(4000) * np.exp2(rng.integers(-130, 127, 4000))).astype(np.float32)
    u = rng.integers(0, 1 << 16, 200).astype(np.uint32)
    ties = ((u << 16) | 0x8000).view(np.float32)  # exactly halfway, both parities
    near = np.concatenate([((u << 16) | 0x7FFF).view(np.float32),
                           ((u << 16) | 0x8001).view(np.float32)])
    special = np.array([0.0, -0.0, np.inf, -np.inf, 3.3895314e38, 1e-40, -1e-45], np.float32)
    allx = np.concatenate([x, ties, near, special])
    allx = allx[np.isfinite(allx) | np.isinf(allx)]
    ours = orc.bf16_round(allx)
    ref = to_bf16_bits(allx)
    assert np.array_equal(ours, ref)
    nan_bits = orc.bf16_round(np.array([np.nan], np.float32))[0]
    assert np.isnan(bits_to_f32([nan_bits])[0])


def test_sane(orc):
    # page: sane -- NaN and +inf become -inf, everything else stays
    assert orc.sane(float("nan")) == -math.inf
    assert orc.sane(math.inf) == -math.inf
    assert orc.sane(-math.inf) == -math.inf
    for v in (0.0, -3.5, 1e30, -1e-30):
        assert orc.sane(v) == np.float32(v)


def test_e2m1_halfway_cases_round_to_even(orc):
    # E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6 (OCP MX v1.0); codes 0..7
    cases = {0.0: 0, 0.2: 0, 0.25: 0, 0.3: 1, 0.5: 1, 0.75: 2, 1.0: 2, 1.25: 2, 1.3: 3,
             1.5: 3, 1.75: 4, 2.0: 4, 2.5: 4, 2.6: 5, 3.0: 5, 3.5: 6, 4.0: 6, 5.0: 6,
             5.1: 7, 6.0: 7, 7.9: 7, 100.0: 7}
    for y, c in cases.items():
        assert orc.e2m1_code(y) == c, y
        assert orc.e2m1_code(-y) == (c | 8 if c else 0), -y
    assert orc.e2m1_code(-0.0) == 0
    assert [orc.e2m1_value(c) for c in range(8)] == [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    assert orc.e2m1_value(8 | 7) == -6.0


def test_e2m1_exhaustive_bf16_inputs(orc):
    # nearest E2M1 magnitude in exact rational arithmetic, ties to the even code
    from fractions import Fraction

    grid = [Fraction(g) for g in ("0", "1/2", "1", "3/2", "2", "3", "4", "6")]
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits_to_f32(bits)
    fin = np.isfinite(vals)
    for b, y in zip(bits[fin], vals[fin]):
        a = abs(Fraction(float(y)))
        d = [abs(a - g) for g in grid]
        best = [i for i, di in enumerate(d) if di == min(d)]
        c = best[0] if len(best) == 1 else [i for i in best if i % 2 == 0][0]
        if c and y < 0:
            c |= 8
        assert orc.e2m1_code(float(y)) == c, (hex(int(b)), y)


def test_mx_block_roundtrip_and_scale_of_amax(orc):
    rng = np.random.default_rng(2)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    for k in range(-20, 21, 3):
        mags = rng.choice(grid, BLK)
        mags[rng.integers(BLK)] = 6.0  # amax = 6 * 2^k
        vals = mags * rng.choice([-1, 1], BLK) * 2.0 ** k
        codes, sc = orc.mx_quant_block(to_bf16_bits(vals))
        assert sc == k + 127
        back = np.array([orc.e2m1_value(int(c)) for c in codes]) * orc.e8m0_value(sc)
        assert np.array_equal(back, vals.astype(np.float32))


def test_mx_scale_puts_amax_in_top_binade(orc):
    # OCP MX: the shared exponent is floor(log2 amax) minus E2M1's emax (2),
    # so amax / scale lands in [4, 8)
    rng = np.random.default_rng(3)
    for e in range(-40, 41, 2):
        blk = to_bf16_bits(rng.standard_normal(BLK) * 2.0 ** e)
        c = orc.mx_scale_code(blk)
        amax = np.abs(bits_to_f32(blk)).max()
        r = amax / 2.0 ** (c - 127)
        assert 4.0 <= r < 8.0, (e, c, r)
    assert orc.mx_scale_code(np.zeros(BLK, np.uint16)) == 1
    tiny = np.zeros(BLK, np.uint16)
    tiny[5] = 0x0001  # smallest bf16 subnormal: clamps to code 1
    assert orc.mx_scale_code(tiny) == 1


def test_e8m0_values_follow_the_ocp_encoding(orc):
    # OCP MX v1.0: an E8M0 scale is 2^(code - 127) for codes 0..254; 0xFF is NaN
    for code in (0, 1, 100, 127, 128, 200, 254):
        assert orc.e8m0_value(code) == 2.0 ** (code - 127)
    assert math.isnan(orc.e8m0_value(255))


def test_mx_nonfinite_block_scale_is_nan(orc):
    # a block whose amax is Inf or NaN has no finite scale: its code is the
    # E8M0 NaN (0xFF), so every element of that block dequantises to NaN; the
    # largest finite bf16 still gets a finite code (floor(log2 amax) = 127)
    for bad in (np.inf, -np.inf, np.nan):
        vals = np.linspace(-3.0, 3.0, BLK)
        vals[7] = bad
        blk = to_bf16_bits(vals)
        assert orc.mx_scale_code(blk) == 255
        _, sc = orc.mx_quant_block(blk)
        assert sc == 255
    big = np.zeros(BLK)
    big[0] = 3.3895314e38
    assert orc.mx_scale_code(to_bf16_bits(big)) == 127 - 2 + 127


def test_mxfp4_inf_latent_poisons_only_its_row(orc):
    # one passthrough latent is +inf: its MX block's scale is NaN, so every
    # output of that (token, head) is NaN (each sums over all 512 latents);
    # every other row stays finite
    from mla_decode_attention_lse_gb300 import synth

    rng = np.random.default_rng(21)
    S, H = 3, 2
    of = rng.standard_normal((1, S, H, D))
    of[0, 1, 0, 300] = np.inf
    wf = torch.from_numpy(rng.standard_normal((H, V, D)) / math.sqrt(D)).float()
    codes, scales = (t.numpy() for t in synth.mxfp4_pack_weights(wf))
    out = bits_to_f32(problem(orc, of, spr=0, w=codes, w_scale=scales, w_fmt=1).full()).reshape(S, H, V)
    assert np.all(np.isnan(out[1, 0]))
    keep = np.ones((S, H), bool)
    keep[1, 0] = False
    assert np.all(np.isfinite(out[keep]))


# ---- layout rule ------------------------------------------------------------

def test_partial_set_layouts(orc):
    assert orc.partial_set(3, 8, 1, 1, 0) == (0, 0, 1)          # passthrough
    assert orc.partial_set(5, 8, 4, 2, 4) == (1, 0, 4)          # compact
    # request-major: 4 requests x q=2, 3 splits each -> P=12
    assert orc.partial_set(0, 8, 12, 2, 3) == (2, 0, 3)
    assert orc.partial_set(5, 8, 12, 2, 3) == (2, 6, 3)
    assert orc.partial_set(7, 8, 12, 2, 3)[0:2] == (2, 9)
    assert orc.partial_set(0, 8, 7, 2, 3)[0] == -1              # neither layout
    assert orc.partial_set(0, 7, 9, 2, 3)[0] == -1              # S % q != 0


# ---- combine: brute force (flash-decoding identity) -----------------------

def _attention_split(rng, L, cuts, dk=64):
    """Full softmax attention of one query over L positions, and the same
    attention cut into chunks: (full [512], [(o_j [512], lse_j)])."""
    qv = rng.standard_normal(dk)
    K = rng.standard_normal((L, dk))
    Vv = rng.standard_normal((L, D))
    s = K @ qv / math.sqrt(dk)
    p = np.exp(s - s.max())
    full = (p / p.sum()) @ Vv
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        if b == a:  # empty chunk: no KV, lse -inf, o garbage
            parts.append((np.full(D, np.nan), -np.inf))
            continue
        sj = s[a:b]
        mj = sj.max()
        pj = np.exp(sj - mj)
        parts.append(((pj / pj.sum()) @ Vv[a:b], mj + math.log(pj.sum())))
    return full, parts


@pytest.mark.parametrize("layout", ["compact", "request_major"])
def test_combine_equals_full_attention(orc, layout):
    rng = np.random.default_rng(4)
    H, spr = 3, 4
    if layout == "compact":
        nreq, q = 5, 1
    else:
        nreq, q = 3, 2
    S = nreq * q
    P = spr if layout == "compact" else nreq * spr
    o = np.full((P, S, H, D), np.nan, np.float32)
    lse = np.full((P, S, H), np.nan, np.float32)
    full = np.zeros((S, H, D))
    for t in range(S):
        for h in range(H):
            L = int(rng.integers(20, 60))
            cuts = sorted([0, L] + list(rng.integers(0, L, spr - 1)))
            if t == 1 and h == 2:
                cuts = [0, 0, L // 2, L // 2, L]  # two empty chunks
            f, parts = _attention_split(rng, L, cuts)
            full[t, h] = f
            r0 = 0 if layout == "compact" else (t // q) * spr
            for j, (oj, lj) in enumerate(parts):
                o[r0 + j, t, h] = oj
                lse[r0 + j, t, h] = lj
    pr = problem(orc, o, lse, q=q, spr=spr)
    for t in range(S):
        for h in range(H):
            lat = pr.latent_f32(t, h)
            r0 = 0 if layout == "compact" else (t // q) * spr
            om = np.nanmax(np.abs(o[r0:r0 + spr, t, h]), axis=0)
            assert np.all(np.abs(lat - full[t, h]) <= 2.0 ** -8 * om + 1e-5), (t, h)


# ---- combine: special cases ----------------------------------------------------

def test_single_partial_is_identity(orc):
    rng = np.random.default_rng(5)
    o = rng.standard_normal((1, 3, 2, D)).astype(np.float32)
    for lv in (0.0, -np.inf, np.nan, 7.0):
        pr = problem(orc, o, np.full((1, 3, 2), lv), spr=0)
        for t in range(3):
            for h in range(2):
                assert np.array_equal(pr.latent_bf16(t, h), to_bf16_bits(o[0, t, h]))
    # P > 1 with exactly one live partial: its row, bit for bit
    o3 = rng.standard_normal((3, 2, 2, D)).astype(np.float32)
    lse = np.array([-np.inf, 2.5, np.nan], np.float32)[:, None, None] * np.ones((3, 2, 2))
    o3b = to_bf16_bits(o3)
    o3b[0] = 0x7FC0  # NaN rows on the dead partials must not leak
    o3b[2] = 0x7FC0
    pr = problem(orc, o_bits=o3b, lse=lse, spr=3)
    for t in range(2):
        for h in range(2):
            assert np.array_equal(pr.latent_bf16(t, h), o3b[1, t, h])


def test_equal_lse_gives_mean(orc):
    rng = np.random.default_rng(6)
    P = 4
    ob = to_bf16_bits(rng.standard_normal((P, 2, 2, D)))
    pr = problem(orc, o_bits=ob, lse=np.full((P, 2, 2), 3.7), spr=P)
    for t in range(2):
        for h in range(2):
            mean = bits_to_f32(ob[:, t, h]).astype(np.float64).mean(0)
            got = bits_to_f32(pr.latent_bf16(t, h)).astype(np.float64)
            ref = bits_to_f32(to_bf16_bits(mean)).astype(np.float64)
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
            assert np.all(np.abs(got - ref) <= ulp)
            assert np.mean(got == ref) > 0.99


@pytest.mark.parametrize("poison", [-np.inf, np.nan, np.inf])
def test_dead_partial_contributes_nothing(orc, poison):
    rng = np.random.default_rng(7)
    P, S, H = 5, 3, 2
    ob = to_bf16_bits(rng.standard_normal((P, S, H, D)))
    lse = (rng.standard_normal((P, S, H)) * 2 + 4).astype(np.float32)
    lse[2] = poison
    ob_poisoned = ob.copy()
    ob_poisoned[2] = 0x7FC0  # NaN everywhere in the dead partial
    keep = [0, 1, 3, 4]
    w, g = dummy_weights(H, rng)
    gate = np.repeat(g, S, axis=0)
    a = problem(orc, o_bits=ob_poisoned, lse=lse, spr=P, w=w, gate=gate)
    b = problem(orc, o_bits=np.ascontiguousarray(ob[keep]),
                lse=np.ascontiguousarray(lse[keep]), spr=P - 1, w=w, gate=gate)
    for t in range(S):
        for h in range(H):
            assert np.array_equal(a.latent_bf16(t, h), b.latent_bf16(t, h))
    assert np.array_equal(a.full(), b.full())


def test_all_dead_row_is_exactly_zero(orc):
    rng = np.random.default_rng(8)
    P, S, H = 3, 2, 2
    ob = to_bf16_bits(rng.standard_normal((P, S, H, D)))
    lse = np.full((P, S, H), 1.0, np.float32)
    lse[:, 1, 0] = [-np.inf, np.nan, np.inf]
    ob[:, 1, 0] = 0x7FC0
    pr = problem(orc, o_bits=ob, lse=lse, spr=P)
    assert np.all(pr.latent_f32(1, 0) == 0.0)
    out = pr.full()
    assert np.all(bits_to_f32(out[1, 0:V]) == 0.0)
    assert np.any(bits_to_f32(out[1, V:2 * V]) != 0.0)


def test_padded_rows_are_zero(orc):
    rng = np.random.default_rng(9)
    ob = to_bf16_bits(rng.standard_normal((2, 3, 2, D)))
    lse = rng.standard_normal((2, 3, 2)).astype(np.float32)
    pr = problem(orc, o_bits=ob, lse=lse, spr=2, S_out=5)
    out = pr.full()
    assert out.shape == (5, 2 * V)
    assert np.all(out[3:] == 0)
    assert np.all(np.any(out[:3] != 0, axis=1))


def test_lse_shift_invariance(orc):
    rng = np.random.default_rng(10)
    P = 6
    ob = to_bf16_bits(rng.standard_normal((P, 1, 1, D)))
    lse = (rng.standard_normal((P, 1, 1)) * 3).astype(np.float32)
    base = problem(orc, o_bits=ob, lse=lse, spr=P).latent_f32(0, 0)
    om = np.abs(bits_to_f32(ob[:, 0, 0])).max(0)
    for c in (10.0, -25.0, 300.0):
        got = problem(orc, o_bits=ob, lse=lse + np.float32(c), spr=P).latent_f32(0, 0)
        assert np.all(np.abs(got - base) <= 1e-5 * om + 1e-7)


def test_natural_log_lse(orc):
    # two partials with lse 0 and ln 3 weigh 1/4 and 3/4 (natural-log LSE)
    ob = np.stack([to_bf16_bits(np.full((1, 1, D), 1.0)), to_bf16_bits(np.full((1, 1, D), 2.0))])
    lse = np.array([0.0, math.log(3.0)], np.float32).reshape(2, 1, 1)
    lat = problem(orc, o_bits=ob, lse=lse, spr=2).latent_f32(0, 0)
    assert np.allclose(lat, 1.75, rtol=1e-6)


# ---- up-projection and gate ---------------------------------------------------

def test_bf16_gemm_gate_matches_torch(orc):
    rng = np.random.default_rng(11)
    S, H = 5, 3
    ob = to_bf16_bits(rng.standard_normal((1, S, H, D)))
    w, _ = dummy_weights(H, rng)
    gate = to_bf16_bits(1 / (1 + np.exp(-rng.standard_normal((S, H * V)))))
    out = problem(orc, o_bits=ob, lse=None, spr=0, w=w, gate=gate).full()
    lat = torch.from_numpy(bits_to_f32(ob[0]).copy())                   # [S, H, 512]
    W = torch.from_numpy(bits_to_f32(w).copy())                          # [H, 128, 512]
    acc = torch.einsum("hvk,shk->shv", W, lat).reshape(S, H * V)
    accb = acc.to(torch.bfloat16).float()
    ref = (accb * torch.from_numpy(bits_to_f32(gate).copy())).to(torch.bfloat16).float().numpy()
    got = bits_to_f32(out)
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-6)
    assert np.mean(got == ref) > 0.98


def test_mxfp4_gemm_is_exact_products(orc):
    from mla_decode_attention_lse_gb300 import synth

    rng = np.random.default_rng(12)
    S, H = 4, 2
    ob = to_bf16_bits(rng.standard_normal((1, S, H, D)))
    wf = torch.from_numpy(rng.standard_normal((H, V, D)) / math.sqrt(D)).float()
    codes, scales = (t.numpy() for t in synth.mxfp4_pack_weights(wf))
    gate = to_bf16_bits(1 / (1 + np.exp(-rng.standard_normal((S, H * V)))))
    pr = problem(orc, o_bits=ob, spr=0, w=codes, w_scale=scales, w_fmt=1, gate=gate)
    out = pr.full()
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6])
    c = np.stack([codes & 15, codes >> 4], -1).reshape(H, V, D)
    Wd = grid[c] * np.exp2(np.repeat(scales.astype(np.float64) - 127, BLK, axis=-1))
    for t in range(S):
        for h in range(H):
            lq = []
            for b in range(D // BLK):
                cc, sc = orc.mx_quant_block(ob[0, t, h, b * BLK:(b + 1) * BLK])
                lq.append(grid[cc] * 2.0 ** (sc - 127))
            lq = np.concatenate(lq)
            acc = (Wd[h] @ lq).astype(np.float32)
            ref = bits_to_f32(to_bf16_bits(bits_to_f32(to_bf16_bits(acc))
                                           * bits_to_f32(gate[t, h * V:(h + 1) * V])))
            got = bits_to_f32(out[t, h * V:(h + 1) * V])
            assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


# ---- hand-worked fixtures -----------------------------------------------------

def test_hand_worked_golden(orc):
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        P, S, H = case["P"], case["S"], case["H"]
        o = np.zeros((P, S, H, D), np.float32)
        for r, val in enumerate(case["o_fill"]):
            o[r] = val
        lse = np.array(case["lse"], np.float32).reshape(P, S, H)
        w = np.zeros((H, V, D), np.float32)
        for v in range(V):
            w[:, v, v] = case["w_diag"]
        gate = np.full((S, H * V), case["gate"], np.float32)
        pr = problem(orc, o_bits=to_bf16_bits(o), lse=lse, spr=P, w=to_bf16_bits(w),
                     gate=to_bf16_bits(gate))
        assert np.allclose(pr.latent_f32(0, 0)[:4], case["latent"], rtol=1e-6, atol=0)
        out = bits_to_f32(pr.full())
        assert np.all(out[:, :V] == np.float32(case["core"])), case["name"]
