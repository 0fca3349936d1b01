"""Shared helpers of the parity tests: inputs to the oracle, the GPU call
through the C ABI, and the element-wise comparison.

Tolerance (the bar the stage is held to): |gpu - oracle| <= 1e-2 + 1e-2 *
|oracle| element-wise for both W_V formats; rows the definition zeroes
(every partial dead, or t >= S) must be exactly zero; outputs past S_out must
stay untouched.
"""
import numpy as np
import torch

V = 128
ATOL = 1e-2
RTOL = 1e-2
CANARY = 0x7E5A  # a bf16 NaN pattern the kernels never write


def to_np16(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def host_inputs(inp):
    """numpy copies of a workload's tensors, strides kept (for the oracle)."""
    import oracle

    return oracle.host_arrays(inp)


def oracle_problem(orc, inp, host=None):
    return orc.problem_from_tensors(inp, host)


def dead_rows(inp):
    """(t, h) rows whose every merged partial has a non-finite-or-+inf LSE."""
    S, H, P, q, spr = (inp[k] for k in ("S", "H", "P", "q", "spr"))
    if P == 1:
        return np.zeros((S, H), bool)
    lse = inp["lse"].detach().cpu()
    live = torch.isfinite(lse)  # NaN, +inf and -inf all sanitise to -inf
    if P == spr:
        return (~live.any(0)).numpy()
    t = torch.arange(S)
    acc = torch.zeros(S, H, dtype=torch.bool)
    for j in range(spr):
        acc |= live[(t // q) * spr + j, t]
    return (~acc).numpy()


def run_gpu(inp, kernel=0, tile=0, extra_rows=2, stream=None):
    """Call the library through the C ABI; returns (out bits, canary rows)."""
    import mla_decode_attention_lse_gb300 as m

    dev = inp["o"].device
    W = inp["H"] * V
    S_out = inp["S_out"]
    buf = torch.full((S_out + extra_rows, W), 0, dtype=torch.int16, device=dev)
    buf.fill_(CANARY)
    out = buf[:S_out].view(torch.bfloat16)
    m.mla_combine_uv(inp["o"], inp["lse"], inp["q"], inp["spr"], inp["w_v"], inp["w_fmt"],
                     inp["gate"], out, w_scale=inp["w_scale"], kernel=kernel, tile_tokens=tile,
                     stream=stream)
    st = m.mla_combine_uv_status(stream)
    assert st == m.MLA_OK, m.mla_status_str(st)
    full = buf.cpu().numpy().view(np.uint16)
    return full[:S_out], full[S_out:]


def compare(gpu_bits, ref_bits, zero_mask_rows=None, what=""):
    """Element-wise check; returns (max abs err, max rel err)."""
    g = bits_to_f32(gpu_bits).astype(np.float64)
    r = bits_to_f32(ref_bits).astype(np.float64)
    assert g.shape == r.shape
    nan_r, nan_g = np.isnan(r), np.isnan(g)
    assert np.array_equal(nan_r, nan_g), f"{what}: NaN positions differ ({nan_g.sum()} vs {nan_r.sum()})"
    inf_r, inf_g = np.isinf(r), np.isinf(g)
    assert np.array_equal(inf_r, inf_g) and np.array_equal(r[inf_r], g[inf_g]), f"{what}: infinities differ"
    ok = ~(nan_r | inf_r)
    err = np.abs(g[ok] - r[ok])
    bound = ATOL + RTOL * np.abs(r[ok])
    bad = err > bound
    if bad.any():
        idx = np.argwhere(ok)[np.argmax(err - bound)]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; worst at {tuple(idx)}: "
                             f"gpu {g[tuple(idx)]} oracle {r[tuple(idx)]}")
    if zero_mask_rows is not None:
        z = g[zero_mask_rows]
        assert np.all(z == 0.0), f"{what}: masked rows not exactly zero"
    rel = err / np.maximum(np.abs(r[ok]), 1e-6)
    return float(err.max(initial=0.0)), float(rel.max(initial=0.0))


def seg_mask(inp):
    """Boolean [S_out, H*128] of outputs that must be exactly zero."""
    S, S_out, H = inp["S"], inp["S_out"], inp["H"]
    mask = np.zeros((S_out, H * V), bool)
    mask[S:] = True
    dr = dead_rows(inp)
    for t, h in zip(*np.nonzero(dr)):
        mask[t, h * V:(h + 1) * V] = True
    return mask
