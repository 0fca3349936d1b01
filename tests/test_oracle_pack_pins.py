"""Pins for the oracle's DCP producer side (stage_push of the vLLM page
"vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"),
independent of the oracle's own code (no GPU): a hand-worked case, the
bijection between source rows and packed rows, and what the masking must do
to the combine downstream (an empty rank contributes nothing, rows past the
batch are zero).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

D, V = 512, 128
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def to_bf16_bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def diag_weights(H):
    w = np.zeros((H, V, D), np.float32)
    for v in range(V):
        w[:, v, v] = 1.0
    return to_bf16_bits(w), to_bf16_bits(np.ones((1, H * V)))


def random_ranks(rng, R, S, H):
    """Every rank's partials over all R*H global heads, and their LSE."""
    o = to_bf16_bits(rng.standard_normal((R, S, R * H, D)))
    lse = (rng.standard_normal((R, S, R * H)) * 2 + 4).astype(np.float32)
    return o, lse


def combine(orc, o, lse, q, H, gate=None, w=None, S_out=None):
    P, S = o.shape[:2]
    if w is None:
        w, g1 = diag_weights(H)
        gate = np.repeat(g1, S, axis=0) if gate is None else gate
    return orc.Problem(o, lse, q, P, w, None, 0, np.ascontiguousarray(gate), S_out).full()


def test_dcp_pack_hand_worked_golden(orc):
    g = json.load(open(os.path.join(GOLDEN, "dcp_pack_hand.json")))
    R, H, S, q, dst = g["R"], g["H"], g["S"], g["q"], g["dst"]
    o = np.empty((R, S, R * H, D), np.uint16)
    lse = np.empty((R, S, R * H), np.float32)
    for r in range(R):
        for t in range(S):
            for gh in range(R * H):
                o[r, t, gh] = to_bf16_bits(16 * r + 4 * t + gh)
                lse[r, t, gh] = 0.5 * (r + 1) + t + 0.125 * gh
    cmb_o, cmb_lse = orc.dcp_pack(o, lse, np.array(g["seq_lens"]), np.array(g["qsl"]), q, dst)
    want_o = to_bf16_bits(np.array(g["cmb_o_fill"], np.float32))
    assert np.array_equal(cmb_o, np.broadcast_to(want_o[:, :, None, None], cmb_o.shape))
    want_lse = np.array([[float(x) for x in row] for row in g["cmb_lse"]], np.float32)[:, :, None]
    assert np.array_equal(cmb_lse, want_lse)
    core = combine(orc, cmb_o, cmb_lse, R, H)  # compact: every token merges the R packed partials
    want_core = to_bf16_bits(np.array(g["core"], np.float32))
    assert np.array_equal(core, np.broadcast_to(want_core[:, None], core.shape))


def test_every_source_row_lands_once(orc):
    # rows carry unique ids; over all destinations every (r, t, g) appears
    # exactly once, at its own rank and token, heads of a destination distinct
    R, H, S, q = 3, 2, 4, 1
    ids = np.arange(R * S * R * H).reshape(R, S, R * H)
    o = np.broadcast_to(to_bf16_bits(ids + 1)[..., None], (R, S, R * H, D)).copy()
    lse = np.zeros((R, S, R * H), np.float32)
    seen = []
    for dst in range(R):
        cmb_o, _ = orc.dcp_pack(o, lse, np.ones((R, S // q), np.int32), np.arange(S // q + 1, dtype=np.int32) * q, q, dst)
        vals = torch.from_numpy(cmb_o[..., 0].view(np.int16)).view(torch.bfloat16).float().numpy().astype(int) - 1
        assert np.all(cmb_o == cmb_o[..., :1])  # whole rows move
        for r in range(R):
            for t in range(S):
                got = vals[r, t]
                assert len(set(got)) == H
                assert all(i // (S * R * H) == r and (i // (R * H)) % S == t for i in got)
        seen.extend(vals.ravel().tolist())
    assert sorted(seen) == list(range(R * S * R * H))


@pytest.mark.parametrize("dst", [0, 2])
def test_empty_rank_contributes_nothing(orc, dst):
    # rank 2 holds no KV of request 1: the packed combine of request 1's tokens
    # equals the combine with rank 2's partial deleted, bit for bit; the other
    # tokens equal the unmasked combine
    rng = np.random.default_rng(7)
    R, H, S, q = 4, 2, 8, 2
    o, lse = random_ranks(rng, R, S, H)
    seq = np.full((R, S // q), 9, np.int32)
    seq[2, 1] = 0
    qsl = np.arange(S // q + 1, dtype=np.int32) * q
    cmb_o, cmb_lse = orc.dcp_pack(o, lse, seq, qsl, q, dst)
    w, g1 = diag_weights(H)
    rw = to_bf16_bits(rng.standard_normal((H, V, D)) / math.sqrt(D))
    gate = to_bf16_bits(1 / (1 + np.exp(-rng.standard_normal((S, H * V)))))
    got = orc.Problem(cmb_o, cmb_lse, q, R, rw, None, 0, gate).full()
    sel = [r for r in range(R) if r != 2]
    heads = slice(dst * H, dst * H + H)
    without = orc.Problem(np.ascontiguousarray(o[sel][:, :, heads]), np.ascontiguousarray(lse[sel][:, :, heads]),
                          q, R - 1, rw, None, 0, gate).full()
    full = orc.Problem(np.ascontiguousarray(o[:, :, heads]), np.ascontiguousarray(lse[:, :, heads]), q, R, rw,
                       None, 0, gate).full()
    req1 = [t for t in range(S) if t // q == 1]
    rest = [t for t in range(S) if t // q != 1]
    assert np.array_equal(got[req1], without[req1])
    assert np.array_equal(got[rest], full[rest])
    assert not np.array_equal(without[req1], full[req1])  # the masked rank did matter


def test_rows_past_the_batch_are_zero(orc):
    rng = np.random.default_rng(8)
    R, H, S, q = 3, 1, 6, 1
    o, lse = random_ranks(rng, R, S, H)
    qsl = np.array([0, 1, 2, 3, 4, 4, 4], np.int32)  # 4 rows live, 2 padding rows
    cmb_o, cmb_lse = orc.dcp_pack(o, lse, np.ones((R, S), np.int32), qsl, q, 1)
    assert np.all(np.isneginf(cmb_lse[:, 4:]))
    assert np.all(np.isfinite(cmb_lse[:, :4]))
    core = combine(orc, cmb_o, cmb_lse, R, H)
    assert np.all(core[4:] == 0) and np.all(np.any(core[:4] != 0, axis=1))


def test_lse_bits_kept_and_mask_is_negative_infinity(orc):
    R, H, S, q = 2, 1, 2, 1
    o = np.zeros((R, S, R * H, D), np.uint16)
    lse_bits = np.full((R, S, R * H), 0x3F800000, np.uint32)
    lse_bits[0, 0, 1] = 0x7FC01234  # a NaN with a payload, in a live row
    lse = lse_bits.view(np.float32)
    seq = np.array([[1, 1], [0, 1]], np.int32)
    _, cmb_lse = orc.dcp_pack(o, lse, seq, np.array([0, 1, 2], np.int32), q, 1)
    bits = cmb_lse.view(np.uint32)
    assert bits[0, 0, 0] == 0x7FC01234
    assert bits[1, 0, 0] == 0xFF800000 and bits[1, 1, 0] == 0x3F800000


def test_pack_rejects_bad_sizes(orc):
    R, H, S = 2, 1, 4
    o = np.zeros((R, S, R * H, D), np.uint16)
    lse = np.zeros((R, S, R * H), np.float32)
    with pytest.raises(ValueError):
        orc.dcp_pack(o, lse, np.ones((R, S), np.int32), np.arange(S + 1, dtype=np.int32), 1, R)
