"""Pins for the oracle's partial producer (split-KV MLA decode attention in
the absorbed form: the page's M1c, whose partials the combine of the vLLM
page "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
merges), each against something other than the oracle's own code (no GPU):
PyTorch's scaled_dot_product_attention and logsumexp in float64, a closed
form for how the splits partition the positions, the flash-decoding merge
identity, a dominant key, and invariance of o under a shift of every score.
"""
import math

import numpy as np
import pytest
import torch

D, R = 512, 64


def bits(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def value(b) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double()


def rand_problem(rng, B, q, H, Lmax, lens):
    qv = bits(rng.standard_normal((B * q, H, D + R)) * 0.3)
    kv = bits(rng.standard_normal((B, Lmax, D + R)))
    return qv, kv, np.array(lens, np.int32)


def sdpa(qv, kv, lens, q, scale):
    """Library attention in float64, token i of a request seeing the
    positions below len - (q - 1 - i); o as bf16 bits, lse as float."""
    S, H, _ = qv.shape
    o = np.zeros((S, H, D), np.uint16)
    lse = np.full((S, H), -np.inf)
    for b, L in enumerate(lens):
        if L == 0:
            continue
        Q = value(qv[b * q:(b + 1) * q]).permute(1, 0, 2)  # [H, q, 576]
        K = value(kv[b, :L]).expand(H, L, D + R)
        Vv = value(kv[b, :L, :D]).expand(H, L, D)
        vis = np.array([L - (q - 1 - i) for i in range(q)])
        mask = torch.from_numpy(np.arange(L)[None, :] < vis[:, None])  # [q, L]
        out = torch.nn.functional.scaled_dot_product_attention(Q, K, Vv, attn_mask=mask, scale=scale)
        scores = (Q @ K.transpose(1, 2)) * scale
        ls = torch.logsumexp(scores.masked_fill(~mask, -math.inf), dim=-1)  # [H, q]
        for i in range(q):
            if vis[i] <= 0:
                continue
            o[b * q + i] = out[:, i].float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            lse[b * q + i] = ls[:, i].numpy()
    return o, lse


@pytest.mark.parametrize("q,lens", [(1, [7, 13, 1]), (3, [9, 4, 3])])
def test_one_split_is_library_attention(orc, q, lens):
    rng = np.random.default_rng(20 + q)
    H, scale = 3, 1 / math.sqrt(D + R)
    qv, kv, lens = rand_problem(rng, len(lens), q, H, 16, lens)
    o, lse = orc.mla_attn_split(qv, kv, lens, q, 1, scale)
    ref_o, ref_lse = sdpa(qv, kv, lens, q, scale)
    assert np.array_equal(o[0], ref_o)
    assert np.allclose(lse[0], ref_lse.astype(np.float32), rtol=1e-6, atol=1e-6)


def test_masked_positions_are_never_read(orc):
    # positions past what a token sees (and past kv_len) may hold anything
    rng = np.random.default_rng(5)
    q, H = 3, 2
    qv, kv, lens = rand_problem(rng, 2, q, H, 12, [8, 5])
    o1, l1 = orc.mla_attn_split(qv, kv, lens, q, 2, 0.05)
    kv2 = kv.copy()
    kv2[0, 6:] = bits(np.full((6, D + R), 1e4))  # token 0 of request 0 sees 0..5
    kv2[1, 5:] = 0x7FC0  # NaN past kv_len
    o2, l2 = orc.mla_attn_split(qv, kv2, lens, q, 2, 0.05)
    assert np.array_equal(o1[:, 0], o2[:, 0]) and np.array_equal(l1[:, 0], l2[:, 0])
    assert np.array_equal(o1[:, q:], o2[:, q:]) and np.array_equal(l1[:, q:], l2[:, q:])
    assert not np.array_equal(o1[:, 1], o2[:, 1])  # token 1 sees position 6


@pytest.mark.parametrize("L,q,spr", [(0, 1, 4), (1, 1, 4), (5, 1, 4), (13, 2, 4), (64, 3, 16), (100, 1, 3)])
def test_split_partition_closed_form(orc, L, q, spr):
    # all scores 0 and latent row j = e_j: split r's o is 1/n on its own
    # positions and 0 elsewhere, its lse ln(n); an empty split is (-inf, 0)
    H = 2
    qv = np.zeros((q, H, D + R), np.uint16)
    kv = np.zeros((1, max(L, 1), D + R), np.float32)
    for j in range(L):
        kv[0, j, j] = 1.0
    o, lse = orc.mla_attn_split(qv, bits(kv), np.array([L], np.int32), q, spr, 0.1)
    C = -(-L // spr)
    for i in range(q):
        vis = max(L - (q - 1 - i), 0)
        for r in range(spr):
            j0, j1 = r * C, min((r + 1) * C, vis)
            n = max(j1 - j0, 0)
            want = np.zeros(D, np.float32)
            if n:
                want[j0:j1] = 1.0 / n
                assert lse[r, i, 0] == np.float32(math.log(n)) and lse[r, i, 1] == lse[r, i, 0]
            else:
                assert lse[r, i, 0] == -np.inf
            assert np.array_equal(o[r, i, 0], bits(want)) and np.array_equal(o[r, i, 1], bits(want))


def test_flash_decoding_identity(orc):
    # the splits, merged exactly with their LSEs, give the unsplit attention
    rng = np.random.default_rng(9)
    q, H, spr = 2, 3, 5
    qv, kv, lens = rand_problem(rng, 3, q, H, 40, [40, 23, 6])
    o1, l1 = orc.mla_attn_split(qv, kv, lens, q, 1, 0.06)
    os_, ls = orc.mla_attn_split(qv, kv, lens, q, spr, 0.06)
    L = torch.logsumexp(torch.from_numpy(ls.astype(np.float64)), dim=0).numpy()
    assert np.allclose(L, l1[0], rtol=1e-6, atol=1e-6)
    w = np.exp(ls.astype(np.float64) - L[None])  # 0 for empty splits
    merged = np.einsum("rsh,rshd->shd", w, value(os_).numpy())
    assert np.allclose(merged, value(o1[0]).numpy(), atol=1e-2)
    assert np.isinf(ls).any()  # request 2 leaves empty splits


def test_dominant_key(orc):
    rng = np.random.default_rng(3)
    H, L = 2, 9
    qv, kv, lens = rand_problem(rng, 1, 1, H, L, [L])
    qd = np.zeros((1, H, D + R), np.float32)
    qd[0, :, D] = 1.0  # rope query picks the first rope coordinate
    kd = value(kv).float().numpy()
    kd[0, :, D] = 0.0
    kd[0, 4, D] = 16.0  # position 4: score 16 * scale above the rest
    o, lse = orc.mla_attn_split(bits(qd), bits(kd), lens, 1, 1, 8.0)
    assert np.array_equal(o[0, 0, 0], bits(kd[0, 4, :D])) and np.array_equal(o[0, 0, 1], o[0, 0, 0])
    assert lse[0, 0, 0] == np.float32(128.0)


def test_score_shift_leaves_o(orc):
    # a rope coordinate equal for every position adds the same constant to
    # every score: o is unchanged, lse moves by that constant
    rng = np.random.default_rng(4)
    H, L = 2, 11
    qv, kv, lens = rand_problem(rng, 1, 1, H, L, [L])
    qd, kd = value(qv).float().numpy(), value(kv).float().numpy()
    qd[0, :, D + R - 1], kd[0, :, D + R - 1] = 0.0, 1.0
    o1, l1 = orc.mla_attn_split(bits(qd), bits(kd), lens, 1, 3, 0.125)
    qd[0, :, D + R - 1] = 2.0
    o2, l2 = orc.mla_attn_split(bits(qd), bits(kd), lens, 1, 3, 0.125)
    assert np.array_equal(o1, o2)
    assert np.allclose(l2 - l1, 0.25, atol=1e-5)


def test_rejects_bad_sizes(orc):
    qv = np.zeros((2, 1, D + R), np.uint16)
    kv = np.zeros((1, 4, D + R), np.uint16)
    with pytest.raises(ValueError):
        orc.mla_attn_split(qv, kv, np.array([-1], np.int32), 2, 1, 1.0)
