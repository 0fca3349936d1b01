"""Pins for the oracle's o_proj shard (the linear layer that takes the core
rows of the vLLM page "vllm.models.kimi_k3.amd.specialized_decode.mono.
attention.mla_back", whose stage ends at "o_proj's input"), against things
other than the oracle's own code (no GPU): PyTorch's float64 matmul, an
identity weight, a permutation, and additivity over the input features."""
import numpy as np
import torch


def bits(x) -> np.ndarray:
    return torch.as_tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def value(b) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double()


def test_equals_library_matmul(orc):
    rng = np.random.default_rng(1)
    x, w = bits(rng.standard_normal((5, 96))), bits(rng.standard_normal((40, 96)) / 10)
    got = orc.o_proj(x, w)
    ref = (value(x) @ value(w).T).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_identity_and_permutation_weights(orc):
    rng = np.random.default_rng(2)
    x = bits(rng.standard_normal((3, 64)))
    assert np.array_equal(orc.o_proj(x, bits(np.eye(64))), x)
    perm = rng.permutation(64)
    assert np.array_equal(orc.o_proj(x, bits(np.eye(64)[perm])), x[:, perm])


def test_additive_over_input_features(orc):
    # small integers: every partial sum exact, so splitting K changes nothing
    rng = np.random.default_rng(3)
    x = bits(rng.integers(-4, 5, (4, 128)))
    w = bits(rng.integers(-4, 5, (16, 128)))
    whole = value(orc.o_proj(x, w))
    lo, hi = value(orc.o_proj(x[:, :64].copy(), w[:, :64].copy())), value(orc.o_proj(x[:, 64:].copy(), w[:, 64:].copy()))
    assert torch.equal(whole, lo + hi)


def test_strided_rows(orc):
    rng = np.random.default_rng(4)
    xb = bits(rng.standard_normal((3, 80)))
    x = xb[:, :64]
    w = bits(rng.standard_normal((8, 64)))
    assert np.array_equal(orc.o_proj(x, w), orc.o_proj(np.ascontiguousarray(x), w))
