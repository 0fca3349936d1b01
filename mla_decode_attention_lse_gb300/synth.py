"""Seeded synthetic inputs for the MLA decode post-attention stage.

This module only draws inputs: partial latents ``o``, their log-sum-exp
values ``lse``, the up-projection ``W_V`` (bf16, or MXFP4 codes + E8M0
scales as a checkpoint would store them) and the ``gate``.  It holds none of
the stage's own arithmetic (no LSE merge, no latent rounding or quantisation,
no GEMM), so the CUDA path and the CPU oracle can both take their inputs from
it without sharing any of the computation under test.

Shapes follow the decode workload of the vLLM page
"vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
(12 heads per rank, 512-wide latents, 128-wide V heads; up to 96 heads in the
large multi-token-prediction batch).

The workloads (``WORKLOADS``):

* ``tiny_split``   S=4 (2 requests x q=2), H=2, 2 splits per request, P=4
                   request-major; lse ~N(4,2) with one -inf and one NaN.
* ``nosplit``      P=1, S=64, H=12: lse unused, pure up-projection + gate.
* ``splitkv``      64 requests x q=1, H=12, 16 splits per request, compact
                   [16, 64, 12, 512]; lse ~N(6,3) with 10% -inf.
* ``splitkv_rm``   the same splits in request-major layout, P=1024
                   ([1024, 64, 12, 512]; only 1/64 of it is read, the rest
                   is NaN so that a wrong read shows).
* ``stacked_mxfp4`` 8 stacked shard partials, S=256 live of S_out=264, H=12;
                   lse ~N(4,2) with 5% -inf, 0.1% NaN and 8 (t, h) rows all
                   -inf; MXFP4 W_V.
* ``mtp``          1024 requests x q=4 (S=4096), H=96, 4 splits per request
                   compact; lse ~N(5,2) with 2% -inf; bf16 W_V.
* ``mtp_mxfp4``    the same with MXFP4 W_V.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D = 512   # latent width
V = 128   # V head dim
BLK = 32  # MX block along K

W_BF16 = 0
W_MXFP4 = 1


@dataclass
class Workload:
    name: str
    S: int
    H: int
    P: int
    q: int
    spr: int
    w_fmt: int
    S_out: int | None = None
    lse_mean: float = 0.0
    lse_std: float = 1.0
    neg_inf_frac: float = 0.0
    nan_frac: float = 0.0
    dead_rows: int = 0            # (t, h) rows whose every partial is -inf
    exact_neg_inf: int = 0        # a fixed count of -inf entries (tiny case)
    exact_nan: int = 0            # a fixed count of NaN entries (tiny case)
    lse_unused: bool = False      # P == 1: lse all 0 and ignored
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def out_rows(self) -> int:
        return self.S if self.S_out is None else self.S_out

    @property
    def requests(self) -> int:
        return self.S // self.q


WORKLOADS = {
    "tiny_split": Workload("tiny_split", S=4, H=2, P=4, q=2, spr=2, w_fmt=W_BF16,
                           lse_mean=4.0, lse_std=2.0, exact_neg_inf=1, exact_nan=1, seed=0),
    "nosplit": Workload("nosplit", S=64, H=12, P=1, q=1, spr=0, w_fmt=W_BF16,
                        lse_unused=True, seed=1),
    "splitkv": Workload("splitkv", S=64, H=12, P=16, q=1, spr=16, w_fmt=W_BF16,
                        lse_mean=6.0, lse_std=3.0, neg_inf_frac=0.10, seed=2),
    "splitkv_rm": Workload("splitkv_rm", S=64, H=12, P=1024, q=1, spr=16, w_fmt=W_BF16,
                           lse_mean=6.0, lse_std=3.0, neg_inf_frac=0.10, seed=2),
    "stacked_mxfp4": Workload("stacked_mxfp4", S=256, S_out=264, H=12, P=8, q=1, spr=8,
                              w_fmt=W_MXFP4, lse_mean=4.0, lse_std=2.0, neg_inf_frac=0.05,
                              nan_frac=0.001, dead_rows=8, seed=3),
    "mtp": Workload("mtp", S=4096, H=96, P=4, q=4, spr=4, w_fmt=W_BF16,
                    lse_mean=5.0, lse_std=2.0, neg_inf_frac=0.02, seed=4),
    "mtp_mxfp4": Workload("mtp_mxfp4", S=4096, H=96, P=4, q=4, spr=4, w_fmt=W_MXFP4,
                          lse_mean=5.0, lse_std=2.0, neg_inf_frac=0.02, seed=4),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype=torch.float32):
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def mxfp4_pack_weights(w: torch.Tensor):
    """Store float weights [H, 128, 512] in the MXFP4 checkpoint format.

    Data preparation only (it is the weight file's format, not a step of the
    stage): each 32-wide block along K gets the smallest power-of-two scale
    that fits its largest magnitude into 6 (so nothing clips), and each
    element takes the nearest E2M1 magnitude, ties away from zero.  Returns
    (codes u8 [H, 128, 256], element 2i in the low nibble of byte i;
    scales u8 [H, 128, 16], E8M0).
    """
    H, Vr, K = w.shape
    blocks = w.float().reshape(H, Vr, K // BLK, BLK)
    amax = blocks.abs().amax(-1)
    # smallest e with amax / 2^e <= 6  ->  e = ceil(log2(amax / 6))
    e = torch.ceil(torch.log2(torch.clamp(amax, min=1e-30) / 6.0))
    e = torch.clamp(e, -126, 127)
    e = torch.where(amax > 0, e, torch.full_like(e, -126))
    scaled = blocks / torch.exp2(e).unsqueeze(-1)
    # midpoints between neighbouring E2M1 magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6;
    # a magnitude at or past a midpoint takes the larger neighbour
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], device=w.device)
    mag = scaled.abs()
    best = (mag.unsqueeze(-1) >= mids).sum(-1)
    codes = best.to(torch.uint8) | ((scaled < 0) & (best > 0)).to(torch.uint8) * 8
    codes = codes.reshape(H, Vr, K)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    scales = (e + 127).to(torch.uint8)
    return packed.contiguous(), scales.contiguous()


def make(wl: Workload | str, device="cpu", seed: int | None = None, w_fmt: int | None = None):
    """Draw one workload's inputs on ``device``.

    Returns a dict of tensors: o [P, S, H, 512] bf16, lse [P, S, H] f32 (or
    None when P == 1 and lse is unused), w_v, w_scale (None for bf16 W_V),
    gate [S, H*128] bf16, plus the integer parameters.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    seed = wl.seed if seed is None else seed
    w_fmt = wl.w_fmt if w_fmt is None else w_fmt
    g = _gen(device, seed)
    S, H, P = wl.S, wl.H, wl.P

    request_major = P > 1 and P != wl.spr
    if request_major and (S % wl.q != 0 or P != (S // wl.q) * wl.spr):
        # the layouts of mla_combine_uv: P == 1, P == spr, or P == (S / q) * spr
        raise ValueError(f"P={P} is none of the layouts for S={S}, q={wl.q}, spr={wl.spr}")
    if request_major:
        # only token t's request's splits are ever read; everything else NaN
        o = torch.full((P, S, H, D), float("nan"), device=device, dtype=torch.bfloat16)
        lse = torch.full((P, S, H), float("nan"), device=device, dtype=torch.float32)
        live_o = _normal((wl.spr, S, H, D), 1.0, g, device, torch.bfloat16)
        live_l = _normal((wl.spr, S, H), wl.lse_std, g, device) + wl.lse_mean
        t = torch.arange(S, device=device)
        for j in range(wl.spr):
            r = (t // wl.q) * wl.spr + j
            o[r, t] = live_o[j]
            lse[r, t] = live_l[j]
        sel_mask = torch.zeros((P, S, H), dtype=torch.bool, device=device)
        for j in range(wl.spr):
            sel_mask[(t // wl.q) * wl.spr + j, t] = True
    else:
        o = _normal((P, S, H, D), 1.0, g, device, torch.bfloat16)
        if wl.lse_unused:
            lse = torch.zeros((P, S, H), device=device, dtype=torch.float32)
        else:
            lse = _normal((P, S, H), wl.lse_std, g, device) + wl.lse_mean
        sel_mask = torch.ones((P, S, H), dtype=torch.bool, device=device)

    if P > 1:
        live_idx = sel_mask.flatten().nonzero().flatten()
        n_live = live_idx.numel()
        flat = lse.view(-1)
        if wl.neg_inf_frac > 0:
            u = torch.rand(n_live, generator=g, device=device)
            flat[live_idx[u < wl.neg_inf_frac]] = float("-inf")
        if wl.nan_frac > 0:
            u = torch.rand(n_live, generator=g, device=device)
            flat[live_idx[u < wl.nan_frac]] = float("nan")
        if wl.exact_neg_inf or wl.exact_nan:
            perm = torch.randperm(n_live, generator=g, device=device)
            k1, k2 = wl.exact_neg_inf, wl.exact_nan
            flat[live_idx[perm[:k1]]] = float("-inf")
            flat[live_idx[perm[k1:k1 + k2]]] = float("nan")
        if wl.dead_rows:
            perm = torch.randperm(S * H, generator=g, device=device)[: wl.dead_rows]
            for i in perm.tolist():
                t, h = divmod(i, H)
                lse[sel_mask[:, t, h], t, h] = float("-inf")
    else:
        lse = None if wl.lse_unused else lse

    w = _normal((H, V, D), 1.0 / math.sqrt(D), g, device)
    if w_fmt == W_BF16:
        w_v, w_scale = w.to(torch.bfloat16).contiguous(), None
    else:
        w_v, w_scale = mxfp4_pack_weights(w)
    gate = torch.sigmoid(_normal((S, H * V), 1.0, g, device)).to(torch.bfloat16).contiguous()
    return dict(o=o, lse=lse, w_v=w_v, w_scale=w_scale, gate=gate, S=S, S_out=wl.out_rows,
                H=H, P=P, q=wl.q, spr=wl.spr, w_fmt=w_fmt, name=wl.name)


def custom(S, H, P, q, spr, w_fmt, S_out=None, seed=0, device="cpu", lse_mean=4.0,
           lse_std=2.0, neg_inf_frac=0.0, nan_frac=0.0, dead_rows=0, lse_unused=False):
    """A workload of any shape with the same recipe (for edge-case tests)."""
    wl = Workload("custom", S=S, H=H, P=P, q=q, spr=spr, w_fmt=w_fmt, S_out=S_out,
                  lse_mean=lse_mean, lse_std=lse_std, neg_inf_frac=neg_inf_frac,
                  nan_frac=nan_frac, dead_rows=dead_rows, lse_unused=lse_unused, seed=seed)
    return make(wl, device=device)


@dataclass
class DcpWorkload:
    """Decode context parallelism over R ranks, all resident on one GPU: every
    rank's attention partials over all R*H global heads, its local KV lengths
    per request (some requests empty on some ranks), the query start
    locations (rows past ``live`` are padding), and destination rank ``dst``'s
    W_V heads and gate."""
    name: str
    R: int
    S: int
    live: int
    H: int
    q: int
    w_fmt: int
    lse_mean: float = 4.0
    lse_std: float = 2.0
    empty_frac: float = 0.05
    dst: int = 0
    seed: int = 0


DCP_WORKLOADS = {
    # 8 ranks x 12 heads (96 global), a decode batch of 264 rows of which 256
    # are live, MXFP4 W_V: the stacked case pushed from its 8 ranks
    "dcp8_mxfp4": DcpWorkload("dcp8_mxfp4", R=8, S=264, live=256, H=12, q=1, w_fmt=W_MXFP4,
                              empty_frac=0.05, seed=11),
}


def make_dcp(wl: DcpWorkload | str, device="cpu", seed: int | None = None, w_fmt: int | None = None):
    """Draw a DCP workload: o_all [R, S, R*H, 512] bf16, lse_all [R, S, R*H]
    f32, seq_lens [R, S/q] int32 (0 = empty), qsl [S/q + 1] int32, and W_V,
    its scales and the gate [S, H*128] of the destination's H heads."""
    if isinstance(wl, str):
        wl = DCP_WORKLOADS[wl]
    seed = wl.seed if seed is None else seed
    w_fmt = wl.w_fmt if w_fmt is None else w_fmt
    g = _gen(device, seed)
    R, S, H, q = wl.R, wl.S, wl.H, wl.q
    nreq = S // q
    o_all = _normal((R, S, R * H, D), 1.0, g, device, torch.bfloat16)
    lse_all = _normal((R, S, R * H), wl.lse_std, g, device) + wl.lse_mean
    seq_lens = torch.randint(1, 4097, (R, nreq), generator=g, device=device, dtype=torch.int32)
    u = torch.rand((R, nreq), generator=g, device=device)
    seq_lens[u < wl.empty_frac] = 0
    j = torch.arange(nreq + 1, device=device, dtype=torch.int32)
    qsl = torch.clamp(j * q, max=wl.live).to(torch.int32)
    w = _normal((H, V, D), 1.0 / math.sqrt(D), g, device)
    if w_fmt == W_BF16:
        w_v, w_scale = w.to(torch.bfloat16).contiguous(), None
    else:
        w_v, w_scale = mxfp4_pack_weights(w)
    gate = torch.sigmoid(_normal((S, H * V), 1.0, g, device)).to(torch.bfloat16).contiguous()
    return dict(o_all=o_all, lse_all=lse_all, seq_lens=seq_lens, qsl=qsl, w_v=w_v, w_scale=w_scale,
                gate=gate, R=R, S=S, S_out=S, H=H, q=q, dst=wl.dst, live=wl.live, w_fmt=w_fmt,
                name=wl.name)


def dcp_pack_bytes(inp) -> int:
    """Bytes the pack must move: every packed row (1 KiB) and its LSE, read and
    written, plus the request lengths and query starts it reads."""
    R, S, H, q = inp["R"], inp["S"], inp["H"], inp["q"]
    rows = R * S * H
    return 2 * rows * (D * 2 + 4) + R * (S // q) * 4 + (S // q + 1) * 4


def algorithmic_bytes(inp) -> int:
    """Bytes the stage must move: every partial row with a finite sanitised
    LSE (the rows whose weight can be non-zero; P == 1 reads every row), all
    selected LSE values, W_V (and its scales), the gate rows and the output."""
    S, S_out, H, P, q, spr = (inp[k] for k in ("S", "S_out", "H", "P", "q", "spr"))
    if P == 1:
        rows = S * H
        lse_bytes = 0
    else:
        lse = inp["lse"]
        n_sel = (S * H * spr)
        fin = torch.isfinite(lse) & (lse < float("inf"))
        if P != spr:  # request-major: only the selected entries count
            t = torch.arange(S, device=lse.device)
            cnt = 0
            for j in range(spr):
                cnt += int(fin[(t // q) * spr + j, t].sum())
            rows = cnt
        else:
            rows = int(fin.sum())
        lse_bytes = 4 * n_sel
    wv = inp["w_v"].numel() * inp["w_v"].element_size()
    if inp["w_scale"] is not None:
        wv += inp["w_scale"].numel()
    return rows * D * 2 + lse_bytes + wv + S * H * V * 2 + S_out * H * V * 2


def algorithmic_bytes_all_rows(inp) -> int:
    """The same count with every selected partial row (live or dead): per
    (t, h) the token's partials (1 KiB + a 4-byte LSE each; P == 1 reads one
    row and no LSE), plus W_V (and its scales), the gate and the output."""
    S, S_out, H, P, spr = (inp[k] for k in ("S", "S_out", "H", "P", "spr"))
    n = 1 if P == 1 else spr
    per_row = D * 2 + (0 if P == 1 else 4)
    wv = inp["w_v"].numel() * inp["w_v"].element_size()
    if inp["w_scale"] is not None:
        wv += inp["w_scale"].numel()
    return S * H * n * per_row + wv + S * H * V * 2 + S_out * H * V * 2


def flops(inp) -> int:
    return 2 * inp["S"] * inp["H"] * V * D


# ---- inputs of the partial producer (split-KV MLA decode attention) -------

@dataclass(frozen=True)
class AttnWorkload:
    """One decode step's attention inputs: B requests of q new tokens, H heads,
    spr splits per request, a cache tensor of Lmax positions per request.
    Request lengths: a fraction ``short_frac`` of the requests is short
    (1 .. 4 * spr positions, which leaves some of its splits empty), the rest
    lies between Lmax / 2 and Lmax."""
    name: str
    B: int
    q: int
    H: int
    spr: int
    Lmax: int
    short_frac: float = 0.1
    seed: int = 0


ATTN_WORKLOADS = {
    # the 16-split decode step of the combine's workloads, produced from a
    # cache of up to 4096 positions per request
    "attn_splitkv": AttnWorkload("attn_splitkv", B=64, q=1, H=12, spr=16, Lmax=4096, short_frac=0.1, seed=21),
}

ATTN_K = D + 64  # latent then rope


def attn_scale() -> float:
    """Softmax scale of the MLA heads: 1 / sqrt(128 + 64), the query-key head
    width before W_UK is absorbed."""
    return 1.0 / math.sqrt(192.0)


def make_attn(wl: AttnWorkload | str, device="cpu", seed: int | None = None):
    """Draw one attention workload's inputs on ``device``: qv [B q, H, 576]
    and kv [B, Lmax, 576] bf16 ~N(0, 1), kv_len [B] int32.  Cached rows past a
    request's length are NaN, so a kernel that reads them shows it."""
    if isinstance(wl, str):
        wl = ATTN_WORKLOADS[wl]
    seed = wl.seed if seed is None else seed
    g = _gen(device, seed)
    S = wl.B * wl.q
    qv = _normal((S, wl.H, ATTN_K), 1.0, g, device, torch.bfloat16)
    kv = _normal((wl.B, wl.Lmax, ATTN_K), 1.0, g, device, torch.bfloat16)
    long_len = torch.randint(wl.Lmax // 2, wl.Lmax + 1, (wl.B,), generator=g, device=device, dtype=torch.int32)
    short_len = torch.randint(1, min(4 * wl.spr, wl.Lmax) + 1, (wl.B,), generator=g, device=device,
                              dtype=torch.int32)
    short = torch.rand(wl.B, generator=g, device=device) < wl.short_frac
    kv_len = torch.where(short, short_len, long_len).to(torch.int32).contiguous()
    past = torch.arange(wl.Lmax, device=device)[None, :] >= kv_len[:, None].long()
    kv[past] = float("nan")
    # the combine that follows: bf16 W_V ~N(0, 1/sqrt(512)), gate sigmoid(N(0, 1))
    w_v = _normal((wl.H, V, D), 1.0 / math.sqrt(D), g, device, torch.bfloat16)
    gate = torch.sigmoid(_normal((S, wl.H * V), 1.0, g, device)).to(torch.bfloat16).contiguous()
    return dict(qv=qv, kv=kv, kv_len=kv_len, q=wl.q, spr=wl.spr, scale=attn_scale(), B=wl.B, H=wl.H,
                Lmax=wl.Lmax, wl=wl, w_v=w_v, w_fmt=W_BF16, w_scale=None, gate=gate)


def attn_bytes(inp) -> int:
    """Algorithmic bytes of one attention call: the cached rows inside the
    requests' lengths (576 bf16 each, once), the query rows, and the o / lse
    partials written."""
    B, q, H, spr = inp["B"], inp["q"], inp["H"], inp["spr"]
    rows = int(inp["kv_len"].long().sum())
    S = B * q
    return rows * ATTN_K * 2 + S * H * ATTN_K * 2 + spr * S * H * (D * 2 + 4)


# ---- inputs of the downstream o_proj shard ---------------------------------

@dataclass(frozen=True)
class OprojWorkload:
    """One rank's o_proj shard: S tokens of core (K = H * 128 wide) times the
    rank's weight slice [Nout, K]."""
    name: str
    S: int
    K: int
    Nout: int
    seed: int = 0


OPROJ_WORKLOADS = {
    # the decode step: 64 tokens, 12 heads per rank (K = 1536), 7168 outputs
    "oproj_decode": OprojWorkload("oproj_decode", S=64, K=12 * V, Nout=7168, seed=31),
}


def make_oproj(wl: OprojWorkload | str, device="cpu", seed: int | None = None):
    """core rows x ~ sigmoid(N(0,1)) * N(0,1) (a gated latent) and the weight
    W ~ N(0, 1/sqrt(K)), both bf16."""
    if isinstance(wl, str):
        wl = OPROJ_WORKLOADS[wl]
    seed = wl.seed if seed is None else seed
    g = _gen(device, seed)
    x = (_normal((wl.S, wl.K), 1.0, g, device) * torch.sigmoid(_normal((wl.S, wl.K), 1.0, g, device)))
    x = x.to(torch.bfloat16).contiguous()
    w = _normal((wl.Nout, wl.K), 1.0 / math.sqrt(wl.K), g, device, torch.bfloat16)
    return dict(x=x, w=w, S=wl.S, K=wl.K, Nout=wl.Nout, wl=wl)


def oproj_bytes(inp) -> int:
    """Algorithmic bytes of one o_proj call: the weight, the core rows, the output."""
    return 2 * (inp["Nout"] * inp["K"] + inp["S"] * inp["K"] + inp["S"] * inp["Nout"])
