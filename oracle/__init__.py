"""CPU oracle for the MLA decode post-attention stage (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it.

The arithmetic lives in ``mla_oracle.c`` (plain single-threaded C, fp32 as
the vLLM page "vllm.models.kimi_k3.amd.specialized_decode.mono.attention.
mla_back" fixes it).  This module only compiles it with gcc and marshals
numpy arrays into it.  bf16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_HDR = os.path.join(_HERE, "mla_oracle.h")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

D, V, BLK = 512, 128, 32


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fused multiply-add: one rounding per op)."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < newest:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True, cwd=_HERE)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Args(ctypes.Structure):
    _fields_ = [
        ("S", ctypes.c_int), ("S_out", ctypes.c_int), ("H", ctypes.c_int),
        ("P", ctypes.c_int), ("q", ctypes.c_int), ("spr", ctypes.c_int),
        ("o", ctypes.c_void_p), ("o_sp", ctypes.c_int64), ("o_st", ctypes.c_int64),
        ("o_sh", ctypes.c_int64),
        ("lse", ctypes.c_void_p), ("l_sp", ctypes.c_int64), ("l_st", ctypes.c_int64),
        ("l_sh", ctypes.c_int64),
        ("w_v", ctypes.c_void_p), ("w_sh", ctypes.c_int64), ("w_sv", ctypes.c_int64),
        ("w_scale", ctypes.c_void_p), ("s_sh", ctypes.c_int64), ("s_sv", ctypes.c_int64),
        ("w_fmt", ctypes.c_int),
        ("gate", ctypes.c_void_p),
    ]


class _PackArgs(ctypes.Structure):
    _fields_ = [
        ("S", ctypes.c_int), ("H", ctypes.c_int), ("R", ctypes.c_int), ("q", ctypes.c_int),
        ("dst", ctypes.c_int),
        ("o", ctypes.c_void_p), ("o_sr", ctypes.c_int64), ("o_st", ctypes.c_int64),
        ("o_sh", ctypes.c_int64),
        ("lse", ctypes.c_void_p), ("l_sr", ctypes.c_int64), ("l_st", ctypes.c_int64),
        ("l_sh", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p), ("sl_sr", ctypes.c_int64),
        ("qsl", ctypes.c_void_p),
    ]


class _AttnArgs(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("q", ctypes.c_int), ("H", ctypes.c_int), ("spr", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("qv", ctypes.c_void_p), ("q_st", ctypes.c_int64), ("q_sh", ctypes.c_int64),
        ("kv", ctypes.c_void_p), ("kv_sb", ctypes.c_int64), ("kv_sl", ctypes.c_int64),
        ("kv_len", ctypes.c_void_p),
    ]


class _OprojArgs(ctypes.Structure):
    _fields_ = [
        ("S", ctypes.c_int), ("K", ctypes.c_int), ("Nout", ctypes.c_int),
        ("x", ctypes.c_void_p), ("x_st", ctypes.c_int64),
        ("w", ctypes.c_void_p), ("w_sj", ctypes.c_int64),
    ]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.POINTER
            L.orc_bf16_to_f32.restype = ctypes.c_float
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f32_to_bf16.restype = ctypes.c_uint16
            L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            L.orc_e2m1_value.restype = ctypes.c_float
            L.orc_e2m1_value.argtypes = [ctypes.c_int]
            L.orc_e8m0_value.restype = ctypes.c_float
            L.orc_e8m0_value.argtypes = [ctypes.c_int]
            L.orc_e2m1_code.restype = ctypes.c_int
            L.orc_e2m1_code.argtypes = [ctypes.c_float]
            L.orc_mx_scale_code.restype = ctypes.c_int
            L.orc_mx_scale_code.argtypes = [ctypes.c_void_p]
            L.orc_mx_quant_block.restype = None
            L.orc_mx_quant_block.argtypes = [ctypes.c_void_p, ctypes.c_void_p, P(ctypes.c_int)]
            L.orc_sane.restype = ctypes.c_float
            L.orc_sane.argtypes = [ctypes.c_float]
            L.orc_partial_set.restype = ctypes.c_int
            L.orc_partial_set.argtypes = [ctypes.c_int] * 5 + [P(ctypes.c_int), P(ctypes.c_int)]
            for name in ("orc_combine_latent", "orc_latent_bf16", "orc_row"):
                f = getattr(L, name)
                f.restype = ctypes.c_int
                f.argtypes = [P(_Args), ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
            L.orc_rows.restype = ctypes.c_int
            L.orc_rows.argtypes = [P(_Args), ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p]
            L.orc_mla_combine_uv.restype = ctypes.c_int
            L.orc_mla_combine_uv.argtypes = [P(_Args), ctypes.c_void_p]
            L.orc_dcp_pack.restype = ctypes.c_int
            L.orc_dcp_pack.argtypes = [P(_PackArgs), ctypes.c_void_p, ctypes.c_void_p]
            L.orc_mla_attn_split.restype = ctypes.c_int
            L.orc_mla_attn_split.argtypes = [P(_AttnArgs), ctypes.c_void_p, ctypes.c_void_p]
            L.orc_o_proj.restype = ctypes.c_int
            L.orc_o_proj.argtypes = [P(_OprojArgs), ctypes.c_void_p]
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _estrides(a):
    return [s // a.itemsize for s in a.strides]


class Problem:
    """One call's inputs as numpy arrays (kept alive while the oracle runs).

    o       uint16 [P, S, H, 512] (bf16 bits; any strides, last dim contiguous)
    lse     float32 [P, S, H] or None (allowed only when P == 1)
    w_v     uint16 [H, 128, 512] (w_fmt 0) or uint8 [H, 128, 256] (w_fmt 1)
    w_scale uint8 [H, 128, 16] (w_fmt 1)
    gate    uint16 [S, H*128] dense
    """

    def __init__(self, o, lse, q, spr, w_v, w_scale, w_fmt, gate, S_out=None):
        self.o, self.lse, self.w_v, self.w_scale, self.gate = o, lse, w_v, w_scale, gate
        P, S, H, d = o.shape
        assert d == D and o.strides[-1] == o.itemsize and o.dtype == np.uint16
        assert gate.dtype == np.uint16 and gate.flags.c_contiguous
        self.S, self.H, self.P = S, H, P
        self.S_out = S if S_out is None else S_out
        a = _Args()
        a.S, a.S_out, a.H, a.P, a.q, a.spr = S, self.S_out, H, P, q, spr
        a.o = _ptr(o)
        a.o_sp, a.o_st, a.o_sh, _ = _estrides(o)
        if lse is not None:
            assert lse.dtype == np.float32
            a.lse = _ptr(lse)
            a.l_sp, a.l_st, a.l_sh = _estrides(lse)
        a.w_v = _ptr(w_v)
        a.w_sh, a.w_sv, _ = _estrides(w_v)
        if w_scale is not None:
            a.w_scale = _ptr(w_scale)
            a.s_sh, a.s_sv, _ = _estrides(w_scale)
        a.w_fmt = w_fmt
        a.gate = _ptr(gate)
        self.args = a

    def full(self) -> np.ndarray:
        out = np.empty((self.S_out, self.H * V), np.uint16)
        rc = lib().orc_mla_combine_uv(ctypes.byref(self.args), _ptr(out))
        if rc != 0:
            raise ValueError("oracle rejected the problem (layout or shape)")
        return out

    def rows(self, ts, hs) -> np.ndarray:
        ts = np.ascontiguousarray(ts, np.int32)
        hs = np.ascontiguousarray(hs, np.int32)
        segs = np.empty((len(ts), V), np.uint16)
        rc = lib().orc_rows(ctypes.byref(self.args), len(ts), _ptr(ts), _ptr(hs), _ptr(segs))
        if rc != 0:
            raise ValueError("oracle rejected the problem (layout or shape)")
        return segs

    def latent_f32(self, t, h) -> np.ndarray:
        lat = np.empty(D, np.float32)
        if lib().orc_combine_latent(ctypes.byref(self.args), t, h, _ptr(lat)) < 0:
            raise ValueError("oracle rejected the problem")
        return lat

    def latent_bf16(self, t, h) -> np.ndarray:
        lat = np.empty(D, np.uint16)
        if lib().orc_latent_bf16(ctypes.byref(self.args), t, h, _ptr(lat)) < 0:
            raise ValueError("oracle rejected the problem")
        return lat


def host_arrays(inp):
    """numpy copies of a workload's tensors (a dict of torch tensors as the
    seeded generator makes them), strides kept: (o bits, lse, W_V, scales,
    gate bits)."""
    import torch

    def bits(t):
        return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)

    o = bits(inp["o"])
    lse = None if inp["lse"] is None else inp["lse"].detach().cpu().numpy()
    w = bits(inp["w_v"]) if inp["w_fmt"] == 0 else inp["w_v"].detach().cpu().numpy()
    ws = None if inp["w_scale"] is None else inp["w_scale"].detach().cpu().numpy()
    gate = bits(inp["gate"].contiguous())
    return o, lse, w, ws, gate


def problem_from_tensors(inp, host=None):
    """The oracle's Problem for a workload dict (tensors copied to the host)."""
    o, lse, w, ws, gate = host or host_arrays(inp)
    return Problem(o, lse, inp["q"], inp["spr"], w, ws, inp["w_fmt"], gate, inp["S_out"])


def dcp_pack(o, lse, seq_lens, qsl, q, dst):
    """stage_push for destination rank ``dst`` (the page's DCP producer side).

    o        uint16 [R, S, R*H, 512] (bf16 bits; any strides, last dim contiguous)
    lse      float32 [R, S, R*H]
    seq_lens int32 [R, S/q] (contiguous rows)
    qsl      int32 [S/q + 1]
    Returns (cmb_o uint16 [R, S, H, 512], cmb_lse float32 [R, S, H]).
    """
    R, S, RH, d = o.shape
    assert d == D and o.strides[-1] == o.itemsize and o.dtype == np.uint16 and RH % R == 0
    assert lse.dtype == np.float32 and lse.shape == (R, S, RH)
    seq_lens = np.ascontiguousarray(seq_lens, np.int32)
    qsl = np.ascontiguousarray(qsl, np.int32)
    assert seq_lens.shape == (R, S // q) and qsl.shape == (S // q + 1,)
    H = RH // R
    a = _PackArgs()
    a.S, a.H, a.R, a.q, a.dst = S, H, R, q, dst
    a.o = _ptr(o)
    a.o_sr, a.o_st, a.o_sh, _ = _estrides(o)
    a.lse = _ptr(lse)
    a.l_sr, a.l_st, a.l_sh = _estrides(lse)
    a.seq_lens, a.sl_sr = _ptr(seq_lens), S // q
    a.qsl = _ptr(qsl)
    cmb_o = np.empty((R, S, H, D), np.uint16)
    cmb_lse = np.empty((R, S, H), np.float32)
    if lib().orc_dcp_pack(ctypes.byref(a), _ptr(cmb_o), _ptr(cmb_lse)) != 0:
        raise ValueError("oracle rejected the pack problem")
    return cmb_o, cmb_lse


def mla_attn_split(qv, kv, kv_len, q, spr, scale):
    """Split-KV MLA decode attention (the partial producer), in double.

    qv     uint16 [S, H, 576] (bf16 bits; any strides, last dim contiguous)
    kv     uint16 [B, Lmax, 576] (bf16 bits; any strides, last dim contiguous)
    kv_len int32 [B]; S = B * q
    Returns (o uint16 [spr, S, H, 512], lse float32 [spr, S, H]).
    """
    S, H, dq = qv.shape
    B, _, dk = kv.shape
    assert dq == D + 64 and dk == D + 64 and S == B * q
    assert qv.dtype == np.uint16 and kv.dtype == np.uint16
    assert qv.strides[-1] == 2 and kv.strides[-1] == 2
    kv_len = np.ascontiguousarray(kv_len, np.int32)
    assert kv_len.shape == (B,) and int(kv_len.max(initial=0)) <= kv.shape[1]
    a = _AttnArgs()
    a.B, a.q, a.H, a.spr, a.scale = B, q, H, spr, scale
    a.qv = _ptr(qv)
    a.q_st, a.q_sh, _ = _estrides(qv)
    a.kv = _ptr(kv)
    a.kv_sb, a.kv_sl, _ = _estrides(kv)
    a.kv_len = _ptr(kv_len)
    o = np.empty((spr, S, H, D), np.uint16)
    lse = np.empty((spr, S, H), np.float32)
    if lib().orc_mla_attn_split(ctypes.byref(a), _ptr(o), _ptr(lse)) != 0:
        raise ValueError("oracle rejected the attention problem")
    return o, lse


def o_proj(x, w):
    """This rank's o_proj shard in double: out[t][j] = sum_k x[t][k] w[j][k].

    x uint16 [S, K] (bf16 bits, unit-stride rows), w uint16 [Nout, K].
    Returns out uint16 [S, Nout] (bf16 bits).
    """
    S, K = x.shape
    Nout, K2 = w.shape
    assert K == K2 and x.dtype == np.uint16 and w.dtype == np.uint16
    assert x.strides[1] == 2 and w.strides[1] == 2
    a = _OprojArgs()
    a.S, a.K, a.Nout = S, K, Nout
    a.x, a.x_st = _ptr(x), x.strides[0] // 2
    a.w, a.w_sj = _ptr(w), w.strides[0] // 2
    out = np.empty((S, Nout), np.uint16)
    if lib().orc_o_proj(ctypes.byref(a), _ptr(out)) != 0:
        raise ValueError("oracle rejected the o_proj problem")
    return out


# ---- scalar helpers for the pins ----------------------------------------

def sane(x: float) -> float:
    return lib().orc_sane(x)


def bf16_round(x) -> np.ndarray:
    x = np.asarray(x, np.float32).ravel()
    f = lib().orc_f32_to_bf16
    return np.array([f(float(v)) for v in x], np.uint16)


def bf16_value(bits) -> np.ndarray:
    bits = np.asarray(bits, np.uint16).ravel()
    f = lib().orc_bf16_to_f32
    return np.array([f(int(b)) for b in bits], np.float32)


def e2m1_code(y: float) -> int:
    return lib().orc_e2m1_code(y)


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e8m0_value(code: int) -> float:
    return lib().orc_e8m0_value(code)


def mx_scale_code(blk_bits) -> int:
    blk = np.ascontiguousarray(blk_bits, np.uint16)
    assert blk.size == BLK
    return lib().orc_mx_scale_code(_ptr(blk))


def mx_quant_block(blk_bits):
    blk = np.ascontiguousarray(blk_bits, np.uint16)
    assert blk.size == BLK
    codes = np.empty(BLK, np.uint8)
    sc = ctypes.c_int()
    lib().orc_mx_quant_block(_ptr(blk), _ptr(codes), ctypes.byref(sc))
    return codes, sc.value


def partial_set(t, S, P, q, spr):
    r0, n = ctypes.c_int(), ctypes.c_int()
    lay = lib().orc_partial_set(t, S, P, q, spr, ctypes.byref(r0), ctypes.byref(n))
    return lay, r0.value, n.value
