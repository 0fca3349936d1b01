"""GB300 (sm_103a) MLA decode post-attention stage: LSE combine -> W_UV -> gate.

A thin ctypes binding of ``libmla_combine_uv.so`` (C ABI in
``include/mla_combine_uv.h``).  It only marshals arguments: every step of the
computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
missing, importing the binding's functions raises.

The operation is the one of the vLLM page
"vllm.models.kimi_k3.amd.specialized_decode.mono.attention.mla_back"
(``mla_post``: dcp_a2a_lse_reduce -> _v_up_proj -> gate).
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmla_combine_uv.so")

MLA_W_BF16 = 0
MLA_W_MXFP4 = 1
MLA_KERNEL_AUTO = 0
MLA_KERNEL_SIMT = 1
MLA_KERNEL_TC = 2
MLA_KERNEL_KSPLIT = 3

MLA_OK = 0
MLA_ERR_NULL = 1
MLA_ERR_SHAPE = 2
MLA_ERR_STRIDE = 3
MLA_ERR_ALIGN = 4
MLA_ERR_FMT = 5
MLA_ERR_LAYOUT = 6
MLA_ERR_CUDA = 7
MLA_ERR_TIMEOUT = 8
MLA_ERR_KERNEL = 9
MLA_ERR_DATA = 10
MLA_ERR_SCRATCH = 11

EXPORTED_SYMBOLS = ("mla_combine_uv", "mla_combine_uv_plan", "mla_combine_uv_status",
                    "mla_dcp_pack", "mla_attn_split_kv", "mla_o_proj", "mla_status_str", "mla_abi_version",
                    "mla_calib_stream_read", "mla_attn_combine_uv", "mla_attn_combine_uv_workspace_words",
                    "mla_attn_combine_uv_noalloc")


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: status {status} ({mla_status_str(status)})" if what else
                         f"status {status} ({mla_status_str(status)})")


class Args(ctypes.Structure):
    """Mirror of ``mla_combine_uv_args``."""
    _fields_ = [
        ("S", ctypes.c_int32), ("S_out", ctypes.c_int32), ("H", ctypes.c_int32),
        ("P", ctypes.c_int32), ("q_per_request", ctypes.c_int32),
        ("splits_per_request", ctypes.c_int32),
        ("o", ctypes.c_void_p), ("o_sp", ctypes.c_int64), ("o_st", ctypes.c_int64),
        ("o_sh", ctypes.c_int64),
        ("lse", ctypes.c_void_p), ("l_sp", ctypes.c_int64), ("l_st", ctypes.c_int64),
        ("l_sh", ctypes.c_int64),
        ("w_v", ctypes.c_void_p), ("w_sh", ctypes.c_int64), ("w_sv", ctypes.c_int64),
        ("w_scale", ctypes.c_void_p), ("s_sh", ctypes.c_int64), ("s_sv", ctypes.c_int64),
        ("w_fmt", ctypes.c_int32),
        ("gate", ctypes.c_void_p), ("out", ctypes.c_void_p),
        ("kernel", ctypes.c_int32), ("tile_tokens", ctypes.c_int32),
        ("wait_ns", ctypes.c_int64), ("ready_flag", ctypes.c_void_p),
    ]


class Plan(ctypes.Structure):
    """Mirror of ``mla_plan``."""
    _fields_ = [(n, ctypes.c_int32) for n in
                ("kernel", "layout", "n_part", "tile_tokens", "units", "grid", "threads",
                 "smem_bytes", "offsets32")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class PackArgs(ctypes.Structure):
    """Mirror of ``mla_dcp_pack_args``."""
    _fields_ = [
        ("S", ctypes.c_int32), ("H", ctypes.c_int32), ("R", ctypes.c_int32),
        ("q_per_request", ctypes.c_int32), ("dst_rank", ctypes.c_int32),
        ("o", ctypes.c_void_p), ("o_sr", ctypes.c_int64), ("o_st", ctypes.c_int64),
        ("o_sh", ctypes.c_int64),
        ("lse", ctypes.c_void_p), ("l_sr", ctypes.c_int64), ("l_st", ctypes.c_int64),
        ("l_sh", ctypes.c_int64),
        ("seq_lens", ctypes.c_void_p), ("sl_sr", ctypes.c_int64),
        ("qsl", ctypes.c_void_p),
        ("cmb_o", ctypes.c_void_p), ("cmb_lse", ctypes.c_void_p),
    ]


class AttnArgs(ctypes.Structure):
    """Mirror of ``mla_attn_split_kv_args``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("q", ctypes.c_int32), ("H", ctypes.c_int32), ("spr", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("qv", ctypes.c_void_p), ("q_st", ctypes.c_int64), ("q_sh", ctypes.c_int64),
        ("kv", ctypes.c_void_p), ("kv_sb", ctypes.c_int64), ("kv_sl", ctypes.c_int64),
        ("Lmax", ctypes.c_int32),
        ("kv_len", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("kernel", ctypes.c_int32),
    ]


class AttnCombineArgs(ctypes.Structure):
    """Mirror of ``mla_attn_combine_uv_args``."""
    _fields_ = [
        ("B", ctypes.c_int32), ("q", ctypes.c_int32), ("H", ctypes.c_int32), ("spr", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("qv", ctypes.c_void_p), ("q_st", ctypes.c_int64), ("q_sh", ctypes.c_int64),
        ("kv", ctypes.c_void_p), ("kv_sb", ctypes.c_int64), ("kv_sl", ctypes.c_int64),
        ("Lmax", ctypes.c_int32),
        ("kv_len", ctypes.c_void_p),
        ("part_o", ctypes.c_void_p), ("part_lse", ctypes.c_void_p),
        ("w_v", ctypes.c_void_p), ("w_sh", ctypes.c_int64), ("w_sv", ctypes.c_int64),
        ("w_scale", ctypes.c_void_p), ("s_sh", ctypes.c_int64), ("s_sv", ctypes.c_int64),
        ("w_fmt", ctypes.c_int32),
        ("gate", ctypes.c_void_p), ("out", ctypes.c_void_p), ("S_out", ctypes.c_int32),
        ("workspace", ctypes.c_void_p), ("workspace_words", ctypes.c_int64),
        ("wait_ns", ctypes.c_int64),
        ("w_o", ctypes.c_void_p), ("w_o_sj", ctypes.c_int64), ("n_out", ctypes.c_int32),
        ("y", ctypes.c_void_p), ("y_st", ctypes.c_int64),
    ]


class OprojArgs(ctypes.Structure):
    """Mirror of ``mla_o_proj_args``."""
    _fields_ = [
        ("S", ctypes.c_int32), ("K", ctypes.c_int32), ("Nout", ctypes.c_int32),
        ("x", ctypes.c_void_p), ("x_st", ctypes.c_int64),
        ("w", ctypes.c_void_p), ("w_sj", ctypes.c_int64),
        ("out", ctypes.c_void_p), ("out_st", ctypes.c_int64),
    ]


_lib = None


def load_library(path: str | None = None):
    """Load the CUDA library (built in-tree by ``build.build()``; the
    environment variable ``MLA_COMBINE_UV_LIB`` names another build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("MLA_COMBINE_UV_LIB") or LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m mla_decode_attention_lse_gb300.build` "
            "(there is no CPU fallback)")
    L = ctypes.CDLL(path)
    L.mla_combine_uv.restype = ctypes.c_int32
    L.mla_combine_uv.argtypes = [ctypes.POINTER(Args), ctypes.c_void_p]
    L.mla_combine_uv_plan.restype = ctypes.c_int32
    L.mla_combine_uv_plan.argtypes = [ctypes.POINTER(Args), ctypes.c_int32, ctypes.POINTER(Plan)]
    L.mla_combine_uv_status.restype = ctypes.c_int32
    L.mla_combine_uv_status.argtypes = [ctypes.c_void_p]
    L.mla_status_str.restype = ctypes.c_char_p
    L.mla_status_str.argtypes = [ctypes.c_int32]
    L.mla_abi_version.restype = ctypes.c_int32
    L.mla_abi_version.argtypes = []
    L.mla_dcp_pack.restype = ctypes.c_int32
    L.mla_dcp_pack.argtypes = [ctypes.POINTER(PackArgs), ctypes.c_void_p]
    L.mla_attn_split_kv.restype = ctypes.c_int32
    L.mla_attn_split_kv.argtypes = [ctypes.POINTER(AttnArgs), ctypes.c_void_p]
    L.mla_o_proj.restype = ctypes.c_int32
    L.mla_o_proj.argtypes = [ctypes.POINTER(OprojArgs), ctypes.c_void_p]
    L.mla_attn_combine_uv.restype = ctypes.c_int32
    L.mla_attn_combine_uv.argtypes = [ctypes.POINTER(AttnCombineArgs), ctypes.c_void_p]
    L.mla_attn_combine_uv_workspace_words.restype = ctypes.c_int64
    L.mla_attn_combine_uv_workspace_words.argtypes = [ctypes.c_int32, ctypes.c_int32]
    L.mla_attn_combine_uv_noalloc.restype = ctypes.c_int32
    L.mla_attn_combine_uv_noalloc.argtypes = [ctypes.POINTER(AttnCombineArgs), ctypes.c_void_p]
    L.mla_calib_stream_read.restype = ctypes.c_int32
    L.mla_calib_stream_read.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                        ctypes.c_void_p]
    _lib = L
    return L


def mla_status_str(status: int) -> str:
    return load_library().mla_status_str(status).decode()


def mla_abi_version() -> int:
    return load_library().mla_abi_version()


def _ptr(t):
    return None if t is None else t.data_ptr()


def make_args(o, lse, q_per_request, splits_per_request, w_v, w_fmt, gate, out, w_scale=None,
              kernel=MLA_KERNEL_AUTO, tile_tokens=0, wait_ns=0, ready_flag=None) -> Args:
    """Fill ``mla_combine_uv_args`` from tensors (pointers and element strides)."""
    P, S, H, _ = o.shape
    a = Args()
    a.S, a.S_out, a.H, a.P = S, out.shape[0], H, P
    a.q_per_request, a.splits_per_request = q_per_request, splits_per_request
    a.o = _ptr(o)
    a.o_sp, a.o_st, a.o_sh = o.stride(0), o.stride(1), o.stride(2)
    if lse is not None:
        a.lse = _ptr(lse)
        a.l_sp, a.l_st, a.l_sh = lse.stride(0), lse.stride(1), lse.stride(2)
    a.w_v = _ptr(w_v)
    a.w_sh, a.w_sv = w_v.stride(0), w_v.stride(1)
    if w_scale is not None:
        a.w_scale = _ptr(w_scale)
        a.s_sh, a.s_sv = w_scale.stride(0), w_scale.stride(1)
    a.w_fmt = w_fmt
    a.gate = _ptr(gate)
    a.out = _ptr(out)
    a.kernel, a.tile_tokens = kernel, tile_tokens
    a.wait_ns = wait_ns
    a.ready_flag = _ptr(ready_flag)
    return a


def _check_tensors(o, lse, w_v, w_scale, gate, out, w_fmt):
    import torch

    if o.dtype != torch.bfloat16 or o.dim() != 4 or o.shape[3] != 512 or o.stride(3) != 1:
        raise ValueError("o must be bf16 [P, S, H, 512] with a unit-stride last dimension")
    if lse is not None and (lse.dtype != torch.float32 or lse.dim() != 3):
        raise ValueError("lse must be float32 [P, S, H]")
    if gate.dtype != torch.bfloat16 or not gate.is_contiguous():
        raise ValueError("gate must be a dense bf16 [S, H*128] tensor")
    if out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a dense bf16 [S_out, H*128] tensor")
    if w_fmt == MLA_W_BF16 and (w_v.dtype != torch.bfloat16 or w_v.stride(-1) != 1):
        raise ValueError("bf16 W_V must be bf16 [H, 128, 512] with a unit-stride last dimension")
    if w_fmt == MLA_W_MXFP4 and (w_v.dtype != torch.uint8 or w_scale is None
                                 or w_scale.dtype != torch.uint8):
        raise ValueError("MXFP4 W_V must be uint8 [H, 128, 256] with uint8 [H, 128, 16] scales")


def mla_combine_uv(o, lse, q_per_request, splits_per_request, w_v, w_fmt, gate, out,
                   w_scale=None, stream=None, kernel=MLA_KERNEL_AUTO, tile_tokens=0,
                   wait_ns=0, ready_flag=None) -> None:
    """Run the stage on CUDA tensors; writes ``out`` [S_out, H*128] bf16.

    o [P, S, H, 512] bf16; lse [P, S, H] f32 (None allowed when P == 1);
    w_v bf16 [H, 128, 512] (w_fmt 0) or uint8 [H, 128, 256] + w_scale uint8
    [H, 128, 16] (w_fmt 1); gate [S, H*128] bf16.  Asynchronous on ``stream``
    (default: PyTorch's current stream).  ``wait_ns`` > 0 sets the limit of
    the tensor-core kernel's bounded waits (default 0.5 s); ``ready_flag`` (a
    one-element int32 CUDA tensor) makes every CTA wait, within that limit,
    until it is non-zero before reading its inputs.
    """
    import torch

    _check_tensors(o, lse, w_v, w_scale, gate, out, w_fmt)
    if stream is None:
        stream = torch.cuda.current_stream(o.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    a = make_args(o, lse, q_per_request, splits_per_request, w_v, w_fmt, gate, out, w_scale,
                  kernel, tile_tokens, wait_ns, ready_flag)
    st = load_library().mla_combine_uv(ctypes.byref(a), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_combine_uv")


def make_pack_args(o, lse, seq_lens, qsl, q_per_request, dst_rank, cmb_o, cmb_lse) -> PackArgs:
    """Fill ``mla_dcp_pack_args`` from tensors (pointers and element strides)."""
    R, S, RH, _ = o.shape
    a = PackArgs()
    a.S, a.H, a.R = S, RH // R, R
    a.q_per_request, a.dst_rank = q_per_request, dst_rank
    a.o = _ptr(o)
    a.o_sr, a.o_st, a.o_sh = o.stride(0), o.stride(1), o.stride(2)
    a.lse = _ptr(lse)
    a.l_sr, a.l_st, a.l_sh = lse.stride(0), lse.stride(1), lse.stride(2)
    a.seq_lens, a.sl_sr = _ptr(seq_lens), seq_lens.stride(0)
    a.qsl = _ptr(qsl)
    a.cmb_o, a.cmb_lse = _ptr(cmb_o), _ptr(cmb_lse)
    return a


def mla_dcp_pack(o, lse, seq_lens, qsl, q_per_request, dst_rank, cmb_o, cmb_lse, stream=None) -> None:
    """The DCP producer side: pack every rank's partials into rank ``dst_rank``'s
    combine buffer on CUDA tensors.

    o [R, S, R*H, 512] bf16 (unit-stride last dimension); lse [R, S, R*H] f32;
    seq_lens [R, S/q] int32 (unit-stride rows); qsl [S/q + 1] int32; cmb_o
    [R, S, H, 512] bf16 dense; cmb_lse [R, S, H] f32 dense.
    """
    import torch

    R, S, RH, d = o.shape
    if o.dtype != torch.bfloat16 or d != 512 or o.stride(3) != 1 or RH % R:
        raise ValueError("o must be bf16 [R, S, R*H, 512] with a unit-stride last dimension")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (R, S, RH):
        raise ValueError("lse must be float32 [R, S, R*H]")
    if S % q_per_request:
        raise ValueError("S must be a multiple of q_per_request")
    if (seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (R, S // q_per_request)
            or seq_lens.stride(1) != 1):
        raise ValueError("seq_lens must be int32 [R, S/q] with unit-stride rows")
    if qsl.dtype != torch.int32 or tuple(qsl.shape) != (S // q_per_request + 1,) or not qsl.is_contiguous():
        raise ValueError("qsl must be a dense int32 [S/q + 1] tensor")
    H = RH // R
    if (cmb_o.dtype != torch.bfloat16 or tuple(cmb_o.shape) != (R, S, H, 512) or not cmb_o.is_contiguous()
            or cmb_lse.dtype != torch.float32 or tuple(cmb_lse.shape) != (R, S, H)
            or not cmb_lse.is_contiguous()):
        raise ValueError("cmb_o / cmb_lse must be dense bf16 [R, S, H, 512] / float32 [R, S, H]")
    if stream is None:
        stream = torch.cuda.current_stream(o.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    a = make_pack_args(o, lse, seq_lens, qsl, q_per_request, dst_rank, cmb_o, cmb_lse)
    st = load_library().mla_dcp_pack(ctypes.byref(a), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_dcp_pack")


def make_attn_args(qv, kv, kv_len, q, spr, scale, o, lse, kernel=0) -> AttnArgs:
    """Fill ``mla_attn_split_kv_args`` from tensors (pointers and element strides)."""
    S, H, _ = qv.shape
    B, Lmax, _ = kv.shape
    a = AttnArgs()
    a.B, a.q, a.H, a.spr, a.scale = B, q, H, spr, float(scale)
    a.qv, a.q_st, a.q_sh = _ptr(qv), qv.stride(0), qv.stride(1)
    a.kv, a.kv_sb, a.kv_sl = _ptr(kv), kv.stride(0), kv.stride(1)
    a.Lmax, a.kv_len = Lmax, _ptr(kv_len)
    a.o, a.lse = _ptr(o), _ptr(lse)
    a.kernel = kernel
    return a


def mla_attn_split_kv(qv, kv, kv_len, q, spr, scale, o, lse, stream=None, kernel=0) -> None:
    """The partial producer: split-KV MLA decode attention on CUDA tensors.

    qv [S, H, 576] bf16 (S = B * q; unit-stride last dimension); kv
    [B, Lmax, 576] bf16 (unit-stride last dimension); kv_len [B] int32; o
    [spr, S, H, 512] bf16 dense; lse [spr, S, H] f32 dense.  ``kernel``: 0
    automatic (one CTA per item), 1 one CTA per item, 2 a 2-CTA cluster per
    item (on request).
    """
    import torch

    S, H, dq = qv.shape
    B, Lmax, dk = kv.shape
    if qv.dtype != torch.bfloat16 or dq != 576 or qv.stride(2) != 1:
        raise ValueError("qv must be bf16 [S, H, 576] with a unit-stride last dimension")
    if kv.dtype != torch.bfloat16 or dk != 576 or kv.stride(2) != 1:
        raise ValueError("kv must be bf16 [B, Lmax, 576] with a unit-stride last dimension")
    if S != B * q:
        raise ValueError("qv must hold B * q token rows")
    if kv_len.dtype != torch.int32 or tuple(kv_len.shape) != (B,) or not kv_len.is_contiguous():
        raise ValueError("kv_len must be a dense int32 [B] tensor")
    if (o.dtype != torch.bfloat16 or tuple(o.shape) != (spr, S, H, 512) or not o.is_contiguous()
            or lse.dtype != torch.float32 or tuple(lse.shape) != (spr, S, H) or not lse.is_contiguous()):
        raise ValueError("o / lse must be dense bf16 [spr, S, H, 512] / float32 [spr, S, H]")
    if stream is None:
        stream = torch.cuda.current_stream(qv.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    a = make_attn_args(qv, kv, kv_len, q, spr, scale, o, lse, kernel)
    st = load_library().mla_attn_split_kv(ctypes.byref(a), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_attn_split_kv")


def mla_attn_combine_uv_workspace_words(B: int, q: int) -> int:
    """int32 words of workspace the fused decode step needs for B requests of q tokens."""
    return load_library().mla_attn_combine_uv_workspace_words(B, q)


def make_attn_combine_args(qv, kv, kv_len, q, spr, scale, part_o, part_lse, w_v, gate, out, workspace,
                           wait_ns=0, w_o=None, y=None) -> AttnCombineArgs:
    """Fill ``mla_attn_combine_uv_args`` from tensors (pointers and element strides)."""
    S, H, _ = qv.shape
    B, Lmax, _ = kv.shape
    a = AttnCombineArgs()
    a.B, a.q, a.H, a.spr, a.scale = B, q, H, spr, float(scale)
    a.qv, a.q_st, a.q_sh = _ptr(qv), qv.stride(0), qv.stride(1)
    a.kv, a.kv_sb, a.kv_sl = _ptr(kv), kv.stride(0), kv.stride(1)
    a.Lmax, a.kv_len = Lmax, _ptr(kv_len)
    a.part_o, a.part_lse = _ptr(part_o), _ptr(part_lse)
    a.w_v, a.w_sh, a.w_sv = _ptr(w_v), w_v.stride(0), w_v.stride(1)
    a.w_fmt = MLA_W_BF16
    a.gate, a.out, a.S_out = _ptr(gate), _ptr(out), out.shape[0]
    a.workspace, a.workspace_words = _ptr(workspace), workspace.numel()
    a.wait_ns = wait_ns
    if w_o is not None:
        a.w_o, a.w_o_sj, a.n_out = _ptr(w_o), w_o.stride(0), w_o.shape[0]
        a.y, a.y_st = _ptr(y), y.stride(0)
    return a


def _check_oproj(w_o, y, S, H):
    import torch

    if (w_o is None) != (y is None):
        raise ValueError("w_o and y go together")
    if w_o is None:
        return
    if w_o.dtype != torch.bfloat16 or w_o.dim() != 2 or w_o.shape[1] != H * 128 or w_o.stride(1) != 1:
        raise ValueError("w_o must be bf16 [n_out, H*128] with a unit-stride last dimension")
    if y.dtype != torch.bfloat16 or y.dim() != 2 or tuple(y.shape) != (S, w_o.shape[0]) or y.stride(1) != 1:
        raise ValueError("y must be bf16 [S, n_out] with a unit-stride last dimension")


def mla_attn_combine_uv(qv, kv, kv_len, q, spr, scale, part_o, part_lse, w_v, gate, out, workspace,
                        stream=None, wait_ns=0, w_o=None, y=None) -> None:
    """The decode step in one launch: split-KV attention, then the combine of
    its partials (bf16 W_V), on CUDA tensors; with ``w_o`` (bf16 [n_out,
    H*128], n_out a multiple of 64) and ``y`` (bf16 [S, n_out]) also the
    o_proj shard y = out[:S] w_o^T, in the same launch.

    qv [S, H, 576] bf16 (S = B * q); kv [B, Lmax, 576] bf16; kv_len [B] int32;
    part_o [spr, S, H, 512] bf16 / part_lse [spr, S, H] f32 dense (scratch for
    the partials); w_v bf16 [H, 128, 512]; gate [S, H*128] bf16; out
    [S_out, H*128] bf16; workspace int32 [mla_attn_combine_uv_workspace_words(B, q)],
    zero before the first call (every call leaves it zero).
    """
    import torch

    S, H, dq = qv.shape
    B, Lmax, dk = kv.shape
    if qv.dtype != torch.bfloat16 or dq != 576 or qv.stride(2) != 1:
        raise ValueError("qv must be bf16 [S, H, 576] with a unit-stride last dimension")
    if kv.dtype != torch.bfloat16 or dk != 576 or kv.stride(2) != 1:
        raise ValueError("kv must be bf16 [B, Lmax, 576] with a unit-stride last dimension")
    if S != B * q:
        raise ValueError("qv must hold B * q token rows")
    if kv_len.dtype != torch.int32 or tuple(kv_len.shape) != (B,) or not kv_len.is_contiguous():
        raise ValueError("kv_len must be a dense int32 [B] tensor")
    if (part_o.dtype != torch.bfloat16 or tuple(part_o.shape) != (spr, S, H, 512) or not part_o.is_contiguous()
            or part_lse.dtype != torch.float32 or tuple(part_lse.shape) != (spr, S, H)
            or not part_lse.is_contiguous()):
        raise ValueError("part_o / part_lse must be dense bf16 [spr, S, H, 512] / float32 [spr, S, H]")
    if w_v.dtype != torch.bfloat16 or tuple(w_v.shape) != (H, 128, 512) or w_v.stride(2) != 1:
        raise ValueError("w_v must be bf16 [H, 128, 512] with a unit-stride last dimension")
    if gate.dtype != torch.bfloat16 or not gate.is_contiguous() or tuple(gate.shape) != (S, H * 128):
        raise ValueError("gate must be a dense bf16 [S, H*128] tensor")
    if out.dtype != torch.bfloat16 or not out.is_contiguous() or out.dim() != 2 or out.shape[1] != H * 128:
        raise ValueError("out must be a dense bf16 [S_out, H*128] tensor")
    if workspace.dtype != torch.int32 or not workspace.is_contiguous():
        raise ValueError("workspace must be a dense int32 tensor")
    if stream is None:
        stream = torch.cuda.current_stream(qv.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    _check_oproj(w_o, y, S, H)
    a = make_attn_combine_args(qv, kv, kv_len, q, spr, scale, part_o, part_lse, w_v, gate, out, workspace, wait_ns,
                               w_o, y)
    st = load_library().mla_attn_combine_uv(ctypes.byref(a), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_attn_combine_uv")


def mla_attn_combine_uv_noalloc(qv, kv, kv_len, q, spr, scale, w_v, gate, out, stream=None, wait_ns=0) -> None:
    """The fused decode step for callers that cannot allocate device memory
    when they run it: the same inputs and output as ``mla_attn_combine_uv``,
    the scratch (partials and counters) in the library's fixed 16 MiB device
    buffer.  Calls that overlap on the GPU race on that buffer."""
    import torch

    S, H, _ = qv.shape
    if stream is None:
        stream = torch.cuda.current_stream(qv.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    B, Lmax, _ = kv.shape
    a = AttnCombineArgs()
    a.B, a.q, a.H, a.spr, a.scale = B, q, H, spr, float(scale)
    a.qv, a.q_st, a.q_sh = _ptr(qv), qv.stride(0), qv.stride(1)
    a.kv, a.kv_sb, a.kv_sl = _ptr(kv), kv.stride(0), kv.stride(1)
    a.Lmax, a.kv_len = Lmax, _ptr(kv_len)
    a.w_v, a.w_sh, a.w_sv = _ptr(w_v), w_v.stride(0), w_v.stride(1)
    a.w_fmt = MLA_W_BF16
    a.gate, a.out, a.S_out = _ptr(gate), _ptr(out), out.shape[0]
    a.wait_ns = wait_ns
    st = load_library().mla_attn_combine_uv_noalloc(ctypes.byref(a), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_attn_combine_uv_noalloc")


def make_oproj_args(x, w, out) -> OprojArgs:
    """Fill ``mla_o_proj_args`` from tensors (pointers and element strides)."""
    a = OprojArgs()
    a.S, a.K = x.shape
    a.Nout = w.shape[0]
    a.x, a.x_st = _ptr(x), x.stride(0)
    a.w, a.w_sj = _ptr(w), w.stride(0)
    a.out, a.out_st = _ptr(out), out.stride(0)
    return a


def mla_o_proj(x, w, out, stream=None) -> None:
    """This rank's o_proj shard on CUDA tensors: out = x @ w.T.

    x [S, K] bf16 (core rows, unit-stride rows), w [Nout, K] bf16 (the linear
    layer's weight slice), out [S, Nout] bf16 (unit-stride rows).
    """
    import torch

    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise ValueError("x, w and out must be bf16")
    if x.dim() != 2 or w.dim() != 2 or out.dim() != 2 or x.shape[1] != w.shape[1]:
        raise ValueError("x [S, K], w [Nout, K], out [S, Nout]")
    if tuple(out.shape) != (x.shape[0], w.shape[0]) or x.stride(1) != 1 or w.stride(1) != 1 or out.stride(1) != 1:
        raise ValueError("out must be [S, Nout]; every last dimension unit-stride")
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    a = make_oproj_args(x, w, out)
    st = load_library().mla_o_proj(ctypes.byref(a), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_o_proj")


def mla_calib_stream_read(src, nbytes: int, dependent_round_trips: int, sink, stream=None) -> None:
    """Measurement aid: one read-only streaming launch over the first ``nbytes``
    bytes of the CUDA tensor ``src`` (``sink``: a one-element int32/uint32
    CUDA tensor, written only for a fixed xor pattern of the data)."""
    import torch

    if nbytes > src.numel() * src.element_size():
        raise ValueError("nbytes exceeds the tensor")
    if stream is None:
        stream = torch.cuda.current_stream(src.device)
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    st = load_library().mla_calib_stream_read(ctypes.c_void_p(src.data_ptr()), nbytes, dependent_round_trips,
                                              ctypes.c_void_p(sink.data_ptr()), ctypes.c_void_p(s))
    if st != MLA_OK:
        raise MlaError(st, "mla_calib_stream_read")


def mla_combine_uv_plan(args: Args, num_sms: int = 0) -> dict:
    """Validate ``args`` and return the launch plan (no GPU needed when
    ``num_sms`` > 0).  Raises ``MlaError`` on a validation error."""
    pl = Plan()
    st = load_library().mla_combine_uv_plan(ctypes.byref(args), num_sms, ctypes.byref(pl))
    if st != MLA_OK:
        raise MlaError(st, "mla_combine_uv_plan")
    return pl.as_dict()


def mla_combine_uv_status(stream=None) -> int:
    """Read and clear the device's error word in order on ``stream`` (then
    synchronised).  The word is one per device, shared by every stream."""
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    s = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return load_library().mla_combine_uv_status(ctypes.c_void_p(s))
