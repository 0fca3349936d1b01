"""C-ABI checks that need no GPU: the library builds and loads, exports every
function ``include/mla_combine_uv.h`` declares, and its host-side validation
and planning behave as documented (``mla_combine_uv_plan`` with an explicit
SM count makes no CUDA call)."""
import ctypes
import os
import re
import subprocess

import pytest

from mla_decode_attention_lse_gb300 import (Args, MlaError, build, load_library, make_args,
                                            mla_combine_uv_plan)
import mla_decode_attention_lse_gb300 as m

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SMS = 152


@pytest.fixture(scope="module")
def lib():
    build.build()
    return load_library()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(m.EXPORTED_SYMBOLS) <= set(names)
    assert len(names) >= 5
    for n in names:
        assert hasattr(lib, n), n


def test_abi_version_and_status_strings(lib):
    assert m.mla_abi_version() == 6
    for s in range(0, 12):
        assert m.mla_status_str(s) and m.mla_status_str(s) != "unknown status"
    assert m.mla_status_str(99) == "unknown status"


def test_args_struct_layout_matches_header(lib, tmp_path):
    # compile a probe against the header and compare every field offset
    fields = [f for f, _ in Args._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_combine_uv.h"',
            "int main(void) {", 'printf("%zu\\n", sizeof(mla_combine_uv_args));']
    prog += [f'printf("%zu\\n", offsetof(mla_combine_uv_args, {f}));' for f in fields]
    prog += ['printf("%zu\\n", sizeof(mla_plan));', "return 0; }"]
    src = tmp_path / "probe.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(Args)
    for f, off in zip(fields, vals[1:-1]):
        assert getattr(Args, f).offset == off, f
    assert vals[-1] == ctypes.sizeof(m.Plan)


def test_pack_args_struct_layout_matches_header(lib, tmp_path):
    fields = [f for f, _ in m.PackArgs._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_combine_uv.h"',
            "int main(void) {", 'printf("%zu\\n", sizeof(mla_dcp_pack_args));']
    prog += [f'printf("%zu\\n", offsetof(mla_dcp_pack_args, {f}));' for f in fields]
    prog += ["return 0; }"]
    src = tmp_path / "probe_pack.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "probe_pack"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(m.PackArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(m.PackArgs, f).offset == off, f


def pack_args(S=8, H=2, R=4, q=2, dst=1, **kw):
    a = m.PackArgs()
    a.S, a.H, a.R, a.q_per_request, a.dst_rank = S, H, R, q, dst
    a.o, a.o_sr, a.o_st, a.o_sh = ALIGNED, S * R * H * 512, R * H * 512, 512
    a.lse, a.l_sr, a.l_st, a.l_sh = ALIGNED * 2, S * R * H, R * H, 1
    a.seq_lens, a.sl_sr = ALIGNED * 3, S // q
    a.qsl = ALIGNED * 4
    a.cmb_o, a.cmb_lse = ALIGNED * 5, ALIGNED * 6
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_pack_validation_errors(lib):
    pack = lib.mla_dcp_pack
    st = lambda a: pack(ctypes.byref(a), None)  # noqa: E731  (errors return before any CUDA call)
    assert st(pack_args(dst=4)) == m.MLA_ERR_SHAPE
    assert st(pack_args(dst=-1)) == m.MLA_ERR_SHAPE
    assert st(pack_args(S=7)) == m.MLA_ERR_SHAPE  # S % q
    assert st(pack_args(R=0)) == m.MLA_ERR_SHAPE
    assert st(pack_args(H=0)) == m.MLA_ERR_SHAPE
    assert st(pack_args(R=300, H=300, dst=0)) == m.MLA_ERR_SHAPE  # R*H > 65535
    assert st(pack_args(qsl=None)) == m.MLA_ERR_NULL
    assert st(pack_args(cmb_lse=None)) == m.MLA_ERR_NULL
    assert st(pack_args(o=ALIGNED + 8)) == m.MLA_ERR_ALIGN
    assert st(pack_args(cmb_o=ALIGNED + 4)) == m.MLA_ERR_ALIGN
    assert st(pack_args(seq_lens=ALIGNED + 2)) == m.MLA_ERR_ALIGN
    assert st(pack_args(o_sh=500)) == m.MLA_ERR_STRIDE
    assert st(pack_args(l_st=-1)) == m.MLA_ERR_STRIDE
    assert st(pack_args(S=0, o=None, qsl=None)) == m.MLA_OK  # nothing to do, nothing read


def test_attn_args_struct_layout_matches_header(lib, tmp_path):
    fields = [f for f, _ in m.AttnArgs._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_combine_uv.h"',
            "int main(void) {", 'printf("%zu\\n", sizeof(mla_attn_split_kv_args));']
    prog += [f'printf("%zu\\n", offsetof(mla_attn_split_kv_args, {f}));' for f in fields]
    prog += ["return 0; }"]
    src = tmp_path / "probe_attn.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "probe_attn"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(m.AttnArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(m.AttnArgs, f).offset == off, f


def attn_args(B=4, q=1, H=12, spr=16, Lmax=256, **kw):
    a = m.AttnArgs()
    a.B, a.q, a.H, a.spr, a.scale = B, q, H, spr, 0.07
    a.qv, a.q_st, a.q_sh = ALIGNED, H * 576, 576
    a.kv, a.kv_sb, a.kv_sl = ALIGNED * 2, Lmax * 576, 576
    a.Lmax, a.kv_len = Lmax, ALIGNED * 3
    a.o, a.lse = ALIGNED * 4, ALIGNED * 5
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_attn_validation_errors(lib):
    fn = lib.mla_attn_split_kv
    st = lambda a: fn(ctypes.byref(a), None)  # noqa: E731  (errors return before any CUDA call)
    assert fn(None, None) == m.MLA_ERR_NULL
    assert st(attn_args(B=-1)) == m.MLA_ERR_SHAPE
    assert st(attn_args(q=0)) == m.MLA_ERR_SHAPE
    assert st(attn_args(q=33)) == m.MLA_ERR_SHAPE
    assert st(attn_args(H=0)) == m.MLA_ERR_SHAPE
    assert st(attn_args(spr=0)) == m.MLA_ERR_SHAPE
    assert st(attn_args(Lmax=0)) == m.MLA_ERR_SHAPE
    assert st(attn_args(scale=float("inf"))) == m.MLA_ERR_SHAPE
    assert st(attn_args(kv_len=None)) == m.MLA_ERR_NULL
    assert st(attn_args(o=None)) == m.MLA_ERR_NULL
    assert st(attn_args(qv=ALIGNED + 8)) == m.MLA_ERR_ALIGN
    assert st(attn_args(kv=ALIGNED + 2)) == m.MLA_ERR_ALIGN
    assert st(attn_args(lse=ALIGNED + 2)) == m.MLA_ERR_ALIGN
    assert st(attn_args(q_sh=580)) == m.MLA_ERR_STRIDE
    assert st(attn_args(kv_sl=568)) == m.MLA_ERR_STRIDE  # rows overlap
    assert st(attn_args(kv_sb=0)) == m.MLA_ERR_STRIDE    # B > 1 requests on one row set
    assert st(attn_args(kernel=3)) == m.MLA_ERR_KERNEL
    assert st(attn_args(B=0, qv=None, kv=None)) == m.MLA_OK  # nothing to do, nothing read


def test_attn_combine_args_struct_layout_matches_header(lib, tmp_path):
    fields = [f for f, _ in m.AttnCombineArgs._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_combine_uv.h"',
            "int main(void) {", 'printf("%zu\\n", sizeof(mla_attn_combine_uv_args));']
    prog += [f'printf("%zu\\n", offsetof(mla_attn_combine_uv_args, {f}));' for f in fields]
    prog += ["return 0; }"]
    src = tmp_path / "probe_fused.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "probe_fused"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(m.AttnCombineArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(m.AttnCombineArgs, f).offset == off, f


def fused_args(B=4, q=1, H=12, spr=16, Lmax=256, **kw):
    a = m.AttnCombineArgs()
    a.B, a.q, a.H, a.spr, a.scale = B, q, H, spr, 0.07
    a.qv, a.q_st, a.q_sh = ALIGNED, H * 576, 576
    a.kv, a.kv_sb, a.kv_sl = ALIGNED * 2, Lmax * 576, 576
    a.Lmax, a.kv_len = Lmax, ALIGNED * 3
    a.part_o, a.part_lse = ALIGNED * 4, ALIGNED * 5
    a.w_v, a.w_sh, a.w_sv = ALIGNED * 6, 128 * 512, 512
    a.w_fmt = 0
    a.gate, a.out, a.S_out = ALIGNED * 7, ALIGNED * 8, B * q
    a.workspace, a.workspace_words = ALIGNED * 9, 3 + (B * q + 7) // 8
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_attn_combine_validation_errors(lib):
    fn = lib.mla_attn_combine_uv
    st = lambda a: fn(ctypes.byref(a), None)  # noqa: E731  (errors return before any CUDA call)
    assert fn(None, None) == m.MLA_ERR_NULL
    assert st(fused_args(w_fmt=1)) == m.MLA_ERR_FMT           # bf16 W_V only
    assert st(fused_args(w_scale=ALIGNED)) == m.MLA_ERR_FMT
    assert st(fused_args(B=-1)) == m.MLA_ERR_SHAPE
    assert st(fused_args(q=33)) == m.MLA_ERR_SHAPE
    assert st(fused_args(spr=33)) == m.MLA_ERR_SHAPE           # one lane per partial in the merge
    assert st(fused_args(spr=0)) == m.MLA_ERR_SHAPE
    assert st(fused_args(S_out=3)) == m.MLA_ERR_SHAPE          # S_out < S
    assert st(fused_args(wait_ns=-1)) == m.MLA_ERR_SHAPE
    assert st(fused_args(workspace_words=2)) == m.MLA_ERR_SHAPE
    assert st(fused_args(workspace_words=2 + 1)) == m.MLA_ERR_SHAPE  # 3 + ceil(4 / 8) = 4 words needed
    # o_proj in the same launch
    op = dict(w_o=ALIGNED * 10, w_o_sj=12 * 128, n_out=128, y=ALIGNED * 11, y_st=128)
    assert st(fused_args(**{**op, "n_out": 96})) == m.MLA_ERR_SHAPE   # not a multiple of 64
    assert st(fused_args(**{**op, "n_out": -64})) == m.MLA_ERR_SHAPE
    assert st(fused_args(**{**op, "w_o": None})) == m.MLA_ERR_NULL
    assert st(fused_args(**{**op, "y": None})) == m.MLA_ERR_NULL
    assert st(fused_args(**{**op, "w_o": ALIGNED + 8})) == m.MLA_ERR_ALIGN
    assert st(fused_args(**{**op, "y": ALIGNED + 1})) == m.MLA_ERR_ALIGN
    assert st(fused_args(**{**op, "w_o_sj": 12 * 128 - 8})) == m.MLA_ERR_STRIDE  # shorter than H*128
    assert st(fused_args(**{**op, "w_o_sj": 12 * 128 + 4})) == m.MLA_ERR_STRIDE  # not a multiple of 8
    assert st(fused_args(**{**op, "y_st": 64})) == m.MLA_ERR_STRIDE
    assert st(fused_args(workspace=None)) == m.MLA_ERR_NULL
    assert st(fused_args(part_o=None)) == m.MLA_ERR_NULL
    assert st(fused_args(out=ALIGNED + 8)) == m.MLA_ERR_ALIGN
    assert st(fused_args(workspace=ALIGNED + 2)) == m.MLA_ERR_ALIGN
    assert st(fused_args(w_sv=500)) == m.MLA_ERR_STRIDE
    assert st(fused_args(kv_sl=568)) == m.MLA_ERR_STRIDE
    for B, q in ((0, 1), (1, 1), (8, 1), (9, 1), (64, 1), (3, 3), (1024, 4)):
        assert lib.mla_attn_combine_uv_workspace_words(B, q) == 3 + (B * q + 7) // 8
    assert lib.mla_attn_combine_uv_workspace_words(-1, 1) == -1


def test_oproj_args_struct_layout_matches_header(lib, tmp_path):
    fields = [f for f, _ in m.OprojArgs._fields_]
    prog = ["#include <stdio.h>", "#include <stddef.h>", '#include "mla_combine_uv.h"',
            "int main(void) {", 'printf("%zu\\n", sizeof(mla_o_proj_args));']
    prog += [f'printf("%zu\\n", offsetof(mla_o_proj_args, {f}));' for f in fields]
    prog += ["return 0; }"]
    src = tmp_path / "probe_oproj.c"
    src.write_text("\n".join(prog))
    exe = tmp_path / "probe_oproj"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                           check=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(m.OprojArgs)
    for f, off in zip(fields, vals[1:]):
        assert getattr(m.OprojArgs, f).offset == off, f


def oproj_args(S=64, K=1536, Nout=7168, **kw):
    a = m.OprojArgs()
    a.S, a.K, a.Nout = S, K, Nout
    a.x, a.x_st = ALIGNED, K
    a.w, a.w_sj = ALIGNED * 2, K
    a.out, a.out_st = ALIGNED * 3, Nout
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_oproj_validation_errors(lib):
    fn = lib.mla_o_proj
    st = lambda a: fn(ctypes.byref(a), None)  # noqa: E731  (errors return before any CUDA call)
    assert fn(None, None) == m.MLA_ERR_NULL
    assert st(oproj_args(S=-1)) == m.MLA_ERR_SHAPE
    assert st(oproj_args(K=100)) == m.MLA_ERR_SHAPE
    assert st(oproj_args(Nout=100)) == m.MLA_ERR_SHAPE
    assert st(oproj_args(w=None)) == m.MLA_ERR_NULL
    assert st(oproj_args(x=ALIGNED + 8)) == m.MLA_ERR_ALIGN
    assert st(oproj_args(x_st=1000)) == m.MLA_ERR_STRIDE   # below K
    assert st(oproj_args(w_sj=1540)) == m.MLA_ERR_STRIDE   # not a multiple of 8
    assert st(oproj_args(out_st=100)) == m.MLA_ERR_STRIDE  # below Nout
    assert st(oproj_args(S=0, x=None, w=None, out=None)) == m.MLA_OK  # nothing to do


# ---- planning / validation without a GPU ---------------------------------

ALIGNED = 1 << 20  # fake, 16-byte aligned device addresses: never dereferenced


def args(S=64, S_out=None, H=12, P=4, q=1, spr=4, w_fmt=0, kernel=0, tile=0, **kw):
    a = Args()
    a.S, a.S_out, a.H, a.P = S, S if S_out is None else S_out, H, P
    a.q_per_request, a.splits_per_request = q, spr
    a.o, a.o_sp, a.o_st, a.o_sh = ALIGNED, S * H * 512, H * 512, 512
    a.lse, a.l_sp, a.l_st, a.l_sh = ALIGNED * 2, S * H, H, 1
    a.w_v = ALIGNED * 3
    a.w_sh, a.w_sv = (128 * 512, 512) if w_fmt == 0 else (128 * 256, 256)
    a.w_scale, a.s_sh, a.s_sv = (ALIGNED * 4, 128 * 16, 16) if w_fmt == 1 else (None, 0, 0)
    a.w_fmt = w_fmt
    a.gate, a.out = ALIGNED * 5, ALIGNED * 6
    a.kernel, a.tile_tokens = kernel, tile
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def status_of(a):
    with pytest.raises(MlaError) as e:
        mla_combine_uv_plan(a, SMS)
    return e.value.status


def test_layouts(lib):
    assert mla_combine_uv_plan(args(P=1, spr=0), SMS)["layout"] == 0
    p = mla_combine_uv_plan(args(P=16, spr=16), SMS)
    assert (p["layout"], p["n_part"]) == (1, 16)
    p = mla_combine_uv_plan(args(S=64, P=1024, q=1, spr=16), SMS)
    assert (p["layout"], p["n_part"]) == (2, 16)
    p = mla_combine_uv_plan(args(S=8, P=12, q=2, spr=3), SMS)
    assert (p["layout"], p["n_part"]) == (2, 3)
    assert status_of(args(S=8, P=7, q=2, spr=3)) == m.MLA_ERR_LAYOUT
    assert status_of(args(S=7, P=9, q=2, spr=3)) == m.MLA_ERR_LAYOUT  # S % q != 0
    assert status_of(args(P=4, spr=0)) == m.MLA_ERR_LAYOUT


def test_kernel_and_tile_choice(lib):
    # even tiny token counts run on the persistent tensor-core kernel (a
    # 16-token tile, mostly empty); split-KV decode sizes with bf16 W_V and
    # 16+ partials: 8-token tiles (two warps per token) while those give each
    # unit its own SM, else 16-token tiles when 32 would not fill the GPU
    p = mla_combine_uv_plan(args(S=4, H=2, P=4, q=2, spr=2), SMS)
    assert (p["kernel"], p["tile_tokens"], p["units"]) == (m.MLA_KERNEL_TC, 16, 2)
    p = mla_combine_uv_plan(args(S=64, P=16, spr=16), SMS)
    assert (p["kernel"], p["tile_tokens"], p["units"], p["grid"], p["threads"]) == (m.MLA_KERNEL_TC, 8, 96, 96, 512)
    assert p["smem_bytes"] <= 227 * 1024
    p = mla_combine_uv_plan(args(S=64, P=1, spr=0), SMS)  # one partial: 16-token tiles
    assert (p["tile_tokens"], p["units"]) == (16, 48)
    p = mla_combine_uv_plan(args(S=64, P=8, spr=8), SMS)  # fewer than 16 partials: 16-token tiles
    assert (p["tile_tokens"], p["units"]) == (16, 48)
    p = mla_combine_uv_plan(args(S=64, P=16, spr=16, w_fmt=1), SMS)  # MXFP4: 8-token tiles on request only
    assert (p["tile_tokens"], p["units"], p["threads"]) == (16, 48, 256)
    p = mla_combine_uv_plan(args(S=64, P=16, spr=16, w_fmt=1, tile=8), SMS)
    assert (p["tile_tokens"], p["units"], p["threads"]) == (8, 96, 512)
    p = mla_combine_uv_plan(args(S=128, P=16, spr=16), SMS)  # 192 8-token units > SMS: 16-token tiles
    assert (p["tile_tokens"], p["units"]) == (16, 96)
    p = mla_combine_uv_plan(args(S=64, P=32, spr=32, tile=8), SMS)
    assert (p["tile_tokens"], p["n_part"]) == (8, 32)
    assert status_of(args(S=64, P=33, spr=33, kernel=m.MLA_KERNEL_TC, tile=8)) == m.MLA_ERR_KERNEL
    # the cluster kernel on request: 4 CTAs of 256 threads per 16-token unit
    p = mla_combine_uv_plan(args(S=64, P=16, spr=16, kernel=m.MLA_KERNEL_KSPLIT), SMS)
    assert (p["kernel"], p["tile_tokens"], p["units"], p["grid"], p["threads"]) == (m.MLA_KERNEL_KSPLIT, 16, 48, 192, 256)
    p = mla_combine_uv_plan(args(S=4, H=2, P=1, spr=0, kernel=m.MLA_KERNEL_KSPLIT), SMS)
    assert (p["kernel"], p["layout"], p["units"], p["grid"]) == (m.MLA_KERNEL_KSPLIT, 0, 2, 8)
    assert p["smem_bytes"] <= 227 * 1024
    assert status_of(args(S=64, P=20, spr=20, kernel=m.MLA_KERNEL_KSPLIT)) == m.MLA_ERR_KERNEL
    assert status_of(args(S=64, kernel=m.MLA_KERNEL_KSPLIT, tile=32)) == m.MLA_ERR_KERNEL
    assert status_of(args(S=64, kernel=m.MLA_KERNEL_KSPLIT, tile=8)) == m.MLA_ERR_KERNEL
    assert status_of(args(S=0, S_out=4, kernel=m.MLA_KERNEL_KSPLIT)) == m.MLA_ERR_KERNEL
    # the large batch: 32-token tiles over a persistent grid of SMS CTAs
    p = mla_combine_uv_plan(args(S=4096, H=96, P=4, q=4, spr=4), SMS)
    assert (p["tile_tokens"], p["units"], p["grid"]) == (32, 96 * 128, SMS)
    assert p["smem_bytes"] <= 227 * 1024
    # 17..32 partials per token: 16-token tiles, one token per warp
    p = mla_combine_uv_plan(args(S=4096, H=96, P=20, spr=20), SMS)
    assert (p["kernel"], p["tile_tokens"], p["threads"]) == (m.MLA_KERNEL_TC, 16, 512)
    assert status_of(args(P=20, spr=20, tile=32)) == m.MLA_ERR_KERNEL
    # MXFP4 16-token tiles run two 8-warp CTAs per SM
    p = mla_combine_uv_plan(args(S=256, H=12, P=8, spr=8, w_fmt=1, tile=16), SMS)
    assert (p["tile_tokens"], p["units"], p["grid"], p["threads"]) == (16, 192, 192, 256)
    # ... but a stacked decode batch with more 16-token units than SMs gets
    # one unit per SM: 12 tiles of 22 tokens per head on the 32-token kernel
    p = mla_combine_uv_plan(args(S=256, H=12, P=8, spr=8, w_fmt=1), SMS)
    assert (p["tile_tokens"], p["units"], p["grid"], p["threads"]) == (22, 144, 144, 512)
    p = mla_combine_uv_plan(args(S=256, H=12, P=8, spr=8, w_fmt=0), SMS)
    assert (p["tile_tokens"], p["units"], p["grid"]) == (22, 144, 144)
    p = mla_combine_uv_plan(args(S=256, H=12, P=8, spr=8, tile=20), SMS)
    assert (p["tile_tokens"], p["units"]) == (20, 12 * 13)
    assert status_of(args(S=256, H=12, P=20, spr=20, tile=20)) == m.MLA_ERR_KERNEL  # <= 16 partials
    # more than 32 partials per token: CUDA cores only
    assert mla_combine_uv_plan(args(P=64, spr=64), SMS)["kernel"] == m.MLA_KERNEL_SIMT
    assert status_of(args(P=64, spr=64, kernel=m.MLA_KERNEL_TC)) == m.MLA_ERR_KERNEL
    assert status_of(args(tile=12)) == m.MLA_ERR_KERNEL
    assert status_of(args(tile=33)) == m.MLA_ERR_KERNEL
    assert status_of(args(kernel=7)) == m.MLA_ERR_KERNEL
    p = mla_combine_uv_plan(args(S=0, S_out=5, kernel=m.MLA_KERNEL_TC), SMS)
    assert p["kernel"] == m.MLA_KERNEL_SIMT  # nothing to merge: zero rows only


def test_offset_width_choice(lib):
    # 32-bit address arithmetic when every dereferenced offset is below 2^32
    assert mla_combine_uv_plan(args(S=4096, H=96, P=4, q=4, spr=4), SMS)["offsets32"] == 1
    # the request-major decode case (P=1024 partials of a 64-token batch) still fits
    assert mla_combine_uv_plan(args(S=64, P=1024, spr=16), SMS)["offsets32"] == 1
    big = 1 << 32
    a = args(S=64, P=2, spr=2)
    a.l_sp = big  # the second partial's LSE lies 2^32 elements on
    assert mla_combine_uv_plan(a, SMS)["offsets32"] == 0
    a = args(S=64, P=2, spr=2)
    a.o_sp = big - 256  # the last partial row ends past 2^32
    assert mla_combine_uv_plan(a, SMS)["offsets32"] == 0
    a = args(S=64, P=2, spr=2)
    a.o_sp = big - 64 * 12 * 512 - 512  # ... and the largest that does not
    assert mla_combine_uv_plan(a, SMS)["offsets32"] == 1
    # out of 2^25 rows x 128 wide reaches 2^32 elements
    assert mla_combine_uv_plan(args(S=64, S_out=1 << 25, H=1, P=2, spr=2), SMS)["offsets32"] == 0
    # a huge stride on a dimension of extent 1 never multiplies
    a = args(S=1, H=1, P=1, spr=0)
    a.o_st = a.o_sh = 1 << 40
    assert mla_combine_uv_plan(a, SMS)["offsets32"] == 1


def test_validation_errors(lib):
    assert status_of(args(w_fmt=3)) == m.MLA_ERR_FMT
    assert status_of(args(S=-1)) == m.MLA_ERR_SHAPE
    assert status_of(args(S=8, S_out=4)) == m.MLA_ERR_SHAPE
    assert status_of(args(H=0)) == m.MLA_ERR_SHAPE
    assert status_of(args(q=0)) == m.MLA_ERR_SHAPE
    assert status_of(args(o=None)) == m.MLA_ERR_NULL
    assert status_of(args(lse=None)) == m.MLA_ERR_NULL
    assert status_of(args(out=None)) == m.MLA_ERR_NULL
    assert status_of(args(w_fmt=1, w_scale=None)) == m.MLA_ERR_NULL
    assert status_of(args(o=ALIGNED + 8)) == m.MLA_ERR_ALIGN
    assert status_of(args(out=ALIGNED + 2)) == m.MLA_ERR_ALIGN
    assert status_of(args(o_st=12 * 512 + 4)) == m.MLA_ERR_STRIDE
    assert status_of(args(o_sh=-512)) == m.MLA_ERR_STRIDE
    assert status_of(args(w_sv=500)) == m.MLA_ERR_STRIDE
    assert status_of(args(w_fmt=1, w_sv=264)) == m.MLA_ERR_STRIDE
    # lse may be NULL only with one partial
    mla_combine_uv_plan(args(P=1, spr=0, lse=None), SMS)
    # nothing to read when S == 0: input pointers are not required
    mla_combine_uv_plan(args(S=0, S_out=3, o=None, lse=None, w_v=None, gate=None), SMS)


def test_make_args_from_strided_views(lib):
    import torch

    big = torch.zeros(2, 8, 16, 512, dtype=torch.bfloat16)
    o = big[:, :, 4:10]  # heads strided view
    lse = torch.zeros(2, 8, 6)
    w = torch.zeros(6, 128, 512, dtype=torch.bfloat16)
    gate = torch.zeros(8, 6 * 128, dtype=torch.bfloat16)
    out = torch.zeros(8, 6 * 128, dtype=torch.bfloat16)
    a = make_args(o, lse, 1, 2, w, 0, gate, out)
    assert (a.P, a.S, a.H, a.S_out) == (2, 8, 6, 8)
    assert (a.o_sp, a.o_st, a.o_sh) == (8 * 16 * 512, 16 * 512, 512)
    assert a.o == o.data_ptr()
    p = mla_combine_uv_plan(a, SMS)
    assert p["layout"] == 1


def test_plan_invariants_on_random_problems(lib):
    """Seeded random problems through the planner: every call either returns
    one of the documented errors or a plan whose launch respects the kernel
    limits (units cover every token, grid no larger than units or resident
    CTAs, shared memory within 227 KB, 32-token tiles only up to 16 partials,
    automatic 8-token tiles only where documented)."""
    import numpy as np

    rng = np.random.default_rng(77)
    errors = {m.MLA_ERR_LAYOUT, m.MLA_ERR_KERNEL, m.MLA_ERR_SHAPE}
    seen = set()
    for _ in range(3000):
        q = int(rng.choice([1, 2, 3, 4]))
        S = int(rng.integers(0, 80)) * q if rng.random() < 0.8 else int(rng.integers(0, 5000))
        H = int(rng.choice([1, 2, 3, 12, 96, 128]))
        layout = rng.choice(["pass", "compact", "request_major", "bad"])
        spr = int(rng.integers(1, 48))
        P = {"pass": 1, "compact": spr, "request_major": max(1, S // q) * spr,
             "bad": spr + 1}[layout]
        if layout == "pass":
            spr = 0
        w_fmt = int(rng.integers(0, 2))
        kernel = int(rng.choice([0, 0, m.MLA_KERNEL_SIMT, m.MLA_KERNEL_TC, m.MLA_KERNEL_KSPLIT]))
        tile = int(rng.choice([0, 0, 8, 16, 32, 24]))
        a = args(S=S, S_out=S + int(rng.integers(0, 4)), H=H, P=P, q=q, spr=spr, w_fmt=w_fmt,
                 kernel=kernel, tile=tile)
        try:
            p = mla_combine_uv_plan(a, SMS)
        except MlaError as e:
            assert e.status in errors, (e.status, S, H, P, q, spr, kernel, tile)
            continue
        n = p["n_part"]
        seen.add((p["kernel"], p["tile_tokens"]))
        assert p["smem_bytes"] <= 227 * 1024
        if p["kernel"] == m.MLA_KERNEL_TC:
            t = p["tile_tokens"]
            assert (t in (8, 16, 32) or 16 < t < 32) and (tile == 0 or t == tile)
            assert p["units"] == H * -(-S // t) and 1 <= p["grid"] <= min(p["units"], 2 * SMS)
            assert n <= (16 if t > 16 else 32)
            if tile == 0 and 16 < t < 32:  # runtime tiles: one unit per SM
                assert p["units"] <= SMS
            assert p["threads"] == (256 if (w_fmt and t == 16 and n <= 16) else 512)
            if tile == 0 and t == 8:
                assert w_fmt == 0 and n >= 16 and H * -(-S // 8) <= SMS
        elif p["kernel"] == m.MLA_KERNEL_KSPLIT:
            assert p["tile_tokens"] == 16 and n <= 16 and p["grid"] == 4 * p["units"]
        else:
            assert p["kernel"] == m.MLA_KERNEL_SIMT and p["grid"] == p["units"]
    # the random draws reached every kernel and every tensor-core tile
    assert {(m.MLA_KERNEL_TC, 8), (m.MLA_KERNEL_TC, 16), (m.MLA_KERNEL_TC, 32), (m.MLA_KERNEL_TC, 24),
            (m.MLA_KERNEL_KSPLIT, 16)} <= seen
    assert any(k == m.MLA_KERNEL_SIMT for k, _ in seen)
