"""Host-side checks of the library (no GPU): it loads, exports every symbol
include/qi21.h declares, rejects bad arguments with the documented codes,
and builds positions / block ids / visibility bit-exactly like the oracle
(RoPE tables within a few ulp)."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import diffusion_transformer_denoiser_qi21_gb300 as q
from diffusion_transformer_denoiser_qi21_gb300 import _binding as B
from oracle import qi21_oracle as O
from synthetic import qi21_inputs as S

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "qi21.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(qi21_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    lib = q.load()
    names = _header_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert set(B.exported_symbols()) == set(names)


def test_version_and_no_error_initially():
    assert b"sm_103a" in q.load().qi21_version()


LAYOUTS = [
    [(0, 3, 0), (1, 2, 3)],
    [(0, 2, 0), (1, 2, 4), (0, 1, 0), (1, 1, 1)],
    [(0, 18, 0), (1, 64, 64), (1, 64, 64)],
    [(0, 5, 0), (1, 4, 6), (0, 3, 0), (1, 3, 2), (1, 10, 13)],
    [(0, 1, 0), (1, 1, 1)],
    [(1, 3, 5), (0, 4, 0), (1, 7, 2)],
] + [S.WORKLOADS[k].segs(s) for k in S.WORKLOADS for s in range(S.WORKLOADS[k].nseq)]


@pytest.mark.parametrize("segs", LAYOUTS)
def test_layout_indices_match_oracle(segs):
    pos, ids, vis, cs, sn = q.layout_indices(segs)
    np.testing.assert_array_equal(pos, O.positions(segs))
    np.testing.assert_array_equal(ids, O.block_ids(segs))
    np.testing.assert_array_equal(vis, O.prefix_visibility(segs))
    oc, osn = O.rope_tables(O.positions(segs))
    # same f32 formula, different libm: a few ulp of values in [-1, 1]
    assert np.max(np.abs(cs - oc)) <= 4e-7 * max(1.0, float(np.abs(pos).max()))
    assert np.max(np.abs(sn - osn)) <= 4e-7 * max(1.0, float(np.abs(pos).max()))
    total, lp, n = q.layout_rows(segs)
    assert (total, lp, n) == (O.total_rows(segs), O.prefix_len(segs), O.seg_len(segs[-1]))


@pytest.mark.parametrize("segs,code", [
    ([(0, 3, 0)], -2),             # no target image
    ([(1, 2, 2)], -2),             # empty prefix
    ([(0, 3, 0), (1, 0, 4)], -2),  # empty target
    ([(0, -1, 0), (1, 2, 2)], -1),  # negative length
    ([(7, 1, 1), (1, 2, 2)], -1),  # unknown kind
])
def test_layout_errors(segs, code):
    with pytest.raises(q.Qi21Error) as e:
        q.layout_rows(segs)
    assert e.value.code == code


@pytest.mark.parametrize("kw,code", [
    (dict(dim=256, heads=2, mlp_hidden=768, layers=1, head_dim=64), -3),
    (dict(dim=256, heads=3, mlp_hidden=768, layers=1), -3),
    (dict(dim=192, heads=1, mlp_hidden=768, layers=1, head_dim=192), -3),
    (dict(dim=256, heads=2, mlp_hidden=700, layers=1), -3),
    (dict(dim=256, heads=2, mlp_hidden=768, layers=0), -3),
    (dict(dim=256, heads=2, mlp_hidden=768, layers=1, axes=(16, 56, 58)), -3),
    (dict(dim=256, heads=2, mlp_hidden=768, layers=1, axes=(15, 57, 56)), -3),
    (dict(dim=256, heads=2, mlp_hidden=768, layers=1, dtype=2), -3),
    (dict(dim=256, heads=2, mlp_hidden=768, layers=1, dtype=-1), -3),
])
def test_geometry_errors(kw, code):
    g = q.geom(**kw)
    assert q.load().qi21_geom_check(C.byref(g)) == code
    assert q.workspace_bytes(g, 10) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_geometry_ok_and_sizes(dtype):
    g = q.geom(4096, 32, 12288, 32, dtype=dtype)
    assert q.load().qi21_geom_check(C.byref(g)) == 0
    H, I = 4096, 12288
    assert q.layer_plane_bytes(g) == 2 * (3 * H * H + H * H + 2 * I * H + H * I)
    M = 4096
    per_row = 4 * H + 2 * H + 6 * H + 2 * H + 2 * I
    fixed = 16 * H + 4096  # the modulation vectors and the GEMMs' K-split merge flags
    assert q.workspace_bytes(g, M) >= M * per_row + fixed
    assert q.workspace_bytes(g, M) < M * per_row + fixed + 8 * 256


def test_empty_inputs_are_no_ops():
    # zero rows (queries, codes) are valid and enqueue nothing: every
    # single-operation entry point returns 0 before it looks at a pointer
    # or touches the device (no CUDA context is needed here)
    lib = q.load()
    for dt in (0, 1):
        assert lib.qi21_op_gemm(dt, 0, 0, 128, 64, None, None, None, 128, None, None) == 0
        assert lib.qi21_op_gemm(dt, 2, 0, 256, 64, None, None, None, 256, None, None) == 0  # residual, no gate
        assert lib.qi21_op_rowop(dt, 0, 256, 1e-6, None, None, None, None, None, None) == 0
        assert lib.qi21_op_qkrope(dt, 0, 2, 1e-6, None, None, None, None, None, None) == 0
        assert lib.qi21_op_attention(dt, 0, 2, None, None, 0, 0, None, None, None) == 0
        assert lib.qi21_op_gemm_split(dt, 0, 0, 128, 64, None, None, None, 128, None, None, 0, None, None) == 0
    assert lib.qi21_op_kvcopy(0, 256, None, None, None) == 0
    assert lib.qi21_op_quant_rows(0, 256, None, None, None, None) == 0
    assert lib.qi21_op_rowop_fp8(0, 256, 1e-6, None, None, None, None, None) == 0
    assert lib.qi21_op_gemm_fp8(1, 0, 256, 128, None, None, None, None, None, 256, None, None) == 0
    # negative sizes are refused
    assert lib.qi21_op_gemm(0, 0, -1, 128, 64, None, None, None, 128, None, None) == -2
    assert lib.qi21_op_attention(0, -1, 2, None, None, 0, 0, None, None, None) == -2


def test_device_entry_points_reject_bad_args_before_touching_the_device():
    lib = q.load()
    g = q.geom(256, 2, 768, 1)
    # null cache / pointers -> ARG, nothing enqueued (no CUDA context needed)
    assert lib.qi21_prefill(C.byref(g), None, None, None, None, None, None, 0, None) == -1
    assert lib.qi21_step(C.byref(g), None, None, None, None, None, None, None, 0, None) == -1
    for dt in (0, 1):
        assert lib.qi21_op_gemm(dt, 0, 128, 100, 64, 8, 8, 8, 128, None, None) == -2  # N % 128
        assert lib.qi21_op_gemm(dt, 9, 128, 128, 64, 8, 8, 8, 128, None, None) == -1  # epilogue
        assert lib.qi21_op_rowop(dt, 4, 6, 1e-6, 8, None, None, 8, 8, None) == -2    # dim % 4
        assert lib.qi21_op_attention(dt, 10, 2, 8, None, 0, 5, None, 8, None) == -2  # nq > own rows
    # an unknown 16-bit type
    assert lib.qi21_op_gemm(5, 0, 128, 128, 64, 8, 8, 8, 128, None, None) == -1
    assert lib.qi21_op_rowop(-1, 4, 8, 1e-6, 8, None, None, 8, 8, None) == -1
    assert lib.qi21_op_attention(2, 1, 2, 8, None, 0, 5, None, 8, None) == -1
    assert lib.qi21_op_qkrope(3, 1, 2, 1e-6, 8, 8, 8, 8, 8, None) == -1
    bad = q.geom(256, 2, 768, 1, head_dim=64)
    assert lib.qi21_prefill(C.byref(bad), None, None, None, None, None, None, 0, None) == -3
    assert b"head_dim" in lib.qi21_last_error()
    # the FP8 variant takes f16 geometries only
    gb = q.geom(256, 2, 768, 1, dtype="bf16")
    assert lib.qi21_layer_fp8_bytes(C.byref(gb)) == 0
    assert lib.qi21_workspace_bytes_fp8(C.byref(gb), 16) == 0
    assert lib.qi21_prefill_fp8(C.byref(gb), None, None, None, None, None, None, 0, None) == -3
    assert b"FP8" in lib.qi21_last_error()
    assert lib.qi21_layer_fp8_bytes(C.byref(g)) > 0
    # the finite scan's element types
    out = C.c_uint64(0)
    assert lib.qi21_count_nonfinite(None, 0, 8, C.byref(out), None) == -1
    assert lib.qi21_count_nonfinite(None, 0, 1, C.byref(out), None) == -1
