"""ctypes binding of libqi21.so (include/qi21.h).

Argument marshalling only: every step of the prefill and the step runs in
the library's CUDA kernels. PyTorch tensors are accepted as device buffers
(their data pointers are passed through); torch never computes on the path.
Loading fails loudly if the library has not been built -- there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libqi21.so")

OK = 0
ERR = {
    -1: "QI21_ERR_ARG", -2: "QI21_ERR_SHAPE", -3: "QI21_ERR_GEOM", -4: "QI21_ERR_MASK",
    -5: "QI21_ERR_OOM", -6: "QI21_ERR_CUDA", -7: "QI21_ERR_STATE", -8: "QI21_ERR_WORKSPACE",
    -9: "QI21_ERR_DEVICE", -10: "QI21_ERR_NONFINITE",
}
SEG_TEXT = 0
SEG_IMAGE = 1
EPI_F16, EPI_F32, EPI_RESID, EPI_SWIGLU = 0, 1, 2, 3
DTYPE_F16, DTYPE_BF16 = 0, 1
ELEM_F16, ELEM_BF16, ELEM_F32 = 2, 3, 4


class Qi21Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERR.get(code, code)}: {msg}")
        self.code = code


class LayerFp8(C.Structure):
    _fields_ = [("wqkv", C.c_void_p), ("wo", C.c_void_p), ("w13", C.c_void_p), ("w2", C.c_void_p),
                ("s_qkv", C.c_void_p), ("s_o", C.c_void_p), ("s_13", C.c_void_p), ("s_2", C.c_void_p),
                ("norm_q", C.c_void_p), ("norm_k", C.c_void_p)]


class Geom(C.Structure):
    _fields_ = [("dim", C.c_int32), ("heads", C.c_int32), ("head_dim", C.c_int32),
                ("mlp_hidden", C.c_int32), ("layers", C.c_int32), ("axes", C.c_int32 * 3),
                ("eps", C.c_float), ("theta", C.c_float), ("dtype", C.c_int32)]


class Seg(C.Structure):
    _fields_ = [("kind", C.c_int32), ("a", C.c_int32), ("b", C.c_int32)]


class Layer(C.Structure):
    _fields_ = [("wqkv", C.c_void_p), ("wo", C.c_void_p), ("w13", C.c_void_p), ("w2", C.c_void_p),
                ("norm_q", C.c_void_p), ("norm_k", C.c_void_p)]


_vp = C.c_void_p
_i32 = C.c_int32
_sz = C.c_size_t
_f = C.c_float

# name -> (restype, argtypes)
_SIGS = {
    "qi21_last_error": (C.c_char_p, []),
    "qi21_version": (C.c_char_p, []),
    "qi21_geom_check": (C.c_int, [C.POINTER(Geom)]),
    "qi21_layout_rows": (C.c_int, [C.POINTER(Seg), _i32, C.POINTER(_i32), C.POINTER(_i32), C.POINTER(_i32)]),
    "qi21_layout_indices": (C.c_int, [C.POINTER(Seg), _i32, C.POINTER(_i32), _f, _vp, _vp, _vp, _vp, _vp]),
    "qi21_layer_plane_bytes": (_sz, [C.POINTER(Geom)]),
    "qi21_workspace_bytes": (_sz, [C.POINTER(Geom), _i32]),
    "qi21_pack_layer": (C.c_int, [C.POINTER(Geom), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                                  C.POINTER(Layer), _vp]),
    "qi21_kvcache_alloc": (C.c_int, [C.POINTER(Geom), C.POINTER(Seg), _i32, C.POINTER(_vp)]),
    "qi21_kvcache_free": (None, [_vp]),
    "qi21_kvcache_info": (C.c_int, [_vp, C.POINTER(_i32), C.POINTER(_i32), C.POINTER(_i32)]),
    "qi21_kvcache_layer": (C.c_int, [_vp, _i32, C.POINTER(_vp)]),
    "qi21_prefill": (C.c_int, [C.POINTER(Geom), C.POINTER(Layer), _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "qi21_step": (C.c_int, [C.POINTER(Geom), C.POINTER(Layer), _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "qi21_step_batch": (C.c_int, [C.POINTER(Geom), C.POINTER(Layer), C.POINTER(_vp), _i32, _vp, _vp, _vp,
                                  _vp, _vp, _sz, _vp]),
    "qi21_embed": (C.c_int, [_i32, _i32, _i32, _vp, _vp, _vp, _vp]),
    "qi21_final": (C.c_int, [_i32, _i32, _i32, _f, _vp, _vp, _vp, _vp, _vp]),
    "qi21_set_checks": (C.c_uint32, [C.c_uint32]),
    "qi21_amax_read": (C.c_int, [_vp, _i32]),
    "qi21_layer_fp8_bytes": (C.c_size_t, [_vp]),
    "qi21_workspace_bytes_fp8": (C.c_size_t, [_vp, _i32]),
    "qi21_pack_layer_fp8": (C.c_int, [_vp, _vp, _vp, C.c_size_t, _vp, _vp]),
    "qi21_prefill_fp8": (C.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, C.c_size_t, _vp]),
    "qi21_step_batch_fp8": (C.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, C.c_size_t, _vp]),
    "qi21_op_quant_rows": (C.c_int, [_i32, _i32, _vp, _vp, _vp, _vp]),
    "qi21_op_rowop_fp8": (C.c_int, [_i32, _i32, _f, _vp, _vp, _vp, _vp, _vp]),
    "qi21_op_gemm_fp8": (C.c_int, [_i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _vp]),
    "qi21_graph_step_batch": (C.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, C.c_size_t, C.POINTER(_vp)]),
    "qi21_graph_denoise_batch": (C.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, C.c_size_t,
                                           C.POINTER(_vp)]),
    "qi21_graph_step_batch_fp8": (C.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp, _vp, C.c_size_t, C.POINTER(_vp)]),
    "qi21_graph_launch": (C.c_int, [_vp, _vp]),
    "qi21_graph_free": (None, [_vp]),
    "qi21_count_nonfinite": (C.c_int, [_vp, C.c_size_t, _i32, C.POINTER(C.c_uint64), _vp]),
    "qi21_timestep_mods": (C.c_int, [_i32, _f, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "qi21_denoise_batch": (C.c_int, [C.POINTER(Geom), C.POINTER(Layer), C.POINTER(_vp), _i32, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _vp, _sz, _vp]),
    "qi21_denoise": (C.c_int, [C.POINTER(Geom), C.POINTER(Layer), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz,
                               _vp]),
    "qi21_step_noalloc": (C.c_int, [C.POINTER(Geom), C.POINTER(Layer), _vp, _vp, _vp, _vp, _vp]),
    "qi21_device_status": (C.c_int, []),
    "qi21_selftest_wait_timeout": (C.c_int, [_vp]),
    "qi21_profile_enable": (C.c_int, [C.c_int]),
    "qi21_profile_read": (C.c_int, [_vp, _vp]),
    "qi21_op_rowop": (C.c_int, [_i32, _i32, _i32, _f, _vp, _vp, _vp, _vp, _vp, _vp]),
    "qi21_op_mods_prep": (C.c_int, [_i32, _vp, _vp, _vp]),
    "qi21_op_gemm": (C.c_int, [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _vp]),
    "qi21_op_gemm_split": (C.c_int, [_i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _sz,
                                     C.POINTER(_i32), _vp]),
    "qi21_op_qkrope": (C.c_int, [_i32, _i32, _i32, _f, _vp, _vp, _vp, _vp, _vp, _vp]),
    "qi21_op_kvcopy": (C.c_int, [_i32, _i32, _vp, _vp, _vp]),
    "qi21_op_attention": (C.c_int, [_i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp, _vp, _vp]),
}

_lib = None


def load() -> C.CDLL:
    """The loaded library. Raises if libqi21.so has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it first (python -m "
                "diffusion_transformer_denoiser_qi21_gb300.build); there is no fallback path")
        lib = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols() -> list:
    return list(_SIGS)


def check(rc: int) -> None:
    if rc != OK:
        raise Qi21Error(rc, load().qi21_last_error().decode())


def geom(dim, heads, mlp_hidden, layers, axes=(16, 56, 56), eps=1e-6, theta=10000.0, head_dim=128,
         dtype=DTYPE_F16) -> Geom:
    """qi21_geom; dtype DTYPE_F16 / DTYPE_BF16 (or "f16" / "bf16")."""
    if isinstance(dtype, str):
        dtype = {"f16": DTYPE_F16, "bf16": DTYPE_BF16}[dtype]
    g = Geom()
    g.dim, g.heads, g.head_dim, g.mlp_hidden, g.layers = dim, heads, head_dim, mlp_hidden, layers
    g.axes[:] = list(axes)
    g.eps, g.theta = eps, theta
    g.dtype = dtype
    return g


def segs_array(segs):
    arr = (Seg * len(segs))()
    for i, (k, a, b) in enumerate(segs):
        arr[i].kind, arr[i].a, arr[i].b = k, a, b
    return arr


def layout_rows(segs):
    t, p, n = _i32(), _i32(), _i32()
    check(load().qi21_layout_rows(segs_array(segs), len(segs), C.byref(t), C.byref(p), C.byref(n)))
    return t.value, p.value, n.value


def layout_indices(segs, axes=(16, 56, 56), theta=10000.0):
    """(pos int64 [rows,3], block_ids int32 [rows], vis uint32 [lp],
    cos f32 [rows, hd/2], sin) from the library's host index construction."""
    total, lp, _ = layout_rows(segs)
    half = sum(axes) // 2
    pos = np.zeros((total, 3), np.int64)
    ids = np.zeros(total, np.int32)
    vis = np.zeros(lp, np.uint32)
    cs = np.zeros((total, half), np.float32)
    sn = np.zeros((total, half), np.float32)
    ax = (_i32 * 3)(*axes)
    check(load().qi21_layout_indices(segs_array(segs), len(segs), ax, theta, pos.ctypes.data,
                                     ids.ctypes.data, vis.ctypes.data, cs.ctypes.data, sn.ctypes.data))
    return pos, ids, vis, cs, sn


def layer_plane_bytes(g: Geom) -> int:
    return load().qi21_layer_plane_bytes(C.byref(g))


def workspace_bytes(g: Geom, rows: int) -> int:
    return load().qi21_workspace_bytes(C.byref(g), rows)


def device_status() -> int:
    return load().qi21_device_status()


CLASSES = ("rowop", "qkv", "qkrope", "kvcopy", "attention", "o", "gateup", "down", "misc", "embed", "final", "temb", "quant")


def profile_enable(on: bool) -> None:
    check(load().qi21_profile_enable(1 if on else 0))


def profile_read():
    """({class: ms since enable/last read}, {class: launches since load})."""
    ms = np.zeros(len(CLASSES), np.float32)
    n = np.zeros(len(CLASSES), np.int64)
    check(load().qi21_profile_read(ms.ctypes.data, n.ctypes.data))
    return dict(zip(CLASSES, ms.tolist())), dict(zip(CLASSES, n.tolist()))
