"""GB300 (sm_103a) Qwen-Image-2.1 single-stream DiT block: prefill of the
prompt prefix into a per-layer K/V cache and the denoiser step against it.

Thin Python face of the C ABI in include/qi21.h (same names, argument
marshalling only). Device buffers are torch CUDA tensors; streams are
torch.cuda streams. There is no CPU fallback: the library must be built
(``build()``) and a CUDA device present for any device call.
"""
from __future__ import annotations

import ctypes as C

from . import _binding as B
from ._binding import (DTYPE_BF16, DTYPE_F16, EPI_F16, EPI_F32, EPI_RESID, EPI_SWIGLU, SEG_IMAGE,  # noqa: F401
                       SEG_TEXT, Geom, Qi21Error,
                       CLASSES, check, device_status, exported_symbols, profile_enable, profile_read, geom, layer_plane_bytes, layout_indices,
                       layout_rows, load, workspace_bytes)

__all__ = [
    "Geom", "Qi21Error", "KVCache", "geom", "layout_rows", "layout_indices", "layer_plane_bytes",
    "workspace_bytes", "pack_layer", "prefill", "step", "step_noalloc", "step_batch", "embed", "final",
    "timestep_mods", "denoise", "set_checks", "PackedLayerFp8", "pack_layer_fp8", "workspace_bytes_fp8",
    "prefill_fp8", "step_batch_fp8", "op_quant_rows", "op_rowop_fp8", "op_gemm_fp8", "Graph", "graph_step_batch", "graph_step_batch_fp8", "graph_denoise_batch", "count_nonfinite", "CHECK_FINITE", "CHECK_AMAX", "AMAX_SITES", "amax_read", "denoise_batch", "device_status", "selftest_wait_timeout", "build",
    "profile_enable", "profile_read", "CLASSES", "op_rowop", "op_mods_prep", "op_gemm", "op_gemm_split", "op_qkrope", "op_kvcopy", "op_attention",
]


def build(**kw) -> str:
    from .make import build as _b
    return _b(**kw)


def _torch():
    import torch
    return torch


def _ptr(t, dtype=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (or None -> NULL)."""
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def dtype_of(g):
    """The torch dtype of a geometry's 16-bit buffers."""
    torch = _torch()
    return torch.bfloat16 if int(getattr(g, "dtype", 0)) == DTYPE_BF16 else torch.float16


def _dt_code(t):
    """QI21_DTYPE_* of a 16-bit torch tensor."""
    torch = _torch()
    if t.dtype == torch.float16:
        return DTYPE_F16
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"expected an f16 or bf16 tensor, got {t.dtype}")


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class PackedLayer:
    """One block's packed device planes (keeps the plane buffer and the norm
    weights alive) and the C struct pointing into them."""

    def __init__(self, planes, norm_q, norm_k, cstruct):
        self.planes = planes
        self.norm_q = norm_q
        self.norm_k = norm_k
        self.c = cstruct


def pack_layer(g: Geom, wq, wk, wv, wo, wgate, wup, wdown, norm_q, norm_k, stream=None) -> PackedLayer:
    """qi21_pack_layer: device weights of the geometry's dtype (f16 or bf16)
    in nn.Linear layout -> packed planes."""
    torch = _torch()
    lib = load()
    nbytes = lib.qi21_layer_plane_bytes(C.byref(g))
    if nbytes == 0:
        check(lib.qi21_geom_check(C.byref(g)))
    planes = torch.empty(nbytes, dtype=torch.uint8, device=wq.device)
    out = B.Layer()
    h = dtype_of(g)
    nq = norm_q.contiguous()
    nk = norm_k.contiguous()
    check(lib.qi21_pack_layer(C.byref(g), _ptr(wq, h, "wq"), _ptr(wk, h, "wk"), _ptr(wv, h, "wv"),
                              _ptr(wo, h, "wo"), _ptr(wgate, h, "wgate"), _ptr(wup, h, "wup"),
                              _ptr(wdown, h, "wdown"), _ptr(nq, torch.float32, "norm_q"),
                              _ptr(nk, torch.float32, "norm_k"), planes.data_ptr(), nbytes, C.byref(out),
                              _stream(stream)))
    return PackedLayer(planes, nq, nk, out)


def _layer_array(layers):
    arr = (B.Layer * len(layers))()
    for i, l in enumerate(layers):
        arr[i] = l.c
    return arr


class KVCache:
    """qi21_kvcache_alloc / qi21_kvcache_free: a per-prompt K/V cache owned
    by the library."""

    def __init__(self, g: Geom, segs):
        self.g = g
        self.segs = list(segs)
        h = C.c_void_p()
        check(load().qi21_kvcache_alloc(C.byref(g), B.segs_array(self.segs), len(self.segs), C.byref(h)))
        self.handle = h
        lp, n, L = C.c_int32(), C.c_int32(), C.c_int32()
        check(load().qi21_kvcache_info(h, C.byref(lp), C.byref(n), C.byref(L)))
        self.lp, self.n, self.layers = lp.value, n.value, L.value

    def layer_ptr(self, layer: int) -> int:
        p = C.c_void_p()
        check(load().qi21_kvcache_layer(self.handle, layer, C.byref(p)))
        return p.value

    def layer_tensor(self, layer: int):
        """A torch [lp, 2H] copy of layer `layer`'s K|V in the geometry's
        dtype (for checks)."""
        torch = _torch()
        raw = _device_view(self.layer_ptr(layer), (self.lp, 2 * self.g.dim), "<i2").clone()
        return raw.view(dtype_of(self.g))

    def free(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            load().qi21_kvcache_free(self.handle)
            self.handle = C.c_void_p()

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class _DevArray:
    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _device_view(ptr: int, shape, typestr):
    """A torch view of library-owned device memory (no copy)."""
    torch = _torch()
    return torch.as_tensor(_DevArray(ptr, shape, typestr), device="cuda")


def prefill(g: Geom, layers, cache: KVCache, x_prefix, mods0, workspace, x_layers=None, stream=None):
    """qi21_prefill."""
    torch = _torch()
    f = torch.float32
    check(load().qi21_prefill(C.byref(g), _layer_array(layers), cache.handle, _ptr(x_prefix, f, "x_prefix"),
                              _ptr(mods0, f, "mods0"), _ptr(x_layers, f, "x_layers"),
                              _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                              _stream(stream)))


def step(g: Geom, layers, cache: KVCache, x_in, x_out, mods, workspace, x_layers=None, stream=None):
    """qi21_step."""
    torch = _torch()
    f = torch.float32
    check(load().qi21_step(C.byref(g), _layer_array(layers), cache.handle, _ptr(x_in, f, "x_in"),
                           _ptr(x_out, f, "x_out"), _ptr(mods, f, "mods"), _ptr(x_layers, f, "x_layers"),
                           _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                           _stream(stream)))


def step_noalloc(g: Geom, layers, cache: KVCache, x_in, x_out, mods, stream=None):
    """qi21_step_noalloc: the step with the library's static device scratch
    instead of a caller workspace (for callers that cannot allocate)."""
    torch = _torch()
    f = torch.float32
    check(load().qi21_step_noalloc(C.byref(g), _layer_array(layers), cache.handle, _ptr(x_in, f, "x_in"),
                                   _ptr(x_out, f, "x_out"), _ptr(mods, f, "mods"), _stream(stream)))


def embed(tok, w_in, x, stream=None):
    """qi21_embed: x [n, dim] = tok [n, 64] w_in^T (f32)."""
    torch = _torch()
    f = torch.float32
    check(load().qi21_embed(tok.shape[0], x.shape[1], tok.shape[1], _ptr(tok, f, "tok"), _ptr(w_in, f, "w_in"),
                            _ptr(x, f, "x"), _stream(stream)))


def final(x, final_scale, w_out, out, eps=1e-6, stream=None):
    """qi21_final: out [n, 64] = (LN(x)(1 + final_scale)) w_out^T (f32)."""
    torch = _torch()
    f = torch.float32
    check(load().qi21_final(x.shape[0], x.shape[1], w_out.shape[0], eps, _ptr(x, f, "x"),
                            _ptr(final_scale, f, "final_scale"), _ptr(w_out, f, "w_out"), _ptr(out, f, "out"),
                            _stream(stream)))


class Graph:
    """A recorded step or denoiser call (qi21_graph_*): replay with
    ``launch``. Bound to the tensors given at capture, which it keeps
    alive; change their contents, not their storage."""

    def __init__(self, handle, keep):
        self.handle = handle
        self._keep = keep

    def launch(self, stream=None):
        check(load().qi21_graph_launch(self.handle, _stream(stream)))

    def free(self):
        if self.handle:
            load().qi21_graph_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


def graph_step_batch(g: Geom, layers, caches, x_in, x_out, mods, workspace) -> Graph:
    """qi21_graph_step_batch: record one step of every cache's sequence."""
    torch = _torch()
    f = torch.float32
    arr = (C.c_void_p * len(caches))(*[c.handle.value for c in caches])
    h = C.c_void_p()
    lay = _layer_array(layers)
    check(load().qi21_graph_step_batch(C.byref(g), lay, arr, len(caches), _ptr(x_in, f, "x_in"),
                                       _ptr(x_out, f, "x_out"), _ptr(mods, f, "mods"),
                                       _ptr(workspace, None, "workspace"),
                                       workspace.numel() * workspace.element_size(), C.byref(h)))
    return Graph(h, (layers, caches, x_in, x_out, mods, workspace, lay))


def graph_step_batch_fp8(g: Geom, layers8, caches, x_in, x_out, mods, workspace) -> Graph:
    """qi21_graph_step_batch_fp8: record one FP8 step of every cache's sequence."""
    torch = _torch()
    f = torch.float32
    arr = (C.c_void_p * len(caches))(*[c.handle.value for c in caches])
    h = C.c_void_p()
    lay = _layer8_array(layers8)
    check(load().qi21_graph_step_batch_fp8(C.byref(g), lay, arr, len(caches), _ptr(x_in, f, "x_in"),
                                           _ptr(x_out, f, "x_out"), _ptr(mods, f, "mods"),
                                           _ptr(workspace, None, "workspace"),
                                           workspace.numel() * workspace.element_size(), C.byref(h)))
    return Graph(h, (layers8, caches, x_in, x_out, mods, workspace, lay))


def graph_denoise_batch(g: Geom, layers, caches, tok, w_in, mods, final_scale, w_out, out, workspace) -> Graph:
    """qi21_graph_denoise_batch: record one latent-tokens -> velocity call."""
    torch = _torch()
    f = torch.float32
    arr = (C.c_void_p * len(caches))(*[c.handle.value for c in caches])
    h = C.c_void_p()
    lay = _layer_array(layers)
    check(load().qi21_graph_denoise_batch(C.byref(g), lay, arr, len(caches), _ptr(tok, f, "tok"),
                                          _ptr(w_in, f, "w_in"), _ptr(mods, f, "mods"),
                                          _ptr(final_scale, f, "final_scale"), _ptr(w_out, f, "w_out"),
                                          _ptr(out, f, "out"), _ptr(workspace, None, "workspace"),
                                          workspace.numel() * workspace.element_size(), C.byref(h)))
    return Graph(h, (layers, caches, tok, w_in, mods, final_scale, w_out, out, workspace, lay))


CHECK_FINITE = 1
CHECK_AMAX = 2
AMAX_SITES = ("attn-in", "qkv", "attn-out", "ffn-in", "hidden")


def amax_read(reset=True) -> dict:
    """qi21_amax_read: {site: largest |value|} of the AMAX probe (synchronises)."""
    import numpy as np
    out = np.zeros(5, np.float32)
    check(load().qi21_amax_read(out.ctypes.data, 1 if reset else 0))
    return dict(zip(AMAX_SITES, out.tolist()))


def set_checks(flags: int) -> int:
    """qi21_set_checks: process-wide optional checks (CHECK_FINITE); returns
    the previous flags."""
    return int(load().qi21_set_checks(int(flags)))


def count_nonfinite(x, stream=None) -> int:
    """qi21_count_nonfinite: NaN/Inf count of a CUDA f32, f16 or bf16 tensor
    (synchronises the stream)."""
    torch = _torch()
    eb = {torch.float32: B.ELEM_F32, torch.float16: B.ELEM_F16, torch.bfloat16: B.ELEM_BF16}.get(x.dtype)
    if eb is None:
        raise TypeError("count_nonfinite takes f32, f16 or bf16 tensors")
    out = C.c_uint64(0)
    check(load().qi21_count_nonfinite(_ptr(x, x.dtype, "x"), x.numel(), eb, C.byref(out), _stream(stream)))
    return int(out.value)


def timestep_mods(t, t_lin1, t_lin2, modulation, norm_out, mods, final_scale, work=None, stream=None):
    """qi21_timestep_mods: mods [4 dim] and final_scale [dim] of the model
    input t (f32 weights t_lin1 [dim, 256], t_lin2, modulation, norm_out)."""
    torch = _torch()
    f = torch.float32
    dim = t_lin2.shape[0]
    if work is None:
        work = torch.empty(2 * dim, dtype=f, device=mods.device)
    check(load().qi21_timestep_mods(dim, float(t), _ptr(t_lin1, f, "t_lin1"), _ptr(t_lin2, f, "t_lin2"),
                                    _ptr(modulation, f, "modulation"), _ptr(norm_out, f, "norm_out"),
                                    _ptr(work, f, "work"), _ptr(mods, f, "mods"),
                                    _ptr(final_scale, f, "final_scale"), _stream(stream)))


def denoise_batch(g: Geom, layers, caches, tok, w_in, mods, final_scale, w_out, out, workspace, stream=None):
    """qi21_denoise_batch: latent tokens -> velocity for one or more sequences."""
    torch = _torch()
    f = torch.float32
    arr = (C.c_void_p * len(caches))(*[c.handle.value for c in caches])
    check(load().qi21_denoise_batch(C.byref(g), _layer_array(layers), arr, len(caches), _ptr(tok, f, "tok"),
                                    _ptr(w_in, f, "w_in"), _ptr(mods, f, "mods"),
                                    _ptr(final_scale, f, "final_scale"), _ptr(w_out, f, "w_out"),
                                    _ptr(out, f, "out"), _ptr(workspace, None, "workspace"),
                                    workspace.numel() * workspace.element_size(), _stream(stream)))


def denoise(g: Geom, layers, cache, tok, w_in, mods, final_scale, w_out, out, workspace, stream=None):
    """qi21_denoise: latent tokens [n, 64] -> velocity [n, 64]."""
    denoise_batch(g, layers, [cache], tok, w_in, mods, final_scale, w_out, out, workspace, stream)


def step_batch(g: Geom, layers, caches, x_in, x_out, mods, workspace, x_layers=None, stream=None):
    """qi21_step_batch (classifier-free-guidance batch of sequences)."""
    torch = _torch()
    f = torch.float32
    arr = (C.c_void_p * len(caches))(*[c.handle.value for c in caches])
    check(load().qi21_step_batch(C.byref(g), _layer_array(layers), arr, len(caches), _ptr(x_in, f, "x_in"),
                                 _ptr(x_out, f, "x_out"), _ptr(mods, f, "mods"), _ptr(x_layers, f, "x_layers"),
                                 _ptr(workspace, None, "workspace"),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


# --------------------------------------------------------- FP8 variant ----

class PackedLayerFp8:
    """One block's E4M3 planes and scales (qi21_pack_layer_fp8); keeps its
    buffer and the f16 layer (for the norm weights) alive."""

    def __init__(self, mem, src, cstruct):
        self.mem = mem
        self.src = src
        self.c = cstruct


def pack_layer_fp8(g: Geom, packed: PackedLayer, stream=None) -> PackedLayerFp8:
    """qi21_pack_layer_fp8: packed f16 planes -> E4M3 planes + row scales."""
    torch = _torch()
    lib = load()
    nbytes = lib.qi21_layer_fp8_bytes(C.byref(g))
    if nbytes == 0:
        check(lib.qi21_geom_check(C.byref(g)))
    mem = torch.empty(nbytes, dtype=torch.uint8, device=packed.planes.device)
    out = B.LayerFp8()
    check(lib.qi21_pack_layer_fp8(C.byref(g), C.byref(packed.c), mem.data_ptr(), nbytes, C.byref(out),
                                  _stream(stream)))
    return PackedLayerFp8(mem, packed, out)


def _layer8_array(layers):
    arr = (B.LayerFp8 * len(layers))()
    for i, l in enumerate(layers):
        arr[i] = l.c
    return arr


def workspace_bytes_fp8(g: Geom, rows: int) -> int:
    return int(load().qi21_workspace_bytes_fp8(C.byref(g), rows))


def prefill_fp8(g: Geom, layers8, cache: KVCache, x_prefix, mods0, workspace, x_layers=None, stream=None):
    """qi21_prefill_fp8."""
    torch = _torch()
    f = torch.float32
    check(load().qi21_prefill_fp8(C.byref(g), _layer8_array(layers8), cache.handle, _ptr(x_prefix, f, "x_prefix"),
                                  _ptr(mods0, f, "mods0"), _ptr(x_layers, f, "x_layers"),
                                  _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                                  _stream(stream)))


def step_batch_fp8(g: Geom, layers8, caches, x_in, x_out, mods, workspace, x_layers=None, stream=None):
    """qi21_step_batch_fp8."""
    torch = _torch()
    f = torch.float32
    arr = (C.c_void_p * len(caches))(*[c.handle.value for c in caches])
    check(load().qi21_step_batch_fp8(C.byref(g), _layer8_array(layers8), arr, len(caches), _ptr(x_in, f, "x_in"),
                                     _ptr(x_out, f, "x_out"), _ptr(mods, f, "mods"), _ptr(x_layers, f, "x_layers"),
                                     _ptr(workspace, None, "workspace"),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def op_quant_rows(a, q, qs, stream=None):
    torch = _torch()
    check(load().qi21_op_quant_rows(a.shape[0], a.shape[1], _ptr(a, torch.float16, "a"), _ptr(q, torch.uint8, "q"),
                                    _ptr(qs, torch.float32, "qs"), _stream(stream)))


def op_rowop_fp8(x, scale, xq, xs, eps=1e-6, stream=None):
    torch = _torch()
    f = torch.float32
    check(load().qi21_op_rowop_fp8(x.shape[0], x.shape[1], eps, _ptr(x, f, "x"), _ptr(scale, f, "scale"),
                                   _ptr(xq, torch.uint8, "xq"), _ptr(xs, f, "xs"), _stream(stream)))


def op_gemm_fp8(epi, A, sa, Bw, sw, out, gate_t=None, stream=None):
    torch = _torch()
    f = torch.float32
    M, K = A.shape
    N = Bw.shape[0]
    check(load().qi21_op_gemm_fp8(epi, M, N, K, _ptr(A, torch.uint8, "A"), _ptr(sa, f, "sa"),
                                  _ptr(Bw, torch.uint8, "B"), _ptr(sw, f, "sw"), _ptr(out, None, "out"),
                                  out.shape[1], _ptr(gate_t, f, "gate_t"), _stream(stream)))


# ------------------------------------------------------- single operations --

def op_rowop(x, scale, xn=None, y=None, gate_t=None, eps=1e-6, stream=None):
    """qi21_op_rowop; xn (f16 or bf16) selects the dtype."""
    torch = _torch()
    rows, dim = x.shape
    dt = _dt_code(xn) if xn is not None else DTYPE_F16
    check(load().qi21_op_rowop(dt, rows, dim, eps, _ptr(x, torch.float32, "x"), _ptr(y, torch.float32, "y"),
                               _ptr(gate_t, torch.float32, "gate_t"), _ptr(scale, torch.float32, "scale"),
                               _ptr(xn, None, "xn"), _stream(stream)))


def op_mods_prep(mods, md, stream=None):
    torch = _torch()
    check(load().qi21_op_mods_prep(mods.numel() // 4, _ptr(mods, torch.float32, "mods"),
                                   _ptr(md, torch.float32, "md"), _stream(stream)))


def op_gemm(epi, A, Bw, out, gate_t=None, stream=None):
    """qi21_op_gemm; A and B both f16 or both bf16."""
    torch = _torch()
    M, K = A.shape
    N = Bw.shape[0]
    check(load().qi21_op_gemm(_dt_code(A), epi, M, N, K, _ptr(A, None, "A"), _ptr(Bw, A.dtype, "B"),
                              _ptr(out, None, "out"), out.shape[1], _ptr(gate_t, torch.float32, "gate_t"),
                              _stream(stream)))


def op_gemm_split(epi, A, Bw, out, scratch, gate_t=None, stream=None):
    """qi21_op_gemm_split: qi21_op_gemm with the K-split tail, merged
    through `scratch` (a 256-byte aligned device buffer); returns the part
    count used (1: no split)."""
    torch = _torch()
    M, K = A.shape
    N = Bw.shape[0]
    parts = C.c_int32(0)
    check(load().qi21_op_gemm_split(_dt_code(A), epi, M, N, K, _ptr(A, None, "A"), _ptr(Bw, A.dtype, "B"),
                                    _ptr(out, None, "out"), out.shape[1], _ptr(gate_t, torch.float32, "gate_t"),
                                    _ptr(scratch, None, "scratch"), scratch.numel() * scratch.element_size(),
                                    C.byref(parts), _stream(stream)))
    return parts.value


def op_qkrope(panel, heads, norm_q, norm_k, cos_, sin_, eps=1e-6, stream=None):
    torch = _torch()
    check(load().qi21_op_qkrope(_dt_code(panel), panel.shape[0], heads, eps, _ptr(panel, None, "panel"),
                                _ptr(norm_q, torch.float32, "norm_q"), _ptr(norm_k, torch.float32, "norm_k"),
                                _ptr(cos_, torch.float32, "cos"), _ptr(sin_, torch.float32, "sin"),
                                _stream(stream)))


def op_kvcopy(panel, kv, stream=None):
    rows = panel.shape[0]
    dim = panel.shape[1] // 3
    _dt_code(panel)
    check(load().qi21_op_kvcopy(rows, dim, _ptr(panel, None, "panel"), _ptr(kv, panel.dtype, "kv"),
                                _stream(stream)))


def op_attention(panel, heads, out, nq, n_own, kv_pre=None, n_pre=0, vis=None, stream=None):
    """qi21_op_attention; panel, kv_pre and out all f16 or all bf16."""
    torch = _torch()
    check(load().qi21_op_attention(_dt_code(panel), nq, heads, _ptr(panel, None, "panel"),
                                   _ptr(kv_pre, panel.dtype, "kv_pre"), n_pre, n_own,
                                   _ptr(vis, torch.int32, "vis"), _ptr(out, panel.dtype, "out"),
                                   _stream(stream)))


def selftest_wait_timeout(stream=None):
    """Enqueue the bounded-wait self-test (qi21_selftest_wait_timeout): one
    CTA whose wait nothing ends gives up after about 2 s and raises the
    device status word."""
    check(load().qi21_selftest_wait_timeout(_stream(stream)))
