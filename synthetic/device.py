"""Device-side setup of a synthetic workload for the library: draws the
seeded tensors of ``synthetic.qi21_inputs``, uploads them as torch CUDA
tensors and packs each layer's planes with the library's own
``qi21_pack_layer``. No arithmetic of the method happens here."""
from __future__ import annotations

import numpy as np

from . import qi21_inputs as S


def geom_of(w: S.Workload):
    import diffusion_transformer_denoiser_qi21_gb300 as q
    return q.geom(w.dim, w.heads, w.mlp_hidden, w.layers, w.axes, w.eps, w.theta, w.head_dim, dtype=w.dtype)


def _pinned_16(shape, dtype):
    import torch
    return torch.empty(shape, dtype=torch.float16 if dtype == "f16" else torch.int16, pin_memory=True)


def upload_layer(w: S.Workload, layer: int, g, stream=None):
    """Draw layer `layer`'s weights on the host, upload and pack them."""
    import torch

    import diffusion_transformer_denoiser_qi21_gb300 as q
    dev = {}
    for tag in S.WEIGHT_TAGS:
        shape = S.weight_shape(w, tag)
        host = _pinned_16(shape, w.dtype)
        hv = host.numpy()
        S.weight(w, layer, tag, out=hv if w.dtype == "f16" else hv.view(np.uint16))
        d = host.to("cuda", non_blocking=True)
        dev[tag] = d if w.dtype == "f16" else d.view(torch.bfloat16)
    nq = torch.from_numpy(S.norm_weight(w, layer, "norm_q")).cuda()
    nk = torch.from_numpy(S.norm_weight(w, layer, "norm_k")).cuda()
    packed = q.pack_layer(g, dev["wq"], dev["wk"], dev["wv"], dev["wo"], dev["wgate"], dev["wup"],
                          dev["wdown"], nq, nk, stream=stream)
    torch.cuda.synchronize()
    del dev
    return packed


def upload_layers(w: S.Workload, g, layers=None):
    return [upload_layer(w, l, g) for l in (range(w.layers) if layers is None else layers)]


def to_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class DeviceWorkload:
    """Geometry, packed layers, caches and activations of a workload on the
    current CUDA device."""

    def __init__(self, w: S.Workload, layers=None):
        """``layers``: already packed layers of an identical geometry and
        seed (the 32-layer workloads share their weights), else drawn here."""
        import torch

        import diffusion_transformer_denoiser_qi21_gb300 as q
        self.w = w
        self.g = geom_of(w)
        self.layers = upload_layers(w, self.g) if layers is None else layers
        self.caches = [q.KVCache(self.g, w.segs(s)) for s in range(w.nseq)]
        self.x_prefix = [to_dev(S.x_prefix(w, s)) for s in range(w.nseq)]
        xt = S.x_target(w)
        self.x_target = to_dev(np.concatenate([xt] * w.nseq, axis=0))
        self.mods_t = to_dev(S.mods_t(w))
        self.mods0 = to_dev(S.mods0(w))
        rows = max([w.nseq * w.n_target] + [c.lp for c in self.caches])
        self.ws = torch.empty(q.workspace_bytes(self.g, rows), dtype=torch.uint8, device="cuda")
        self.x_out = torch.empty_like(self.x_target)

    def prefill_all(self, x_layers=None, stream=None):
        import diffusion_transformer_denoiser_qi21_gb300 as q
        for s, c in enumerate(self.caches):
            q.prefill(self.g, self.layers, c, self.x_prefix[s], self.mods0, self.ws,
                      x_layers=None if x_layers is None else x_layers[s], stream=stream)

    def step(self, x_in=None, x_out=None, x_layers=None, stream=None):
        import diffusion_transformer_denoiser_qi21_gb300 as q
        x_in = self.x_target if x_in is None else x_in
        x_out = self.x_out if x_out is None else x_out
        if len(self.caches) == 1:
            q.step(self.g, self.layers, self.caches[0], x_in, x_out, self.mods_t, self.ws,
                   x_layers=x_layers, stream=stream)
        else:
            q.step_batch(self.g, self.layers, self.caches, x_in, x_out, self.mods_t, self.ws,
                         x_layers=x_layers, stream=stream)
        return x_out
