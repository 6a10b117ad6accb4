"""Shared helpers of the block-level GPU parity tests: a device run of a
workload (prefill + one step, with every block's output kept) and the
comparisons of its blocks against the oracle. Expected values come from
oracle/ only; the inputs from synthetic/."""
import numpy as np

from oracle import qi21_oracle as O
from synthetic import device as D
from synthetic import qi21_inputs as S


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def host(t):
    import torch
    torch.cuda.synchronize()
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


class DeviceRun:
    """Prefill + one step of a workload on the GPU with per-block outputs."""

    def __init__(self, w, layers=None, keep_prefill_x=True):
        import torch

        import diffusion_transformer_denoiser_qi21_gb300 as q
        self.w = w
        self.dw = D.DeviceWorkload(w, layers=layers)
        H, L = w.dim, w.layers
        self.xpre = [torch.full((L, c.lp, H), float("nan"), device="cuda") if keep_prefill_x else None
                     for c in self.dw.caches]
        self.dw.prefill_all(x_layers=self.xpre)
        n = w.n_target
        self.xl = torch.full((L, w.nseq * n, H), float("nan"), device="cuda")
        self.out = self.dw.step(x_layers=self.xl)
        torch.cuda.synchronize()
        assert q.device_status() == 0

    def kv(self, s, layer):
        return self.dw.caches[s].layer_tensor(layer)

    def step_x(self, layer, s, rows=None):
        import torch
        n = self.w.n_target
        t = self.xl[layer, s * n:(s + 1) * n]
        if rows is not None:
            t = t[torch.as_tensor(rows, device="cuda")]
        return host(t)

    def step_in(self, layer, s, rows=None):
        if layer == 0:
            x = S.x_target(self.w)
            return x if rows is None else x[rows]
        return self.step_x(layer - 1, s, rows)

    def pre_x(self, layer, s):
        return host(self.xpre[s][layer])

    def pre_in(self, layer, s):
        return S.x_prefix(self.w, s) if layer == 0 else self.pre_x(layer - 1, s)


def check_block(got_out, x_in, ref_out, what, x_tol, delta_tol):
    """rel L2 of the block output and of the block's own contribution."""
    e = rel_l2(got_out, ref_out)
    assert e <= x_tol, f"{what}: rel L2 {e:.3e}"
    d = rel_l2(np.asarray(got_out, np.float64) - x_in, np.asarray(ref_out, np.float64) - x_in)
    assert d <= delta_tol, f"{what}: block delta rel L2 {d:.3e}"
    return e, d


def teacher_forced_layer(run, layer, s, W, cfg, tol, rows_pre=None, rows_step=None):
    """Oracle block `layer` on the GPU's inputs: prefill (K/V and output) and
    step (output), optionally on sampled rows. tol = (x, delta, kv)."""
    x_tol, delta_tol, kv_tol = tol
    w = run.w
    segs = w.segs(s)
    lp = O.prefix_len(segs)
    pos = O.positions(segs)
    cp, sp = O.rope_tables(pos[:lp], cfg["axes"], cfg["theta"])
    vis = O.prefix_visibility(segs)
    # prefill: this layer's K/V from the GPU's prefix input of the layer
    xin = run.pre_in(layer, s)
    xo, k, v = O.block(xin, W, S.mods0(w), cp, sp, cfg, None, vis, rows=rows_pre)
    kv = host(run.kv(s, layer)).astype(np.float64)
    H = w.dim
    ek = rel_l2(kv[:, :H], k)
    ev = rel_l2(kv[:, H:], v)
    assert ek <= kv_tol and ev <= kv_tol, f"layer {layer} seq {s}: cache K {ek:.2e} V {ev:.2e}"
    if layer + 1 < w.layers:
        got = run.pre_x(layer, s)
        if rows_pre is not None:
            got = got[rows_pre]
            xin_r = xin[rows_pre]
        else:
            xin_r = xin
        check_block(got, xin_r, xo, f"prefill layer {layer} seq {s}", x_tol, delta_tol)
    # step: the GPU's input of the layer against the GPU's cache of the layer
    ct, st = O.target_rope(segs, cfg["axes"], cfg["theta"])
    x_in = run.step_in(layer, s)
    ref, _, _ = O.block(x_in, W, S.mods_t(w), ct, st, cfg, (kv[:, :H], kv[:, H:]), None, rows=rows_step)
    got = run.step_x(layer, s, rows_step)
    x_in_r = x_in if rows_step is None else x_in[rows_step]
    return check_block(got, x_in_r, ref, f"step layer {layer} seq {s}", x_tol, delta_tol)


def end_to_end(run, weights, cfg, tol):
    """Each side runs its own chain: every block output of the step and every
    layer's cache against the oracle's prefill + step. Returns the worst
    block rel L2."""
    import numpy.testing as npt
    x_tol, delta_tol, kv_tol = tol
    w = run.w
    worst = 0.0
    for s in range(w.nseq):
        segs = w.segs(s)
        cache, _ = O.prefill(S.x_prefix(w, s), weights, S.mods0(w), segs, cfg)
        _, xs = O.step(S.x_target(w), weights, S.mods_t(w), segs, cache, cfg, keep_x=True)
        x_in = S.x_target(w)
        for l in range(w.layers):
            e, _ = check_block(run.step_x(l, s), x_in, xs[l], f"{w.name} e2e step layer {l} seq {s}",
                               x_tol, delta_tol)
            worst = max(worst, e)
            x_in = xs[l]
            kv = host(run.kv(s, l)).astype(np.float64)
            H = w.dim
            assert rel_l2(kv[:, :H], cache[l][0]) <= kv_tol
            assert rel_l2(kv[:, H:], cache[l][1]) <= kv_tol
        n = w.n_target
        npt.assert_array_equal(host(run.out[s * n:(s + 1) * n]), run.step_x(w.layers - 1, s))
    return worst


def sample_rows(n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 2, 17, 18, 19, 126, 127, 128, 129, n // 2, n - 129, n - 128, n - 2, n - 1]
    rnd = rng.choice(n, size=min(n, 48), replace=False).tolist()
    return np.array(sorted(set(r for r in fixed + rnd if 0 <= r < n)), dtype=np.int64)
