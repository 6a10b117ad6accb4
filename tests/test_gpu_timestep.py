"""Timestep conditioning through the C ABI (qi21_timestep_mods) against the
CPU oracle, and a whole sampler call built on it: the prefix prefilled with
the t = 0 modulation, then latent tokens -> velocity with the modulation of t.

Tolerance of mods / final_scale, derived from the f32 sinusoid: the angle
a_i = (1000 t) f_i is rounded in f32 on both sides, but f_i comes from
each side's own f32 exp (at most 2 ulp apart), so a_i can differ by up to
|a_i| 2^-22 <= 1000 t 2.4e-7 rad. Over the 256 channels that bounds the
sinusoid's error at 16 * 2.4e-4 t against its norm sqrt(128), a relative
3.4e-4 t, which the contractions carry through unchanged in size. On top of
that the device sums in f32 (about 1e-6 relative). So: rel L2 <=
1e-5 + 3.4e-4 t.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from oracle import qi21_oracle as O  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def tol(t):
    return 1e-5 + 3.4e-4 * t


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert q.device_status() == 0


def _run(wd, t):
    dim = wd["t_lin2"].shape[0]
    mods = torch.full((4 * dim,), float("nan"), device="cuda")
    fs = torch.full((dim,), float("nan"), device="cuda")
    q.timestep_mods(t, wd["t_lin1"], wd["t_lin2"], wd["modulation"], wd["norm_out"], mods, fs)
    return mods, fs


@pytest.mark.parametrize("name", ["tiny_block_d256", "ragged_d512", "block_d4096_n4096"])
@pytest.mark.parametrize("t", [0.0, 0.001, 0.25, 0.731, 1.0])
def test_timestep_mods_match_oracle(name, t):
    w = S.WORKLOADS[name]
    W = S.timestep_weights(w)
    wd = {k: T(v) for k, v in W.items()}
    mods, fs = _run(wd, t)
    ref_m, ref_f = O.timestep_mods(t, W["t_lin1"], W["t_lin2"], W["modulation"], W["norm_out"])
    got_m, got_f = host(mods), host(fs)
    assert np.all(np.isfinite(got_m)) and np.all(np.isfinite(got_f))
    assert rel_l2(got_m, ref_m) <= tol(t), rel_l2(got_m, ref_m)
    assert rel_l2(got_f, ref_f) <= tol(t), rel_l2(got_f, ref_f)


def test_timestep_mods_odd_width_and_errors():
    # dim 260 is not a multiple of 128 or of the 8-row CTA: ragged warps and
    # a ragged last CTA
    rng = np.random.default_rng(3)
    dim = 260
    W = {"t_lin1": rng.standard_normal((dim, 256)).astype(np.float32) / 16,
         "t_lin2": rng.standard_normal((dim, dim)).astype(np.float32) / dim ** 0.5,
         "modulation": rng.standard_normal((4 * dim, dim)).astype(np.float32) / dim ** 0.5,
         "norm_out": rng.standard_normal((dim, dim)).astype(np.float32) / dim ** 0.5}
    wd = {k: T(v) for k, v in W.items()}
    mods, fs = _run(wd, 0.4)
    ref_m, ref_f = O.timestep_mods(0.4, W["t_lin1"], W["t_lin2"], W["modulation"], W["norm_out"])
    assert rel_l2(host(mods), ref_m) <= tol(0.4)
    assert rel_l2(host(fs), ref_f) <= tol(0.4)
    # host-detectable errors enqueue nothing
    before = host(mods).copy()
    with pytest.raises(q.Qi21Error):
        q.timestep_mods(float("nan"), wd["t_lin1"], wd["t_lin2"], wd["modulation"], wd["norm_out"], mods, fs)
    with pytest.raises(q.Qi21Error):
        q.timestep_mods(0.5, wd["t_lin1"], wd["t_lin2"], wd["modulation"], wd["norm_out"], mods, fs,
                        work=torch.empty(2 * dim + 1, device="cuda")[1:])
    np.testing.assert_array_equal(host(mods), before)


@pytest.mark.parametrize("name", ["tiny_block_d256", "cfg_pair_d256"])
def test_sampler_call_from_timestep(name):
    # the page's sampler call: prefix at t = 0 (causal_condition), target at t
    w = S.WORKLOADS[name]
    t = 0.6
    W = S.timestep_weights(w)
    wd = {k: T(v) for k, v in W.items()}
    dw = D.DeviceWorkload(w)
    m0, _ = _run(wd, 0.0)
    dw.mods0 = m0
    dw.prefill_all()
    mt, fs = _run(wd, t)
    tok, w_in, w_out = S.tokens(w), S.w_in(w), S.w_out(w)
    n = w.n_target
    out = torch.empty((w.nseq * n, 64), device="cuda")
    q.denoise_batch(dw.g, dw.layers, dw.caches, T(np.concatenate([tok] * w.nseq)), T(w_in), mt, fs, T(w_out),
                    out, dw.ws)
    got = host(out)
    cfg = O.cfg_of(w)
    weights = [S.layer_weights(w, l) for l in range(w.layers)]
    ref_m0, _ = O.timestep_mods(0.0, W["t_lin1"], W["t_lin2"], W["modulation"], W["norm_out"])
    ref_mt, ref_fs = O.timestep_mods(t, W["t_lin1"], W["t_lin2"], W["modulation"], W["norm_out"])
    for s in range(w.nseq):
        segs = w.segs(s)
        cache, _ = O.prefill(S.x_prefix(w, s), weights, ref_m0, segs, cfg)
        ref = O.denoise(tok, w_in, weights, ref_mt, ref_fs, w_out, segs, cache, cfg)
        assert rel_l2(got[s * n:(s + 1) * n], ref) <= 2e-3, (name, s)
