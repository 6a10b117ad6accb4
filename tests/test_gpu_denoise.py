"""The ends of the denoiser call through the C ABI: qi21_embed, qi21_final
and the whole qi21_denoise / qi21_denoise_batch (latent tokens -> velocity)
against the CPU oracle on the same seeded inputs.

Tolerances: embed and final are f32 contractions (64 and dim terms):
rel L2 <= 1e-5. The whole call inherits the blocks' bar: rel L2 <= 2e-3 of
the velocity.
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


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert q.device_status() == 0


@pytest.mark.parametrize("n,dim", [(1, 256), (130, 512), (4096, 4096)])
def test_embed_matches_oracle(n, dim):
    tok = S.op_tensor(20, n, 0, (n, 64), 1.0)
    w_in = S.op_tensor(20, n, 1, (dim, 64), 0.125)
    x = torch.empty((n, dim), device="cuda")
    q.embed(T(tok), T(w_in), x)
    assert rel_l2(host(x), O.embed_image(tok, w_in)) <= 1e-5


@pytest.mark.parametrize("n,dim", [(1, 256), (33, 512), (130, 4096), (4096, 4096)])
def test_final_matches_oracle(n, dim):
    x = S.op_tensor(21, n, 0, (n, dim), 2.0, offset=0.3)
    fs = S.op_tensor(21, n, 1, (dim,), 0.1)
    w_out = S.op_tensor(21, n, 2, (64, dim), dim ** -0.5)
    out = torch.empty((n, 64), device="cuda")
    q.final(T(x), T(fs), T(w_out), out)
    rows = slice(None) if n <= 256 else np.arange(0, n, 97)
    ref = O.final_layer(x[rows], fs, w_out, 1e-6)
    assert rel_l2(host(out)[rows], ref) <= 1e-5


def _io(w):
    return (S.tokens(w), S.w_in(w), S.w_out(w), S.final_scale(w))


@pytest.mark.parametrize("name", ["tiny_block_d256", "ragged_d512", "cfg_pair_d256", "single_row_d256"])
def test_denoise_end_to_end(name):
    w = S.WORKLOADS[name]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    tok, w_in, w_out, fsc = _io(w)
    n = w.n_target
    out = torch.full((w.nseq * n, 64), float("nan"), device="cuda")
    q.denoise_batch(dw.g, dw.layers, dw.caches, T(np.concatenate([tok] * w.nseq)), T(w_in), dw.mods_t, T(fsc),
                    T(w_out), out, dw.ws)
    got = host(out)
    cfg = O.cfg_of(w)
    weights = [S.layer_weights(w, l) for l in range(w.layers)]
    for s in range(w.nseq):
        segs = w.segs(s)
        cache, _ = O.prefill(S.x_prefix(w, s), weights, S.mods0(w), segs, cfg)
        ref = O.denoise(tok, w_in, weights, S.mods_t(w), fsc, w_out, segs, cache, cfg)
        assert rel_l2(got[s * n:(s + 1) * n], ref) <= 2e-3, (name, s)


def test_denoise_full_width_composition_and_final_rows():
    # the whole call equals embed -> step -> final launched one by one
    # (bit-exact), and its final layer matches the oracle on sampled rows of
    # the GPU's own hidden state after the 32 blocks
    w = S.WORKLOADS["step32_cond4114_n4096"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    tok, w_in, w_out, fsc = (T(a) for a in _io(w))
    n = w.n_target
    out = torch.empty((n, 64), device="cuda")
    q.denoise(dw.g, dw.layers, dw.caches[0], tok, w_in, dw.mods_t, fsc, w_out, out, dw.ws)
    x = torch.empty((n, w.dim), device="cuda")
    q.embed(tok, w_in, x)
    q.step(dw.g, dw.layers, dw.caches[0], x, x, dw.mods_t, dw.ws)
    out2 = torch.empty_like(out)
    q.final(x, fsc, w_out, out2)
    np.testing.assert_array_equal(host(out), host(out2))
    rows = np.array([0, 1, 127, 128, 2048, 4095])
    xs = x[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = O.final_layer(xs, S.final_scale(w), S.w_out(w), w.eps)
    assert rel_l2(host(out)[rows], ref) <= 1e-5
    assert np.all(np.isfinite(host(out)))
