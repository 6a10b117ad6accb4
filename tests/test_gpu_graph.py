"""Recorded calls (qi21_graph_step_batch / qi21_graph_denoise_batch /
qi21_graph_launch): a replay runs the very launches of the direct call, so
its results must equal the direct call's bit for bit, also after the
caller changes the contents of the bound buffers between replays."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import diffusion_transformer_denoiser_qi21_gb300 as q  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

pytestmark = pytest.mark.gpu


def T(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


@pytest.fixture(autouse=True)
def _status_clean():
    yield
    assert q.device_status() == 0


def _direct_step(dw, x_in, mods):
    out = torch.empty_like(x_in)
    q.step_batch(dw.g, dw.layers, dw.caches, x_in, out, mods, dw.ws)
    return host(out)


@pytest.mark.parametrize("name", ["tiny_block_d256", "cfg_pair_d256", "ragged_d512", "block_d4096_n4096"])
def test_graph_step_equals_direct_step(name):
    w = S.WORKLOADS[name]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    x_in = dw.x_target.clone()
    mods = dw.mods_t.clone()
    x_out = torch.full_like(x_in, float("nan"))
    gr = q.graph_step_batch(dw.g, dw.layers, dw.caches, x_in, x_out, mods, dw.ws)
    assert np.all(np.isnan(host(x_out)))  # recording runs nothing
    ref = _direct_step(dw, x_in, mods)
    gr.launch()
    np.testing.assert_array_equal(host(x_out), ref)
    # new contents in the bound buffers: the replay follows them
    rng = np.random.default_rng(7)
    x_in.copy_(T(rng.standard_normal(tuple(x_in.shape)).astype(np.float32)))
    mods.copy_(T((0.1 * rng.standard_normal(mods.numel())).astype(np.float32)))
    ref2 = _direct_step(dw, x_in, mods)
    gr.launch()
    np.testing.assert_array_equal(host(x_out), ref2)
    assert not np.array_equal(ref, ref2)
    # repeated replays on a side stream agree too
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            gr.launch(stream=s)
    s.synchronize()
    np.testing.assert_array_equal(host(x_out), ref2)
    gr.free()


def test_graph_denoise_equals_direct_and_in_place_chain():
    w = S.WORKLOADS["cfg_pair_d256"]
    dw = D.DeviceWorkload(w)
    dw.prefill_all()
    tok = T(np.concatenate([S.tokens(w)] * w.nseq))
    w_in, w_out, fs = T(S.w_in(w)), T(S.w_out(w)), T(S.final_scale(w))
    out = torch.empty((tok.shape[0], 64), device="cuda")
    gr = q.graph_denoise_batch(dw.g, dw.layers, dw.caches, tok, w_in, dw.mods_t, fs, w_out, out, dw.ws)
    ref = torch.empty_like(out)
    q.denoise_batch(dw.g, dw.layers, dw.caches, tok, w_in, dw.mods_t, fs, w_out, ref, dw.ws)
    gr.launch()
    np.testing.assert_array_equal(host(out), host(ref))
    # a few Euler-like updates of the tokens through the graph vs direct calls
    tok2 = tok.clone()
    for _ in range(3):
        gr.launch()
        torch.cuda.synchronize()
        tok.sub_(0.1 * out)
        q.denoise_batch(dw.g, dw.layers, dw.caches, tok2, w_in, dw.mods_t, fs, w_out, ref, dw.ws)
        torch.cuda.synchronize()
        tok2.sub_(0.1 * ref)
    np.testing.assert_array_equal(host(tok), host(tok2))
    gr.free()


def test_graph_capture_refuses_what_the_call_refuses():
    w = S.WORKLOADS["tiny_block_d256"]
    dw = D.DeviceWorkload(w)
    # caches not prefilled: the capture fails like the direct call, nothing recorded
    with pytest.raises(q.Qi21Error):
        q.graph_step_batch(dw.g, dw.layers, dw.caches, dw.x_target, dw.x_out, dw.mods_t, dw.ws)
    dw.prefill_all()
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(q.Qi21Error):
        q.graph_step_batch(dw.g, dw.layers, dw.caches, dw.x_target, dw.x_out, dw.mods_t, small)
    # and the library is still usable afterwards
    gr = q.graph_step_batch(dw.g, dw.layers, dw.caches, dw.x_target, dw.x_out, dw.mods_t, dw.ws)
    gr.launch()
    ref = _direct_step(dw, dw.x_target, dw.mods_t)
    np.testing.assert_array_equal(host(dw.x_out), ref)


def test_graph_fp8_step_equals_direct():
    w = S.WORKLOADS["cfg_pair_d256"]
    dw = D.DeviceWorkload(w)
    l8 = [q.pack_layer_fp8(dw.g, l) for l in dw.layers]
    rows = max(w.nseq * w.n_target, max(c.lp for c in dw.caches))
    ws = torch.empty(q.workspace_bytes_fp8(dw.g, rows), dtype=torch.uint8, device="cuda")
    for s, c in enumerate(dw.caches):
        q.prefill_fp8(dw.g, l8, c, dw.x_prefix[s], dw.mods0, ws)
    x_out = torch.empty_like(dw.x_target)
    gr = q.graph_step_batch_fp8(dw.g, l8, dw.caches, dw.x_target, x_out, dw.mods_t, ws)
    ref = torch.empty_like(x_out)
    q.step_batch_fp8(dw.g, l8, dw.caches, dw.x_target, ref, dw.mods_t, ws)
    gr.launch()
    np.testing.assert_array_equal(host(x_out), host(ref))
    gr.free()
