"""End-to-end parity of the 32-layer, dim-4096 workloads against the oracle:
each side runs its own chain (the prefill of every prefix row, then the step
of every target row through all 32 blocks) and every block's output is
compared, not only teacher-forced samples.

The oracle chain of these workloads takes tens of minutes of float64 CPU
work, so its results are stored by tests/golden/make_fullwidth_golden.py
(which calls only oracle/ and synthetic/) in tests/golden/fullwidth_*.npz:
per layer a few target rows element by element, and Gaussian sketches
A X B^T of the step output, of the prefill output and of the cached K and V
(32 x 32 numbers that weigh every row and column; their relative L2
difference estimates that of the whole tensor). A stored file whose oracle
source hash or input summary no longer matches is skipped with the
reason, never trusted.

Bar: rel L2 <= 2e-3 for every block output (step and prefill) and for the
cache (6e-3 for the bf16 cache: one bf16 rounding of a stored value), on
the stored rows and on the sketches.
"""
import os
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from blockcheck import DeviceRun, host, rel_l2  # noqa: E402
from synthetic import device as D  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_fullwidth_golden as G  # noqa: E402

pytestmark = pytest.mark.gpu

X_TOL = 2e-3
KV_TOL = 2e-3


def _golden(name):
    meta, arr = G.load(name)
    why = G.stale_reason(meta, name)
    if why is not None:
        pytest.skip(why)
    return meta, arr


@pytest.fixture(scope="module")
def layers32():
    w = S.WORKLOADS["step32_cond4114_n4096"]
    layers = D.upload_layers(w, D.geom_of(w))
    yield layers
    del layers
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["step32_cond4114_n4096", "step32_n16384", "cfg_pair32_n1024"])
def test_full_width_32_layers_end_to_end(name, layers32):
    _end_to_end(name, layers32, X_TOL, KV_TOL)


def test_full_width_bf16_end_to_end():
    # the bench workload in bf16 (weights, activation rows and cache): the
    # same bar on the block outputs; the cache within bf16's one-rounding
    # bar (6e-3: relative RMS 2^-8 / sqrt(3) of a stored value)
    name = "step32_cond4114_n4096_bf16"
    _golden(name)
    w = S.WORKLOADS[name]
    layers = D.upload_layers(w, D.geom_of(w))
    _end_to_end(name, layers, X_TOL, 6e-3)
    del layers
    torch.cuda.empty_cache()


def _end_to_end(name, layers, x_tol, kv_tol):
    w = S.WORKLOADS[name]
    meta, arr = _golden(name)
    run = DeviceRun(w, layers=layers)
    H, L, n = w.dim, w.layers, w.n_target
    K = meta["sketch_k"]
    B = S.sketch(H, K, 1)
    An = S.sketch(n, K, 0)
    rows = arr["rows"]
    worst = {"step_rows": 0.0, "step": 0.0, "prefill": 0.0, "kv": 0.0}
    for s in range(w.nseq):
        lp = w.prefix_rows(s)
        Ap = S.sketch(lp, K, 0)
        for layer in range(L):
            x = run.step_x(layer, s)
            e_rows = rel_l2(x[rows], arr[f"step_rows_s{s}"][layer])
            e_sk = rel_l2(G.sketch_of(x, An, B), arr[f"step_sketch_s{s}"][layer])
            kv = host(run.kv(s, layer))
            e_k = rel_l2(G.sketch_of(kv[:, :H], Ap, B), arr[f"k_sketch_s{s}"][layer])
            e_v = rel_l2(G.sketch_of(kv[:, H:], Ap, B), arr[f"v_sketch_s{s}"][layer])
            e_pre = 0.0
            if layer + 1 < L:
                e_pre = rel_l2(G.sketch_of(run.pre_x(layer, s), Ap, B), arr[f"pre_sketch_s{s}"][layer])
            print(f"{name} seq {s} layer {layer}: step rows {e_rows:.2e} sketch {e_sk:.2e}, "
                  f"prefill {e_pre:.2e}, K {e_k:.2e} V {e_v:.2e}")
            assert e_rows <= x_tol, f"seq {s} layer {layer}: sampled rows rel L2 {e_rows:.3e}"
            assert e_sk <= x_tol, f"seq {s} layer {layer}: step sketch rel L2 {e_sk:.3e}"
            assert e_pre <= x_tol, f"seq {s} layer {layer}: prefill sketch rel L2 {e_pre:.3e}"
            assert e_k <= kv_tol and e_v <= kv_tol, f"seq {s} layer {layer}: K {e_k:.3e} V {e_v:.3e}"
            worst["step_rows"] = max(worst["step_rows"], e_rows)
            worst["step"] = max(worst["step"], e_sk)
            worst["prefill"] = max(worst["prefill"], e_pre)
            worst["kv"] = max(worst["kv"], e_k, e_v)
        np.testing.assert_array_equal(host(run.out[s * n:(s + 1) * n]), run.step_x(L - 1, s))
    print(f"{name}: worst " + ", ".join(f"{k} {v:.2e}" for k, v in worst.items()))
    del run
    torch.cuda.empty_cache()
