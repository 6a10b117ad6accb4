"""The stored end-to-end expectations of the 32-layer, dim-4096 workloads
(tests/golden/fullwidth_*.npz, written by tests/golden/make_fullwidth_golden.py
from oracle/ and synthetic/ only) are current and come from the oracle: their
keys match the present oracle source and seeded inputs, and a piece of one
of them is recomputed here from the oracle directly. No GPU."""
import dataclasses
import os
import sys

import numpy as np
import pytest

from oracle import qi21_oracle as O
from synthetic import qi21_inputs as S

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))
import make_fullwidth_golden as G  # noqa: E402

NAMES = ["step32_cond4114_n4096", "step32_n16384", "cfg_pair32_n1024", "step32_cond4114_n4096_bf16"]


@pytest.mark.parametrize("name", NAMES)
def test_stored_file_is_current(name):
    meta, arr = G.load(name)
    if meta is None:
        pytest.skip(f"fullwidth_{name}.npz not written yet")
    w = S.WORKLOADS[name]
    assert meta["workload"] == name and meta["layers"] == w.layers and meta["nseq"] == w.nseq
    assert meta["oracle_sha256"] == G.oracle_sha256(), "the oracle changed: rewrite the stored file"
    assert G.stale_reason(meta, name) is None
    L, K = w.layers, meta["sketch_k"]
    np.testing.assert_array_equal(arr["rows"], G.sample_rows(w.n_target))
    for s in range(w.nseq):
        assert arr[f"step_rows_s{s}"].shape == (L, len(arr["rows"]), w.dim)
        assert arr[f"step_sketch_s{s}"].shape == (L, K, K)
        assert arr[f"pre_sketch_s{s}"].shape == (L - 1, K, K)
        assert arr[f"k_sketch_s{s}"].shape == (L, K, K) and arr[f"v_sketch_s{s}"].shape == (L, K, K)
        assert np.all(np.isfinite(arr[f"step_rows_s{s}"]))


def test_first_layer_of_the_cfg_pair_recomputed_from_the_oracle():
    # sequence 1 of the CFG pair has a one-row prefix, so its layer 0 is
    # cheap: the prefill block of that row, then the step block of every
    # target row against it, restricted on the query side to the stored rows
    name = "cfg_pair32_n1024"
    meta, arr = G.load(name)
    if meta is None:
        pytest.skip("fullwidth_cfg_pair32_n1024.npz not written yet")
    w = S.WORKLOADS[name]
    cfg = O.cfg_of(w)
    s = 1
    segs = w.segs(s)
    W0 = S.layer_weights(w, 0)
    cache, _ = O.prefill(S.x_prefix(w, s), [W0], S.mods0(w), segs, cfg)
    rows = arr["rows"]
    ct, st = O.target_rope(segs, cfg["axes"], cfg["theta"])
    got, _, _ = O.block(S.x_target(w), W0, S.mods_t(w), ct, st, cfg, cache[0], None, rows=rows)
    want = arr[f"step_rows_s{s}"][0].astype(np.float64)
    assert np.max(np.abs(got - want)) <= 1e-6 * np.max(np.abs(want))
    Ap = S.sketch(O.prefix_len(segs), meta["sketch_k"], 0)
    B = S.sketch(w.dim, meta["sketch_k"], 1)
    k_sk = G.sketch_of(cache[0][0], Ap, B)
    want_k = arr[f"k_sketch_s{s}"][0].astype(np.float64)
    assert np.max(np.abs(k_sk - want_k)) <= 1e-5 * np.max(np.abs(want_k))


def test_input_summary_tolerates_last_place_noise_only():
    w = S.WORKLOADS["cfg_pair_d256"]
    now = G.inputs_summary(w)
    assert G.summary_matches(now, now)
    # a last-place change of a few elements is tolerated
    noisy = [[n, c, s_ * (1 + 1e-9), q_ * (1 + 1e-9)] for n, c, s_, q_ in now]
    assert G.summary_matches(now, noisy)
    # another seed is not
    other = G.inputs_summary(dataclasses.replace(w, seed=1))
    assert not G.summary_matches(now, other)
    shifted = [[n, c, s_ + 1e-3 * np.sqrt(q_), q_] for n, c, s_, q_ in now]
    assert not G.summary_matches(now, shifted)


def test_sketch_estimates_the_whole_relative_error():
    # the statistic the GPU test relies on: for a dense error the sketched
    # relative L2 difference is close to the whole one
    rng = np.random.default_rng(3)
    n, H, K = 1024, 512, 32
    X = rng.standard_normal((n, H))
    E = 1e-3 * rng.standard_normal((n, H))
    A, B = S.sketch(n, K, 0), S.sketch(H, K, 1)
    whole = np.linalg.norm(E) / np.linalg.norm(X)
    sk = np.linalg.norm(G.sketch_of(X + E, A, B) - G.sketch_of(X, A, B)) / np.linalg.norm(G.sketch_of(X, A, B))
    assert 0.8 < sk / whole < 1.25
    # an error confined to one row is still seen
    E1 = np.zeros((n, H))
    E1[517] = 0.05 * rng.standard_normal(H)
    sk1 = np.linalg.norm(G.sketch_of(X + E1, A, B) - G.sketch_of(X, A, B)) / np.linalg.norm(G.sketch_of(X, A, B))
    whole1 = np.linalg.norm(E1) / np.linalg.norm(X)
    assert 0.3 < sk1 / whole1 < 3.0
