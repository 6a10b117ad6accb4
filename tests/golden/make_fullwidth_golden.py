"""Write the expected values of the end-to-end parity test of the 32-layer,
dim-4096 workloads (tests/test_gpu_fullwidth_e2e.py).

Calls only the oracle (oracle/qi21_oracle.py) and the seeded input
generators (synthetic/qi21_inputs.py). For every sequence of the workload
the whole chain runs on the CPU, as the page's CPU-exact path does it
(qwen_image21.rs, Qi21Dit::prefill, then the block loop of
Qi21Dit::step_cpu): the prefix through all L blocks with the t = 0
modulation and the block-causal mask, keeping each layer's post-RoPE K/V,
then the target rows through all L blocks against [cache of the layer, own
rows]. Every row is computed (the next layer's keys need every row); what
is stored per layer is small:

* ``step_rows``: the hidden state after each block on a few fixed target
  rows (the first row, the last row of the first 128-row tile, an interior
  row and the last row), float32 [L][R][H];
* ``step_sketch``, ``pre_sketch``, ``k_sketch``, ``v_sketch``: the matrix
  A X B^T of the step output after each block, of the prefill output after
  each block but the last, and of the layer's cached K and V, with A and B
  the seeded Gaussian sketches of ``synthetic.qi21_inputs.sketch`` (32 x
  rows, 32 x dim). Their relative L2 difference estimates that of the whole
  output, every row and column included.

The file is keyed by the sha256 of the oracle functions on the path and by
a summary of the seeded inputs (per tensor: count, sum and sum of squares),
so a test can tell a stale file. The summary is compared within a relative
1e-6, not bit for bit: float32 normal draws can differ in the last place
between platforms' libm (rare tail samples), which moves no result here.
One workload per run:

    python tests/golden/make_fullwidth_golden.py step32_cond4114_n4096

writes tests/golden/fullwidth_step32_cond4114_n4096.npz (about 40 min of
float64 CPU work for the 16384-row workload on 8 cores, a few minutes for
the CFG pair).
"""
from __future__ import annotations

import hashlib
import inspect
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import qi21_oracle as O  # noqa: E402
from synthetic import qi21_inputs as S  # noqa: E402

SKETCH_K = 32
FORMAT = 1


def sample_rows(n: int) -> np.ndarray:
    """Fixed target rows stored element by element."""
    return np.array(sorted({0, min(127, n - 1), n // 2 + 37 if n > 80 else n // 2, n - 1}),
                    dtype=np.int64)


# The oracle functions the chain runs through (a change to any other part of
# the oracle file does not make a stored file stale).
ORACLE_PATH = ("seg_len", "total_rows", "prefix_len", "validate", "block_ids", "positions",
               "prefix_visibility", "rope_tables", "target_rope", "silu", "layer_norm",
               "norm_mod", "gated_add", "rms_norm", "rope_rotate", "qk_norm_rope",
               "masked_softmax", "attention", "block", "cfg_of", "prefill", "step")


def oracle_sha256() -> str:
    """sha256 over the source text of the oracle functions on the path."""
    h = hashlib.sha256()
    for fn in ORACLE_PATH:
        h.update(inspect.getsource(getattr(O, fn)).encode())
    return h.hexdigest()


def inputs_fingerprint(w: S.Workload) -> str:
    """sha256 over the draws the chain starts from: every sequence's prefix,
    the target rows, both modulations and the first and last layers'
    weights (a change of the recipe changes at least these)."""
    h = hashlib.sha256()
    for s in range(w.nseq):
        h.update(S.x_prefix(w, s).tobytes())
    h.update(S.x_target(w).tobytes())
    h.update(S.mods_t(w).tobytes())
    h.update(S.mods0(w).tobytes())
    for layer in sorted({0, w.layers - 1}):
        W = S.layer_weights(w, layer)
        for tag in S.WEIGHT_TAGS + ("norm_q", "norm_k"):
            h.update(np.ascontiguousarray(W[tag]).tobytes())
    return h.hexdigest()


def _input_tensors(w: S.Workload):
    """(name, values) of the draws the chain starts from: every sequence's
    prefix, the target rows, both modulations and the first and last
    layers' weights."""
    for s in range(w.nseq):
        yield f"x_prefix_{s}", S.x_prefix(w, s)
    yield "x_target", S.x_target(w)
    yield "mods_t", S.mods_t(w)
    yield "mods0", S.mods0(w)
    for layer in sorted({0, w.layers - 1}):
        W = S.layer_weights(w, layer)
        for tag in S.WEIGHT_TAGS + ("norm_q", "norm_k"):
            yield f"{tag}_{layer}", W[tag]


def inputs_summary(w: S.Workload) -> list:
    """[name, count, sum, sum of squares] (float64) of each input tensor."""
    out = []
    for name, a in _input_tensors(w):
        v = np.asarray(a, dtype=np.float64).ravel()
        out.append([name, int(v.size), float(v.sum()), float((v * v).sum())])
    return out


def summary_matches(stored, now, rtol=1e-6) -> bool:
    """Same tensors, counts, and sums within rtol of the tensor's L2 scale."""
    if len(stored) != len(now):
        return False
    for (n0, c0, s0, q0), (n1, c1, s1, q1) in zip(stored, now):
        scale = max(np.sqrt(q0), 1e-30)
        if n0 != n1 or c0 != c1 or abs(s0 - s1) > rtol * scale or abs(q0 - q1) > rtol * max(q0, 1e-30):
            return False
    return True


def stale_reason(meta, name: str):
    """Why a stored file cannot be used for workload `name` (None: usable)."""
    if meta is None:
        return f"tests/golden/fullwidth_{name}.npz has not been written"
    if meta.get("oracle_sha256") != oracle_sha256():
        return f"fullwidth_{name}.npz was written by another oracle version"
    if "inputs_summary" not in meta or not summary_matches(meta["inputs_summary"], inputs_summary(S.WORKLOADS[name])):
        return f"fullwidth_{name}.npz was written for other seeded inputs"
    return None


def sketch_of(X: np.ndarray, A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """A X B^T in float64 (the parity statistic; not part of the method)."""
    return (A @ np.asarray(X, dtype=np.float64)) @ B.T


class _Layers:
    """The workload's layer weights, drawn one layer at a time while the
    oracle iterates (32 layers of dim 4096 would hold 14 GB at once)."""

    def __init__(self, w: S.Workload):
        self.w = w

    def __len__(self):
        return self.w.layers

    def __iter__(self):
        for layer in range(self.w.layers):
            yield S.layer_weights(self.w, layer)


def run(name: str, out_dir: str = HERE) -> str:
    w = S.WORKLOADS[name]
    cfg = O.cfg_of(w)
    H, L, n = w.dim, w.layers, w.n_target
    rows = sample_rows(n)
    B = S.sketch(H, SKETCH_K, 1)
    An = S.sketch(n, SKETCH_K, 0)
    arrays = {"rows": rows}
    t0 = time.time()
    for s in range(w.nseq):
        segs = w.segs(s)
        lp = O.prefix_len(segs)
        Ap = S.sketch(lp, SKETCH_K, 0)
        # prefill: every layer's cache; the hidden state after each block
        cache, xs_pre = O.prefill(S.x_prefix(w, s), _Layers(w), S.mods0(w), segs, cfg, keep_x=True)
        arrays[f"pre_sketch_s{s}"] = np.stack([sketch_of(x, Ap, B) for x in xs_pre[:L - 1]]).astype(np.float32)
        arrays[f"k_sketch_s{s}"] = np.stack([sketch_of(k, Ap, B) for k, _ in cache]).astype(np.float32)
        arrays[f"v_sketch_s{s}"] = np.stack([sketch_of(v, Ap, B) for _, v in cache]).astype(np.float32)
        del xs_pre
        print(f"{name} seq {s}: prefill of {lp} rows done at {time.time() - t0:.0f} s", flush=True)
        # step: one layer at a time through the oracle's own step
        x = S.x_target(w)
        srows, ssk = [], []
        for layer in range(L):
            x, _ = O.step(x, [S.layer_weights(w, layer)], S.mods_t(w), segs, [cache[layer]], cfg)
            cache[layer] = None
            srows.append(x[rows].astype(np.float32))
            ssk.append(sketch_of(x, An, B).astype(np.float32))
            print(f"{name} seq {s}: step layer {layer} done at {time.time() - t0:.0f} s", flush=True)
        arrays[f"step_rows_s{s}"] = np.stack(srows)
        arrays[f"step_sketch_s{s}"] = np.stack(ssk)
    meta = {
        "workload": name,
        "format": FORMAT,
        "oracle_sha256": oracle_sha256(),
        "inputs_fingerprint": inputs_fingerprint(w),
        "inputs_summary": inputs_summary(w),
        "sketch_k": SKETCH_K,
        "seed": w.seed,
        "nseq": w.nseq,
        "layers": L,
        "cpu_seconds": round(time.time() - t0, 1),
        "written_by": "tests/golden/make_fullwidth_golden.py (oracle only)",
    }
    arrays["meta"] = np.frombuffer(json.dumps(meta).encode(), dtype=np.uint8)
    path = os.path.join(out_dir, f"fullwidth_{name}.npz")
    np.savez_compressed(path, **arrays)
    print(f"wrote {path} in {time.time() - t0:.0f} s", flush=True)
    return path


def load(name: str, golden_dir: str = HERE):
    """(meta dict, arrays) of a stored file, or (None, None) if absent."""
    path = os.path.join(golden_dir, f"fullwidth_{name}.npz")
    if not os.path.exists(path):
        return None, None
    z = np.load(path)
    arrays = {k: z[k] for k in z.files if k != "meta"}
    meta = json.loads(bytes(z["meta"]).decode())
    return meta, arrays


def refresh_meta(name: str, golden_dir: str = HERE) -> None:
    """Rewrite only the keys of a stored file (the oracle source hash and
    the input summary, recomputed here); its arrays are kept as written."""
    path = os.path.join(golden_dir, f"fullwidth_{name}.npz")
    z = np.load(path)
    arrays = {k: z[k] for k in z.files if k != "meta"}
    meta = json.loads(bytes(z["meta"]).decode())
    w = S.WORKLOADS[name]
    if meta["inputs_fingerprint"] != inputs_fingerprint(w):
        raise SystemExit(f"{name}: the inputs here are not the ones the file was written for")
    meta["inputs_summary"] = inputs_summary(w)
    arrays["meta"] = np.frombuffer(json.dumps(meta).encode(), dtype=np.uint8)
    np.savez_compressed(path, **arrays)
    print(f"refreshed the keys of {path}")


if __name__ == "__main__":
    if len(sys.argv) > 2 and sys.argv[1] == "--refresh-meta":
        for nm in sys.argv[2:]:
            refresh_meta(nm)
    else:
        for nm in sys.argv[1:]:
            run(nm)
