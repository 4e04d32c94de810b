"""GPU parity of the sequence-tiled SwiGLU MLP (upipe_mlp_fwd / upipe_mlp_bwd,
through the C ABI) against the float64 oracle (oracle/mlp.py) on the same
seeded inputs.  Tiling is exact by definition (a token's output depends on
that token alone), and the CUDA path computes every row the same way in any
tile: y and dx must be bit-identical across tile sizes; the weight gradients
sum over the tiles with fp32 reduce-adds in no fixed order."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import MLP_WORKLOADS, MlpWorkload, make_mlp_inputs, sample_rows
from tests._util import f64, assert_close
from tests._guard import guarded

pytestmark = pytest.mark.gpu


def U():
    import headwise_chunked_attention_gb300 as mod
    mod.lib()
    return mod


def shape_of(u, w):
    return u.MlpShape(w.S, w.hidden, w.ffn, w.tile_rows)


def run_fwd(w, t):
    u = U()
    sh = shape_of(u, w)
    g = {"y": guarded((w.S, w.hidden), fill=float("nan")),
         "workspace": guarded((u.mlp_workspace_bytes(sh, 0),), torch.uint8)}
    u.mlp_fwd(sh, t["x"], t["Wg"], t["Wu"], t["Wd"], g["y"].t, g["workspace"].t)
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == 0, f"device error word {rc}"
    for name, b in g.items():
        b.check(name)
    return g["y"].t


def run_bwd(w, t):
    u = U()
    sh = shape_of(u, w)
    g = {"dx": guarded((w.S, w.hidden), fill=float("nan")),
         "dWg": guarded((w.ffn, w.hidden), fill=float("nan")),
         "dWu": guarded((w.ffn, w.hidden), fill=float("nan")),
         "dWd": guarded((w.hidden, w.ffn), fill=float("nan")),
         "workspace": guarded((u.mlp_workspace_bytes(sh, 1),), torch.uint8)}
    u.mlp_bwd(sh, t["x"], t["Wg"], t["Wu"], t["Wd"], t["dy"], g["dx"].t, g["dWg"].t,
              g["dWu"].t, g["dWd"].t, g["workspace"].t)
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == 0, f"device error word {rc}"
    for name, b in g.items():
        b.check(name)
    return {k: g[k].t for k in ("dx", "dWg", "dWu", "dWd")}


SMALL = [
    # three tiles, the last one ragged (300 = 128 + 128 + 44)
    MlpWorkload("mlp-s300", S=300, hidden=256, ffn=384, tile_rows=128),
    # sequence shorter than one tile
    MlpWorkload("mlp-s77", S=77, hidden=128, ffn=128, tile_rows=256),
    # wider: 256-wide output tiles of y and dx, two split-K partitions
    MlpWorkload("mlp-s2500", S=2500, hidden=512, ffn=1024, tile_rows=1024),
    # 18 row blocks in the first tile: the gate/up and dA GEMMs' grouped tile
    # order runs a full group of 16 row blocks, then a partial group of 2;
    # the second tile (296 rows) is ragged
    MlpWorkload("mlp-s2600-groups", S=2600, hidden=256, ffn=384, tile_rows=2304),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_mlp_matches_oracle(w):
    inp = make_mlp_inputs(w, seed=0, with_grad=True)
    t = {k: v.cuda() for k, v in inp.items()}
    a = {k: f64(v) for k, v in inp.items()}
    ref = O.mlp_backward(a["x"], a["Wg"], a["Wu"], a["Wd"], a["dy"])
    y = run_fwd(w, t)
    assert_close(f64(y), ref["y"], f"{w.name} y")
    g = run_bwd(w, t)
    for name in ("dx", "dWg", "dWu", "dWd"):
        assert_close(f64(g[name]), ref[name], f"{w.name} {name}")


def test_mlp_rows_do_not_depend_on_the_tile_size():
    base = MlpWorkload("mlp-tiles", S=1000, hidden=256, ffn=512, tile_rows=1024)
    t = {k: v.cuda() for k, v in make_mlp_inputs(base, seed=2, with_grad=True).items()}
    y0 = run_fwd(base, t).clone()
    g0 = {k: v.clone() for k, v in run_bwd(base, t).items()}
    for tile in (128, 384):
        w = base.with_(tile_rows=tile)
        assert torch.equal(run_fwd(w, t), y0), tile
        g = run_bwd(w, t)
        assert torch.equal(g["dx"], g0["dx"]), tile
        for name in ("dWg", "dWu", "dWd"):
            # fp32 reduce-adds over a different number of tiles: summation order
            assert_close(f64(g[name]), f64(g0[name]), f"{name} tile={tile}", 1e-4, 1e-5)


def test_mlp_full_size_sampled_rows():
    # the benchmark's MLP (Llama-3-8B widths, one rank's 131072 tokens, tiles
    # of 8192): y and dx on a seeded sample of rows against the oracle on
    # those rows alone (rows are independent; dx of a row needs only its own
    # x and dy); the weight gradients must be finite
    w = MLP_WORKLOADS["llama3-8b-mlp-rank-s1m"]
    t = make_mlp_inputs(w, seed=0, device="cuda", with_grad=True)
    rows = np.asarray(sample_rows(w.S, 256, tile=w.tile_rows))
    y = f64(run_fwd(w, t)[rows])
    g = run_bwd(w, t)
    for name in ("dWg", "dWu", "dWd"):
        assert torch.isfinite(g[name]).all(), name
    dx = f64(g["dx"][rows])
    idx = torch.from_numpy(rows).cuda()
    a = {k: f64(v) for k, v in t.items() if k not in ("x", "dy")}
    ref = O.mlp_backward(f64(t["x"][idx]), a["Wg"], a["Wu"], a["Wd"], f64(t["dy"][idx]))
    assert_close(y, ref["y"], "y rows")
    assert_close(dx, ref["dx"], "dx rows")


def test_mlp_weight_gradients_at_full_widths():
    # Llama-3-8B's MLP widths (hidden 4096, ffn 14336) on 3000 tokens in tiles
    # of 1024 (three tiles, the last one ragged): every gradient in full,
    # against the whole float64 backward
    w = MlpWorkload("mlp-widths-s3000", S=3000, hidden=4096, ffn=14336, tile_rows=1024)
    inp = make_mlp_inputs(w, seed=5, with_grad=True)
    t = {k: v.cuda() for k, v in inp.items()}
    g = run_bwd(w, t)
    a = {k: f64(v) for k, v in inp.items()}
    ref = O.mlp_backward(a["x"], a["Wg"], a["Wu"], a["Wd"], a["dy"])
    for name in ("dx", "dWg", "dWu", "dWd"):
        assert_close(f64(g[name]), ref[name], f"{name} at full widths")
