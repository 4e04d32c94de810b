"""GPU parity of the sequence-tiled cross-entropy loss (upipe_loss_fwd /
upipe_loss_bwd, through the C ABI) against the float64 oracle
(oracle/loss.py) on the same seeded inputs.  Each token's loss depends on
that token alone and the CUDA path computes every row the same way in any
tile: the losses, log-sum-exps and dh must be bit-identical across tile
sizes; dW sums over the tiles with fp32 reduce-adds in no fixed order."""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import LOSS_WORKLOADS, LossWorkload, make_loss_inputs, sample_rows
from tests._util import f64, assert_close, LSE_ABS
from tests._guard import guarded

pytestmark = pytest.mark.gpu


def U():
    import headwise_chunked_attention_gb300 as mod
    mod.lib()
    return mod


def shape_of(u, w):
    return u.LossShape(w.S, w.hidden, w.vocab, w.tile_rows)


def run_fwd(w, t, expect_error=0):
    u = U()
    sh = shape_of(u, w)
    g = {"loss": guarded((w.S,), fill=float("nan")), "lse": guarded((w.S,), fill=float("nan")),
         "workspace": guarded((u.loss_workspace_bytes(sh, 0),), torch.uint8)}
    u.loss_fwd(sh, t["h"], t["W"], t["targets"], g["loss"].t, g["lse"].t, g["workspace"].t)
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == expect_error, f"device error word {rc}, expected {expect_error}"
    for name, b in g.items():
        b.check(name)
    return g["loss"].t, g["lse"].t


def run_bwd(w, t, lse, scale):
    u = U()
    sh = shape_of(u, w)
    g = {"dh": guarded((w.S, w.hidden), fill=float("nan")),
         "dW": guarded((w.vocab, w.hidden), fill=float("nan")),
         "workspace": guarded((u.loss_workspace_bytes(sh, 1),), torch.uint8)}
    u.loss_bwd(sh, t["h"], t["W"], t["targets"], lse, scale, g["dh"].t, g["dW"].t,
               g["workspace"].t)
    torch.cuda.synchronize()
    rc = u.last_error()
    assert rc == 0, f"device error word {rc}"
    for name, b in g.items():
        b.check(name)
    return g["dh"].t, g["dW"].t


SMALL = [
    # three tiles, the last one ragged; 256-wide vocabulary tiles
    LossWorkload("loss-s300", S=300, hidden=256, vocab=1024, tile_rows=128),
    # one tile shorter than tile_rows; vocabulary 384: 128-wide tiles
    LossWorkload("loss-s77", S=77, hidden=128, vocab=384, tile_rows=256),
    # wider, several split-K partitions of dW
    LossWorkload("loss-s2500", S=2500, hidden=512, vocab=4096, tile_rows=1024),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_loss_matches_oracle(w):
    inp = make_loss_inputs(w, seed=0)
    t = {k: v.cuda() for k, v in inp.items()}
    h, W, tg = f64(inp["h"]), f64(inp["W"]), inp["targets"].numpy()
    ref = O.loss_forward(h, W, tg)
    loss, lse = run_fwd(w, t)
    dl = np.abs(f64(lse) - ref["lse"]).max()
    assert dl <= LSE_ABS, f"{w.name} lse {dl:.3e}"
    dl = np.abs(f64(loss) - ref["loss_rows"]).max()
    assert dl <= LSE_ABS, f"{w.name} loss {dl:.3e}"
    scale = 1.0 / w.S
    gref = O.loss_backward(h, W, tg, scale)
    dh, dW = run_bwd(w, t, lse, scale)
    assert_close(f64(dh), gref["dh"], f"{w.name} dh")
    assert_close(f64(dW), gref["dW"], f"{w.name} dW")


def test_loss_rows_do_not_depend_on_the_tile_size():
    base = LossWorkload("loss-tiles", S=1000, hidden=256, vocab=2048, tile_rows=1024)
    t = {k: v.cuda() for k, v in make_loss_inputs(base, seed=2).items()}
    loss0, lse0 = (x.clone() for x in run_fwd(base, t))
    dh0, dW0 = (x.clone() for x in run_bwd(base, t, lse0, 1e-3))
    for tile in (128, 384):
        w = base.with_(tile_rows=tile)
        loss, lse = run_fwd(w, t)
        assert torch.equal(loss, loss0) and torch.equal(lse, lse0), tile
        dh, dW = run_bwd(w, t, lse, 1e-3)
        assert torch.equal(dh, dh0), tile
        # fp32 reduce-adds over a different number of tiles: summation order
        assert_close(f64(dW), f64(dW0), f"dW tile={tile}", 1e-4, 1e-5)


def test_loss_reports_targets_outside_the_vocabulary():
    w = LossWorkload("loss-bad-target", S=200, hidden=128, vocab=256, tile_rows=128)
    inp = make_loss_inputs(w, seed=4)
    inp["targets"][17] = w.vocab        # one past the last word
    inp["targets"][150] = -1
    t = {k: v.cuda() for k, v in inp.items()}
    loss, _ = run_fwd(w, t, expect_error=U().ERR_TARGET)
    bad = torch.isnan(loss).nonzero().flatten().tolist()
    assert bad == [17, 150], bad
    # the next call starts with a clear error word
    inp["targets"][17] = 3
    inp["targets"][150] = 0
    run_fwd(w, {k: v.cuda() for k, v in inp.items()})


def test_loss_full_size_sampled_rows():
    # the benchmark's loss (Llama-3-8B's vocabulary of 128256, one rank's
    # 131072 tokens, tiles of 4096): losses, lse and dh on a seeded sample of
    # rows against the oracle on those rows alone; dW must be finite
    w = LOSS_WORKLOADS["llama3-8b-loss-rank-s1m"]
    t = make_loss_inputs(w, seed=0, device="cuda")
    rows = np.asarray(sample_rows(w.S, 256, tile=w.tile_rows))
    loss, lse = run_fwd(w, t)
    scale = 1.0 / w.S
    dh, dW = run_bwd(w, t, lse, scale)
    assert torch.isfinite(dW).all()
    idx = torch.from_numpy(rows).cuda()
    h = f64(t["h"][idx])
    W = f64(t["W"])
    tg = t["targets"][idx].cpu().numpy()
    ref = O.loss_forward(h, W, tg)
    assert np.abs(f64(lse[idx]) - ref["lse"]).max() <= LSE_ABS
    assert np.abs(f64(loss[idx]) - ref["loss_rows"]).max() <= LSE_ABS
    gref = O.loss_backward(h, W, tg, scale)
    assert_close(f64(dh[idx]), gref["dh"], "dh rows")


def test_loss_weight_gradient_at_full_vocabulary():
    # Llama-3's vocabulary (128256) and width (4096) on 1500 tokens in tiles
    # of 512 (three tiles, the last one ragged): dW and dh in full against the
    # whole float64 backward
    w = LossWorkload("loss-vocab-s1500", S=1500, hidden=4096, vocab=128256, tile_rows=512)
    inp = make_loss_inputs(w, seed=6)
    t = {k: v.cuda() for k, v in inp.items()}
    loss, lse = run_fwd(w, t)
    scale = 1.0 / w.S
    dh, dW = run_bwd(w, t, lse, scale)
    h, W, tg = f64(inp["h"]), f64(inp["W"]), inp["targets"].numpy()
    ref = O.loss_forward(h, W, tg)
    assert np.abs(f64(loss) - ref["loss_rows"]).max() <= LSE_ABS
    gref = O.loss_backward(h, W, tg, scale)
    assert_close(f64(dh), gref["dh"], "dh at full vocabulary")
    assert_close(f64(dW), gref["dW"], "dW at full vocabulary")
