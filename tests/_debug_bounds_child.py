"""Child process of test_debug_bounds: run with UPIPE_DEBUG_BOUNDS=1 (and
UPIPE_BWD_WALK=4, so that the backward also runs its split query walks), it
loads the bounds-checked build of the library and runs every entry point
(attention, MLP and loss) on small shapes against the float64 oracle.  Each call must leave the device
error word clear (a failed bounds check would report UPIPE_ERR_BOUNDS) and
the guard margins untouched.  Exits non-zero on any failure."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import headwise_chunked_attention_gb300 as u  # noqa: E402
from tests import test_parity_bwd as PB  # noqa: E402
from tests import test_parity_fused as PF  # noqa: E402
from tests import test_parity_fwd as PW  # noqa: E402
from tests._util import f64, assert_close, GAIN_MAX_REL, GAIN_MEAN_REL  # noqa: E402
from workloads import Workload, make_inputs  # noqa: E402


def main():
    assert u.DEBUG_BOUNDS and u.debug_bounds(), "not the debug build"
    assert os.environ.get("UPIPE_BWD_WALK"), "run with UPIPE_BWD_WALK set"
    # the checks fire: the self-test's write past its declared view is
    # refused and reported, and the next read of the error word is clear
    assert u.selftest_bounds() is False
    assert u.last_error() == u.ERR_BOUNDS
    assert u.last_error() == 0
    # forward and fused forward (every call asserts a clear error word)
    for w in PW.SMALL:
        inp = make_inputs(w, seed=0, norm_gains="random")
        ref = PF.oracle_fwd(w, inp)
        for ch in w.chunk_heads:
            PW.check_full(w, ch, inp)
            PF.check(w, ch, inp, ref)
    for S in (1, 129, 257):
        w = Workload("ragged", S=S, hidden=256, Hq=2, Hkv=1, d=128, chunk_heads=(1,),
                     rope_theta=1e4)
        inp = make_inputs(w, seed=S)
        PF.check(w, 1, inp, PF.oracle_fwd(w, inp))
    # rows long enough to fold O into the per-SM rows (d = 64, 70000 tokens)
    w = Workload("d64-s70000", S=70000, hidden=256, Hq=1, Hkv=1, d=64, chunk_heads=(1,),
                 rope_theta=1e4)
    t = {k: v.cuda() for k, v in make_inputs(w, seed=6).items()}
    out, lse = PF.run_fused(w, 1, t)
    out_u, lse_u = PF.run_unfused(w, 1, t)
    assert torch.equal(lse, lse_u)
    # backward with recompute and with the saved attention output
    for w, chs in PB.CASES:
        inp = make_inputs(w, seed=0, with_grad=True, norm_gains="random")
        ref = PB.oracle_bwd(w, inp)
        for ch in chs:
            for saved in (False, True):
                g = PB.run_fwd_bwd(w, ch, inp, saved_o=saved)
                for name in ("dx", "dWq", "dWk", "dWv", "dWo"):
                    assert_close(f64(g[name]), ref[name], f"{w.name} {name} ch={ch}")
                if w.qk_norm:
                    for name in ("dq_gamma", "dk_gamma"):
                        assert_close(f64(g[name]), ref[name], f"{w.name} {name} ch={ch}",
                                     GAIN_MAX_REL, GAIN_MEAN_REL)
    # the sequence-tiled MLP, forward and backward
    from tests import test_parity_mlp as PM
    from workloads import make_mlp_inputs
    import oracle as O
    for w in PM.SMALL:
        inp = make_mlp_inputs(w, seed=0, with_grad=True)
        t = {k: v.cuda() for k, v in inp.items()}
        a = {k: f64(v) for k, v in inp.items()}
        ref = O.mlp_backward(a["x"], a["Wg"], a["Wu"], a["Wd"], a["dy"])
        assert_close(f64(PM.run_fwd(w, t)), ref["y"], f"{w.name} y")
        g = PM.run_bwd(w, t)
        for name in ("dx", "dWg", "dWu", "dWd"):
            assert_close(f64(g[name]), ref[name], f"{w.name} {name}")
    # the sequence-tiled loss, forward and backward
    from tests import test_parity_loss as PL
    for w in PL.SMALL:
        PL.test_loss_matches_oracle(w)
    print("debug bounds ok")


if __name__ == "__main__":
    main()
