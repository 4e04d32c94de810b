"""Child process of test_parity_bwd.test_backward_segmented_walks: run with
UPIPE_BWD_WALK set (read once per process), it checks the backward against
the float64 oracle on small shapes and exits non-zero on a mismatch."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from tests.test_parity_bwd import CASES, oracle_bwd, run_fwd_bwd  # noqa: E402
from tests._util import f64, assert_close, GAIN_MAX_REL, GAIN_MEAN_REL  # noqa: E402
from workloads import make_inputs  # noqa: E402


def main():
    assert os.environ.get("UPIPE_BWD_WALK"), "run with UPIPE_BWD_WALK set"
    for w, chs in (CASES[1], CASES[2], CASES[4]):
        inp = make_inputs(w, seed=0, with_grad=True, norm_gains="random")
        ref = oracle_bwd(w, inp)
        for ch in chs:
            g = run_fwd_bwd(w, ch, inp)
            for name in ("dx", "dWq", "dWk", "dWv", "dWo"):
                assert_close(f64(g[name]), ref[name], f"{w.name} {name} ch={ch}")
            if w.qk_norm:
                for name in ("dq_gamma", "dk_gamma"):
                    assert_close(f64(g[name]), ref[name], f"{w.name} {name} ch={ch}",
                                 GAIN_MAX_REL, GAIN_MEAN_REL)
    print("segmented walks ok")


if __name__ == "__main__":
    main()
