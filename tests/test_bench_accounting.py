"""The benchmark's FLOP accounting (the numerator of its TFLOP/s figures),
checked on the CPU."""
import pytest

import bench
from workloads import WORKLOADS, Workload


@pytest.mark.parametrize("S", [1, 2, 5, 129])
def test_attention_flops_count_unmasked_pairs(S):
    # causal mask with the diagonal: query i sees keys 0..i; each visible pair
    # costs d multiply-adds for q.k and d for p v, per query head
    w = Workload("count", S=S, hidden=128, Hq=3, Hkv=1, d=64, chunk_heads=(1,), rope_theta=1e4)
    pairs = sum(1 for i in range(S) for j in range(S) if j <= i)
    _, attn = bench.layer_flops(w, "fwd")
    assert attn == 2 * 2 * w.d * w.Hq * pairs


def test_projection_and_wo_flops():
    # x [S, hidden] times Wq^T, Wk^T, Wv^T ([hidden, (Hq + 2 Hkv) d]) and
    # O [S, Hq d] times Wo^T ([Hq d, hidden]): 2 FLOPs per multiply-add
    w = Workload("gemms", S=7, hidden=256, Hq=4, Hkv=2, d=64, chunk_heads=(1,), rope_theta=1e4)
    total, attn = bench.layer_flops(w, "fwd")
    macs = w.S * w.hidden * (w.Hq + 2 * w.Hkv) * w.d + w.S * (w.Hq * w.d) * w.hidden
    assert total - attn == 2 * macs


# hand-computed model FLOPs of the five workloads: forward, backward
EXPECTED = {
    "tiny-s2048": (2.95e9, 6.98e9),
    "llama3.2-3b-s65536": (29.7e12, 72.6e12),
    "llama3-8b-rank-s1m": (1.137e15, 2.84e15),
    "llama3-8b-rank-s5m": (28.2e15, 70.5e15),
    "qwen3-32b-rank-s1m": (2.28e15, 5.68e15),
}


@pytest.mark.parametrize("name", list(EXPECTED))
def test_layer_flops_of_the_workloads(name):
    w = WORKLOADS[name]
    fwd, _ = bench.layer_flops(w, "fwd")
    both, _ = bench.layer_flops(w, "fwdbwd")
    ef, eb = EXPECTED[name]
    assert abs(fwd / ef - 1) < 5e-3, (fwd, ef)
    assert abs((both - fwd) / eb - 1) < 5e-3, (both - fwd, eb)
    # the backward's model count: twice each GEMM of the forward and 10 d per
    # visible pair and head for the attention backward (2.5 times its forward)
    _, attn = bench.layer_flops(w, "fwd")
    assert abs((both - fwd) - (2 * (fwd - attn) + 2.5 * attn)) <= 1e-9 * both


def test_recompute_flops():
    # hardware FLOPs of the backward add the recomputed projections and, unless
    # the forward's attention output is kept, the recomputed attention forward
    w = WORKLOADS["llama3.2-3b-s65536"]
    fwd, attn = bench.layer_flops(w, "fwd")
    wo = 2.0 * w.S * w.Hq * w.d * w.hidden
    proj = fwd - attn - wo
    assert bench.recompute_flops(w) == pytest.approx(proj + attn, rel=1e-12)
    assert bench.recompute_flops(w, saved_o=True) == pytest.approx(proj, rel=1e-12)


def test_ncu_traffic_is_reported_only_for_the_captured_kernel_and_size():
    # the DRAM bytes per launch belong to one kernel source and one workload
    # size: a different S or an edited kernel reports null, never a stale figure
    w = WORKLOADS["llama3-8b-rank-s1m"]
    for kernel in ("attn_fwd_kernel", "attn_bwd_kernel"):
        got = bench.traffic_of(kernel, w.name, 1, w.S)
        ent = bench.NCU_TRAFFIC[(kernel, w.name, 1)]
        assert got == (ent[0] if ent[1] == bench.kernel_source_sha(kernel) else None)
        assert bench.traffic_of(kernel, w.name, 1, 65536) is None
        assert bench.traffic_of(kernel, w.name, 2, w.S) is None
    # the scaled 1M figures are 16x the 256K captures (the causal pairs ratio)
    S1, S2 = w.S, 262144
    assert abs(S1 * (S1 + 1) / (S2 * (S2 + 1)) - 16.0) < 1e-4
