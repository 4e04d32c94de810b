"""CPU checks of the persistent GEMM's tile walk (upipe_gemm_tile_order, the
host copy of the device function every GEMM launch uses to map a tile index
to its work).  What is checked are the properties the kernels rely on, not
the formula: every output tile's K range is covered exactly once across the
split-K partitions, each partition is one contiguous run of tile indices,
and each order keeps the promise it makes about which operand stays in L2
(one contiguous run per A row block, per B column tile, or per column tile
within a group of G row blocks)."""
import itertools

import pytest


@pytest.fixture(scope="module")
def u():
    import os
    import headwise_chunked_attention_gb300 as mod
    if not os.path.exists(mod.lib_path()):
        from headwise_chunked_attention_gb300.build import build
        build()
    mod.lib()
    return mod


SHAPES = list(itertools.product([1, 2, 15, 16, 17, 33, 64, 70], [1, 3, 16, 112],
                                [1, 2, 3], [1, 7, 64]))


def runs(seq):
    """Number of maximal runs of equal consecutive values."""
    return sum(1 for i, v in enumerate(seq) if i == 0 or v != seq[i - 1])


@pytest.mark.parametrize("m_fastest", [0, 1, 2, 16, 100])
def test_every_tile_and_k_block_is_covered_once(u, m_fastest):
    for num_m, num_n, ksplit, kb_total in SHAPES:
        walk = u.gemm_tile_order(num_m, num_n, kb_total, ksplit, m_fastest)
        per_split = num_m * num_n
        assert len(walk) == per_split * ksplit
        covered = {}
        for t, (m, n, k0, k1) in enumerate(walk):
            assert 0 <= m < num_m and 0 <= n < num_n, (t, m, n)
            assert 0 <= k0 and k1 <= kb_total
            covered.setdefault((m, n), []).append((t // per_split, k0, k1))
        assert len(covered) == per_split
        for (m, n), parts in covered.items():
            # one entry per partition, and the non-empty K ranges tile [0, kb_total)
            assert sorted(p[0] for p in parts) == list(range(ksplit)), (m, n)
            ranges = sorted((k0, k1) for _, k0, k1 in parts if k1 > k0)
            assert ranges[0][0] == 0 and ranges[-1][1] == kb_total, (m, n, ranges)
            for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
                assert a1 == b0, (m, n, ranges)
        # a partition is a contiguous run of tile indices with one K range
        for ks in range(ksplit):
            part = walk[ks * per_split:(ks + 1) * per_split]
            assert len({(k0, k1) for _, _, k0, k1 in part}) == 1


def test_k_partitions_are_as_even_as_the_block_count_allows(u):
    # ceil-sized partitions: all but the last non-empty one hold ceil(kb/ks)
    for kb_total, ksplit in [(64, 3), (65, 2), (7, 7), (5, 8), (128, 5)]:
        walk = u.gemm_tile_order(1, 1, kb_total, ksplit, 0)
        sizes = [k1 - k0 for _, _, k0, k1 in walk if k1 > k0]
        per = -(-kb_total // ksplit)
        assert all(s == per for s in sizes[:-1]) and 0 < sizes[-1] <= per
        assert sum(sizes) == kb_total


def test_column_fastest_keeps_each_a_row_block_in_one_run(u):
    for num_m, num_n, ksplit, kb_total in SHAPES:
        walk = u.gemm_tile_order(num_m, num_n, kb_total, ksplit, 0)
        for ks in range(ksplit):
            part = walk[ks * num_m * num_n:(ks + 1) * num_m * num_n]
            assert runs([m for m, _, _, _ in part]) == num_m


def test_row_fastest_keeps_each_b_column_tile_in_one_run(u):
    for num_m, num_n, ksplit, kb_total in SHAPES:
        walk = u.gemm_tile_order(num_m, num_n, kb_total, ksplit, 1)
        for ks in range(ksplit):
            part = walk[ks * num_m * num_n:(ks + 1) * num_m * num_n]
            assert runs([n for _, n, _, _ in part]) == num_n


@pytest.mark.parametrize("G", [2, 16])
def test_grouped_order_sweeps_the_columns_once_per_group(u, G):
    # the walk visits the row blocks group by group (G row blocks each, the
    # last group ragged); within a group each B column tile is one run over
    # the group's row blocks, so only G row blocks of A need stay in L2 while
    # B is read once per group
    for num_m, num_n, ksplit, kb_total in SHAPES:
        walk = u.gemm_tile_order(num_m, num_n, kb_total, ksplit, G)
        part = walk[:num_m * num_n]
        t = 0
        for g0 in range(0, num_m, G):
            gm = min(G, num_m - g0)
            block = part[t:t + gm * num_n]
            t += gm * num_n
            assert {m for m, _, _, _ in block} == set(range(g0, g0 + gm)), (num_m, num_n, g0)
            assert runs([n for _, n, _, _ in block]) == num_n
            assert [n for _, n, _, _ in block[::gm]] == list(range(num_n))
        assert t == len(part)


def test_grouped_order_with_one_group_is_row_fastest(u):
    # G at least the row-block count: one group, the same walk as row fastest
    for num_m, num_n in [(1, 5), (16, 3), (17, 112)]:
        assert (u.gemm_tile_order(num_m, num_n, 8, 2, max(num_m, 2)) ==
                u.gemm_tile_order(num_m, num_n, 8, 2, 1))


def test_invalid_arguments_are_rejected(u):
    import ctypes
    L = u.lib()
    code = {name: c for c, name in u.ERR_NAMES.items()}
    invalid = code["UPIPE_ERR_INVALID_ARG"]
    buf = (ctypes.c_int32 * 64)()
    assert L.upipe_gemm_tile_order(2, 2, 4, 1, 0, buf, 64) == code["UPIPE_OK"]
    for args in [(0, 2, 4, 1, 0), (2, 0, 4, 1, 0), (2, 2, 0, 1, 0), (2, 2, 4, 0, 0),
                 (2, 2, 4, 1, -1), (2, 2, 4, 1, 2 ** 30)]:
        assert L.upipe_gemm_tile_order(*args, buf, 64) == invalid, args
    # short output buffer, NULL output
    assert L.upipe_gemm_tile_order(4, 4, 4, 1, 0, buf, 63) == invalid
    assert L.upipe_gemm_tile_order(2, 2, 4, 1, 0, None, 64) == invalid
