"""Host logic of bench.py on CPU (not gpu): the end-to-end step's copy groups
and the per-entry source digests of the committed DRAM-traffic figures."""
import json
import os

import pytest

import bench

CAP = 4 << 20


def _check_groups(calls, bounds, cap=CAP):
    # the groups cover every call once, in step order
    assert [a for a, _ in bounds] == [0] + [e for _, e in bounds[:-1]]
    assert bounds[-1][1] == len(calls)
    for i0, i1 in bounds:
        assert i1 > i0
        ms = {calls[i][0] for i in range(i0, i1)}
        assert len(ms) == 1, "one batch size per group"
        if i1 - i0 > 1:
            assert sum(calls[i][1] for i in range(i0, i1)) <= cap
    # and they are maximal: each group ends because the next call could not join it
    for (i0, i1), (j0, _) in zip(bounds, bounds[1:]):
        assert calls[j0][0] != calls[i0][0] or sum(calls[i][1] for i in range(i0, j0 + 1)) > cap


@pytest.mark.parametrize("name", ["decode7b", "small", "w8a8-3b", "prefill", "stack-decode", "stack-prefill"])
def test_e2e_groups_of_each_workload(name):
    lins, _ = bench.workload_calls(name)
    calls = [(l.M, l.M * l.K * 2) for l in lins]
    bounds = bench.e2e_group_bounds(calls)
    _check_groups(calls, bounds)


def test_e2e_groups_decode_sweep_shape():
    """The decode sweep (M = 1, 8, 32, 128, 256; q, gate_up, down each): small
    batches share one group per batch size; at M = 256 the 9.7 MB down_proj
    input is a group of its own."""
    lins, _ = bench.workload_calls("decode7b")
    calls = [(l.M, l.M * l.K * 2) for l in lins]
    bounds = bench.e2e_group_bounds(calls)
    by_m = {}
    for i0, i1 in bounds:
        by_m.setdefault(calls[i0][0], []).append(i1 - i0)
    assert by_m[1] == [3] and by_m[8] == [3] and by_m[32] == [3]
    assert sum(by_m[256]) == 3 and len(by_m[256]) >= 2


def test_e2e_groups_edge_cases():
    assert bench.e2e_group_bounds([]) == []
    assert bench.e2e_group_bounds([(4, 10 * CAP)]) == [(0, 1)]
    assert bench.e2e_group_bounds([(1, 8), (2, 8), (1, 8)]) == [(0, 1), (1, 2), (2, 3)]
    calls = [(7, CAP // 3)] * 7
    b = bench.e2e_group_bounds(calls)
    assert b == [(0, 3), (3, 6), (6, 7)]
    _check_groups(calls, b)


def test_traffic_entries_name_existing_sources():
    """Each committed traffic figure names the kernel sources its digest covers;
    the digest depends on exactly those files."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    csrc = set(os.listdir(os.path.join(bench.ROOT, "bit_quantized_linear_gb300", "csrc")))
    for key, e in d.items():
        files = e.get("digest_files")
        assert files and set(files) <= csrc, key
        assert len(e["kernel_digest"]) == 16
        assert e["dram_bytes_per_launch"] > 0
    some = ["common.cuh", "kernels.h"]
    assert bench.kernel_digest(some) != bench.kernel_digest(some + ["tc_ptx.cuh"])
    assert bench.kernel_digest(some) == bench.kernel_digest(list(reversed(some)))
