"""bench.py's host-side bookkeeping, without a GPU: the decode step's products
and bytes, and the provenance of every recorded DRAM-traffic figure."""
import os
import re
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_decode_step_products_and_bytes():
    items = bench.workload_list(4)
    assert len(items) == 28 * 6 + 1 and items[-1][0] == "lm_head"
    # affine 4-bit gs64: half a byte per code plus two bf16 per 64 values
    total = sum(bench.packed_bytes(n, k, 4) for _, n, k in items)
    assert total == sum(n * k // 2 + 2 * n * (k // 64) * 2 for _, n, k in items) == 302211072
    assert bench.config_dict(4, 1)["weight_bytes_per_step"] == total


def test_traffic_figures_name_their_capture():
    # every recorded figure comes from a committed ncu summary of the same kernel version
    profiles = os.path.join(ROOT, "profiles")
    texts = [open(os.path.join(profiles, f)).read() for f in os.listdir(profiles) if f.endswith((".md", ".txt"))]
    for key, (value, commit) in bench.TRAFFIC.items():
        if value is None:
            assert commit is None and bench.traffic(key) == (None, None), key
            continue
        assert value > 0, key
        assert any(re.search(r"commit\s+" + commit, t) for t in texts), (key, commit)
        v, why = bench.traffic(key)
        assert v == value and commit in why and "profiles/" not in why
    assert bench.traffic("dequant", False) == (None, None)


def test_grouped_step_calls():
    # products that read the same activations share a call: per layer q/k/v and
    # gate/up, with down_proj and lm_head alone -- 85 calls over the same 169 products
    items = [(name, n, k, None, None, None) for name, n, k in bench.workload_list(4)]
    groups = bench.step_groups(items, True)
    assert len(groups) == 28 * 3 + 1
    assert [it for g in groups for it in g] == items
    names = [[it[0].split(".")[-1] for it in g] for g in groups[:3]]
    assert names == [["q_proj", "k_proj", "v_proj"], ["gate_proj", "up_proj"], ["down_proj"]]
    assert all(len({it[2] for it in g}) == 1 for g in groups)  # one k per call
    assert [len(g) for g in bench.step_groups(items, False)] == [1] * 169
    # algorithmic bytes of a call: its packed weights, x once, every output
    g = groups[0]
    assert bench.group_algo_bytes(g, 4, 1) == sum(bench.packed_bytes(n, k, 4) + 2 * n for _, n, k, *_ in g) + 2 * 1024
