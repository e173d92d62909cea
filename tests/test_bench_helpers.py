"""Host-side logic of bench.py (no GPU): the launch count it claims, the
profile-validity hash, the traffic lookup and the algorithmic-work figures."""

import json
import os

import numpy as np

import bench
import synthetic


def test_launches_per_pass_follows_the_gram_plan():
    # one launch per stage (importance, redundancy, select + compact); the dense
    # Gram adds the single-CTA launch after the CTA-pair one on odd counts of at
    # least 17 key tiles (N = 2176 -> 17 tiles)
    counts = {i: bench.launches_per_pass(synthetic.WORKLOADS[i], "gram") for i in range(5)}
    assert counts == {0: 3, 1: 3, 2: 4, 3: 3, 4: 3}
    # closed form: a kernel of its own; fused: importance and redundancy in one launch
    assert all(bench.launches_per_pass(synthetic.WORKLOADS[i], "closed") == 3 for i in range(5))
    assert all(bench.launches_per_pass(synthetic.WORKLOADS[i], "closed-fused") == 2 for i in range(5))


def test_source_hash_ignores_comments_and_whitespace_only():
    code = "int f(int x)\n{\n    return x + 1; // one more\n}\n"
    same = "/* header */\nint f(int x) {   return x + 1;   }\n"
    other = "int f(int x)\n{\n    return x + 2; // one more\n}\n"
    assert bench.source_code_hash(code) == bench.source_code_hash(same)
    assert bench.source_code_hash(code) != bench.source_code_hash(other)


def test_traffic_lookup_needs_matching_source_and_workload():
    path = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    entries = json.load(open(path))
    for kernel, entry in entries.items():
        if entry.get("source_sha") == bench.kernel_source_hash(kernel):
            assert bench.ncu_traffic(kernel, entry["workload"]) == entry["dram_bytes_per_launch"]
        assert bench.ncu_traffic(kernel, entry["workload"] + "-other") is None


def test_algorithmic_work_of_the_headline_workload():
    s = synthetic.WORKLOADS[1]
    lens = np.full(s.batch, s.max_seq_len)
    keep = np.tile(np.arange(s.budget, dtype=np.int32), (s.layers, s.batch, s.kv_heads, 1))
    work = bench.algorithmic_work(s, lens, keep)
    heads = s.layers * s.batch * s.kv_heads
    # dense Gram: 2 N^2 d flops per head
    assert np.isclose(work["rkv_redundancy"]["work"], heads * 2.0 * s.max_seq_len ** 2 * s.head_dim)
    # importance: K read + the query block + two fp32 outputs per key
    per_head = s.max_seq_len * 256 + s.window * (s.q_heads // s.kv_heads) * 256 + s.max_seq_len * 8
    assert np.isclose(work["rkv_importance"]["work"], heads * per_head)
    # select + compact: identity kept indices move no row; what is left is
    # reading the two score rows and writing the kept indices
    assert np.isclose(work["rkv_select_compact"]["work"], heads * (s.max_seq_len * 8 + s.budget * 4))
