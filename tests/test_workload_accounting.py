"""The harness's byte/FLOP accounting against the figures the page states."""
import json
import os

from compressed_sparse_attention_compress_gb300 import workload
from compressed_sparse_attention_compress_gb300.inputs import WORKLOADS

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "paper_facts.json")))


def test_replicated_state_matches_page():
    f = GOLD["replicated_state_1M"]
    b = workload.compressed_state_bytes(f["tokens"], f["ratio"], f["main_kv_dims"] + f["indexer_dims"],
                                        f["bytes_per_elem"])
    assert round(b / 2**20) == f["approx_mib"]
    g = GOLD["replicated_state_21_layers"]
    assert round(g["layers"] * b / 2**30, 1) == g["approx_gib"]


def test_headline_counts():
    c = workload.counts(WORKLOADS["warmup32k"])
    assert c["queries"] == 32768
    assert c["attn_flops"] == 4 * 64 * 128 * c["attn_pairs"]
    # causal visible pairs: sum_t floor((t+1)/4)
    assert c["visible_pairs"] == sum((t + 1) // 4 for t in range(32768))
    assert abs(c["total_flops"] - 4.40e12) / 4.40e12 < 0.01


def test_thd_lengths_and_capacity():
    wl = WORKLOADS["thd128k"]
    assert wl.T == 140343 and wl.T_cap % 128 == 0 and wl.n_cmp == 35081
