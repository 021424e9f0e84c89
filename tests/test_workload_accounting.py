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


def test_backward_counts():
    # attention backward: S recompute, dP, dQ, dK, dV at 2 H d FLOPs each per (query, candidate key);
    # indexer backward: the teacher once plus the indexer dots, dqI and dkI at 2 H_I d_I each
    wl = WORKLOADS["warmup32k"]
    c = workload.counts(wl)
    assert c["attn_bwd_flops"] == 5 * 2 * 64 * 128 * c["attn_pairs"]
    assert c["teacher_pairs"] == c["visible_pairs"]          # dense teacher: every visible entry
    assert c["indexer_bwd_flops"] == (2 * 64 * 128 + 3 * 2 * 8 * 64) * c["teacher_pairs"]
    # the selected teacher counts the selected entries instead
    s = workload.counts(WORKLOADS["csa8k"])
    assert s["teacher_pairs"] == sum(min(512, (t + 1) // 4) for t in range(8192))
