"""Host-side pieces of bench.py on CPU: the oracle leg (timing and the parity record it adds
to each bench leg) and the compact summary that closes the bench line."""
import argparse

import numpy as np

import bench
from oracle import oracle
from workloads import config_case


def test_oracle_leg_parity_and_units():
    case = config_case(1)
    kp, vp = case.k_pool.copy(), case.v_pool.copy()
    slots = oracle.slot_mapping(case.block_table, case.context_lens, case.q_indptr,
                                case.page_size)
    oracle.store(kp, vp, case.k_new, case.v_new, slots)
    ref, _ = oracle.attention(case.q, kp, vp, case.block_table, case.context_lens,
                              case.q_indptr)
    off = ref.copy()
    off[0, 0, 0] += 0.5                       # one element off by 0.5
    r = bench.oracle_leg(case, ref, "GB/s", seconds=0.0, also={"shifted": off})
    assert r["kind"] == "oracle" and r["cores"] >= 1 and r["value"] > 0
    assert r["parity_vs_gpu"]["max_abs"] == 0.0 and r["parity_vs_gpu"]["ok"]
    assert r["parity_shifted"]["max_abs"] == 0.5 and not r["parity_shifted"]["ok"]
    assert r["parity_shifted"]["elements"] == ref.size
    # the bytes of the step over all sequences: K/V of every position, Q, O, the store
    seqs = np.arange(case.num_seqs)
    assert bench._sub_bytes(case, seqs) == bench.decode_bytes(case) + bench.store_bytes(case)


def test_append_units_match_the_gpu_leg():
    case = config_case(4, num_seqs=3)
    _, flops = bench.append_work(case)
    assert abs(bench._sub_case_units(case, np.arange(3), "TFLOP/s") - flops / 1e12) < 1e-15


def test_summary_is_compact_and_last():
    leg = {"cpu_baseline": {"seconds_per_pass": 0.5,
                            "parity_vs_gpu": {"max_abs": 1e-3, "mean_abs": 1e-5}}}
    line = {"value": 5000.0, "roofline": {"frac": 0.8}, **leg,
            "tiny_decode": {"us": 9.0, **leg},
            "append": {"p16": {"roofline_frac": 0.7, "tflops": 600.0, "int8": {
                "roofline_frac": 0.5}, **leg}},
            "decode_legs": {"long_decode": {"frac_of_hbm": 0.95, **leg},
                            "shared_prefix": {"grouped_frac_of_hbm": 0.8, **leg}}}
    s = bench.summary_of(line)
    assert s["decode_frac"] == 0.8 and s["append_p16_frac"] == 0.7
    assert s["int8_append_p16_frac"] == 0.5 and s["long_decode_parity"] == [1e-3, 1e-5]
    assert s["tiny_us"] == 9.0 and s["shared_prefix_oracle_s"] == 0.5
    assert len(str(s)) < 1500


def test_both_arms_print_the_same_config():
    case = config_case(2)
    args = argparse.Namespace(flush_mb=512)
    assert bench.headline_config(case, args, 1)["workload"] == bench.WORKLOAD
    assert bench.headline_config(case, args, 1) == bench.headline_config(case, args, 1)
