"""The benchmark's JSON contract and bookkeeping, on the CPU: the keys of the line, one
config object for both arms, the median of the timed runs, whole-job throughput over
ranks, and that every profile summary the line reads its DRAM traffic from was taken on
the current attention sources."""
import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

bench = pytest.importorskip("bench")


def _args(**kw):
    a = argparse.Namespace(steps=50, warmup=10)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_line_has_the_contract_keys():
    line = bench.base_line("c2", 1, _args(), 7300.0, 2343.5)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["config"]["workload"] == "llama8b-32layer-b16-ctx8192-full-stack"
    assert line["ms_per_step"] == pytest.approx(2.3435)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["n_gpus"] == 1


@pytest.mark.parametrize("workload", ["c2", "c2-layer", "c1", "c4", "c3"])
def test_both_arms_share_one_config_object(workload):
    # the GPU arm and the reference arm both call config_dict: same object for the same
    # workload and world size, with the fields a reader needs to tell workloads apart
    a, b = bench.config_dict(workload, 2), bench.config_dict(workload, 2)
    assert a == b
    assert a["parallelism"] == "replicas2"
    assert {"workload", "batch", "q_heads", "kv_heads", "head_dim", "page_tokens"} <= set(a)


def test_runs_summary_reports_the_median():
    # five runs of a 50-step graph, in ms; the median run is the 3rd smallest
    ms = [120.0, 117.5, 118.0, 130.0, 117.0]
    r = bench.runs_summary(ms, 50)
    assert r["n"] == 5
    assert r["us_per_step_median"] == pytest.approx(118.0 * 1e3 / 50)
    assert r["us_per_step_runs"][3] == pytest.approx(130.0 * 1e3 / 50)


def test_job_throughput_counts_every_rank():
    # 4 ranks, 1 GB each per step, 10 steps in 10 ms -> 4 TB/s whole job
    assert bench.job_throughput(4, 10**9, 10, 10.0) == pytest.approx(4000.0)


@pytest.mark.parametrize("workload", ["c1", "c2", "c2-layer", "c4"])
def test_profiles_match_the_current_attention_sources(workload):
    # a profile taken on older kernel sources gives no traffic (the line reports null)
    assert bench.profiled_traffic(workload) is not None, (
        f"profiles/k_attn_compressed_{workload}.md was not taken on the current attention sources "
        f"({bench.kernel_source_hash()})")
    assert bench.profiled_traffic("c1", "tiles") is not None


def test_layer_workloads_are_single_layers_of_the_configs():
    import kvgen

    for name, base in (("c1", kvgen.C1), ("c2-layer", kvgen.C2), ("c4", kvgen.C4)):
        cfg = bench.layer_cfg(name)
        assert cfg.layers == 1
        assert (cfg.batch, cfg.hq, cfg.hkv, cfg.full_pages) == (base.batch, base.hq, base.hkv, base.full_pages)
