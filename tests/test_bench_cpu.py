"""The bench's CPU-side contract: the reference arm (the oracle timed on the
host) prints one JSON line with the keys the driver reads, for a MoE
workload and for the attention leg; the roofline bound follows the ridge of
the measured peaks; the workload table covers every leg."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def run_reference(workload):
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                          workload, "--steps", "1", "--warmup", "1"], cwd=ROOT,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_line_for_a_moe_workload():
    d = run_reference("tiny")
    assert KEYS <= set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens/s"
    assert d["config"]["workload"] == "tiny"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_line_for_the_attention_leg():
    d = run_reference("attn_decode")
    assert KEYS <= set(d)
    assert d["config"]["workload"] == "attn_decode" and d["config"]["L"] == 32768
    assert d["value"] > 0 and d["higher_is_better"] is True


def test_algorithmic_counts():
    """Bytes of an expert, the layer's bytes and FLOPs from a histogram, and
    the attention call's bytes, from their definitions."""
    H, I = 2048, 512
    # packed nibbles (0.5 B per weight) and two bf16 per 64-weight group
    assert bench.expert_bytes(H, I) == 3 * H * I // 2 + 2 * 2 * (3 * H * I // 64)
    S = synth.CONFIGS["prefill"].shape
    counts = np.zeros(S.E, np.int64)
    counts[:3] = [10, 5, 1]
    algo, flops, ffn_bytes, ffn_flops = bench.layer_algo(16, S, counts)
    assert ffn_bytes == 4 * bench.expert_bytes(S.H, S.I) + 16 * S.H * 2 * 2
    assert ffn_flops == 2 * 3 * S.I * S.H * (16 * S.K + 16)
    assert flops == ffn_flops + 2 * S.E * S.H * 16
    c = bench.ATTN_WORKLOADS["attn_decode"]
    assert bench.attn_bytes(c) == c["L"] * 2 * 128 * 4 + 512 * 4 + 2 * 16 * 128 * 2
    # one chunked DeltaNet call at T=2048: q and k (16 heads), v and o (32
    # heads) in bf16, the two fp32 gates, the fp32 state read and written
    g = bench.GDN_WORKLOADS["gdn_prefill"]
    assert (g["T"], g["n_k"], g["n_v"], g["dk"], g["dv"]) == (2048, 16, 32, 128, 128)
    assert bench.gdn_bytes(g) == (2 * 2048 * 16 * 128 * 2 + 2 * 2048 * 32 * 128 * 2 +
                                  2 * 2048 * 32 * 4 + 2 * 32 * 128 * 128 * 4)


def test_tensor_or_hbm_bound_by_the_ridge():
    """At T=512 the grouped GEMMs sit below the ridge of the measured peaks
    (HBM-bound); a Zipf T=2048 layer with about 140 touched experts sits
    above it (tensor-bound)."""
    hbm, bf16, _, _ = bench.peaks()
    ridge = bf16 * 1e3 / hbm
    S = synth.CONFIGS["prefill"].shape
    uniform = np.full(S.E, 16)
    _, _, b512, f512 = bench.layer_algo(512, S, uniform)
    assert f512 / b512 < ridge
    skew = np.zeros(S.E, np.int64)
    skew[:140] = 2048 * S.K // 140
    _, _, b2k, f2k = bench.layer_algo(2048, S, skew)
    assert f2k / b2k > ridge


def test_step_spread_quartiles():
    """Per-step event times are summarised by their median and quartiles."""
    d = bench.step_spread([1.0, 2.0, 3.0, 4.0, 5.0])
    assert d["median"] == 3.0 and d["p25"] == 2.0 and d["p75"] == 4.0 and d["iqr"] == 2.0
    assert d["min"] == 1.0 and d["max"] == 5.0 and d["n"] == 5
    assert bench.step_spread([]) is None


def test_default_run_times_every_graded_workload():
    """The headline plus its legs cover T=1 (decode, 40 layers), T=512 and the
    skewed T=2048 layer."""
    names = {"prefill", *bench.LEGS}
    Ts = {synth.CONFIGS[n].T for n in names}
    assert Ts == {1, 512, 2048}
    assert synth.CONFIGS["decode"].layers == 40 and synth.CONFIGS["skewed"].zipf_s > 0
