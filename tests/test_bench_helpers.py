"""The bench's byte and FLOP accounting and its roofline bound, checked by hand counts."""
import json
import os

import bench
from workload import make_scenario


def test_attention_bytes_and_flops_by_hand():
    scn = make_scenario(3, V=1000, stream_len=5000)  # B=1, Hq=32, Hkv=8, d=128, N=60, bf16
    P = int(scn.prefix_len[0])
    kv = (P + 60) * 8 * 128 * 2 * 2          # K and V rows of every KV head, bf16
    qo = 2 * 1 * 60 * 32 * 128 * 2           # Q read and O written
    assert bench.attn_bytes(scn) == kv + qo
    assert bench.attn_flops(scn) == 4 * 4 * 60 * (P + 60) * 128 * 8   # 4 g N (P+n) d per head
    scn4 = make_scenario(4, V=1000, P=(100, 900), B=3, stream_len=5000)
    keys = sum(int(p) + 60 for p in scn4.prefix_len)
    assert bench.attn_bytes(scn4) == keys * 8 * 128 * 2 * 2 + 2 * 3 * 60 * 64 * 128 * 2


def test_roofline_bound_follows_the_measured_ridge():
    hbm, _ = bench._peaks()
    tpeak, _ = bench._tensor_peak()
    ridge = tpeak * 1e12 / (hbm * 1e9)
    peaks = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks):  # written per machine; the fallback figures apply otherwise
        with open(peaks) as f:
            assert json.load(f)["hbm_gbs"] == hbm
    # workload 3 sits below the ridge (HBM-bound), workloads 4 and 5 above it (tensor-bound)
    for cid, tensor in ((3, False), (4, True), (5, True)):
        scn = make_scenario(cid, V=1000, stream_len=5000)
        assert (bench.attn_flops(scn) / bench.attn_bytes(scn) > ridge) == tensor, cid


def test_config_objects_describe_the_workload_only():
    """Both arms print the same `config` for a workload: sizes and the L2 rotation, no
    measured value."""
    scn = make_scenario(3, V=1000, stream_len=5000)
    c = bench.workload_config(scn, 3, 0.0)
    assert c["workload"] == scn.name and c["config_id"] == 3 and c["slots"] == 60
    assert c["step_bytes"] == bench.step_bytes(scn) and c["parallelism"] == "single GPU"
    per_set, nsets = bench.rotation(scn)
    assert per_set * nsets >= 4 * bench.L2_BYTES and nsets >= 2
    assert not any("frac" in k for k in c)


def test_reference_arm_line_carries_the_contract_keys():
    """The reference arm times the oracle on the host: one JSON-ready line with the GPU arm's
    metric and unit, impl "reference", a CPU baseline describing the run and an e2e object
    that moves no bytes; ranks other than 0 return nothing."""
    import argparse
    args = argparse.Namespace(config=1, steps=1, warmup=3, ref_budget=0.0, temperature=0.0,
                              seed=1)
    line = bench.run_reference(args, 0, 1)
    json.dumps(line)  # serialisable as printed
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "steps/s"
    assert line["higher_is_better"] is True and line["steps"] >= 1 and line["value"] > 0
    assert line["config"] == bench.workload_config(bench.make_scenario(1), 1, 0.0)
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": "steps/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert bench.run_reference(args, 1, 2) is None
