"""bench.py's JSON line on the CPU: the reference arm (the oracle on the host cores) on the
tiny workload, and the helpers the GPU arm reports with."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "1",
                          "--steps", "2", "--warmup", "3", "--cpu-budget", "1"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [x for x in out.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["metric"] == bench.METRIC and j["unit"] == bench.UNIT
    assert j["steps"] == 2 and j["warmup"] == 3 and j["higher_is_better"] is True
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle"
    assert 1 <= j["cpu_baseline"]["cores"] <= j["cpu_baseline"]["cores_available"]
    assert j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert j["config"]["workload"] == "tiny-decode"


def test_warmup_below_three_is_refused():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "1"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "--warmup must be >= 3" in out.stderr


def test_threads_used_is_cpu_time_over_wall_time():
    assert bench.threads_used(16.0, 1.0) == 16
    assert bench.threads_used(0.4, 1.0) == 1
    assert bench.threads_used(0.0, 0.0) == 1


def test_percentiles_nearest_rank():
    assert bench.percentiles([5, 1, 2, 3, 4, 6, 7, 8, 9, 10]) == [2, 5, 9]
    assert bench.percentiles([0.25]) == [0.25, 0.25, 0.25]
    assert bench.percentiles([]) is None


@pytest.mark.parametrize("index", [1, 2])
def test_small_workloads_are_timed_with_an_l2_flush(index):
    # the tiny and Qwen2.5-0.5B batches hold far less KV than twice the 129 MB L2, so the GPU
    # arm flushes L2 (a scratch write of FLUSH_BYTES) before each of their timed steps
    from paged_kv_gqa_14_gb300 import workloads as W

    bt = W.config(index, poison=False)
    assert bench.kv_unique_bytes(bt) < 2 * bench.L2_BYTES
    assert bench.FLUSH_BYTES >= 2 * bench.L2_BYTES


def test_gpu_count_must_match_the_launched_processes():
    # without torchrun there is one process: --gpus 2 is refused instead of printing n_gpus 1
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                          "--workload", "1"], capture_output=True, text=True, timeout=120, cwd=ROOT, env=env)
    assert out.returncode != 0 and "--gpus 2 but 1 process" in out.stderr


def test_prefill_flops_count_unmasked_pairs():
    # a 3-row span over 5 keys sees 3 + 4 + 5 keys; decode rows are not counted
    from paged_kv_gqa_14_gb300 import workloads as W

    bt = W.make_batch([5, 9], [3, 1], 4, 2, 64, 4, seed=0)
    assert bench.prefill_flops(bt) == 4 * 64 * 4 * (3 + 4 + 5)
    # the mixed workload: 2,098,176 pairs per head x 16 heads x 4 x 128
    bt5 = W.config(5, poison=False)
    assert bench.prefill_flops(bt5) == 2_098_176 * 16 * 4 * 128


def test_traffic_record_is_read_back_only_for_the_same_sources(tmp_path, monkeypatch):
    csv = tmp_path / "cap.csv"
    csv.write_text(
        '"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
        '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n'
        '"3","1","p","h","void pkv::decode_tc_kernel<128, 2, 16>(pkv::DecodeTcParams)","1","7","(288, 1, 1)",'
        '"(152, 1, 1)","0","10.3","m","dram__bytes_read.sum","byte","1,000"\n'
        '"3","1","p","h","void pkv::decode_tc_kernel<128, 2, 16>(pkv::DecodeTcParams)","1","7","(288, 1, 1)",'
        '"(152, 1, 1)","0","10.3","m","dram__bytes_write.sum","Kbyte","2"\n')
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "traffic.json"))
    rec = bench.record_traffic(str(csv), "decode", "w3", "ncu ...")
    assert rec["dram_bytes_per_launch"] == 3000 and rec["launches"] == 1
    assert bench.kernel_traffic("decode", "w3") == 3000.0
    assert bench.kernel_traffic("decode", "other") is None
    monkeypatch.setattr(bench, "source_sha256", lambda: "changed")
    assert bench.kernel_traffic("decode", "w3") is None


@pytest.mark.parametrize("index", [1, 2])
def test_early_streaming_rule_small_batches(index):
    # PKV_ATTN_STREAM_EARLY is set for batches whose block tables hold at least 2^17 key slots:
    # not for the two small workloads, at any block size (the rule counts tokens, not blocks)
    from paged_kv_gqa_14_gb300 import ops
    from paged_kv_gqa_14_gb300 import workloads as W

    for bs in (8, 16, 128):
        bt = W.config(index, poison=False, block_size=bs)
        assert not ops.stream_early_pays(bt.num_seqs, bt.block_tables.shape[1], bt.block_size)


def test_early_streaming_rule_large_batches():
    # the three large workloads (sequences x longest context): 256 x 2048, 50 x 8192, 204 x 2048
    from paged_kv_gqa_14_gb300 import ops

    for seqs, keys in [(256, 2048), (50, 8192), (204, 2048)]:
        for bs in (8, 16, 128):
            assert ops.stream_early_pays(seqs, keys // bs, bs)
    assert ops.stream_early_pays(1, 1 << 13, 16) and not ops.stream_early_pays(1, (1 << 13) - 1, 16)
