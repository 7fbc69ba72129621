"""The bench's roofline classification of the lm_head: the bound follows the
launch's arithmetic intensity (2 M flops per weight element of 2 bytes, so
M flops per byte for M block rows) against the ridge point of the measured
peaks, so a drafting round at batch 1 or 4 is weight-streaming (HBM) and a
batch of 64 requests is a dense contraction (tensor)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workload import get_config  # noqa: E402

HBM_GBS, TFLOPS = 6789.6, 1721.3  # a measured copy bandwidth and sustained bf16 rate of this part


def _lm_head(name, batch):
    cfg = get_config(name)
    M = cfg.block * batch
    flops = 2.0 * M * cfg.vocab * cfg.hidden
    nbytes = cfg.vocab * cfg.hidden * 2 + M * cfg.hidden * 2
    return flops, nbytes


def test_drafting_workloads_classified_by_intensity():
    assert bench.roofline_bound(*_lm_head("qwen3-8b", 1), HBM_GBS, TFLOPS) == "hbm"
    assert bench.roofline_bound(*_lm_head("llama3.1-8b", 1), HBM_GBS, TFLOPS) == "hbm"
    assert bench.roofline_bound(*_lm_head("long-8layer", 4), HBM_GBS, TFLOPS) == "hbm"
    assert bench.roofline_bound(*_lm_head("batched-qwen3-8b", 64), HBM_GBS, TFLOPS) == "tensor"


def test_ridge_point():
    ridge = TFLOPS * 1e12 / (HBM_GBS * 1e9)  # about 253 flops per byte
    assert bench.roofline_bound(0.99 * ridge, 1.0, HBM_GBS, TFLOPS) == "hbm"
    assert bench.roofline_bound(1.01 * ridge, 1.0, HBM_GBS, TFLOPS) == "tensor"


def test_lm_head_traffic_only_for_the_captured_build_and_workload():
    """The committed DRAM-traffic figure is reported only while the GEMM's
    sources hash to the captured build, and only for the workload it scales to."""
    import re
    text = open(os.path.join(ROOT, "profiles", "lm_head_traffic_mid.md")).read()
    want = re.search(r"^source_sha256: ([0-9a-f]{64})$", text, re.M).group(1)
    traffic = int(re.search(r"^traffic_bytes_per_launch: (\d+)$", text, re.M).group(1))
    expect = traffic if bench.gemm_source_hash() == want else None
    assert bench.lm_head_traffic(get_config("qwen3-8b")) == expect
    assert bench.lm_head_traffic(get_config("long-8layer")) is None
    # a traffic figure is DRAM bytes of one launch: at least the weights it streams
    if expect is not None:
        cfg = get_config("qwen3-8b")
        assert expect >= cfg.vocab * cfg.hidden * 2
