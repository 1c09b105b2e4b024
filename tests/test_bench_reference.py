"""The reference arm of bench.py (the CPU oracle, timed) prints one well-formed JSON line on
the same metric and workload string as the GPU arm.  CPU only."""
import io
import json
from contextlib import redirect_stdout

import bench


def test_reference_arm_line():
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC
    assert line["value"] > 0 and line["unit"] in ("GB/s", "TOPS")
    assert line["higher_is_better"] is True and line["steps"] == 1 and line["warmup"] == 3
    assert line["config"]["workload"] == bench.workload_desc("tiny")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["h2d_bytes_per_step"] == 0
