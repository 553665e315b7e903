"""bench.py's command line on CPU: the reference arm (the fp64 oracle on the
host cores) runs without a GPU, so the workload options can be checked
end to end here. The line carries the contract's keys and names the shape
it ran."""
import contextlib
import io
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(argv):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(argv) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_on_an_ad_hoc_shape():
    line = _run(["--impl", "reference", "--shape", "48x40x24",
                 "--steps", "2", "--warmup", "3"])
    assert line["impl"] == "reference"
    assert line["config"]["workload"] == "shape_48x40x24"
    assert (line["config"]["M"], line["config"]["N"],
            line["config"]["K"]) == (48, 40, 24)
    assert line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["warmup"] == 3 and line["steps"] == 2


def test_reference_arm_on_a_named_workload():
    line = _run(["--impl", "reference", "--workload", "ragged_127x129x33",
                 "--steps", "1", "--warmup", "3"])
    assert line["config"]["workload"] == "ragged_127x129x33"
    assert line["config"]["inputs"] == "uniform, seed 3"


def test_bad_ops_are_refused():
    sys.path.insert(0, ROOT)
    import bench
    with pytest.raises(SystemExit):
        with contextlib.redirect_stderr(io.StringIO()):
            bench.main(["--ops", "XY"])
