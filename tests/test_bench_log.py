"""The bench's run record (CPU only): the clock verdict over sampled clocks
(a run counts only with no slowdown reason other than the power cap and the
SM clock at or above 85% of its maximum) and the append-only JSON-lines log,
each line with the commit it ran from."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(tmp_path, rows):
    c = bench.Clocks(0)
    c.proc = object()  # a sampler that ran
    c.path = str(tmp_path / "clocks.csv")
    with open(c.path, "w") as f:
        for r in rows:
            f.write(", ".join(r) + "\n")
    return c.summary()


def _row(mhz, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    return ["0", str(mhz), "2070", "900.0", "0x0"] + flags


def test_clock_verdict(tmp_path):
    assert _summary(tmp_path, [_row(2070)] * 5)["ok"] is True
    assert _summary(tmp_path, [_row(2070, ("sw_power_cap",))] * 5)["ok"] is True
    s = _summary(tmp_path, [_row(2070), _row(2070, ("hw_slowdown",)), _row(2070)])
    assert s["ok"] is False and s["reasons"] == ["hw_slowdown"]
    s = _summary(tmp_path, [_row(1500)] * 5)          # held below 85% of 2070 with no reason
    assert s["ok"] is False and s["sm_mhz"] == 1500.0


def test_log_appends_with_commit(tmp_path, capsys):
    path = str(tmp_path / "runs.jsonl")
    bench.emit({"metric": "m", "value": 1.0}, path)
    bench.emit({"metric": "m", "value": 2.0}, path)
    printed = capsys.readouterr().out.strip().splitlines()
    assert [json.loads(x)["value"] for x in printed] == [1.0, 2.0]
    recs = [json.loads(x) for x in open(path)]
    assert [r["value"] for r in recs] == [1.0, 2.0]
    assert all("commit" in r and "logged_at" in r for r in recs)


def test_memory_pre_check_records_why_a_workload_is_skipped():
    """A workload is run only when its device tensors fit in the free memory
    with 10% and 256 MB of headroom; otherwise the line records why."""
    GB = 1 << 30
    assert bench.skip_reason(10 * GB, 100 * GB) is None
    assert bench.skip_reason(int(100 * GB / 1.1), 100 * GB) is not None  # no room left for the headroom
    why = bench.skip_reason(300 * GB, 280 * GB)
    assert why is not None and "322.12 GB" in why and "300.65 GB free" in why


def test_require_clean_refuses_a_modified_or_unknown_tree():
    assert bench.require_clean("ab12cd3") is None
    assert bench.require_clean("ab12cd3+dirty") == "--require-clean: tracked files differ from ab12cd3"
    assert bench.require_clean(None) == "--require-clean: not a git work tree"
