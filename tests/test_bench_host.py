"""Host logic of bench.py: the ncu launch list -> per-op DRAM bytes mapping
that stamps profiles/traffic.json, and the fingerprint check that keeps
counters taken on other kernel sources out of the bench line."""
import csv
import json

import pytest

import bench

# ncu's kernel names for one eager step, in launch order (template flags as
# ncu prints them)
STEP_NAMES = [
    "void sel::(anonymous namespace)::argmax_kernel<true, false, 0>(sel::(anonymous namespace)::ArgmaxArgs)",
    "sel::(anonymous namespace)::argmax_finish_kernel(unsigned long long *, unsigned int *, unsigned int)",
    "void sel::(anonymous namespace)::topk_kernel<true, false, true>(sel::(anonymous namespace)::TopkArgs)",
    "void sel::(anonymous namespace)::topk_finish_kernel<0, 0>(sel::(anonymous namespace)::TopkArgs)",
    "void sel::(anonymous namespace)::topk_kernel<true, false, true>(sel::(anonymous namespace)::TopkArgs)",
    "void sel::(anonymous namespace)::topk_finish_kernel<1, 0>(sel::(anonymous namespace)::TopkArgs)",
    "void sel::(anonymous namespace)::spec_phase1_kernel<1, 1>(sel::(anonymous namespace)::SpecArgs)",
    "sel::(anonymous namespace)::spec_decide_draw_cl_kernel(sel::(anonymous namespace)::SpecArgs, "
    "sel::(anonymous namespace)::DrawArgs, unsigned int)",
    "void sel::(anonymous namespace)::argmax_kernel<true, false, 0>(sel::(anonymous namespace)::ArgmaxArgs)",
    "sel::(anonymous namespace)::spec_argmax_finish_kernel(sel::(anonymous namespace)::SpecArgs)",
]


def _write_csv(path, launches, first_id=30):
    """An ncu --csv launch list: a preamble, the header, then three metric
    rows per launch (time, DRAM read, DRAM write) in mixed byte units."""
    with open(path, "w", newline="") as f:
        f.write("==PROF== Connected to process 1 (python)\n")
        w = csv.writer(f)
        w.writerow(["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream",
                    "Block Size", "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit",
                    "Metric Value"])
        for n, (name, rd, wr) in enumerate(launches):
            lid = str(first_id + n)
            base = [lid, "1", "python", "127.0.0.1", name, "1", "7", "(256, 1, 1)", "(1, 1, 1)", "0", "10.3",
                    "Command line profiler metrics"]
            w.writerow(base + ["gpu__time_duration.sum", "ns", "1,000"])
            w.writerow(base + ["dram__bytes_read.sum", "Kbyte", f"{rd / 1e3:,.3f}"])
            w.writerow(base + ["dram__bytes_write.sum", "byte", f"{wr:,}"])


def test_step_table_names_every_op_once_per_launch_slot():
    assert len(bench.STEP_LAUNCHES) == len(STEP_NAMES)
    for (op, pat), name in zip(bench.STEP_LAUNCHES, STEP_NAMES):
        assert pat in name, (op, pat, name)
    assert {op for op, _ in bench.STEP_LAUNCHES} == {"argmax", "topk", "sample", "spec_rejection", "spec_argmax"}


def test_traffic_is_the_mean_bytes_per_call_of_each_op(tmp_path, monkeypatch):
    out = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(out))
    launches = []
    for step in range(2):
        for j, name in enumerate(STEP_NAMES):
            rd = 1_000_000 * (j + 1) + 1000 * step   # bytes, a multiple of 1 KB
            launches.append((name, rd, 64 * j))
    path = tmp_path / "launches.csv"
    _write_csv(path, launches)
    got = bench.write_traffic(str(path))
    want = {}
    for j, (op, _) in enumerate(bench.STEP_LAUNCHES):
        per_call = sum(1_000_000 * (j + 1) + 1000 * st + 64 * j for st in range(2)) / 2
        want[op] = want.get(op, 0) + per_call
    assert got["ops"] == {op: round(v) for op, v in want.items()}
    assert got["sources"] == bench.sources_fingerprint()
    assert json.loads(out.read_text()) == got


def test_a_capture_that_starts_inside_a_step_is_refused(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tmp_path / "traffic.json"))
    launches = [(name, 1000, 0) for name in STEP_NAMES[1:] + STEP_NAMES]  # shifted by one launch
    path = tmp_path / "launches.csv"
    _write_csv(path, launches)
    with pytest.raises(SystemExit):
        bench.write_traffic(str(path))
    assert not (tmp_path / "traffic.json").exists()


def test_counters_from_other_sources_are_not_reported(tmp_path, monkeypatch):
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(path))
    path.write_text(json.dumps({"sources": "0" * 16, "ops": {"argmax": 5}}))
    assert bench.load_traffic("argmax") is None
    path.write_text(json.dumps({"sources": bench.sources_fingerprint(), "ops": {"argmax": 5}}))
    assert bench.load_traffic("argmax") == 5
    assert bench.load_traffic("topk") is None
