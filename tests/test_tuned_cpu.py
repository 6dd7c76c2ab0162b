"""Host logic of the benchmark's launch configurations: the autotuner cache
entries are read back into knobs (latest entry wins, timing-log lines and
other shapes are ignored), and without an entry the measured defaults stand."""
import json

from chunk_scheduled_communication_gb300 import tuned
from chunk_scheduled_communication_gb300 import workloads as wl


def _line(op, w, **kn):
    base = dict(op=op, R=w.R, rank=0, M=w.M, N=w.N, K=w.K, backend=2, comm_sms=8, tile_m=256, tile_n=256,
                group_m=8, stages=0, reduce_warps=0, direct_fetch=0, split=1, order=0, us=100.0)
    base.update(kn)
    return json.dumps(base)


def test_cache_entries_override_defaults(tmp_path, monkeypatch):
    cache = tmp_path / "tune.jsonl"
    w = wl.QWEN2_7B_DOWN_AR
    cache.write_text("\n".join([
        _line(2, w, backend=3, stages=5, split=2),
        _line(2, w, backend=3, stages=4, split=3, order=2, group_m=16),            # latest wins
        _line(2, w, backend=0, split=4, phase="final"),                           # a timing log line
        _line(2, wl.scaled(w, M=8192), backend=1),                                 # another shape
    ]) + "\n")
    monkeypatch.setenv("SYN_TUNE_CACHE", str(cache))
    knobs, source = tuned.bench_knobs()
    assert source["ar"] == "autotuner cache" and source["ag"] == "measured defaults"
    assert knobs["ar"] == dict(backend="tma_colocated_smem", split=3, order="grouped", tile_m=256, tile_n=256,
                               comm_sms=8, group_m=16, stages=4, reduce_warps=0, direct_fetch=0)
    assert knobs["ag"] == tuned.STEP_KNOBS["ag"]
    split, order, kn = tuned.knobs_for("ar")
    assert (split, order, kn["stages"]) == (3, "grouped", 4)


def test_missing_cache_keeps_defaults(tmp_path, monkeypatch):
    monkeypatch.setenv("SYN_TUNE_CACHE", str(tmp_path / "absent.jsonl"))
    knobs, source = tuned.bench_knobs()
    assert knobs == tuned.STEP_KNOBS and set(source.values()) == {"measured defaults"}
