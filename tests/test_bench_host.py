"""Host-side logic of the benchmark on CPU: the provenance rule of the
profiled DRAM traffic and the phase table of the draft launch's marks."""
import bench


def test_profiled_traffic_is_null_once_the_kernel_sources_change(monkeypatch):
    """The bench reports a captured DRAM figure only for the sources it was
    captured on (hash of the kernel files); any other hash gives null."""
    t = dict(bench.PROFILED_TRAFFIC["draft"])
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "draft", {**t, "source_sha": bench.source_sha("draft")})
    assert bench.traffic_of("draft") == t["dram_bytes"]
    assert "ncu" in bench.traffic_note("draft")
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "draft", {**t, "source_sha": "0" * 16})
    assert bench.traffic_of("draft") is None
    assert "no ncu capture" in bench.traffic_note("draft")


def test_timeline_phases_on_synthetic_marks():
    """The phase table of the profiling build's marks: first marks stored
    complemented, last marks plain, sums per block; times relative to the
    launch's first block."""
    import numpy as np
    buf = np.zeros((8, 256, 48), np.uint64)
    ev = bench.TL_EVENTS
    for sl in range(8):
        base = 10 ** 9 + sl * 30000
        for b in range(4):
            for j, nm in enumerate(ev):
                if nm in bench.TL_SUM_EV:
                    buf[sl, b, j] = 10 + b
                elif nm in bench.TL_FIRST_EV:
                    buf[sl, b, j] = ~np.uint64(base + 1000 * j + 100 * b)
                else:
                    buf[sl, b, j] = base + 1000 * j + 100 * b
    t = bench.timeline_phases(buf, range(1, 8), 4)
    assert t["entry"]["min"] == 0.0 and abs(t["entry"]["max"] - 0.3) < 1e-9
    j = ev.index("dn_last")
    assert abs(t["dn_last"]["median"] - (j + 0.15)) < 1e-9
    assert t["bytes"]["per_block_mean"] == 11.5 and t["bytes"]["total"] == 46
    assert abs(t["launch_period_us"] - 30.0) < 1e-9
