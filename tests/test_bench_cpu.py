"""Host-side pieces of the benchmark that need no GPU: the code digest that
keeps a committed DRAM-traffic figure tied to the kernels it was measured on,
and the reading of those figures."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_keeps_literals():
    src = 'int a = 1; // note\n/* block\n comment */ const char *s = "//kept /*too*/"; char c = \'/\';\n'
    assert bench.code_only(src) == 'int a = 1; const char *s = "//kept /*too*/"; char c = \'/\';'


def _reader(overrides):
    def read(rel):
        if rel in overrides:
            return overrides[rel]
        return open(os.path.join(ROOT, rel), encoding="utf-8").read()
    return read


def test_digest_ignores_documentation_but_not_code():
    rel = "tenant_composite_lora_gb300/csrc/decode.cu"
    text = open(os.path.join(ROOT, rel), encoding="utf-8").read()
    base = bench.sources_digest("decode")
    assert bench.sources_digest("decode", _reader({rel: "// a new comment line\n" + text})) == base
    assert bench.sources_digest("decode", _reader({rel: text.replace("{", "{ ", 1)})) == base
    assert bench.sources_digest("decode", _reader({rel: text + "\nint extra_symbol;\n"})) != base
    # a header shared by every path changes every path's digest; a path's own file only its own
    hdr = "tenant_composite_lora_gb300/csrc/internal.h"
    htext = open(os.path.join(ROOT, hdr), encoding="utf-8").read() + "\nint extra_symbol;\n"
    for path in bench.PATH_SOURCES:
        assert bench.sources_digest(path, _reader({hdr: htext})) != bench.sources_digest(path)
    assert bench.sources_digest("mma", _reader({rel: text + "\nint extra_symbol;\n"})) == \
        bench.sources_digest("mma")


def test_traffic_files_parse(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic_demo_decode.txt").write_text(
        "# header\ndram_bytes_per_apply: 1234\nsources_sha256_16: %s\n" % bench.sources_digest("decode"))
    (prof / "traffic_stale_decode.txt").write_text("dram_bytes_per_apply: 99\nsources_sha256_16: 0000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "sources_digest", lambda path, read=None: bench_digest[path])
    bench_digest = {"decode": open(prof / "traffic_demo_decode.txt").read().split()[-1]}
    assert bench.ncu_traffic("demo", "decode") == 1234
    assert bench.ncu_traffic("stale", "decode") is None  # taken with other kernel code
    assert bench.ncu_traffic("absent", "decode") is None


def test_cpu_baseline_reports_threads_model_and_single_thread():
    import workloads as W
    cb = bench.oracle_baseline(W.make("tiny"), 0.5)
    assert cb["kind"] == "oracle" and cb["unit"] == "tokens/s" and cb["value"] > 0
    assert cb["cores"] >= 1 and cb["nproc"] >= 1 and isinstance(cb["cpu_model"], str) and cb["cpu_model"]
    st = cb["single_thread"]
    assert st["unit"] == "tokens/s" and st["value"] > 0 and "one thread" in st["sample"]


def test_pass_times_and_spread():
    """Per-pass event timing and its percentiles, with events that tick a
    fake device clock on every replay."""
    clock = {"t": 0.0}
    durations = iter([2.0, 4.0, 3.0, 1.0, 5.0])

    class Event:
        def __init__(self, enable_timing=False):
            assert enable_timing
            self.t = None

        def record(self, stream):
            assert stream == "s"
            self.t = clock["t"]

        def synchronize(self):
            assert self.t is not None

        def elapsed_time(self, other):
            return other.t - self.t

    def replay():
        clock["t"] += next(durations)

    ms = bench.pass_times_ms(replay, 5, "s", Event)
    assert ms == [2.0, 4.0, 3.0, 1.0, 5.0]
    sp = bench.spread([m * 1e3 / 4 for m in ms])  # 4 steps per pass, microseconds
    assert sp["median"] == 750.0 and sp["samples"] == 5
    assert sp["p10"] == 350.0 and sp["p90"] == 1150.0


def test_cold_blocks_subtract_the_read_per_block():
    """Each block's work time is its [read, work] mean less the next block of
    the read alone; the mean and the percentiles are over the blocks."""
    work = iter([0.050, 0.052, 0.051, 0.060])
    flush = iter([0.040, 0.041, 0.040, 0.040])
    mean, sp = bench.cold_blocks_us(lambda: next(work), lambda: next(flush), 4)
    diffs = [10.0, 11.0, 11.0, 20.0]
    assert abs(mean - sum(diffs) / 4) < 1e-9
    assert sp["samples"] == 4 and abs(sp["median"] - 11.0) < 1e-9
    assert sp["p10"] <= sp["median"] <= sp["p90"]
    neg, _ = bench.cold_blocks_us(lambda: 0.039, lambda: 0.040, 3)
    assert neg == 0.0
