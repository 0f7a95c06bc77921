"""The committed ncu summaries: well-formed traffic records, and every ncu command leaves the clocks alone."""
import json
import re
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
PROFILES = ROOT / "profiles"


def test_traffic_records_are_consistent():
    recs = sorted(PROFILES.glob("*.traffic.json"))
    assert recs
    for f in recs:
        rec = json.loads(f.read_text())
        for key in ("kernel", "workload", "dram_bytes_per_launch", "algorithmic_bytes_per_launch",
                    "dram_bytes_per_algorithmic_byte", "kernel_source_sha256", "command"):
            assert key in rec, (f.name, key)
        ratio = rec["dram_bytes_per_launch"] / rec["algorithmic_bytes_per_launch"]
        assert abs(ratio - rec["dram_bytes_per_algorithmic_byte"]) < 1e-4, f.name
        assert re.fullmatch(r"[0-9a-f]{64}", rec["kernel_source_sha256"]), f.name
        assert rec["command"].startswith("ncu ") and "--clock-control none" in rec["command"], f.name


def test_ncu_commands_in_summaries_keep_clocks():
    for f in sorted(PROFILES.glob("*.md")):
        text = f.read_text()
        # join continuation lines, then look at every command that starts with ncu
        text = re.sub(r"\\\n\s*", " ", text)
        for line in text.splitlines():
            cmd = line.strip().lstrip("`")
            if cmd.startswith("ncu ") and " -i " not in cmd:
                assert "--clock-control none" in cmd, (f.name, cmd)


def test_traffic_scales_with_algorithmic_bytes(tmp_path, monkeypatch):
    import bench
    rec = json.loads((PROFILES / "paged_prefill_prefill30k.traffic.json").read_text())
    monkeypatch.setattr(bench, "ROOT", tmp_path)
    (tmp_path / "profiles").mkdir()
    csrc = tmp_path / "paged_kv_cache_258_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for i, name in enumerate(bench.PREFILL_SOURCES):
        (csrc / name).write_text(f"// {name}\nint v{i} = {i};  /* a value */\n")
    rec["kernel_source_sha256"] = bench.kernel_source_hash(bench.PREFILL_SOURCES)
    (tmp_path / "profiles" / "t.json").write_text(json.dumps(rec))
    got = bench.traffic_per_launch("x", 1.0e8, "t.json", bench.PREFILL_SOURCES)
    assert got == int(rec["dram_bytes_per_algorithmic_byte"] * 1.0e8)
    # a comment or layout edit keeps the record; a code edit voids it
    (csrc / bench.PREFILL_SOURCES[0]).write_text("// reworded\nint   v0 =\n 0; // a value\n")
    assert bench.traffic_per_launch("x", 1.0e8, "t.json", bench.PREFILL_SOURCES) == got
    (csrc / bench.PREFILL_SOURCES[0]).write_text("int v0 = 1;\n")
    assert bench.traffic_per_launch("x", 1.0e8, "t.json", bench.PREFILL_SOURCES) is None
    (csrc / bench.PREFILL_SOURCES[0]).write_text('int v0 = 0; const char* s = "// kept";\n')
    assert bench.traffic_per_launch("x", 1.0e8, "t.json", bench.PREFILL_SOURCES) is None
