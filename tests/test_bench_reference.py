"""The benchmark's reference arm (the oracle on the host cores) keeps the JSON contract, and
ranks other than 0 exit without work."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "1"], capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"].startswith("MoE-layer tokens/s") and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 1 and d["n_gpus"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("decode T=1")


def test_reference_arm_other_ranks_exit_without_work():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_traffic_record_from_ncu_raw_page(tmp_path, monkeypatch):
    """--record-traffic: mean DRAM bytes over the matching launches of ncu's raw page (header
    row, units row, one row per launch), stamped with the digest of the decode FFN sources;
    the bench reads it back only while that digest still matches."""
    import bench
    raw = tmp_path / "raw.csv"
    raw.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
                   '"","","byte","byte"\n'
                   '"0","void fp4moe::route_decode_kernel<1, 12>(RouteArgs)","4000000","1000"\n'
                   '"1","void fp4moe::mxf4_decode_kernel<8>(fp4moe::DecParams)","113000000","2000000"\n'
                   '"2","void fp4moe::mxf4_decode_kernel<8>(fp4moe::DecParams)","113200000","2200000"\n')
    out = tmp_path / "rec.json"
    monkeypatch.setattr(bench, "ROOT", str(bench.ROOT))
    rec = bench.record_traffic(str(raw), bench.FFN_KERNEL, str(out), "ncu ...")
    assert rec["launches"] == 2 and rec["dram_bytes_per_launch"] == 115200000
    assert rec["digest"] == bench.sources_digest(bench.FFN_SOURCES)
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(out))
    assert bench.ffn_traffic() == 115200000
    rec["digest"] = "0" * 16
    out.write_text(json.dumps(rec))
    assert bench.ffn_traffic() is None
