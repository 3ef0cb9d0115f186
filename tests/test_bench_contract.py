"""bench.py's reference arm (the CPU oracle on a bounded sample of the
128K-context decode step): one JSON line with the contract's keys on rank 0,
nothing and exit status 0 on any other rank."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _oracle_built():
    from nvfp4_kv_cache_bd_gb300 import build
    build.build_oracle()


def run_bench(env_extra):
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env.update(env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                           "--warmup", "1"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = run_bench({})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "µs/step" and d["higher_is_better"] is False
    assert d["steps"] == 1 and d["warmup"] == 1 and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in d["config"] and "model" not in d["config"]


def test_reference_arm_is_silent_on_other_ranks():
    r = run_bench({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def test_traffic_record_hash_ignores_comments_and_whitespace():
    """The measured-traffic record follows the decode sources' code only:
    comments and whitespace runs leave the hash alone, anything else (string
    contents included) changes it."""
    sys.path.insert(0, ROOT)
    import bench
    code = 'int a = 1; /* block */ const char* s = "x // y";  // line\nfloat b;'
    assert bench.code_only(code) == 'int a = 1; const char* s = "x // y"; float b;'
    assert bench.code_only("a\n\n   b // c\n") == bench.code_only("a b")
    assert bench.code_only('s = "/* kept */";') == 's = "/* kept */";'
    assert bench.code_only("x = 1;") != bench.code_only("x = 2;")
    assert len(bench.decode_sources_hash()) == 16
