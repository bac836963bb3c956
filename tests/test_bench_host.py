"""Host-side logic of bench.py that needs no GPU: the oracle's CPU rate and the
gate that drops committed ncu traffic once its kernel sources have changed."""

from __future__ import annotations

import hashlib
import os

import bench


def test_cpu_oracle_rate_all_and_one_thread():
    gbs, sps, done, k, threads = bench.cpu_oracle_rate(1, budget_s=0.2)
    assert gbs > 0 and sps > 0 and done >= 1 and k == 4 and threads >= 1
    gbs1, sps1, done1, _, threads1 = bench.cpu_oracle_rate(1, budget_s=0.2, threads=1)
    assert gbs1 > 0 and sps1 > 0 and done1 >= 1 and threads1 == 1


def _write_profile(tmp_path, srcs, shas, value="123456"):
    prof = tmp_path / "profiles"
    prof.mkdir(exist_ok=True)
    (prof / "t.traffic.txt").write_text(
        "# comment: source_sha256 lines in comments are ignored\n"
        f"source: {','.join(srcs)}\nsource_sha256: {','.join(shas)}\n"
        f"dram_bytes_per_launch: {value}\n")


def test_profile_traffic_follows_source_hashes(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_cache_287_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cuh").write_bytes(b"kernel a\n")
    (csrc / "b.cuh").write_bytes(b"kernel b\n")
    sha = lambda p: hashlib.sha256(p.read_bytes()).hexdigest()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))

    _write_profile(tmp_path, ["a.cuh", "b.cuh"], [sha(csrc / "a.cuh"), sha(csrc / "b.cuh")])
    assert bench.profile_traffic("t.traffic.txt") == 123456.0

    (csrc / "b.cuh").write_bytes(b"kernel b, changed\n")  # one source changed: no traffic
    assert bench.profile_traffic("t.traffic.txt") is None

    _write_profile(tmp_path, ["a.cuh", "b.cuh"], [sha(csrc / "a.cuh")])  # count mismatch
    assert bench.profile_traffic("t.traffic.txt") is None
    _write_profile(tmp_path, ["gone.cuh"], ["0" * 64])  # missing source
    assert bench.profile_traffic("t.traffic.txt") is None
    assert bench.profile_traffic("absent.traffic.txt") is None


def test_committed_profiles_match_current_sources():
    """Every committed traffic file names sources that exist; those whose hashes
    match give a positive byte count (a stale one is simply reported as null)."""
    prof = os.path.join(bench.ROOT, "profiles")
    names = [f for f in os.listdir(prof) if f.endswith(".traffic.txt")]
    assert names
    for name in names:
        fields = {}
        with open(os.path.join(prof, name)) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        for src in fields["source"].split(","):
            assert os.path.exists(os.path.join(bench.ROOT, "paged_kv_cache_287_gb300", "csrc",
                                               src.strip())), (name, src)
        t = bench.profile_traffic(name)
        assert t is None or t > 0
