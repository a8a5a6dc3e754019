"""bench.py's `roofline.traffic`: the DRAM bytes per launch come from the
committed ncu summary only while the kernel's sources hash as when the
counters were taken, and only on the workload they were taken on (the bytes
of a launch depend on its parameters); otherwise the field is null."""
import hashlib
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _tree(tmp_path, sources):
    csrc = tmp_path / "long_context_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name, text in sources.items():
        (csrc / name).write_bytes(text)
    (tmp_path / "profiles").mkdir()
    return csrc


def _sha(csrc, files):
    return hashlib.sha1(b"".join((csrc / f).read_bytes() for f in files)).hexdigest()[:12]


def _args(**kw):
    a = dict(workload=bench.TRAFFIC_WORKLOAD, cand_bp=None, rho=None, topk=None, topk_order="score")
    a.update(kw)
    return types.SimpleNamespace(**a)


def test_traffic_follows_the_source_hash_and_the_workload(tmp_path, monkeypatch):
    files = {f: f"// {f}\n".encode() for fs in bench.TRAFFIC_SOURCES.values() for f in fs}
    csrc = _tree(tmp_path, files)
    h_dec = _sha(csrc, bench.TRAFFIC_SOURCES["decode"])
    h_den = _sha(csrc, bench.TRAFFIC_SOURCES["dense"])
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        f"# comment line\ndecode {h_dec} 48790272\ndense {h_den} 540388864\ndecode 000000000000 1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_record("decode", _args()) == 48790272.0
    assert bench.traffic_record("dense", _args()) == 540388864.0
    # another workload, or the same workload at other parameters: no record
    assert bench.traffic_record("decode", _args(workload="1m-hbm")) is None
    assert bench.traffic_record("decode", _args(topk=2048)) is None
    assert bench.traffic_record("decode", _args(topk_order="position")) is None
    assert bench.traffic_record("attend", _args()) is None
    # a changed header shared by both kernels voids both records
    (csrc / "paris_device.cuh").write_bytes(b"// changed\n")
    assert bench.traffic_record("decode", _args()) is None
    assert bench.traffic_record("dense", _args()) is None


def test_committed_records_name_every_kernel_once():
    seen = {}
    for line in open(os.path.join(ROOT, "profiles", "dram_traffic.txt")):
        if line.startswith("#") or not line.strip():
            continue
        kernel, sha, nbytes = line.split()
        assert kernel in bench.TRAFFIC_SOURCES and len(sha) == 12 and float(nbytes) > 0
        seen[kernel] = seen.get(kernel, 0) + 1
    assert seen == {k: 1 for k in bench.TRAFFIC_SOURCES}
