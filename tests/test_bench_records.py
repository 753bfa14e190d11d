"""Host-side pieces of bench.py that need no GPU: the recorded ncu traffic
(profiles/ncu_traffic.txt) and its lookup, and the varlen profiling
workload's guard."""
import argparse
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORKLOADS = {"llama8b_decode", "mixed_prefill_decode", "head_sweep_kv1", "head_sweep_kv8",
             "head_sweep_kv32", "long_context_decode", "tiny_gqa_decode",
             "cross_attention_decode", "cross_attention_prefill", "varlen_prefill_llama8b"}


def _load_bench():
    spec = importlib.util.spec_from_file_location("bench_records_under_test",
                                                  os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _records(path):
    out = []
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            out.append(dict(kv.split("=", 1) for kv in line.split()))
    return out


def test_traffic_records_are_well_formed():
    recs = _records(os.path.join(ROOT, "profiles", "ncu_traffic.txt"))
    assert recs, "no traffic record"
    seen = set()
    for r in recs:
        assert r["kernel"] in ("decode_kernel", "prefill_tc_kernel")
        assert r["workload"] in WORKLOADS
        assert len(r["source_sha"]) == 16 and int(r["source_sha"], 16) >= 0
        assert int(r["bytes_per_launch"]) == int(r["read"]) + int(r["write"]) > 0
        key = (r["kernel"], r["workload"])
        assert key not in seen, f"two records for {key}"
        seen.add(key)


def test_traffic_lookup_follows_the_source_hash(tmp_path, monkeypatch):
    bench = _load_bench()
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.txt").write_text(
        "# comment\n"
        "kernel=decode_kernel source_sha=00000000000000aa workload=llama8b_decode "
        "bytes_per_launch=30 read=20 write=10\n"
        "kernel=prefill_tc_kernel source_sha=00000000000000aa workload=llama8b_decode "
        "bytes_per_launch=99 read=90 write=9\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda src: "00000000000000aa")
    assert bench.ncu_traffic("decode_kernel", "decode.cu", "llama8b_decode") == 30.0
    assert bench.ncu_traffic("prefill_tc_kernel", "prefill_tc.cu", "llama8b_decode") == 99.0
    assert bench.ncu_traffic("decode_kernel", "decode.cu", "head_sweep_kv1") is None
    # a changed source (another hash) reports no traffic
    monkeypatch.setattr(bench, "kernel_source_sha", lambda src: "00000000000000bb")
    assert bench.ncu_traffic("decode_kernel", "decode.cu", "llama8b_decode") is None


def test_source_hash_covers_the_shared_headers(tmp_path, monkeypatch):
    bench = _load_bench()
    csrc = tmp_path / "mqa_paged_kv_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("decode.cu", "pa_common.cuh", "pa_kernels.cuh"):
        (csrc / name).write_text(name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha("decode.cu")
    (csrc / "pa_common.cuh").write_text("changed")
    assert bench.kernel_source_sha("decode.cu") != h0


def test_varlen_profiling_workload_has_no_reference_arm():
    bench = _load_bench()
    args = argparse.Namespace(workload="varlen_prefill_llama8b", impl="reference", seed=0,
                              steps=3, warmup=3)
    with pytest.raises(SystemExit):
        bench.run_varlen_only(args)
