"""Host-side logic of bench.py that the JSON line rests on: how the end-to-end
step splits the batch, which kernels count as the backward, and how DRAM
traffic captures are keyed by the sources they ran on (so that a capture of
older sources is never reported as current)."""
import json
import os
import shutil

import pytest

import bench


def test_end_to_end_chunks_partition_the_batch():
    assert bench.e2e_chunk_sizes(8) == [2, 2, 2, 2]
    assert bench.e2e_chunk_sizes(64) == [16, 16, 16, 16]
    assert bench.e2e_chunk_sizes(4) == [2, 2]
    assert bench.e2e_chunk_sizes(2) == [1, 1]
    assert bench.e2e_chunk_sizes(3) == [3]
    assert bench.e2e_chunk_sizes(1) == [1]
    assert bench.e2e_chunk_sizes(4, "1,3") == [1, 3]
    for spec in ("2,3", "0,4", "5"):
        with pytest.raises(ValueError):
            bench.e2e_chunk_sizes(4, spec)


def test_backward_time_of_both_kernel_layouts():
    assert bench.backward_ms({"fwd": 0.2, "bwd": 0.5, "dq_finish": 0.03}) == 0.5
    assert bench.backward_ms({"fwd": 0.6, "bwd_kv": 0.9, "bwd_q": 0.65}) == pytest.approx(1.55)
    assert bench.backward_ms({"fwd": 0.4}) is None


def _ncu_csv(path):
    # two launches of each tensor-core kernel, units as ncu prints them
    rows = [
        ("1", "void saf::fwd_tc_kernel(saf::FwdParams)", "dram__bytes_read.sum", "Mbyte", "100"),
        ("1", "void saf::fwd_tc_kernel(saf::FwdParams)", "dram__bytes_write.sum", "Mbyte", "50"),
        ("2", "void saf::fwd_tc_kernel(saf::FwdParams)", "dram__bytes_read.sum", "Mbyte", "110"),
        ("2", "void saf::fwd_tc_kernel(saf::FwdParams)", "dram__bytes_write.sum", "Kbyte", "40,000"),
        ("3", "void saf::bwd_tc_kernel<false>(saf::BwdParams)", "dram__bytes_read.sum", "Gbyte", "0.25"),
        ("3", "void saf::bwd_tc_kernel<false>(saf::BwdParams)", "dram__bytes_write.sum", "Mbyte", "125"),
        ("4", "void saf::call_init_kernel(...)", "dram__bytes_read.sum", "Kbyte", "7"),
    ]
    with open(path, "w") as f:
        f.write("==PROF== a line ncu prints that is not CSV\n")
        f.write('"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"\n')
        for r in rows:
            f.write(",".join(f'"{c}"' for c in r) + "\n")


def test_traffic_records_are_keyed_by_the_current_sources(tmp_path):
    csv_path, out = str(tmp_path / "t.csv"), str(tmp_path / "traffic.json")
    _ncu_csv(csv_path)
    # an entry of sources that no longer exist is dropped when new captures are stored
    with open(out, "w") as f:
        json.dump({"bwd|w|000000000000": 1.0}, f)
    assert bench.record_traffic(csv_path, "w", out) == 0
    tt = json.load(open(out))
    assert tt == {f"fwd|w|{bench._src_hash('fwd')}": pytest.approx((150e6 + 150e6) / 2),
                  f"bwd|w|{bench._src_hash('bwd')}": pytest.approx(375e6)}


def test_a_source_change_changes_the_key(tmp_path, monkeypatch):
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "softmax_attention_hybrid_gb300", "csrc"),
                    root / "softmax_attention_hybrid_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "include"), root / "include")
    monkeypatch.setattr(bench, "ROOT", str(root))
    before = {k: bench._src_hash(k) for k in ("fwd", "bwd", None)}
    p = root / "softmax_attention_hybrid_gb300" / "csrc" / "bwd_tc.cu"
    p.write_text(p.read_text() + "\n// edited\n")
    assert bench._src_hash("bwd") != before["bwd"]
    assert bench._src_hash("fwd") == before["fwd"]   # not among the forward's sources
    assert bench._src_hash() != before[None]
