"""Host-side logic of the benchmark: workload selection and the L2 statement of its JSON line."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def test_head_dim_option_changes_only_the_head_dimension():
    base = W.named("qwen3")
    a = bench.parse_args(["--workload", "qwen3", "--head-dim", "64"])
    w = bench.workload_of(a)
    assert w.head_dim == 64
    assert w == base.with_(head_dim=64)
    assert bench.workload_of(bench.parse_args([])) == W.named("fulldepth")  # the default headline workload
    cfg = bench.workload_config(w, a)
    assert "d=64" in cfg["workload"] and cfg["head_dim"] == 64


def test_l2_statement_follows_the_bytes_one_round_reads():
    for name, expect in (("qwen3", "1024 MiB"), ("tree", "2048 MiB"), ("fulldepth", "1024 MiB")):
        a = bench.parse_args(["--workload", name])
        l2 = bench.workload_config(bench.workload_of(a), a)["l2"]
        assert expect in l2 and "more than the 129 MB L2" in l2, (name, l2)
    a = bench.parse_args(["--workload", "tiny"])
    l2 = bench.workload_config(bench.workload_of(a), a)["l2"]
    assert "128 KiB" in l2 and "stays in" in l2
    a = bench.parse_args(["--workload", "qwen3", "--head-dim", "64"])
    assert "512 MiB" in bench.workload_config(bench.workload_of(a), a)["l2"]


def test_layers_option_keeps_every_launch_shape():
    w = bench.workload_of(bench.parse_args(["--layers", "2"]))
    assert w == W.named("fulldepth").with_(n_layers=2)
    cfg = bench.workload_config(w, bench.parse_args([]))
    assert cfg["n_layers"] == 2 and "2 layers x 2 requests" in cfg["workload"]


def test_copy_rates_skip_pushes_without_copies():
    import numpy as np
    iv = np.array([[0.0, 1.0, 1.0, 1.1], [np.nan, np.nan, 1.1, 1.5], [1.0, 3.0, 3.0, 3.1]])
    r = bench.copy_rates(iv, [200e6, 200e6, 200e6])
    assert r["pushes"] == 2 and abs(r["max"] - 200.0) < 1e-9 and abs(r["min"] - 100.0) < 1e-9
    assert r["below_150_frac"] == 0.5


def test_step_overlap_takes_the_union_of_transfers_inside_each_step():
    import numpy as np
    nan = np.nan
    # two steps of one layer with two pushes each; push 1 of step 0 is read in place (no copy interval)
    iv = np.array([[0.0, 2.0, 2.0, 2.5], [nan, nan, 2.5, 4.0],
                   [10.0, 12.0, 12.0, 12.4], [12.1, 14.0, 14.0, 14.3]])
    rounds = np.array([[-0.5, 4.0, 4.2], [9.8, 14.3, 14.5]])
    so = bench.step_overlap(iv, rounds, 1)
    assert len(so) == 2
    (t0, b0), (t1, b1) = so
    assert abs(t0 - 4.7) < 1e-9 and abs(b0 - 3.5) < 1e-9  # [0, 2] and the in-place kernel [2.5, 4]
    assert abs(t1 - 4.7) < 1e-9 and abs(b1 - 3.9) < 1e-9  # [10, 12] and [12.1, 14]
    # a step with a different number of intervals (an adaptive in-place round launched once) is cut by time
    iv2 = np.array([[0.0, 2.0, 2.0, 2.5], [nan, nan, 2.5, 4.0], [nan, nan, 10.2, 14.0]])
    (t0, b0), (t1, b1) = bench.step_overlap(iv2, rounds, 1)
    assert abs(b0 - 3.5) < 1e-9 and abs(b1 - 3.8) < 1e-9


def test_default_run_records_and_profiling_switches():
    a = bench.parse_args([])
    assert a.workload == "fulldepth" and a.method and a.draft_load
    assert [n for n in a.sub_workloads.split(",")] == ["tiny", "qwen3", "internlm", "tree"]
    assert set(a.tp_sub_workloads.split(",")) == {"qwen3", "internlm", "tree"}
    p = bench.parse_args(["--no-method", "--no-draft-load", "--sub-workloads="])
    assert not p.method and not p.draft_load and p.sub_workloads == ""


def test_code_digest_ignores_comments_only():
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        f1, f2, f3 = (os.path.join(d, n) for n in ("a.cu", "b.cu", "c.cu"))
        open(f1, "w").write("int x = 1;  // one\n\n// note\nint y = 2;\n")
        open(f2, "w").write("int x = 1;\nint y = 2;   // two\n")
        open(f3, "w").write("int x = 1;\nint y = 3;\n")
        assert bench.code_digest(f1) == bench.code_digest(f2)
        assert bench.code_digest(f1) != bench.code_digest(f3)


def test_committed_traffic_summary_matches_the_kernel_source():
    """The DRAM-traffic summary under profiles/ was taken on the chunk kernel as it is: the benchmark
    reports its figures as roofline.traffic only then."""
    for name, d in (("fulldepth", 128), ("qwen3", 128), ("internlm", 128), ("tree", 128), ("qwen3", 64),
                    ("internlm", 64), ("tree", 64)):
        t = bench.profiled_traffic(W.named(name).with_(head_dim=d))
        assert t is not None and t > 0, (name, d)
