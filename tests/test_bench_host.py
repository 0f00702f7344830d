"""Host-side arithmetic of bench.py that its reported numbers rest on (CPU only)."""
import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_prefill_flop_count_matches_counting_pairs():
    b = _bench()
    H, d_c, d_h, d_r = 3, 8, 4, 2
    lengths, n_new = [5, 9, 4], [5, 3, 0]
    up, att = b.prefill_flop(lengths, n_new, H=H, d_c=d_c, d_h=d_h, d_r=d_r)
    # every cached row is up-projected to K_nope and V for every head
    assert up == sum(lengths) * 2 * d_c * 2 * H * d_h
    # every new token k of a sequence with L rows sees rows 0 .. L - n + k
    pairs = 0
    for L, n in zip(lengths, n_new):
        for k in range(n):
            pairs += len(range(0, L - n + k + 1))
    assert att == pairs * H * 2 * (d_h + d_r + d_h)


def test_committed_traffic_follows_the_source_digest():
    b = _bench()
    # a kernel with no committed figure, or a workload never captured, reports none
    assert b.committed_traffic("attend_tc", "no_such_workload") is None
    assert b.committed_traffic("no_such_kernel", "long_b4") is None


def test_cpu_baseline_times_both_oracle_forms():
    # the host-core baseline: the fp64 oracle's absorbed form, and beside it the explicit form
    import mla_synth as S
    b = _bench()
    inp = S.make_inputs(S.shape_with("dsv2_b16", batch=2, lengths=(70, 130)))
    r = b.cpu_baseline(inp, 0.3)
    assert r["kind"] == "oracle" and r["cores"] == (os.cpu_count() or 1)
    assert r["value"] > 0 and r["explicit"]["value"] > 0
    assert "absorbed" in r["sample"] and "explicit" in r["explicit"]["sample"]
