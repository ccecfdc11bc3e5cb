"""Host-side helpers of bench.py (no GPU): the interleaved timing rounds and the
keys that tie a committed ncu summary to a kernel source and plan."""
import bench


def test_interleaved_alternates_order_and_averages():
    calls = []

    def fake_timer(fn, n, stream):
        calls.append((fn(), n))
        return {"a": 1.0, "b": 3.0}[calls[-1][0]] + len(calls) * 0.0

    arms = {"a": lambda: "a", "b": lambda: "b"}
    res = bench.interleaved(arms, 4, 7, None, timer=fake_timer)
    assert [c[0] for c in calls] == ["a", "b", "b", "a", "a", "b", "b", "a"]
    assert all(n == 7 for _, n in calls)
    assert res == {"a": 1.0, "b": 3.0}


def test_interleaved_sees_a_drift_equally():
    """A clock that slows every call by the same step affects both arms alike
    when the order alternates."""
    t = [0]

    def drifting(fn, n, stream):
        t[0] += 1
        return fn() + 0.1 * t[0]

    res = bench.interleaved({"x": lambda: 1.0, "y": lambda: 1.0}, 4, 1, None, timer=drifting)
    assert abs(res["x"] - res["y"]) < 1e-12


def test_plan_keys():
    assert bench.plan_key({"bm": 256, "bn": 256, "stages": 7, "grid": 152, "colgroup": 8,
                           "rowgroup": 2, "rank_order": 1, "reduce_mode": 0}) == \
        "bm=256 bn=256 colgroup=8 rowgroup=2 rank_order=1 reduce_mode=0"
    assert bench.plan_key({"grid": 152, "stages": 7, "slice_rows": 8, "slices": 64}) == \
        "grid=152 stages=7 slice_rows=8 slices=64"
    assert bench.kernel_name({"bm": 256}) == "gemm_rs_pair_kernel"
    assert bench.kernel_name({"bm": 128}) == "gemm_rs_fused_kernel"


def test_recorded_traffic_needs_a_matching_plan():
    plan = {"bm": 256, "bn": 256, "stages": 7, "grid": 152, "colgroup": 3, "rowgroup": 2,
            "rank_order": 1, "reduce_mode": 0}
    assert bench.recorded_traffic("gemm_rs_pair_kernel", "ffn_w8_m4096", plan) is None
    assert bench.recorded_traffic("gemm_rs_pair_kernel", "no_such_workload", plan) is None


def test_kernel_identity_ignores_comments_but_not_code():
    src = 'int f(int x) { // a comment\n  return x + 1; /* another */\n}\nconst char *s = "a // b";\n'
    edited_comment = src.replace("a comment", "edited")
    edited_code = src.replace("x + 1", "x + 2")
    assert bench.code_only(src) == bench.code_only(edited_comment)
    assert bench.code_only(src) != bench.code_only(edited_code)
    assert '"a // b"' in bench.code_only(src)          # a string literal is kept whole
    assert "comment" not in bench.code_only(src) and "another" not in bench.code_only(src)


def test_sustained_run_blocks_and_averages(monkeypatch):
    """The sustained region times blocks of about 0.2 s of calls until the
    requested wall time has passed, and reports their mean per call."""
    from tensor_gemm_reduce_tcgen05_gb300.inputs import WORKLOADS
    w = WORKLOADS["ffn_w8_m4096"]
    seen = []

    def fake_b2b(fn, n, stream):
        seen.append(n)
        return 0.5  # ms per call

    monkeypatch.setattr(bench, "time_loop_b2b", fake_b2b)
    res = bench.sustained_run(lambda: None, w, None, 0.02, False, None)
    assert seen[0] >= 1 and all(n == 400 for n in seen[1:])  # 0.2 s / 0.5 ms
    assert res["calls"] == 400 * (len(seen) - 1)
    assert abs(res["ms_per_call"] - 0.5) < 1e-12
    assert abs(res["tflops"] - w.flops / 0.5e-3 / 1e12) < 1e-6


def test_headline_profile_is_current():
    """The committed ncu summary of the default workload was taken on the
    current kernel source and the default plan, so the bench line reports its
    DRAM traffic (a stale summary would make it null)."""
    plan = {"bm": 256, "bn": 256, "stages": 7, "grid": 152, "colgroup": 32, "rowgroup": 4,
            "rank_order": 1, "reduce_mode": 0}
    t = bench.recorded_traffic("gemm_rs_pair_kernel", "ffn_w8_m8192_bias", plan)
    assert t is not None and 5e9 < t < 2e10
