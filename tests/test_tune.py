"""Host logic of the offline tuner: choosing the best variant per size bucket
and rendering the table, without a GPU."""
from symmetric_matrix_vector_gb300 import tune


def rec(kind, uplo, n, variant, name, ms):
    return {"kind": kind, "uplo": uplo, "n": n, "variant": variant, "variant_name": name,
            "ms": ms, "gbs": 1.0}


def test_choose_picks_fastest_and_buckets():
    done = {}
    for r in (rec("s", "U", 4096, 0, "a", 2.0), rec("s", "U", 4096, 1, "b", 1.0),
              rec("s", "U", 8192, 0, "a", 3.0), rec("s", "U", 8192, 1, "b", 4.0)):
        done[(r["kind"], r["uplo"], r["n"], r["variant_name"])] = r
    e = tune.choose(done)
    assert [(k, u, nmax, r["variant"]) for k, u, nmax, r in e] == [
        ("s", 1, (4096 + 8192) // 2, 1), ("s", 1, tune.INT_MAX, 0)]


def test_choose_maps_names_to_current_indices():
    # results recorded against an older table: "gone" no longer exists and
    # "b" moved from index 1 to index 0
    done = {}
    for r in (rec("d", "L", 8192, 0, "gone", 0.5), rec("d", "L", 8192, 1, "b", 1.0),
              rec("d", "L", 8192, 2, "c", 1.5)):
        done[(r["kind"], r["uplo"], r["n"], r["variant_name"])] = r
    index_of = {("d", "b"): 0, ("d", "c"): 1}
    (entry,) = tune.choose(done, index_of)
    assert entry[3]["variant_name"] == "b" and entry[3]["variant"] == 0


def test_render_table_fills_missing_kinds():
    done = {("z", "U", 16384, "x"): rec("z", "U", 16384, 3, "x", 1.0)}
    text = tune.render_table(tune.choose(done))
    assert "{'z', 1, %d, \"x\"}" % tune.INT_MAX in text
    for k in "sdcw":
        assert "{'%s', -1, %d, \"\"}," % (k, tune.INT_MAX) in text


def test_choose_breaks_near_ties_by_back_to_back_time():
    done = {}
    for r in (dict(rec("s", "U", 8192, 0, "a", 1.000), ms_b2b=0.95),
              dict(rec("s", "U", 8192, 1, "b", 1.005), ms_b2b=0.80),
              dict(rec("s", "U", 8192, 2, "c", 1.100), ms_b2b=0.50)):
        done[(r["kind"], r["uplo"], r["n"], r["variant_name"])] = r
    (entry,) = tune.choose(done)
    assert entry[3]["variant_name"] == "b"      # c is fastest back to back but 10 % slower alone


def test_results_of_several_runs_are_averaged(tmp_path):
    import json

    path = tmp_path / "r.jsonl"
    rows = [rec("w", "L", 8192, 0, "a", 3.6), rec("w", "L", 8192, 1, "b", 3.7),
            rec("w", "L", 8192, 0, "a", 3.8), rec("w", "L", 8192, 1, "b", 3.7)]
    path.write_text("".join(json.dumps(r) + "\n" for r in rows))
    done = tune.load_results(str(path))
    assert abs(done[("w", "L", 8192, "a")]["ms"] - 3.7) < 1e-12
    assert done[("w", "L", 8192, "a")]["runs"] == 2


def test_choose_counts_sub_quarter_microsecond_gaps_as_ties():
    """small calls: 12.34 against 12.52 us is 1.5 % apart but under 0.25 us
    (below the event timer's resolution): back to back decides; 0.3 us
    apart is a real difference"""
    a = dict(rec("s", "L", 1024, 0, "one_launch", 0.01234), ms_b2b=0.0100)
    b = dict(rec("s", "L", 1024, 1, "two_kernels", 0.01252), ms_b2b=0.0045)
    best = tune.choose({("s", "L", 1024, r["variant_name"]): r for r in (a, b)})
    assert best[0][3]["variant_name"] == "two_kernels"
    c = dict(rec("s", "L", 1024, 1, "two_kernels", 0.01264), ms_b2b=0.0045)
    best = tune.choose({("s", "L", 1024, r["variant_name"]): r for r in (a, c)})
    assert best[0][3]["variant_name"] == "one_launch"


def test_one_launch_variant_counts_its_twin_back_to_back():
    """the library runs a one-launch variant's two-kernel twin for
    back-to-back calls, so the tie-break charges it the twin's time"""
    assert tune.twin_name("vr2_u2_r0_w8_b4_g12_c2_f") == ["vr2_u2_r0_w8_b4_g12_c2",
                                                          "vr2_u2_r0_w8_b4_g12"]
    assert tune.twin_name("vr4_u2_r0_w8_b0_g5_c8_f") == ["vr4_u2_r0_w8_b0_g5_c8"]
    assert tune.twin_name("vr4_u2_r0_w8_b0_g5_c8") is None
    one = dict(rec("s", "L", 1024, 0, "vr1_u2_r0_w8_b6_g11_c2_f", 0.01234), ms_b2b=0.0100)
    twin = dict(rec("s", "L", 1024, 1, "vr1_u2_r0_w8_b6_g11", 0.01270), ms_b2b=0.0044)
    other = dict(rec("s", "L", 1024, 2, "vr1_u2_r0_w8_b0_g9", 0.01252), ms_b2b=0.0045)
    done = {("s", "L", 1024, r["variant_name"]): r for r in (one, twin, other)}
    (entry,) = tune.choose(done)
    assert entry[3]["variant_name"] == "vr1_u2_r0_w8_b6_g11_c2_f"
    assert one["ms_b2b"] == 0.0100          # the caller's records are not changed
