"""Offline tuner: times every compiled kernel variant on the current GPU and
writes the per-(kind, uplo, n) choice into csrc/xsymv_tuned.h.

The report tunes (Tx, Ty, U) thread-block shapes offline and builds the best
kernels into its library, with an if-then table over n per GPU
("CUDA-xSYMV の実装と評価", §3 and Tables I, 2, 3).  The GB300 kernels'
parameter space is the variant list compiled into libxsymv.so (vectors per
lane, columns in flight, shared-memory ring depth, warps per block); this
script measures each one with CUDA events on synthetic problems and keeps the
fastest per size.

Results are appended to a JSONL file (one line per measurement) and reused on
a rerun, so an interrupted sweep resumes where it stopped.

    python -m symmetric_matrix_vector_gb300.tune --kinds s --n 8192,16384,32768 \\
        --results /tmp/tune.jsonl --write-header /tmp/xsymv_tuned.h
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import time

from . import _build, inputs

# the sizes each kind is tuned at: the small, L2-resident sizes (triangles of
# at most a few tens of MB) separately from the HBM-bound ones
DEFAULT_N = {"s": [512, 1024, 2048, 3072, 4096, 8192, 12288, 16384, 20480, 24576, 28672, 32768],
             "d": [1024, 2048, 4096, 8192, 16384, 24576], "c": [1024, 2048, 4096, 8192, 16384],
             "z": [1024, 2048, 4096, 8192, 16384], "w": [1024, 2048, 4096, 8192]}
TUNED_H = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc", "xsymv_tuned.h")
INT_MAX = 2147483647
L2_BYTES = 129e6          # GB300's L2
COLD_BELOW = 4 * L2_BYTES  # smaller stored triangles are timed with L2 flushed before each call


def trimmed_mean(values, cut=0.1):
    """mean of the values without the lowest and highest `cut` fraction.
    CUDA event times are quantised (on GB300 to about 2 us); over many calls
    the quantum's phase varies, so a mean resolves what a median cannot."""
    v = sorted(values)
    k = int(len(v) * cut)
    v = v[k:len(v) - k] or v
    return sum(v) / len(v)


def measure(xs, kind, uplo, n, variant, reps, prob, cold=False):
    """ms of one call.  Back-to-back calls (median of three runs), or, with
    cold=True, each call after writing a 512 MB buffer and reading another
    (nothing of the problem left in L2, and no dirty lines left to write back
    during the call; the trimmed mean of many such calls) -- the protocol the
    benchmark uses for triangles near L2's size."""
    import torch

    assert xs.xsymv_set_variant(kind, variant) == 0
    try:
        A, x, y, lda = prob["A"], prob["x"], prob["y"], prob["lda"]
        alpha = prob["alpha"]
        beta = prob["beta"]
        for _ in range(3):
            xs.check(xs.symv(kind, uplo, n, alpha, A, lda, x, 1, beta, y, 1))
        torch.cuda.synchronize()
        if cold:
            flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
            clean = torch.zeros(64 << 20, dtype=torch.int64, device="cuda")
            evs = []
            for _ in range(max(60, min(reps, 120))):
                flush.fill_(1)
                clean.sum()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record()
                xs.check(xs.symv(kind, uplo, n, alpha, A, lda, x, 1, beta, y, 1))
                e1.record()
                evs.append((e0, e1))
            torch.cuda.synchronize()
            return trimmed_mean([a.elapsed_time(b) for a, b in evs])
        def call():
            xs.check(xs.symv(kind, uplo, n, alpha, A, lda, x, 1, beta, y, 1))

        # the host's cost of enqueueing `reps` calls: the GPU spins at least
        # that long first, so that the calls run back to back on the GPU and
        # the events time the GPU, not the host's rate of issuing calls
        t0 = time.perf_counter()
        for _ in range(10):
            call()
        host_s = (time.perf_counter() - t0) / 10 * reps
        torch.cuda.synchronize()
        times = []
        for _ in range(3):
            torch.cuda._sleep(int((1.5 * host_s + 2e-4) * 2.07e9))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                call()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) / reps)
        return statistics.median(times)
    finally:
        xs.xsymv_set_variant(kind, -1)


def load_results(path):
    """(kind, uplo, n, variant name) -> record.  A file may hold several
    measurements of one key (runs on different GPUs of the same model,
    appended one after another): their times are averaged, so that the
    choice does not follow one GPU's quirks."""
    groups = {}
    if path and os.path.exists(path):
        with open(path) as f:
            for line in f:
                try:
                    r = json.loads(line)
                except ValueError:
                    continue
                groups.setdefault((r["kind"], r["uplo"], r["n"], r["variant_name"]), []).append(r)
    done = {}
    for key, rs in groups.items():
        r = dict(rs[-1])
        r["ms"] = sum(x["ms"] for x in rs) / len(rs)
        b2b = [x["ms_b2b"] for x in rs if "ms_b2b" in x]
        if b2b:
            r["ms_b2b"] = sum(b2b) / len(b2b)
        r["runs"] = len(rs)
        tri = r["gbs"] * rs[-1]["ms"]   # stored bytes / 1e6, from the record's own figures
        r["gbs"] = tri / r["ms"]
        done[key] = r
    return done


def sweep(kinds, sizes, uplos, results_path, reps_bytes=8e9, only=None):
    import torch

    import symmetric_matrix_vector_gb300 as xs

    _build.build()
    xs.load()
    done = load_results(results_path)
    out = open(results_path, "a") if results_path else None
    es = inputs.ELEM_BYTES
    for kind in kinds:
        for uplo in uplos:
            for n in sizes.get(kind, DEFAULT_N[kind]):
                prob = None
                for v in range(xs.xsymv_variant_count(kind)):
                    name = xs.xsymv_variant_name(kind, v)
                    if only and name not in only:
                        continue
                    if (kind, uplo, n, name) in done:
                        continue
                    if prob is None:
                        al = {"s": 1.0, "d": 1.0, "c": 1.0, "z": 1.0, "w": (1.0, 0.0)}[kind]
                        be = {"s": 0.0, "d": 0.0, "c": 0.0, "z": 0.0, "w": (0.0, 0.0)}[kind]
                        prob = inputs.device_problem(kind, uplo, n, lda=n, alpha=al, beta=be,
                                                     seed=n)
                    tri = n * (n + 1) / 2 * es[kind]
                    reps = int(max(5, min(500, reps_bytes / tri)))
                    cold = tri < COLD_BELOW
                    ms = measure(xs, kind, uplo, n, v, reps, prob, cold=cold)
                    rec = {"kind": kind, "uplo": uplo, "n": n, "variant": v, "variant_name": name,
                           "ms": ms, "gbs": tri / (ms * 1e-3) / 1e9,
                           "l2": "flushed" if cold else "back-to-back",
                           "gpu": torch.cuda.get_device_name()}
                    if cold:   # the same calls back to back too, for the tie-break in choose()
                        rec["ms_b2b"] = measure(xs, kind, uplo, n, v, max(reps, 100), prob)
                    done[(kind, uplo, n, name)] = rec
                    if out:
                        out.write(json.dumps(rec) + "\n")
                        out.flush()
                    print("%s %s n=%6d %-16s %8.4f ms %8.1f GB/s" % (kind, uplo, n, name, ms,
                                                                     rec["gbs"]), flush=True)
                del prob
                torch.cuda.empty_cache()
    if out:
        out.close()
    return done


TIE = 0.01        # variants within 1 % of the fastest isolated call count as equal,
TIE_MS = 0.00025  # or within 0.25 us of it: an eighth of the event timer's ~2 us tick,
                  # about the spread of a trimmed mean of 60 flushed calls


def twin_name(name):
    """the two-kernel twin of a one-launch variant name ("..._f"): the name
    without "_f", and without "_c<R>" when R is U (the default); the
    library runs it for back-to-back calls.  None for other names."""
    if not name.endswith("_f"):
        return None
    base = name[:-2]
    m = re.match(r"vr\d+_u(\d+)_.*_c(\d+)$", base)
    if m and m.group(1) == m.group(2):
        return [base, base[: base.rindex("_c")]]
    return [base]


def choose(done, index_of=None):
    """best variant per (kind, uplo, n) -> table entries with n_max buckets.

    The fastest call decides (an isolated call with the L2 flushed for the
    small triangles, back to back for the large ones); among small-triangle
    variants within TIE (relative) or TIE_MS (absolute) of the fastest, the
    one fastest back to back wins, a one-launch variant counting its
    two-kernel twin's time there (the library runs the twin back to back).

    ``index_of`` maps (kind, variant name) to the variant's index in the
    library being tuned; results for names it does not know (variants since
    removed) are skipped and the indices come from it, not from the results
    file, whose indices may belong to an older variant table."""
    groups = {}
    for (kind, uplo, n, name), r in done.items():
        if index_of is not None:
            if (kind, name) not in index_of:
                continue
            r = dict(r, variant=index_of[(kind, name)])
        groups.setdefault((kind, uplo, n), []).append(r)
    best = {}
    for key, rs in groups.items():
        # back to back, a one-launch variant runs as its two-kernel twin
        by_name = {r["variant_name"]: r for r in rs}

        def effective(r):
            for t in twin_name(r["variant_name"]) or []:
                tr = by_name.get(t)
                if tr is not None and "ms_b2b" in tr and "ms_b2b" in r:
                    return dict(r, ms_b2b=min(r["ms_b2b"], tr["ms_b2b"]))
            return r

        rs = [effective(r) for r in rs]
        fastest = min(r["ms"] for r in rs)
        near = [r for r in rs if r["ms"] <= max(fastest * (1 + TIE), fastest + TIE_MS)]
        if all("ms_b2b" in r for r in near):
            best[key] = min(near, key=lambda r: (r["ms_b2b"], r["ms"]))
        else:
            best[key] = min(rs, key=lambda r: r["ms"])
    entries = []
    for kind in "sdczw":
        for uplo in ("U", "L"):
            ns = sorted(n for (k, u, n) in best if k == kind and u == uplo)
            for i, n in enumerate(ns):
                n_max = INT_MAX if i + 1 == len(ns) else (n + ns[i + 1]) // 2
                entries.append((kind, 1 if uplo == "U" else 0, n_max, best[(kind, uplo, n)]))
    return entries


def render_table(entries, kinds_all="sdczw"):
    lines = ["static const TunedEntry kTuned[] = {"]
    have = set()
    for kind, upper, n_max, r in entries:
        have.add(kind)
        lines.append("    {'%s', %d, %d, \"%s\"},   // %.1f GB/s at n=%d" % (
            kind, upper, n_max, r["variant_name"], r["gbs"], r["n"]))
    for kind in kinds_all:
        if kind not in have:
            lines.append("    {'%s', -1, %d, \"\"},   // not tuned: variant 0" % (kind, INT_MAX))
    lines.append("};")
    return "\n".join(lines)


def write_header(entries, path):
    with open(TUNED_H) as f:
        src = f.read()
    table = render_table(entries)
    new = re.sub(r"// BEGIN TUNED TABLE\n.*?// END TUNED TABLE",
                 "// BEGIN TUNED TABLE\n" + table + "\n// END TUNED TABLE", src, flags=re.S)
    with open(path, "w") as f:
        f.write(new)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kinds", default="s")
    ap.add_argument("--n", default="", help="comma-separated sizes (default: per kind)")
    ap.add_argument("--uplo", default="U,L")
    ap.add_argument("--results", default="tune_results.jsonl")
    ap.add_argument("--write-header", default="", help="write the tuned header here")
    ap.add_argument("--variants", default="",
                    help="comma-separated variant names: time only these (default: all)")
    args = ap.parse_args()
    kinds = [k for k in args.kinds.split(",") if k]
    sizes = {}
    if args.n:
        ns = [int(v) for v in args.n.split(",")]
        sizes = {k: ns for k in kinds}
    only = set(v for v in args.variants.split(",") if v)
    done = sweep(kinds, sizes, args.uplo.split(","), args.results, only=only or None)
    if args.write_header:
        import symmetric_matrix_vector_gb300 as xs

        index_of = {(k, xs.xsymv_variant_name(k, i)): i
                    for k in "sdczw" for i in range(xs.xsymv_variant_count(k))}
        write_header(choose(done, index_of), args.write_header)
        print("wrote", args.write_header)


if __name__ == "__main__":
    main()
