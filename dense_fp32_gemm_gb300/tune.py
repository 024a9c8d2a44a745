"""Per-shape-class autotuner: tile configuration x persistent-schedule policy.

The pages tune one problem (M = N = K = 4096) over sixteen hand-picked
tuples and keep the fastest ("Autotuning: Searching the Tile-Shape Space",
sections "What The Sweep Found" and "What Could Be Improved"). Here:

1. the candidates are generated (configgen.py: every legal tuple of a bounded
   space, pruned by measured rules, the best two per tile shape);
2. a separate library of all candidates is built (``_lib_cand/``, row-major
   operands only) and loaded instead of the product library;
3. stage 1 times every candidate on every representative shape of a class
   with the default schedule policy and keeps the best few;
4. stage 2 times those few under every schedule policy of ``POLICIES``
   (hybrid stream-K, hybrid with only the last wave split, whole tiles,
   stream-K, split-K; raster group heights; split thresholds);
5. the winner of a class is the (configuration, policy) with the least
   geometric mean, over the class's shapes, of its time over the best time
   seen for that shape; a pair with the default policy within NOISE of that
   score is preferred (the policies differ by less than run-to-run noise on
   most classes, and the default is the one every other call path shares).

It writes

  * ``csrc/configs.inc``     -- the configurations the product library
    compiles: each class winner (built for every operand layout) plus the
    pages' own sweep winner (a reference point, row-major only);
  * ``csrc/tuned_table.inc`` -- class -> (configuration, policy);
  * ``tuned_table.json``     -- every timing behind the choice, with the GPU.

Run on the GPU (then rebuild the product library):

    python -m dense_fp32_gemm_gb300.tune --search

``--run CLASS`` only runs the product library's choice (or ``--config ID``)
on the first shape of a class, repeatedly, so that a profiler can capture
the launch that backs a choice.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# (M, N, K, alpha, beta) per class; the first shape of a class is the one a
# profiler capture backs the choice with.
CLASS_SHAPES = {
    "square_large": [(4096, 4096, 4096, 0.5, 3.0), (8192, 8192, 2048, 1.0, 0.0),
                     (6144, 4096, 4096, 1.0, 1.0)],
    "square_mid": [(8191, 1000, 777, 1.25, -0.5), (2048, 2048, 2048, 1.0, 0.0),
                   (3072, 2048, 1536, 1.0, 1.0)],
    "square_small": [(1024, 1024, 1024, 1.0, 0.0), (1536, 768, 1024, 1.0, 1.0),
                     (2048, 1024, 768, 1.0, 0.0)],
    "k_dominant": [(1024, 1024, 16384, 1.0, 1.0), (512, 512, 8192, 1.0, 0.0),
                   (2048, 1024, 16384, 1.0, 0.0)],
    "skinny_n": [(16384, 64, 4096, 1.0, 1.0), (8192, 32, 8192, 1.0, 0.0),
                 (32768, 96, 2048, 1.0, 0.0)],
    "skinny_m": [(64, 16384, 4096, 1.0, 1.0), (32, 8192, 8192, 1.0, 0.0),
                 (96, 32768, 2048, 1.0, 0.0)],
    # the persistent kernel's tiny class starts above 2^25 (smaller row-major
    # problems go to the tiny kernel)
    "tiny": [(512, 512, 512, 1.0, 0.0), (384, 384, 384, 1.0, 0.0), (256, 512, 1024, 1.25, -0.5),
             (640, 640, 640, 1.0, 1.0)],
}
# Names as the C++ table spells the classes.
CLASS_TOKENS = {"square_large": "SquareLarge", "square_small": "SquareSmall",
                "k_dominant": "KDominant", "skinny_n": "SkinnyN", "skinny_m": "SkinnyM",
                "tiny": "Tiny", "square_mid": "SquareMid"}

H, HT, DP, SK, SPK = 0, 1, 2, 3, 4
DEFAULT_POLICY = (H, 8, 4, 1)
# (mode, raster group, min split units, splits)
POLICIES = [DEFAULT_POLICY, (H, 4, 4, 1), (H, 16, 4, 1), (H, 8, 2, 1), (H, 8, 8, 1),
            (HT, 8, 4, 1), (HT, 4, 4, 1), (HT, 16, 4, 1),
            (DP, 8, 4, 1), (DP, 4, 4, 1), (DP, 16, 4, 1),
            (SK, 8, 2, 1), (SK, 8, 4, 1), (SK, 8, 8, 1),
            (SPK, 8, 4, 2), (SPK, 8, 4, 3), (SPK, 8, 4, 4), (SPK, 8, 4, 6), (SPK, 8, 4, 8)]
# The pages' sweep winner on this kernel's pipeline (128 x 64 x 16, warp
# 64 x 32, WNITER 2, 4 x 4 patches, 128 threads), kept as a reference point.
PAGES_WINNER = (128, 64, 16, 64, 32, 2, 4, 4, 128, 3, 3, 4, 0)
CAND_DIR = os.path.join(HERE, "_lib_cand")
# Relative score margin within which the default policy is preferred.
NOISE = 0.005


def config_token(full_name: str) -> str:
    """The configuration's registry token (the part before any '_')."""
    return full_name.split("_", 1)[0]


def relative_scores(times):
    """times: {key: [ms per shape or None]} -> {key: geometric mean over the
    shapes of ms / (best ms of that shape)}; keys that failed on any shape
    are left out."""
    ok = {k: v for k, v in times.items() if v and all(x is not None for x in v)}
    if not ok:
        return {}
    n = len(next(iter(ok.values())))
    best = [min(v[i] for v in ok.values()) for i in range(n)]
    return {k: math.exp(sum(math.log(v[i] / best[i]) for i in range(n)) / n) for k, v in ok.items()}


def pick_best(times):
    """The key of least relative score (ties: the smaller key)."""
    sc = relative_scores(times)
    if not sc:
        raise RuntimeError("nothing ran")
    return min(sorted(sc), key=lambda k: sc[k])


def pick_with_default(times, default=DEFAULT_POLICY, noise=NOISE):
    """times: {(config, policy): [ms]} -> the best key, except that the best
    key with the default policy wins when its score is within `noise` of the
    overall best."""
    sc = relative_scores(times)
    if not sc:
        raise RuntimeError("nothing ran")
    best = min(sorted(sc), key=lambda k: sc[k])
    dflt = [k for k in sorted(sc) if k[1] == default and sc[k] <= sc[best] * (1.0 + noise)]
    return min(dflt, key=lambda k: sc[k]) if dflt else best


def table_text(winners, gpu_name, sms):
    """winners: {class: (config name, policy tuple)}."""
    lines = ["// tuned_table.inc -- fastest tile configuration and schedule policy per shape class.",
             "// Generated by dense_fp32_gemm_gb300/tune.py on %s (%d SMs);" % (gpu_name, sms),
             "// the timings behind each row are in tuned_table.json.",
             "#define SGEMM_GB300_TUNED_TABLE(X) \\"]
    rows = []
    for c, tok in CLASS_TOKENS.items():
        name, pol = winners[c]
        rows.append(f"  X({tok}, {config_token(name)}, {pol[0]}, {pol[1]}, {pol[2]}, {pol[3]})")
    lines += [r + " \\" for r in rows[:-1]] + [rows[-1], ""]
    return "\n".join(lines)


def product_entries(winner_tuples, extras=(PAGES_WINNER,)):
    """The product configuration list: the winners (every layout, in first-win
    order) then the extras (row-major only) that are not winners."""
    seen, entries = set(), []
    for t in winner_tuples:
        if t not in seen:
            seen.add(t)
            entries.append((t, True))
    for t in extras:
        if t not in seen:
            seen.add(t)
            entries.append((t, False))
    return entries


def _inputs(M, N, K, seed):
    from dense_fp32_gemm_gb300.workloads import Workload, make_inputs
    w = Workload("tune", M, N, K, 1.0, 0.0, "uniform", seed)
    A, B, C = make_inputs(w)
    return A.cuda(), B.cuda(), C.cuda()


def time_call(cid, policy, shape, bufs, min_ms=30.0, min_reps=5):
    """Mean device time (ms) of one sgemm launch with configuration `cid`
    and schedule `policy` forced."""
    import torch
    from dense_fp32_gemm_gb300 import binding
    M, N, K, alpha, beta = shape
    dA, dB, dC = bufs
    s = torch.cuda.current_stream().cuda_stream
    assert binding.sgemm_force_config(cid) == 0
    assert binding.sgemm_force_schedule(policy) == 0
    try:
        def call():
            st = binding.sgemm(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                               dC.data_ptr(), N, s)
            if st != 0:
                raise binding.SgemmError(st, "sgemm")
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        one = max(e0.elapsed_time(e1), 1e-3)
        reps = max(min_reps, int(min_ms / one))
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize()
        st, detail = binding.sgemm_poll_device_status(s)
        if st != 0:
            raise binding.SgemmError(st, f"device status detail {detail}")
        return e0.elapsed_time(e1) / reps
    finally:
        binding.sgemm_force_config(-1)
        binding.sgemm_force_schedule(None)


def search_class(cls, names, measure, top=4, policies=POLICIES, log=print):
    """Two-stage search for one class. measure(si, cid, policy) -> ms (or
    raises). Returns (winner (cid, policy), stage-1 times {cid: [ms]},
    stage-2 times {(cid, policy): [ms]})."""
    shapes = CLASS_SHAPES[cls]

    def run(cid, pol):
        out = []
        for si in range(len(shapes)):
            try:
                out.append(measure(si, cid, pol))
            except Exception as e:  # a configuration that cannot run this shape
                log(f"{cls} {shapes[si][:3]} {names[cid]} {pol}: failed: {e}")
                out.append(None)
        return out
    stage1 = {cid: run(cid, DEFAULT_POLICY) for cid in range(len(names))}
    sc = relative_scores(stage1)
    best = sorted(sc, key=lambda c: (sc[c], c))[:top]
    for cid in best:
        log(f"{cls:13s} stage 1 {names[cid]:42s} {sc[cid]:.4f}")
    stage2 = {(cid, DEFAULT_POLICY): stage1[cid] for cid in best}
    for cid in best:
        for pol in policies:
            if (cid, pol) not in stage2:
                stage2[(cid, pol)] = run(cid, pol)
    win = pick_with_default(stage2)
    sc2 = relative_scores(stage2)
    log(f"{cls:13s} winner  {names[win[0]]:42s} policy {win[1]} score {sc2[win]:.4f} "
        f"(default policy {sc2.get((win[0], DEFAULT_POLICY), float('nan')):.4f})")
    return win, stage1, stage2


def build_candidates(out_dir=CAND_DIR):
    """A library of every candidate (row-major operands; the first candidate
    also for every layout, as the list's fallback) in out_dir; returns its
    path and the candidate tuples in registry order."""
    from dense_fp32_gemm_gb300 import build as cuda_build
    from dense_fp32_gemm_gb300 import configgen
    cands = configgen.candidates()
    fb = (128, 256, 32, 64, 64, 2, 4, 4, 256, 4, 1, 32, 2)
    if fb not in cands:
        cands = [fb] + cands
    entries = [(t, t == fb) for t in cands]
    os.makedirs(out_dir, exist_ok=True)
    inc = os.path.join(out_dir, "candidates.inc")
    configgen.write_configs_inc(entries, fb, "the tuner's candidate set.", path=inc)
    table = os.path.join(out_dir, "candidates_table.inc")
    name = configgen.config_name(fb)
    rows = [f"  X({tok}, {name}, 0, 8, 4, 1)" for tok in CLASS_TOKENS.values()]
    with open(table, "w") as f:
        f.write("#define SGEMM_GB300_TUNED_TABLE(X) \\\n" + " \\\n".join(rows) + "\n")
    path = cuda_build.build(config_list=inc, tuned_table=table, out_dir=out_dir)
    return path, cands


def search(out_dir=None, classes=None, top=4, log=print):
    """The whole search on the candidate library; writes the product list,
    the table and the timings (csrc/ and the package unless out_dir)."""
    lib_path, cands = build_candidates()
    os.environ["SGEMM_GB300_LIB"] = lib_path
    import torch
    from dense_fp32_gemm_gb300 import binding, configgen
    assert binding.library_path() == lib_path
    names = [binding.sgemm_config_info(i)[0] for i in range(binding.sgemm_config_count())]
    assert names == [configgen.config_name(t) for t in cands], "candidate registry order"
    props = torch.cuda.get_device_properties(0)
    classes = list(classes or CLASS_SHAPES)
    record = {"gpu": props.name, "sms": props.multi_processor_count,
              "when": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime()),
              "candidates": names, "policies": [list(p) for p in POLICIES],
              "shapes": {c: CLASS_SHAPES[c] for c in classes}, "stage1_ms": {}, "stage2_ms": {},
              "winners": {}}
    winners = {}
    for ci, cls in enumerate(classes):
        bufs = {}

        def measure(si, cid, pol):
            if si not in bufs:
                bufs.clear()
                torch.cuda.empty_cache()
                bufs[si] = _inputs(*CLASS_SHAPES[cls][si][:3], seed=100 + 10 * ci + si)
            return time_call(cid, pol, CLASS_SHAPES[cls][si], bufs[si])
        (cid, pol), st1, st2 = search_class(cls, names, measure, top=top, log=log)
        winners[cls] = (names[cid], pol)
        record["stage1_ms"][cls] = {names[c]: v for c, v in st1.items()}
        record["stage2_ms"][cls] = {f"{names[c]} {list(p)}": v for (c, p), v in st2.items()}
        record["winners"][cls] = {"config": names[cid], "policy": list(pol)}
        bufs.clear()
    csrc = out_dir or os.path.join(HERE, "csrc")
    json_path = os.path.join(out_dir or HERE, "tuned_table.json")
    with open(json_path, "w") as f:
        json.dump(record, f, indent=1)
    if set(classes) == set(CLASS_SHAPES):
        write_product(winners, csrc, props.name, props.multi_processor_count)
    return winners


def winners_from_record(record, noise=NOISE):
    """Re-derive {class: (config name, policy)} from a saved search record
    (tuned_table.json), with the current selection rule."""
    out = {}
    for cls, st2 in record["stage2_ms"].items():
        times = {}
        for key, v in st2.items():
            name, pol = key.split(" ", 1)
            times[(name, tuple(json.loads(pol)))] = v
        out[cls] = pick_with_default(times, noise=noise)
    return out


def write_product(winners, csrc, gpu_name, sms):
    """configs.inc and tuned_table.inc for {class: (config name, policy)}."""
    from dense_fp32_gemm_gb300 import configgen
    order = list(CLASS_TOKENS)
    tuples = [configgen.parse_name(winners[c][0]) for c in order]
    configgen.write_configs_inc(product_entries(tuples), tuples[0],
                                "each shape class's measured winner (tune.py) and the "
                                "pages' sweep winner.", path=os.path.join(csrc, "configs.inc"))
    with open(os.path.join(csrc, "tuned_table.inc"), "w") as f:
        f.write(table_text(winners, gpu_name, sms))


def run_one(cls, cid, reps):
    from dense_fp32_gemm_gb300 import binding
    shape = CLASS_SHAPES[cls][0]
    bufs = _inputs(*shape[:3], seed=100)
    st, pol = binding.sgemm_choose_policy(*shape[:3])
    for _ in range(reps):
        time_call(cid, pol, shape, bufs, min_ms=0.0, min_reps=1)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--search", action="store_true",
                    help="build the candidate library and search every class")
    ap.add_argument("--out-dir", default=None,
                    help="where configs.inc, tuned_table.inc/json go (default: csrc/ and the package)")
    ap.add_argument("--classes", default=None, help="comma-separated subset of classes")
    ap.add_argument("--top", type=int, default=4, help="configurations kept for stage 2")
    ap.add_argument("--from-json", default=None,
                    help="rewrite configs.inc and tuned_table.inc from a saved search record")
    ap.add_argument("--run", default=None, help="only run CLASS's first shape (for profiling)")
    ap.add_argument("--config", type=int, default=None)
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    if args.run:
        from dense_fp32_gemm_gb300 import binding
        cid = args.config if args.config is not None else binding.sgemm_choose_config(
            *CLASS_SHAPES[args.run][0][:3])[0]
        run_one(args.run, cid, args.reps)
        return
    if args.from_json:
        rec = json.load(open(args.from_json))
        winners = winners_from_record(rec)
        write_product(winners, args.out_dir or os.path.join(HERE, "csrc"), rec["gpu"], rec["sms"])
        print(json.dumps(winners, indent=1))
        return
    if args.search:
        classes = args.classes.split(",") if args.classes else None
        winners = search(args.out_dir, classes, top=args.top)
        print(json.dumps(winners, indent=1))
        return
    ap.print_help()


if __name__ == "__main__":
    main()
