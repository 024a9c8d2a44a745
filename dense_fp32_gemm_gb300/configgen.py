"""The tile-configuration space of the FFMA kernel: enumeration, legality,
pruning, and the generated configuration list the library is built from.

"Autotuning: Searching the Tile-Shape Space" sweeps sixteen hand-picked
tuples ("What The Sweep Found") and finds most of the space illegal ("Most
Configurations Are Not Wrong By A Little"). Here the space is generated:

1. enumerate every tuple (BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES,
   MINB, KU, ORDER) over bounded ranges (``SPACE``);
2. keep the legal ones: the kernel's own constexpr checker ``cfg_check`` in
   csrc/tile_config.hpp, compiled for the host with g++ (one source of truth:
   the kernel static_asserts the same function);
3. prune with the rules below, each backed by a measurement or by arithmetic;
4. rank what is left per tile shape and keep the best two (``candidates``).

The tuner (tune.py) builds a library of all candidates, times them per shape
class together with the schedule policies, and writes the winners back here
as ``csrc/configs.inc``: the X-macro list configs.hpp compiles. build.py
generates one translation unit per listed configuration from that list.

Pruning rules (a tuple must pass all):
  P1 TM = TN = 4: one float4 per fragment group; the FMA count per shared
     load depends only on the lane's rows x columns (WMITER*TM x WNITER*TN),
     so larger patches change the lane map, not the balance.
  P2 ORDER 2 (paired FMA, two rows of a column per instruction): halves the
     FMA instruction count; every paired configuration beat its scalar twin
     in the first sweep (tuned_table.json history: 2.02 vs 2.48 ms at 4096^3).
  P3 KU = BK (each k-slice one fully unrolled block), BK in {16, 24, 32}:
     full unrolling measured 1-5 % faster than KU 8 or 16; BK 48 lost every
     class and spills once unrolled beyond 16.
  P4 residency: MINB is the most CTAs per SM that shared memory and the
     register estimate allow, then STAGES the most (at most 5) that keep it.
  P5 at least 8 resident warps per SM (two per scheduler, to hide the
     paired FMA's dependent-issue latency).
  P6 at least 64 accumulators per lane (the pages' "at least four FMAs per
     shared load" balance, "Shared Memory Tiling", "What Could Be Improved").
Ranking per (BM, BN, BK): more accumulators, then a lane patch closest to
16 x 8 (the measured best), then the squarest warp tile, then more CTAs per
SM; the best two are candidates.
"""
from __future__ import annotations

import ctypes
import itertools
import os
import subprocess
import tempfile
import threading
from collections import defaultdict

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
CONFIGS_INC = os.path.join(CSRC, "configs.inc")
BUILD_DIR = os.path.join(HERE, "_lib")

FIELDS = ("BM", "BN", "BK", "WM", "WN", "WNITER", "TM", "TN", "NT", "STAGES", "MINB", "KU", "ORDER")

SPACE = {
    "BM": (64, 128, 256), "BN": (64, 128, 256), "BK": (16, 24, 32),
    "WM": (32, 64, 128), "WN": (32, 64, 128), "WNITER": (1, 2, 4),
    "TM": (4,), "TN": (4,), "STAGES": (5, 4, 3), "MINB": (8, 6, 4, 3, 2, 1), "ORDER": (2,),
}

_lock = threading.Lock()
_checker = None

_SHIM = r'''
#include "tile_config.hpp"
using namespace sgemm_gb300;
extern "C" int cg_check(const int* p, int* d) {
  const TileShape s{p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7], p[8], p[9], p[10], p[11], p[12]};
  const int r = cfg_check(s);
  if (r == 0 && d != nullptr) {
    d[0] = wmiter(s);
    d[1] = acc_per_thread(s);
    d[2] = smem_bytes(s);
    d[3] = est_registers(s);
  }
  return r;
}
'''


def checker():
    """The kernel's legality checker (csrc/tile_config.hpp) compiled for the
    host with g++: cg_check(params[13], derived[4]) -> 0 or the failed rule."""
    global _checker
    with _lock:
        if _checker is None:
            os.makedirs(BUILD_DIR, exist_ok=True)
            out = os.path.join(BUILD_DIR, "libcfgcheck.so")
            hdr = os.path.join(CSRC, "tile_config.hpp")
            if not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(hdr):
                with tempfile.TemporaryDirectory() as d:
                    src = os.path.join(d, "shim.cpp")
                    with open(src, "w") as f:
                        f.write(_SHIM)
                    subprocess.check_call(["g++", "-std=c++17", "-O1", "-shared", "-fPIC",
                                           "-I", CSRC, src, "-o", out + ".tmp"])
                os.replace(out + ".tmp", out)
            lib = ctypes.CDLL(out)
            lib.cg_check.restype = ctypes.c_int
            lib.cg_check.argtypes = [ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
            _checker = lib
        return _checker


def check(t):
    """(rule, derived): rule 0 = legal; derived = (WMITER, accumulators per
    lane, shared bytes per CTA, register estimate) when legal."""
    p = (ctypes.c_int * 13)(*[int(x) for x in t])
    d = (ctypes.c_int * 4)()
    r = checker().cg_check(p, d)
    return r, tuple(d) if r == 0 else None


def enumerate_legal():
    """Every tuple of SPACE (with NT derived from the warp grid and KU = BK)
    that the checker accepts, as (tuple, derived)."""
    out = []
    S = SPACE
    for BM, BN, BK, WM, WN, WNI, TM, TN, ORD in itertools.product(
            S["BM"], S["BN"], S["BK"], S["WM"], S["WN"], S["WNITER"], S["TM"], S["TN"], S["ORDER"]):
        if BM % WM or BN % WN:
            continue
        NT = (BM // WM) * (BN // WN) * 32
        for MINB, ST in itertools.product(S["MINB"], S["STAGES"]):
            t = (BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, BK, ORD)
            r, d = check(t)
            if r == 0:
                out.append((t, d))
    return out


def prune(legal):
    """Rules P4-P6 over the legal tuples (P1-P3 are built into SPACE): one
    (MINB, STAGES) per warp layout, at least 8 warps per SM, at least 64
    accumulators per lane."""
    by_layout = defaultdict(list)
    for t, d in legal:
        by_layout[t[:9] + (t[11], t[12])].append((t, d))
    kept = []
    for _, v in sorted(by_layout.items()):
        minb = max(t[10] for t, _ in v)
        v = [(t, d) for t, d in v if t[10] == minb]
        st = max(t[9] for t, _ in v)
        t, d = [(t, d) for t, d in v if t[9] == st][0]
        if (t[8] // 32) * t[10] < 8 or d[1] < 64:
            continue
        kept.append((t, d))
    return kept


def _rank_key(item):
    t, d = item
    rm, rn = d[0] * t[6], t[5] * t[7]
    return (-d[1], abs(rm - 16) + abs(rn - 8), abs(t[3] - t[4]), -t[10], t)


def candidates(per_shape=2):
    """The tuner's candidate tuples: the best `per_shape` per (BM, BN, BK)."""
    groups = defaultdict(list)
    for t, d in prune(enumerate_legal()):
        groups[t[:3]].append((t, d))
    out = []
    for key in sorted(groups):
        out += [t for t, _ in sorted(groups[key], key=_rank_key)[:per_shape]]
    return out


def config_name(t):
    """Registry name of a tuple: a C identifier that spells its parameters."""
    BM, BN, BK, WM, WN, WNI, TM, TN, NT, ST, MINB, KU, ORD = t
    return f"T{BM}x{BN}x{BK}w{WM}x{WN}n{WNI}p{TM}x{TN}t{NT}s{ST}m{MINB}u{KU}o{ORD}"


def parse_name(name):
    """Inverse of config_name (the registry token before any '_')."""
    import re
    m = re.fullmatch(r"T(\d+)x(\d+)x(\d+)w(\d+)x(\d+)n(\d+)p(\d+)x(\d+)t(\d+)s(\d+)m(\d+)u(\d+)o(\d+)",
                     name.split("_", 1)[0])
    if not m:
        raise ValueError(f"not a generated configuration name: {name}")
    return tuple(int(x) for x in m.groups())


def configs_inc_text(entries, fallback, note):
    """The X-macro list: entries = [(tuple, all_layouts)]; `fallback` (a tuple
    built for every layout) serves transposed operands whose class winner is
    built for row-major operands only."""
    names = [config_name(t) for t, _ in entries]
    if config_name(fallback) not in names:
        raise ValueError("the fallback configuration must be in the list")
    if not dict((config_name(t), a) for t, a in entries)[config_name(fallback)]:
        raise ValueError("the fallback configuration must be built for every layout")
    if len(set(names)) != len(names):
        raise ValueError("duplicate configuration")
    for t, _ in entries:
        r, _ = check(t)
        if r != 0:
            raise ValueError(f"{config_name(t)} breaks legality rule {r}")
    lines = ["// configs.inc -- the tile configurations compiled into the library.",
             "// Generated by dense_fp32_gemm_gb300/configgen.py; " + note,
             "//   X(Name, BM, BN, BK, WM, WN, WNITER, TM, TN, NT, STAGES, MINB, KU, ORDER, ALL_LAYOUTS)",
             f"#define SGEMM_GB300_FALLBACK_CONFIG {config_name(fallback)}",
             "#define SGEMM_GB300_CONFIGS(X) \\"]
    rows = [f"  X({config_name(t)}, {', '.join(str(x) for x in t)}, {1 if a else 0})"
            for t, a in entries]
    lines += [r + " \\" for r in rows[:-1]] + [rows[-1], ""]
    return "\n".join(lines)


def read_configs_inc(path=CONFIGS_INC):
    """[(tuple, all_layouts)] and the fallback tuple of a configs.inc."""
    import re
    text = open(path).read()
    rows = re.findall(r"X\((T\w+), ([\d, ]+)\)", text)
    entries = []
    for name, nums in rows:
        v = [int(x) for x in nums.split(",")]
        t, a = tuple(v[:13]), bool(v[13])
        if config_name(t) != name:
            raise ValueError(f"{name} does not spell its parameters")
        entries.append((t, a))
    fb = re.search(r"#define SGEMM_GB300_FALLBACK_CONFIG (\w+)", text).group(1)
    return entries, parse_name(fb)


def write_configs_inc(entries, fallback, note, path=CONFIGS_INC):
    with open(path + ".tmp", "w") as f:
        f.write(configs_inc_text(entries, fallback, note))
    os.replace(path + ".tmp", path)


if __name__ == "__main__":
    legal = enumerate_legal()
    kept = prune(legal)
    cands = candidates()
    print(f"{len(legal)} legal tuples, {len(kept)} after pruning, {len(cands)} candidates")
    for t in cands:
        print(config_name(t))
