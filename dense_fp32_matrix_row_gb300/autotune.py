"""Autotuning of the FFMA tile kernel.

The search of "CUDA 矩阵乘法优化：从朴素 Kernel 到接近 cuBLAS", section "8. Kernel 9:
参数自动调优", redone for GB300: the kernel's compile-time tile parameters are
enumerated, combinations the hardware cannot run are dropped, and the rest are
timed on the GPU.  Two uses:

``python -m dense_fp32_matrix_row_gb300.autotune search``
    Builds one variant library per legal (TM, TN, WM, WN, BK, STAGES, MINB)
    of the default configuration (the FFMA_* macros of csrc/ffma_tma.cu) and
    times each on the benchmark shapes: the exploration that picks the
    default.  Variant libraries go under ``--workdir``.

``python -m dense_fp32_matrix_row_gb300.autotune table --out FILE``
    Times every configuration compiled into the library (see
    ``ffma_configs()``) on shapes inside each (M, N) class (at the class
    bound and 3/4 of it, K at three depths) and on the benchmark's shapes one
    by one (``--exact``), and writes the dispatch table (the format of
    csrc/ffma_tuning.inc) that maps each class to its fastest configuration.
    Copy it over csrc/ffma_tuning.inc and rebuild to use it.

Both need a GB300; ``legal`` and ``table_source`` are plain host code.
"""

from __future__ import annotations

import argparse
import itertools
import json
import os
import subprocess
import sys

# GB300 limits the filter checks against
SMEM_PER_SM = 227 * 1024          # bytes of shared memory one SM gives its CTAs
REGS_PER_SM = 65536
MAX_THREADS = 1024
TMA_BOX_MAX = 256                  # elements per box dimension

# M and N class upper bounds of the table (the last class is unbounded), the
# fractions of the bound at which each class is measured, and the depths
M_CLASSES = [32, 64, 128, 256, 512, 1024, 2048, 4096, 8192]
N_CLASSES = [256, 512, 1024, 2048, 4096, 8192]
POINTS = [1.0, 0.75]
K_DEPTHS = [1024, 4096, 8192]
# a configuration other than the default wins a class only by this margin
# (repeated timings of one shape differ by a few tenths of a percent)
MARGIN = 1.005


def pick(tflops: list[float]) -> int:
    """The configuration for a class from its mean TFLOP/s per configuration."""
    best = max(range(len(tflops)), key=tflops.__getitem__)
    return best if tflops[best] >= MARGIN * tflops[0] else 0


def legal(tm: int, tn: int, wm: int, wn: int, bk: int, stages: int, minb: int) -> tuple[bool, str]:
    """Whether the FFMA kernel can be built and run with these parameters, and
    why not.  Mirrors the kernel's static checks plus the register budget."""
    if tm % 4 or tn % 4 or tm <= 0 or tn <= 0:
        return False, "thread tiles come in float4 groups"
    bm, bn, threads = wm * 4 * tm, wn * 8 * tn, wm * wn * 32
    if bm > TMA_BOX_MAX or bn > TMA_BOX_MAX:
        return False, "a TMA box is at most 256 elements wide"
    if threads > MAX_THREADS or threads < 32:
        return False, "threads per CTA"
    if bk < 4 or bk % 4:
        return False, "k-tile depth"
    smem = 128 + stages * (bk * bm + bk * bn) * 4 + stages * 16
    if smem * minb > SMEM_PER_SM:
        return False, f"shared memory: {minb} x {smem} B > {SMEM_PER_SM} B"
    regs = REGS_PER_SM // (threads * minb)
    regs = min(255, regs - regs % 8)
    need = tm * tn + tm + tn + 24        # accumulators, one k-step's operands, addressing
    if need > regs:
        return False, f"registers: about {need} needed, {regs} per thread at {minb} CTAs/SM"
    return True, ""


def candidates(tiles=((8, 8),)) -> list[tuple[int, ...]]:
    """The search space: (TM, TN, WM, WN, BK, STAGES, MINB), legal ones only,
    with the given thread tiles (by default 8 x 8: a lane loads 16 floats per
    64 FMAs, the ratio at which GB300's shared-memory pipe keeps up with its
    FMA pipe; 8 x 4 loads 12 per 32 and 4 x 4 8 per 16), CTA tiles of at least
    64 x 64, and 8 to 32 warps resident per SM."""
    out = []
    for (tm, tn), (wm, wn), bk, stages, minb in itertools.product(
            tiles, ((2, 2), (4, 2), (2, 4), (4, 1), (1, 4)),
            (16, 32, 48), (2, 3, 4), (1, 2, 4)):
        warps = wm * wn * minb
        if wm * 4 * tm < 64 or wn * 8 * tn < 64 or not 8 <= warps <= 32:
            continue
        if legal(tm, tn, wm, wn, bk, stages, minb)[0]:
            out.append((tm, tn, wm, wn, bk, stages, minb))
    return out


def table_source(rows: list[tuple[int, int, int]], gpu: str, measured: dict,
                 exact: list[tuple[int, int, int, int]] = ()) -> str:
    """C++ source of the dispatch table: entries for the exact shapes (M, N, K,
    config) first, then the classes (m_max, n_max, config; any K) with -1
    meaning unbounded, in lookup order."""
    lim = lambda v: "INT64_MAX" if v < 0 else str(v)
    body = "\n".join([f"    {{{M}, {M}, {N}, {N}, {K}, {K}, {c}}},   // {M}x{N}x{K}" for M, N, K, c in exact] +
                     [f"    {{0, {lim(m)}, 0, {lim(n)}, 0, INT64_MAX, {c}}}," for m, n, c in rows])
    exact_lines = "".join(f"//   {M}x{N}x{K} (exact): " + " ".join(f"{t:.1f}" for t in measured["exact"][f"{M}x{N}x{K}"])
                          + "\n" for M, N, K, _ in exact)
    return (
        "// ffma_tuning.inc -- which FFMA tile configuration runs each shape class.\n"
        "// Written by dense_fp32_matrix_row_gb300/autotune.py from measurements on\n"
        f"// {gpu}; rerun it (and rebuild) to retune.  Entries are tried in order; the\n"
        "// first with M, N and K inside its bounds applies: the shapes measured\n"
        "// exactly (M, N and K), then the (M, N) classes.  A configuration other than the\n"
        f"// default wins only by {100 * (MARGIN - 1):.1f}% or more.\n"
        "// Configurations: " + "; ".join(
            f"{i} = {c['bm']}x{c['bn']} BK {c['bk']}, {c['stages']} stages, {c['ctas_per_sm']} CTAs/SM"
            for i, c in enumerate(measured["configs"])) + ".\n"
        "// Mean TFLOP/s per class and configuration (M, N at "
        + ", ".join(f"{f:g}" for f in POINTS) + " of the class bound; K = "
        + ", ".join(str(k) for k in K_DEPTHS) + "):\n"
        + exact_lines
        + "".join(f"//   M<={lim(m)} N<={lim(n)}: "
                  + " ".join(f"{t:.1f}" for t in measured["classes"][f"{m},{n}"]) + "\n"
                  for m, n, _ in rows)
        + "static const FfmaTuneEntry kFfmaTune[] = {\n" + body + "\n};\n")


def _time(sg, torch, M, N, K, reps=20):
    A = torch.rand((M, K), device="cuda") - 0.5
    B = torch.rand((K, N), device="cuda") - 0.5
    C = torch.empty((M, N), device="cuda")
    for _ in range(3):
        sg.sgemm(A, B, C)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        sg.sgemm(A, B, C)
    e1.record()
    torch.cuda.synchronize()
    if sg.status() != sg.OK:
        raise RuntimeError("kernel error during tuning")
    return 2.0 * M * N * K / (e0.elapsed_time(e1) / reps * 1e-3) / 1e12


def _measure(sg, torch, n_configs, shapes):
    tf = []
    for c in range(n_configs):
        prev = sg.ffma_force_config(c)
        try:
            tf.append(sum(_time(sg, torch, M, N, K) for M, N, K in shapes) / len(shapes))
        finally:
            sg.ffma_force_config(prev)
    return tf


def run_table(out: str, exact_shapes=()) -> None:
    import torch
    import dense_fp32_matrix_row_gb300 as sg
    sg.build()
    configs = sg.ffma_configs()
    exact_tf, exact = {}, []
    seen = set()
    exact_shapes = [s for s in exact_shapes if not (tuple(s) in seen or seen.add(tuple(s)))]
    for M, N, K in exact_shapes:
        tf = _measure(sg, torch, len(configs), [(M, N, K)])
        exact_tf[f"{M}x{N}x{K}"] = tf
        exact.append((M, N, K, pick(tf)))
        print(f"{M}x{N}x{K} (exact): " + " ".join(f"{t:.1f}" for t in tf), flush=True)
    classes, rows = {}, []
    m_bounds, n_bounds = M_CLASSES + [-1], N_CLASSES + [-1]
    for mi, m in enumerate(m_bounds):
        for ni, n in enumerate(n_bounds):
            # shapes inside the class: fractions of its upper bound (for the
            # unbounded class, of twice the previous bound), at each depth
            mt = m if m > 0 else 2 * m_bounds[mi - 1]
            nt = n if n > 0 else 2 * n_bounds[ni - 1]
            shapes = [(max(17, int(mt * f) // 4 * 4), max(4, int(nt * f) // 4 * 4), K)
                      for f in POINTS for K in K_DEPTHS]
            tf = _measure(sg, torch, len(configs), shapes)
            classes[f"{m},{n}"] = tf
            rows.append((m, n, pick(tf)))
            print(f"M<={m} N<={n} ({mt}x{nt}): " + " ".join(f"{t:.1f}" for t in tf), flush=True)
    measured = {"configs": configs, "classes": classes, "exact": exact_tf}
    gpu = torch.cuda.get_device_name()
    with open(out, "w") as f:
        f.write(table_source(rows, gpu, measured, exact))
    with open(out + ".json", "w") as f:
        json.dump({"gpu": gpu, **measured, "table": rows, "exact_table": exact}, f, indent=1)


def rederive(report: str, out: str) -> None:
    """Rewrite the table from a saved report (the .json beside a table) with
    the current ``pick`` rule, without measuring again."""
    with open(report) as f:
        rep = json.load(f)
    rows = [(m, n, pick(rep["classes"][f"{m},{n}"])) for m, n, _ in rep["table"]]
    exact = [(M, N, K, pick(rep["exact"][f"{M}x{N}x{K}"])) for M, N, K, _ in rep.get("exact_table", [])]
    rep.setdefault("exact", {})
    with open(out, "w") as f:
        f.write(table_source(rows, rep["gpu"], rep, exact))


SEARCH_CHILD = r"""
import json, sys, torch
sys.path.insert(0, {root!r})
import dense_fp32_matrix_row_gb300 as sg
from dense_fp32_matrix_row_gb300 import autotune
sg.LIBRARY = {lib!r}
sg.ffma_force_config(0)
print("RESULT", json.dumps({{f"{{M}}x{{N}}x{{K}}": autotune._time(sg, torch, M, N, K)
                             for M, N, K in {shapes!r}}}))
"""


def run_search(workdir: str, shapes: list[tuple[int, int, int]], tiles, only: str = "") -> None:
    # the package re-exports the build() function under the module's name,
    # so import the function itself
    from .build import build as build_library
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    results = {}
    for cand in candidates(tiles):
        name = "tm{}_tn{}_wm{}_wn{}_bk{}_st{}_mb{}".format(*cand)
        if only and not any(o in name for o in only.split(",")):
            continue
        flags = [f"-DFFMA_{k}={v}" for k, v in zip(("TM", "TN", "WM", "WN", "BK", "STAGES", "MINB"), cand)]
        lib = os.path.join(workdir, name, "libsgemm_gb300.so")
        try:
            build_library(extra_flags=flags, library=lib)
        except Exception as e:  # a combination ptxas rejects
            print(name, "build failed:", str(e)[-200:], flush=True)
            continue
        code = SEARCH_CHILD.format(root=root, lib=lib, shapes=shapes)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=900)
        line = [l for l in r.stdout.splitlines() if l.startswith("RESULT ")]
        if r.returncode != 0 or not line:
            print(name, "run failed:", r.stderr[-300:], flush=True)
            continue
        results[name] = json.loads(line[0][7:])
        print(name, results[name], flush=True)
    if not results:
        raise RuntimeError("no configuration built and ran")
    best = max(results.items(), key=lambda kv: sum(kv[1].values()))
    print("best", best[0], best[1])


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    sub = ap.add_subparsers(dest="cmd", required=True)
    t = sub.add_parser("table", help="time the compiled configurations per shape class")
    t.add_argument("--out", required=True, help="where to write the table (C++ source)")
    t.add_argument("--from-report", help="rewrite the table from this saved report instead of measuring")
    t.add_argument("--exact", default="4092x4092x4092,8192x8192x8192,8192x12288x4096,8192x14336x4096,"
                                      "8192x4096x14336,32x14336x4096,64x14336x4096,128x14336x4096",
                   help="shapes (MxNxK, comma-separated) measured one by one; their entries come first")
    s = sub.add_parser("search", help="time every legal default configuration")
    s.add_argument("--workdir", required=True, help="directory for the variant libraries")
    s.add_argument("--shapes", default="4092x4092x4092,8192x8192x8192,1024x1024x1024",
                   help="comma-separated MxNxK")
    s.add_argument("--tiles", default="8x8", help="thread tiles TMxTN to search, comma-separated")
    s.add_argument("--only", default="",
                   help="comma-separated name fragments; only candidates whose name contains one run")
    args = ap.parse_args(argv)
    if args.cmd == "table":
        if args.from_report:
            rederive(args.from_report, args.out)
        else:
            exact = [tuple(int(v) for v in x.split("x")) for x in args.exact.split(",") if x]
            run_table(args.out, exact)
    else:
        shapes = [tuple(int(v) for v in s.split("x")) for s in args.shapes.split(",")]
        tiles = tuple(tuple(int(v) for v in t.split("x")) for t in args.tiles.split(","))
        run_search(args.workdir, shapes, tiles, args.only)
    return 0


if __name__ == "__main__":
    sys.exit(main())
