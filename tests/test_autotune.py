"""Host side of the FFMA autotuning: the legality filter of the search, the
generated dispatch table, and the library's table lookup (no GPU needed)."""

import os
import re
import subprocess

import pytest

import dense_fp32_matrix_row_gb300 as sg
from dense_fp32_matrix_row_gb300 import autotune

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "dense_fp32_matrix_row_gb300", "csrc", "ffma_tuning.inc")

# (TM, TN, WM, WN, BK, STAGES, MINB) of the configurations compiled into the library
COMPILED = [(8, 8, 4, 2, 48, 2, 2), (8, 8, 2, 4, 32, 2, 2), (8, 8, 4, 1, 32, 2, 4),
            (8, 8, 4, 2, 16, 4, 2), (8, 8, 1, 4, 32, 2, 3), (8, 8, 4, 2, 32, 2, 2)]


@pytest.fixture(scope="module")
def L():
    sg.build()
    return sg.lib()


def test_compiled_configurations_are_legal_and_reported(L):
    got = sg.ffma_configs()
    assert len(got) == len(COMPILED)
    for (tm, tn, wm, wn, bk, st, mb), info in zip(COMPILED, got):
        assert autotune.legal(tm, tn, wm, wn, bk, st, mb) == (True, "")
        assert info == {"bm": wm * 4 * tm, "bn": wn * 8 * tn, "bk": bk, "stages": st,
                        "threads": wm * wn * 32, "ctas_per_sm": mb}


@pytest.mark.parametrize("cfg,why", [
    ((8, 8, 4, 2, 32, 4, 2), "shared memory"),       # 2 x 128 KB > 227 KB
    ((16, 8, 4, 2, 32, 2, 2), "registers"),          # 128 accumulators at 128 registers
    ((8, 16, 4, 4, 32, 2, 1), "256 elements"),       # BN = 512
    ((6, 8, 4, 2, 32, 2, 2), "float4"),
    ((8, 8, 8, 4, 32, 2, 1), "registers"),           # 1024 threads: 64 registers each
])
def test_illegal_configurations_are_rejected(cfg, why):
    ok, reason = autotune.legal(*cfg)
    assert not ok and why in reason


def test_search_space():
    c = autotune.candidates()
    assert (8, 8, 4, 2, 48, 2, 2) in c                # the default is searched
    assert all(autotune.legal(*x)[0] for x in c)
    assert all(8 <= x[2] * x[3] * x[6] <= 32 for x in c)
    assert len(autotune.candidates(((8, 8), (8, 4), (4, 8)))) > len(c)


def _compile_table(tmp_path, text):
    src = tmp_path / "t.cc"
    src.write_text("#include <cstdint>\n#include <cstdio>\n"
                   "struct FfmaTuneEntry { int64_t m_lo, m_max, n_lo, n_max, k_lo, k_max; int config; };\n" + text +
                   "int main() { std::printf(\"%d\\n\", (int)(sizeof(kFfmaTune) / sizeof(kFfmaTune[0]))); }\n")
    exe = tmp_path / "t"
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", str(src), "-o", str(exe)], check=True)
    return int(subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout)


def _entries(text):
    """(m_lo, m_max, n_lo, n_max, k_lo, k_max, config) of every table entry."""
    v = r"(INT64_MAX|\d+)"
    rows = re.findall(r"\{\s*" + r",\s*".join([v] * 6) + r",\s*(\d+)\s*\}", text)
    big = 2 ** 63 - 1
    num = lambda x: big if x == "INT64_MAX" else int(x)
    return [tuple(num(x) for x in r[:6]) + (int(r[6]),) for r in rows]


def _lookup(entries, M, N, K):
    return next(e[6] for e in entries
                if e[0] <= M <= e[1] and e[2] <= N <= e[3] and e[4] <= K <= e[5])


def test_generated_table_compiles(tmp_path):
    configs = [dict(bm=128, bn=128, bk=32, stages=2, ctas_per_sm=2)] * 2
    rows = [(64, 256, 1), (64, -1, 0), (-1, -1, 0)]
    measured = {"configs": configs, "exact": {"4092x4092x4092": [60.0, 62.0]},
                "classes": {"64,256": [10.0, 12.0], "64,-1": [11.0, 9.0], "-1,-1": [60.0, 55.0]}}
    text = autotune.table_source(rows, "test GPU", measured, [(4092, 4092, 4092, 1)])
    assert _compile_table(tmp_path, text) == 4
    big = 2 ** 63 - 1
    assert _entries(text) == [(4092, 4092, 4092, 4092, 4092, 4092, 1), (0, 64, 0, 256, 0, big, 1),
                              (0, 64, 0, big, 0, big, 0), (0, big, 0, big, 0, big, 0)]


def test_committed_table(tmp_path, L):
    text = open(TABLE).read()
    n = _compile_table(tmp_path, text)
    entries = _entries(text)
    assert len(entries) == n and n >= 1
    big = 2 ** 63 - 1
    assert entries[-1][:6] == (0, big, 0, big, 0, big), "the last entry must catch every shape"
    assert all(0 <= e[6] < len(COMPILED) for e in entries)
    # the library's lookup is the first matching entry
    for M in (17, 64, 65, 128, 300, 1024, 4092, 8192, 9000):
        for N in (8, 256, 257, 1024, 4092, 12288, 14336):
            for K in (64, 1024, 4092, 4096, 8192):
                assert sg.ffma_config_for(M, N, K) == _lookup(entries, M, N, K), (M, N, K)
    # exact shapes match on K too
    for e in entries:
        if e[0] == e[1] and e[4] == e[5]:
            assert sg.ffma_config_for(e[0], e[2], e[4]) == e[6]


def test_forcing_a_configuration(L):
    assert sg.ffma_force_config(len(COMPILED)) == sg.ERR_BAD_ARG
    prev = sg.ffma_force_config(2)
    try:
        assert prev == -1
        assert sg.ffma_config_for(4092, 4092, 4092) == 2
    finally:
        sg.ffma_force_config(-1)
    assert sg.ffma_config_for(4092, 4092, 4092) == _lookup(_entries(open(TABLE).read()), 4092, 4092, 4092)


def test_pick_keeps_the_default_within_the_margin():
    assert autotune.pick([60.0, 60.2, 59.0]) == 0          # 0.3% is noise
    assert autotune.pick([60.0, 61.0, 59.0]) == 1
    assert autotune.pick([10.0, 9.0, 9.5]) == 0


def test_search_runs_only_the_named_candidates(monkeypatch, tmp_path, capsys):
    # the search builds and times a variant library per candidate; here the
    # build and the timing child are stand-ins, so only the selection and
    # the report are exercised
    import json as _json
    import importlib
    build_mod = importlib.import_module("dense_fp32_matrix_row_gb300.build")
    built = []

    def fake_build(extra_flags=None, library=None, **kw):
        built.append((tuple(extra_flags), library))
        return library

    class Done:
        def __init__(self, out):
            self.returncode, self.stdout, self.stderr = 0, out, ""

    def fake_run(cmd, capture_output, text, timeout):
        tflops = 60.0 + len(built)   # later candidates "measure" faster
        return Done("RESULT " + _json.dumps({"4092x4092x4092": tflops}) + "\n")

    monkeypatch.setattr(build_mod, "build", fake_build)
    monkeypatch.setattr(autotune.subprocess, "run", fake_run)
    autotune.run_search(str(tmp_path), [(4092, 4092, 4092)], ((8, 8),),
                        only="wm2_wn2_bk32_st2_mb4,wm4_wn1_bk32_st2_mb4")
    names = [os.path.basename(os.path.dirname(lib)) for _, lib in built]
    assert names == ["tm8_tn8_wm2_wn2_bk32_st2_mb4", "tm8_tn8_wm4_wn1_bk32_st2_mb4"]
    assert all("-DFFMA_MINB=4" in flags for flags, _ in built)
    out = capsys.readouterr().out
    assert "best tm8_tn8_wm4_wn1_bk32_st2_mb4" in out
    with pytest.raises(RuntimeError):
        autotune.run_search(str(tmp_path), [(4092, 4092, 4092)], ((8, 8),), only="no_such_name")
