"""CPU-side checks of the C ABI: the library builds and loads, it exports every
entry point the header declares (and nothing else), and a plain C99 program
compiled with -std=c99 -Wall -Werror -pedantic links against it and gets the
documented status from every entry point's early-return path. No GPU needed."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tts_bb.h")


def _lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location("ttsbb_build", os.path.join(ROOT, "codec_token_tts_gb300", "build.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m.build()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tts_bb_[a-z_0-9]+)\s*\(", text)))


def exported_symbols(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib], capture_output=True, text=True, check=True).stdout
    return sorted({ln.split()[-1] for ln in out.splitlines() if " T " in ln})


def test_library_exports_exactly_the_header():
    lib = _lib()
    decl = declared_symbols()
    assert len(decl) >= 14
    assert exported_symbols(lib) == decl


def test_python_binding_loads_every_symbol():
    _lib()
    import codec_token_tts_gb300 as tb
    assert sorted(tb.EXPORTED) == declared_symbols()
    c = tb.tts_bb_default_config()
    assert (c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.ffn) == (28, 1024, 16, 8, 128, 3072)
    assert abs(c.rms_eps - 1e-6) < 1e-12 and c.rope_theta == 1e6
    assert tb.tts_bb_version().startswith("0.1.0")


def test_c99_consumer_compiles_and_runs(tmp_path):
    lib = _lib()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_c")
    cuda_lib = "/usr/local/cuda/lib64"
    cmd = [cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I" + os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "abi", "abi_c.c"), "-o", exe, lib,
           "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + cuda_lib]
    subprocess.run(cmd, check=True)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = cuda_lib + ":" + env.get("LD_LIBRARY_PATH", "")
    r = subprocess.run([exe], capture_output=True, text=True, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_c: ok" in r.stdout


def test_maskgit_schedule_matches_oracle():
    """Host-only schedule of the library against the oracle's (same reading of
    the shifted time steps); bad arguments are rejected."""
    import numpy as np

    import oracle as O
    _lib()
    import codec_token_tts_gb300 as m
    for n_step, n_total, s in ((32, 6144, 0.1), (8, 100, 0.1), (1, 5, 0.1), (16, 2800, 0.1), (10, 1000, 1.0),
                               (7, 0, 0.3)):
        got = m.tts_bb_maskgit_schedule(n_step, n_total, s)
        assert np.array_equal(got, O.maskgit_schedule(n_step, n_total, s)), (n_step, n_total, s)
    buf = np.zeros(4, np.int32)
    for args in ((0, 10, 0.1), (4, -1, 0.1), (4, 10, 0.0)):
        assert m.lib.tts_bb_maskgit_schedule(*args, buf.ctypes.data) == m.E_INVALID
    assert m.lib.tts_bb_maskgit_schedule(4, 10, 0.1, None) == m.E_INVALID
