"""The C ABI from plain C: tests/c_abi/dg_pass_example.c includes only include/dgcanvas.h and the
CUDA runtime header, links libdgcanvas.so, and runs one bf16 pass; on the GPU its outputs are
checked against the oracle on the inputs it wrote out."""
import os
import subprocess
from pathlib import Path

import numpy as np
import pytest

ROOT = Path(__file__).resolve().parents[1]
PKG = ROOT / "uniform_state_denoising_vocab_b300"
CUDA = Path(os.environ.get("CUDA_HOME", "/usr/local/cuda"))


def _build(tmp_path: Path) -> Path:
    from uniform_state_denoising_vocab_b300 import build
    build.build()
    exe = tmp_path / "dg_pass_example"
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           str(ROOT / "tests" / "c_abi" / "dg_pass_example.c"), "-I", str(ROOT / "include"),
           "-I", str(CUDA / "include"), "-L", str(PKG), "-ldgcanvas", "-L", str(CUDA / "lib64"),
           "-lcudart", f"-Wl,-rpath,{PKG}:{CUDA / 'lib64'}", "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_example_compiles_and_links(tmp_path):
    """The header is valid C99 and every call the example makes resolves in the library."""
    assert _build(tmp_path).exists()


def _read(path: Path):
    b = path.read_bytes()
    hdr = np.frombuffer(b, np.int32, 6, 0)
    B, S, V, d, K, p = (int(x) for x in hdr)
    off = 24
    seed = int(np.frombuffer(b, np.uint64, 1, off)[0])
    off += 8
    R = B * S
    out = {"B": B, "S": S, "V": V, "d": d, "K": K, "pass": p, "seed": seed}
    for name, dt, n in (("h", np.uint16, R * d), ("w", np.uint16, V * d), ("canvas_in", np.int32, R),
                        ("canvas", np.int32, R), ("argmax", np.int32, R), ("conf", np.float32, R),
                        ("entropy", np.float32, R), ("kept", np.uint8, R),
                        ("mean_entropy", np.float32, B), ("status", np.uint32, 1)):
        out[name] = np.frombuffer(b, dt, n, off).copy()
        off += n * np.dtype(dt).itemsize
    assert off == len(b)
    return out


@pytest.mark.gpu
def test_c_example_pass_matches_oracle(tmp_path, orc):
    from parity import TOL, check_select, check_stats
    exe = _build(tmp_path)
    out = tmp_path / "pass.bin"
    args = [str(out), "2", "200", "3001", "264", "40", "12345", "7"]
    r = subprocess.run([str(exe), *args], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout
    g = _read(out)
    assert int(g["status"][0]) == 0
    B, S, V, d, K, p, seed = g["B"], g["S"], g["V"], g["d"], g["K"], g["pass"], g["seed"]
    o = orc.step(B, S, V, d, "bf16", g["h"], g["w"], K, seed, p)
    check_stats(g, o, TOL["bf16"])
    check_select(g, o, B, S, V, K, seed, p, orc.draw)
    assert np.allclose(g["mean_entropy"], o["mean_entropy"], atol=TOL["bf16"])
