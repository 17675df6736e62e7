"""The C ABI from plain C: the header compiles as C99 and a C program links and runs.

tests/c_abi/hicache_c_roundtrip.c uses only include/hicache.h, the CUDA runtime
and the CPU oracle (test infrastructure).  Without a GPU the program is
compiled and linked only; on a GPU it runs a backup and a single-launch burst
and checks every byte against the oracle.
"""
import os
import subprocess

import pytest

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _build(tmp_path):
    from hierarchical_kv_cache_gb300.build import _cuda_home, build
    import oracle

    lib = build()
    orc = oracle.build_oracle()
    cuda = _cuda_home()
    exe = str(tmp_path / "hicache_c_roundtrip")
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Werror", "-o", exe,
           os.path.join(REPO, "tests", "c_abi", "hicache_c_roundtrip.c"),
           "-I", os.path.join(REPO, "include"), "-I", os.path.join(REPO, "oracle"),
           "-I", os.path.join(cuda, "include"),
           lib, orc, "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.dirname(orc) + ":" +
           os.path.join(cuda, "lib64")]
    subprocess.run(cmd, check=True)
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_program_round_trip_on_gpu(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, f"rc={r.returncode}\n{r.stdout}\n{r.stderr}"
    assert "round trip ok" in r.stdout
