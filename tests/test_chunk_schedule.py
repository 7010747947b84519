"""The codec kernels' order of chunks, on the CPU: the launchers' grid (wave_grid) and each
CTA's chunks (cta_chunks) cover every chunk exactly once, wave by wave, for sizes from one
chunk to several hundred thousand and any resident CTA count.  The check is a host program
compiled with nvcc from tests/cuda/chunk_schedule.cu against the library's own headers."""
import os
import subprocess

from compressed_pseudo_gradient_gb300 import build as lib_build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_every_chunk_taken_once(tmp_path):
    exe = os.path.join(tmp_path, "chunk_schedule")
    src = os.path.join(HERE, "cuda", "chunk_schedule.cu")
    subprocess.run([lib_build.nvcc(), *lib_build.NVCC_FLAGS, "-o", exe, src], check=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert ", 0 failed" in out.stdout
