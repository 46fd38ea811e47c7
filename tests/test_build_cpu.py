"""Build switches of libmoe.so that the default build does not exercise (no GPU needed)."""

import os
import subprocess

from sparse_mixture_experts_61_b300 import build as moe_build


def test_trace_ranges_compile_in(tmp_path):
    """MOE_NVTX=1 compiles NVTX ranges around moe_forward's stages into the C ABI."""
    obj = str(tmp_path / "moe_api_nvtx.o")
    src = os.path.join(moe_build.CSRC, "moe_api.cu")
    subprocess.run([moe_build.NVCC, *moe_build.ARCH, *moe_build.FLAGS, "-DMOE_NVTX=1", "-c", src,
                    "-o", obj], check=True, capture_output=True, text=True)
    syms = subprocess.run(["nm", obj], capture_output=True, text=True, check=True).stdout
    assert "nvtx" in syms.lower()
