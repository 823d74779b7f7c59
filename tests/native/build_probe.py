"""Compile the test-only tcgen05 layout probes into tests/native/libumma_probe.so,
tests/native/libumma_pair_probe.so and tests/native/libumma_f8_probe.so."""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))


def build_one(name: str) -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = os.path.join(HERE, f"lib{name}.so")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-lineinfo",
           "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared", "-o", out,
           os.path.join(HERE, f"{name}.cu")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"probe build failed: {name}")
    return out


def build() -> list:
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=3) as ex:
        return list(ex.map(build_one, ["umma_probe", "umma_pair_probe", "umma_f8_probe"]))


if __name__ == "__main__":
    print(build())
