"""Builds and runs the instruction-rate microbenchmark (issue_rates.cu) on GPU 0:
python -m rank_latent_routing_gb300.micro"""
import os
import subprocess
import sys

from rank_latent_routing_gb300.build import ARCH, LIBDIR, nvcc

HERE = os.path.dirname(os.path.abspath(__file__))


def main() -> int:
    os.makedirs(LIBDIR, exist_ok=True)
    exe = os.path.join(LIBDIR, "issue_rates")
    subprocess.run([nvcc(), *ARCH, "-O3", os.path.join(HERE, "issue_rates.cu"), "-o", exe], check=True)
    return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
