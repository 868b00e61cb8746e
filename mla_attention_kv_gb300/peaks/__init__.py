"""Measured compute roofs that MEASURED_PEAKS.json does not carry.

``measure()`` compiles and runs mma_sync_rates.cu (nvcc, sm_103a) and
returns its report: the throughput of mma.sync f16 / bf16 / s8 and FFMA.
The s8 figure is the roof bench.py uses for the W8A8 integer GEMMs.
"""
import os
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def measure() -> str:
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "mma_sync_rates")
        subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                        os.path.join(HERE, "mma_sync_rates.cu")], check=True)
        return subprocess.run([exe], check=True, capture_output=True, text=True).stdout


if __name__ == "__main__":
    print(measure())
