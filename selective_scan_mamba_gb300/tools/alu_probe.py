"""Builds and runs alu_probe.cu (nvcc, sm_103a) and prints its JSON line.

    python -m selective_scan_mamba_gb300.tools.alu_probe
"""
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))


def main() -> int:
    from selective_scan_mamba_gb300.build import ARCH, nvcc
    with tempfile.TemporaryDirectory() as tmp:
        exe = os.path.join(tmp, "alu_probe")
        r = subprocess.run([nvcc(), *ARCH, "-O3", os.path.join(HERE, "alu_probe.cu"), "-o", exe],
                           capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stderr)
            return r.returncode
        return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
