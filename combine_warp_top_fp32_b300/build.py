"""Build libep_b300.so in-tree with nvcc for sm_103a.

    python -m combine_warp_top_fp32_b300.build [--force] [--ptxas-info]

No fast-math: the int8 code needs IEEE division and ties-to-even rounding and
the weights need an accurate expf, so denormals are kept (-ftz=false) and
division and square root are IEEE (-prec-div/-prec-sqrt). Bit-exact spots use
explicit __fadd_rn/__fmul_rn/__fmaf_rn/__fdiv_rn, which are never contracted.
"""
from __future__ import annotations

import argparse
import subprocess
import sys
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB = PKG / "libep_b300.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
              "-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-cudart", "static"]


def sources() -> list[Path]:
    return sorted(CSRC.glob("*.cu"))


def _deps() -> list[Path]:
    return sources() + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + sorted(INCLUDE.glob("*.h"))


def up_to_date(lib: Path = LIB) -> bool:
    if not lib.exists():
        return False
    t = lib.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _deps())


def build(force: bool = False, ptxas_info: bool = False, out: Path = LIB, extra: list[str] | None = None) -> Path:
    if not force and up_to_date(out) and not ptxas_info and not extra:
        return out
    cmd = ["nvcc", *ARCH, *NVCC_FLAGS, "-I", str(INCLUDE), "-I", str(CSRC)]
    if ptxas_info:
        cmd += ["-Xptxas", "-v"]
    cmd += list(extra or [])
    cmd += [str(s) for s in sources()] + ["-o", str(out)]
    subprocess.run(cmd, check=True)
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers/spills/shared memory per kernel")
    args = ap.parse_args(argv)
    p = build(force=args.force, ptxas_info=args.ptxas_info)
    print(p)
    return 0


if __name__ == "__main__":
    sys.exit(main())
