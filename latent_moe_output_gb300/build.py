"""Build the CUDA library in-tree: csrc/*.cu -> _lib/liblatent_tail.so.

sm_103a only (``-gencode arch=compute_103a,code=sm_103a``), one nvcc process
per translation unit in parallel, then one link step. No CMake.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
OUT = PKG / "_lib" / "liblatent_tail.so"

GENCODE = "arch=compute_103a,code=sm_103a"


def cuda_home() -> Path:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and (Path(cand) / "bin" / "nvcc").exists():
            return Path(cand)
    nvcc = shutil.which("nvcc")
    if nvcc:
        return Path(nvcc).resolve().parent.parent
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def nvcc_flags(extra=()) -> list[str]:
    return ["-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}", f"-I{CSRC}",
            "--expt-relaxed-constexpr", *extra]


def build(out: Path = OUT, extra_flags=(), verbose: bool = False, force: bool = False) -> Path:
    sources = sorted(CSRC.glob("*.cu"))
    deps = sources + sorted(CSRC.glob("*.cuh")) + sorted(CSRC.glob("*.h")) + \
        sorted(INCLUDE.glob("*.h"))
    if out.exists() and not force and not extra_flags:
        newest = max(p.stat().st_mtime for p in deps)
        if out.stat().st_mtime >= newest:
            return out
    home = cuda_home()
    nvcc = str(home / "bin" / "nvcc")
    objdir = BUILD / ("release" if not extra_flags else "variant")
    objdir.mkdir(parents=True, exist_ok=True)
    flags = nvcc_flags(extra_flags)

    def compile_one(src: Path) -> Path:
        obj = objdir / (src.stem + ".o")
        cmd = [nvcc, *flags, "-c", str(src), "-o", str(obj)]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src.name}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        objs = list(ex.map(compile_one, sources))
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_name(out.name + f".tmp{os.getpid()}")
    cmd = [nvcc, "-shared", "-gencode", GENCODE, *[str(o) for o in objs], "-o", str(tmp),
           "-cudart", "shared", f"-Xlinker", f"-rpath,{home / 'lib64'}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv[1:], force=True))
