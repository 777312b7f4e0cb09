"""Build libdec.so (the C-ABI decode-step library) for sm_103a with nvcc.

Each CUDA translation unit is compiled in parallel, then linked into a shared
library next to this file.  The CUDA runtime is linked statically, so the
library only needs the NVIDIA driver at run time.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import pathlib
import shutil
import subprocess
import sys

HERE = pathlib.Path(__file__).resolve().parent
CSRC = HERE / "csrc"
BUILD = HERE / "_build"
LIB = HERE / "libdec.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def sources() -> list[pathlib.Path]:
    return sorted(CSRC.glob("*.cu"))


def _stale(obj: pathlib.Path, src: pathlib.Path) -> bool:
    if not obj.exists():
        return True
    deps = [src] + list(CSRC.glob("*.cuh")) + [HERE.parent / "include" / "dec.h"]
    return any(d.stat().st_mtime > obj.stat().st_mtime for d in deps)


def build(verbose: bool = False, force: bool = False, extra: list[str] | None = None) -> pathlib.Path:
    """Compile every stale translation unit and link libdec.so.

    DEC_TIMELINE=1 in the environment compiles in the per-launch %globaltimer
    stamps of dec_set_timeline.  A change of flags rebuilds everything.
    """
    BUILD.mkdir(exist_ok=True)
    extra = list(extra or [])
    if os.environ.get("DEC_TIMELINE", "0") == "1":
        extra.append("-DDEC_TIMELINE=1")
    stamp = BUILD / "flags.txt"
    flags = " ".join(ARCH + FLAGS + extra)
    if not stamp.exists() or stamp.read_text() != flags:
        force = True
    cmds = []
    objs = []
    for src in sources():
        obj = BUILD / (src.stem + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            cmds.append([nvcc(), *ARCH, *FLAGS, *extra, "-c", str(src), "-o", str(obj)])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {cmd[-3]}")
        return r

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(cmds), os.cpu_count() or 4))) as ex:
        list(ex.map(run, cmds))
    if cmds or force or not LIB.exists():
        tmp = LIB.with_suffix(".so.tmp")
        run([nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", str(tmp), *map(str, objs)])
        os.replace(tmp, LIB)
    stamp.write_text(flags)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
