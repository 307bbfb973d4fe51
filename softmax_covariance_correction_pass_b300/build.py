"""Build libparallax_attn.so in-tree with nvcc for sm_103a.

    python -m softmax_covariance_correction_pass_b300.build [--force] [--verbose] [--debug]

Each ``csrc/*.cu`` is compiled to an object in ``_build/`` (in parallel), then
linked into ``softmax_covariance_correction_pass_b300/libparallax_attn.so``
with the CUDA runtime linked statically, so the library loads without a GPU
and without a CUDA runtime on the loader path.  ``-Xptxas -v`` output (registers,
spills, shared memory per kernel) is kept in ``_build/ptxas.log``.

``--debug`` builds ``libparallax_attn_debug.so`` instead (objects in ``_build/debug``)
with ``-DPARALLAX_DEBUG_CHECKS``: every global write and bulk copy the kernels guard is
checked against the extent of its tensor on the device, and a failed check raises
PARALLAX_DEVERR_BOUNDS in the device error word instead of touching memory outside the
tensor.  The binding loads it when ``PARALLAX_LIBRARY=debug`` is set.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libparallax_attn.so")
DEBUG_LIB = os.path.join(PKG, "libparallax_attn_debug.so")
DEBUG_FLAGS = ["-DPARALLAX_DEBUG_CHECKS"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, build_dir: str, extra: tuple = ()) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


# Kernels that hand registers between warpgroups (setmaxnreg) must be launched
# with exactly the per-thread register count their hand-over arithmetic assumes;
# a smaller launch allocation would make the raising warpgroups wait forever.
LAUNCH_REGISTERS = {"prefill_pair_kernel": 168}


def kernel_registers(log: str) -> dict:
    """Map each compiled kernel (mangled name) to the registers ptxas assigned."""
    regs, name = {}, None
    for line in log.splitlines():
        if "Compiling entry function" in line:
            name = line.split("'")[1]
        elif name and "Used" in line and "registers" in line:
            regs[name] = int(line.split("Used")[1].split("registers")[0])
            name = None
    return regs


def check_registers(log: str) -> None:
    regs = kernel_registers(log)
    for key, want in LAUNCH_REGISTERS.items():
        found = {n: r for n, r in regs.items() if key in n}
        if not found:
            raise RuntimeError(f"no kernel matching {key} in the ptxas report")
        bad = {n: r for n, r in found.items() if r != want}
        if bad:
            raise RuntimeError(f"{key}: ptxas assigned {sorted(set(bad.values()))} registers, "
                               f"the register hand-over needs exactly {want}")


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = DEBUG_LIB if debug else LIB
    if not force and up_to_date(lib):
        return lib
    build_dir = os.path.join(BUILD, "debug") if debug else BUILD
    extra = tuple(DEBUG_FLAGS) if debug else ()
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda p: _compile(p, build_dir, extra), srcs))
    log = "\n".join(r[1] for r in results)
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        f.write(log)
    check_registers(log)
    if verbose:
        print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[r[0] for r in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--debug", action="store_true",
                    help="build libparallax_attn_debug.so with device-side bounds checks")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, debug=args.debug))
    return 0


if __name__ == "__main__":
    sys.exit(main())
