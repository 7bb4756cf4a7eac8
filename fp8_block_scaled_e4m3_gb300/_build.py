"""Build libfp8bs.so in-tree with nvcc for sm_103a (no CMake, parallel TUs)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libfp8bs.so")
SOURCES = ["api.cu", "bs_kernel.cu", "bs2_kernel.cu", "mx_kernel.cu", "mx2_kernel.cu", "mxd_kernel.cu"]
HEADERS = ["ptx.cuh", "common.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "fp8bs.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def parse_ptxas(log_path: str) -> dict:
    """{kernel symbol: {"registers": int, "stack": int, "spill_stores": int, "spill_loads": int}} from ptxas -v."""
    import re
    out, cur = {}, None
    with open(log_path) as f:
        for line in f:
            m = re.search(r"Function properties for (\S+)", line)
            if m:
                cur = m.group(1)
                out[cur] = {}
                continue
            m = re.search(r"(\d+) bytes stack frame", line)
            if m and cur:
                out[cur]["stack"] = int(m.group(1))
            m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and cur:
                out[cur]["spill_stores"] = int(m.group(1))
                out[cur]["spill_loads"] = int(m.group(2))
            m = re.search(r"Used (\d+) registers", line)
            if m and cur:
                out[cur]["registers"] = int(m.group(1))
    return out


def check_resources(log_path: str) -> None:
    """The blockscale kernels (one CTA and CTA pair) and the stream-K MXFP8 and
    tensor-scale kernels re-split their registers with setmaxnreg (4 warps
    low, 8 high) out of a launch allotment of 384 threads x 168; that split is
    only valid when the kernel is compiled to exactly 168 registers. No kernel
    may spill or keep an array in local memory (a stack frame)."""
    info = parse_ptxas(log_path)
    for sym, r in info.items():
        split = any(k in sym for k in ("fp8bs_blockscale_kernel", "fp8bs_blockscale_pair_kernel",
                                       "fp8bs_mxfp8_sk_kernel", "fp8bs_tensorscale_sk_kernel"))
        if split and r.get("registers") != 168:
            raise RuntimeError(f"{sym}: {r.get('registers')} registers, the setmaxnreg split needs 168")
        if r.get("spill_stores", 0) or r.get("spill_loads", 0) or r.get("stack", 0):
            raise RuntimeError(f"{sym}: register spills or stack frame {r}")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared library.

    ptxas register / spill / shared-memory reports go to _build/ptxas.log.
    """
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
                     "-I", os.path.join(ROOT, "include")]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src + ".log"), "w")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log, src, cmd))
        objs.append(obj)
    failed = []
    for p, log, src, cmd in procs:
        rc = p.wait()
        log.close()
        if rc != 0:
            failed.append(src)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as out:
        for src in SOURCES:
            with open(os.path.join(BUILD, src + ".log")) as f:
                txt = f.read()
            out.write(f"==== {src}\n{txt}\n")
            if verbose or src in failed:
                sys.stderr.write(txt)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}; see {BUILD}/*.log")
    check_resources(os.path.join(BUILD, "ptxas.log"))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, LIB)
    return LIB


def resources_table(log_path: str) -> str:
    """One line per kernel instance from a ptxas -v log: registers, stack, spills, static shared memory."""
    import re
    smem, cur = {}, None
    with open(log_path) as f:
        for line in f:
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                cur = m.group(1)
            m = re.search(r"Used \d+ registers.*?(\d+) bytes smem", line)
            if m and cur:
                smem[cur] = int(m.group(1))
    rows = ["registers  stack  spill_st  spill_ld  static_smem  kernel (mangled symbol)"]
    for sym, r in sorted(parse_ptxas(log_path).items()):
        rows.append(f"{r.get('registers', 0):9d}  {r.get('stack', 0):5d}  {r.get('spill_stores', 0):8d}  "
                    f"{r.get('spill_loads', 0):8d}  {smem.get(sym, 0):11d}  {sym}")
    return "\n".join(rows)


if __name__ == "__main__":
    lib = build(force="--force" in sys.argv, verbose="--resources" not in sys.argv)
    if "--resources" in sys.argv:
        print(resources_table(os.path.join(BUILD, "ptxas.log")))
    else:
        print(lib)
