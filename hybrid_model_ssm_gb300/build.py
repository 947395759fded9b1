"""Build librssm.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own process, in parallel. The shared
library lands next to this file, and the objects go to ``_build/``. The
build reruns only when a source or header is newer than the library.
Usage: ``python -m hybrid_model_ssm_gb300.build [--force] [--verbose]``, or
``--resources`` for a table of each kernel's registers, stack, spills and static
shared memory as ptxas reports them.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librssm.so")
HEADERS = [os.path.join(ROOT, "include", "rssm.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librssm.so")
    return cand


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    return sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + HEADERS


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link librssm.so in-tree. Returns its path."""
    lib = LIB
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


_MODES = {"0": "decode", "1": "verify", "2": "flush", "3": "quantize", "4": "conventional", "5": "snapshot verify"}
_TILES = {"0": "FP32", "1": "E4M3 copy", "2": "E2M1 copy", "3": "FP16 ckpt", "4": "delta rule"}


def _kernel_label(name: str) -> str:
    """A readable label for a demangled kernel name (mode and tile format spelled out)."""
    import re
    m = re.match(r"void rssm::head_kernel<(\d), (\d+), ([^,]+), (\d)>", name)
    if m:
        return f"head_kernel {_MODES[m[1]]}, N={m[2]}, {m[3].replace('__nv_bfloat16', 'bf16')}, {_TILES[m[4]]}"
    m = re.match(r"void rssm::nonflush_kernel<(\d+), ([^,]+), (\d)>", name)
    if m:
        return f"nonflush_kernel N={m[1]}, {m[2].replace('__nv_bfloat16', 'bf16')}, {_TILES[m[3]]}"
    m = re.match(r"void rssm::verify_tc_kernel<(\d+), (\d+)>", name)
    if m:
        return f"verify_tc_kernel N={m[1]}, P={m[2]}"
    return name.split("(")[0].replace("rssm::", "")


def resources() -> list[dict]:
    """Registers, stack frame, spills and static shared memory of every kernel, as ptxas
    reports them (-Xptxas -v) for sm_103a. Compiles into _build/resources; no GPU needed."""
    import re
    out_dir = os.path.join(BUILD, "resources")
    os.makedirs(out_dir, exist_ok=True)

    def one(src):
        cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-Xptxas", "-v", "-c", src, "-o",
               os.path.join(out_dir, os.path.basename(src).replace(".cu", ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
        return os.path.basename(src), r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        logs = list(ex.map(one, sources()))
    rows, cur = [], None
    for src, log in logs:
        for line in log.splitlines():
            m = re.search(r"Compiling entry function '([^']+)'", line)
            if m:
                cur = {"source": src, "mangled": m[1], "stack": 0, "spill_st": 0, "spill_ld": 0, "smem": 0}
                rows.append(cur)
                continue
            if cur is None:
                continue
            m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m:
                cur["stack"], cur["spill_st"], cur["spill_ld"] = int(m[1]), int(m[2]), int(m[3])
            m = re.search(r"Used (\d+) registers", line)
            if m:
                cur["regs"] = int(m[1])
                sm = re.search(r"(\d+) bytes smem", line)
                cur["smem"] = int(sm[1]) if sm else 0
    filt = shutil.which("c++filt")
    names = [r["mangled"] for r in rows]
    if filt and names:
        dem = subprocess.run([filt], input="\n".join(names), capture_output=True, text=True).stdout.splitlines()
        if len(dem) == len(names):
            names = dem
    for r, n in zip(rows, names):
        r["kernel"] = _kernel_label(n)
    return sorted(rows, key=lambda r: (r["source"], r["kernel"]))


def resources_table() -> str:
    rows = resources()
    lines = ["| source | kernel | registers | stack B | spill st/ld B | static smem B |", "|---|---|---|---|---|---|"]
    for r in rows:
        lines.append(f"| {r['source']} | {r['kernel']} | {r.get('regs', '?')} | {r['stack']} | "
                     f"{r['spill_st']}/{r['spill_ld']} | {r['smem']} |")
    return "\n".join(lines)


if __name__ == "__main__":
    if "--resources" in sys.argv:
        print(resources_table())
    else:
        print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
