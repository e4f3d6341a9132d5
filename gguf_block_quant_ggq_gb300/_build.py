"""Build libggq.so in-tree with nvcc for sm_103a (no CMake).

Translation units compile in parallel; the register/spill report of every
kernel (``-Xptxas -v``) is written next to the library as ``ptxas_report.txt``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libggq.so")
BUILD = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libggq needs the CUDA toolkit to build")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "ggq.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, jobs: int | None = None) -> str:
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src: str):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-6000:]}")
        return obj, r.stderr

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    with open(os.path.join(PKG, "ptxas_report.txt"), "w") as f:
        for (obj, log), src in zip(results, srcs):
            f.write(f"== {os.path.basename(src)}\n{log}\n")
    return LIB


def ptxas_summary(report: str | None = None) -> str:
    """Markdown table of every kernel's registers, stack and spills from the
    ``-Xptxas -v`` report that build() writes (one row per kernel instance)."""
    import re

    text = open(report or os.path.join(PKG, "ptxas_report.txt")).read()
    rows = []
    cur = None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = {"name": m.group(1)}
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            cur["stack"], cur["st"], cur["ld"] = (int(g) for g in m.groups())
        m = re.search(r"Used (\d+) registers", line)
        if m:
            cur["regs"] = int(m.group(1))
            rows.append(cur)
            cur = None
    def pretty(mangled):
        # _ZN3ggq<len><name>I<template args>E... -> name<args> (Li5E -> 5, Lb1E -> true)
        m = re.match(r"_ZN3ggq(\d+)", mangled)
        if not m:
            return mangled
        n = int(m.group(1))
        start = m.end()
        name = mangled[start:start + n]
        args = re.findall(r"L([ib])(\d+)E", mangled[start + n:])
        vals = [("true" if v == "1" else "false") if t == "b" else v for t, v in args]
        return f"{name}<{', '.join(vals)}>" if vals else name
    out = ["| kernel | registers | stack (B) | spill stores (B) | spill loads (B) |", "|---|---|---|---|---|"]
    for r in sorted(rows, key=lambda r: pretty(r["name"])):
        out.append(f"| `{pretty(r['name'])}` | {r['regs']} | {r.get('stack', 0)} | {r.get('st', 0)} | {r.get('ld', 0)} |")
    return "\n".join(out) + "\n"


if __name__ == "__main__":
    import sys

    if len(sys.argv) > 2 and sys.argv[1] == "--ptxas-summary":
        build()
        with open(sys.argv[2], "w") as f:
            f.write("# Registers, stack and spills of every kernel instance (nvcc -Xptxas -v, sm_103a)\n\n"
                    "Command:\n\n    python -m gguf_block_quant_ggq_gb300._build --ptxas-summary "
                    f"{os.path.relpath(sys.argv[2], ROOT)}\n\n"
                    "Template arguments: k_stream<kind, format, tokens, activation kind, row chunks>, "
                    "k_gemv_mma<format, dump, chunk width>, k_group<kind, format, dump>, "
                    "k_gmm<kind, format, dump>, k_gmmtc<format, dump>, k_direct<kind, format, "
                    "tokens, dump>; formats 0 Q4_0, 1 Q8_0, 2 Q4_K, 3 Q5_K, 4 Q6_K, 5 MXFP4, 6 Q2_K, 7 Q3_K.\n\n")
            f.write(ptxas_summary())
    else:
        print(build(force=True))
