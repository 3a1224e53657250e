"""Build the in-tree shared libraries with nvcc for sm_103a.

``python -m exact_attention_16_gb300.build`` (or ``__graft_entry__.build()``)
compiles, in parallel:

* ``_lib/libfa_gb300.so``  the C-ABI attention library (include/fa.h);
* ``_lib/libfa_probes.so`` single-tile primitive probes used by the GPU tests.

The CUDA runtime is linked statically, so loading a library needs no GPU
driver; only calls that touch the device do.
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "_lib")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
    "-shared",
]

TARGETS = {
    "libfa_gb300.so": ["fa_api.cu", "fa_merge.cu", "fa_decode.cu", "fa_decode_noalloc.cu", "fa_host.cu"],
    "libfa_probes.so": ["probes.cu"],
}


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources_newer(lib: str, srcs) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(PKG), "include", "fa.h"))
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> dict:
    os.makedirs(LIBDIR, exist_ok=True)
    procs = {}
    for lib, srcs in TARGETS.items():
        out = os.path.join(LIBDIR, lib)
        if not force and not _sources_newer(out, srcs):
            continue
        cmd = [nvcc(), *NVCC_FLAGS, "-o", out + ".tmp", *[os.path.join(CSRC, s) for s in srcs]]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs[lib] = (subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True), out)
    logs = {}
    failed = []
    for lib, (pr, out) in procs.items():
        text, _ = pr.communicate()
        logs[lib] = text
        if pr.returncode != 0:
            failed.append(lib)
        else:
            os.replace(out + ".tmp", out)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(failed) + ":\n" + "\n".join(logs[f] for f in failed))
    return logs


if __name__ == "__main__":
    logs = build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    for lib, text in logs.items():
        print(f"== {lib}\n{text}")
