"""Build the C-ABI shared library in-tree with nvcc (sm_103a only).

    python -m rank_adapter_apply_gb300.build        # -> rank_adapter_apply_gb300/_build/librank_adapter_apply.so
    python -m rank_adapter_apply_gb300.build --sanitize
        # -> _build_sanitize/: host code with AddressSanitizer and UBSan, for
        #    checking the host paths (run with LD_PRELOAD of libasan and
        #    libubsan, ASAN_OPTIONS=detect_leaks=0 and RANK_ADAPTER_APPLY_LIB
        #    pointing at that library)

Translation units compile in parallel; cudart is linked statically so the
library needs only the NVIDIA driver at run time (loaded lazily on the first
CUDA call, which lets the symbol table be inspected on a machine without one).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "librank_adapter_apply.so")
SOURCES = ["lora_abi.cu", "group.cu", "decode.cu", "decode_cluster.cu", "static_scratch.cu",
           "prefill_tc.cu", "upload.cu", "slot_table.cpp"]
HEADERS = ["kernels.cuh", "slot_table.h", "device_util.cuh", "tc_util.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         f"-I{os.path.join(ROOT, 'include')}"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


SANITIZE_FLAGS = ["-Xcompiler", "-fsanitize=address,-fsanitize=undefined,-fno-omit-frame-pointer", "-g"]


def build(force: bool = False, verbose: bool = False, sanitize: bool = False) -> str:
    out_dir = BUILD + "_sanitize" if sanitize else BUILD
    lib_path = os.path.join(out_dir, os.path.basename(LIB))
    flags = FLAGS + (SANITIZE_FLAGS if sanitize else [])
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    common_deps = [os.path.join(CSRC, h) for h in HEADERS] + [
        os.path.join(ROOT, "include", "rank_adapter_apply.h")]
    objs, jobs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(out_dir, src + ".o")
        objs.append(obj)
        if force or _stale(obj, [path] + common_deps):
            cmd = [nvcc, *ARCH, *flags, "-c", path, "-o", obj]
            if src.endswith(".cpp"):
                cmd = [nvcc, *flags, "-x", "c++", "-c", path, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{p.stdout}\n{p.stderr}")
        return p.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        for err in ex.map(run, jobs):
            if verbose and err:
                print(err, flush=True)
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        link_extra = ["-Xcompiler", "-fsanitize=address,-fsanitize=undefined"] if sanitize else []
        run([nvcc, *ARCH, "-shared", "-cudart", "static", *objs, *link_extra, "-o", tmp])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, sanitize="--sanitize" in sys.argv))
