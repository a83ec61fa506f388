"""Build libjepa_gb300.so in place with nvcc for sm_103a (no cmake, one -gencode).

Each translation unit (.cu, and the host-only .cpp) compiles in parallel to an object under _build/, then one link
step writes jepa_vision_encoder_gb300/libjepa_gb300.so. Host code is compiled with
floating-point contraction off so that the seeded weight generator (synth/jepa_synth.h)
produces the same bits on x86-64 and aarch64.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libjepa_gb300.so")
SOURCES = ["runtime.cu", "gemm_tc.cu", "gemm_tc2.cu", "attention_tc.cu", "simt.cu", "rowops.cu", "postab.cu",
           "predictor.cu", "head.cu", "gguf.cpp"]
HEADERS = ["ptx.cuh", "epilogue.cuh", "kernels.h", "internal.h", "seq.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libjepa_gb300.so")


def _flags():
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-ffp-contract=off",
                   "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "synth"), "-I", CSRC]


def _deps():
    deps = [os.path.join(CSRC, h) for h in HEADERS]
    deps += [os.path.join(ROOT, "include", "jepa.h"), os.path.join(ROOT, "synth", "jepa_synth.h")]
    return deps


def _stale(target, sources) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    deps = _deps()
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + deps):
            jobs.append([nvcc()] + _flags() + list(extra_flags) + ["-c", s, "-o", o])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            futs = [ex.submit(subprocess.run, cmd, capture_output=True, text=True) for cmd in jobs]
            for cmd, f in zip(jobs, futs):
                r = f.result()
                if verbose or r.returncode:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc()] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
        if r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link of libjepa_gb300.so failed")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ())
    print(LIB)
