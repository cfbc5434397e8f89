"""Build libbq.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit compiles in parallel to an object file under
csrc/_build/, and the objects link into block_quantized_weight_row_gb300/libbq.so.
No CPU fallback is built: the library is CUDA-only.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ_DIR = os.path.join(CSRC, "_build")
LIB = os.path.join(HERE, "libbq.so")
# measurement probe (tensor-op rates for the roofline denominators); not part of the libbq ABI
PROBE_SRC = "probe_mma.cu"
PROBE_LIB = os.path.join(HERE, "libbq_probe.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["bq_api.cu", "quantize.cu", "gemv.cu", "gemv_seq.cu", "gemm.cu", "gemm_tc.cu", "gemm_noalloc.cu", "attn.cu",
           "attn_fixed_q4k.cu", "attn_fixed_q8k.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [os.path.join(INCLUDE, "bq.h"), __file__]


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(OBJ_DIR, exist_ok=True)
    cc = nvcc()
    deps = _deps()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + deps):
            jobs.append([cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    probe_src = os.path.join(CSRC, PROBE_SRC)
    probe_tmp = PROBE_LIB + f".tmp{os.getpid()}"
    build_probe = force or _stale(PROBE_LIB, [probe_src, __file__] + deps)
    if build_probe:
        jobs.append([cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-shared", probe_src, "-o", probe_tmp])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES) + 1) as ex:
        for out in ex.map(run, jobs):
            if verbose and out:
                print(out, file=sys.stderr)
    if build_probe:
        os.replace(probe_tmp, PROBE_LIB)
    if force or any("-c" in j for j in jobs) or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        run([cc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    flags = [a for a in sys.argv[1:] if a.startswith("-X")]
    print(build(force="--force" in sys.argv, verbose=True, extra_flags=flags))
