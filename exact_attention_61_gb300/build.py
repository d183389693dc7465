"""Build the sm_103a CUDA library ``libattn.so`` in-tree with nvcc.

Translation units (compiled in parallel, then linked into one shared library
with the CUDA runtime linked statically):
  attn_host.cu                       C ABI, validation, tensor maps, dispatch
  attn_static_scratch.cu             device scratch of attn_fwd_kv_static (own module)
  probe.cu                           one-tile tensor-core probe (test hook)
  attn_merge.cu                      merge of split-key partials
  attn_decode.cu                     streaming decode kernel (up to 4 query rows)
  attn_fwd_inst.cu x 4               forward kernel, one unit per (d, dtype)
  attn_bwd_aux.cu                    backward prologue (D, lse2) and dQ cast
  attn_bwd_inst.cu x 4               backward kernel, one unit per (d, dtype)
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", f"-I{INCLUDE}"]

UNITS = [
    ("attn_host.cu", [], "attn_host.o"),
    ("attn_static_scratch.cu", [], "attn_static_scratch.o"),
    ("probe.cu", [], "probe.o"),
    ("attn_merge.cu", [], "attn_merge.o"),
    ("attn_decode.cu", [], "attn_decode.o"),
    ("attn_fwd_inst.cu", ["-DATTN_INST_D=64", "-DATTN_INST_BF16=0"], "attn_fwd_d64_f16.o"),
    ("attn_fwd_inst.cu", ["-DATTN_INST_D=64", "-DATTN_INST_BF16=1"], "attn_fwd_d64_bf16.o"),
    ("attn_fwd_inst.cu", ["-DATTN_INST_D=128", "-DATTN_INST_BF16=0"], "attn_fwd_d128_f16.o"),
    ("attn_fwd_inst.cu", ["-DATTN_INST_D=128", "-DATTN_INST_BF16=1"], "attn_fwd_d128_bf16.o"),
    ("attn_bwd_aux.cu", [], "attn_bwd_aux.o"),
    ("attn_bwd_inst.cu", ["-DATTN_INST_D=64", "-DATTN_INST_BF16=0"], "attn_bwd_d64_f16.o"),
    ("attn_bwd_inst.cu", ["-DATTN_INST_D=64", "-DATTN_INST_BF16=1"], "attn_bwd_d64_bf16.o"),
    ("attn_bwd_inst.cu", ["-DATTN_INST_D=128", "-DATTN_INST_BF16=0"], "attn_bwd_d128_f16.o"),
    ("attn_bwd_inst.cu", ["-DATTN_INST_D=128", "-DATTN_INST_BF16=1"], "attn_bwd_d128_bf16.o"),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def _newest_source() -> float:
    files = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every unit that is out of date, then link ``libattn.so``."""
    os.makedirs(BUILD, exist_ok=True)
    newest = _newest_source()
    cc = nvcc()
    procs = []
    for src, defs, obj in UNITS:
        out = os.path.join(BUILD, obj)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
            continue
        cmd = [cc, *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", out]
        log = open(os.path.join(BUILD, obj + ".log"), "w")
        procs.append((obj, cmd, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for obj, cmd, p, log in procs:
        rc = p.wait()
        log.close()
        if rc != 0:
            failed.append(obj)
            with open(os.path.join(BUILD, obj + ".log")) as f:
                sys.stderr.write(f"--- nvcc failed for {obj}:\n{' '.join(cmd)}\n{f.read()}\n")
        elif verbose:
            print(f"built {obj}")
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    objs = [os.path.join(BUILD, obj) for _, _, obj in UNITS]
    if force or procs or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(map(os.path.getmtime, objs)):
        fd, tmp = tempfile.mkstemp(suffix=".so", dir=BUILD)
        os.close(fd)
        subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
