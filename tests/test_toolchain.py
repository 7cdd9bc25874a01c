"""What the sm_103a toolchain accepts for the prefill GEMM's tensor-core path.

The W8A8 variant's natural prefill form would multiply int8 codes on the
5th-generation tensor cores (tcgen05.mma kind::i8).  ptxas accepts that
instruction for sm_100a but rejects it for sm_103a (GB300), so the M > 32
path stays on kind::f16 (bf16 operands).  Compile-only checks (nvcc
cross-compiles here without a GPU); the kernels are one instruction each.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

KERNEL = r"""
#include <cstdint>
__global__ void k(uint32_t tm, uint64_t da, uint64_t db, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %%4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::%s [%%0], %%1, %%2, %%3, p;\n\t}"
                 :: "r"(tm), "l"(da), "l"(db), "r"(idesc), "r"(1));
}
"""


def _compile(kind, arch):
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "k.cu")
        with open(src, "w") as f:
            f.write(KERNEL % kind)
        r = subprocess.run([NVCC, "-gencode", f"arch=compute_{arch},code=sm_{arch}", "-c", src, "-o",
                            os.path.join(d, "k.o")], capture_output=True, text=True)
        return r.returncode, r.stdout + r.stderr


pytestmark = pytest.mark.skipif(not (os.path.exists(NVCC) or shutil.which("nvcc")), reason="nvcc not found")


def test_kind_f16_compiles_for_sm103a():
    rc, out = _compile("f16", "103a")
    assert rc == 0, out


def test_kind_i8_is_rejected_for_sm103a():
    rc, out = _compile("i8", "103a")
    assert rc != 0 and "kind::i8" in out and "sm_103a" in out, out


def test_kind_i8_compiles_for_sm100a():
    rc, out = _compile("i8", "100a")
    assert rc == 0, out
