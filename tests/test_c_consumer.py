"""A plain C program builds against include/cpt.h and libcpt.so and calls the
host-side entry points: the ABI needs no C++ and no Python."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "cpt.h"

int main(void)
{
    const int32_t cu[4] = {0, 16, 40, 64};
    if (cpt_validate_layout(CPT_LAYOUT_DUAL_CHUNK_SWAP, 2, cu, 3, 64) != CPT_OK) return 1;
    if (cpt_validate_layout(CPT_LAYOUT_DUAL_CHUNK_SWAP, 3, cu, 3, 64) != CPT_ERR_NOT_DIVISIBLE) return 2;
    if (strlen(cpt_last_error_string()) == 0) return 3;
    if (cpt_plan_workspace_bytes(CPT_LAYOUT_DUAL_CHUNK_SWAP, 2, 3, 64) == 0) return 4;
    cpt_kernel_path k = CPT_KERNEL_LOADS;
    if (cpt_kernel_path_of(CPT_CALL_GRAD_RETURN, 4, CPT_BF16, CPT_BF16, 0, 5120, 2 * 262144, &k) != CPT_OK)
        return 5;
    if (k != CPT_KERNEL_BULK) return 6;
    printf("%s|%s\n", cpt_status_string(CPT_OK), cpt_status_string(CPT_ERR_NOT_DIVISIBLE));
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_builds_and_runs(cpt):
    lib_dir = os.path.dirname(cpt._LIB_PATH)
    work = os.path.join(ROOT, "_build", "c_consumer")  # the build folder, kept out of git
    os.makedirs(work, exist_ok=True)
    src = os.path.join(work, "consumer.c")
    exe = os.path.join(work, "consumer")
    with open(src, "w") as f:
        f.write(PROGRAM)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src,
                    "-o", exe, "-L", lib_dir, "-lcpt", f"-Wl,-rpath,{lib_dir}"], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    ok, nd = out.stdout.strip().split("|")
    assert ok and nd and ok != nd
