"""The Python example in README.md runs as written and computes what the
README says: the partition puts rank r's tokens in q_local[r], and the
gradient return is the ordered binary32 sum of the writers' rows."""
import os
import re

import pytest
import torch

pytestmark = pytest.mark.gpu

README = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")


def test_readme_example_runs_and_is_right(cpt, cuda_device):
    with open(README) as f:
        blocks = re.findall(r"```python\n(.*?)```", f.read(), flags=re.S)
    assert len(blocks) == 1
    env = {}
    exec(compile(blocks[0], "README.md", "exec"), env)
    torch.cuda.synchronize()
    P, S = env["P"], env["S"]
    plan = env["plan"]
    l2g = torch.empty(S, dtype=torch.int32, device="cuda")
    cpt.cpt_index_map(plan, l2g, None)
    idx = l2g.long()
    assert torch.equal(env["q_local"].view(S, 20, 128), env["q"].index_select(0, idx))
    w = env["dk_writers"]
    acc = w[0].index_select(0, idx).float()
    for k in range(1, P):
        acc = acc + w[k].index_select(0, idx).float()
    assert torch.equal(acc.bfloat16().view(torch.int16), env["dk_owner"].view(S, 20, 128).view(torch.int16))


def test_readme_c_example_builds_and_runs(cpt, cuda_device):
    """The C block of README.md, built as the README says (gcc, then nvcc to
    link the CUDA runtime), runs on the GPU and prints ok: every owner
    element is the ordered sum 1 + 2 + 3 + 4."""
    import shutil
    import subprocess

    gcc, nvcc = shutil.which("gcc"), shutil.which("nvcc")
    if gcc is None or nvcc is None:
        pytest.skip("needs gcc and nvcc")
    with open(README) as f:
        blocks = re.findall(r"```c\n(.*?)```", f.read(), flags=re.S)
    assert len(blocks) == 1
    root = os.path.dirname(README)
    work = os.path.join(root, "_build", "readme_c")  # the build folder, kept out of git
    os.makedirs(work, exist_ok=True)
    src, obj, exe = (os.path.join(work, n) for n in ("example.c", "example.o", "example"))
    with open(src, "w") as f:
        f.write(blocks[0])
    cuda_home = os.path.dirname(os.path.dirname(nvcc))
    lib_dir = os.path.dirname(cpt._LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"), "-I",
                    os.path.join(cuda_home, "include"), "-c", src, "-o", obj], check=True)
    subprocess.run([nvcc, obj, "-o", exe, "-L", lib_dir, "-lcpt", "-Xlinker", f"-rpath,{lib_dir}"], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.strip() == "ok"
