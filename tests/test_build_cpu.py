"""The kernel-source digest (which stamps the committed DRAM-traffic records) is the same in any
checkout: it hashes the sources and the build flags, with the include directory written relative
to the repository."""
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def digest_in(root):
    code = ("import sys; sys.path.insert(0, sys.argv[1]); "
            "from exact_attention_fa_gb300 import build; print(build.source_digest())")
    out = subprocess.run([sys.executable, "-c", code, root], capture_output=True, text=True,
                         check=True, env={**os.environ, "FA_NVCC_EXTRA": ""})
    return out.stdout.strip()


def test_source_digest_does_not_depend_on_the_checkout_path(tmp_path):
    copy = tmp_path / "elsewhere" / "checkout"
    pkg = copy / "exact_attention_fa_gb300"
    (pkg / "csrc").mkdir(parents=True)
    for f in ("__init__.py", "build.py", "binding.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "exact_attention_fa_gb300", f), pkg / f)
    for f in os.listdir(os.path.join(ROOT, "exact_attention_fa_gb300", "csrc")):
        if f.endswith((".cu", ".cuh", ".h")):
            shutil.copy(os.path.join(ROOT, "exact_attention_fa_gb300", "csrc", f), pkg / "csrc" / f)
    shutil.copytree(os.path.join(ROOT, "include"), copy / "include")
    assert digest_in(str(copy)) == digest_in(ROOT)


def test_source_digest_changes_with_a_kernel_source(tmp_path):
    copy = tmp_path / "co"
    shutil.copytree(os.path.join(ROOT, "exact_attention_fa_gb300"), copy / "exact_attention_fa_gb300",
                    ignore=shutil.ignore_patterns("_build", "*.so", "__pycache__"))
    shutil.copytree(os.path.join(ROOT, "include"), copy / "include")
    before = digest_in(str(copy))
    with open(copy / "exact_attention_fa_gb300" / "csrc" / "fa_api.cu", "a") as f:
        f.write("\n// edited\n")
    assert digest_in(str(copy)) != before
