"""The DRAM-traffic record that bench.py reports is keyed by the gradient
return kernels' device code: host launch edits keep it, kernel edits void it,
and the committed record matches the committed kernels."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = os.path.join(ROOT, "context_attention_token_gb300", "csrc", "grad_return.cu")


def _text():
    with open(SRC) as f:
        return f.read()


def test_device_code_holds_every_kernel_and_constant():
    code = bench._device_code(_text())
    assert "grad_return_kernel(const GradReturnParams p)" in code
    assert "grad_return_bulk_kernel(const GradReturnParams p)" in code
    assert "constexpr int kBulkWarps" in code
    assert "cudaOccupancyMaxActiveBlocksPerMultiprocessor" not in code  # host launch code


def test_host_edit_keeps_and_kernel_edit_changes_the_key():
    text = _text()
    base = bench._device_code(text)
    host = text.replace("cudaError_t launch_grad_return(", "// note\ncudaError_t launch_grad_return(", 1)
    assert host != text and bench._device_code(host) == base
    i = text.index("grad_return_bulk_kernel(const GradReturnParams p)")
    j = text.index("add_rn", i)
    kernel = text[:j] + "add_rn_x" + text[j + len("add_rn"):]
    assert bench._device_code(kernel) != base


def test_committed_record_matches_committed_kernels():
    value, note = bench.profiled_traffic("grad_return", 262144)
    assert value is not None, note
