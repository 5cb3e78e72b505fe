"""The usage example in the binding's module docstring stays in step with the binding: it runs on the CPU under
tests/fake_cuda.py (host stand-ins for CUDA, the library stubbed), so every call in it passes the binding's
argument and buffer checks.  The numbers it computes there are meaningless."""
import os
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _example():
    from decode_attention_19_b300 import binding
    doc = binding.__doc__
    at = doc.index("::\n")
    return textwrap.dedent(doc[at + 3:])


def test_binding_example_passes_the_binding_checks():
    code = "import sys\nsys.path[:0] = [%r, %r]\nimport fake_cuda\nfake_cuda.install()\n" % (
        os.path.join(ROOT, "tests"), ROOT) + _example()
    assert "lowram_decode_attn(" in code
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
