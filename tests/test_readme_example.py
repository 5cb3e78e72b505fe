"""The README's usage example stays in step with the binding: it runs on the CPU under tests/fake_cuda.py (host
stand-ins for CUDA, the library stubbed), so every call in it passes the binding's argument and buffer checks.
The numbers it computes there are meaningless."""
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_passes_the_binding_checks():
    text = open(os.path.join(ROOT, "README.md")).read()
    blocks = re.findall(r"```python\n(.*?)```", text, flags=re.S)
    assert blocks, "no python example in README.md"
    code = "import sys\nsys.path[:0] = [%r, %r]\nimport fake_cuda\nfake_cuda.install()\n" % (
        os.path.join(ROOT, "tests"), ROOT) + blocks[0]
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
