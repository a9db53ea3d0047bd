"""Layout rules the product keeps: the oracle is reached only from the tests, the smoke entry and
the benchmark; nothing product-side reads the scratch folder; profiles hold text summaries only."""
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SKIP_DIRS = {".git", "_work", "gpurun_out", "_build", "__pycache__", ".pytest_cache", "baseline"}


def _files(top, exts):
    for d, dirs, files in os.walk(os.path.join(ROOT, top)):
        dirs[:] = [x for x in dirs if x not in SKIP_DIRS]
        for f in files:
            if f.endswith(exts):
                yield os.path.join(d, f)


def _text(p):
    with open(p, encoding="utf-8", errors="replace") as f:
        return f.read()


def test_product_code_does_not_reach_the_oracle():
    """The library, its binding and the input recipes never import, load or include the oracle."""
    pat = re.compile(r"\boracle\b")
    for top in ("chunkwise_linear_attention_gb300", "workloads", "include"):
        for p in _files(top, (".py", ".cu", ".cuh", ".h", ".c", ".cpp")):
            for line in _text(p).splitlines():
                s = line.strip()
                if s.startswith(("import", "from")) or "#include" in s or "CDLL" in s or "liboracle" in s:
                    assert not pat.search(s), f"{os.path.relpath(p, ROOT)}: {s}"


def test_oracle_does_not_reach_the_product():
    """The oracle shares no code with the CUDA path: no include of the library's headers or sources,
    no import of the package."""
    for p in _files("oracle", (".py", ".c", ".h")):
        t = _text(p)
        assert "chunkwise_linear_attention_gb300" not in t, p
        assert "cla.h" not in t and "csrc" not in t, p


def test_nothing_committed_reads_the_scratch_folder():
    for top in ("chunkwise_linear_attention_gb300", "workloads", "oracle", "tests", "include", "profiles"):
        for p in _files(top, (".py", ".cu", ".cuh", ".h", ".c", ".md", ".txt", ".json")):
            if os.path.abspath(p) == os.path.abspath(__file__):
                continue
            assert "_work/" not in _text(p), os.path.relpath(p, ROOT)
    for f in ("bench.py", "__graft_entry__.py"):
        assert "_work/" not in _text(os.path.join(ROOT, f)), f


def test_profiles_hold_text_summaries_only():
    for f in os.listdir(os.path.join(ROOT, "profiles")):
        assert f.endswith((".md", ".txt", ".json")), f
        assert os.path.getsize(os.path.join(ROOT, "profiles", f)) < 64 * 1024, f
