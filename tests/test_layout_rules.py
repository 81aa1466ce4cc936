"""Repository rules that the code must keep (no GPU): the library and its
binding never reach the oracle, and nothing committed reads the git-ignored
scratch folder."""
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _tracked(suffixes):
    out = subprocess.run(["git", "ls-files"], cwd=ROOT, capture_output=True, text=True)
    if out.returncode != 0:
        files = []
        for d, _, fs in os.walk(ROOT):
            if "/." in d or "/_work" in d:
                continue
            files += [os.path.relpath(os.path.join(d, f), ROOT) for f in fs]
    else:
        files = out.stdout.split()
    return [f for f in files if f.endswith(suffixes)]


def test_library_never_imports_the_oracle():
    for f in _tracked((".py", ".cu", ".cuh", ".h", ".c")):
        if not f.startswith(("serial_draft_head_gb300/", "include/")):
            continue
        text = open(os.path.join(ROOT, f)).read()
        assert not re.search(r"^\s*(import|from)\s+oracle\b", text, flags=re.M), f
        assert "oracle.h" not in text and "liboracle" not in text, f


def test_nothing_committed_uses_the_scratch_folder():
    for f in _tracked((".py", ".cu", ".cuh", ".h", ".c", ".sh", ".toml", ".cfg", ".txt")):
        if f.startswith("_work/") or f == "tests/test_layout_rules.py":
            continue
        text = open(os.path.join(ROOT, f), errors="replace").read()
        assert not re.search(r"(^|[\s'\"/(])_work/", text), f
