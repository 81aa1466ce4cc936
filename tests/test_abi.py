"""The C-ABI library builds, loads and exports every symbol its header
declares (no compute: this runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(dspark_\w+)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ["dspark_walk_create", "dspark_walk_run", "dspark_walk_run_host",
              "dspark_walk_status", "dspark_walk_get_plan", "dspark_walk_set_limits",
              "dspark_walk_strerror", "dspark_walk_destroy"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    from serial_draft_head_gb300 import walk
    L = walk.load(build_if_missing=True)
    lib = ctypes.CDLL(walk.library_path())
    for n in declared_symbols():
        assert hasattr(lib, n), "%s declared but not exported" % n
    assert set(walk.EXPORTS) <= set(declared_symbols())
    assert L.dspark_walk_strerror(-4).decode() == "cross-CTA rendezvous timed out"


def test_plan_struct_matches_header():
    from serial_draft_head_gb300 import walk
    text = open(os.path.join(ROOT, "include", "dspark_walk.h")).read()
    body = text[text.index("struct dspark_walk_plan {"):]
    body = body[:body.index("};")]
    fields = re.findall(r"^\s*(int64_t|int)\s+(\w+);", body, flags=re.M)
    assert [f for _, f in fields] == [n for n, _ in walk.dspark_walk_plan._fields_]


def test_create_without_a_device_fails_cleanly():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    from serial_draft_head_gb300 import walk
    with pytest.raises(walk.WalkError):
        walk.dspark_walk_create(16, 16, 100, 256, 1, 1)


def test_binding_constants_match_the_header():
    """Every DSPARK_* value the header defines has the same value in the binding."""
    from serial_draft_head_gb300 import walk
    text = open(os.path.join(ROOT, "include", "dspark_walk.h")).read()
    defs = re.findall(r"^#define DSPARK_(\w+)\s+\(?(-?\d+)\)?", text, flags=re.M)
    assert len(defs) >= 20
    for name, value in defs:
        assert hasattr(walk, name), "DSPARK_%s has no binding constant" % name
        assert getattr(walk, name) == int(value), "DSPARK_%s differs" % name
