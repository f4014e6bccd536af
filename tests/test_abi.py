"""The C-ABI library builds, loads and exports every entry point include/moe.h declares, and
its host-side validation rejects bad arguments before touching a GPU.  CPU only: no call here
launches a kernel."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_batches_gb300 import build, load_library
    build.build()
    return load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_layer_entry_points():
    names = declared_functions()
    for required in ("moe_plan_create", "moe_layer_forward", "moe_route", "moe_permute", "moe_combine",
                     "moe_route_logits", "moe_plan_destroy", "moe_plan_set_weights", "moe_plan_set_workspace"):
        assert required in names


def _params(name):
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
    assert m, name
    return [" ".join(p.split()) for p in m.group(1).split(",")]


def test_combine_takes_fp32_expert_outputs():
    """The boundary's combine call takes y and shared_y as fp32 (the layer keeps its own
    intermediates in fp16 and calls the kernel internally)."""
    params = _params("moe_combine")
    assert params[1] == "const float* y" and params[4] == "const float* shared_y", params
    assert params[2] == "const float* gates" and params[3] == "const int32_t* inv_perm"


def test_every_declaration_cites_its_source_or_says_it_has_none():
    """Each entry point's comment names the page passage it implements, or states that the pages
    have no counterpart."""
    text = open(os.path.join(ROOT, "include", "moe.h")).read()
    for name in declared_functions():
        m = re.search(r"\n[a-z_ *]*\b" + name + r"\s*\(", text)
        assert m, name
        lines = text[:m.start()].split("\n")
        i = len(lines)                         # back to the end of the previous declaration
        while i > 0 and not (lines[i - 1].rstrip().endswith(");") and not lines[i - 1].lstrip().startswith("*")
                             and "/*" in "\n".join(lines[i:])):
            i -= 1                             # (declarations that share one comment share its citation)
        doc = "\n".join(lines[i:])
        assert ('"' in doc) or ("no counterpart" in " ".join(doc.lower().replace("*", " ").split())), name


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libmoe.so does not export {name}"
    import decode_batches_gb300 as pkg
    assert set(pkg.EXPORTED) <= set(declared_functions())


def test_plan_create_validates_shapes(lib):
    bad = [(0, 1, 64, 64, 0, 0), (8, 9, 64, 64, 0, 0), (2000, 8, 64, 64, 0, 0), (8, 2, 60, 64, 0, 0),
           (8, 2, 64, 64, 0, 1 + 1), (8, 2, 48, 64, 0, 1), (8, 40, 64, 64, 0, 0), (8, 2, 64, 64, -1, 0)]
    for args in bad:
        assert lib.moe_plan_create(*args) is None, args
        assert lib.moe_last_error()
    p = lib.moe_plan_create(8, 2, 256, 512, 0, 0)
    assert p
    lib.moe_plan_destroy(p)
    lib.moe_plan_destroy(None)


def test_entry_points_reject_bad_arguments_before_any_launch(lib):
    from decode_batches_gb300 import MOE_ERR_INVALID_ARG, MOE_ERR_NOT_READY, MOE_ERR_UNSUPPORTED
    p = lib.moe_plan_create(8, 2, 256, 512, 1, 0)
    try:
        assert lib.moe_plan_set_weights(p, None, None, None, None, None, None, None, None) == MOE_ERR_INVALID_ARG
        assert lib.moe_layer_forward(p, None, 4, 0, None, None) == MOE_ERR_NOT_READY
        assert lib.moe_layer_forward(None, None, 4, 0, None, None) == MOE_ERR_INVALID_ARG
        assert lib.moe_route(p, None, -1, None, None, None, None) == MOE_ERR_INVALID_ARG
        assert lib.moe_plan_set_shared(p, 12, None, None, None) == MOE_ERR_INVALID_ARG
        assert lib.moe_plan_set_path(p, 7) == MOE_ERR_INVALID_ARG
        assert lib.moe_plan_set_path(p, 1) == 0
        assert lib.moe_combine(p, None, None, None, None, 0, None, None) == 0          # T = 0 is a no-op
        assert lib.moe_combine(p, None, None, None, None, 3, None, None) == MOE_ERR_INVALID_ARG
        b1, b2 = lib.moe_plan_workspace_bytes(p, 16), lib.moe_plan_workspace_bytes(p, 4096)
        assert 0 < b1 < b2
        assert b"required" in lib.moe_last_error() or lib.moe_last_error()
    finally:
        lib.moe_plan_destroy(p)
    q = lib.moe_plan_create(8, 2, 96, 64, 0, 0)          # d not a multiple of 128: no tensor-core path
    try:
        assert lib.moe_plan_set_path(q, 2) == MOE_ERR_UNSUPPORTED
    finally:
        lib.moe_plan_destroy(q)
