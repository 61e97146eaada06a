"""The C-ABI library builds, loads without a GPU and exports every entry point
that include/*.h declares; host-side argument checks reject bad calls before
any launch.  No GPU needed (no compute call reaches a kernel)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from tree_verify_linear_gb300 import build, lbx
    build.build()
    return lbx.load()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"\b(lbx_\w+)\s*\(", text)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "lbx_verify_step" in names and len(names) >= 6
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_every_declared_symbol():
    from tree_verify_linear_gb300 import lbx
    assert sorted(lbx.EXPORTS) == declared_functions()


def declared_arity():
    """Parameter count of every function include/*.h declares."""
    arity = {}
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for name, params in re.findall(r"\b(lbx_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
            params = params.strip()
            arity[name] = 0 if params in ("", "void") else params.count(",") + 1
    return arity


def test_binding_argument_counts_match_the_header(lib):
    """Each ctypes prototype the binding sets has as many arguments as the C
    declaration (a mismatch would shift every argument after it)."""
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, n in arity.items():
        assert len(getattr(lib, name).argtypes) == n, (name, len(getattr(lib, name).argtypes), n)


def test_strerror_and_workspace(lib):
    from tree_verify_linear_gb300 import lbx
    assert lbx.strerror(0) == "ok"
    assert "tree" in lbx.strerror(lbx.LBX_ETREE)
    cfg = lbx.make_cfg(48, 5, 22, 16, 48, 128, 4, 7)
    assert lbx.lbx_workspace_size(cfg) >= 48 * 5 * 16 * 4
    assert lbx.lbx_workspace_size(cfg) % 256 == 0


@pytest.mark.parametrize("field,value", [("d", 48), ("Hv", 47), ("K", 5), ("K", 0), ("N", 0),
                                         ("n_slots", 0), ("L", 0)])
def test_bad_config_rejected_on_host(lib, field, value):
    from tree_verify_linear_gb300 import lbx
    cfg = lbx.make_cfg(1, 1, 8, 2, 4, 32, 4, 1)
    setattr(cfg, field, value)
    assert lbx.lbx_workspace_size(cfg) == 0
    # the checks run before any pointer is touched, so NULL pointers are safe here
    rc = lib.lbx_verify_step(ctypes.byref(cfg), *([None] * 10), None, 0, None, None)
    assert rc == lbx.LBX_EINVAL


def test_null_pointers_and_limits_rejected_on_host(lib):
    from tree_verify_linear_gb300 import lbx
    cfg = lbx.make_cfg(1, 1, 8, 2, 4, 32, 4, 1)
    assert lib.lbx_verify_step(ctypes.byref(cfg), *([None] * 10), None, 0, None, None) == \
        lbx.LBX_EINVAL
    assert lib.lbx_tree_conv(ctypes.byref(cfg), *([None] * 8)) == lbx.LBX_EINVAL
    assert lib.lbx_tree_deltanet(ctypes.byref(cfg), *([None] * 10)) == lbx.LBX_EINVAL
    assert lib.lbx_tree_persist(ctypes.byref(cfg), *([None] * 9)) == lbx.LBX_EINVAL
    big = lbx.make_cfg(1, 1, lbx.LBX_MAX_TREE_NODES + 1, 2, 4, 32, 4, 1, mode=lbx.LBX_MODE_TREE)
    fake = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: rejected first
    args = [fake] * 10
    assert lib.lbx_verify_step(ctypes.byref(big), *args, fake, 1 << 20, None, None) == \
        lbx.LBX_EINVAL
    assert lib.lbx_tree_conv(ctypes.byref(big), *([fake] * 6), None, None) == lbx.LBX_EINVAL
