"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/polestar.h declares, sizes workspaces, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cdll():
    from drift_aware_kv_spherical_gb300 import _build, polestar
    if not os.path.exists(polestar.LIB_PATH):
        _build.build()
    return polestar.Library.load().cdll


def _declared():
    src = open(os.path.join(ROOT, "include", "polestar.h")).read()
    return sorted(set(re.findall(r"^\s*(?:ps_status|size_t|int|const char\*)\s+(ps_\w+)\(",
                                 src, re.M)))


def test_every_declared_symbol_is_exported(cdll):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(cdll, n), n


def test_workspace_sizes_are_shape_only(cdll):
    from drift_aware_kv_spherical_gb300 import polestar as ps
    a = ps.ps_workspace_bytes(ps.OP_KMEANS, B=1, N=1024, d=4096, C=64)
    assert a > 0 and a % 256 == 0
    assert ps.ps_workspace_bytes(ps.OP_KMEANS, B=0, N=1024, d=4096, C=64) == 0
    assert ps.ps_workspace_bytes(ps.OP_TOPK, B=4, N=10, C=2, k=1) == 0
    assert ps.ps_workspace_bytes(ps.OP_PROXY_KL, B=1, N=1024, d=4096, C=64, Hq=32,
                                 Hkv=32, dh=128) >= 64 * 4096 * 4
    assert ps.ps_workspace_bytes(ps.OP_COMMIT, B=1, P=32, V=126464) > 0


def test_status_strings(cdll):
    for s in range(6):
        assert cdll.ps_status_string(s)


def test_null_handle_and_bad_args_rejected_on_host(cdll):
    from drift_aware_kv_spherical_gb300 import polestar as ps
    # every op returns PS_ERR_ARG for a NULL handle before any CUDA call
    assert cdll.ps_kmeans_spherical(None, None, 0, 1, 8, 16, 2, 1, 0, None, None, None,
                                    None, None, None, None, None, 0, None) == ps.PS_ERR_ARG
    assert cdll.ps_topk_drift(None, None, None, None, 1, 8, 2, 1, None, None, None, None,
                              None, None, 0, None) == ps.PS_ERR_ARG
    assert cdll.ps_commit(None, None, 0, 1, 2, 8, None, None, None, 2, None, None, None,
                          None, 2, ps.CommitParams(0.9, 1, 0.1, 0, 1), None, None, None,
                          None, 0, None) == ps.PS_ERR_ARG
    h = ctypes.c_void_p()
    st = cdll.ps_create(-1, ctypes.byref(h))
    assert st == ps.PS_ERR_ARG
