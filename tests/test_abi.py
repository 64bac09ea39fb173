"""The C-ABI library loads (no GPU needed), exports every symbol include/cosa.h declares,
and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_long_gb300 import build
    build.build()
    from block_sparse_long_gb300 import cosa as C
    return C


def declared_functions():
    text = open(os.path.join(ROOT, "include", "cosa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cosa_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    assert "cosa_proxy_select" in names and "cosa_sparse_prefill" in names
    assert len(names) == 7


def test_exports_every_declared_symbol(lib):
    L = lib.library()
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(declared_functions()) == set(lib.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (cosa_\w+)", out))
    assert exported == set(declared_functions())


def test_no_driver_or_runtime_link(lib):
    out = subprocess.run(["ldd", lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = lib.cosa_status_string(code)
        assert s and s != "unknown status"
    assert lib.cosa_status_string(12345) == "unknown status"
    assert lib.cosa_version() >= 1


def _params(lib, **kw):
    base = dict(num_reqs=1, num_q_heads=4, num_kv_heads=2, head_dim=128, block_size=128, page_size=64, stride=16,
                total_tokens=1000, max_seqlen=1000, num_pages=16, max_pages_per_req=16, mask_pitch=8,
                budget_ppm=500_000, sm_scale=0.088, skip_delta=-1.0)
    base.update(kw)
    return lib.make_params(**base)


def test_host_validation(lib):
    L = lib.library()
    fake = ctypes.c_void_p(4096)
    def kap(p, ws_bytes=1 << 30, q=fake):
        return L.cosa_proxy_select(ctypes.byref(p), q, fake, fake, fake, fake, fake, fake, ws_bytes, None, None)
    def osk(p, q=fake):
        return L.cosa_sparse_prefill(ctypes.byref(p), q, fake, fake, fake, fake, fake, fake, fake, None, None, 0,
                                     None, None)
    assert kap(_params(lib, head_dim=96)) == lib.COSA_ERR_UNSUPPORTED
    assert kap(_params(lib, block_size=96)) == lib.COSA_ERR_UNSUPPORTED
    assert kap(_params(lib, page_size=256)) == lib.COSA_ERR_UNSUPPORTED
    assert kap(_params(lib, stride=64)) == lib.COSA_ERR_UNSUPPORTED          # two samples per block
    assert kap(_params(lib, num_q_heads=3)) == lib.COSA_ERR_INVALID_ARG
    assert kap(_params(lib, budget_ppm=0)) == lib.COSA_ERR_INVALID_ARG
    assert kap(_params(lib, mask_pitch=3)) == lib.COSA_ERR_INVALID_ARG       # K_i up to 4 at 50 % of 8 blocks
    assert kap(_params(lib, max_pages_per_req=15)) == lib.COSA_ERR_INVALID_ARG
    assert kap(_params(lib), q=None) == lib.COSA_ERR_INVALID_ARG
    assert kap(_params(lib), q=ctypes.c_void_p(4097)) == lib.COSA_ERR_INVALID_ARG   # misaligned
    assert kap(_params(lib), ws_bytes=16) == lib.COSA_ERR_WORKSPACE
    assert kap(_params(lib, max_seqlen=128 * 4097, total_tokens=10, max_pages_per_req=8194,
                       mask_pitch=4097)) == lib.COSA_ERR_UNSUPPORTED
    assert osk(_params(lib, head_dim=80)) == lib.COSA_ERR_UNSUPPORTED
    assert osk(_params(lib, sm_scale=0.0)) == lib.COSA_ERR_INVALID_ARG
    assert osk(_params(lib), q=None) == lib.COSA_ERR_INVALID_ARG
    assert osk(_params(lib, flags=1 << 5)) == lib.COSA_ERR_INVALID_ARG      # unknown flag bit
    assert kap(_params(lib, flags=1 << 5)) == lib.COSA_ERR_INVALID_ARG
    assert kap(_params(lib, flags=lib.COSA_FLAG_TOP_P, mask_pitch=7)) == lib.COSA_ERR_INVALID_ARG   # K_i up to 8
    assert osk(_params(lib, total_tokens=0)) == lib.COSA_OK                 # nothing to do
    # the GQA page-union kernel serves 128-token blocks of ID-list masks only
    assert osk(_params(lib, flags=lib.COSA_FLAG_GQA_UNION, block_size=64, stride=8)) == lib.COSA_ERR_UNSUPPORTED
    assert osk(_params(lib, flags=lib.COSA_FLAG_GQA_UNION | lib.COSA_FLAG_BINARY_MASK)) == lib.COSA_ERR_UNSUPPORTED
    assert osk(_params(lib, flags=lib.COSA_FLAG_GQA_UNION, total_tokens=0)) == lib.COSA_OK


def test_kap_stride_validation(lib):
    """A stride of 0, or one that does not divide the block, is refused by the workspace query and
    by both select calls before any size is computed (no division by the stride on the host)."""
    L = lib.library()
    fake = ctypes.c_void_p(4096)
    for stride, code in ((0, lib.COSA_ERR_INVALID_ARG), (3, lib.COSA_ERR_INVALID_ARG),
                         (-16, lib.COSA_ERR_INVALID_ARG), (64, lib.COSA_ERR_UNSUPPORTED)):
        p = _params(lib, stride=stride)
        assert lib.cosa_proxy_workspace_size(p) == 0, stride
        rc = L.cosa_proxy_select(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, 1 << 30, None, None)
        assert rc == code, (stride, rc)
        rc = L.cosa_proxy_select_static(ctypes.byref(p), fake, fake, fake, fake, fake, fake, None, None)
        assert rc == code, (stride, rc)
    # a budget or mask pitch the select calls refuse gives no workspace size either
    assert lib.cosa_proxy_workspace_size(_params(lib, budget_ppm=0)) == 0
    assert lib.cosa_proxy_workspace_size(_params(lib, mask_pitch=3)) == 0


def test_workspace_sizes(lib):
    p = _params(lib)
    n = lib.cosa_proxy_workspace_size(p)
    assert n > 0 and n % 1 == 0
    big = lib.cosa_proxy_workspace_size(_params(lib, total_tokens=131072, max_seqlen=131072,
                                                 max_pages_per_req=2048, mask_pitch=1024, num_q_heads=32,
                                                 num_kv_heads=8))
    assert big > n
    assert lib.cosa_proxy_workspace_size(_params(lib, head_dim=96)) == 0
    assert lib.cosa_prefill_workspace_size(p) == 0
