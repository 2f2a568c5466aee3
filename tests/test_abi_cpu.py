"""The C ABI library on a machine without a GPU: it builds, loads, exports
every function include/spconv.h declares, and rejects bad arguments before
touching the device."""
import ctypes
import os
import re

import pytest

import submanifold_voxel_gather_gb300 as sv
from submanifold_voxel_gather_gb300 import build as svbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spconv.h")


@pytest.fixture(scope="module")
def lib():
    svbuild.build()
    return sv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spconv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("spconv_build_nmap", "spconv_submconv3d", "spconv_build_nmap_workspace_size",
                     "spconv_last_error", "spconv_version", "spconv_count_valid_pairs",
                     "spconv_device_status", "spconv_submconv3d_ex", "spconv_submconv3d_dgrad",
                     "spconv_submconv3d_wgrad", "spconv_build_nmap_async", "spconv_tile_order",
                     "spconv_submconv3d_ordered"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_version_and_workspace_size(lib):
    assert sv.version() == 1
    assert sv.workspace_size(-1) == 0
    assert sv.workspace_size(0) == 256 + 64 * 16
    assert sv.workspace_size(32) == 256 + 64 * 16
    assert sv.workspace_size(33) == 256 + 128 * 16
    assert sv.workspace_size(11_773_199) == 256 + (1 << 25) * 16


def _status(code):
    return code, sv.load_library().spconv_last_error().decode()


def test_argument_validation_without_gpu(lib):
    offs = sv.default_offsets()
    optr = offs.ctypes.data_as(ctypes.c_void_p)
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: validation fails first
    # build_nmap
    assert _status(lib.spconv_build_nmap(fake, -1, optr, 27, fake, fake, 1 << 30, None))[0] == -1
    assert _status(lib.spconv_build_nmap(fake, 10, optr, 0, fake, fake, 1 << 30, None))[0] == -1
    assert _status(lib.spconv_build_nmap(fake, 10, None, 27, fake, fake, 1 << 30, None))[0] == -1
    assert _status(lib.spconv_build_nmap(None, 10, optr, 27, fake, fake, 1 << 30, None))[0] == -1
    code, msg = _status(lib.spconv_build_nmap(fake, 10, optr, 27, fake, fake, 100, None))
    assert code == -3 and "workspace" in msg
    code, msg = _status(lib.spconv_build_nmap(fake, 10, optr, 27, fake, ctypes.c_void_p(0x100010),
                                              1 << 30, None))
    assert code == -1 and "256-byte" in msg
    assert _status(lib.spconv_build_nmap(fake, 0, optr, 27, None, None, 0, None))[0] == 0
    # submconv3d
    assert _status(lib.spconv_submconv3d(fake, fake, fake, None, fake, -5, 27, 16, 16, 2, None))[0] == -1
    assert _status(lib.spconv_submconv3d(fake, fake, fake, None, fake, 10, 0, 16, 16, 2, None))[0] == -1
    assert _status(lib.spconv_submconv3d(fake, fake, fake, None, fake, 10, 27, 16, 16, 7, None))[0] == -1
    code, msg = _status(lib.spconv_submconv3d(fake, fake, fake, None, fake, 10, 27, 24, 16, 2, None))
    assert code == -2 and "multiples of 16" in msg
    code, msg = _status(lib.spconv_submconv3d(ctypes.c_void_p(0x100008), fake, fake, None, fake, 10, 27,
                                              16, 16, 2, None))
    assert code == -1 and "aligned" in msg
    assert _status(lib.spconv_submconv3d(None, fake, fake, None, fake, 10, 27, 16, 16, 0, None))[0] == -1
    assert _status(lib.spconv_submconv3d(None, None, None, None, None, 0, 27, 16, 16, 2, None))[0] == 0
    # submconv3d_ex: same checks plus the activation code and residual alignment
    ex = lib.spconv_submconv3d_ex
    assert _status(ex(fake, fake, fake, None, None, fake, 10, 27, 16, 16, 2, 3, None))[0] == -1
    assert _status(ex(fake, fake, fake, None, None, fake, 10, 27, 16, 16, 2, -1, None))[0] == -1
    code, msg = _status(ex(fake, fake, fake, None, ctypes.c_void_p(0x100001), fake, 10, 27, 16, 16, 2, 1,
                           None))
    assert code == -1 and "residual" in msg
    assert _status(ex(fake, fake, fake, None, None, fake, -5, 27, 16, 16, 2, 0, None))[0] == -1
    assert _status(ex(None, None, None, None, None, None, 0, 27, 16, 16, 2, 2, None))[0] == 0
    # submconv3d_dgrad: forward sizes, same checks
    dg = lib.spconv_submconv3d_dgrad
    assert _status(dg(fake, fake, fake, fake, -1, 27, 16, 16, 2, None))[0] == -1
    assert _status(dg(fake, fake, fake, fake, 10, 27, 24, 16, 2, None))[0] == -2
    assert _status(dg(None, fake, fake, fake, 10, 27, 16, 16, 2, None))[0] == -1
    assert _status(dg(None, None, None, None, 0, 27, 16, 16, 2, None))[0] == 0
    # submconv3d_wgrad
    wg = lib.spconv_submconv3d_wgrad
    assert _status(wg(fake, fake, fake, None, None, 10, 27, 16, 16, 2, None))[0] == -1
    assert _status(wg(fake, fake, fake, fake, None, 10, 27, 16, 16, 9, None))[0] == -1
    assert _status(wg(fake, fake, fake, ctypes.c_void_p(0x100002), None, 10, 27, 16, 16, 2, None))[0] == -1
    assert _status(wg(None, fake, fake, fake, None, 10, 27, 16, 16, 2, None))[0] == -1
    # build_nmap_async: host-side checks as build_nmap, plus the status pointer
    ba = lib.spconv_build_nmap_async
    assert _status(ba(fake, 10, optr, 27, fake, fake, 1 << 30, None, None))[0] == -1
    assert _status(ba(fake, 10, optr, 27, fake, fake, 1 << 30, ctypes.c_void_p(0x100002), None))[0] == -1
    assert _status(ba(fake, 10, optr, 27, fake, fake, 100, fake, None))[0] == -3
    assert _status(ba(fake, -1, optr, 27, fake, fake, 1 << 30, fake, None))[0] == -1
    # count
    assert _status(lib.spconv_count_valid_pairs(fake, 10, 27, None, None))[0] == -1


def test_order_entry_points_validate_without_gpu(lib):
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: validation fails first
    to = lib.spconv_tile_order
    assert _status(to(fake, -1, 27, fake, None))[0] == -1
    assert _status(to(fake, 10, 0, fake, None))[0] == -1
    assert _status(to(None, 10, 27, fake, None))[0] == -1
    assert _status(to(fake, 10, 27, None, None))[0] == -1
    assert _status(to(fake, 10, 27, ctypes.c_void_p(0x100002), None))[0] == -1
    assert _status(to(None, 0, 27, None, None))[0] == 0
    od = lib.spconv_submconv3d_ordered
    code, msg = _status(od(fake, fake, None, fake, None, fake, 10, 27, 16, 16, 2, None))
    assert code == -1 and "order" in msg
    code, msg = _status(od(fake, fake, ctypes.c_void_p(0x100002), fake, None, fake, 10, 27, 16, 16, 2, None))
    assert code == -1 and "order" in msg
    assert _status(od(fake, fake, fake, fake, None, fake, 10, 27, 24, 16, 2, None))[0] == -2
    assert _status(od(None, None, None, None, None, None, 0, 27, 16, 16, 2, None))[0] == 0


def test_xrun_entry_points_validate_without_gpu(lib):
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: validation fails first
    n = 10
    cap = lib.spconv_xrun_slot_capacity(n)
    ws = lib.spconv_xrun_workspace_size(n)
    assert cap == 3 * n + 1
    assert ws >= n + 8
    assert lib.spconv_xrun_slot_capacity(-1) == 0 and lib.spconv_xrun_workspace_size(-1) == 0
    xl = lib.spconv_xrun_layout
    assert _status(xl(fake, fake, 0, 27, fake, cap, fake, fake, ws, None))[0] == -1
    assert _status(xl(fake, fake, 1 << 30, 27, fake, 1 << 32, fake, fake, 1 << 40, None))[0] == -1
    assert _status(xl(fake, fake, n, 26, fake, cap, fake, fake, ws, None))[0] == -2
    assert _status(xl(None, fake, n, 27, fake, cap, fake, fake, ws, None))[0] == -1
    assert _status(xl(fake, fake, n, 27, fake, cap - 1, fake, fake, ws, None))[0] == -1
    assert _status(xl(fake, fake, n, 27, fake, cap, ctypes.c_void_p(0x100004), fake, ws, None))[0] == -1
    assert _status(xl(fake, fake, n, 27, fake, cap, fake, fake, ws - 1, None))[0] == -3
    xc = lib.spconv_submconv3d_xrun
    assert _status(xc(fake, fake, fake, 31, fake, fake, None, fake, n, 27, 128, 128, 0, None))[0] == -2
    assert _status(xc(fake, fake, fake, 31, fake, fake, None, fake, n, 27, 64, 128, 2, None))[0] == -2
    assert _status(xc(fake, fake, fake, 31, fake, fake, None, fake, n, 27, 128, 256, 2, None))[0] == -2
    assert _status(xc(fake, fake, fake, 31, fake, fake, None, fake, n, 27, 128, 24, 2, None))[0] == -2
    assert _status(xc(fake, fake, fake, 31, fake, fake, None, fake, n, 125, 128, 128, 2, None))[0] == -2
    assert _status(xc(fake, fake, None, 31, fake, fake, None, fake, n, 27, 128, 128, 2, None))[0] == -1
    assert _status(xc(fake, fake, fake, 31, fake, ctypes.c_void_p(0x100008), None, fake, n, 27, 128, 128, 2,
                      None))[0] == -1
    assert _status(xc(fake, fake, fake, 31, fake, fake, None, fake, 0, 27, 128, 128, 2, None))[0] == -1
    assert _status(xc(fake, fake, fake, 0, fake, fake, None, fake, n, 27, 128, 128, 2, None))[0] == -1
    xe = lib.spconv_submconv3d_xrun_ex
    assert _status(xe(fake, fake, fake, 31, fake, fake, None, fake, fake, n, 27, 128, 128, 2, 3, None))[0] == -1
    assert _status(xe(fake, fake, fake, 31, fake, fake, None, ctypes.c_void_p(0x100008), fake, n, 27, 128, 128,
                      2, 1, None))[0] == -1
    assert _status(xe(fake, fake, fake, 31, fake, fake, None, fake, fake, n, 27, 64, 128, 2, 2, None))[0] == -2
    assert _status(xe(fake, None, fake, 31, fake, fake, None, fake, fake, n, 27, 128, 128, 2, 0, None))[0] == -1
    xd = lib.spconv_submconv3d_dgrad_xrun
    assert _status(xd(fake, fake, fake, 31, fake, fake, fake, n, 27, 128, 64, 2, None))[0] == -2
    assert _status(xd(fake, fake, fake, 31, fake, fake, fake, n, 27, 256, 128, 2, None))[0] == -2
    assert _status(xd(fake, fake, fake, 31, fake, fake, fake, n, 27, 64, 128, 0, None))[0] == -2
    assert _status(xd(fake, fake, None, 31, fake, fake, fake, n, 27, 64, 128, 2, None))[0] == -1
    assert _status(xd(fake, fake, fake, 31, fake, ctypes.c_void_p(0x100008), fake, n, 27, 64, 128, 2,
                      None))[0] == -1
    assert _status(xd(fake, fake, fake, 0, fake, fake, fake, n, 27, 64, 128, 2, None))[0] == -1


def test_fused_build_and_layout_validates_without_gpu(lib):
    fake = ctypes.c_void_p(0x100000)  # never dereferenced: validation fails first
    n = 10
    cap = lib.spconv_xrun_slot_capacity(n)
    ws = lib.spconv_build_nmap_xrun_workspace_size(n)
    assert ws >= lib.spconv_build_nmap_workspace_size(n) + lib.spconv_xrun_workspace_size(n)
    assert lib.spconv_build_nmap_xrun_workspace_size(-1) == 0
    bx = lib.spconv_build_nmap_xrun
    assert _status(bx(fake, 0, fake, fake, cap, fake, fake, ws, None, None))[0] == -1
    assert _status(bx(fake, 1 << 30, fake, fake, 1 << 32, fake, fake, 1 << 40, None, None))[0] == -1
    assert _status(bx(None, n, fake, fake, cap, fake, fake, ws, None, None))[0] == -1
    assert _status(bx(fake, n, fake, fake, cap - 1, fake, fake, ws, None, None))[0] == -1
    assert _status(bx(fake, n, fake, fake, cap, ctypes.c_void_p(0x100004), fake, ws, None, None))[0] == -1
    assert _status(bx(fake, n, fake, fake, cap, fake, ctypes.c_void_p(0x100080), ws, None, None))[0] == -1
    assert _status(bx(fake, n, fake, fake, cap, fake, fake, ws, ctypes.c_void_p(0x100002), None))[0] == -1
    assert _status(bx(fake, n, fake, fake, cap, fake, fake, ws - 1, None, None))[0] == -3


def test_python_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    with pytest.raises(TypeError):
        sv.build_nmap(torch.zeros((4, 3), dtype=torch.int32))
    with pytest.raises(TypeError):
        sv.submconv3d(torch.zeros((4, 16)), torch.zeros((27, 4), dtype=torch.int32),
                      torch.zeros((27, 16, 16)))


def test_default_offsets_order():
    offs = sv.default_offsets()
    assert offs.shape == (27, 3)
    for k, (dz, dy, dx) in enumerate(offs):
        assert k == 9 * (dz + 1) + 3 * (dy + 1) + (dx + 1)
