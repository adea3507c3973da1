"""C ABI checks that need no GPU: the library builds, loads and exports every
function include/vla.h declares, and argument errors come back as codes."""
import ctypes
import os

import pytest
import torch

from _util import ensure_built, header_functions


@pytest.fixture(scope="module")
def lib():
    ensure_built()
    import sherman_morrison_inverse_gb300 as vla
    return vla.load_library()


def test_header_declares_the_boundary():
    names = header_functions()
    for fn in ("vla_create", "vla_scan_fwd", "vla_status", "vla_last_error", "vla_destroy"):
        assert fn in names, names


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_null_handle_is_rejected_before_any_cuda_call(lib):
    code = lib.vla_scan_fwd(None, None, None, None, None, None, None, None, None,
                            1, 1, 4, 64, 64, 1, 0, 0.0, 1.0, 0, 0, 0, 16, None)
    assert code == 1  # VLA_ERR_INVALID_ARG
    assert b"handle" in lib.vla_last_error(None)


def test_status_and_destroy_with_null(lib):
    assert lib.vla_status(None, None, None) == 1
    assert lib.vla_destroy(None) == 0


def test_create_rejects_null_out_pointer(lib):
    assert lib.vla_create(None, 0) == 1


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_create_without_a_gpu_reports_an_error(lib):
    h = ctypes.c_void_p()
    code = lib.vla_create(ctypes.byref(h), 0)
    assert code in (1, 3) and not h.value
    assert lib.vla_last_error(None)


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    import sherman_morrison_inverse_gb300 as vla
    monkeypatch.setattr(vla, "_lib", None)
    monkeypatch.setattr(vla, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        vla.load_library()


def test_host_entry_point_and_path_info_reject_a_null_handle(lib):
    code = lib.vla_scan_fwd_host(None, None, None, None, None, None, None, None, None,
                                 1, 1, 4, 64, 64, 1, 0, 0.0, 1.0, 0, 0, 0, 0, 0, None)
    assert code == 1  # VLA_ERR_INVALID_ARG
    assert b"handle" in lib.vla_last_error(None)
    g, seg = ctypes.c_int(), ctypes.c_longlong()
    assert lib.vla_host_path_info(None, ctypes.byref(g), ctypes.byref(seg)) == 1


def test_projection_rejects_a_null_handle(lib):
    assert lib.vla_project_u(None, None, None, None, 4, 64, 1, 0, None) == 1


def test_header_and_library_serve_a_plain_c_program(lib, tmp_path):
    """include/vla.h compiles as strict C99 and a C program links against libvla.so and
    calls through it (NULL handles only: no GPU needed)."""
    import shutil
    import subprocess
    from _util import HEADER
    import sherman_morrison_inverse_gb300 as vla
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_vla.c"
    src.write_text(
        '#include "vla.h"\n'
        "#include <string.h>\n"
        "int main(void) {\n"
        "  vla_status_t st;\n"
        "  if (vla_destroy(0) != VLA_OK) return 1;\n"
        "  if (vla_status(0, 0, &st) != VLA_ERR_INVALID_ARG) return 2;\n"
        "  if (vla_scan_fwd(0, 0, 0, 0, 0, 0, 0, 0, 0, 1, 1, 4, 64, 64, 1, 0, 0.f, 1.f, 0, VLA_F32,\n"
        "                   VLA_SEQUENTIAL, 0, 0) != VLA_ERR_INVALID_ARG) return 3;\n"
        "  return strlen(vla_last_error(0)) > 0 ? 0 : 4;\n"
        "}\n")
    libdir = os.path.dirname(vla.library_path())
    exe = tmp_path / "use_vla"
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.dirname(HEADER),
           str(src), "-L", libdir, "-lvla", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    assert subprocess.run([str(exe)]).returncode == 0
