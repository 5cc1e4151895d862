"""The C ABI without a GPU: libcc.so builds, loads, exports every function
include/*.h declares, and rejects bad arguments on the host before touching
the device. No compute call is made here."""

import ctypes
import os
import re

import pytest

from causal_convolution_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include"))) if f.endswith(".h")]


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from causal_convolution_gb300 import build
        build.build()
    return _lib.load()


def declared_functions():
    names = set()
    for path in HEADERS:
        text = open(path).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(cc_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_headers_declare_the_boundary():
    names = declared_functions()
    for required in ("cc_conv3d_causal", "cc_resample_up2", "cc_attn_frame", "cc_head_out", "cc_check_device",
                     "cc_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_python_binding_declares_every_symbol():
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_every_entry_point_has_an_exported_wrapper():
    from causal_convolution_gb300 import api
    # cc_last_error is read by the wrappers themselves (CCError messages)
    missing = [n for n in declared_functions() if n != "cc_last_error" and n not in api.__all__]
    assert not missing, missing
    assert all(callable(getattr(api, n)) for n in api.__all__ if n.startswith("cc_"))


def test_version_and_workspace_arithmetic(lib):
    assert lib.cc_version() >= 100
    assert lib.cc_resample_workspace_bytes(1, 8, 88, 156, 512) == 4 * 8 * 88 * 156 * 512 * 2
    assert lib.cc_head_workspace_bytes(1, 16, 352, 624) == 16 * 352 * 624 * 112 * 2
    assert lib.cc_attn_ld(3432) == 3440
    assert lib.cc_attn_ld(3440) == 3440
    assert lib.cc_attn_ld(3441) == 3456
    ld = 3440
    assert lib.cc_attn_workspace_bytes(4, 3432) == 4 * 3432 * ld * 4 + 4 * 3432 * ld * 2
    assert lib.cc_resample_workspace_bytes(0, 1, 1, 1, 1) == 0
    assert lib.cc_attn_exp_key_tiles(3432) == 14
    assert lib.cc_attn_exp_key_tiles(256) == 1 and lib.cc_attn_exp_key_tiles(257) == 2
    assert lib.cc_attn_exp_workspace_bytes(4, 3432) == 4 * 3432 * ld * 2 + 4 * 3432 * 14 * 8


def test_host_validation_rejects_before_any_launch(lib):
    # null pointers, misalignment and bad sizes come back as CC_ERR_INVALID /
    # CC_ERR_UNSUPPORTED without a device (no CUDA call is reached)
    buf = ctypes.create_string_buffer(1 << 12)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.cc_conv3d_causal(None, p, None, p, 1, 1, 1, 1, 64, 64, 0, None) == 1
    assert b"null" in lib.cc_last_error()
    assert lib.cc_conv3d_causal(p + 2, p, None, p, 1, 1, 1, 1, 64, 64, 0, None) == 1
    assert b"aligned" in lib.cc_last_error()
    assert lib.cc_conv3d_causal(p, p, None, p, 1, 1, 1, 1, 64, 64, 1, None) == 1  # hist must be 0 or 2
    assert lib.cc_conv3d_causal(p, p, None, p, 1, 1, 1, 1, 48, 64, 0, None) == 2  # C_in % 64
    assert b"multiple of 64" in lib.cc_last_error()
    assert lib.cc_resample_interleave(p, p, p, p, 1, 1, 1, 1, 12, None) == 2  # C % 8
    assert lib.cc_resample_up2_fused(p, p, p, p, p, 1, 1, 1, 1, 64, 64, 0, 2, None) == 1  # temporal flag
    assert lib.cc_attn_softmax(p, p, 1, 16, 16, 16, ctypes.c_float(-1.0), None) == 1  # scale > 0
    assert lib.cc_attn_frame(p, p, p, p, 1, 16, 64, 64, 64, 64, 64, ctypes.c_float(0.125), p, 16, None) == 1
    assert b"workspace" in lib.cc_last_error()
    assert lib.cc_head_out(p, p, p, p, 1, 1, 4, 4, 64, 0, p, 10, None) == 1
    assert lib.cc_attn_scores_exp(p, p, p, None, 1, 16, 64, 64, 64, 16, ctypes.c_float(0.125), None) == 1
    assert b"null" in lib.cc_last_error()
    assert lib.cc_attn_scores_exp(p, p, p, p, 1, 16, 64, 64, 64, 16, ctypes.c_float(0.0), None) == 1  # scale
    assert lib.cc_attn_scores_exp(p, p, p, p, 1, 16, 48, 48, 48, 16, ctypes.c_float(0.125), None) == 2  # C % 64
    assert lib.cc_attn_pv_exp(p, p + 4, p, p, 1, 16, 64, 16, 64, 64, None) == 1  # stats misaligned
    assert lib.cc_attn_exp_rescale(p, p, 1, 16, 12, None) == 1  # ld_e % 8
    assert lib.cc_attn_frame_exp(p, p, p, p, 1, 16, 64, 64, 64, 64, 64, ctypes.c_float(0.125), p, 16, None) == 1
    assert b"workspace" in lib.cc_last_error()
    assert lib.cc_debug_wait_timeout(0, None) == 1
    assert lib.cc_debug_im2col_tile(p, p, 1, 1, 1, 1, 64, -17, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, None) == 1


def test_empty_requests_succeed_without_a_launch(lib):
    # a zero count of images, frames, rows, columns or positions: CC_OK with
    # NULL pointers and no device (nothing is launched, no pointer is read)
    f = ctypes.c_float(0.125)
    assert lib.cc_conv3d_causal(None, None, None, None, 0, 4, 8, 8, 64, 64, 0, None) == 0
    assert lib.cc_conv3d_causal(None, None, None, None, 1, 0, 8, 8, 64, 64, 2, None) == 0
    assert lib.cc_conv3d_causal(None, None, None, None, 1, 4, 8, 0, 64, 64, 0, None) == 0
    assert lib.cc_resample_phase_conv(None, None, None, 1, 1, 0, 4, 64, 64, 0, None) == 0
    assert lib.cc_resample_interleave(None, None, None, None, 1, 0, 4, 4, 64, None) == 0
    assert lib.cc_resample_up2(None, None, None, None, None, 0, 1, 4, 4, 64, 64, 0, None, 0, None) == 0
    assert lib.cc_resample_up2_fused(None, None, None, None, None, 1, 1, 4, 0, 64, 64, 0, 1, None) == 0
    assert lib.cc_attn_scores(None, None, None, 0, 16, 64, 64, 64, 16, None) == 0
    assert lib.cc_attn_softmax(None, None, 2, 0, 16, 16, f, None) == 0
    assert lib.cc_attn_pv(None, None, None, 0, 16, 64, 16, 64, 64, None) == 0
    assert lib.cc_attn_frame(None, None, None, None, 2, 0, 64, 64, 64, 64, 64, f, None, 0, None) == 0
    assert lib.cc_attn_scores_exp(None, None, None, None, 0, 16, 64, 64, 64, 16, f, None) == 0
    assert lib.cc_attn_exp_rescale(None, None, 3, 0, 16, None) == 0
    assert lib.cc_attn_pv_exp(None, None, None, None, 0, 16, 64, 16, 64, 64, None) == 0
    assert lib.cc_attn_frame_exp(None, None, None, None, 0, 5, 64, 64, 64, 64, 64, f, None, 0, None) == 0
    assert lib.cc_head_temporal(None, None, None, 1, 0, 4, 4, 256, 0, None) == 0
    assert lib.cc_head_stencil(None, None, None, 1, 2, 0, 4, None) == 0
    assert lib.cc_head_out(None, None, None, None, 0, 2, 4, 4, 256, 0, None, 0, None) == 0
    assert lib.cc_head_out_noalloc(None, None, None, None, 1, 0, 4, 4, 256, 2, None) == 0
    assert lib.cc_attn_exp_workspace_bytes(0, 16) == 0 and lib.cc_head_workspace_bytes(1, 0, 4, 4) == 0
    # a negative count stays invalid, whatever the other counts
    assert lib.cc_conv3d_causal(None, None, None, None, 0, -1, 8, 8, 64, 64, 0, None) == 1
    assert b"negative" in lib.cc_last_error()
    assert lib.cc_attn_frame_exp(None, None, None, None, -2, 0, 64, 64, 64, 64, 64, f, None, 0, None) == 1
    assert lib.cc_head_out_noalloc(None, None, None, None, 1, 1, -4, 4, 256, 0, None) == 1


def test_copy_to_host_argument_checks(lib):
    buf = ctypes.create_string_buffer(1 << 12)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    assert lib.cc_copy_to_host(None, None, 0, 8, None) == 0  # nothing to copy
    assert lib.cc_copy_to_host(None, p, 64, 8, None) == 1
    assert lib.cc_copy_to_host(p + 4, p, 64, 8, None) == 1
    assert b"aligned" in lib.cc_last_error()
    assert lib.cc_copy_to_host(p, p, 40, 8, None) == 1
    assert b"multiple of 16" in lib.cc_last_error()
    assert lib.cc_copy_to_host(p, p, 64, 0, None) == 1 and lib.cc_copy_to_host(p, p, 64, 1025, None) == 1
    # memory the device cannot address (no device here at all): rejected, not launched
    assert lib.cc_copy_to_host(p, p, 64, 8, None) == 1
    assert b"page-locked" in lib.cc_last_error()



def test_size_limits_rejected_on_the_host(lib):
    # requests past the kernels' index ranges come back CC_ERR_UNSUPPORTED
    # before any device call (no device here)
    buf = ctypes.create_string_buffer(1 << 12)
    p = (ctypes.addressof(buf) + 15) // 16 * 16
    big = 1 << 16
    assert lib.cc_conv3d_causal(p, p, None, p, 1, 1, big, big, 64, 64, 0, None) == 2
    assert b"too many positions" in lib.cc_last_error()
    assert lib.cc_resample_up2_fused(p, p, p, p, p, 1, 1, big, big // 2, 64, 64, 0, 0, None) == 2
    assert lib.cc_head_temporal(p, p, p, 1, 1, big, big, 256, 0, None) == 2
    assert lib.cc_resample_interleave(p, p, p, p, 1, big, big, 1, 64, None) == 2
    assert lib.cc_head_stencil(p, p, p, 1, big, big, big, None) == 2
    hw = 1 << 30  # 2^23 query tiles x 2^22 key tiles
    f = ctypes.c_float(0.125)
    assert lib.cc_attn_scores_exp(p, p, p, p, 1, hw, 64, 64, 64, hw, f, None) == 2
    assert b"too many output tiles" in lib.cc_last_error()
    assert lib.cc_attn_scores(p, p, p, 1, hw, 64, 64, 64, hw, None) == 2


C_CALLER = r"""
#include <stdio.h>
#include "cc.h"
#include "cc_debug.h"
int main(void) {
  if (cc_version() < 100) return 2;
  /* a rejected request: no device needed, nothing launched */
  if (cc_conv3d_causal(NULL, NULL, NULL, NULL, 1, 1, 1, 1, 64, 64, 0, NULL) != CC_ERR_INVALID) return 3;
  if (cc_last_error()[0] == 0) return 4;
  /* an empty request succeeds */
  if (cc_head_out(NULL, NULL, NULL, NULL, 0, 1, 1, 1, 64, 0, NULL, 0, NULL) != CC_OK) return 5;
  printf("ok\n");
  return 0;
}
"""


def test_headers_compile_and_link_as_plain_c(lib, tmp_path):
    # the boundary is a C ABI: a C99 caller (pedantic, warnings as errors)
    # includes the headers, links libcc.so and calls it
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = str(tmp_path / "abi_caller.c")
    exe = str(tmp_path / "abi_caller")
    with open(src, "w") as f:
        f.write(C_CALLER)
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-L", libdir, "-lcc", f"-Wl,-rpath,{libdir}", "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
