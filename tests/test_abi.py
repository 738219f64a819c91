"""Host-side checks of the C ABI: the library loads, exports every function that
include/*.h declares, and rejects bad arguments synchronously (no GPU needed:
every call here returns before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import linear_attention_elu_gb300 as la
    return la


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(la_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("la_noncausal_fwd", "la_causal_fwd", "la_decode_step", "la_workspace_size",
                     "la_workspace_init", "la_query_status", "la_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.library_path())
    missing = [n for n in _declared() if not hasattr(so, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in range(6):
        assert lib.la_status_string(code).startswith("LA_")
    assert "unknown" in lib.la_status_string(99)
    assert lib.la_version() >= 1


def test_workspace_size(lib):
    assert lib.la_workspace_size(lib.LA_OP_DECODE, 512, 8, 1, 64, 64, lib.LA_BF16) == 0
    for op in (lib.LA_OP_CAUSAL, lib.LA_OP_NONCAUSAL):
        n = lib.la_workspace_size(op, 8, 8, 3072, 64, 64, lib.LA_BF16)
        assert n >= 256 and n % 256 == 0
        # Empty problems need only the header.
        assert lib.la_workspace_size(op, 8, 8, 0, 64, 64, lib.LA_BF16) == 256


def test_feature_map_entries_reject_bad_arguments_without_a_gpu(lib):
    so = ctypes.CDLL(lib.library_path())
    P = ctypes.c_void_p
    so.la_noncausal_fwd_phi.argtypes = [P, P, P, P] + [ctypes.c_int] * 7 + [ctypes.c_float, P,
                                                                            ctypes.c_size_t, P]
    # An unknown feature map is refused before anything is launched.
    assert so.la_noncausal_fwd_phi(None, None, None, None, 1, 1, 0, 64, 64, 1, 5, 1e-6, None, 0,
                                   None) == 1
    so.la_positive_random_features.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_float, P]
    assert so.la_positive_random_features(None, None, None, 10, 129, 64, 1, 0.0, None) == 1
    assert so.la_positive_random_features(None, None, None, 10, 64, 0, 1, 0.0, None) == 1
    assert so.la_positive_random_features(None, None, None, 10, 64, 64, 1, float("inf"), None) == 1
    assert so.la_positive_random_features(None, None, None, 10, 64, 64, 1, 0.0, None) == 1  # null x
    assert so.la_positive_random_features(None, None, None, 0, 64, 64, 1, 0.0, None) == 0   # empty


def test_backward_workspace_and_launches(lib):
    # Both backward directions use the same scratch: per-chunk forward and reverse
    # sums (B*H*ceil(N/64)*(Dk*Dv + Dk) floats each) and per-row (dnum, dden)
    # (B*H*N*(Dv + 1) floats), after the 256-byte header.
    B, H, N, D = 8, 8, 3072, 64
    body = 4 * (2 * B * H * (N // 64) * (D * D + D) + B * H * N * (D + 1))
    for op in (lib.LA_OP_CAUSAL_BWD, lib.LA_OP_NONCAUSAL_BWD):
        assert lib.la_workspace_size(op, B, H, N, D, D, lib.LA_BF16) == 256 + (body + 255) // 256 * 256
        assert lib.la_launch_count(op, B, H, N, D, D, lib.LA_BF16) == 5
        assert lib.la_launch_count(op, B, H, 0, D, D, lib.LA_BF16) == 0
    so = ctypes.CDLL(lib.library_path())
    n = ctypes.c_size_t(0)
    assert so.la_workspace_size(lib.LA_OP_NONCAUSAL_BWD, 1, 1, 64, 128, 64, 1, ctypes.byref(n)) == 2


def _raw(lib):
    return ctypes.CDLL(lib.library_path())


def test_bad_arguments_are_rejected_synchronously(lib):
    so = _raw(lib)
    n = ctypes.c_size_t(0)
    # Null out-parameter, bad op, bad dtype, negative and oversized dims.
    assert so.la_workspace_size(1, 1, 1, 1, 64, 64, 1, None) == 1
    assert so.la_workspace_size(7, 1, 1, 1, 64, 64, 1, ctypes.byref(n)) == 1
    assert so.la_workspace_size(1, 1, 1, 1, 64, 64, 5, ctypes.byref(n)) == 1
    assert so.la_workspace_size(1, -1, 1, 1, 64, 64, 1, ctypes.byref(n)) == 1
    assert so.la_workspace_size(1, 1, 1, 1, 0, 64, 1, ctypes.byref(n)) == 1
    assert so.la_workspace_size(1, 1, 1, 1, 256, 256, 1, ctypes.byref(n)) == 2
    assert so.la_workspace_size(1, 1000, 1000, 1, 64, 64, 1, ctypes.byref(n)) == 2
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    so.la_causal_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, P, P, Z, P]
    so.la_noncausal_fwd.argtypes = [P, P, P, P, I, I, I, I, I, I, F, P, Z, P]
    so.la_decode_step.argtypes = [P, P, P, P, P, P, I, I, I, I, I, F, P]
    fake = 1 << 20  # aligned, never dereferenced: every call below fails its checks first
    # Null tensors.
    assert so.la_causal_fwd(None, fake, fake, fake, 1, 1, 64, 64, 64, 1, 1e-6, None, None,
                            fake, 1 << 30, None) == 1
    # Misaligned tensor.
    assert so.la_noncausal_fwd(fake + 2, fake, fake, fake, 1, 1, 64, 64, 64, 1, 1e-6, fake,
                               1 << 30, None) == 1
    # Negative / NaN eps.
    assert so.la_causal_fwd(fake, fake, fake, fake, 1, 1, 64, 64, 64, 1, -1.0, None, None,
                            fake, 1 << 30, None) == 1
    assert so.la_causal_fwd(fake, fake, fake, fake, 1, 1, 64, 64, 64, 1, float("nan"), None,
                            None, fake, 1 << 30, None) == 1
    # Workspace missing, too small, misaligned.
    assert so.la_causal_fwd(fake, fake, fake, fake, 1, 1, 64, 64, 64, 1, 1e-6, None, None,
                            None, 0, None) == 3
    assert so.la_causal_fwd(fake, fake, fake, fake, 1, 1, 64, 64, 64, 1, 1e-6, None, None,
                            fake, 300, None) == 3
    assert so.la_noncausal_fwd(fake, fake, fake, fake, 1, 1, 64, 64, 64, 1, 1e-6, fake + 16,
                               1 << 30, None) == 3
    # Decode: null state.
    assert so.la_decode_step(fake, fake, fake, fake, None, fake, 1, 1, 64, 64, 1, 1e-6,
                             None) == 1
    # Empty problems are valid no-ops that touch nothing.
    assert so.la_noncausal_fwd(None, None, None, None, 0, 4, 64, 64, 64, 1, 1e-6, None, 0,
                               None) == 0
    assert so.la_causal_fwd(None, None, None, None, 2, 0, 64, 64, 64, 1, 1e-6, None, None,
                            None, 0, None) == 0
    assert so.la_decode_step(None, None, None, None, None, None, 0, 8, 64, 64, 1, 1e-6,
                             None) == 0


def test_host_staging_size(lib):
    # Two buffers of one head group (a quarter of B*H rounded up to a multiple of
    # 4 heads), each holding q, k, v, o of the group plus 256-byte alignment.
    per_head = 3072 * (2 * 64 + 2 * 64) * 2
    assert lib.la_host_staging_size(8, 8, 3072, 64, 64, lib.LA_BF16) == 2 * (16 * per_head + 1024)
    assert lib.la_host_staging_size(1, 1, 100, 32, 32, lib.LA_F32) == 2 * (4 * 100 * 128 * 4 + 1024)
    with pytest.raises(lib.LinAttnError):
        lib.la_host_staging_size(1, 1, 100, 0, 32, lib.LA_F32)


def test_host_entry_rejects_bad_arguments_without_a_gpu(lib):
    raw = _raw(lib)
    raw.la_causal_fwd_host.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 6 + [
        ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
        ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]
    buf = ctypes.create_string_buffer(4096)
    p = ctypes.cast(buf, ctypes.c_void_p)
    # Missing host tensors, then a missing staging buffer: rejected before any CUDA call.
    assert raw.la_causal_fwd_host(None, None, None, None, 1, 1, 8, 64, 64, 1, 1e-6, None, None,
                                  p, 4096, p, 4096, None) == 1
    assert raw.la_causal_fwd_host(p, p, p, p, 1, 1, 8, 64, 64, 1, 1e-6, None, None,
                                  None, 0, p, 4096, None) == 3


def test_layer_decode_workspace(lib):
    # Projection buffers ([B, 3 d_model] and [B, d_model] in the dtype, each
    # rounded up to 256 bytes) after the header; two projections and the decode
    # step are three launches.
    B, H, D = 512, 8, 64
    dm = H * D
    body = B * 3 * dm * 2 + B * dm * 2
    assert lib.la_workspace_size(lib.LA_OP_LAYER_DECODE, B, H, 1, D, D, lib.LA_BF16) == 256 + body
    assert lib.la_launch_count(lib.LA_OP_LAYER_DECODE, B, H, 1, D, D, lib.LA_BF16) == 3
    so = ctypes.CDLL(lib.library_path())
    n = ctypes.c_size_t(0)
    assert so.la_workspace_size(lib.LA_OP_LAYER_DECODE, B, H, 1, 64, 32, 1, ctypes.byref(n)) == 2


def test_header_is_plain_c_and_links(lib, tmp_path):
    # A C caller (no C++, no CUDA headers) compiles against the header and links
    # against the library: every entry point is taken by address, so a missing
    # or mangled symbol fails the link.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    names = _declared()
    src = tmp_path / "use_abi.c"
    src.write_text(
        '#include "linattn.h"\n#include <stdio.h>\n'
        "int main(void) {\n"
        "    const void* fns[] = {" + ", ".join(f"(const void*)&{n}" for n in names) + "};\n"
        '    size_t n = 0;\n'
        '    la_status s = la_workspace_size(LA_OP_CAUSAL, 8, 8, 3072, 64, 64, LA_BF16, &n);\n'
        '    printf("%d %zu %d\\n", (int)s, n, (int)(sizeof(fns) / sizeof(fns[0])));\n'
        "    return s == LA_OK ? 0 : 1;\n}\n")
    exe = tmp_path / "use_abi"
    libdir = os.path.dirname(lib.library_path())
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(root, "include"),
                        str(src), "-L", libdir, "-llinattn", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    # Running it needs only the CUDA runtime to load; the size query touches no GPU.
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    status, size, count = r.stdout.split()
    assert int(status) == 0 and int(size) == lib.la_workspace_size(lib.LA_OP_CAUSAL, 8, 8, 3072, 64, 64, lib.LA_BF16)
    assert int(count) == len(names)


def test_binding_sets_a_signature_for_every_declared_function(lib):
    # A function called through ctypes without argtypes would pass every
    # argument as a C int: the binding must declare each one.
    with open(os.path.join(ROOT, "linear_attention_elu_gb300", "__init__.py")) as f:
        text = f.read()
    bound = set(re.findall(r"lib\.(la_[a-z0-9_]+)\.argtypes", text))
    missing = sorted(set(_declared()) - bound)
    assert not missing, missing


def test_wrappers_refuse_host_tensors_before_any_launch(lib):
    import torch
    q = torch.zeros(1, 1, 4, 64)
    for fn in (lib.la_causal_fwd, lib.la_noncausal_fwd, lib.la_causal_fwd_noalloc):
        with pytest.raises(ValueError):
            fn(q, q, q)
