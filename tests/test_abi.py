"""libkivi.so host-side checks that need no GPU: the library loads, exports
every entry point include/kivi.h declares, validates its arguments with the
documented status codes, and its byte accounting agrees with the oracle's
closed form.  No call here reaches a CUDA API."""
import ctypes as C
import os
import re

import numpy as np
import pytest

from conftest import ROOT


def header_functions():
    src = open(os.path.join(ROOT, "include", "kivi.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kivi_\w+)\s*\(", src)))


def test_header_symbols_exported(kivi_lib):
    from kivi_bit_kv_gb300 import abi
    names = header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(kivi_lib, n), f"{n} declared in include/kivi.h but not exported"
    assert sorted(abi.EXPORTS) == names


def test_abi_version_and_status_strings(kivi_lib):
    from kivi_bit_kv_gb300 import abi
    assert abi.kivi_abi_version() == 1
    for st in range(6):
        assert abi.kivi_status_string(st) and abi.kivi_status_string(st) != "unknown status"
    assert abi.kivi_status_string(99) == "unknown status"


def _desc(**kw):
    from kivi_bit_kv_gb300 import abi
    base = dict(B=2, H=4, D=128, bits_k=2, bits_v=2, G=32, R=128, Tmax=4096)
    base.update(kw)
    return abi.kivi_cache(**base)


def _with_ptrs(d, base=0x10000, misalign=None):
    for i, name in enumerate(["kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "len"]):
        setattr(d, name, base + 0x100000 * (i + 1) + (4 if name == misalign else 0))
    return d


@pytest.mark.parametrize("field,value,needle", [
    ("D", 96, "head dim"), ("D", 32, "head dim"), ("bits_k", 3, "bits"), ("bits_v", 16, "bits"),
    ("G", 16, "group size"), ("G", 128, "multiple of G"), ("R", 48, "residual"),
    ("R", -32, "residual"), ("Tmax", 100, "capacity"), ("Tmax", 0, "capacity"), ("B", 0, "B=0"),
])
def test_validation_rejects_bad_sizes(kivi_lib, field, value, needle):
    from kivi_bit_kv_gb300 import abi
    d = _with_ptrs(_desc(**{field: value}, **({"D": 64} if field == "G" and value == 128 else {})))
    st = abi.kivi_cache_validate(d)
    assert st == abi.KIVI_EINVAL
    assert needle in abi.kivi_last_error(), abi.kivi_last_error()


def test_validation_pointers(kivi_lib):
    from kivi_bit_kv_gb300 import abi
    assert abi.kivi_cache_validate(_with_ptrs(_desc())) == abi.KIVI_OK
    assert abi.kivi_last_error() == ""
    d = _with_ptrs(_desc())
    d.vzero = None
    assert abi.kivi_cache_validate(d) == abi.KIVI_EINVAL and "vzero is NULL" in abi.kivi_last_error()
    d = _with_ptrs(_desc(), misalign="kres")
    assert abi.kivi_cache_validate(d) == abi.KIVI_EINVAL and "aligned" in abi.kivi_last_error()
    assert kivi_lib.kivi_cache_validate(None) == abi.KIVI_EINVAL


def test_entry_points_reject_bad_arguments_before_launch(kivi_lib):
    """Argument errors return before any CUDA call (no device is touched)."""
    from kivi_bit_kv_gb300 import abi
    L = kivi_lib
    d = _with_ptrs(_desc())
    ref = C.byref(d)
    assert L.kivi_quant_keys(ref, None, 16, None, None) == abi.KIVI_EINVAL     # K NULL
    assert L.kivi_quant_values(ref, 0x20000, 5000, None, None) == abi.KIVI_EINVAL  # T > Tmax
    assert L.kivi_quant_keys(ref, 0x20004, 16, None, None) == abi.KIVI_EINVAL  # misaligned
    assert L.kivi_dequant(ref, 2, 0x20000, 16, None) == abi.KIVI_EINVAL        # which
    assert L.kivi_append_token(ref, 0x20000, 0x30000, None, None) == abi.KIVI_EINVAL
    assert L.kivi_decode_qk(ref, 0x20000, 6, C.c_float(1.0), 0x30000, 4096, None) == abi.KIVI_EINVAL
    assert "multiple of H" in abi.kivi_last_error()
    assert L.kivi_decode_qk(ref, 0x20000, 4, C.c_float(1.0), 0x30000, 4095, None) == abi.KIVI_EINVAL
    assert L.kivi_decode_qk(ref, 0x20000, 4 * 17, C.c_float(1.0), 0x30000, 4096, None) == abi.KIVI_EINVAL
    need = abi.kivi_workspace_bytes(type("c", (), {"desc": d})(), 4)
    assert need > 0
    # undersized workspaces: rejected before any launch (the pointers are fake)
    assert L.kivi_decode_pv(ref, 0x30000, 4096, 4, 0x40000, 0x50000, 16, None) == abi.KIVI_EWORKSPACE
    assert L.kivi_decode_attention(ref, 0x20000, 4, C.c_float(1.0), 0x40000, 0x50000, 16,
                                   None) == abi.KIVI_EWORKSPACE
    assert L.kivi_decode_attention(ref, 0x20000, 6, C.c_float(1.0), 0x40000, 0x50000, need,
                                   None) == abi.KIVI_EINVAL
    # mixed key / value widths pass validation (an undersized workspace is
    # what stops this call before any launch)
    mixed = _with_ptrs(_desc(bits_v=4))
    assert L.kivi_decode_attention(C.byref(mixed), 0x20000, 4, C.c_float(1.0), 0x40000, 0x50000,
                                   16, None) == abi.KIVI_EWORKSPACE


def test_buffer_bytes(kivi_lib):
    from kivi_bit_kv_gb300 import abi
    d = _desc(B=3, H=5, D=128, bits_k=2, bits_v=4, G=32, R=64, Tmax=1024)
    BH = 15
    assert abi.kivi_buffer_bytes(d, abi.KIVI_BUF_KQ) == BH * (1024 // 16) * 128 * 4
    assert abi.kivi_buffer_bytes(d, abi.KIVI_BUF_KSCALE) == BH * (1024 // 32) * 128 * 4
    assert abi.kivi_buffer_bytes(d, abi.KIVI_BUF_VQ) == BH * 1024 * (128 // 8) * 4
    assert abi.kivi_buffer_bytes(d, abi.KIVI_BUF_VZERO) == BH * 1024 * 4 * 4
    assert abi.kivi_buffer_bytes(d, abi.KIVI_BUF_KRES) == BH * 96 * 128 * 2
    assert abi.kivi_buffer_bytes(d, abi.KIVI_BUF_LEN) == 12
    assert abi.kivi_buffer_bytes(d, 9) == 0


def test_cache_bytes_matches_oracle_closed_form(kivi_lib, ref):
    from kivi_bit_kv_gb300 import abi
    rng = np.random.default_rng(0)
    for _ in range(300):
        G = int(rng.choice([32, 64, 128]))
        D = int(rng.choice([64, 128, 256]))
        if D % G:
            continue
        bits = int(rng.choice([2, 4, 8]))
        R = G * int(rng.integers(0, 5))
        T = int(rng.integers(0, 40000))
        for which in (0, 1):
            assert abi.kivi_cache_bytes(T, D, bits, G, R, which) == ref.cache_bytes(T, D, bits, G, R, which)
    assert abi.kivi_cache_bytes(10, 128, 3, 32, 0, 0) == 0


def test_missing_library_fails_loudly(tmp_path):
    from kivi_bit_kv_gb300 import abi
    with pytest.raises(ImportError):
        abi.load(str(tmp_path / "libkivi.so"))


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "kivi.h"

int main(void)
{
    kivi_cache c;
    memset(&c, 0, sizeof c);
    c.B = 1; c.H = 1; c.D = 100; c.bits_k = 2; c.bits_v = 2; c.G = 32; c.R = 32; c.Tmax = 64;
    const int32_t st = kivi_cache_validate(&c);
    printf("%d %d %zu %d %s|%s\n", kivi_abi_version(), st, kivi_cache_bytes(100, 64, 2, 32, 32, 0),
           st == KIVI_EINVAL, kivi_status_string(st), kivi_last_error());
    return 0;
}
"""


def test_plain_c_client_links_and_calls(kivi_lib, tmp_path):
    """The boundary is usable from C99 with nothing but include/kivi.h and
    libkivi.so: a strict C program compiles, links and calls host-side entry
    points (no CUDA call is reached)."""
    import shutil
    import subprocess
    from kivi_bit_kv_gb300 import abi
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    src, exe = tmp_path / "client.c", tmp_path / "client"
    src.write_text(C_CLIENT)
    libdir = os.path.dirname(abi.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                    f"-I{os.path.join(ROOT, 'include')}", str(src), "-o", str(exe),
                    f"-L{libdir}", "-lkivi", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.strip()
    head, err = out.split("|", 1)
    version, status, nbytes, is_einval, text = head.split(" ", 4)
    assert int(version) == abi.kivi_abi_version()
    assert int(status) == abi.KIVI_EINVAL and is_einval == "1" and text == "invalid argument"
    assert int(nbytes) == abi.kivi_cache_bytes(100, 64, 2, 32, 32, 0)
    assert "D=100" in err
