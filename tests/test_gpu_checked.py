"""The bounds-checked build of the library (KIVI_CHECKS defined) on hard
shapes, through the whole path.

In that build every global access of the encode, materialize, append,
payload and split-decode kernels is checked against the cache's arrays and
the call's buffers, and the streamed decode checks its copies, tiles, output
rows and partial slots; a failed check is reported as KIVI_ECHECK (by
kivi_check_status, and in the fused decode's workspace status word) and the
access is skipped.  Each case runs through both builds (each in a process of
its own, KIVI_LIB selecting the checked library): every status stays KIVI_OK,
the encoded cache, the materialized K and V, the state after an append with
a group flush, the split decode and the payload round trip agree bit for bit
between the builds, and the fused decode agrees to rounding order (which
consumer warp takes which tile varies from run to run).
"""
import os
import subprocess
import sys

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# (B, H, Hq, D, bits_k, bits_v, G, R, lengths)
CASES = [
    (3, 2, 8, 128, 2, 2, 32, 128, [700, 1, 4000]),      # GQA, ragged, a residual-only sequence
    (1, 1, 1, 128, 2, 2, 32, 128, [60000]),              # one row spread over every CTA
    (4, 4, 8, 64, 4, 4, 32, 32, [513, 2048, 0, 95]),     # D = 64, int4, an empty sequence
    (2, 2, 2, 256, 8, 8, 64, 64, [3000, 1500]),          # D = 256, int8, G = 64
    (2, 2, 4, 128, 2, 4, 32, 128, [2500, 2600]),         # key and value widths differ
    (2, 1, 4, 128, 4, 2, 128, 128, [9000, 4097]),        # G = 128
]


def run_cases(path):
    """Runs every case through the library KIVI_LIB names (or the default
    one) and saves the results and status words to `path`."""
    sys.path.insert(0, ROOT)
    import torch
    from kivi_bit_kv_gb300 import KiviCache, abi
    dev = torch.device("cuda", 0)
    res = {}
    for i, (B, H, Hq, D, bk, bv, G, R, lens) in enumerate(CASES):
        g = torch.Generator().manual_seed(100 + i)
        T = max(lens)
        Tmax = (T + 2 * G) // G * G + G
        K = torch.randn((B, H, T, D), generator=g).to(torch.float16).to(dev)
        V = torch.randn((B, H, T, D), generator=g).to(torch.float16).to(dev)
        q = torch.randn((B, Hq, D), generator=g).to(torch.float16).to(dev)
        kn = torch.randn((B, H, D), generator=g).to(torch.float16).to(dev)
        vn = torch.randn((B, H, D), generator=g).to(torch.float16).to(dev)
        cache = KiviCache(B, H, D, bk, bv, G, R, Tmax, device=dev)
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)
        abi.kivi_quant_keys(cache, K, sl)
        abi.kivi_quant_values(cache, V, sl)
        for which, name in ((0, "kh"), (1, "vh")):
            o = torch.zeros((B, H, T, D), dtype=torch.float16, device=dev)
            abi.kivi_dequant(cache, which, o)
            res[f"{name}{i}"] = o.view(torch.int16).cpu().numpy()
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        # append until some sequence flushes a group into the packed cache
        for _ in range(G + 1):
            abi.kivi_append_token(cache, kn, vn, status)
        for name in ("kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "lens"):
            t = getattr(cache, name)
            # bit patterns (fp32 statistics as int32, fp16 ring slots as int16)
            bits = {torch.float32: torch.int32, torch.float16: torch.int16}.get(t.dtype)
            res[f"{name}{i}"] = (t.view(bits) if bits is not None else t).cpu().numpy()
        ld = (Tmax + 3) // 4 * 4
        logits = torch.zeros((B, Hq, ld), dtype=torch.float32, device=dev)
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev)
        abi.kivi_decode_qk(cache, q, logits)
        abi.kivi_decode_pv(cache, logits, out, cache.workspace(Hq))
        res[f"split{i}"] = out.view(torch.int32).cpu().numpy()
        res[f"logits{i}"] = logits.view(torch.int32).cpu().numpy()
        fused = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev)
        ws = cache.workspace(Hq)
        abi.kivi_decode_attention(cache, q, fused, ws)
        torch.cuda.synchronize(dev)
        res[f"fused{i}"] = fused.cpu().numpy()
        res[f"fstatus{i}"] = np.int32(ws[:1].view(torch.int32).item())
        n = abi.kivi_payload_bytes(cache.desc, cache.lens.cpu().tolist())
        host = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        abi.kivi_export(cache, host, status)
        torch.cuda.synchronize(dev)
        res[f"payload{i}"] = host.numpy().copy()
        other = KiviCache(B, H, D, bk, bv, G, R, Tmax, device=dev)
        abi.kivi_import(other, host, status)
        torch.cuda.synchronize(dev)
        res[f"imported_vq{i}"] = other.vq.cpu().numpy()
        res[f"appstatus{i}"] = np.int32(status.item())
        res[f"check{i}"] = np.int32(abi.kivi_check_status())
    np.savez(path, **res)


@pytest.mark.gpu
def test_checked_build_passes_every_device_check(tmp_path):
    """Both builds, each in a process of its own; see the module docstring."""
    sys.path.insert(0, ROOT)
    from kivi_bit_kv_gb300 import build
    checked = build.build(variant="checked")
    paths = {}
    for name, lib in (("checked", checked), ("default", None)):
        env = dict(os.environ)
        env.pop("KIVI_LIB", None)
        if lib:
            env["KIVI_LIB"] = lib
        paths[name] = str(tmp_path / f"{name}.npz")
        subprocess.run([sys.executable, os.path.abspath(__file__), paths[name]], env=env, check=True,
                       timeout=900)
    a, b = np.load(paths["checked"]), np.load(paths["default"])
    for i in range(len(CASES)):
        for key in ("check", "fstatus", "appstatus"):
            assert int(a[f"{key}{i}"]) == 0, f"case {i}: {key} {int(a[f'{key}{i}'])} in the checked build"
            assert int(b[f"{key}{i}"]) == 0, f"case {i}: {key}"
        for key in ("kh", "vh", "kq", "kscale", "kzero", "vq", "vscale", "vzero", "kres", "vres", "lens",
                    "logits", "split", "payload", "imported_vq"):
            assert np.array_equal(a[f"{key}{i}"], b[f"{key}{i}"]), f"case {i}: {key}"
        x, y = a[f"fused{i}"], b[f"fused{i}"]
        assert np.isfinite(x).all() and np.isfinite(y).all(), f"case {i}"
        np.testing.assert_allclose(x, y, rtol=1e-5, atol=1e-6, err_msg=f"case {i}")


if __name__ == "__main__":
    run_cases(sys.argv[1])
