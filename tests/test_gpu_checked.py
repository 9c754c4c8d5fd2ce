"""The bounds-checked build of the library (KIVI_CHECKS defined) on the fused
decode's hardest shapes.

In that build the streamed decode checks, on the device, that every copy it
issues reads inside the cache arrays and lands inside its shared-memory
region, that every tile lies inside its sequence, and that every output row
and partial slot it writes exists; the combine kernel checks its pieces and
rows.  A failed check would leave KIVI_ECHECK in the workspace status word.
Each case below runs through both builds (each in a process of its own,
KIVI_LIB selecting the checked library): the status word stays KIVI_OK and the
outputs of the two builds agree.  They agree to rounding order, not bit for
bit: which consumer warp takes which tile varies from run to run.
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
    """Encodes and decodes every case with the library KIVI_LIB names (or the
    default one) and saves outputs and status words to `path`."""
    sys.path.insert(0, ROOT)
    import torch
    from kivi_bit_kv_gb300 import KiviCache, abi
    dev = torch.device("cuda", 0)
    res = {}
    for i, (B, H, Hq, D, bk, bv, G, R, lens) in enumerate(CASES):
        g = torch.Generator().manual_seed(100 + i)
        T = max(lens)
        Tmax = (T + G) // G * G + G
        K = torch.randn((B, H, T, D), generator=g).to(torch.float16).to(dev)
        V = torch.randn((B, H, T, D), generator=g).to(torch.float16).to(dev)
        q = torch.randn((B, Hq, D), generator=g).to(torch.float16).to(dev)
        cache = KiviCache(B, H, D, bk, bv, G, R, Tmax, device=dev)
        sl = torch.tensor(lens, dtype=torch.int32, device=dev)
        abi.kivi_quant_keys(cache, K, sl)
        abi.kivi_quant_values(cache, V, sl)
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=dev)
        ws = cache.workspace(Hq)
        abi.kivi_decode_attention(cache, q, out, ws)
        torch.cuda.synchronize(dev)
        res[f"out{i}"] = out.cpu().numpy()
        res[f"status{i}"] = np.int32(ws[:1].view(torch.int32).item())
    np.savez(path, **res)


@pytest.mark.gpu
def test_checked_build_passes_every_device_check(tmp_path):
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
        assert int(a[f"status{i}"]) == 0, f"case {i}: a device check failed (status {int(a[f'status{i}'])})"
        assert int(b[f"status{i}"]) == 0
        x, y = a[f"out{i}"], b[f"out{i}"]
        assert np.isfinite(x).all() and np.isfinite(y).all(), f"case {i}"
        np.testing.assert_allclose(x, y, rtol=1e-5, atol=1e-6, err_msg=f"case {i}")


if __name__ == "__main__":
    run_cases(sys.argv[1])
