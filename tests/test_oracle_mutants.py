"""Planted mistakes in the CPU oracle must fail its pins.

Each mutant below is a copy of kivi_ref.c with one plausible mistake: a
wrong rounding mode, a dropped or swapped term, an off-by-one, a transposed
index, a wrong byte order.  Every copy is compiled with the oracle's own
flags, and the pin suite (test_oracle_pins.py and the oracle payload tests)
runs against it in a child process, with KIVI_REF_LIB pointing the oracle at
that build.  A mutant passes this test only if some pin fails on it.  The
unmodified source, compiled the same way, must pass every pin; that control
shows that the mutants fail for their mistake and not for the harness.  The
same is done for the oracle's Python front end (oracle/ref.py): each mutant
there runs the pins from a copy of oracle/ and tests/ whose ref.py carries
the mistake.

Nothing here touches a GPU or the CUDA library.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from oracle import build as oracle_build  # noqa: E402

PINS = [
    "tests/test_oracle_pins.py",
    "tests/test_payload_host.py::test_fnv1a64_specification_vectors",
    "tests/test_payload_host.py::test_oracle_payload_layout",
    "tests/test_payload_host.py::test_oracle_payload_round_trip",
]

# name -> (text in kivi_ref.c, replacement).  Each text occurs exactly once.
MUTANTS = {
    # codes
    "code_ties_away_from_zero": ("c = (int)nearbyintf(qf);", "c = (int)roundf(qf);"),
    "scale_over_2_pow_b": ("float s = range / (float)M;", "float s = range / (float)(M + 1);"),
    "zero_is_the_maximum": ("*zero = mn;", "*zero = mx;"),
    "scan_skips_an_element": ("for (int i = 1; i < n; ++i) {", "for (int i = 2; i < n; ++i) {"),
    "offset_from_the_maximum": ("volatile float a = v - mn;", "volatile float a = mx - v;"),
    "split_off_by_one": ("int n = T - R;", "int n = T - R + 1;"),
    # packing
    "pack_big_endian": ("w |= ((uint32_t)codes[i]) << (i * bits);",
                        "w |= ((uint32_t)codes[i]) << ((P - 1 - i) * bits);"),
    "unpack_mask_too_wide": ("uint32_t mask = (1u << bits) - 1u;", "uint32_t mask = (2u << bits) - 1u;"),
    "value_code_reversed": ("return codes[d % P];", "return codes[P - 1 - d % P];"),
    "key_word_of_the_next_channel": ("kref_unpack_word(kq[(size_t)(t / P) * D + d], bits, codes);",
                                     "kref_unpack_word(kq[(size_t)(t / P) * D + (d ^ 1)], bits, codes);"),
    "value_groups_overlap": ("const uint16_t* row = V + (size_t)t * D + (size_t)g * G;",
                             "const uint16_t* row = V + (size_t)t * D + (size_t)g;"),
    # dequantization and fp16
    "dequant_without_fma": ("return kref_float_to_half(fmaf((float)code, scale, zero));",
                            "return kref_float_to_half((float)code * scale + zero);"),
    "half_ties_away_from_zero": ("if (diff > 0.5 || (diff == 0.5 && fmod(r, 2.0) != 0.0))",
                                 "if (diff >= 0.5)"),
    "half_subnormal_scale": ("v = ldexpf((float)mant, -24);", "v = ldexpf((float)mant, -25);"),
    # residual ring and append
    "ring_slot_from_the_split": ("kres[(size_t)(t % RG) * D + d] = K[(size_t)t * D + d];",
                                 "kres[(size_t)(t - Tq) * D + d] = K[(size_t)t * D + d];"),
    "flush_at_R_tokens": ("if (len - Tq == RG) {", "if (len - Tq == R + 1) {"),
    # attention
    "softmax_not_normalized": ("acc += (s[t] / sum) *", "acc += s[t] *"),
    "softmax_scale_dropped": ("s[t] = (double)sm_scale * acc;", "s[t] = acc;"),
    "every_head_uses_head_0": ("const uint16_t* qh = q + (size_t)h * D;", "const uint16_t* qh = q;"),
    "key_hat_stats_of_next_channel": ("        size_t si = (size_t)(t / G) * D + d;\n        return (double)key_code",
                                      "        size_t si = ((size_t)(t / G) * D + d) ^ 1;\n"
                                      "        return (double)key_code"),
    "value_hat_stats_of_group_0": ("size_t si = (size_t)t * (D / G) + d / G;", "size_t si = (size_t)t * (D / G);"),
    # storage accounting and payload
    "key_stats_counted_once": ("size_t stats = which == 0 ? (Tq / (size_t)G) * (size_t)D * 8",
                               "size_t stats = which == 0 ? (Tq / (size_t)G) * (size_t)D * 4"),
    "fnv_prime": ("h *= 1099511628211ull;", "h *= 1099511628213ull;"),
    "payload_big_endian": ("out[k] = (uint8_t)(v >> (8 * k));", "out[k] = (uint8_t)(v >> (8 * (3 - k)));"),
    "payload_ring_bytes_swapped": ("bytes[o] = (uint8_t)(row[d] & 0xFFu);\n"
                                   "                bytes[o + 1] = (uint8_t)(row[d] >> 8);",
                                   "bytes[o] = (uint8_t)(row[d] >> 8);\n"
                                   "                bytes[o + 1] = (uint8_t)(row[d] & 0xFFu);"),
    "payload_key_zero_before_scale": ("    o += words_io(io + o, ks, (size_t)(Tq / G) * D, put);\n"
                                      "    o += words_io(io + o, kz, (size_t)(Tq / G) * D, put);",
                                      "    o += words_io(io + o, kz, (size_t)(Tq / G) * D, put);\n"
                                      "    o += words_io(io + o, ks, (size_t)(Tq / G) * D, put);"),
}


# Mistakes in the Python front end of the oracle (oracle/ref.py), which maps
# query heads to KV heads, applies the default softmax scale, honours ragged
# lengths and keeps the append bookkeeping.
PY_MUTANTS = {
    "gqa_heads_interleaved": ("qs = np.ascontiguousarray(q[b, h * NQ:(h + 1) * NQ])",
                              "qs = np.ascontiguousarray(q[b, h::self.H])"),
    "default_scale_1_over_D": ("sm = float(1.0 / np.sqrt(D)) if sm_scale is None else float(sm_scale)",
                               "sm = float(1.0 / D) if sm_scale is None else float(sm_scale)"),
    "encode_ignores_lengths": ("Tb = int(lens[b])\n", "Tb = T\n"),
    "append_keeps_the_length": ("                self.lens[b] = new", "                self.lens[b] = n"),
    "append_ignores_overflow": ("            if new < 0:\n                overflow[b] = True",
                                "            if False:\n                overflow[b] = True"),
}


def _copy_tree(dst: str, ref_text: str):
    """The oracle and the tests under dst, with ref.py replaced by ref_text."""
    ignore = shutil.ignore_patterns("__pycache__", "*.so", "*.so.tmp*")
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"), ignore=ignore)
    shutil.copytree(os.path.join(ROOT, "tests"), os.path.join(dst, "tests"), ignore=ignore)
    with open(os.path.join(dst, "oracle", "ref.py"), "w") as f:
        f.write(ref_text)


def _compile(src_text: str, out: str):
    src = out[:-3] + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    cmd = ["gcc", *oracle_build.CFLAGS, f"-I{os.path.dirname(oracle_build.SRC)}", src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)


def _run_pins(lib: str | None, root: str = ROOT) -> subprocess.CompletedProcess:
    env = dict(os.environ)
    env.pop("KIVI_REF_LIB", None)
    if lib:
        env["KIVI_REF_LIB"] = lib
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu", *PINS]
    return subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)


def test_mutant_texts_are_unique():
    src = open(oracle_build.SRC).read()
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, name
        assert old != new, name
    py = open(os.path.join(ROOT, "oracle", "ref.py")).read()
    for name, (old, new) in PY_MUTANTS.items():
        assert py.count(old) == 1, name
        assert old != new, name


def test_every_planted_mistake_in_the_front_end_fails_a_pin(tmp_path):
    py = open(os.path.join(ROOT, "oracle", "ref.py")).read()
    texts = {"control": py}
    texts.update({name: py.replace(old, new) for name, (old, new) in PY_MUTANTS.items()})
    for name, text in texts.items():
        _copy_tree(str(tmp_path / name), text)
    with ThreadPoolExecutor(max(2, min(8, os.cpu_count() or 2))) as ex:
        results = dict(zip(texts, ex.map(lambda n: _run_pins(None, str(tmp_path / n)), texts)))
    control = results.pop("control")
    assert control.returncode == 0, "unmodified front end failed its pins:\n" + control.stdout[-2000:]
    survivors = [n for n, r in results.items() if r.returncode == 0]
    assert not survivors, f"planted mistakes that no pin catches: {survivors}"
    crashed = [n for n, r in results.items() if r.returncode not in (0, 1)]
    assert not crashed, {n: results[n].stdout[-500:] for n in crashed}


def test_every_planted_mistake_fails_a_pin(tmp_path):
    src = open(oracle_build.SRC).read()
    builds = {"control": str(tmp_path / "control.so")}
    texts = {"control": src}
    for name, (old, new) in MUTANTS.items():
        builds[name] = str(tmp_path / f"{name}.so")
        texts[name] = src.replace(old, new)
    workers = max(2, min(16, os.cpu_count() or 2))
    with ThreadPoolExecutor(workers) as ex:
        list(ex.map(lambda n: _compile(texts[n], builds[n]), builds))
        results = dict(zip(builds, ex.map(lambda n: _run_pins(builds[n]), builds)))
    control = results.pop("control")
    assert control.returncode == 0, "unmodified oracle failed its pins:\n" + control.stdout[-2000:]
    survivors = [n for n, r in results.items() if r.returncode == 0]
    assert not survivors, f"planted mistakes that no pin catches: {survivors}"
    # a mutant must fail a pin, not crash the interpreter or the collection
    crashed = [n for n, r in results.items() if r.returncode not in (0, 1)]
    assert not crashed, {n: results[n].stdout[-500:] for n in crashed}
