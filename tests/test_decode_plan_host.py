"""Host checks of the decode chunk plan and shared-memory layout, for every
supported shape.

The decode kernels size their shared memory from decode_chunk_plan() and
decode_layout() (csrc/decode_mma.cuh) and rely on invariants that nothing
checks at run time: the layout fits the per-SM budget for the planned number
of resident CTAs; every region starts on a 16-byte boundary (cp.async,
ldmatrix and float4 accesses); the overlays (B fragments on the staged keys,
split partials on the value statistics, zero terms on the logits) fit inside
what they overlay; and no chunk holds more quantized tokens than the TC staged
rows or more tokens than the TC + S logit rows.  The GPU tests cover a
handful of shapes.  This test compiles the real header into a host program
with nvcc and enumerates all of them: D in {64, 128, 256}, key and value
widths in {2, 4, 8}, G in {32, 64, 128}, residuals from 0 to 2^20 tokens, and
1 to 16 query heads per KV head.
"""
import json
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kivi_bit_kv_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <map>
#include <tuple>
#include "decode_mma.cuh"
using namespace kivi;

template <int BITS, int NQB> constexpr int tok() { return KeyTile<BITS, NQB>::TOK; }
static int key_tile_tokens(int bits, int nqb)
{
    switch (bits * 10 + nqb) {
    case 21: return tok<2, 1>(); case 22: return tok<2, 2>(); case 24: return tok<2, 4>();
    case 41: return tok<4, 1>(); case 42: return tok<4, 2>(); case 44: return tok<4, 4>();
    case 81: return tok<8, 1>(); case 82: return tok<8, 2>(); default: return tok<8, 4>();
    }
}

static void layout_json(const char* name, const DecodeLayout& L)
{
    printf("\"%s\": {\"kw\": %zu, \"ks\": %zu, \"kz\": %zu, \"vw\": %zu, \"vs\": %zu, \"vz\": %zu, "
           "\"p\": %zu, \"bb\": %zu, \"part\": %zu, \"zs\": %zu, \"total\": %zu, "
           "\"bb_on_keys\": %d, \"part_on_vstats\": %d, \"zs_on_p\": %d}",
           name, L.kw, L.ks, L.kz, L.vw, L.vs, L.vz, L.p, L.bb, L.part, L.zs, L.total,
           (int)L.bb_on_keys, (int)L.part_on_vstats, (int)L.zs_on_p);
}

// Chunk bounds as the decode kernels derive them (chunk_range): chunk ci of a
// sequence of n tokens covers [ci TC, ci TC + TC), the last one [ci TC, n);
// its quantized tokens end at min(t_end, Tq).
static long chunk_violations(int TC, int S, int G, int R)
{
    static std::map<std::tuple<int, int, int, int>, long> memo;
    const auto key = std::make_tuple(TC, S, G, R);
    const auto hit = memo.find(key);
    if (hit != memo.end())
        return hit->second;
    long bad = 0;
    for (int n = 0; n <= 6 * 1024 + 300; ++n) {
        const int nch = decode_chunks(n, TC, S), Tq = quantized_tokens(n, G, R);
        int covered = 0;
        for (int ci = 0; ci < nch; ++ci) {
            const int tb = ci * TC, te = ci == nch - 1 ? n : tb + TC;
            const int tq_end = tb > (te < Tq ? te : Tq) ? tb : (te < Tq ? te : Tq);
            if (tb != covered || te <= tb || te - tb > TC + S || tq_end - tb > TC || tb % G != 0)
                ++bad;
            covered = te;
        }
        if (covered != n || nch > decode_chunks(n + 1, TC, S))
            ++bad;
    }
    memo[key] = bad;
    return bad;
}

int main()
{
    const int Ds[] = {64, 128, 256}, bitss[] = {2, 4, 8}, Gs[] = {32, 64, 128};
    printf("[\n");
    bool first = true;
    for (int D : Ds)
        for (int bk : bitss)
            for (int bv : bitss)
                for (int G : Gs) {
                    if (D % G != 0)
                        continue;
                    const int Rs[] = {0, G, 2 * G, 4 * G, 1024, 1 << 20};
                    for (int R : Rs)
                        for (int NQ = 1; NQ <= 16; ++NQ) {
                            const ChunkPlan cp = decode_chunk_plan(D, bk, bv, G, R, NQ);
                            const int NQB = heads_per_pass(NQ);
                            const bool mp = NQ > NQB;
                            const int TX = cp.TC + cp.S;
                            printf("%s{\"D\": %d, \"bk\": %d, \"bv\": %d, \"G\": %d, \"R\": %d, \"NQ\": %d, "
                                   "\"NQB\": %d, \"TC\": %d, \"S\": %d, \"ctas\": %d, \"tok\": %d, "
                                   "\"static\": %zu, \"bb_words\": %zu, \"part_words\": %zu, "
                                   "\"zs_words\": %zu, \"p_words\": %zu, \"chunk_violations\": %ld, ",
                                   first ? "" : ",\n", D, bk, bv, G, R, NQ, NQB, cp.TC, cp.S,
                                   cp.ctas_per_sm, key_tile_tokens(bk, NQB), decode_static_smem(D, NQB),
                                   bb_words(TX, D, G, NQB), part_words(D, NQB), zs_words(D, G, NQB),
                                   (size_t)NQB * prob_stride(TX),
                                   chunk_violations(cp.TC, cp.S, G, R));
                            first = false;
                            layout_json("fused", decode_layout(cp.TC, TX, D, bk, bv, G, NQB, mp, true, true,
                                                               cp.zs_on_p));
                            printf(", ");
                            layout_json("qk", decode_layout(cp.TC, TX, D, bk, bv, G, NQB, mp, true, false,
                                                            cp.zs_on_p));
                            printf(", ");
                            layout_json("pv", decode_layout(cp.TC, TX, D, bk, bv, G, NQB, mp, false, true,
                                                            cp.zs_on_p));
                            printf("}");
                        }
                }
    printf("\n]\n");
    return 0;
}
"""

MAX_DYNAMIC_SMEM = 227 * 1024  # per-CTA opt-in limit


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("plan")
    src, exe = d / "plan.cu", d / "plan"
    src.write_text(PROGRAM)
    subprocess.run([nvcc, "-std=c++17", "-O1", f"-I{CSRC}", f"-I{os.path.join(ROOT, 'include')}",
                    str(src), "-o", str(exe)], check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    rows = json.loads(out)
    assert len(rows) > 1000
    return rows


def _regions(L, keys, values, x):
    """(name, start, words) of the regions a layout gives their own words."""
    regs = []
    if keys:
        regs += [("kw", L["kw"], L["ks"] - L["kw"]), ("ks", L["ks"], L["kz"] - L["ks"]),
                 ("kz", L["kz"], L["kz"] - L["ks"])]
    if values:
        regs += [("vw", L["vw"], L["vs"] - L["vw"]), ("vs", L["vs"], L["vz"] - L["vs"]),
                 ("vz", L["vz"], L["vz"] - L["vs"]), ("p", L["p"], x["p_words"])]
        if not L["bb_on_keys"]:
            regs.append(("bb", L["bb"], x["bb_words"]))
        if not L["part_on_vstats"]:
            regs.append(("part", L["part"], x["part_words"]))
        if not L["zs_on_p"]:
            regs.append(("zs", L["zs"], x["zs_words"]))
    return regs


def test_plan_is_well_formed(plans):
    for x in plans:
        TC, S, G = x["TC"], x["S"], x["G"]
        assert TC & (TC - 1) == 0 and 64 <= TC <= 1024, x
        assert TC % G == 0 and TC % x["tok"] == 0, x
        assert S % 16 == 0 and 0 <= S <= min(x["R"], TC // 4), x
        assert 1 <= x["ctas"] <= 3, x
        assert x["chunk_violations"] == 0, x


def test_layouts_fit_the_budget(plans):
    for x in plans:
        budget = 228 * 1024 // x["ctas"] - 1024
        for name in ("fused", "qk", "pv"):
            dyn = 4 * x[name]["total"]
            assert dyn + x["static"] <= budget, (name, x)
            assert dyn <= MAX_DYNAMIC_SMEM, (name, x)


def test_regions_are_aligned_disjoint_and_inside(plans):
    for x in plans:
        for name, keys, values in (("fused", True, True), ("qk", True, False), ("pv", False, True)):
            L = x[name]
            regs = _regions(L, keys, values, x)
            for r, start, n in regs:
                assert start % 4 == 0, (name, r, x)  # 16-byte boundary
                assert start + n <= L["total"], (name, r, x)
            spans = sorted((s, s + n, r) for r, s, n in regs if n > 0)
            for (s0, e0, r0), (s1, e1, r1) in zip(spans, spans[1:]):
                assert e0 <= s1, (name, r0, r1, x)


def test_overlays_fit_what_they_overlay(plans):
    for x in plans:
        L = x["fused"]
        key_words = L["vw"] - L["kw"]
        vstat_words = 2 * (L["vz"] - L["vs"])
        if L["bb_on_keys"]:
            assert L["bb"] == L["kw"] and x["bb_words"] <= key_words, x
        if L["part_on_vstats"]:
            assert L["part"] == L["vs"] and x["part_words"] <= vstat_words, x
            assert x["NQ"] == x["NQB"], x  # one pass: the statistics are dead after it
        if L["zs_on_p"]:
            assert L["zs"] == L["p"] and x["zs_words"] <= x["p_words"], x
