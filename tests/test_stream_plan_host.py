"""Host checks of the streamed fused decode's compile-time plan, for every
shape it is instantiated for.

decode_stream_kernel (csrc/decode_stream.cuh) sizes its stage ring, per-warp
scratch and merge area from StreamCfg and relies on invariants that nothing
checks at run time: the shared memory of one CTA holds at least one stage
more than there are consumer warps; every stage region starts on a 16-byte
boundary and lies inside the stage slot (bulk copies and 16-byte loads);
every bulk copy moves a multiple of 16 bytes, for every group size and every
partial tile; the stage's key statistic rows cover the groups of any stage
at G = 32, 64 and 128; the tile sizes are whole key warp tiles and MMA
slices; the per-warp scratch holds the logit rows, the scaled query, the
value weights and the row's query heads.  This test compiles the real header into a host program with
nvcc and enumerates key and value widths {2, 4, 8}, 1, 2 or 4 query heads per
pass and D in {64, 128, 256}.
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
#include "decode_stream.cuh"
using namespace kivi;

template <int BK, int BV, int NQB, int D>
void one(bool& first)
{
    constexpr int NC = stream_consumers<BK, BV, NQB, D>();
    using C = StreamCfg<BK, BV, NQB, D, NC>;
    printf("%s{\"bk\": %d, \"bv\": %d, \"nqb\": %d, \"D\": %d, \"NC\": %d, \"TS\": %d, \"RT\": %d, "
           "\"TOK\": %d, \"PK\": %d, \"DW\": %d, \"NGM\": %d, \"KSR\": %d, "
           "\"O_KW\": %d, \"O_KS\": %d, \"O_KZ\": %d, \"O_VW\": %d, \"O_VS\": %d, \"O_VZ\": %d, \"Q_END\": %d, "
           "\"O_KR\": %d, \"O_VR\": %d, \"R_END\": %d, \"SLOT\": %d, \"LS\": %d, \"QWS\": %d, \"UNITS\": %d, "
           "\"UB\": %d, \"UTS\": %d, \"W_LG\": %d, \"W_QW\": %d, \"W_UB\": %d, \"W_Q\": %d, \"WARP_FLOATS\": %d, "
           "\"M_END\": %d, \"NMB\": %d, \"FIXED\": %d, \"ns\": %d, \"THREADS\": %d}",
           first ? "" : ",\n", BK, BV, NQB, D, NC, C::TS, C::RT, C::TOK, C::PK, C::DW, C::NGM, C::KSR,
           C::O_KW, C::O_KS, C::O_KZ, C::O_VW, C::O_VS, C::O_VZ, C::Q_END, C::O_KR, C::O_VR, C::R_END,
           C::SLOT, C::LS, C::QWS, C::UNITS, C::UB, C::UTS, C::W_LG, C::W_QW, C::W_UB, C::W_Q, C::WARP_FLOATS,
           C::M_END, C::NMB, C::FIXED_BYTES, stream_stages<C>(), C::THREADS);
    first = false;
}
template <int BK, int BV, int D> void nq(bool& f) { one<BK, BV, 1, D>(f); one<BK, BV, 2, D>(f); one<BK, BV, 4, D>(f); }
template <int BK, int D> void bv(bool& f) { nq<BK, 2, D>(f); nq<BK, 4, D>(f); nq<BK, 8, D>(f); }
template <int D> void bk(bool& f) { bv<2, D>(f); bv<4, D>(f); bv<8, D>(f); }
int main()
{
    bool first = true;
    printf("{\"smem\": %d, \"max_ctas\": %d, \"shapes\": [\n", kStreamSmemBytes, kMaxStreamCTAs);
    bk<64>(first);
    bk<128>(first);
    bk<256>(first);
    printf("]}\n");
    return 0;
}
"""


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    d = tmp_path_factory.mktemp("stream_plan")
    src, exe = d / "plan.cu", d / "plan"
    src.write_text(PROGRAM)
    r = subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
                        f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}", "-o", str(exe),
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    return json.loads(out)


def test_every_shape_is_planned(plan):
    assert len(plan["shapes"]) == 81


def test_stages_outnumber_consumers_and_fit(plan):
    for s in plan["shapes"]:
        assert 1 <= s["NC"] <= 8, s
        assert s["THREADS"] == 384  # three warpgroups: 8 consumer warps, 2 producers, 2 idle
        assert s["ns"] >= s["NC"] + 1 and s["ns"] >= 2, s
        assert s["ns"] <= 32, s  # the per-slot consumed counters are a static array of 32
        dyn = s["ns"] * s["SLOT"] + s["FIXED"] - 512 + 2 * 8 * s["ns"]
        # dynamic shared memory plus the kernel's static arrays (< 512 bytes)
        assert dyn + 512 <= plan["smem"], s


def test_stage_slot_regions(plan):
    for s in plan["shapes"]:
        D, TS, RT, PK, DW, NGM = s["D"], s["TS"], s["RT"], s["PK"], s["DW"], s["NGM"]
        assert s["O_KW"] == 0
        assert s["O_KS"] == s["O_KW"] + (TS // PK) * D * 4
        assert s["O_KZ"] == s["O_KS"] + s["KSR"] * D * 4
        assert s["O_VW"] == s["O_KZ"] + s["KSR"] * D * 4
        assert s["O_VS"] == s["O_VW"] + TS * DW * 4
        assert s["O_VZ"] == s["O_VS"] + TS * NGM * 4
        assert s["Q_END"] == s["O_VZ"] + TS * NGM * 4 <= s["SLOT"]
        assert s["O_KR"] == 0 and s["O_VR"] == s["O_KR"] + RT * D * 2
        assert s["R_END"] == s["O_VR"] + RT * D * 2 <= s["SLOT"]
        for k in ("O_KW", "O_KS", "O_KZ", "O_VW", "O_VS", "O_VZ", "O_KR", "O_VR"):
            assert s[k] % 16 == 0, (k, s)
        assert s["SLOT"] % 128 == 0


def test_tile_shapes(plan):
    for s in plan["shapes"]:
        TS, RT = s["TS"], s["RT"]
        assert TS % s["TOK"] == 0 and TS % 16 == 0 and TS >= 32
        assert RT % 16 == 0 and RT <= TS
        assert TS & (TS - 1) == 0  # a power of two: G divides TS or TS divides G
        for G in (32, 64, 128):
            if s["D"] % G:
                continue
            # key statistic rows of a stage (whole groups, or one group holding the stage)
            assert max(1, TS // G) <= s["KSR"]
            assert s["D"] // G <= s["NGM"]


def test_bulk_copy_sizes(plan):
    """Every copy the producer issues is a multiple of 16 bytes, from a source
    offset that is a multiple of 16 bytes, for every group size and every
    length of a partial tile (quantized tiles hold a multiple of G tokens,
    residual tiles any count, split at most once by the ring's end)."""
    for s in plan["shapes"]:
        D, TS, RT, PK, DW = s["D"], s["TS"], s["RT"], s["PK"], s["DW"]
        assert (D * 2) % 16 == 0
        for G in (32, 64, 128):
            if D % G:
                continue
            NG = D // G
            for n in range(G, TS + 1, G) if TS >= G else [TS]:
                assert (n // PK) * D * 4 % 16 == 0
                assert n * DW * 4 % 16 == 0 and n * NG * 4 % 16 == 0
                ngr = -(-n // G)
                assert ngr * D * 4 % 16 == 0
            # source offsets: t0 is a multiple of TS (quantized) and of G
            assert (TS // PK) * D * 4 % 16 == 0 and TS * NG * 4 % 16 == 0
        for n in range(1, RT + 1):
            assert n * D * 2 % 16 == 0


def test_warp_scratch(plan):
    for s in plan["shapes"]:
        nqb = s["nqb"]
        assert s["LS"] >= s["TS"] + 2 * ((s["TS"] - 1) // 16) + 1  # padded logit rows
        assert s["W_QW"] == s["W_LG"] + nqb * s["LS"]
        # the value weights overlay the scaled query (dead once q . K is done)
        assert s["W_UB"] == s["W_QW"]
        assert s["UNITS"] == s["NGM"] * nqb
        assert s["UB"] % 16 == 0 and s["TS"] % s["UB"] == 0 and s["UTS"] >= s["UB"]
        # 2 parts x UNITS rows of UTS fp16 weights
        assert s["W_UB"] + s["UNITS"] * s["UTS"] <= s["W_Q"] and s["W_QW"] + nqb * s["QWS"] <= s["W_Q"]
        # the row's query heads, fp16, in 16-byte pieces
        assert s["W_Q"] % 4 == 0 and s["W_Q"] + nqb * s["D"] // 2 <= s["WARP_FLOATS"]
        assert s["WARP_FLOATS"] % 4 == 0 and s["QWS"] % 4 == 0 and s["LS"] % 2 == 0
