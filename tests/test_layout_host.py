"""Host-only checks of the main kernel's pipeline layout (csrc/qmm_layout.h) for
every code format, row tile and consumer layout the library compiles: the
activation-slot ownership rule the staging warps rely on, the stage and slot
counts the two consumer parities need, the shared-memory opt-in limit and the
register budget of one CTA per SM. The header is plain C++ without CUDA; a
small program built with the host compiler prints its values. No GPU needed."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "bit_affine_quantized_group_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "qmm_layout.h"
using namespace qmmk;
int main() {
    const int bits[] = {2, 3, 4, 5, 6, 8};
    const int groups[] = {32, 64};
    const int mbs[] = {8, 16};
    const int lays[] = {kNarrow, kWide, kPair};
    for (int b : bits) for (int g : groups) for (int mb : mbs) for (int lay : lays) {
        if (mb == 16 && lay == kWide) continue;   // not compiled
        std::printf("%d %d %d %d %d %d %d %d %d %d\n", b, g, mb, lay, stage_count(b, g, mb, lay),
                    act_slots(b, g, mb, lay), staging_per_tile(mb, g, lay), consumer_parities(lay),
                    main_smem_bytes(b, g, mb, lay), main_threads(mb, g, lay));
    }
    std::printf("optin %d\n", kSmemOptin);
    return 0;
}
"""


@pytest.fixture(scope="module")
def layouts(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("layout")
    src = d / "layout.cpp"
    src.write_text(PROGRAM)
    exe = d / "layout"
    subprocess.run([cxx, "-std=c++17", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    optin = int([l for l in out if l.startswith("optin")][0].split()[1])
    rows = [tuple(int(v) for v in l.split()) for l in out if l and not l.startswith("optin")]
    return rows, optin


def test_every_configuration_is_listed(layouts):
    rows, _ = layouts
    assert len(rows) == 6 * 2 * (3 + 2)


def test_slot_ownership_and_parities(layouts):
    """Each staging warp owns whole slots (F at most the warps per tile, or a
    multiple of them), so every phase of a slot's barriers is awaited by one warp
    in order; both consumer parities own as many weight stages and slots."""
    rows, _ = layouts
    for b, g, mb, lay, S, F, spt, cpar, smem, threads in rows:
        cfg = (b, g, mb, lay)
        assert F >= 2 and (F <= spt or F % spt == 0), cfg
        assert F % cpar == 0, cfg
        if S:
            assert S >= 2 and S % cpar == 0, cfg


def test_narrow_layout_always_fits(layouts):
    """The narrow layout serves every call, so it must have at least two weight
    stages in the opt-in shared memory for every format and row tile."""
    rows, optin = layouts
    for b, g, mb, lay, S, F, spt, cpar, smem, threads in rows:
        if lay == 0:
            assert S >= 2 and smem <= optin, (b, g, mb)


def test_shared_memory_and_registers(layouts):
    """A configuration with stages fits the opt-in limit, and its CTA fits one
    SM's 64 K registers at no fewer than 128 registers a thread: at most four
    warps share one of the four schedulers."""
    rows, optin = layouts
    for b, g, mb, lay, S, F, spt, cpar, smem, threads in rows:
        if S == 0:
            continue
        assert smem <= optin, (b, g, mb, lay)
        warps = threads // 32
        assert warps <= 16 and (warps + 3) // 4 * 4 * 32 * 128 <= 65536, (b, g, mb, lay, warps)


def test_wide_groups_of_32_take_three_staging_warps(layouts):
    """The 8-row wide kernel with groups of 32 runs 12 warps (8 consumers, 3
    staging, 1 producer): three a scheduler, so up to 168 registers a thread."""
    rows, _ = layouts
    for b, g, mb, lay, S, F, spt, cpar, smem, threads in rows:
        if mb == 8 and lay == 1 and g == 32:
            assert threads == 12 * 32 and spt == 3, (b, g)
