"""Host-side checks of the small-batch decode kernel's launch plan.

The plan (gsi_plan.h, integer arithmetic only) places every shared-memory
region of the kernel, the tensor-map boxes its copies land in and the W ring
that reuses the call's scratch; a region that overlaps another, a box that is
not 1024-byte aligned (128-byte swizzle) or an index past its buffer would
only show on a GPU.  A small C++ harness (batch_plan_dump.cpp) prints plans
for the 6B and 13B maps, ragged and random shapes, and this test replays the
kernel's address arithmetic for each plan on the CPU.
"""
import json
import os
import random
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "gated_rank_subspace_gb300", "csrc")
BUDGET = 232448  # shared memory a CTA may opt into on an sm_100-class GPU

SHAPES_6B = [(4096, 12288, 256), (4096, 4096, 256), (4096, 16384, 256), (16384, 4096, 256)]
SHAPES_13B = [(5120, 15360, 320), (5120, 5120, 320), (5120, 13824, 320), (13824, 5120, 320)]


def cases():
    out = []
    for ncta in (112, 128, 144):
        for T in (2, 3, 4, 8, 9, 16):
            for d, d_out, k in SHAPES_6B + SHAPES_13B:
                out.append((d, d_out, k, T, ncta))
            out += [(520, 333, 64, T, ncta), (1032, 2056, 128, T, ncta), (16, 8, 64, T, ncta),
                    (8200, 520, 64, T, ncta), (4096, 4096, 384, T, ncta), (4096, 4096, 512, T, ncta),
                    (4104, 12296, 192, T, ncta)]
    rng = random.Random(11)
    for _ in range(400):
        k = 64 * rng.randint(1, 8)
        d = 8 * rng.randint(2, 40000 // 8)
        d_out = rng.randint(1, 20000)
        out.append((d, d_out, k, rng.randint(1, 17), 16 * rng.randint(1, 16)))
    return out


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ is not available")
    exe = str(tmp_path_factory.mktemp("bplan") / "batch_plan_dump")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "batch_plan_dump.cpp"), "-o", exe],
                   check=True)
    lines = [f"{d} {d_out} {k} {T} {ncta} {BUDGET}" for d, d_out, k, T, ncta in cases()]
    r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
    return [json.loads(x) for x in r.stdout.splitlines()]


def test_benchmark_maps_fit(plans):
    # every 6B and 13B map fits at T = 2 .. 16 on a grid of 112 CTAs (7 clusters)
    for p in plans:
        if p["ncta"] == 112 and 2 <= p["T"] <= 16 and (p["d"], p["d_out"], p["k"]) in SHAPES_6B + SHAPES_13B:
            assert p["ok"], p


def test_rejects_out_of_range(plans):
    for p in plans:
        if p["T"] < 2 or p["T"] > p["maxT"] or p["k"] % 64 or p["k"] > p["max_k"] or p["d"] % 8:
            assert not p["ok"], p


def test_regions_and_indices(plans):
    n_ok = 0
    for p in plans:
        if not p["ok"]:
            continue
        n_ok += 1
        d, d_out, k, T, ncta = p["d"], p["d_out"], p["k"], p["T"], p["ncta"]
        vr, rpc, ks, kb, S, SB = p["vr"], p["rpc"], p["ks"], p["kb"], p["stages"], p["stage_bytes"]
        maxT, CS, NW = p["maxT"], p["cluster"], p["warps"]
        limit = p["smem"] - p["slack"]  # bytes usable after aligning the base to 1024
        assert p["smem"] <= p["budget"]
        # grid covers the map
        assert vr % 16 == 0 and rpc % 16 == 0 and vr * ncta >= d and rpc * ncta >= d_out
        assert rpc <= 16 * p["max_mt"] and vr <= 256 and rpc <= 256  # box heights
        assert ks * CS == k and kb * 64 == k and ks % 2 == 0
        # regions in order, non-overlapping, inside the limit
        regions = [
            ("bars", 0, 512 + 8), ("gbf", p["off_gbf"], 2 * maxT * p["gbf_pitch"]),
            ("dec", p["off_dec"], 2 * maxT * 4), ("wsh", p["off_wsh"], NW * maxT * 2 * 4),
            ("fs", p["off_fs"], T * ks * 4 + maxT * 4), ("nx", p["off_nx"], maxT * 4),
            ("v", p["off_v"], kb * vr * 128), ("xs", p["off_xs"], maxT * p["xs_pitch"]),
            ("in", p["off_in"], CS * T * ks * 4), ("nin", p["off_nin"], CS * maxT * 4),
            ("g32", p["off_g32"], T * k * 4 + maxT * 4), ("qin", p["off_qin"], CS * maxT * 8),
            ("gram", p["off_gram"], ks * k * 4), ("m", p["off_m"], kb * rpc * 128)]
        end = 0
        for name, off, size in regions:
            assert off >= end, (name, p)
            end = off + size
        assert end <= limit, p
        # barriers: 8 named + 2 x stages, below the words at 512
        assert (8 + 2 * p["max_stages"]) * 8 <= 512
        # swizzled boxes start on 1024-byte boundaries, bulk copies on 16
        for off in (p["off_scr"], p["off_v"], p["off_m"]):
            assert off % 1024 == 0, p
        assert (vr * 128) % 1024 == 0 and (rpc * 128) % 1024 == 0 and SB % 1024 == 0
        assert p["off_gram"] % 16 == 0 and p["gbf_pitch"] % 16 == 0 and p["xs_pitch"] % 16 == 0
        assert p["off_in"] % 8 == 0 and p["off_nin"] % 8 == 0 and p["off_g32"] % 16 == 0 and p["off_qin"] % 8 == 0
        # the scratch starts after the regions that live through the call
        assert p["off_scr"] >= p["off_nx"] + maxT * 4 and p["off_scr"] <= p["off_v"]
        # the partial g by column slice [16][T][ks] float32 fits in the bf16 g region it precedes
        assert T * k * 4 <= 2 * maxT * p["gbf_pitch"]
        # bulk copies between CTAs: 16-byte aligned sources, destinations and sizes
        assert (T * ks * 4) % 16 == 0 and p["off_fs"] % 16 == 0 and p["off_nx"] % 16 == 0
        assert p["off_in"] % 16 == 0 and p["off_nin"] % 16 == 0 and p["off_gbf"] % 16 == 0
        assert p["off_g32"] % 16 == 0 and (T * k * 4) % 16 == 0
        # ring: S stages of W (2 boxes of rpc rows) + X (2 boxes of up to 16 rows), inside the limit
        assert 2 <= S <= p["max_stages"]
        assert SB >= 2 * rpc * 128 + 2 * maxT * 128
        assert p["off_scr"] + S * SB <= limit, p
        # the warps' partial sums [NW][16][rpc] float32 fit the ring
        assert NW * maxT * rpc * 4 <= S * SB
        # token slab: vectors written and fragments read stay in a row
        assert (vr // 8) * 16 <= p["xs_pitch"] and ((vr // 16 - 1) * 2 + 1) * 16 + 16 <= p["xs_pitch"]
        # g in bf16: the last chunk read of a token row stays inside its pitch
        assert (k // 8) * 16 <= p["gbf_pitch"]
        # workspace words: [16 clusters][T][k] and [16 clusters][16]
        assert p["ws_part_x"] - p["ws_part_g"] >= p["max_clusters"] * T * k * 8
        assert p["ws_total"] - p["ws_part_x"] >= p["max_clusters"] * maxT * 8
        assert ncta // CS <= p["max_clusters"]
        # exchange items: the reduce loop covers T * ks / 2 pairs (+ 8 norm pairs)
        assert T * (ks // 2) + maxT // 2 <= 2 * NW * 32 + NW * 32
        # share pushes: one thread per (token, rank)
        assert T * CS <= NW * 32
    assert n_ok > 100
