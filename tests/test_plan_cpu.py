"""Host-side checks of the single-token decode kernel's launch plan.

The plan (gsi_plan.h, pure integer arithmetic) places every shared-memory
region of the kernel and sizes its W rings; a region that overlaps another,
runs past the budget or breaks a bulk copy's 16-byte alignment would only
show on a GPU.  A small C++ harness (plan_dump.cpp) prints the plans for many
shapes -- the 6B and 13B maps, config 1, ragged and random shapes, several
grid sizes and both element types -- and this test checks them on the CPU.
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

SHAPES_6B = [(4096, 12288), (4096, 4096), (4096, 16384), (16384, 4096)]
SHAPES_13B = [(5120, 15360), (5120, 5120), (5120, 13824), (13824, 5120)]


def cases():
    out = []
    for ncta in (112, 128, 144):
        for d, d_out in SHAPES_6B:
            out += [(d, d_out, 256, 2, ncta), (d, d_out, 64, 2, ncta)]
        for d, d_out in SHAPES_13B:
            out.append((d, d_out, 320, 2, ncta))
        out += [(256, 256, 16, 4, ncta), (520, 333, 24, 2, ncta), (1032, 2056, 40, 2, ncta), (16, 8, 8, 2, ncta),
                (8200, 520, 64, 2, ncta), (512, 512, 64, 2, ncta), (4096, 4096, 128, 4, ncta)]
    rng = random.Random(7)
    for _ in range(300):
        es = rng.choice((2, 4))
        step = 8 if es == 2 else 4
        k = step * rng.randint(1, 512 // step)
        d = step * rng.randint(1, 20000 // step)
        d_out = rng.randint(1, 20000)
        out.append((d, d_out, k, es, 16 * rng.randint(1, 16)))
    return out


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ is not available")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_dump")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "plan_dump.cpp"), "-o", exe],
                   check=True)
    lines = []
    for d, d_out, k, es, ncta in cases():
        for grid in (0, 1):
            lines.append(f"{d} {d_out} {k} {es} {ncta} {BUDGET} {grid}")
    r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
    return [json.loads(x) for x in r.stdout.splitlines()]


def cdiv(a, b):
    return -(-a // b)


def test_plans_cover_the_benchmark_maps(plans):
    """Every 6B map at k = 256 has a plan on a 112-CTA grid: the cluster
    projection for the 4096-wide maps, the grid projection for the down map;
    the 13B maps (k = 320) have grid-projection plans."""
    by = {(p["d"], p["d_out"], p["k"], p["es"], p["ncta"], p["grid_req"]): p for p in plans}
    for d, d_out in SHAPES_6B:
        cl, gr = by[(d, d_out, 256, 2, 112, 0)], by[(d, d_out, 256, 2, 112, 1)]
        if d == 4096:
            assert cl["ok"] and not cl["grid"]
        else:
            assert not cl["ok"] and gr["ok"] and gr["grid"]
    for d, d_out in SHAPES_13B:
        assert by[(d, d_out, 320, 2, 112, 1)]["ok"]


def test_plan_invariants(plans):
    n_ok = 0
    for p in plans:
        if not p["ok"]:
            continue
        n_ok += 1
        d, d_out, k, es, ncta = p["d"], p["d_out"], p["k"], p["es"], p["ncta"]
        nw, cs = p["nw"], p["cluster"]
        mrow_b, row_b = k * es, d * es
        ctx = json.dumps(p)
        # what a plan promises the kernel
        assert p["smem"] <= p["budget"], ctx
        assert p["grid"] == p["grid_req"], ctx
        assert mrow_b % 16 == 0 and row_b % 16 == 0 and k % 4 == 0, ctx
        assert cdiv(mrow_b, 16) <= 64, ctx                       # at most two vectors a lane
        assert p["rw"] <= 32 and nw * p["rw"] >= p["vr"], ctx    # one token element a lane
        assert p["vr"] * (ncta if p["grid"] else cs) >= d, ctx   # every V row projected
        assert p["rpc"] * ncta >= d_out, ctx                     # every output row applied
        assert p["ks"] * cs >= k, ctx                            # every column owned by a rank
        if p["grid"]:
            assert k % cs == 0 and ncta <= cs * p["max_clusters"], ctx
        # regions in order, 128-byte aligned, no overlap
        bars = (nw + p["bars"] + nw * p["max_stages"]) * 8
        # the CTA words (call epoch / launch number, error flag) follow the
        # mbarriers at one offset for every map, before the g area
        assert p["words_off"] == bars and p["words_off"] % 4 == 0, ctx
        bars += 4 * p["words"]
        g_bytes = (k + cs + 2 * cs * nw + 4 + nw * 32) * 4
        regions = [("g", p["off_g"], g_bytes), ("y", p["off_y"], p["rpc"] * 4),
                   ("in", p["off_in"], max(cs * p["ks"] * 4, row_b)), ("gram", p["off_gram"], p["ks"] * k * 4)]
        alias = p["off_red"] == p["off_v"]
        if not alias:
            regions.append(("red", p["off_red"], nw * (k + 4) * 4))
        assert p["off_g"] >= bars, ctx
        end = 0
        for name, off, size in regions:
            assert off % 128 == 0, (name, ctx)
            assert off >= end, (name, ctx)
            end = off + size
        assert p["off_v"] >= end and p["off_v"] % 128 == 0, ctx
        v_bytes = nw * p["rw"] * mrow_b
        m_bytes = p["rpc"] * mrow_b
        assert p["off_v"] + v_bytes <= p["smem"], ctx
        assert p["off_m"] % 16 == 0 and p["off_m"] + m_bytes <= p["smem"], ctx
        if p["m_late"]:
            assert p["off_m"] == p["off_v"] and not alias, ctx
        else:
            assert p["off_m"] >= p["off_v"] + v_bytes, ctx
        # a warp's partial g and ||x||^2 fit its slot (its own V rows when aliased)
        if alias:
            assert p["red_stride"] * 4 == p["rw"] * mrow_b and p["rw"] * mrow_b >= (k + 4) * 4, ctx
        else:
            assert p["red_stride"] == k + 4, ctx
        assert p["red_stride"] * 4 % 16 == 0, ctx
        # the W rings of a slow token fit the V / M space (and what follows it)
        assert p["seg_bytes"] == min(row_b, 4096) and p["seg_bytes"] % 16 == 0, ctx
        assert 2 <= p["sw"] <= p["max_stages"], ctx
        assert p["off_v"] + nw * p["sw"] * p["seg_bytes"] <= p["smem"], ctx
        # the mbarriers initialised by the kernel (one per thread, every ring
        # slot a map could use) fit the bars region
        assert nw + p["bars"] + nw * p["max_stages"] <= 256, ctx
        # grid projection: the clusters' epoch-tagged words fit the workspace's
        # partial areas ([clusters][k] and [clusters] 64-bit words)
        if p["grid"]:
            assert p["ws_part_g"] >= (ncta // cs) * k * 8 and p["ws_part_x"] >= (ncta // cs) * 8, ctx
    assert n_ok > 100
