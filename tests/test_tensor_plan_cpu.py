"""Host-side checks of the tensor-core path's workspace layout and of its
finalize plan (the per-token norms pass and the Gram form).

The plan (gsi_plan.h, integer arithmetic only) sizes the workspace regions
of a call, the Gram form's row blocks (one thread-block cluster per 16-token
chunk), its shared-memory ring and the bulk copies that fill it; an
overlapping region, a cluster above the portable size, a copy that is not a
multiple of 16 bytes or a transaction count past an mbarrier's limit would
only show on a GPU.  A small C++ harness (tensor_plan_dump.cpp) prints plans
for the benchmark's prefill map, the 13B widths and random shapes, and this
test replays the kernels' index arithmetic for each plan on the CPU.
"""
import json
import os
import random
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "gated_rank_subspace_gb300", "csrc")
SMEM_MAX = 232448 - 1024  # dynamic shared memory a CTA may opt into, less the static part's allowance
MBAR_TX_MAX = (1 << 20) - 1  # an mbarrier phase's transaction count


def cases():
    out = [(4096, 256, 2048), (5120, 320, 2048), (4096, 256, 129), (1032, 136, 300), (512, 64, 160),
           (2048, 320, 160), (1024, 512, 136), (16384, 256, 4096), (13824, 320, 17), (4096, 512, 1)]
    rng = random.Random(5)
    for _ in range(600):
        k = 8 * rng.randint(1, 64)  # bf16 maps: k a multiple of 8, at most 512
        d = max(k, 8 * rng.randint(1, 3000))
        out.append((d, k, rng.choice([rng.randint(1, 40), rng.randint(1, 5000)])))
    return out


@pytest.fixture(scope="module")
def plans(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ is not available")
    exe = str(tmp_path_factory.mktemp("tplan") / "tensor_plan_dump")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "tensor_plan_dump.cpp"), "-o", exe],
                   check=True)
    lines = [f"{d} {k} {T}" for d, k, T in cases()]
    r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
    return [json.loads(x) for x in r.stdout.splitlines()]


def cdiv(a, b):
    return -(-a // b)


def test_workspace_regions(plans):
    for p in plans:
        d, k, T, F = p["d"], p["k"], p["T"], p["fin_tok"]
        regions = [("ctrl", p["ctrl"], 256), ("vt", p["vt"], k * d * 2), ("g", p["g"], p["gsplit"] * T * k * 4),
                   ("gbf", p["gbf"], T * k * 2), ("gfast", p["gfast"], T * k * 2), ("xslow", p["xslow"], T * d * 2),
                   ("idx", p["idx"], 2 * T * 4), ("gt", p["gt"], cdiv(T, F) * F * k * 4), ("norms", p["norms"], T * 8)]
        end = 0
        for name, off, size in regions:
            assert off >= end and off % 256 == 0, (name, p)
            end = off + size
        assert end <= p["total"], p
        assert p["gsplit"] <= p["gsplit_max"]


def test_gram_form_plan(plans):
    for p in plans:
        k, T, nb, F = p["k"], p["T"], p["nb"], p["fin_tok"]
        # a portable cluster of row blocks, each with at least one Gram row
        assert 1 <= nb <= p["fin_max_blocks"] <= 8, p
        for b in range(nb):
            i0, i1 = k * b // nb, k * (b + 1) // nb
            assert i1 > i0, p
        # about three CTAs an SM of a GB300 where k allows it
        chunks = cdiv(T, F)
        if chunks * nb < 456:
            assert nb == min(p["fin_max_blocks"], max(1, k // 32)), p
        # passes over the Gram and the ring of bulk copies, one a row
        npass = 1 if k <= p["fin_cols"] else 2
        assert k <= npass * p["fin_cols"] <= 512
        ks = npass * p["fin_cols"]                     # ring row stride (floats)
        rows = p["fin_stage_bytes"] // (ks * 4)         # Gram rows a stage
        assert 1 <= rows <= 32                         # one copy warp lane a row
        assert (k * 4) % 16 == 0 and k * 4 <= ks * 4   # a row copy: 16-byte multiple, inside its slot
        assert rows * k * 4 <= MBAR_TX_MAX             # a stage's transactions
        assert F * k * 4 <= MBAR_TX_MAX and (F * k * 4) % 16 == 0  # the chunk's g, one copy
        # shared memory: ring, g by row, the warps' q partials
        need = p["fin_stages"] * p["fin_stage_bytes"] + F * k * 4 + 4 * F * 4
        assert p["fin_smem"] == need and need <= SMEM_MAX, p
        assert (p["fin_stages"] * p["fin_stage_bytes"]) % 16 == 0  # g by row starts 16-byte aligned
        # compute threads: two token octets x 64 column quads cover 16 tokens x one 256-column pass
        assert p["fin_threads"] == 2 * 64 and F == 2 * 8 and p["fin_cols"] == 64 * 4


def test_norms_pass_plan(plans):
    for p in plans:
        k, d = p["k"], p["d"]
        # four columns a thread: k a multiple of 4; x in 16-byte vectors: d a multiple of 8
        assert k % 4 == 0 and d % 8 == 0
        # g by chunk: [chunk][column][slot]; the last token's last column stays inside the region
        T, F = p["T"], p["fin_tok"]
        last = ((T - 1) // F) * k * F + (k - 1) * F + (T - 1) % F
        assert last < cdiv(T, F) * F * k
