"""Host-side tests of the C ABI (no GPU): the library loads and exports every
symbol include/w8.h declares; w8_validate refuses the planes the PR page's
bind step turns away (Changes: any FP8 format other than E4M3fn, a plane
without padding, a bias term, a build that mixes bf16 and FP8 planes;
Limitations: e4m3fnuz and the remaining formats); the
packed address map is a bijection that keeps each lane's 16-byte vector
inside one (row tile, K block); the launch planner covers K exactly and does
not depend on the weight dtype.  No compute call is made here.
"""
from __future__ import annotations

import os
import re
import subprocess
import sys

import pytest

from fp8_weight_only_w8a16_gb300 import w8

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w8.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\([^;{]*\)\s*;", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


def test_every_declared_function_is_exported():
    declared = _declared_functions()
    assert "w8_gemv" in declared and "bf16_gemv" in declared and "w8_bind" in declared
    assert sorted(w8.EXPORTS) == declared
    for name in declared:
        assert hasattr(w8.lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", w8.LIB_PATH], capture_output=True,
                        text=True)
    if nm.returncode == 0:
        exported = set(line.split()[-1] for line in nm.stdout.splitlines() if line.strip())
        assert set(declared) <= exported


def test_abi_version_and_status_strings():
    assert w8.lib.w8_abi_version() == 8
    for code in range(15):
        assert w8.status_str(code)
    assert w8.status_str(99) == "unknown status"


FAKE = 0x10000  # a 16-byte aligned address; validate never dereferences it


def _desc(**kw):
    d = dict(w=FAKE, dtype=w8.DT_E4M3FN, layout=0, n=64, k=128, ldw=128, scale=FAKE + 4096,
             bias=None, block_scale=None, ldb=0)
    d.update(kw)
    return w8.PlaneDesc(d["w"], d["dtype"], d["layout"], d["n"], d["k"], d["ldw"], d["scale"],
                        d["bias"], d["block_scale"], d["ldb"])


MX = dict(dtype=w8.DT_MXFP4, scale=None, block_scale=FAKE + 8192, ldb=4)
B128 = dict(dtype=w8.DT_E4M3FN_B128, ldb=1)


def _status(*descs):
    arr = (w8.PlaneDesc * len(descs))(*descs)
    return w8.lib.w8_validate(arr, len(descs))


@pytest.mark.parametrize("kw,want", [
    ({}, "W8_OK"),
    ({"dtype": w8.DT_BF16, "scale": None, "ldw": 128}, "W8_OK"),
    ({"w": None}, "W8_ERR_NULL"),
    ({"dtype": w8.DT_E4M3FNUZ}, "W8_ERR_DTYPE"),
    ({"dtype": w8.DT_E5M2}, "W8_ERR_DTYPE"),
    ({"dtype": w8.DT_FP16}, "W8_ERR_DTYPE"),
    ({"dtype": 99}, "W8_ERR_DTYPE"),
    ({"layout": 2}, "W8_ERR_LAYOUT"),
    ({"layout": -1}, "W8_ERR_LAYOUT"),
    ({"layout": w8.SRC_GATE_UP}, "W8_OK"),                 # n = 64: I = 32
    ({"layout": w8.SRC_GATE_UP, "n": 48}, "W8_OK"),        # I = 24
    ({"layout": w8.SRC_GATE_UP, "n": 40}, "W8_ERR_SHAPE"),  # I = 20: not a multiple of 8
    ({"layout": w8.SRC_GATE_UP, "n": 8}, "W8_ERR_SHAPE"),
    ({"layout": w8.SRC_GATE_UP, "n": 7}, "W8_ERR_SHAPE"),
    ({"bias": FAKE}, "W8_ERR_BIAS"),
    ({"n": 0}, "W8_ERR_SHAPE"),
    ({"k": 0}, "W8_ERR_SHAPE"),
    ({"ldw": 64}, "W8_ERR_SHAPE"),
    ({"n": 1 << 31}, "W8_ERR_SHAPE"),
    ({"scale": None}, "W8_ERR_SCALE"),
    ({"dtype": w8.DT_BF16}, "W8_ERR_SCALE"),
    ({"w": FAKE + 8}, "W8_ERR_UNPADDED"),
    ({"ldw": 136}, "W8_ERR_UNPADDED"),
    ({"k": 130, "ldw": 130}, "W8_ERR_UNPADDED"),
    ({"k": 130, "ldw": 144}, "W8_OK"),
    ({"dtype": w8.DT_BF16, "scale": None, "ldw": 132}, "W8_ERR_UNPADDED"),
    ({"dtype": w8.DT_BF16, "scale": None, "ldw": 136}, "W8_OK"),
    # MXFP4: E8M0 block scales instead of row scales; rows of a multiple of 16 bytes
    (dict(MX), "W8_OK"),
    (dict(MX, k=100, ldw=128), "W8_OK"),
    (dict(MX, block_scale=None), "W8_ERR_SCALE"),
    (dict(MX, scale=FAKE + 4096), "W8_ERR_SCALE"),
    (dict(MX, ldb=3), "W8_ERR_SCALE"),           # 128 columns need 4 blocks
    (dict(MX, ldw=144), "W8_ERR_UNPADDED"),      # 72 bytes a row
    (dict(MX, ldw=129, k=100), "W8_ERR_UNPADDED"),
    (dict(MX, ldw=160), "W8_OK"),                # 80 bytes a row
    ({"block_scale": FAKE + 8192, "ldb": 4}, "W8_ERR_SCALE"),  # FP8 plane with block scales
    # block-scaled FP8: fp32 factors [ceil(n/128)][ldb] in scale, ldb >= ceil(k/128)
    (dict(B128), "W8_OK"),
    (dict(B128, k=300, ldw=304, ldb=3), "W8_OK"),
    (dict(B128, k=300, ldw=304, ldb=2), "W8_ERR_SCALE"),
    (dict(B128, ldb=0), "W8_ERR_SCALE"),
    (dict(B128, scale=None), "W8_ERR_SCALE"),
    (dict(B128, block_scale=FAKE + 8192), "W8_ERR_SCALE"),
    (dict(B128, layout=w8.SRC_GATE_UP), "W8_ERR_LAYOUT"),
    (dict(B128, ldw=136), "W8_ERR_UNPADDED"),
])
def test_validate_refusal_matrix(kw, want):
    assert w8.STATUS[_status(_desc(**kw))] == want


def test_mixed_build_refused_and_empty_list():
    bf = _desc(dtype=w8.DT_BF16, scale=None)
    assert w8.STATUS[_status(_desc(), bf)] == "W8_ERR_MIXED"
    assert w8.STATUS[_status(bf, _desc())] == "W8_ERR_MIXED"
    assert w8.STATUS[_status(_desc(), _desc(n=7, k=33, ldw=48))] == "W8_OK"
    assert w8.STATUS[w8.lib.w8_validate(None, 0)] == "W8_ERR_NULL"
    # row-scaled and block-scaled FP8 are different dtypes too
    assert w8.STATUS[_status(_desc(), _desc(**B128))] == "W8_ERR_MIXED"
    # a bad plane anywhere in the list is reported before the mix check
    assert w8.STATUS[_status(_desc(), _desc(bias=FAKE))] == "W8_ERR_BIAS"


def test_packed_bytes_mxfp4():
    # [100, 200]: 7 tiles x 7 blocks x 288 B (codes and the rows' bf16 block scales)
    assert w8.packed_bytes([_desc(n=100, k=200, ldw=224, **{k: v for k, v in MX.items()
                                                          if k != "ldb"}, ldb=7)]) == \
        -(-7 * 7 * 288 // 256) * 256


def test_mxfp4_bit_map_is_a_bijection_onto_the_code_bits():
    rt, kb = 3, 4
    bits = [b for r in range(rt * 16) for c in range(kb * 32)
            for b in w8.mxfp4_code_bits(kb, r, c)]
    # every code bit of every 288-byte run exactly once; its last 256 bits
    # hold the block scales
    assert sorted(bits) == [run * 2304 + b for run in range(rt * kb) for b in range(2048)]
    assert w8.packed_offset(w8.DT_MXFP4, kb, 0, 0) == -1
    for r in (0, 5, 8, 13):
        for c in (0, 7, 8, 31):
            m, e0, e1, sg = w8.mxfp4_code_bits(1, r, c)
            # lane (g, t) owns bytes 8 (4g + t) .. + 7 of the run
            assert all(b // 64 == 4 * (r % 8) + c // 8 for b in (m, e0, e1, sg))
            # one shift carries the magnitude to bf16 bits 6..8 and the sign to
            # 15 (low element) or 22..24 and 31 (high element) of its word:
            # consecutive magnitude bits except in the spare register (13)
            assert e0 == m + 1 and (e1 == m + 2 or e1 == m + 3)
    with pytest.raises(w8.W8Error):
        w8.mxfp4_code_bits(1, 0, 32)


def test_packed_bytes_block_scaled():
    # [300, 500]: 19 tiles x 16 blocks x 512 B, row copy 19*16*4 B, factors 3 x 4 x 4 B
    d = _desc(n=300, k=500, ldw=512, **B128)
    d.ldb = 4
    want = 19 * 16 * 512 + (-(-19 * 16 * 4 // 256)) * 256 + 256
    assert w8.packed_bytes([d]) == want


def test_packed_bytes_formula():
    # FP8 [100, 200]: 7 tiles x 7 blocks x 512 B, scales 7*16*4 B (each 256-aligned)
    assert w8.packed_bytes([_desc(n=100, k=200, ldw=208)]) == 25088 + 512
    # bf16 [16, 32]: one run of 1024 B
    assert w8.packed_bytes([_desc(dtype=w8.DT_BF16, scale=None, n=16, k=32, ldw=32)]) == 1024
    two = w8.packed_bytes([_desc(n=100, k=200, ldw=208), _desc(n=16, k=32, ldw=32)])
    assert two == 25088 + 512 + 512 + 256


@pytest.mark.parametrize("n", [16, 48, 64, 4096])
def test_gate_up_packed_row_interleaves_gate_and_up(n):
    half = n // 2
    rows = [w8.gate_up_packed_row(n, r) for r in range(n)]
    assert sorted(rows) == list(range(n))  # a permutation of the packed rows
    for j in range(half):
        g, u = rows[j], rows[half + j]
        # gate row j and up row j share a 16-row tile, eight rows apart
        assert g // 16 == u // 16 == j // 8
        assert g % 16 == j % 8 and u == g + 8
    for bad in (-1, n):
        assert w8.gate_up_packed_row(n, bad) == -1
    for bad_n in (0, 8, 24, -16):
        assert w8.gate_up_packed_row(bad_n, 0) == -1


@pytest.mark.parametrize("dtype,elt", [(w8.DT_E4M3FN, 1), (w8.DT_E4M3FN_B128, 1),
                                       (w8.DT_BF16, 2)])
def test_packed_offset_is_a_bijection(dtype, elt):
    rt, kb = 3, 4
    offs = [w8.packed_offset(dtype, kb, r, c) for r in range(rt * 16) for c in range(kb * 32)]
    assert all(o % elt == 0 for o in offs)
    assert sorted(o // elt for o in offs) == list(range(rt * 16 * kb * 32))


@pytest.mark.parametrize("dtype,run", [(w8.DT_E4M3FN, 512), (w8.DT_BF16, 1024)])
def test_packed_offset_lane_vectors(dtype, run):
    """Each 16-byte vector holds rows g and g+8 of one tile and columns 8t..8t+7
    of one block, with lane = 4g + t; runs are tile-major then block."""
    kb = 5
    for r in range(32):
        for c in range(kb * 32):
            o = w8.packed_offset(dtype, kb, r, c)
            tile, blk = r // 16, c // 32
            assert o // run == tile * kb + blk
            lane = (o % 512) // 16
            assert lane == 4 * (r % 8) + (c % 32) // 8
    # the 8 columns of one lane split 4 + 4 between the two tensor-core steps
    for c in range(32):
        o = w8.packed_offset(dtype, 1, 0, c)
        step = (o % 16) // 8 if dtype == w8.DT_E4M3FN else (o // 512)
        assert step == (c % 8) // 4


def test_packed_offset_rejects_bad_arguments():
    assert w8.packed_offset(w8.DT_E4M3FN, 0, 0, 0) == -1
    assert w8.packed_offset(w8.DT_E4M3FN, 2, 0, 64) == -1
    assert w8.packed_offset(w8.DT_E5M2, 2, 0, 0) == -1
    assert w8.packed_offset(w8.DT_BF16, 2, -1, 0) == -1


SHAPES = [(256, 512), (2624, 6144), (6144, 16384), (4096, 6144), (6144, 2048),
          (16384, 2048), (28672, 512), (4096, 2048), (128, 6144), (32, 6144),
          (154880, 6144), (1, 1), (37, 77), (100, 4096), (8192, 4096), (6144, 8192)]


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("m", [1, 2, 4, 8, 9, 16, 17, 32, 33, 64, 65, 96, 97, 128, 200, 256])
def test_plan_invariants(n, k, m):
    p = w8.plan_shape(n, k, m, 152)
    kb = -(-k // 32)
    rt = -(-n // 16)
    assert p.grid == p.row_groups * p.splits
    assert p.kernel == (1 if m > 64 or (m >= 17 and -(-n // 128) >= 48) else 0)
    if p.kernel == 1:
        # the tensor-memory kernel: 128 rows x one K range per CTA, tokens
        # padded to 16, about two CTAs per SM, at least one 4-block stage per split
        assert p.kernel == 1 and p.block == 352
        npad = -(-m // 16) * 16 if m <= 64 else min(x for x in (96, 128, 192, 256) if x >= m)
        occ = 2 if npad <= 64 else 1
        deep = npad == 64 and p.ctas_per_sm == 1
        if npad == 64:
            # one CTA per SM (a deeper ring) exactly where one wave of
            # unclustered CTAs covers 3/4 of the SMs or more
            rg = -(-n // 128)
            sg = min(8, 152 // rg)
            while sg > 1 and kb // sg < 32:
                sg -= 1
            cl = 1
            while cl < 8 and rg * cl * 2 <= 152 and kb // (cl * 2) >= 4:
                cl *= 2
            one_wave = rg * (sg if sg > cl else cl)
            assert deep == ((sg > cl or cl == 1) and 114 <= one_wave <= 152)
            if deep:
                occ = 1
        assert p.ctas_per_sm == occ
        assert p.row_groups == -(-n // 128) and p.n_tiles * 8 == npad
        assert p.splits == 1 or kb // p.splits >= 4
        assert p.grid <= 2 * 152 or p.splits == 1
        assert p.k_blocks_per_warp_max == -(-kb // p.splits)
        if p.cluster == 1 and p.splits > 1:
            # K ranges that meet in the workspace: as many as fill the
            # resident slots (at most 8), more than the power-of-two
            # cluster plan would take
            assert npad <= 64 and (2 < p.splits <= 8 or p.row_groups * 2 <= occ * 152 or deep)
            assert p.splits == min(8, occ * 152 // p.row_groups, kb // 32)
            assert p.grid <= occ * 152
            assert p.workspace_bytes >= p.splits * rt * 16 * m * 4
            return
        assert p.cluster == p.splits and p.splits in (1, 2, 4, 8)
        nw, nb = {16: (5, 6), 32: (4, 5), 48: (4, 3), 64: (3, 3), 96: (5, 5), 128: (5, 4),
                  192: (4, 3), 256: (4, 2)}[npad]  # FP8 stage slots
        if deep:
            nw, nb = 8, 4
        # about 100 KB (two CTAs per SM), about 200 KB (one), plus 1 KB to
        # start the stages on a 1024-byte boundary
        limit = 105 * 1024 if occ == 2 else 209 * 1024
        assert p.smem_bytes == nw * 8 * 4 * 512 + nb * 4 * npad * 64 + 1024 <= limit
        assert p.grid <= occ * 152 or p.splits == 1
        assert p.workspace_bytes == 0  # split partials meet on chip
        return
    assert p.cluster == 1
    assert p.block == 256
    assert p.warps_k in (1, 2, 4, 8) and p.depth >= 1
    assert 1 <= p.splits <= kb
    tiles_per_cta = (8 // p.warps_k) * p.row_tiles_per_warp
    assert p.row_groups * tiles_per_cta >= rt > (p.row_groups - 1) * tiles_per_cta
    assert p.n_tiles * 8 >= m and (p.n_tiles == 1 or p.n_tiles * 4 < m)
    assert p.smem_bytes == 8 * p.row_tiles_per_warp * p.n_tiles * 128 * 4 <= 64 * 1024
    assert (p.workspace_bytes == 0) == (p.splits == 1)
    if p.splits > 1:
        assert p.workspace_bytes >= p.splits * rt * 16 * m * 4
    # CTA splits and warp K parts tile the K blocks exactly (floor boundaries);
    # every warp gets at least one block unless K is shorter than the warps
    parts = []
    for s in range(p.splits):
        c0, c1 = (s * kb) // p.splits, ((s + 1) * kb) // p.splits
        for q in range(p.warps_k):
            parts.append((c0 + (q * (c1 - c0)) // p.warps_k,
                          c0 + ((q + 1) * (c1 - c0)) // p.warps_k))
    assert parts[0][0] == 0 and parts[-1][1] == kb
    assert all(a1 == b0 for (_, a1), (b0, _) in zip(parts, parts[1:]))
    assert max(b - a for a, b in parts) == p.k_blocks_per_warp_max
    if kb >= p.warps_k * p.splits:
        assert min(b - a for a, b in parts) >= 1


PLAN_FIELDS = ("kernel", "grid", "block", "smem_bytes", "n_tiles", "row_tiles_per_warp",
               "warps_k", "row_groups", "splits", "workspace_bytes", "cluster", "ctas_per_sm")


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("m", [1, 4, 8, 16, 17, 32, 64, 65, 200])
def test_plan_shape_dtype_row_and_bf16_planes_match_the_shape_plan(n, k, m):
    """E4M3FN and bf16 planes of one shape launch the same plan (the same
    summation order); only the ring depth differs."""
    base = w8.plan_shape(n, k, m, 152)
    for dt in (w8.DT_E4M3FN, w8.DT_BF16):
        p = w8.plan_shape_dtype(n, k, m, 152, dt)
        assert all(getattr(p, f) == getattr(base, f) for f in PLAN_FIELDS), dt
        assert p.k_blocks_per_warp_max == base.k_blocks_per_warp_max
    assert w8.plan_shape_dtype(n, k, m, 152, w8.DT_E4M3FN).depth == base.depth
    if base.kernel == 1 and base.ctas_per_sm == 1 and m <= 64:
        # the one-CTA-per-SM instance at 49..64 tokens: 8 FP8 or 4 bf16
        # weight stages of 4 K blocks
        assert base.depth == 32
        assert w8.plan_shape_dtype(n, k, m, 152, w8.DT_BF16).depth == 16


@pytest.mark.parametrize("n,k", SHAPES)
@pytest.mark.parametrize("m", [1, 2, 8, 9, 16, 17, 32, 33, 64])
def test_plan_shape_dtype_ring_only_planes(n, k, m):
    """MXFP4 and block-scaled planes run the register ring at every m; MXFP4
    takes the ring plan FP8 would take there, block-scaled planes a ring of
    whole column blocks, with K split among CTAs and warps in whole column
    blocks."""
    kb = -(-k // 32)
    mx = w8.plan_shape_dtype(n, k, m, 152, w8.DT_MXFP4)
    b1 = w8.plan_shape_dtype(n, k, m, 152, w8.DT_E4M3FN_B128)
    for p in (mx, b1):
        assert p.kernel == 0 and p.block == 256 and p.grid == p.row_groups * p.splits
        assert p.n_tiles * 8 >= m and p.depth >= 1
    fp8 = w8.plan_shape(n, k, m, 152)
    if fp8.kernel == 0:
        assert all(getattr(mx, f) == getattr(fp8, f) for f in PLAN_FIELDS)
    assert b1.depth % 4 == 0
    # the block-scaled K parts: units of 4 blocks, floor boundaries, the last cut at kb
    nu = -(-kb // 4)
    parts = []
    for s in range(b1.splits):
        c0, c1 = (s * nu) // b1.splits, ((s + 1) * nu) // b1.splits
        for q in range(b1.warps_k):
            a0 = 4 * (c0 + (q * (c1 - c0)) // b1.warps_k)
            a1 = min(4 * (c0 + ((q + 1) * (c1 - c0)) // b1.warps_k), kb)
            parts.append((min(a0, kb), max(a1, min(a0, kb))))
    assert parts[0][0] == 0 and parts[-1][1] == kb
    assert all(a1 == b0 for (_, a1), (b0, _) in zip(parts, parts[1:]))
    assert all(a0 % 4 == 0 for a0, a1 in parts if a1 > a0)
    assert max(b - a for a, b in parts) == b1.k_blocks_per_warp_max


def test_plan_shape_dtype_refusals():
    for dt in (w8.DT_MXFP4, w8.DT_E4M3FN_B128):
        with pytest.raises(w8.W8Error) as e:
            w8.plan_shape_dtype(2624, 6144, 65, 152, dt)
        assert e.value.name == "W8_ERR_SHAPE"
    for dt in (w8.DT_E4M3FNUZ, w8.DT_E5M2, w8.DT_FP16, 0, 99):
        with pytest.raises(w8.W8Error) as e:
            w8.plan_shape_dtype(2624, 6144, 1, 152, dt)
        assert e.value.name == "W8_ERR_DTYPE"
    with pytest.raises(w8.W8Error) as e:
        w8.plan_shape_dtype(2624, 6144, 0, 152, w8.DT_E4M3FN)
    assert e.value.name == "W8_ERR_SHAPE"


TC_SHAPES = [(256, 512), (2624, 6144), (6144, 16384), (6144, 2048), (16384, 2048), (28672, 512),
             (4096, 2048), (160, 6144), (6144, 8192), (8192, 4096), (20480, 2048), (37, 77)]


@pytest.mark.parametrize("sms", [1, 2, 8, 66, 132, 148, 160, 264])
def test_tensor_memory_plans_on_other_sm_counts(sms):
    """The tensor-memory plan's invariants hold whatever the SM count: the
    grid tiles row blocks x K ranges, the splits meet on chip (a cluster of
    at most 8) or in the workspace (cluster 1, workspace > 0), every K block
    is covered, the shared memory fits the CTAs per SM the plan is built
    for, and the one-CTA-per-SM instance at 49..64 tokens appears only where
    one wave of unclustered CTAs covers 3/4 of the SMs or more."""
    seen = 0
    for n, k in TC_SHAPES:
        kb = -(-k // 32)
        for m in (17, 33, 49, 64, 65, 128, 256):
            p = w8.plan_shape(n, k, m, sms)
            if p.kernel != 1:
                continue
            seen += 1
            assert p.grid == p.row_groups * p.splits and p.row_groups == -(-n // 128)
            assert p.ctas_per_sm in (1, 2) and 1 <= p.cluster <= 8
            assert p.cluster in (1, p.splits)
            assert p.k_blocks_per_warp_max * p.splits >= kb
            assert (p.workspace_bytes > 0) == (p.splits > 1 and p.cluster == 1)
            if m <= 64 and p.ctas_per_sm == 1:
                assert -(-m // 16) * 16 == 64 and p.cluster == 1
                assert p.grid <= sms and 4 * p.grid >= 3 * sms
            if m > 64:
                assert p.ctas_per_sm == 1 and p.workspace_bytes == 0
            # two CTAs of 352 threads share an SM's 228 KB, one may take 227 KB
            assert p.smem_bytes <= (113 if p.ctas_per_sm == 2 else 227) * 1024
    assert seen > 0


def test_plan_does_not_depend_on_anything_but_shape():
    a = w8.plan_shape(2624, 6144, 4, 152)
    b = w8.plan_shape(2624, 6144, 4, 152)
    assert bytes(a) == bytes(b)


def test_plan_refuses_bad_shapes():
    for args in [(0, 32, 1, 152), (16, 0, 1, 152), (16, 32, 0, 152), (16, 32, 257, 152),
                 (16, 32, 1, 0)]:
        with pytest.raises(w8.W8Error) as e:
            w8.plan_shape(*args)
        assert e.value.name == "W8_ERR_SHAPE"


def test_binding_fails_loudly_without_the_library(tmp_path):
    """With libw8.so absent the binding raises on import: no CPU fallback."""
    code = (
        "import sys; sys.path.insert(0, %r)\n"
        "from fp8_weight_only_w8a16_gb300 import build_lib\n"
        "build_lib.LIB = %r\n"
        "try:\n"
        "    import fp8_weight_only_w8a16_gb300.w8\n"
        "except ImportError as e:\n"
        "    print('raised', e)\n"
        "else:\n"
        "    print('imported')\n" % (ROOT, str(tmp_path / "missing" / "libw8.so")))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert "raised" in r.stdout and "no CPU fallback" in r.stdout, r.stdout + r.stderr


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "fp8_weight_only_w8a16_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cpp", ".cuh")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "w8_oracle" not in text and "liboracle" not in text, f
