"""Every fp16 kernel configuration against the oracle.

The dispatcher picks one tile width (64/128/192/256 columns); for 128 and 256,
pairs of blocks running 2-SM MMAs across the pair; and a schedule: whole tiles,
or the K steps of a last, part-filled round of tiles shared out over the
persistent grid (stream-K, shared tiles finished by their last contributor).
Each configuration is forced here in its own process (the switches are read
once per process from GEMM_GB300_HG_PAIR, GEMM_GB300_HG_BN and
GEMM_GB300_HG_SK; SK=2 and SK=3 share every tile, so every tile goes through
the partial-sum path, finished inside the kernel (2) or by the reduction
kernel (3)) and checked on ragged, multi-tile problems in all four variants,
exact on small-integer inputs.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from dense_gemm_tiled_gb300 import inputs
from helpers import check_problem
for v in ("nn", "tn", "nt", "tt"):
    tA, tB = inputs.VARIANTS[v]
    # 3 tile rows (odd: the last pair has a block past M), ragged N and K
    p = inputs.make_problem(384, 640, 448, tA, tB, "f16", "integer", seed=600)
    check_problem(p, exact=True)
    p = inputs.make_problem(300, 520, 264, tA, tB, "f16", "uniform", seed=601, beta=0.5)
    check_problem(p)
    # odd N: C rows off 16-byte alignment
    p = inputs.make_problem(300, 523, 264, tA, tB, "f16", "uniform", seed=604, beta=0.5)
    check_problem(p)
    p = inputs.make_problem(1024, 768, 1000, tA, tB, "f16", "uniform", seed=602)
    check_problem(p)
    # 2048 x 3072 with 256-wide tiles: 96 pair units (192 single tiles) over
    # 76 pairs (152 blocks) leaves a last round part-filled, whose K steps
    # stream-K shares out
    p = inputs.make_problem(2048, 3072, 512, tA, tB, "f16", "uniform", seed=603, beta=0.5)
    check_problem(p)
    # few tiles, long K: shared tiles with many contributors each
    p = inputs.make_problem(260, 96, 3000, tA, tB, "f16", "integer", seed=605)
    check_problem(p, exact=True)
    p = inputs.make_problem(130, 200, 2056, tA, tB, "f16", "uniform", seed=606, beta=0.5)
    check_problem(p)
print("ok")
"""


@pytest.mark.parametrize("pair,bn,sk", [("2", "256", "1"), ("2", "256", "2"), ("2", "256", "3"),
                                        ("2", "256", "0"), ("2", "128", "1"), ("2", "128", "2"),
                                        ("2", "128", "3"), ("0", "256", "2"), ("0", "256", "3"),
                                        ("0", "256", "0"), ("0", "128", "2"), ("0", "192", "2"),
                                        ("0", "64", "2"), ("0", "64", "3"), ("0", "64", "1")])
def test_forced_kernel_configuration(lib_path, gpu, pair, bn, sk):
    env = dict(os.environ, GEMM_GB300_HG_PAIR=pair, GEMM_GB300_HG_BN=bn, GEMM_GB300_HG_SK=sk)
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-3000:] + r.stderr[-3000:]


SCRIPT_F32 = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from dense_gemm_tiled_gb300 import binding, inputs
from helpers import check_problem
# (the 128 x 128 tile's counts; the 128 x 256 tile splits the first three
# shapes over K instead)
want = ("ffma",) if {tile!r} == "0" else ("ffma", "ffma_splitk")
for v in ("nn", "tn", "nt", "tt"):
    tA, tB = inputs.VARIANTS[v]
    # above the packing threshold (M*N*K >= 2^30) with more output tiles
    # than the split-K rule splits (> 152), ragged in every dimension
    p = inputs.make_problem(1000, 2600, 620, tA, tB, "f32", "uniform", seed=610, beta=0.5)
    r = check_problem(p)
    assert r["path"] in want, r
    p = inputs.make_problem(2048, 1408, 384, tA, tB, "f32", "integer", seed=611)
    r = check_problem(p, exact=True)
    assert r["path"] in want, r
    # odd leading dimensions everywhere (rows off 16-byte alignment)
    p = inputs.make_problem(1001, 2601, 621, tA, tB, "f32", "uniform", seed=612, beta=0.5)
    r = check_problem(p)
    assert r["path"] in want, r
    # 176 tiles of 128 x 256 (stream-K for that tile too), integer: exact
    p = inputs.make_problem(2048, 2600, 400, tA, tB, "f32", "integer", seed=613, beta=1.0,
                            c_fill="integer")
    r = check_problem(p, exact=True)
    assert r["path"] == "ffma", r
    # fewer tiles than SMs on a large problem (64 of 128 x 128, 32 of
    # 128 x 256, 128 of 128 x 64): every tile's K steps shared over all blocks
    # in one launch, up to 5 contributors a tile; otherwise split K; exact
    p = inputs.make_problem(1000, 1000, 1100, tA, tB, "f32", "integer", seed=614, beta=1.0,
                            c_fill="integer")
    r = check_problem(p, exact=True)
    assert r["path"] == ("ffma" if {all_shared} else "ffma_splitk"), r
print("ok")
"""


@pytest.mark.parametrize("pack,sk,tile,ws", [("1", "1", "0", "1"), ("0", "1", "0", "1"),
                                             ("1", "0", "0", "1"), ("1", "1", "0", "0"),
                                             ("1", "0", "0", "0"), ("1", "1", "2", "1"),
                                             ("0", "1", "2", "1"), ("1", "0", "2", "1"),
                                             ("1", "1", "3", "1"), ("0", "1", "3", "1"),
                                             ("1", "1", "3", "0")])
def test_forced_fp32_configuration(lib_path, gpu, pack, sk, tile, ws):
    """The fp32 transposing pre-pass (default on large problems) or the kernel
    reading every layout directly (GEMM_GB300_SG_PACK=0); the persistent
    stream-K launch (default when the tiles are not a whole number of rounds
    of the SMs; the shapes here have 168 and 176 tiles of 128 x 128, 84 and 88
    of 128 x 256, 336 and 352 of 128 x 64 against 304 resident blocks) or one
    block per tile (GEMM_GB300_SG_SK=0); the 128 x 128 tile, the 128 x 256
    one (lanes of 8 x 16 outputs) or the 128 x 64 one (GEMM_GB300_SG_TILE 0,
    2, 3); operands stored k-major (packed, or tn as given) staged by the
    warp-specialised TMA kernel (default for the 128 x 128 and 128 x 64
    tiles) or by every warp's cp.async copies (GEMM_GB300_SG_WS=0)."""
    env = dict(os.environ, GEMM_GB300_SG_PACK=pack, GEMM_GB300_SG_SK=sk, GEMM_GB300_SG_TILE=tile,
               GEMM_GB300_SG_WS=ws)
    all_shared = pack == "1" and sk == "1" and ws == "1"
    code = SCRIPT_F32.format(root=ROOT, tests=os.path.join(ROOT, "tests"), tile=tile,
                             all_shared=all_shared)
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-3000:] + r.stderr[-3000:]


SCRIPT_NARROW = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from dense_gemm_tiled_gb300 import binding, inputs
from helpers import check_problem
for v in ("nn", "tn", "nt", "tt"):
    tA, tB = inputs.VARIANTS[v]
    # rank-32 output with a long K (split over K), a ragged N below 32 with
    # beta, every dimension ragged, and odd leading dimensions on a problem
    # large enough for the pre-pass copies
    p = inputs.make_problem(4096, 32, 2048, tA, tB, "f32", "uniform", seed=620)
    check_problem(p)
    p = inputs.make_problem(300, 17, 5000, tA, tB, "f32", "uniform", seed=621, beta=0.5)
    check_problem(p)
    p = inputs.make_problem(777, 31, 333, tA, tB, "f32", "integer", seed=622, beta=1.0,
                            c_fill="integer")
    check_problem(p, exact=True)
    p = inputs.make_problem(8191, 29, 4601, tA, tB, "f32", "uniform", seed=623)
    check_problem(p)
    # aligned rows, N = 32 and N = 24 (B tile past N), split over K and
    # not, integer inputs: exact
    p = inputs.make_problem(2304, 32, 1024, tA, tB, "f32", "integer", seed=624, beta=1.0,
                            c_fill="integer")
    check_problem(p, exact=True)
    p = inputs.make_problem(40000, 24, 256, tA, tB, "f32", "integer", seed=625)
    check_problem(p, exact=True)
print("ok")
"""


@pytest.mark.parametrize("narrow,ws", [("1", "1"), ("1", "0"), ("0", "1")])
def test_fp32_narrow_tile(lib_path, gpu, narrow, ws):
    """N <= 32 on the fp32 path: the 256 x 32 tile (default) or the general
    128 x 128 tile (GEMM_GB300_SG_NARROW=0), split over K or not; with
    aligned rows and B stored [K, N], the narrow tile's operands arrive by TMA
    (A row tiles 128-byte swizzled when A is stored [M, K]), else
    (GEMM_GB300_SG_WS=0, or unaligned rows) by every warp's cp.async copies."""
    env = dict(os.environ, GEMM_GB300_SG_NARROW=narrow, GEMM_GB300_SG_WS=ws)
    code = SCRIPT_NARROW.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-3000:] + r.stderr[-3000:]


SCRIPT_LAUNCHES = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
from dense_gemm_tiled_gb300 import binding, inputs
from helpers import check_problem
# a LoRA adapter product (rank-32 output, K = 2048): 4 tiles shared by 16 ranges
p = inputs.make_problem(512, 32, 2048, False, True, "f16", "uniform", seed=242)
r = check_problem(p)
print(r["path"], binding.last_launches())
"""


@pytest.mark.parametrize("sk,launches", [("2", 1), ("3", 2)])
def test_shared_tile_finishing_launches(lib_path, gpu, sk, launches):
    """Shared tiles finished inside the GEMM kernel by each tile's last
    contributor take one launch (GEMM_GB300_HG_SK=2); finished by the
    reduction kernel over every contributor's published sums, two
    (GEMM_GB300_HG_SK=3)."""
    env = dict(os.environ, GEMM_GB300_HG_SK=sk)
    code = SCRIPT_LAUNCHES.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert r.stdout.split()[-2:] == ["tc_splitk", str(launches)], r.stdout
