"""The GEMM's launch plan on the host, without a GPU: how many CTA pairs launch,
and when the nearly empty last round of tiles is divided along K (the split
tail). The rule: split when a workspace of the full size is given, the tiles do
not fit one round, the leftover round is at most a quarter full, and each tile has
at least 32 K-steps of 128 (K >= 4096); the first pairs + leftover tiles are then
divided. The workspace holds 10240 bytes of arrival counters plus two 256 KB
partial-sum slots per pair, for at most 80 pairs."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "microscaled_precision_gemm_gb300", "csrc")
COUNTERS = 10240
SLOT = 2 * 128 * 256 * 4


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    cxx = shutil.which("g++")
    cuda_inc = "/usr/local/cuda/include"
    if cxx is None or not os.path.isdir(cuda_inc):
        pytest.skip("g++ or the CUDA headers are not available")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_probe")
    subprocess.run([cxx, "-std=c++17", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
                    "-I", cuda_inc, os.path.join(ROOT, "tests", "helpers", "plan_probe.cpp"), "-o", exe], check=True)

    def run(m, n, k, clusters=76, ws=None, halves=False, lead=False):
        full = COUNTERS + 2 * min(80, max(1, ((m + 255) // 256) * (n // 256) - 1)) * SLOT
        ws_bytes = full if ws is None else ws
        out = subprocess.run([exe], input=f"{m} {n} {k} {clusters} {ws_bytes} {int(halves)}\n", capture_output=True,
                             text=True, check=True).stdout.split()
        vals = tuple(int(v) for v in out)
        if lead:
            return vals[5]
        return vals[:5] if halves else vals[:4]

    return run


def test_dit_down_projection_splits_its_leftover_round(plan):
    # 64 x 12 = 768 pair tiles on 76 pairs: 10 rounds + 8; K = 12288 is 96 K-steps
    assert plan(16384, 3072, 12288) == (768, 76, 76 + 8, COUNTERS + 2 * 80 * SLOT)


def test_full_leftover_rounds_stay_whole(plan):
    assert plan(20480, 12288, 3072)[:3] == (3840, 76, 0)    # 40 left over > 76 / 4
    assert plan(20480, 3072, 12288)[:3] == (960, 76, 0)     # 48 left over


def test_short_tiles_never_split(plan):
    # M = 4096 up-projection: 768 tiles, 8 left over, but 24 K-steps per tile
    tiles, pairs, split, ws = plan(4096, 12288, 3072)
    assert (tiles, pairs, split, ws) == (768, 76, 0, 0)
    assert plan(16384, 3072, 3968)[2] == 0                  # 31 K-steps
    assert plan(16384, 3072, 4096)[2] == 76 + 8             # 32 K-steps


def test_workspace_decides(plan):
    assert plan(16384, 3072, 12288, ws=-1)[2] == 0                            # none given
    assert plan(16384, 3072, 12288, ws=COUNTERS + 2 * 76 * SLOT - 1)[2] == 0  # one byte short
    assert plan(16384, 3072, 12288, ws=COUNTERS + 2 * 76 * SLOT)[2] == 84     # enough for 76 pairs


def test_pairs_never_exceed_tiles_or_residency(plan):
    assert plan(256, 256, 8192)[:3] == (1, 1, 0)
    assert plan(300, 512, 8192)[:3] == (4, 4, 0)            # ragged M: 2 row tiles x 2
    assert plan(20480, 3072, 12288, clusters=10)[:2] == (960, 10)
    # leftover 0 (tiles a multiple of the pairs): nothing to split
    assert plan(256 * 76, 256, 8192)[:3] == (76, 76, 0)
    assert plan(256 * 152, 256, 8192)[:3] == (152, 76, 0)
    # leftover 1 of 76: split the first 77 tiles
    assert plan(256 * 153, 256, 8192)[:3] == (153, 76, 77)


def test_workspace_bytes_query(plan):
    assert plan(16384, 3072, 3072)[3] == 0                  # K < 4096
    assert plan(256, 256, 8192)[3] == 0                     # one tile
    assert plan(512, 256, 8192)[3] == COUNTERS + 2 * 1 * SLOT
    assert plan(20480, 3072, 12288)[3] == COUNTERS + 2 * 80 * SLOT


def test_half_tiles(plan):
    """Without a split, the last round's tiles run as halves when at most pairs / 2
    are left over, and a GEMM of at most pairs / 2 tiles runs all of them as halves
    on twice as many pairs; never where the split tail is taken, nor when the
    epilogue cannot (halves_ok false). Output: tiles, pairs, split, ws, half tiles."""
    # M = 4096 up-projection: 768 tiles = 10 rounds + 8 (K = 3072: no split)
    assert plan(4096, 12288, 3072, halves=True)[:3] + plan(4096, 12288, 3072, halves=True)[4:] == (768, 76, 0, 8)
    assert plan(4096, 12288, 3072, halves=False)[:3] == (768, 76, 0)
    # 38 left over of 76: halves; 39: not
    assert plan(256 * 114, 256, 3072, halves=True)[4] == 38
    assert plan(256 * 115, 256, 3072, halves=True)[4] == 0
    # a round's worth exactly: nothing left over
    assert plan(256 * 152, 256, 3072, halves=True)[4] == 0
    # few tiles: all halves on twice the pairs (PR1: 1 x 2 tiles)
    assert plan(128, 512, 256, halves=True) == (2, 4, 0, 0, 2)
    assert plan(256 * 38, 256, 3072, halves=True)[1:] == (76, 0, 0, 38)
    assert plan(256 * 39, 256, 3072, halves=True)[1:] == (39, 0, 0, 0)
    # the split tail wins where it applies (DiT down-projection)
    assert plan(16384, 3072, 12288, halves=True)[2:] == (84, COUNTERS + 2 * 80 * SLOT, 0)


def test_leading_rows_cover_row_block_zero(plan):
    """The GEMM that quantizes its own activations leaves the rows of its first round
    of tiles to the quantize kernel; when it encodes any rows itself (leading rows <
    M) they are a whole number of 256-row pair tiles, at least one, so 128-row block
    0 always lies in the leading rows. Its counter word is then free, and the
    quantizer warps use it as their work counter."""
    # the full block's up-projection: 48 column tiles, 76 pairs -> row tiles 0 and 1
    assert plan(20480, 12288, 3072, lead=True) == 512
    assert plan(4096, 12288, 3072, lead=True) == 512
    # 16384 wide (the SwiGLU gate/up GEMM): 64 column tiles -> row tiles 0 and 1
    assert plan(20480, 16384, 3072, lead=True) == 512
    # narrower than 12288: every row up front
    assert plan(20480, 3072, 3072, lead=True) == 20480
    assert plan(20480, 8192, 3072, lead=True) == 20480
    # few pairs, ragged M, M inside the first round
    for m, n, clusters in [(20480, 12288, 1), (20480, 12288, 10), (1300, 12288, 76), (300, 12288, 76),
                           (257, 12288, 2), (100000, 65536, 76), (5000, 24576, 30)]:
        lead_rows = plan(m, n, 3072, clusters=clusters, lead=True)
        assert lead_rows == m or (lead_rows % 256 == 0 and 256 <= lead_rows < m), (m, n, clusters, lead_rows)
