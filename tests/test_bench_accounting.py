"""Host-side flop accounting of bench.py (no GPU): the issued-flop count
follows the kernels' tile enumeration."""
import bench


def test_issued_equals_algorithmic_on_exact_pair_tiles_for_update():
    # 512 x 1024: two 256-row pair rows, four 256-column tiles, K = 512
    got = bench.ns_stage_issued_flops(512, 1024)
    assert got["ns_update"] == 2 * 512 * 1024 * 512 == bench.ns_stage_flops(512, 1024)["ns_update"]


def test_pair_triangle_counts_whole_diagonal_tiles():
    # T = 2 pair rows -> tiles (0,0), (0,1), (1,1), each 256 x 256
    got = bench.ns_stage_issued_flops(512, 1024)
    assert got["ns_syrk"] == 2 * 3 * 256 * 256 * 1024
    assert got["ns_poly"] == 2 * 3 * 256 * 256 * 512


def test_single_cta_triangle_skips_left_half_of_odd_diagonal_tiles():
    # m' = 300: 44 rows past 256 waste > 1/8 -> single CTAs, 128 x 256 tiles.
    # Row tiles 0..2, column tiles 0..1 (second one 44 wide -> 48 issued).
    # ti=0: tj 0,1 -> 256 + 48; ti=1: tj 0 (right half 128) + tj 1 (48);
    # ti=2: tj 1 (48).
    cols = (256 + 48) + (128 + 48) + 48
    got = bench.ns_stage_issued_flops(300, 1000)
    assert got["ns_poly"] == 2 * 128 * cols * 320  # K = 300 rounded up to 320
    assert got["ns_syrk"] == 2 * 128 * cols * 1024


def test_issued_never_below_algorithmic():
    for mp, np_ in [(1, 1), (7, 13), (64, 64), (256, 512), (1408, 2048), (2048, 5632), (7168, 18432)]:
        iss = bench.ns_stage_issued_flops(mp, np_)
        alg = bench.ns_stage_flops(mp, np_)
        for k in alg:
            assert iss[k] >= alg[k], (mp, np_, k)
