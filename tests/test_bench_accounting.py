"""Host-side flop accounting of bench.py (no GPU): the issued-flop count
follows the kernels' tile enumeration."""
import bench


def test_issued_equals_algorithmic_on_exact_pair_tiles_for_update():
    # 1024 x 2048: four 256-row pair rows, eight 256-column tiles, K = 1024
    got = bench.ns_stage_issued_flops(1024, 2048)
    assert got["ns_update"] == 2 * 1024 * 2048 * 1024 == bench.ns_stage_flops(1024, 2048)["ns_update"]


def test_pair_triangle_counts_whole_diagonal_tiles():
    # 1024 rows: 4 pair rows -> tiles (I, J >= I), 10 of 256 x 256
    got = bench.ns_stage_issued_flops(1024, 2048)
    assert got["ns_syrk"] == 2 * 10 * 256 * 256 * 2048
    assert got["ns_poly"] == 2 * 10 * 256 * 256 * 1024


def test_up_to_512_rows_run_on_single_ctas():
    # 512 rows, no pair padding, but single CTAs: 4 row tiles of 128 over
    # 2 column tiles of 256, odd diagonal tiles issuing only their right half:
    # ti=0: 256 + 256; ti=1: 128 + 256; ti=2: 256; ti=3: 128
    got = bench.ns_stage_issued_flops(512, 1024)
    assert got["ns_syrk"] == 2 * 128 * (512 + 384 + 256 + 128) * 1024
    assert got["ns_poly"] == 2 * 128 * (512 + 384 + 256 + 128) * 512
    assert got["ns_update"] == 2 * 512 * 1024 * 512


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


def test_e2e_pieces_cover_every_element_once():
    """The end-to-end run's pieces: runs of consecutive matrices whose
    W, G, M fit a staging slot (one matrix per piece at least), then AdamW
    chunks that tile each buffer exactly, every chunk starting 16-byte
    aligned so the vector path stays on."""
    from types import SimpleNamespace
    import torch
    import workloads

    w = workloads.get("c3")
    w.matrices = w.matrices[:40]                    # 4 attention + 36 expert matrices
    n = sum(s.rows * s.cols for s in w.matrices)
    storage = (torch.empty(n), torch.empty(n), torch.empty(n))
    adamw = [SimpleNamespace(p=torch.empty(k), g=torch.empty(k), m=torch.empty(k), v=torch.empty(k))
             for k in (1000, 37)]
    ws = SimpleNamespace(w=w, tens=SimpleNamespace(storage=storage), adamw=adamw)
    slot = 200 << 20
    pieces = bench.e2e_pieces(ws, slot)
    muon = [p for p in pieces if p[0] == "muon"]
    ranges = [p[3] for p in muon]
    assert ranges[0][0] == 0 and ranges[-1][1] == len(w.matrices)
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    for kind, ins, outs, (a, b) in muon:
        nbytes = sum(t.numel() * t.element_size() for t in ins)
        assert b - a == 1 or nbytes <= slot
        assert len(ins) == 3 and len(outs) == 2 and outs[0].data_ptr() == ins[0].data_ptr()
    small = bench.e2e_pieces(ws, 64)                 # a slot smaller than any piece: one unit each
    assert len([p for p in small if p[0] == "muon"]) == len(w.matrices)
    for buf, want in zip(adamw, (1000, 37)):
        chunks = [p[3] for p in small if p[0] == "adamw" and p[3][0].untyped_storage().data_ptr()
                  == buf.p.untyped_storage().data_ptr()]
        assert sum(q[0].numel() for q in chunks) == want
        assert all(q[0].storage_offset() % 4 == 0 for q in chunks)
