"""Host-side paging recipes: the ring layout of window layers keeps every
retained position in its own live block, and the write of a new position
only ever lands on a block whose positions have all left the window."""
import pytest

from int4_quantized_paged_gb300 import workloads as wl


@pytest.mark.parametrize("window,bs", [(40, 16), (128, 16), (16, 16), (17, 16), (512, 32)])
def test_ring_paging_live_blocks_distinct_and_overwrites_dead(window, bs):
    w = wl.Workload("ring", Hq=8, Hkv=2, D=64, block_size=bs,
                    context_lens=(1, 15, 16, 17, 90, 333, 1024), windows=(window,), seed=5)
    pg = wl.ring_paging(w, window, "cpu")
    R = (window + bs - 1) // bs + 1
    assert pg.num_blocks == w.B * R
    bt = pg.block_table
    for b, L in enumerate(w.context_lens):
        for Lc in range(1, L + 1):                  # every intermediate context length
            lo = max(0, Lc - window)
            live = [int(bt[b][p // bs]) for p in range(lo, Lc)]
            logical = sorted({p // bs for p in range(lo, Lc)})
            assert len({int(bt[b][j]) for j in logical}) == len(logical)
            assert all(0 <= x < pg.num_blocks for x in live)
            # the block the newest position was written into held, before this
            # write, only positions below the window's start
            p = Lc - 1
            j = p // bs
            for older in range(j - R, -1, -R):
                assert int(bt[b][older]) == int(bt[b][j])
                assert (older + 1) * bs <= lo
