"""Host models of kernel loop structures whose warp collectives need every lane of a warp.

A full-mask shuffle executed by only some lanes of a warp is undefined and can stall the warp, so a
loop whose body shuffles must give every lane of a warp the same trip count.  These models restate
the index arithmetic of such loops and check it over chunk lengths of every residue."""
import pytest


@pytest.mark.parametrize("t1", [1, 2, 3, 4, 5, 31, 32, 33, 544, 713, 1023, 1024])
def test_key_norm_loop_is_warp_uniform_and_covers_every_entry(t1):
    # prefill_key_norm_kernel: 256 threads, eight per entry, a warp takes four consecutive entries per
    # step; the loop runs on the warp's first entry tw and lanes past the chunk's end add nothing
    blk, t0 = 256, 0
    seen = []
    for warp in range(blk // 32):
        trips = set()
        for lane in range(32):
            x, n = warp * 32 + lane, 0
            tw = t0 + ((x >> 5) << 2)
            while tw < t1:
                t = tw + ((x & 31) >> 3)
                if t < t1 and (x & 7) == 0:
                    seen.append(t)
                tw += blk >> 3
                n += 1
            trips.add(n)
        assert len(trips) == 1, f"warp {warp}: lanes make different trip counts {trips}"
    assert sorted(seen) == list(range(t0, t1))
