"""GPU parity of a decoder stack's step (csa2_stack_step): the 20-layer decoder as 5 groups of 4,
the first led by a Full layer that appends the step's token, the other four by Reindex layers that
reuse its cache (and, hierarchical, the pool it kept).  Every layer's indices, outputs and lse are
compared with the oracle's group step over the 20 layers in order; groups that do not share one
batch, cache and append are rejected before anything runs."""
import numpy as np
import pytest

from tests._cases import GroupCase, check_stack

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402

F, RX, R = c.MODE_FULL, c.MODE_REINDEX, c.MODE_REUSE


def _stack(seed, T, hierarchical=False):
    g0 = GroupCase(seed, T, [F, R, R, R], hierarchical=hierarchical)
    return [g0] + [GroupCase(seed, T, [RX, R, R, R], hierarchical=hierarchical, share=g0, layer0=4 * i)
                   for i in range(1, 5)]


def test_decoder_stack_20_layers_flat(orc):
    gs = _stack(71, [3000, 700, 2049, 9])
    c.csa2_stack_step([g.desc() for g in gs], gs[0].ws)
    torch.cuda.synchronize()
    check_stack(orc, gs)


def test_decoder_stack_20_layers_hierarchical(orc):
    """Reindex-led groups rescore the pool the first group's Full layer kept (more than 2048 blocks
    in one sequence, fewer in the other; the append completes a block in one of them)."""
    gs = _stack(72, [8 * 2600 + 3, 8 * 900], hierarchical=True)
    c.csa2_stack_step([g.desc() for g in gs], gs[0].ws)
    torch.cuda.synchronize()
    check_stack(orc, gs)


def test_stack_rejects_mismatched_groups():
    gs = _stack(73, [500, 300])
    descs = [g.desc() for g in gs]
    bad_append = [g.desc() for g in gs]
    bad_append[2].n_new = 1
    bad_append[2].kv_new = descs[0].kv_new
    other = torch.zeros_like(gs[0].codes)
    bad_cache = [g.desc() for g in gs]
    bad_cache[3].codes = other.data_ptr()
    bad_shape = [g.desc() for g in gs]
    bad_shape[1].B = 1
    for bad in (bad_append, bad_cache, bad_shape):
        with pytest.raises(c.Csa2Error) as e:
            c.csa2_stack_step(bad, gs[0].ws)
        assert e.value.status == c.ERR_INVALID_ARG
    torch.cuda.synchronize()
    for g in gs:  # nothing ran
        assert all(int(o.abs().sum()) == 0 for o in g.out)
    c.csa2_stack_step(descs, gs[0].ws)
    torch.cuda.synchronize()
    assert all(int(o.abs().sum()) > 0 for g in gs for o in g.out)
