"""The C-ABI library builds, loads and exports every entry point the header declares; argument
validation answers without a GPU (no kernel is launched on a rejected call)."""
import ctypes
import os
import re

import pytest

import compressed_sparse_attention_step_gb300 as csa2
from compressed_sparse_attention_step_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "csa2.h")


@pytest.fixture(scope="module")
def L():
    _build.build()
    return csa2.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n


def test_struct_layout_and_status_strings(L):
    assert L.csa2_group_desc_size() == ctypes.sizeof(csa2.GroupDesc)
    for s in range(5):
        assert L.csa2_status_string(s)
    assert L.csa2_status_string(99) == b"unknown status"


def test_workspace_sizes(L):
    assert csa2.workspace_size(csa2.OP_TOPK, B=4, Nq=1, n=8192, k=512) == 0      # one CTA per row
    assert csa2.workspace_size(csa2.OP_TOPK, B=4, Nq=1, n=131072, k=512) > 4 * 4096 * 4
    a = csa2.workspace_size(csa2.OP_SPARSE_ATTN, B=64, Nq=1, k=512, W=128)
    ns = L.csa2_attn_auto_split(64, 512, 128)
    n_tiles = L.csa2_attn_auto_split(1, 512, 128)          # one query: one split per row tile
    assert n_tiles >= 2 and 1 < ns <= n_tiles
    assert a == 64 * ns * (16 * 512 + 32) * 4 + 64 * 4     # partials + one ticket per query
    # an explicit split larger than the tile count is clamped to it
    assert csa2.workspace_size(csa2.OP_SPARSE_ATTN, B=64, Nq=1, k=512, W=128, n_split=32) == \
        64 * n_tiles * (16 * 512 + 32) * 4 + 64 * 4
    assert csa2.workspace_size(csa2.OP_SPARSE_ATTN, B=4096, Nq=1, k=512, W=128) == 0   # one split
    g = csa2.group_workspace_size(64, 1, 131072)
    assert g >= 64 * 131072 * 4 + a
    h = csa2.group_workspace_size(8, 1, 1 << 20, hierarchical=True)
    assert h >= 8 * (1 << 17) * 4
    assert L.csa2_workspace_size(csa2.OP_GROUP_STEP, None) == 0


def test_argument_validation_without_gpu(L):
    fake = ctypes.c_void_p(0x10000)       # aligned, never dereferenced on a rejected call
    odd = ctypes.c_void_p(0x10001)
    # wrong latent width
    assert L.csa2_fp4_quantize_append(fake, 1, 1, 256, fake, fake, 4, None, None) == 2
    assert L.csa2_fp4_dequantize(fake, fake, 1, 500, fake, None) == 2
    # null / misaligned pointers, bad sizes
    assert L.csa2_fp4_quantize_append(None, 1, 1, 512, fake, fake, 4, None, None) == 1
    assert L.csa2_fp4_quantize_append(odd, 1, 1, 512, fake, fake, 4, None, None) == 1
    assert L.csa2_fp4_quantize_append(fake, 1, 5, 512, fake, fake, 4, None, None) == 1   # n_new > cap
    assert L.csa2_topk(fake, 1, 10, 10, None, 0, None, 0, fake, None, None, 0, None) == 1
    assert L.csa2_topk(fake, 1, 10, 10, None, 4096, None, 0, fake, None, None, 0, None) == 1
    assert L.csa2_topk(fake, 1, 10, 5, None, 4, None, 0, fake, None, None, 0, None) == 1   # ld < n
    assert L.csa2_index_score(fake, fake, 1, 1, fake, 16, fake, None, None, 0, 0, None, fake, None, None) == 1
    assert L.csa2_sparse_attn_decode(fake, 1, 1, fake, fake, 16, fake, None, 1024, None, None, 0,
                                     0.1, fake, None, 0, None, 0, None) == 1               # k > 512
    assert L.csa2_sparse_attn_decode(fake, 1, 1, fake, fake, 16, fake, None, 512, fake, fake, 256,
                                     0.1, fake, None, 0, None, 0, None) == 1               # W > 128
    # the auto split needs workspace: NULL workspace is reported, nothing launched
    assert L.csa2_sparse_attn_decode(fake, 1, 1, fake, fake, 16, fake, None, 512, None, None, 0,
                                     0.1, fake, None, 0, None, 0, None) == 4
    # empty problems are no-ops
    assert L.csa2_fp4_quantize_append(None, 0, 0, 512, None, None, 0, None, None) == 0
    assert L.csa2_topk(None, 0, 0, 0, None, 1, None, 0, None, None, None, 0, None) == 0
    assert L.csa2_topk(fake, 2, 1 << 17, 1 << 17, None, 512, None, 0, fake, None, None, 0, None) == 4  # needs ws
    # group descriptor checks
    g = csa2.GroupDesc()
    g.n_layers = 0
    assert L.csa2_group_step(ctypes.byref(g), None, 0, None) == 1
    g.n_layers, g.B, g.Nq, g.K, g.W, g.ratio, g.cap = 2, 1, 1, 512, 128, 1, 1024
    g.modes[0] = csa2.MODE_REUSE
    assert L.csa2_group_step(ctypes.byref(g), None, 0, None) == 1                            # Reuse first
    assert L.csa2_group_step(None, None, 0, None) == 1
