"""GPU parity of the prefill selection on the tensor cores (csa2_index_select_prefill and the group
step's prefill route) against the oracle: the index sets are bit-exact with the oracle's canonical
scores and Top-k, for partial query tiles, several sequences, queries that see fewer than k (or
fewer than k groups of 32) positions, massive ties (every key survives the filter and streams
through the candidate list), all-negative head weights (ties at 0), k = 2048, small-integer indexer
data (every tensor-core and canonical score is then exact, so both must agree bit for bit, with
heavy ties), a prefill group step, and the full 2048-query x 131072-entry chunk on every row."""
import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import DI, HOST_THREADS, GroupCase, bf16_dev, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402

F, R = c.MODE_FULL, c.MODE_REUSE


def _visible(T, Nq, ratio, q_pos, b, i):
    p = int(q_pos[b, i]) if q_pos is not None else ratio * T[b] - Nq + i
    return 0 if p + 1 < 0 else min((p + 1) // ratio, T[b])


def _expected(orc, KI, qI, w, T, Nq, ratio, q_pos, k, rows):
    out = {}
    for (b, i) in rows:
        nv = _visible(T, Nq, ratio, q_pos, b, i)
        s = orc.index_score(qI[b, i], w[b, i], KI[b], n=nv) if nv > 0 else np.zeros(0, np.float32)
        out[(b, i)] = orc.topk(s, k)[0] if nv > 0 else np.full(k, -1, np.int32)
    return out


def _run(KI, qI, w, T, ratio, q_pos, k):
    B, Nq = qI.shape[0], qI.shape[1]
    idx = torch.full((B * Nq, k), -7, dtype=torch.int32, device="cuda")
    n_sel = torch.zeros(B * Nq, dtype=torch.int32, device="cuda")
    c.csa2_index_select_prefill(bf16_dev(qI), torch.from_numpy(w).cuda(), bf16_dev(KI),
                                to_dev(np.array(T, np.int32)), idx, k=k, ratio=ratio,
                                q_pos=None if q_pos is None else to_dev(q_pos.reshape(-1)), n_sel=n_sel)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), n_sel.cpu().numpy()


def _inputs(seed, B, cap, Nq):
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, b, (cap, DI)) for b in range(B)])
    qI = np.stack([syn.normal_bf16(seed, syn.T_QI, b, (Nq, 4, DI)) for b in range(B)])
    w = np.stack([syn.normal_f32(seed, syn.T_W, b, (Nq, 4)) for b in range(B)]).astype(np.float32)
    return KI, qI, w


def _check_all(orc, KI, qI, w, T, ratio, q_pos, k, rows=None):
    B, Nq = qI.shape[0], qI.shape[1]
    got, n_sel = _run(KI, qI, w, T, ratio, q_pos, k)
    rows = rows if rows is not None else [(b, i) for b in range(B) for i in range(Nq)]
    exp = _expected(orc, KI, qI, w, T, Nq, ratio, q_pos, k, rows)
    for (b, i), e in exp.items():
        r = b * Nq + i
        assert np.array_equal(got[r], e), f"row {(b, i)}"
        assert n_sel[r] == int((e >= 0).sum())


def test_prefill_select_partial_tiles_two_sequences(orc):
    """96 queries (one full and one partial tile of 64) per sequence, ratio 2, causal at the end."""
    B, Nq, k = 2, 96, 512
    T = [20000, 17000]
    KI, qI, w = _inputs(61, B, 20480, Nq)
    _check_all(orc, KI, qI, w, T, 2, None, k, rows=[(b, i) for b in range(B) for i in (0, 1, 37, 63, 64, 95)])


def test_prefill_select_arbitrary_positions(orc):
    """Query positions spread over the context: some see fewer than k entries, some fewer than
    512 groups of 32 (every visible key survives the filter), some the whole cache."""
    B, Nq, k = 1, 64, 256
    T = [30000]
    q_pos = np.linspace(0, 2 * 30000 - 1, Nq).astype(np.int32)[None]
    KI, qI, w = _inputs(62, B, 30720, Nq)
    _check_all(orc, KI, qI, w, T, 2, q_pos, k, rows=[(0, i) for i in (0, 1, 3, 10, 20, 40, 63)])


def test_prefill_select_massive_ties(orc):
    """All keys equal: every score ties, every key survives the filter (more than the candidate
    list holds), and the selection returns the k lowest visible positions."""
    B, Nq, k, T = 1, 64, 512, [14000]
    KI = np.zeros((B, 14336, DI), np.uint16)
    _, qI, w = _inputs(63, B, 16, Nq)
    got, n_sel = _run(KI, qI, w, T, 1, None, k)
    for i in (0, 31, 63):
        nv = _visible(T, Nq, 1, None, 0, i)
        assert nv > 10240
        assert np.array_equal(got[i], np.arange(k, dtype=np.int32))
    _check_all(orc, KI, qI, w, T, 1, None, k, rows=[(0, 5)])


def test_prefill_select_negative_weights_stream_ties(orc):
    """Rows whose four head weights are all negative score <= 0 everywhere: thousands of keys tie at
    0 and survive the filter, more than the candidate list holds, so the list is cut back to its k
    best while the marked keys stream through.  k = 2048 (every visible key is marked: fewer than
    2048 groups of 32) and k = 64 (ties at the threshold)."""
    B, Nq, T = 1, 64, 24000
    KI, qI, w = _inputs(64, B, 24576, Nq)
    w[0, ::2] = -np.abs(w[0, ::2])
    rows = [(0, i) for i in (0, 1, 2, 31, 62, 63)]
    for k in (64, 2048):
        _check_all(orc, KI, qI, w, [T], 2, None, k, rows=rows)


def test_prefill_select_rounding_adversarial(orc):
    """Indexer data from {0, +-1, +-2, +-2^12}, whose fp32 scores depend on the order of every
    addition: the tensor-core filter's error bound is large relative to the spread of the scores, so
    nearly every key is rescored in the canonical order, and the selection (ties included) must
    still be the oracle's exactly."""
    from tests.test_gpu_score_topk import _adversarial
    B, Nq, cap, k = 1, 64, 6144, 512
    KI = _adversarial(3, (B, cap, DI))
    qI = _adversarial(4, (B, Nq, 4, DI))
    w = np.broadcast_to(np.array([1.0, -1.0, np.float32(1.0 + 2.0 ** -23), 3.0], np.float32), (B, Nq, 4)).copy()
    T = [6000]
    exp, _ = orc.index_select(KI, qI, w, T, k, ratio=1, threads=HOST_THREADS)
    got, _ = _run(KI, qI, w, T, 1, None, k)
    assert np.array_equal(got.reshape(B, Nq, k), exp)


def _int_inputs(seed, B, cap, Nq):
    KI = np.stack([syn.integer_bf16(seed, syn.T_KI, b, (cap, DI), -8, 8) for b in range(B)])
    qI = np.stack([syn.integer_bf16(seed, syn.T_QI, b, (Nq, 4, DI), -8, 8) for b in range(B)])
    w = np.stack([syn.bf16_bits_to_f32(syn.integer_bf16(seed, syn.T_W, b, (Nq, 4), -4, 4)) for b in range(B)])
    return KI, qI, w.astype(np.float32)


@pytest.mark.parametrize("k", [64, 512, 2048])
def test_prefill_select_integer_data_every_row(orc, k):
    """Small-integer indexer keys, queries and head weights: every dot product, weighted sum and
    score is an integer below 2^24, exact in fp32 in any summation order, so the tensor-core filter
    scores equal the canonical scores bit for bit and a fault anywhere in the contraction (operand,
    head, key or query order) changes the selection.  Scores tie heavily.  A quarter of the rows
    get all-negative weights (every score <= 0, ties at 0).  Two sequences of 128 queries (two full
    query tiles), ratio 2, causal at the end; every row against the oracle."""
    B, Nq = 2, 128
    T = [20000, 13001]
    KI, qI, w = _int_inputs(65 + k, B, 20480, Nq)
    w[:, ::4] = -np.abs(w[:, ::4]) - 1.0
    exp, n_exp = orc.index_select(KI, qI, w, T, k, ratio=2, threads=HOST_THREADS)
    got, n_sel = _run(KI, qI, w, T, 2, None, k)
    assert np.array_equal(got.reshape(B, Nq, k), exp)
    assert np.array_equal(n_sel.reshape(B, Nq), n_exp)


def test_prefill_group_step_integer_data(orc):
    """The prefill group step (Full + Reuse) on small-integer indexer data selects exactly the
    oracle's indices for every query (tensor-core scores are exact on such data), and attends as the
    oracle does."""
    Nq, T = 128, 9000
    q_pos = np.arange(2 * T - Nq, 2 * T, dtype=np.int32)[None]
    gc = GroupCase(66, [T], [F, R], Nq=Nq, ratio=2, K=512, W=128, append=False, q_pos=q_pos, integer_index=True)
    assert (gc.h_w(0, 0) < 0).all(axis=1).any()
    gc.run()
    gc.check(orc)


def test_prefill_group_step_ratio2(orc):
    """A prefill chunk of 64 queries through the group step (Full + 2 Reuse) selects on the tensor
    cores; indices and attention outputs match the oracle."""
    Nq, T = 64, 6000
    q_pos = np.arange(2 * T - Nq, 2 * T, dtype=np.int32)[None]
    gc = GroupCase(64, [T], [F, R, R], Nq=Nq, ratio=2, K=256, W=64, append=False, q_pos=q_pos)
    gc.run()
    gc.check(orc)


def test_prefill_select_full_chunk_2048x131072(orc):
    """The encoder prefill chunk: 2048 queries at the end of 262144 tokens (131072 compressed
    entries), Top-512 per query; every row against the oracle."""
    B, Nq, k, T = 1, 2048, 512, [131072]
    seed = syn.SEEDS["prefill_group_1f5r_ratio2_q2048"]
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, 0, (131072, DI))])
    qI = np.stack([syn.normal_bf16(seed, syn.T_QI, 0, (Nq, 4, DI))])
    w = np.stack([syn.normal_f32(seed, syn.T_W, 0, (Nq, 4))]).astype(np.float32)
    got, n_sel = _run(KI, qI, w, T, 2, None, k)
    assert np.all(n_sel == k)
    exp, n_exp = orc.index_select(KI, qI, w, T, k, ratio=2, threads=HOST_THREADS)
    bad = np.nonzero(~np.all(got == exp[0], axis=1))[0]
    assert bad.size == 0, f"{bad.size} of {Nq} rows differ, first {bad[:8]}"
    assert np.array_equal(n_sel, n_exp[0])


def test_prefill_group_full_size_1f5r_q2048_t131072(orc):
    """The encoder prefill chunk through the group step: 1 Full + 5 Reuse layers, ratio 2, 2048
    queries at the end of 262144 tokens (131072 compressed entries), Top-512, 128-token window.
    Every query of every layer against the oracle (indices bit-exact, outputs and lse within the
    tolerance, per (query, head) row); the chunk includes queries whose Full-layer head weights are
    all negative."""
    Nq, T = 2048, 131072
    q_pos = np.arange(2 * T - Nq, 2 * T, dtype=np.int32)[None]
    gc = GroupCase(syn.SEEDS["prefill_group_1f5r_ratio2_q2048"], [T], [F, R, R, R, R, R], Nq=Nq, ratio=2,
                   append=False, q_pos=q_pos)
    assert (gc.h_w(0, 0) < 0).all(axis=1).any()
    gc.run()
    gc.check(orc)

