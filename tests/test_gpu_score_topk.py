"""GPU parity of the indexer-score, Top-K, block-key and block-pool kernels against the oracle:
bit-exact fp32 scores, index sets, block keys and pools, including ragged contexts, causal
masking over compressed entries, candidate pools, heavy ties (the fallback selection path),
k = 2048, and rows at the full context of the decode workloads."""
import numpy as np
import pytest

import csa2_synth as syn
from tests._cases import bf16_dev, bf16_host, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)
import compressed_sparse_attention_step_gb300 as c  # noqa: E402


def _score_inputs(seed, B, Nq, cap):
    qI = np.stack([syn.normal_bf16(seed, syn.T_QI, b, (Nq, 4, 128)) for b in range(B)])
    w = np.stack([syn.normal_f32(seed, syn.T_W, b, (Nq, 4)) for b in range(B)])
    KI = np.stack([syn.normal_bf16(seed, syn.T_KI, b, (cap, 128)) for b in range(B)])
    return qI, w, KI


def _adversarial(seed, shape):
    """bf16 values from {0, +-1, +-2, +-2^12}: products of 2^24, 2^13, 2^12 and small integers make
    fp32 sums absorb and tie, so any summation order other than the canonical one changes bits."""
    g = np.random.default_rng(seed)
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0, 4096.0, -4096.0], np.float32)
    p = np.array([0.6, 0.12, 0.12, 0.05, 0.05, 0.03, 0.03])
    return syn.f32_to_bf16_bits(g.choice(vals, size=shape, p=p).astype(np.float32))


def test_scores_rounding_order_adversarial(orc):
    """Scores of crafted keys and queries whose fp32 sums depend on the order of every addition (see
    _adversarial) are bit-identical to the oracle's canonical order; head weights include 1 + 2^-23
    and 3 so that each weighted product's own rounding matters."""
    B, Nq, cap = 2, 3, 4096
    qI = _adversarial(1, (B, Nq, 4, 128))
    KI = _adversarial(2, (B, cap, 128))
    w = np.array([[1.0, -1.0, np.float32(1.0 + 2.0 ** -23), 3.0], [0.5, 1.0, 1.0, 1.0], [-1.0, 2.0, 0.25, 1.0]],
                 np.float32)
    w = np.broadcast_to(w[None], (B, Nq, 4)).copy()
    sc = torch.zeros((B * Nq, cap), device="cuda")
    c.csa2_index_score(bf16_dev(qI), to_dev(w), bf16_dev(KI), to_dev(np.full(B, cap, np.int32)), sc)
    sc = sc.cpu().numpy()
    for b in range(B):
        for i in range(Nq):
            n = cap - Nq + i + 1
            exp = orc.index_score(qI[b, i], w[b, i], KI[b], n=n)
            assert np.array_equal(sc[b * Nq + i, :n].view(np.uint32), exp.view(np.uint32)), (b, i)


def test_scores_flat_ragged(orc):
    B, Nq, cap = 3, 2, 1000
    lens = [1000, 517, 3]
    qI, w, KI = _score_inputs(31, B, Nq, cap)
    sc = torch.full((B * Nq, cap), 123.0, device="cuda")
    nv = torch.zeros(B * Nq, dtype=torch.int32, device="cuda")
    c.csa2_index_score(bf16_dev(qI), to_dev(w), bf16_dev(KI), to_dev(np.array(lens, np.int32)), sc, n_valid=nv)
    sc, nv = sc.cpu().numpy(), nv.cpu().numpy()
    for b in range(B):
        for i in range(Nq):
            r = b * Nq + i
            n = lens[b] - Nq + i + 1          # query i sits at position T - Nq + i
            assert nv[r] == n
            exp = orc.index_score(qI[b, i], w[b, i], KI[b], n=n)
            assert np.array_equal(sc[r, :n].view(np.uint32), exp.view(np.uint32))
            assert np.all(np.isneginf(sc[r, n:]))


def test_scores_causal_ratio2_and_pool(orc):
    B, Nq, cap = 2, 4, 700
    lens = [700, 450]
    qI, w, KI = _score_inputs(32, B, Nq, cap)
    q_pos = np.array([[3, 100, 901, 1399], [0, 1, 899, 2000]], np.int32)
    sc = torch.zeros((B * Nq, cap), device="cuda")
    nv = torch.zeros(B * Nq, dtype=torch.int32, device="cuda")
    c.csa2_index_score(bf16_dev(qI), to_dev(w), bf16_dev(KI), to_dev(np.array(lens, np.int32)), sc, ratio=2,
                       q_pos=to_dev(q_pos.reshape(-1)), n_valid=nv)
    sc, nv = sc.cpu().numpy(), nv.cpu().numpy()
    for b in range(B):
        for i in range(Nq):
            n = min(lens[b], (q_pos[b, i] + 1) // 2)
            assert nv[b * Nq + i] == n
            exp = orc.index_score(qI[b, i], w[b, i], KI[b], n=n)
            assert np.array_equal(sc[b * Nq + i, :n], exp)
    # candidate pool (ascending positions, ragged lengths), causal prefix inside the pool
    g = np.random.default_rng(0)
    n_cand = 300
    cand = np.full((B * Nq, n_cand), -1, np.int32)
    clen = np.array([300, 250, 120, 0, 300, 17, 299, 1], np.int32)
    for r in range(B * Nq):
        cand[r, :clen[r]] = np.sort(g.choice(lens[r // Nq], clen[r], replace=False))
    sc = torch.zeros((B * Nq, n_cand), device="cuda")
    nv = torch.zeros(B * Nq, dtype=torch.int32, device="cuda")
    c.csa2_index_score(bf16_dev(qI), to_dev(w), bf16_dev(KI), to_dev(np.array(lens, np.int32)), sc,
                       cand=to_dev(cand), cand_len=to_dev(clen), ratio=2, q_pos=to_dev(q_pos.reshape(-1)),
                       n_valid=nv)
    sc, nv = sc.cpu().numpy(), nv.cpu().numpy()
    for r in range(B * Nq):
        b, i = divmod(r, Nq)
        vis = min(lens[b], (q_pos[b, i] + 1) // 2)
        m = int(np.sum(cand[r, :clen[r]] < vis))
        assert nv[r] == m
        exp = orc.index_score(qI[b, i], w[b, i], KI[b], pos=cand[r, :m])
        assert np.array_equal(sc[r, :m], exp) and np.all(np.isneginf(sc[r, m:]))


def _topk_rows(n):
    g = np.random.default_rng(n)
    rows = [
        g.standard_normal(n).astype(np.float32),                               # generic
        np.round(g.standard_normal(n) * 3).astype(np.float32),                 # ties
        np.full(n, 0.5, np.float32),                                           # all equal: fallback
        g.choice(np.array([0.0, -0.0, 2.0, -2.0], np.float32), n),             # +-0, heavy ties
        (g.standard_normal(n) * 1e-3 + 7.0).astype(np.float32),                # one narrow bin
        -np.abs(g.standard_normal(n)).astype(np.float32),                      # all negative
    ]
    s = np.stack(rows)
    s[0, 5] = np.inf
    s[0, 6] = -np.inf
    return s


@pytest.mark.parametrize("n,k", [(1000, 512), (131072, 512), (131072, 2048), (4096, 1), (600, 512), (16384, 512),
                                 (16384, 2048), (12000, 512), (16385, 512)])
def test_topk_matches_oracle(orc, n, k):
    s = _topk_rows(n)
    rows = s.shape[0]
    nvalid = np.array([n, n - 7, n, n // 2, min(n, k - 1), n], np.int32)
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(rows, dtype=torch.int32, device="cuda")
    c.csa2_topk(to_dev(s), k, idx, n_valid=to_dev(nvalid), n_sel=nsel)
    idx, nsel = idx.cpu().numpy(), nsel.cpu().numpy()
    for r in range(rows):
        exp, cnt = orc.topk(s[r, :nvalid[r]], k)
        assert nsel[r] == cnt
        assert np.array_equal(idx[r], exp), r


def test_topk_long_rows_bound_and_overflow(orc):
    """Rows longer than 8192 columns, at the edges of the group-key bound: fewer than k groups of
    16 (every key is a candidate; the list holds them, or overflows to the whole-row selection),
    a valid prefix one past a group, all keys equal over 262144 columns (more groups at the bound
    than the group list holds), and a row where only the top group keys' bin survives."""
    g = np.random.default_rng(11)
    n, k = 262144, 2048
    s = np.stack([g.standard_normal(n).astype(np.float32) for _ in range(4)] +
                 [np.full(n, -1.25, np.float32), (g.standard_normal(n) * 1e-4).astype(np.float32)])
    nvalid = np.array([9000, 20000, 16 * 2048 + 1, 8193, n, n - 3], np.int32)
    idx = torch.full((s.shape[0], k), -5, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(s.shape[0], dtype=torch.int32, device="cuda")
    c.csa2_topk(to_dev(s), k, idx, n_valid=to_dev(nvalid), n_sel=nsel)
    idx, nsel = idx.cpu().numpy(), nsel.cpu().numpy()
    for r in range(s.shape[0]):
        exp, cnt = orc.topk(s[r, :nvalid[r]], k)
        assert nsel[r] == cnt
        assert np.array_equal(idx[r], exp), r


def _cluster_rows(n, k, g):
    """Rows for the one-cluster-per-row selection (8193 to 131072 columns)."""
    rows = []
    r = g.standard_normal(n).astype(np.float32)
    r[g.choice(n, k + 700, replace=False)] = 5.0       # the largest key k + 700 times: its k lowest columns
    rows.append(r)
    r = g.standard_normal(n).astype(np.float32)
    r[g.choice(n, k, replace=False)] = 5.0             # exactly k times
    rows.append(r)
    r = g.standard_normal(n).astype(np.float32)
    pos = g.choice(n, k + 9, replace=False)
    r[pos[:k - 1]] = 5.0                               # k - 1 times, then ten ties one key lower
    r[pos[k - 1:]] = 4.0
    rows.append(r)
    rows.append(np.where(g.random(n) < 0.5, 0.0, -0.0).astype(np.float32))  # +0 and -0 only: one key
    r = (g.standard_normal(n) * 1e-4).astype(np.float32)
    r[n // 4 - 3:n // 4 + 3] = 1.0                     # ties across the boundary of the first CTA's run
    r[n // 2 - 8:n // 2 + 8] = 1.0
    rows.append(r)
    rows.append(np.round(g.standard_normal(n) * 8).astype(np.float32))  # wide bins, many ties at the cut
    return np.stack(rows)


@pytest.mark.parametrize("k", [512, 2048])
@pytest.mark.parametrize("reps", [1, 8])
def test_topk_cluster_rows(orc, k, reps):
    """One thread-block cluster per row (eight CTAs for the 6 rows, four for 48): the largest key held
    by at least k columns (each CTA writes its share of the k lowest in column order), by exactly k
    and by k - 1 (then the list), signed zeros only, ties across the CTAs' runs, and valid prefixes
    whose every key is listed (8000: the list holds them; 8193 and 9000: the whole-row fallback)."""
    g = np.random.default_rng(31 + k)
    n = 131072
    s = np.concatenate([_cluster_rows(n, k, g) for _ in range(reps)])
    rows = s.shape[0]
    nvalid = np.full(rows, n, np.int32)
    nvalid[5::6] = [8000, 8193, 9000, n - 5, 40000, 131071, 70000, 16 * k + 1][:len(nvalid[5::6])]
    idx = torch.full((rows, k), -5, dtype=torch.int32, device="cuda")
    nsel = torch.zeros(rows, dtype=torch.int32, device="cuda")
    c.csa2_topk(to_dev(s), k, idx, n_valid=to_dev(nvalid), n_sel=nsel)
    idx, nsel = idx.cpu().numpy(), nsel.cpu().numpy()
    for r in range(rows):
        exp, cnt = orc.topk(s[r, :nvalid[r]], k)
        assert nsel[r] == cnt
        assert np.array_equal(idx[r], exp), r


def test_topk_with_map(orc):
    g = np.random.default_rng(5)
    n, k = 16384, 512
    s = g.standard_normal((3, n)).astype(np.float32)
    mp = np.stack([np.sort(g.choice(1 << 20, n, replace=False)) for _ in range(3)]).astype(np.int32)
    idx = torch.empty((3, k), dtype=torch.int32, device="cuda")
    c.csa2_topk(to_dev(s), k, idx, map_=to_dev(mp))
    idx = idx.cpu().numpy()
    for r in range(3):
        exp, _ = orc.topk(s[r], k, mp[r])
        assert np.array_equal(idx[r], exp)


def test_block_keys_and_pool(orc):
    B, cap = 3, 8 * 3000
    lens = [8 * 3000, 8 * 1200 + 5, 8 * 2500 + 7]
    KI = np.stack([syn.normal_bf16(33, syn.T_KI, b, (cap, 128)) for b in range(B)])
    bk = torch.zeros((B, cap // 8, 128), dtype=torch.bfloat16, device="cuda")
    lens_d = to_dev(np.array(lens, np.int32))
    c.csa2_block_keys_build(bf16_dev(KI), lens_d, bk)
    bkh = bf16_host(bk)
    obk = []
    for b in range(B):
        o = orc.block_keys(KI[b, :lens[b]])
        assert np.array_equal(bkh[b, :lens[b] // 8], o)
        obk.append(o)
    qI = np.stack([syn.normal_bf16(33, syn.T_QI, b, (1, 4, 128)) for b in range(B)])
    w = np.stack([syn.normal_f32(33, syn.T_W, b, (1, 4)) for b in range(B)])
    keep = 2048
    pool = torch.full((B, keep * 8), -3, dtype=torch.int32, device="cuda")
    plen = torch.zeros(B, dtype=torch.int32, device="cuda")
    c.csa2_block_pool(bf16_dev(qI), to_dev(w), bk, cap, lens_d, keep, pool, plen)
    pool, plen = pool.cpu().numpy(), plen.cpu().numpy()
    for b in range(B):
        ep, en = orc.block_pool(qI[b, 0], w[b, 0], obk[b], lens[b] // 8, keep)
        assert plen[b] == en and np.array_equal(pool[b], ep)


def test_full_context_rows_of_decode_workload(orc):
    """Rows at the 128K context of the batched decode workload: scores and Top-512 of two
    sampled sequences, computed in one launch over a batch of 64."""
    B, T = 64, 131072
    seed = syn.SEEDS["decode_group_1f3r_b64_t131072"]
    KI = syn.device_normal_bf16((B, T, 128), seed, syn.T_KI * 1000)
    qI = syn.device_normal_bf16((B, 1, 4, 128), seed, syn.T_QI)
    w = syn.device_normal_bf16((B, 1, 4), seed, syn.T_W).float()
    sampled = [3, 50]
    host = {}
    for b in sampled:
        host[b] = (syn.normal_bf16(seed, syn.T_KI, b, (T, 128)), syn.normal_bf16(seed, syn.T_QI, b, (1, 4, 128)),
                   syn.normal_f32(seed, syn.T_W, b, (1, 4)))
        KI[b].copy_(bf16_dev(host[b][0]))
        qI[b].copy_(bf16_dev(host[b][1]))
        w[b].copy_(to_dev(host[b][2]))
    lens = torch.full((B,), T, dtype=torch.int32, device="cuda")
    sc = torch.empty((B, T), device="cuda")
    nv = torch.empty(B, dtype=torch.int32, device="cuda")
    c.csa2_index_score(qI, w, KI, lens, sc, n_valid=nv)
    idx = torch.empty((B, 512), dtype=torch.int32, device="cuda")
    c.csa2_topk(sc, 512, idx, n_valid=nv)
    for b in sampled:
        ki, qi, wi = host[b]
        exp = orc.index_score(qi[0], wi[0], ki)
        assert np.array_equal(sc[b].cpu().numpy(), exp)
        ei, _ = orc.topk(exp, 512)
        assert np.array_equal(idx[b].cpu().numpy(), ei)
