"""Case builders shared by the GPU parity tests and the smoke check.

Every input comes from the seeded generators in `csa2_synth`.  Small cases draw everything on the
host and upload it; full-size cases fill the device with torch's generator and overwrite the
sampled sequences with the host draw, so the oracle (which only ever sees host draws) and the
CUDA path get identical bytes for every sequence that is compared.  Nothing here computes any
part of the method: the GPU cache is filled by the library's own quantiser, the oracle's by the
oracle's.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import csa2_synth as syn

# host threads for the oracle and for drawing many sequences (numpy's generators release the GIL)
HOST_THREADS = max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))

D, H, HI, DI = 512, 16, 4, 128
SCALE = float(np.float32(1.0 / np.sqrt(D)))

# attention outputs: |gpu - oracle| <= ATOL everywhere, and ||gpu - oracle|| <= RTOL ||oracle|| for
# every (query, head) row of 512 channels on its own as well as over the whole tensor
ATOL, RTOL = 2e-2, 1e-2


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(a):
    import torch
    return to_dev(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)


def bf16_host(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_attn_close(got_bf16_bits, ref, what=""):
    """Attention outputs [..., 512] against the oracle: element-wise max-abs ATOL, and relative
    error RTOL per (query, head) row and over the whole tensor.  A row the oracle gives as exactly
    zero (a query with no rows) must be exactly zero."""
    got = syn.bf16_bits_to_f32(got_bf16_bits).astype(np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    g2, r2 = got.reshape(-1, got.shape[-1]), ref.reshape(-1, ref.shape[-1])
    rn = np.linalg.norm(r2, axis=1)
    en = np.linalg.norm(g2 - r2, axis=1)
    zero = rn == 0.0
    assert not np.any(en[zero] > 0.0), f"{what}: {int(np.sum(en[zero] > 0))} rows should be exactly zero"
    row_rel = en[~zero] / rn[~zero]
    worst = float(row_rel.max()) if row_rel.size else 0.0
    assert err.max() <= ATOL and rel <= RTOL and worst <= RTOL, \
        f"{what}: max abs {err.max():.3e}, rel {rel:.3e}, worst row rel {worst:.3e}"


class GroupCase:
    """One CSA2 layer group: inputs on host (per sequence) and on the device.

    T: per-sequence context after the step's append (list).  The device cache is filled for rows
    [0, T_b - 1) by the library's quantiser; the step itself appends row T_b - 1 (kv_new/ki_new)
    when `append` is set, otherwise rows [0, T_b) are filled up front.
    """

    def __init__(self, seed, T, modes, *, Nq=1, K=512, W=128, ratio=1, hierarchical=False, keep=2048,
                 cap=None, append=True, host_seqs=None, q_pos=None, share=None, layer0=0, swa_fp8=False,
                 integer_index=False):
        """share: a case whose cache, lengths, block keys and pool this one uses (a later group of
        a decoder stack: no append of its own); layer0: the stack index of this group's first
        layer (its per-layer draws use tensor ids offset by it); swa_fp8: 8-bit (E4M3) window rows,
        quantised from the bf16 draws by the oracle for host-drawn sequences (both sides see the
        same bytes) and by the library elsewhere; integer_index: indexer keys and queries are small
        integers in [-8, 8] and head weights integers in [-4, 4] (every indexer score is then exact
        in fp32 in any summation order, and ties are plentiful); host-drawn sequences only."""
        self.integer_index = integer_index
        assert not integer_index or host_seqs is None
        import torch
        import compressed_sparse_attention_step_gb300 as c
        self.c = c
        self.seed, self.T, self.modes = seed, list(T), list(modes)
        self.B, self.L = len(T), len(modes)
        self.Nq, self.K, self.W, self.ratio = Nq, K, W, ratio
        self.hierarchical, self.keep = hierarchical, keep
        self.cap = cap if cap is not None else max(T)
        self.append = append and Nq == 1 and share is None
        self.layer0 = layer0
        self.swa_fp8 = swa_fp8
        self.host_seqs = list(range(self.B)) if host_seqs is None else list(host_seqs)
        self.q_pos = q_pos
        B, L, cap, SW = self.B, self.L, self.cap, W - 1 + Nq
        dev = "cuda"
        self.lens = torch.tensor(self.T, dtype=torch.int32, device=dev)
        self.swa_len_np = np.minimum(np.array(self.T), SW).astype(np.int32)
        self.swa_len = to_dev(self.swa_len_np)
        # device tensors
        self.codes = torch.zeros((B, cap, 256), dtype=torch.uint8, device=dev)
        self.scales = torch.zeros((B, cap, 32), dtype=torch.uint8, device=dev)
        self.KI = torch.zeros((B, cap, DI), dtype=torch.bfloat16, device=dev)
        full_host = len(self.host_seqs) == B
        if full_host:
            self.q = [bf16_dev(np.stack([self.h_q(l, b) for b in range(B)])) for l in range(L)]
            self.qI = [bf16_dev(np.stack([self.h_qI(l, b) for b in range(B)])) for l in range(L)]
            self.w = [to_dev(np.stack([self.h_w(l, b) for b in range(B)])) for l in range(L)]
            self.swa = [self._dev_win(np.stack([self.h_swa(l, b) for b in range(B)])) for l in range(L)]
        else:
            l0 = layer0
            self.q = [syn.device_normal_bf16((B, Nq, H, D), seed, syn.T_Q + l0 + l) for l in range(L)]
            self.qI = [syn.device_normal_bf16((B, Nq, HI, DI), seed, syn.T_QI + l0 + l) for l in range(L)]
            self.w = [syn.device_normal_bf16((B, Nq, HI), seed, syn.T_W + l0 + l).float() for l in range(L)]
            self.swa = [self._dev_win_device(syn.device_normal_bf16((B, SW, D), seed, syn.T_SWA + l0 + l))
                        for l in range(L)]
            for b in self.host_seqs:
                for l in range(L):
                    self.q[l][b].copy_(bf16_dev(self.h_q(l, b)))
                    self.qI[l][b].copy_(bf16_dev(self.h_qI(l, b)))
                    self.w[l][b].copy_(to_dev(self.h_w(l, b)))
                    self.swa[l][b].copy_(self._dev_win(self.h_swa(l, b)))
        # cache rows (kept before the step; the last row comes from the step's append)
        self.kv_new = torch.zeros((B, 1, D), dtype=torch.bfloat16, device=dev)
        self.ki_new = torch.zeros((B, 1, DI), dtype=torch.bfloat16, device=dev)
        if share is not None:
            self.codes, self.scales, self.KI, self.lens = share.codes, share.scales, share.KI, share.lens
            self.__dict__["_kv"] = share.__dict__.setdefault("_kv", {})
            self.__dict__["_ki"] = share.__dict__.setdefault("_ki", {})
        if share is None and len(self.host_seqs) > 2:   # draw the host sequences' caches in parallel
            with cf.ThreadPoolExecutor(min(HOST_THREADS, 8)) as ex:
                list(ex.map(lambda b: (self.h_kv(b), self.h_ki(b)), self.host_seqs))
        for b in (range(B) if share is None else ()):
            Tb = self.T[b]
            pre = Tb - 1 if self.append else Tb
            if b in self.host_seqs:
                kv = bf16_dev(self.h_kv(b))
                ki = bf16_dev(self.h_ki(b))
            else:
                kv = syn.device_normal_bf16((cap, D), seed, syn.T_KV * 1000 + b)
                ki = syn.device_normal_bf16((cap, DI), seed, syn.T_KI * 1000 + b)
            if pre > 0:
                c.csa2_fp4_quantize_append(kv[:pre].unsqueeze(0).contiguous(), self.codes[b:b + 1], self.scales[b:b + 1])
                self.KI[b, :pre].copy_(ki[:pre])
            if self.append:
                self.kv_new[b, 0].copy_(kv[Tb - 1])
                self.ki_new[b, 0].copy_(ki[Tb - 1])
            del kv, ki
        if self.append:   # garbage where the step must write
            for b in range(B):
                self.codes[b, self.T[b] - 1].fill_(0xFF)
                self.scales[b, self.T[b] - 1].fill_(0x7E)
                self.KI[b, self.T[b] - 1].fill_(7.0)
        self.block_keys = None
        if share is not None and hierarchical:
            self.block_keys, self.pool, self.pool_len = share.block_keys, share.pool, share.pool_len
        elif hierarchical:
            self.block_keys = torch.zeros((B, cap // 8, DI), dtype=torch.bfloat16, device=dev)
            pre_lens = self.lens - (1 if self.append else 0)
            c.csa2_block_keys_build(self.KI, pre_lens.contiguous(), self.block_keys)
            self.pool = torch.full((B * Nq, keep * 8), -7, dtype=torch.int32, device=dev)
            self.pool_len = torch.zeros(B * Nq, dtype=torch.int32, device=dev)
        else:
            self.pool = self.pool_len = None
        self.out = [torch.zeros((B, Nq, H, D), dtype=torch.bfloat16, device=dev) for _ in range(L)]
        self.lse = [torch.zeros((B, Nq, H), dtype=torch.float32, device=dev) for _ in range(L)]
        self.idx = [torch.full((B * Nq, K), -9, dtype=torch.int32, device=dev) for _ in range(L)]
        self.qp_dev = to_dev(np.asarray(q_pos, np.int32)) if q_pos is not None else None
        self.ws = torch.empty(c.group_workspace_size(B, Nq, cap, K, W, hierarchical, keep), dtype=torch.uint8,
                              device=dev)

    # host draws, one sequence at a time (cache rows are kept once drawn) ----------------------
    def h_kv(self, b):
        cache = self.__dict__.setdefault("_kv", {})
        if b not in cache:
            cache[b] = syn.normal_bf16(self.seed, syn.T_KV, b, (self.cap, D))
        return cache[b]

    def h_ki(self, b):
        cache = self.__dict__.setdefault("_ki", {})
        if b not in cache:
            cache[b] = (syn.integer_bf16(self.seed, syn.T_KI, b, (self.cap, DI), -8, 8) if self.integer_index
                        else syn.normal_bf16(self.seed, syn.T_KI, b, (self.cap, DI)))
        return cache[b]

    def h_q(self, l, b): return syn.normal_bf16(self.seed, syn.T_Q + self.layer0 + l, b, (self.Nq, H, D))

    def h_qI(self, l, b):
        tid = syn.T_QI + self.layer0 + l
        if self.integer_index:
            return syn.integer_bf16(self.seed, tid, b, (self.Nq, HI, DI), -8, 8)
        return syn.normal_bf16(self.seed, tid, b, (self.Nq, HI, DI))

    def h_w(self, l, b):
        tid = syn.T_W + self.layer0 + l
        if self.integer_index:
            return syn.bf16_bits_to_f32(syn.integer_bf16(self.seed, tid, b, (self.Nq, HI), -4, 4))
        return syn.normal_f32(self.seed, tid, b, (self.Nq, HI))
    def h_swa(self, l, b):
        return syn.normal_bf16(self.seed, syn.T_SWA + self.layer0 + l, b, (self.W - 1 + self.Nq, D))

    def h_win(self, l, b):
        """Window rows as the step reads them: bf16 bits, or the oracle's E4M3 bytes."""
        if not self.swa_fp8:
            return self.h_swa(l, b)
        import oracle
        oracle.build()
        return oracle.fp8_quantize(self.h_swa(l, b))

    def _dev_win(self, host_bf16):
        if not self.swa_fp8:
            return bf16_dev(host_bf16)
        import oracle
        oracle.build()
        return to_dev(oracle.fp8_quantize(host_bf16))

    def _dev_win_device(self, dev_bf16):
        if not self.swa_fp8:
            return dev_bf16
        import torch
        out = torch.empty(dev_bf16.shape, dtype=torch.uint8, device=dev_bf16.device)
        self.c.csa2_fp8_quantize(dev_bf16, out)
        return out

    def desc(self, events=None, n_split=0, seq_chunks=0):
        c = self.c
        return c.make_group_desc(
            self.modes, B=self.B, Nq=self.Nq, cap=self.cap, lens=self.lens, codes=self.codes, scales=self.scales,
            KI=self.KI, q=self.q, qI=self.qI, w=self.w, swa=self.swa, swa_len=self.swa_len, out=self.out,
            idx=self.idx, K=self.K, W=self.W, ratio=self.ratio, hierarchical=self.hierarchical, keep=self.keep,
            n_split=n_split, q_pos=self.qp_dev, block_keys=self.block_keys, pool=self.pool,
            pool_len=self.pool_len, kv_new=self.kv_new if self.append else None,
            ki_new=self.ki_new if self.append else None, lse=self.lse, events=events, seq_chunks=seq_chunks,
            swa_fp8=self.swa_fp8)

    def run(self, n_split=0, seq_chunks=0):
        import torch
        d = self.desc(n_split=n_split, seq_chunks=seq_chunks)
        self.c.csa2_group_step(d, self.ws)
        torch.cuda.synchronize()

    def oracle(self, orc, seqs=None, threads=HOST_THREADS):
        """Oracle of the sequences `seqs` (host draws only)."""
        return stack_oracle(orc, [self], seqs, threads)

    def check(self, orc, seqs=None, threads=HOST_THREADS):
        """Compare the device results of `seqs` with the oracle: bit-exact indices (and pools),
        attention outputs within the tolerance, lse within 1e-2 absolute."""
        return check_stack(orc, [self], seqs, threads)


def stack_oracle(orc, groups, seqs=None, threads=HOST_THREADS):
    """The oracle of the groups of a decoder stack, run in order on the first group's cache: one
    group step over all their layers (a Reindex layer rescores the latest Full layer's pool)."""
    g0 = groups[0]
    seqs = g0.host_seqs if seqs is None else seqs
    Nq = g0.Nq
    Ts = [g0.T[b] for b in seqs]
    cap = max(Ts)
    codes = np.zeros((len(seqs), cap, 256), np.uint8)
    scales = np.zeros((len(seqs), cap, 32), np.uint8)
    KI = np.zeros((len(seqs), cap, DI), np.uint16)
    for i, b in enumerate(seqs):
        kv = g0.h_kv(b)[:g0.T[b]]
        codes[i, :g0.T[b]], scales[i, :g0.T[b]] = orc.fp4_quantize(kv, threads=threads)
        KI[i, :g0.T[b]] = g0.h_ki(b)[:g0.T[b]]
    layers = [(g, l) for g in groups for l in range(g.L)]
    modes = [g.modes[l] for g, l in layers]
    q = np.stack([np.stack([g.h_q(l, b) for b in seqs]) for g, l in layers])
    qI = np.stack([np.stack([g.h_qI(l, b) for b in seqs]) for g, l in layers])
    w = np.stack([np.stack([g.h_w(l, b) for b in seqs]) for g, l in layers])
    swa = np.stack([np.stack([g.h_win(l, b) for b in seqs]) for g, l in layers])
    qp = None if g0.q_pos is None else np.asarray(g0.q_pos, np.int32).reshape(g0.B, Nq)[seqs]
    return orc.group_step(modes, Ts, codes, scales, KI, q, qI, w, swa, g0.swa_len_np[seqs],
                          Nq=Nq, K=g0.K, W=g0.W, ratio=g0.ratio, hierarchical=g0.hierarchical,
                          keep=g0.keep, q_pos=qp, softmax_scale=SCALE, threads=threads, swa_fp8=g0.swa_fp8)


def check_stack(orc, groups, seqs=None, threads=HOST_THREADS):
    """Compare the device results of the groups of a stack (run in order) for the sequences `seqs`
    with stack_oracle: bit-exact indices (and pools), attention outputs within the tolerance, lse
    within 1e-2 absolute."""
    g0 = groups[0]
    seqs = g0.host_seqs if seqs is None else seqs
    ref = stack_oracle(orc, groups, seqs, threads)
    Nq = g0.Nq
    rows = np.concatenate([np.arange(b * Nq, (b + 1) * Nq) for b in seqs])
    layers = [(g, l) for g in groups for l in range(g.L)]
    for j, (g, l) in enumerate(layers):
        gi = g.idx[l].cpu().numpy()[rows].reshape(len(seqs), Nq, g.K)
        assert np.array_equal(gi, ref["idx"][j]), f"layer {j}: indices differ"
        out = bf16_host(g.out[l])[seqs]
        assert_attn_close(out, ref["out"][j], f"layer {j} out")
        lse = g.lse[l].cpu().numpy()[seqs]
        fin = np.isfinite(ref["lse"][j])
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.all(np.abs(lse[fin] - ref["lse"][j][fin]) <= 1e-2), f"layer {j} lse"
    if g0.hierarchical:
        gp = g0.pool.cpu().numpy()[rows]
        gl = g0.pool_len.cpu().numpy()[rows]
        assert np.array_equal(gl, ref["pool_len"].reshape(-1))
        for i in range(len(rows)):
            n = gl[i]
            assert np.array_equal(gp[i, :n], ref["pool"].reshape(len(rows), -1)[i, :n])
    return ref

