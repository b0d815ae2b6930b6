"""GPU parity of the paged, ragged batch path (kvq_paged_append,
kvq_paged_decode_attn): sequences of different lengths share pools of
physical key blocks through a shuffled block table.

Every sequence's blocks, gathered through the table, must equal the oracle's
encoding of that sequence's tokens bit for bit; every sequence's output must be
within the decode tolerance of the oracle's float64 attention over its own
tokens, its query at its newest token. Prefills go one sequence at a time (a
one-sequence view), then decode steps append one token to every sequence at
its own position; a sequence without tokens must give zeros.
"""
import numpy as np
import pytest
import torch

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
import kvq_inputs as ki
import kvq_testlib as tl

pytestmark = pytest.mark.gpu

W = ki.Workload
CASES = {
    # name: (workload with B sequences, prefill lengths, prefill pieces per sequence, decode steps)
    "gqa_int4_outliers": (W("pg4", 3, 8, 2, 128, 0, 4, 64, 64, 0.01, 5e5, 31), [200, 64, 1], 2, 3),
    "int3_bk128_gv32": (W("pg3", 3, 8, 2, 128, 0, 3, 128, 32, 0.01, 5e5, 32), [130, 300, 127], 3, 2),
    "mha_int4_rope": (W("pgm", 2, 4, 4, 128, 0, 4, 64, 64, 0.0, 1e4, 33), [65, 190], 1, 2),
    "d64_int2_g2": (W("pg64", 3, 4, 2, 64, 0, 2, 64, 32, 0.04, 1e4, 34), [70, 5, 128], 2, 2),
    "with_empty_sequence": (W("pge", 3, 8, 2, 128, 0, 4, 64, 64, 0.01, 5e5, 35), [100, 0, 40], 1, 0),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


def _gather(cache, b, h, T):
    """Sequence b, head h of the pools in logical order, shaped like the
    contiguous cache's per-stream views (first T tokens)."""
    v = {k: t.cpu().numpy() for k, t in cache.views().items()}
    Bk = cache.cfg.key_block
    table = cache.block_table[b].cpu().numpy()
    nbk = -(-T // Bk)
    nb = T // Bk
    blocks = [int(table[j]) for j in range(nbk)]
    cat = lambda name: (np.concatenate([v[name][p, h] for p in blocks])[:T] if blocks else v[name][0, h][:0])
    out = {"v_codes": cat("v_codes"), "v_meta": cat("v_meta"), "k_codes": cat("k_codes")[:nb * Bk],
           "k_meta": (np.stack([v["k_meta"][p, h] for p in blocks[:nb]]) if nb else v["k_meta"][0:0, h]),
           "k_tail": v["k_tail"][b, h, :T - nb * Bk]}
    if cache.n_out:
        out["v_outl"] = cat("v_outl")
        out["k_outl"] = cat("k_outl")[:nb * Bk]
    return out


def _compare(cache, b, w, enc, T):
    Bk = w.key_block
    nb = T // Bk
    for h in range(w.H_kv):
        got = _gather(cache, b, h, T)
        want = {"v_codes": enc["v_codes"][h], "v_meta": enc["v_meta"][h],
                "k_codes": enc["k_codes"][h, :nb * Bk], "k_meta": enc["k_meta"][h],
                "k_tail": enc["k_tail"][h, :T - nb * Bk]}
        if cache.n_out:
            want["v_outl"] = enc["v_outl"][h]
            want["k_outl"] = enc["k_outl"][h, :nb * Bk]
        for name, g in got.items():
            gb = np.ascontiguousarray(g).view(np.uint8)
            ob = np.ascontiguousarray(want[name]).view(np.uint8)
            assert gb.shape == ob.shape and np.array_equal(gb, ob), f"{name} differs: sequence {b}, head {h}"


@pytest.mark.parametrize("name", list(CASES))
def test_paged_ragged_parity(name):
    w, lens, pieces, steps = CASES[name]
    Bk = w.key_block
    T_max = (max(lens) + steps) // Bk * Bk + Bk
    per_seq = T_max // Bk
    n_blocks = w.B * per_seq + 3                     # a few blocks never used
    cache = kvq.PagedKVCache(w.B, w.H_kv, w.D, T_max, n_blocks, w.bits, Bk, w.value_group, w.outlier_frac,
                             H_q=w.H_q, rope_theta=w.rope_theta)
    rng = np.random.default_rng(w.seed)
    perm = rng.permutation(n_blocks)[:w.B * per_seq].reshape(w.B, per_seq)
    cache.block_table.copy_(torch.from_numpy(perm.astype(np.int32)))
    T_all = max(lens) + steps
    K, V = ki.kv_torch(w.replace(T=T_all), 0, 0, T_all, "cuda")      # [B, H_kv, T_all, D]
    # prefill: one sequence at a time, in pieces
    for b, L in enumerate(lens):
        cuts = np.linspace(0, L, pieces + 1).astype(int)
        for t0, t1 in zip(cuts[:-1], cuts[1:]):
            if t1 > t0:
                cache.append_seq(b, K[b:b + 1, :, t0:t1].contiguous(), V[b:b + 1, :, t0:t1].contiguous())
    assert cache.lengths == lens
    assert cache.seq_len.cpu().tolist() == lens
    cur = list(lens)
    for s in range(steps + 1):
        if s > 0:                                     # one token for every sequence, at its own position
            idx = torch.tensor(cur, device="cuda").view(-1, 1, 1, 1).expand(-1, w.H_kv, 1, w.D)
            cache.append(torch.gather(K, 2, idx).contiguous(), torch.gather(V, 2, idx).contiguous())
            cur = [t + 1 for t in cur]
            assert cache.seq_len.cpu().tolist() == cur
        q = ki.queries_torch(w, 0, s, "cuda")
        out = cache.decode(q).cpu().numpy()
        tl.sync()
        qn = q.cpu().numpy()
        for b, T in enumerate(cur):
            if T == 0:
                assert not out[b].any(), "a sequence without tokens must give zeros"
                continue
            streams = [(b, h) for h in range(w.H_kv)]
            Kh, Vh = tl.host_streams(w.replace(T=T_all), streams, T)
            enc = tl.oracle_encode(w, Kh, Vh)
            _compare(cache, b, w, enc, T)
            ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(qn, w, streams), T - 1)
            tl.check_decode(tl.q_of_streams(out, w, streams), ref, f"{name} step {s} sequence {b}")
