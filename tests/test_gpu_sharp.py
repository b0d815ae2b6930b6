"""GPU parity on peaked attention: planted "needle" keys aligned with a query.

The random caches of the other parity tests give near-uniform attention (a
spread of log2-logits of about 3 to 5), where a score error barely moves the
weights. Here every stream gets keys whose score against the first query head
of their kv head is tens of nats above the rest, so that:
  * a split's running maximum jumps by more than 2^64 after its frame is set
    (the kernel moves its shared sums to the new frame),
  * the combine merges splits whose maxima differ by more than 64 in log2,
  * two needles of close scores in distant splits share the weight, so the
    score precision shows in the output.
Needles sit in the first block, inside splits, in the fp16 tail and at the
last position; the cases cover INT4 with outliers at sm_scale 1 and 4, INT2
with 128-token key blocks, MHA without outliers, the paged path, the fused
decode step and one layer of the 1M-token workload. Every case asserts from
the oracle's own logits that the spread exceeds 64 (log2 units).

Logits of tens of nats need more score precision than fp16 operands give, so
every case runs with the precise-score flag (KVQ_FLAG_PRECISE_SCORES: fp32
key arithmetic, hi + lo fp16 operands) and is compared at the decode
tolerance (2e-3 max-abs, 1e-2 relative). The default fp16-operand path runs
the same cases against the bound its arithmetic gives (fast_path_bound).
"""
import math

import numpy as np
import pytest
import torch

import bit_quantized_kv_append_gb300 as kvq
from bit_quantized_kv_append_gb300 import build as kbuild
import kvq_inputs as ki
import kvq_testlib as tl
from oracle import oracle_cpp as oc
from oracle import oracle_np as on

pytestmark = pytest.mark.gpu
W = ki.Workload
LOG2E = 1.4426950408889634


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    kbuild.build()
    kvq.lib()


def _needle_key(q_head, q_pos, t, nats, sm_scale, theta):
    """Pre-RoPE key at position t whose score against q_head (at q_pos) is
    `nats`: c * R(q_pos - t) q, since <R(q_pos) q, R(t) R(q_pos - t) q> = |q|^2."""
    qd = q_head.astype(np.float64)
    c = nats / (sm_scale * float(qd @ qd))
    k = qd if theta == 0 else on.rope(qd, q_pos - t, theta)
    return (c * k).astype(np.float16)


def _plant(w, K, qn, q_pos, needles, sm_scale):
    """needles: {stream index p: [(t, nats), ...]} for head h_kv * G of stream p."""
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    for p, lst in needles.items():
        b, h = streams[p]
        for t, nats in lst:
            K[p, t] = _needle_key(qn[b, h * w.G], q_pos, t, nats, sm_scale, w.rope_theta)
    return streams


def _logit_spread(w, enc, T, qn, streams, q_pos, sm_scale):
    """log2-logit spread (max - min over t) of the first head of every stream,
    from the oracle's dequantized cache."""
    Kh, _ = oc.dequant(enc, T, w.D, w.bits, w.key_block, w.value_group, tl.n_out_of(w))
    out = []
    for p, (b, h) in enumerate(streams):
        qd = qn[b, h * w.G].astype(np.float64)
        if w.rope_theta > 0:
            kr = on.rope(Kh[p], np.arange(T, dtype=np.float64), w.rope_theta)
            qr = on.rope(qd, q_pos, w.rope_theta)
        else:
            kr, qr = Kh[p], qd
        lg = sm_scale * (kr @ qr) * LOG2E
        out.append((float(lg.max() - lg.min()), lg))
    return out


def fast_path_bound(w, enc, T, qn, streams, q_pos, sm_scale, v_max):
    """Output error bound of the fp16-operand scores. Each operand is rounded
    to fp16 (relative 2^-11): q, the dequantized key, and the two products of
    the rotation, so a token's score (nats) is off by at most
    delta_t = 4 * 2^-11 * sm_scale * sum_c |q_c| (|x_c| + |x_c'|), c' the
    rotation partner of channel c. Scores off by at most delta move the
    normalized weights by a factor within exp(+-2 delta); with the fp16
    rounding of p * s and of the output this bounds |out - ref| by
    2e-3 + 2 (exp(2 delta) - 1) max|v| + 2^-10 max|v|."""
    Kh, _ = oc.dequant(enc, T, w.D, w.bits, w.key_block, w.value_group, tl.n_out_of(w))
    H = w.D // 2
    delta = 0.0
    for p, (b, h) in enumerate(streams):
        x = np.abs(Kh[p])
        xx = x + np.concatenate([x[:, H:], x[:, :H]], axis=1)
        qabs = np.abs(qn[b, h * w.G:(h + 1) * w.G].astype(np.float64))         # |q| is rotation-invariant per pair
        qpair = np.sqrt(qabs[:, :H] ** 2 + qabs[:, H:] ** 2)
        qq = np.concatenate([qpair, qpair], axis=1)
        delta = max(delta, float((qq @ xx.T).max()) * 4 * 2.0 ** -11 * sm_scale)
    return 2e-3 + 2 * math.expm1(2 * delta) * v_max + 2.0 ** -10 * v_max


def _needles_for(w, T, P, strong=60.0, pair=False):
    """Per stream: a needle in block 1..7 at a stream-dependent offset (so that
    across streams it falls at many offsets inside a split), a second one in the
    last third (pair: 0.7 nats weaker, else 30 nats weaker), one in the fp16 tail
    for some streams and one at the last position for others."""
    Bk = w.key_block
    nd = {}
    n_full = T // Bk
    for p in range(P):
        t1 = Bk * (1 + p % min(7, max(1, n_full - 1))) + (13 * p) % Bk
        t2 = (2 * T) // 3 + (29 * p) % (T // 4)
        lst = [(min(t1, T - 1), strong), (min(t2, T - 1), strong - (0.7 if pair else 30.0))]
        if p % 3 == 1 and T % Bk:
            lst.append((n_full * Bk + (p % (T % Bk)), strong - 20.0))
        if p % 3 == 2:
            lst.append((T - 1, strong - 15.0))
        nd[p] = lst
    return nd


CASES = {
    # name: (workload, T, sm_scale, pair)
    "gqa_int4_outliers_s1": (W("sharp4", 4, 32, 8, 128, 4096 + 37, 4, 64, 64, 0.01, 5e5, 51), 1.0, False),
    "gqa_int4_outliers_s4_pair": (W("sharp4p", 4, 32, 8, 128, 4096 + 37, 4, 64, 64, 0.01, 5e5, 52), 4.0, True),
    "int2_bk128_gv32": (W("sharp2", 4, 32, 8, 128, 8192 + 77, 2, 128, 32, 0.01, 5e5, 53), 1.0, True),
    "int3_bk128_gv32": (W("sharp3", 2, 16, 8, 128, 8192 + 5, 3, 128, 32, 0.01, 5e5, 54), 4.0, False),
    "mha_g1_no_outliers": (W("sharpg1", 4, 16, 16, 128, 4096 + 11, 4, 64, 64, 0.0, 1e4, 55), 1.0, True),
}


def _cache(w, T_max, precise):
    return kvq.QuantizedKVCache(w.B, w.H_kv, w.D, T_max, w.bits, w.key_block, w.value_group, w.outlier_frac,
                                H_q=w.H_q, rope_theta=w.rope_theta, device="cuda", precise=precise)


def _check(precise, got, ref, what, bound):
    if precise:
        return tl.check_decode(got, ref, what)
    err = float(np.abs(got.astype(np.float64) - ref).max())
    assert err <= bound, f"{what} (fp16 scores): max abs error {err:.3g} above its bound {bound:.3g}"
    return err, None


@pytest.mark.parametrize("precise", [True, False], ids=["precise", "fp16"])
@pytest.mark.parametrize("name", list(CASES))
def test_sharp_attention(name, precise):
    w, sm_scale, pair = CASES[name]
    T = w.T
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    K, V = tl.host_streams(w, streams, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    qn = q.cpu().numpy()
    q_pos = T - 1
    _plant(w, K, qn, q_pos, _needles_for(w, T, len(streams), pair=pair), sm_scale)
    enc = tl.oracle_encode(w, K, V)
    spreads = _logit_spread(w, enc, T, qn, streams, q_pos, sm_scale)
    assert min(s for s, _ in spreads) > 64.0, "the planted needles must give a log2-logit spread above 64"
    cache = _cache(w, (T // w.key_block + 1) * w.key_block, precise)
    Kd = torch.from_numpy(K.reshape(w.B, w.H_kv, T, w.D)).cuda()
    Vd = torch.from_numpy(V.reshape(w.B, w.H_kv, T, w.D)).cuda()
    tl.append_pieces(cache, Kd, Vd, [T - 300, 299, 1])
    tl.sync()
    tl.compare_streams(cache, streams, enc, T)
    out = cache.decode(q, q_pos=q_pos, sm_scale=sm_scale).cpu().numpy()
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(qn, w, streams), q_pos, sm_scale=sm_scale)
    bound = 0.0 if precise else fast_path_bound(w, enc, T, qn, streams, q_pos, sm_scale, float(np.abs(V).max()))
    _check(precise, tl.q_of_streams(out, w, streams), ref, name, bound)


@pytest.mark.parametrize("precise", [True, False], ids=["precise", "fp16"])
def test_sharp_fused_step(precise):
    """The appended token is the needle: kvq_decode_step attends the new query
    at its own position, where its key scores 60 nats above the rest."""
    w = W("sharpstep", 4, 32, 8, 128, 2048 + 20, 4, 64, 64, 0.01, 5e5, 56)
    T, sm_scale = w.T, 1.0
    streams = [(b, h) for b in range(w.B) for h in range(w.H_kv)]
    K, V = tl.host_streams(w, streams, T)
    q = ki.queries_torch(w, 0, 0, "cuda")
    qn = q.cpu().numpy()
    nd = {p: [(T - 1, 60.0), (64 * (1 + p % 5) + 7, 59.5)] for p in range(len(streams))}
    _plant(w, K, qn, T - 1, nd, sm_scale)
    enc = tl.oracle_encode(w, K, V)
    assert min(s for s, _ in _logit_spread(w, enc, T, qn, streams, T - 1, sm_scale)) > 64.0
    cache = _cache(w, (T // w.key_block + 1) * w.key_block, precise)
    Kd = torch.from_numpy(K.reshape(w.B, w.H_kv, T, w.D)).cuda()
    Vd = torch.from_numpy(V.reshape(w.B, w.H_kv, T, w.D)).cuda()
    cache.append(Kd[:, :, :T - 1].contiguous(), Vd[:, :, :T - 1].contiguous())
    out = cache.decode_step(Kd[:, :, T - 1:].contiguous(), Vd[:, :, T - 1:].contiguous(), q,
                            sm_scale=sm_scale).cpu().numpy()
    tl.sync()
    tl.compare_streams(cache, streams, enc, T)
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(qn, w, streams), T - 1, sm_scale=sm_scale)
    bound = 0.0 if precise else fast_path_bound(w, enc, T, qn, streams, T - 1, sm_scale, float(np.abs(V).max()))
    _check(precise, tl.q_of_streams(out, w, streams), ref, "fused step", bound)


@pytest.mark.parametrize("precise", [True, False], ids=["precise", "fp16"])
def test_sharp_paged(precise):
    """Paged, ragged batch with needles in every sequence (shuffled block table)."""
    w = W("sharppg", 4, 32, 8, 128, 0, 4, 64, 64, 0.01, 5e5, 57)
    sm_scale = 1.0
    lens = [3000, 2111, 1500, 777]
    Bk = w.key_block
    T_max = (max(lens) // Bk + 1) * Bk
    per_seq = T_max // Bk
    n_blocks = w.B * per_seq + 3
    cache = kvq.PagedKVCache(w.B, w.H_kv, w.D, T_max, n_blocks, w.bits, Bk, w.value_group, w.outlier_frac,
                             H_q=w.H_q, rope_theta=w.rope_theta, precise=precise)
    perm = np.random.default_rng(w.seed).permutation(n_blocks)[:w.B * per_seq].reshape(w.B, per_seq)
    cache.block_table.copy_(torch.from_numpy(perm.astype(np.int32)))
    q = ki.queries_torch(w, 0, 0, "cuda")
    qn = q.cpu().numpy()
    refs, bounds = {}, {}
    for b, n in enumerate(lens):
        ss = [(b, h) for h in range(w.H_kv)]
        K, V = ki.streams_np(w.replace(T=n), ss, n)
        for h in range(w.H_kv):
            for t, nats in [(Bk * (1 + (b + h) % 5) + 3 * h, 60.0), (n - 1 - 5 * h, 59.4)]:
                K[h, t] = _needle_key(qn[b, h * w.G], n - 1, t, nats, sm_scale, w.rope_theta)
        cache.append_seq(b, torch.from_numpy(K[None]).cuda(), torch.from_numpy(V[None]).cuda())
        enc = tl.oracle_encode(w, K, V)
        spreads = _logit_spread(w, enc, n, qn[b:b + 1], [(0, h) for h in range(w.H_kv)], n - 1, sm_scale)
        assert min(s for s, _ in spreads) > 64.0
        refs[b] = tl.oracle_decode(w, enc, n, tl.q_of_streams(qn, w, ss), n - 1, sm_scale=sm_scale)
        bounds[b] = 0.0 if precise else fast_path_bound(w, enc, n, qn[b:b + 1], [(0, h) for h in range(w.H_kv)],
                                                        n - 1, sm_scale, float(np.abs(V).max()))
    out = cache.decode(q, sm_scale=sm_scale).cpu().numpy()
    for b in range(w.B):
        got = tl.q_of_streams(out, w, [(b, h) for h in range(w.H_kv)])
        _check(precise, got, refs[b], f"paged sequence {b}", bounds[b])


@pytest.mark.parametrize("precise", [True, False], ids=["precise", "fp16"])
def test_sharp_long_context_layer(precise):
    """One layer of the 1M-token workload: needles 2^19 tokens apart, the far one
    at a RoPE distance of about 10^6 positions."""
    w = ki.WORKLOADS["long1m"]
    T, layer, sm_scale = w.T, 9, 1.0
    streams = [(0, h) for h in range(w.H_kv)]
    q = ki.queries_torch(w, layer, 0, "cuda")
    qn = q.cpu().numpy()
    cache = _cache(w, T + w.key_block, precise)
    p_s = 3                                    # the stream checked against the oracle
    needles = [(1000, 60.0), ((1 << 19) + 17, 59.6), (T - 1, 45.0)]
    t0 = 0
    for chunk in (1 << 18,) * 4:
        K, V = ki.kv_torch(w, layer, t0, chunk, "cuda")
        for t, nats in needles:
            if t0 <= t < t0 + chunk:
                K[0, p_s, t - t0] = torch.from_numpy(_needle_key(qn[0, p_s * w.G], T - 1, t, nats, sm_scale,
                                                                 w.rope_theta)).cuda()
        cache.append(K, V)
        t0 += chunk
        del K, V
    out = cache.decode(q, sm_scale=sm_scale).cpu().numpy()
    Kh, Vh = tl.host_streams(w, [(0, p_s)], T, layer=layer)
    for t, nats in needles:
        Kh[0, t] = _needle_key(qn[0, p_s * w.G], T - 1, t, nats, sm_scale, w.rope_theta)
    enc = tl.oracle_encode(w, Kh, Vh)
    tl.compare_streams(cache, [(0, p_s)], enc, T)
    spread = _logit_spread(w, enc, T, qn, [(0, p_s)], T - 1, sm_scale)[0][0]
    assert spread > 64.0
    ref = tl.oracle_decode(w, enc, T, tl.q_of_streams(qn, w, [(0, p_s)]), T - 1, sm_scale=sm_scale)
    bound = 0.0 if precise else fast_path_bound(w, enc, T, qn, [(0, p_s)], T - 1, sm_scale, float(np.abs(Vh).max()))
    _check(precise, tl.q_of_streams(out, w, [(0, p_s)]), ref, "long1m needles", bound)
