"""Pins of the CPU oracle to facts it does not produce itself.

Each test checks the oracle against a closed form, a hand-worked example
(tests/golden/hand_examples.json), a library routine the step reduces to, an
invariant, or brute force on tiny inputs.  ``tests/test_oracle_mutations.py``
plants plausible mistakes in the oracle and checks that these pins catch
each one, so the functions here must reach the oracle through the module
attribute ``O`` (which the mutation harness patches).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import csa_synth
from oracle import csa_oracle as O
from tests._common import f64, oracle_comp, oracle_layer, oracle_state, rel_err_rows, step_tuple

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")))


def _tiny_layer(dtype="f32", ratio=4, **kw):
    base = dict(dtype=dtype, H=4, D=16, R=8, W=8, ratio=ratio, Hi=3, Di=8, topk=5, X=24)
    base.update(kw)
    return O.Layer(**base)


def _tiny_comp(layer, d, rng, gate_scale=1.0):
    L = layer.lanes
    return O.Compressor(
        wkv=O.store(rng.standard_normal((L * d, layer.X)) / math.sqrt(layer.X), layer.dtype),
        wgate=O.store(gate_scale * rng.standard_normal((L * d, layer.X)) / math.sqrt(layer.X), layer.dtype),
        ape=O.round_f32(rng.standard_normal((layer.ratio, L * d))),
        norm_w=O.round_f32(1.0 + 0.1 * rng.standard_normal(d)),
        d=d)


def _inv_freq(R, base=10000.0):
    return (base ** (-2.0 * np.arange(R // 2) / R)).astype(np.float32)


# --------------------------------------------------------------------------- storage rounding

def test_round_bf16_matches_torch_cast():
    """fp32 inputs: single rounding to bf16 equals torch's RNE cast (a library routine)."""
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.float32([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0, 1e-40, -3e-39])
                        ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = O.round_bf16(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_round_bf16_is_nearest_for_float64():
    """float64 inputs: the result is a bf16 value and no bf16 neighbour is closer."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal(5000) * 3.0
    r = O.round_bf16(x)
    assert np.array_equal(torch.from_numpy(r.astype(np.float32)).to(torch.bfloat16).double().numpy(), r)
    ulp = np.ldexp(1.0, np.frexp(r)[1] - 8)
    for cand in (r - ulp, r + ulp, r - ulp / 2, r + ulp / 2):
        c = torch.from_numpy(cand.astype(np.float32)).to(torch.bfloat16).double().numpy()
        assert np.all(np.abs(x - r) <= np.abs(x - c) + 1e-300)


# --------------------------------------------------------------------------- RoPE

def test_rope_hand_example():
    g = GOLDEN["rope_pair"]
    out = O.rope(np.array(g["v"]), g["p"], np.float32(g["inv_freq"]))
    assert np.allclose(out, g["expected"], rtol=0, atol=1e-15)
    back = O.rope(out, g["p"], np.float32(g["inv_freq"]), inverse=True)
    assert np.allclose(back, g["v"], rtol=0, atol=1e-15)


def test_rope_pairs_are_interleaved_on_last_dims():
    """Closed form per pair: dims (D-R+2i, D-R+2i+1) rotate by p*inv_freq[i]; others unchanged."""
    D, R, p = 12, 6, 3
    invf = np.float32([1.0, 0.25, 0.0625])
    rng = np.random.default_rng(3)
    v = rng.standard_normal(D)
    out = O.rope(v, p, invf)
    assert np.array_equal(out[:D - R], v[:D - R])
    for i in range(R // 2):
        th = p * float(invf[i])
        a, b = v[D - R + 2 * i], v[D - R + 2 * i + 1]
        assert out[D - R + 2 * i] == pytest.approx(a * math.cos(th) - b * math.sin(th), abs=1e-14)
        assert out[D - R + 2 * i + 1] == pytest.approx(a * math.sin(th) + b * math.cos(th), abs=1e-14)


def test_rope_preserves_norm_and_inverts():
    rng = np.random.default_rng(4)
    invf = _inv_freq(16)
    for p in (0, 1, 7, 1000, 65535):
        v = rng.standard_normal((5, 64))
        r = O.rope(v, p, invf)
        assert np.allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(v, axis=-1), rtol=1e-13)
        assert np.allclose(O.rope(r, p, invf, inverse=True), v, atol=1e-13)


def test_rope_dot_depends_only_on_relative_position():
    """RoPE(q,p).RoPE(k,t) = RoPE(q,p+s).RoPE(k,t+s); power-of-two frequencies keep fp32 angles exact."""
    rng = np.random.default_rng(5)
    invf = np.float32([2.0 ** -e for e in range(8)])
    q, k = rng.standard_normal(32), rng.standard_normal(32)
    base = O.rope(q, 9, invf) @ O.rope(k, 4, invf)
    for s in (1, 5, 100, 4096):
        assert O.rope(q, 9 + s, invf) @ O.rope(k, 4 + s, invf) == pytest.approx(base, abs=1e-9)


def test_rope_angle_is_fp32_product():
    """R8: theta is fp32(p) * fp32(inv_freq) rounded to fp32 (not the exact product)."""
    invf = np.float32([0.1234567])
    p = 70001
    th = O.rope_angles(p, invf)[0]
    assert th == float(np.float32(p) * invf[0])
    assert th != p * float(invf[0])
    out = O.rope(np.array([1.0, 0.0]), p, invf)
    assert out[0] == pytest.approx(math.cos(th), abs=1e-15)
    assert abs(out[0] - math.cos(p * float(invf[0]))) > 1e-5


# --------------------------------------------------------------------------- RMSNorm

def test_rms_norm_closed_forms():
    c, w, eps = 3.0, np.array([1.0, 2.0, -1.0, 0.5]), 1e-6
    y = O.rms_norm(np.full(4, c), w, eps)
    assert np.allclose(y, c / math.sqrt(c * c + eps) * w, rtol=1e-15)
    rng = np.random.default_rng(6)
    u = rng.standard_normal(64)
    y = O.rms_norm(u, np.ones(64), 0.0)
    assert np.mean(y * y) == pytest.approx(1.0, rel=1e-13)
    assert np.allclose(O.rms_norm(7.5 * u, np.ones(64), 0.0), y, rtol=1e-13)


# --------------------------------------------------------------------------- compressor

def test_pool_weights_sum_to_one():
    rng = np.random.default_rng(7)
    s = rng.standard_normal((8, 100)) * 5
    w = O.pool_weights(s)
    assert np.all(w > 0)
    assert np.allclose(w.sum(axis=0), 1.0, atol=1e-15)
    assert np.allclose(O.pool_weights(np.zeros((8, 3))), 1 / 8)
    ref = scipy.special.softmax(s, axis=0)
    assert np.allclose(w, ref, rtol=1e-13)


def test_compressor_hand_example_overlap_row():
    g = GOLDEN["compressor_overlap_row1"]
    layer = _tiny_layer(ratio=4)
    comp = O.Compressor(wkv=None, wgate=None, ape=np.zeros((4, 2)), norm_w=np.ones(1), d=1)
    tok = {}
    for t in range(4):
        tok[t] = (np.array([g["kv_lane0"][t], -99.0]), np.array([g["gate_lane0"][t], 50.0]))
    for t in range(4, 8):
        tok[t] = (np.array([-99.0, g["kv_lane1"][t - 4]]), np.array([50.0, g["gate_lane1"][t - 4]]))
    kv, s = O.window_entries(layer, comp, 1, tok)
    u = (O.pool_weights(s) * kv).sum(axis=0)
    assert u[0] == pytest.approx(g["expected_u"], rel=1e-14)


def test_projection_hand_example():
    """kv = Wkv x and g = Wgate x with weights stored [out, in], each rounded once to bf16 (a tie to even
    included): pins which weight feeds which output, the contraction axis and the storage rounding."""
    g = GOLDEN["projection"]
    layer = _tiny_layer(dtype="bf16", ratio=4, X=2)
    comp = O.Compressor(wkv=np.array(g["wkv"]), wgate=np.array(g["wgate"]), ape=np.zeros((4, 2)),
                        norm_w=np.ones(1), d=1)
    kv, gate = O.project(layer, comp, np.array(g["x"])[None])  # one sequence of two tokens
    assert kv.shape == gate.shape == (1, 2, 2)
    assert np.array_equal(kv[0], np.array(g["expected_kv_bf16"]))
    assert np.array_equal(gate[0], np.array(g["expected_gate_bf16"]))


def _entries_pooled(layer, comp, j, tok):
    kv, s = O.window_entries(layer, comp, j, tok)
    return (O.pool_weights(s) * kv).sum(axis=0)


@pytest.mark.parametrize("ratio", [4, 128])
def test_compressor_constant_and_mean(ratio):
    """All entries equal v -> pooled v; equal gates and zero APE -> arithmetic mean of the entries."""
    layer = _tiny_layer(ratio=ratio)
    L, d, r = layer.lanes, 6, ratio
    rng = np.random.default_rng(8)
    comp = O.Compressor(wkv=None, wgate=None, ape=rng.standard_normal((r, L * d)), norm_w=np.ones(d), d=d)
    v = rng.standard_normal(d)
    tok = {t: (np.tile(v, L), rng.standard_normal(L * d)) for t in range(3 * r)}
    for j in range(3):
        assert np.allclose(_entries_pooled(layer, comp, j, tok), v, rtol=1e-13)
    comp.ape[:] = 0.0
    tok = {t: (rng.standard_normal(L * d), np.full(L * d, 0.7)) for t in range(3 * r)}
    for j in range(3):
        got = _entries_pooled(layer, comp, j, tok)
        if L == 1:
            want = np.mean([tok[t][0] for t in range(j * r, (j + 1) * r)], axis=0)
        else:
            cur = [tok[t][0][d:] for t in range(j * r, (j + 1) * r)]
            prev = [tok[t][0][:d] for t in range((j - 1) * r, j * r)] if j > 0 else []
            want = np.mean(prev + cur, axis=0)
        assert np.allclose(got, want, rtol=1e-13)


def test_compressor_lane_and_ape_assignment():
    """R1: previous window through lane 0, current through lane 1, APE indexed by t mod ratio.

    One dominant gate selects exactly one entry: putting it on token t and lane
    l must return that token's lane-l kv."""
    layer = _tiny_layer(ratio=4)
    d, r = 3, 4
    comp = O.Compressor(wkv=None, wgate=None, ape=np.zeros((r, 2 * d)), norm_w=np.ones(d), d=d)
    kvs = {t: np.arange(2 * d) + 100.0 * t for t in range(8)}
    for t_hot, lane in [(0, 0), (2, 0), (3, 0), (4, 1), (7, 1)]:
        tok = {t: (kvs[t], np.full(2 * d, -40.0)) for t in range(8)}
        tok[t_hot][1][lane * d:(lane + 1) * d] = 40.0
        got = _entries_pooled(layer, comp, 1, tok)
        assert np.allclose(got, kvs[t_hot][lane * d:(lane + 1) * d], rtol=1e-12)
    # APE: a large APE on slot 2 selects token 4+2 of the current window (lane 1)
    comp.ape[2, d:] = 80.0
    tok = {t: (kvs[t], np.zeros(2 * d)) for t in range(8)}
    assert np.allclose(_entries_pooled(layer, comp, 1, tok), kvs[6][d:], rtol=1e-12)
    # ... and of the previous window on lane 0 when that lane's APE dominates instead
    comp.ape[:] = 0.0
    comp.ape[1, :d] = 80.0
    assert np.allclose(_entries_pooled(layer, comp, 1, tok), kvs[1][:d], rtol=1e-12)
    # row 0 has no previous window: only lane 1 of tokens 0..3 contributes
    comp.ape[:] = 0.0
    tok = {t: (kvs[t], np.zeros(2 * d)) for t in range(4)}
    assert np.allclose(_entries_pooled(layer, comp, 0, tok),
                       np.mean([kvs[t][d:] for t in range(4)], axis=0), rtol=1e-13)


@pytest.mark.parametrize("ratio", [4, 128])
def test_compress_streaming_is_chunking_invariant(ratio):
    """Token-by-token, one-shot and random chunkings give bit-identical state and rows;
    n_rows == floor(tokens / ratio) after every call; each row equals a from-scratch rebuild."""
    layer = _tiny_layer(ratio=ratio, X=16)
    d = 8
    rng = np.random.default_rng(9)
    comp = _tiny_comp(layer, d, rng)
    invf = _inv_freq(layer.R)
    T = 3 * ratio + 3
    x = O.store(rng.standard_normal((1, T, layer.X)), layer.dtype)
    F, cap = layer.frontier_slots, T // ratio + 2

    def run(splits):
        fr, pool, n = np.zeros((1, F, 2 * layer.lanes * d)), np.zeros((1, cap, d)), np.zeros(1, np.int64)
        p = 0
        for s in splits:
            fr, pool, n, err = O.compress_append(layer, comp, x[:, p:p + s], np.array([p]), fr, pool, n, invf)
            assert err == 0
            p += s
            assert n[0] == p // ratio
        return fr, pool, n

    one = run([T])
    for splits in ([1] * T, [ratio - 1, ratio + 2, T - 2 * ratio - 1], [5, 1, T - 6]):
        other = run(splits)
        for a, b in zip(one, other):
            assert np.array_equal(a, b)
    _, pool, n = one
    kv, g = O.project(layer, comp, x[0])
    tok = {t: (kv[t], g[t]) for t in range(T)}
    for j in range(int(n[0])):
        lo = max(0, (j - 1) * ratio) if layer.lanes == 2 else j * ratio
        only = {t: tok[t] for t in range(lo, (j + 1) * ratio)}
        assert np.array_equal(O.compressor_row(layer, comp, j, only, invf), pool[0, j])


def test_compressed_row_is_normed_and_roped_at_window_start():
    """finalize_row = RoPE(j*r) of RMSNorm(u); rotating back gives a row with unit RMS (w = 1)."""
    layer = _tiny_layer(ratio=4, dtype="f32")
    d = 16
    comp = O.Compressor(wkv=None, wgate=None, ape=None, norm_w=np.ones(d), d=d)
    invf = _inv_freq(layer.R)
    rng = np.random.default_rng(10)
    u = rng.standard_normal(d) * 4
    for j in (0, 1, 5):
        row = O.finalize_row(layer, comp, u, j, invf)
        unrot = O.rope(row, j * 4, invf, inverse=True)
        assert np.mean(unrot ** 2) == pytest.approx(1.0, rel=1e-5)
        assert np.allclose(unrot, u / np.sqrt(np.mean(u * u)), rtol=1e-5)


def test_compress_refuses_inconsistent_state_and_capacity():
    layer = _tiny_layer(ratio=4, X=16)
    rng = np.random.default_rng(11)
    comp = _tiny_comp(layer, 8, rng)
    invf = _inv_freq(layer.R)
    x = O.store(rng.standard_normal((2, 4, 16)), "f32")
    fr, pool = rng.standard_normal((2, 8, 32)), np.zeros((2, 3, 8))
    fr2, pool2, n2, err = O.compress_append(layer, comp, x, np.array([4, 8]), fr, pool, np.array([0, 2]), invf)
    assert err == O.ERR_STATE
    assert np.array_equal(fr2[0], fr[0]) and np.array_equal(pool2[0], pool[0]) and n2[0] == 0
    assert n2[1] == 3
    _, pool3, n3, err = O.compress_append(layer, comp, x, np.array([8, 8]), fr, pool, np.array([2, 2]), invf)
    assert err == 0
    _, _, n4, err = O.compress_append(layer, comp, x, np.array([12, 8]), fr, pool3, np.array([3, 2]), invf)
    assert err == O.ERR_CAPACITY and n4[0] == 3


# --------------------------------------------------------------------------- indexer / top-k

def test_indexer_hand_example():
    g = GOLDEN["indexer_scores"]
    layer = _tiny_layer(Hi=2, Di=2, R=2, topk=g["topk"])
    s = O.index_scores(layer, np.array(g["iq"]), np.array(g["iw"]), np.array(g["keys"]), 0, np.float32([1.0]))
    assert np.allclose(s, g["expected_scores"], rtol=1e-15)
    assert list(O.topk_select(s, g["topk"])) == g["expected_sel"]
    s = O.index_scores(layer, np.array(g["iq"]), np.array(g["iw_neg"]), np.array(g["keys"]), 0,
                       np.float32([1.0]))
    assert np.allclose(s, g["expected_scores_neg"], rtol=1e-15)
    assert list(O.topk_select(s, g["topk"])) == g["expected_sel_neg"]


def test_indexer_single_head_reduces_to_relu_dot():
    """Hi = 1 with iw = sqrt(Di): score_j = ReLU(RoPE(q,p) . key_j)."""
    Di = 16
    layer = _tiny_layer(Hi=1, Di=Di, R=8, dtype="f32")
    rng = np.random.default_rng(12)
    invf = _inv_freq(8)
    q, keys = rng.standard_normal((1, Di)), rng.standard_normal((30, Di))
    s = O.index_scores(layer, q, np.array([math.sqrt(Di)]), keys, 17, invf)
    want = np.maximum(O.round_f32(O.rope(q[0], 17, invf)) @ keys.T, 0.0)
    assert np.allclose(s, want, rtol=1e-12)
    assert np.all(s >= 0) and np.any(s == 0)


def test_topk_against_full_sort_brute_force():
    rng = np.random.default_rng(13)
    for trial in range(300):
        n = int(rng.integers(1, 40))
        k = int(rng.integers(1, 12))
        s = rng.integers(-3, 4, n).astype(np.float64)  # many exact ties
        want = sorted(sorted(range(n), key=lambda j: (-s[j], j))[:k])
        assert list(O.topk_select(s, k)) == want
    s = np.array([0.0, -0.0, 0.0, -1.0])
    assert list(O.topk_select(s, 2)) == [0, 1]


def test_visibility_hand_cases():
    g = GOLDEN["visibility"]
    layer = _tiny_layer(ratio=g["ratio"])
    for p, want in g["cases"]:
        assert O.visible_rows(layer, g["n"], p) == want
    # decode sees every row emitted up to and including its own token
    for p in range(64):
        n = (p + 1) // 4
        assert O.visible_rows(layer, n, p) == n


# --------------------------------------------------------------------------- attention

def test_attention_hand_example():
    g = GOLDEN["attention_with_sink"]
    layer = _tiny_layer(H=1, D=g["D"], scale=g["scale"])
    o = O.attend(layer, np.array(g["q"]), np.array(g["keys"]), np.array(g["sink"]))
    assert np.allclose(o, g["expected"], rtol=1e-14)


def test_attention_sink_limits():
    """Sink -inf: plain softmax (scipy); sink 0: o = o_plain * S / (S + 1), S = sum e^logit."""
    layer = _tiny_layer(H=3, D=16)
    rng = np.random.default_rng(14)
    q, keys = rng.standard_normal((3, 16)), rng.standard_normal((11, 16))
    logits = layer.softmax_scale * q @ keys.T
    plain = scipy.special.softmax(logits, axis=1) @ keys
    assert np.allclose(O.attend(layer, q, keys, np.full(3, -np.inf)), plain, rtol=1e-13)
    S = np.exp(logits).sum(axis=1)
    assert np.allclose(O.attend(layer, q, keys, np.zeros(3)), plain * (S / (S + 1))[:, None], rtol=1e-13)
    big = O.attend(layer, 200 * q, keys, np.zeros(3))  # logits in the hundreds: no overflow
    assert np.all(np.isfinite(big))


def test_split_merge_equals_unsplit():
    layer = _tiny_layer(H=4, D=16)
    rng = np.random.default_rng(15)
    q, keys, sink = rng.standard_normal((4, 16)), rng.standard_normal((37, 16)), rng.standard_normal(4)
    full = O.attend(layer, q, keys, sink)
    for trial in range(20):
        cuts = np.sort(rng.integers(0, 38, int(rng.integers(0, 6))))
        parts = np.split(np.arange(37), cuts)
        got = O.merge_partials([O.attend_partial(layer, q, keys[ix]) for ix in parts], sink)
        assert np.allclose(got, full, rtol=1e-12, atol=1e-14)


def test_topk_covering_all_rows_equals_dense_attention():
    """When topk >= visible rows, the indexer path equals attending every row (brute force)."""
    layer = _tiny_layer(H=4, D=16, R=8, W=8, topk=64, Hi=2, Di=8)
    rng = np.random.default_rng(16)
    invf = _inv_freq(8)
    B, cap, p = 1, 20, 60
    pool = O.round_f32(rng.standard_normal((B, cap, 16)))
    window = O.round_f32(rng.standard_normal((B, 8, 16)))
    q, kv, sink = rng.standard_normal((B, 4, 16)), rng.standard_normal((B, 16)), rng.standard_normal(4)
    n = np.array([15])
    sel, n_sel = O.index_topk(layer, rng.standard_normal((B, 2, 8)), rng.standard_normal((B, 2)),
                              rng.standard_normal((B, cap, 8)), n, np.array([p]), invf)
    assert n_sel[0] == 15
    a, w1, _ = O.attend_decode(layer, q, kv, sink, window, pool, n, sel, n_sel, np.array([p]), invf)
    b, _, _ = O.attend_decode(layer, q, kv, sink, window, pool, n, None, None, np.array([p]), invf)
    assert np.array_equal(a, b)
    # brute force: explicit key list, plain softmax with the sink column
    keys = list(pool[0, :15]) + [w1[0, t % 8] for t in range(p - 7, p + 1)]
    qr = O.round_f32(O.rope(q[0], p, invf))
    logits = layer.softmax_scale * qr @ np.array(keys).T
    full = np.concatenate([logits, sink[:, None]], axis=1)
    wts = scipy.special.softmax(full, axis=1)[:, :-1]
    o = O.round_f32(O.rope(O.round_f32(wts @ np.array(keys)), p, invf, inverse=True))
    assert np.allclose(a[0], o, rtol=1e-6, atol=1e-7)


def test_window_holds_the_last_W_tokens():
    """R4: the window is [p-W+1, p]; early on, ring slots of tokens that do not exist yet are ignored."""
    layer = _tiny_layer(W=8, D=16, R=8)
    invf = _inv_freq(8)
    assert list(O.window_tokens(layer, 3)) == [0, 1, 2, 3]
    assert list(O.window_tokens(layer, 20)) == list(range(13, 21))
    pool = np.zeros((1, 4, 16))
    q = np.zeros((1, 4, 16))
    kv = np.zeros((1, 16))
    for p, seen in ((3, False), (5, True)):
        w = np.zeros((1, 8, 16))
        w[0, 5] = 1.0  # token 5's slot; at p = 3 it holds stale data that must not be attended
        kv_p = kv if p != 5 else np.ones((1, 16))
        out, _, _ = O.attend_decode(layer, q, kv_p, np.full(4, -np.inf), w, pool, np.array([0]), None, None,
                                    np.array([p]), invf)
        assert (np.abs(out).max() > 0) == seen


# --------------------------------------------------------------------------- decode == prefill

def _decode_vs_prefill(ratio, T, ctx_tokens, topk):
    """Run a chunk token by token (decode path) and as one prefill chunk; compare."""
    cfg = csa_synth.CONFIGS[1].replace(ratio=ratio, topk=topk)
    layer = oracle_layer(cfg)
    ca, ci = oracle_comp(csa_synth.compressor(cfg, "attn")), None
    if cfg.has_indexer:
        ci = oracle_comp(csa_synth.compressor(cfg, "index"))
    invf = f64(csa_synth.inv_freq(cfg)).astype(np.float32)
    sink = f64(csa_synth.sinks(cfg))
    cap = (ctx_tokens + T) // ratio + 2
    st0 = oracle_state(csa_synth.empty_cache(cfg, cap, B=1))
    # build a context by decoding ctx_tokens of hidden states through the compressors only
    xs = f64(csa_synth.hidden(cfg, ctx_tokens, B=1))
    if ctx_tokens:
        st0["front_a"], st0["pool"], n, _ = O.compress_append(layer, ca, xs, st0["pos"], st0["front_a"],
                                                              st0["pool"], st0["n_rows"], invf)
        if ci is not None:
            st0["front_i"], st0["ikeys"], _, _ = O.compress_append(layer, ci, xs, st0["pos"], st0["front_i"],
                                                                   st0["ikeys"], st0["n_rows"], invf)
        st0["n_rows"] = n
        st0["pos"] = np.array([ctx_tokens])
        rng = np.random.default_rng(18)
        st0["window"] = O.round_f32(rng.standard_normal(st0["window"].shape))
    ch = csa_synth.chunk_inputs(cfg, T)
    x, q, kv, iq, iw = f64(ch.x), f64(ch.q), f64(ch.kv), f64(ch.iq), f64(ch.iw)
    # decode path
    st = {k: (v.copy() if v is not None else None) for k, v in st0.items()}
    outs, sels = [], []
    for i in range(T):
        out, sel, n_sel, err = O.decode_step(layer, ca, ci, st, (x[:, i:i + 1], q[i:i + 1], kv[i:i + 1],
                                             iq[i:i + 1], iw[i:i + 1]), sink, invf)
        assert err == 0
        outs.append(out[0])
        sels.append(None if sel is None else sel[0, :n_sel[0]])
    # prefill path
    pf = {k: (v.copy() if v is not None else None) for k, v in st0.items()}
    pf["front_a"], pf["pool"], n, _ = O.compress_append(layer, ca, x, pf["pos"], pf["front_a"], pf["pool"],
                                                        pf["n_rows"], invf)
    if ci is not None:
        pf["front_i"], pf["ikeys"], _, _ = O.compress_append(layer, ci, x, pf["pos"], pf["front_i"],
                                                             pf["ikeys"], pf["n_rows"], invf)
    out_p, sel_p, nsel_p, win_p = O.attend_prefill_chunk(layer, q, kv, iq, iw, sink, int(pf["pos"][0]),
                                                         pf["window"][0], pf["pool"][0], pf["ikeys"][0]
                                                         if ci is not None else None, int(n[0]), invf)
    assert np.array_equal(st["pool"], pf["pool"])
    assert np.array_equal(st["window"][0], win_p)
    assert rel_err_rows(np.stack(outs), out_p) <= 4e-6
    if cfg.has_indexer:
        for i in range(T):
            assert list(sels[i]) == list(sel_p[i, :nsel_p[i]])
    return np.stack(outs), out_p


def test_decode_equals_prefill_from_empty_cache():
    """Crosses window eviction (W = 32), 16 ratio-4 boundaries and the dense->sparse switch (topk 8)."""
    _decode_vs_prefill(ratio=4, T=70, ctx_tokens=0, topk=8)


def test_decode_equals_prefill_mid_sequence():
    _decode_vs_prefill(ratio=4, T=37, ctx_tokens=41, topk=6)


def test_decode_equals_prefill_ratio128():
    _decode_vs_prefill(ratio=128, T=140, ctx_tokens=130, topk=16)


# --------------------------------------------------------------------------- exact trim (R15)

def _rollback_setup(ratio, rollback, W=8, topk=5, seed=31):
    layer = _tiny_layer(ratio=ratio, W=W, topk=topk, rollback=rollback)
    rng = np.random.default_rng(seed)
    ca = _tiny_comp(layer, layer.D, rng)
    ci = _tiny_comp(layer, layer.Di, rng) if layer.has_indexer else None
    invf = _inv_freq(layer.R)
    sink = rng.standard_normal(layer.H)
    return layer, ca, ci, invf, sink, rng


def _empty_state(layer, cap, extra):
    """One sequence's empty state with `extra` rollback slots in every ring."""
    L = layer.lanes
    F = layer.frontier_slots + extra
    return dict(pool=np.zeros((1, cap, layer.D)), ikeys=np.zeros((1, cap, layer.Di)),
                window=np.zeros((1, layer.W + extra, layer.D)),
                front_a=np.zeros((1, F, 2 * L * layer.D)), front_i=np.zeros((1, F, 2 * L * layer.Di)),
                n_rows=np.zeros(1, dtype=np.int64), pos=np.zeros(1, dtype=np.int64))


def _tokens(layer, rng, n):
    return [(rng.standard_normal((1, 1, layer.X)), rng.standard_normal((1, layer.H, layer.D)),
             rng.standard_normal((1, layer.D)), rng.standard_normal((1, layer.Hi, layer.Di)),
             rng.standard_normal((1, layer.Hi))) for _ in range(n)]


def _decode(layer, ca, ci, st, tok, sink, invf):
    out, sel, n_sel, err = O.decode_step(layer, ca, ci, st, tok, sink, invf)
    assert err == 0
    return out, (None if sel is None else list(sel[0, :n_sel[0]]))


@pytest.mark.parametrize("ratio,n_true,drafts", [
    (4, 40, [(9, 3), (18, 4), (21, 2), (30, 6)]),  # drafts crossing emissions at 12, 20, 24 and 32; dense->sparse at 23
    (128, 300, [(125, 5), (254, 6)]),               # drafts crossing the ratio-128 emissions at 128 and 256
])
def test_trim_then_redecode_equals_never_decoded(ratio, n_true, drafts):
    """R15 against its definition: decoding k draft tokens, trimming them and decoding the true tokens gives, step
    for step, exactly the outputs, selections and state of decoding only the true tokens (with or without rollback
    slots in the rings)."""
    R = 6
    layer, ca, ci, invf, sink, rng = _rollback_setup(ratio, R)
    true = _tokens(layer, rng, n_true)
    cap = n_true // ratio + 4
    ref = _empty_state(layer, cap, 0)  # no rollback slots: rings of exactly W / frontier_slots
    ref_out = [_decode(layer, ca, ci, ref, t, sink, invf) for t in true]
    st = _empty_state(layer, cap, R)
    hw = np.zeros(1, dtype=np.int64)
    at = dict(drafts)
    for i, t in enumerate(true):
        if i in at:
            k = at[i]
            for d in _tokens(layer, rng, k):
                _decode(layer, ca, ci, st, d, sink, invf)
            assert O.trim(layer, st, np.array([k]), hw) == 0
            assert int(st["pos"][0]) == i and int(st["n_rows"][0]) == i // ratio
        out, sel = _decode(layer, ca, ci, st, t, sink, invf)
        assert np.array_equal(out, ref_out[i][0]), f"step {i}"
        assert sel == ref_out[i][1], f"step {i} selection"
    n = int(ref["n_rows"][0])
    assert int(st["n_rows"][0]) == n and int(st["pos"][0]) == n_true
    assert np.array_equal(st["pool"][:, :n], ref["pool"][:, :n])
    if layer.has_indexer:
        assert np.array_equal(st["ikeys"][:, :n], ref["ikeys"][:, :n])
    Wr, F = layer.W + R, layer.frontier_slots + R
    for tk in range(n_true - layer.W, n_true):  # the window tokens the next query attends
        assert np.array_equal(st["window"][0, tk % Wr], ref["window"][0, tk % layer.W])
    for tk in range(n_true - layer.frontier_slots, n_true):  # the frontier entries the next emission pools
        assert np.array_equal(st["front_a"][0, tk % F], ref["front_a"][0, tk % layer.frontier_slots])


def test_trim_refuses_beyond_the_margin():
    """R15: a trim past the rollback margin, below position 0, by a negative count, or on an inconsistent state is
    refused and changes nothing; the margin counts from the highest position reached, so two trims of 4 after
    decoding 6 draft tokens exceed a margin of 6 even though each alone would not."""
    layer, ca, ci, invf, sink, rng = _rollback_setup(4, 6)
    st = _empty_state(layer, 16, 6)
    hw = np.zeros(1, dtype=np.int64)
    for t in _tokens(layer, rng, 20):
        _decode(layer, ca, ci, st, t, sink, invf)
    snap = {k: v.copy() for k, v in st.items()}
    for n in (7, 21, -1):
        assert O.trim(layer, st, np.array([n]), hw) == O.ERR_ROLLBACK
        assert all(np.array_equal(st[k], snap[k]) for k in st)
    assert O.trim(layer, st, np.array([4]), hw) == 0 and int(hw[0]) == 20
    for t in _tokens(layer, rng, 2):  # back to 18, still below the high-water mark 20
        _decode(layer, ca, ci, st, t, sink, invf)
    assert O.trim(layer, st, np.array([5]), hw) == O.ERR_ROLLBACK  # 13 < 20 - 6
    assert O.trim(layer, st, np.array([4]), hw) == 0 and int(st["pos"][0]) == 14
    st["n_rows"][0] += 1
    assert O.trim(layer, st, np.array([1]), hw) == O.ERR_STATE
    zero = _rollback_setup(4, 0)[0]
    st2 = _empty_state(zero, 16, 0)
    st2["pos"][0], st2["n_rows"][0] = 8, 2
    assert O.trim(zero, st2, np.array([1]), np.zeros(1, dtype=np.int64)) == O.ERR_ROLLBACK  # no margin: no trim
    assert O.trim(zero, st2, np.array([0]), np.zeros(1, dtype=np.int64)) == 0


# --------------------------------------------------------------------------- cross-layer sharing (R16)

def test_consumer_layer_reads_the_owner_caches():
    """R16: a consumer layer with the owner's own queries, new token and window reproduces the owner's selection and
    output exactly (as an index-source layer and reusing the owner's selection alike); with its own queries it
    selects through the owner's keys, equal to the indexer run directly on them; severing the sharing (an empty
    pool in place of the owner's) changes the output, the negative control of the V4.1 port's tests."""
    layer, ca, ci, invf, sink, rng = _rollback_setup(4, 0, topk=5)
    st = _empty_state(layer, 16, 0)
    for t in _tokens(layer, rng, 40):
        _decode(layer, ca, ci, st, t, sink, invf)
    tok = _tokens(layer, rng, 1)[0]
    win0 = st["window"].copy()
    out_o, sel_o, nsel_o, _ = O.decode_step(layer, ca, ci, st, tok, sink, invf)
    owner = dict(pool=st["pool"], ikeys=st["ikeys"], n_rows=st["n_rows"], pos=st["pos"] - 1)
    pool_before = st["pool"].copy()
    for owner_sel in (None, (sel_o, nsel_o)):
        out_c, sel_c, nsel_c, _, err = O.consumer_decode_step(layer, owner, win0.copy(), tok, sink, invf, owner_sel)
        assert err == 0
        assert np.array_equal(out_c, out_o) and np.array_equal(sel_c, sel_o)
    assert np.array_equal(st["pool"], pool_before)
    own = _tokens(layer, rng, 1)[0]
    own_win = rng.standard_normal(win0.shape)
    out_c, sel_c, nsel_c, _, _ = O.consumer_decode_step(layer, owner, own_win, own, sink, invf)
    s2, n2 = O.index_topk(layer, own[3], own[4], owner["ikeys"], owner["n_rows"], owner["pos"], invf)
    assert np.array_equal(sel_c, s2) and np.array_equal(nsel_c, n2)
    out_p, sel_p, _, _, _ = O.consumer_decode_step(layer, owner, own_win, own, sink, invf, (sel_o, nsel_o))
    assert np.array_equal(sel_p, sel_o)  # a plain consumer attends the owner's selection, not its own
    keys = np.concatenate([owner["pool"][0][sel_o[0, :nsel_o[0]]]] +
                          [O.store(O.rope(own[2][0], int(owner["pos"][0]), invf), layer.dtype)[None]
                           if t == int(owner["pos"][0]) else own_win[0, t % layer.W][None]
                           for t in O.window_tokens(layer, int(owner["pos"][0]))])
    qr = O.store(O.rope(own[1][0], int(owner["pos"][0]), invf), layer.dtype)
    ref = O.output_rows(layer, O.attend(layer, qr, keys, sink), int(owner["pos"][0]), invf)
    assert np.allclose(out_p[0], ref, rtol=0, atol=0)
    severed = dict(owner, pool=np.zeros_like(owner["pool"]))
    out_s, _, _, _, _ = O.consumer_decode_step(layer, severed, own_win, own, sink, invf)
    assert rel_err_rows(out_s, out_c) > 0.05


# ---------------------------------------------------------------- fp8 index keys (R19)

def test_e4m3_format_values():
    """E4M3 as the OCP 8-bit floating-point format defines it: bias 7, 3 mantissa bits, subnormals m * 2^-9,
    S.1111.111 the only NaN encodings, largest finite magnitude 448 = 1.75 * 2^8."""
    v = O.e4m3_decode(np.arange(256))
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x01] == 2.0 ** -9 and v[0x07] == 7 * 2.0 ** -9 and v[0x08] == 2.0 ** -6
    assert v[0x38] == 1.0 and v[0x39] == 1.125 and v[0xB8] == -1.0 and v[0x58] == 16.0
    assert set(np.nonzero(np.isnan(v))[0].tolist()) == {0x7F, 0xFF}
    pos = v[:0x7F]
    assert np.all(np.diff(pos) > 0)  # codes 0 .. 0x7E increase strictly


def test_e4m3_rounding_ties_to_even_and_saturation():
    """Every finite code round-trips; midpoints go to the even code; magnitudes past 448 saturate."""
    c = np.arange(256)
    v = O.e4m3_decode(c)
    fin = ~np.isnan(v)
    assert np.array_equal(O.e4m3_encode(v[fin]), c[fin])
    mids = [(2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02), (1.0625, 0x38), (1.1875, 0x3A), (17.0, 0x58),
            (-1.0625, 0xB8), (432.0, 0x7E), (2.0 ** -6 + 2.0 ** -10, 0x08)]
    for x, want in mids:
        assert O.e4m3_encode([x])[0] == want, x
    # on either side of the midpoint 1.0625 between 1.0 (0x38) and 1.125 (0x39)
    assert O.e4m3_encode([1.06])[0] == 0x38 and O.e4m3_encode([1.07])[0] == 0x39
    assert O.e4m3_encode([449.0, 1e6, -1e6]).tolist() == [0x7E, 0x7E, 0xFE]


def test_fwht_is_the_hadamard_transform():
    """The fp32 butterflies equal the Sylvester Hadamard matrix (built independently by scipy) up to fp32 rounding,
    transform a one-hot into a row of (-1)^popcount(i & k), and applied twice give 128 x exactly on small integers."""
    import scipy.linalg
    H = scipy.linalg.hadamard(128).astype(np.float64)
    rng = np.random.default_rng(19)
    x = rng.standard_normal(128).astype(np.float32)
    assert np.max(np.abs(O.fwht_f32(x) - H @ x.astype(np.float64))) < 64 * 2.0 ** -23 * np.abs(x).sum()
    k = 37
    sign = np.array([(-1) ** bin(i & k).count("1") for i in range(128)], dtype=np.float64)
    assert np.array_equal(O.fwht_f32(np.eye(128, dtype=np.float32)[k]), sign)
    xi = rng.integers(-8, 9, 128).astype(np.float32)
    assert np.array_equal(O.fwht_f32(O.fwht_f32(xi)), 128 * xi)


def test_fp8_row_quantization():
    """The largest rotated element maps to +-448; every decoded element is within half an E4M3 step of the rotated
    value (scaled); a zero row keeps scale 0 and zero codes."""
    rng = np.random.default_rng(7)
    v = O.store(rng.standard_normal(128), "bf16")
    codes, scale = O.quantize_fp8_row(v)
    u = H_apply(v)
    assert np.max(np.abs(O.e4m3_decode(codes))) == 448.0
    y = u / np.float64(scale)
    step = np.where(np.abs(y) < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 1e-30))) - 3))
    assert np.all(np.abs(O.e4m3_decode(codes) - y) <= 0.5 * step + 1e-12 * np.abs(y))
    c0, s0 = O.quantize_fp8_row(np.zeros(128))
    assert s0 == 0 and not np.any(c0)


def H_apply(v):
    import scipy.linalg
    return scipy.linalg.hadamard(128).astype(np.float64) @ np.asarray(v, dtype=np.float64)


def test_fp8_scores_equal_the_exact_definition_on_representable_operands():
    """When the rotated query heads and key rows lie on the E4M3 grid with their largest element at 448 times a
    power-of-two scale, quantisation loses nothing and the fp8 score equals sum_h w_h ReLU(q_h . k_j) exactly
    (the rotation cancels: H H^T = 128 I)."""
    layer = O.Layer(dtype="bf16", H=4, D=16, R=8, W=8, ratio=4, Hi=3, Di=128, topk=2, X=24)
    rng = np.random.default_rng(23)
    grid = O.e4m3_decode(np.arange(0x7F))

    def representable(scale):
        u = rng.choice(grid, 128) * rng.choice([-1.0, 1.0], 128)
        u[rng.integers(128)] = 448.0
        return u * scale

    q_rot = np.stack([representable(2.0 ** -6) for _ in range(layer.Hi)])
    k_rot = np.stack([representable(2.0 ** -7) for _ in range(5)])
    q = np.stack([O.fwht_f32(r.astype(np.float32)) for r in q_rot]).astype(np.float64) / 128
    k = np.stack([O.fwht_f32(r.astype(np.float32)) for r in k_rot]).astype(np.float64) / 128
    qc = [O.quantize_fp8_row(r) for r in q]
    kc = [O.quantize_fp8_row(r) for r in k]
    assert all(s == 2.0 ** -6 for _, s in qc) and all(s == 2.0 ** -7 for _, s in kc)
    iw = rng.standard_normal(layer.Hi)
    got = O.index_scores_fp8(layer, np.stack([c for c, _ in qc]), np.array([s for _, s in qc]), iw,
                             np.stack([c for c, _ in kc]), np.array([s for _, s in kc]))
    w = iw * layer.Di ** -0.5 * layer.Hi ** -0.5
    want = (w[:, None] * np.maximum(q @ k.T, 0.0)).sum(axis=0)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-15)
