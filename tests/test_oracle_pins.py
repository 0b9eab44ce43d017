"""Pins of the CPU oracle to things other than itself (no GPU needed).

The source pages print no worked numeric example, so the oracle is pinned by:
  * brute force: a pure-Python ``math.fsum`` evaluation with no max shift and
    no NumPy, on tiny inputs;
  * closed forms: one key, equal keys, a dominant key, two keys with known
    logits, the GQA head mapping, exact bf16 decoding, the pool row layout;
  * invariants: merge(single partial) == partial bitwise, invariance of the
    merged result under any tiling of the keys (size-1 and empty tiles too),
    under permutation of physical pages, and a logit shift moving only the LSE;
  * a library second opinion: torch's float64 scaled_dot_product_attention and
    logsumexp on CPU.
Each pin is a function of an implementation namespace; the mutation tests at
the bottom plant plausible mistakes in copies of the oracle and require every
planted mistake to fail at least one pin.
"""

import math
import types

import numpy as np
import pytest
import torch

import oracle
from oracle import paged_attention as oa
from paged_decode_attention_attn_gb300 import workloads as wl

RTOL_BRUTE = 1e-12


def real_impl():
    return types.SimpleNamespace(
        attention=oa.attention, tile_attention=oa.tile_attention,
        lse_merge=oa.lse_merge, request_history=oa.request_history,
        bf16_bits_to_f64=oa.bf16_bits_to_f64,
        merge_stress_partials=oa.merge_stress_partials)


def impl_with(**over):
    ns = real_impl()
    for k, v in over.items():
        setattr(ns, k, v)
    if "attention" in over and "tile_attention" not in over:
        att = over["attention"]

        def tile_attention(q, K, V, tiles, scale):
            q = np.asarray(q, dtype=np.float64)
            outs = np.zeros((len(tiles),) + q.shape)
            lses = np.zeros((len(tiles), q.shape[0]))
            for i, (s, e) in enumerate(tiles):
                outs[i], lses[i] = att(q, K[s:e], V[s:e], scale)
            return outs, lses
        ns.tile_attention = tile_attention
    return ns


# ---------------------------------------------------------------------------
# brute force reference: pure Python, no max shift, math.fsum
# ---------------------------------------------------------------------------

def brute_attention(q, K, V, scale):
    n_q = len(q)
    n_kv = len(K[0])
    d = len(q[0])
    group = n_q // n_kv
    out, lse = [], []
    for h in range(n_q):
        g = h // group
        e = [math.exp(scale * math.fsum(q[h][i] * K[j][g][i] for i in range(d)))
             for j in range(len(K))]
        z = math.fsum(e)
        out.append([math.fsum(e[j] * V[j][g][i] for j in range(len(K))) / z
                    for i in range(d)])
        lse.append(math.log(z))
    return out, lse


def small_case(rng, n_q=4, n_kv=2, d=4, n_keys=7, scale=0.5):
    q = rng.standard_normal((n_q, d))
    K = rng.standard_normal((n_keys, n_kv, d))
    V = rng.standard_normal((n_keys, n_kv, d))
    return q, K, V, scale


# ---------------------------------------------------------------------------
# pins (each takes an implementation namespace and asserts)
# ---------------------------------------------------------------------------

def pin_bruteforce(impl):
    rng = np.random.default_rng(101)
    for n_keys in (1, 2, 5, 16):
        for (n_q, n_kv) in ((4, 2), (6, 1), (3, 3)):
            q, K, V, scale = small_case(rng, n_q, n_kv, 4, n_keys, 0.5)
            out, lse = impl.attention(q, K, V, scale)
            bo, bl = brute_attention(q.tolist(), K.tolist(), V.tolist(), scale)
            np.testing.assert_allclose(out, np.array(bo), rtol=RTOL_BRUTE, atol=1e-13)
            np.testing.assert_allclose(lse, np.array(bl), rtol=RTOL_BRUTE, atol=1e-13)


def pin_single_key(impl):
    rng = np.random.default_rng(102)
    q, K, V, scale = small_case(rng, 6, 2, 8, 1, 1.0 / 16)
    out, lse = impl.attention(q, K, V, scale)
    for h in range(6):
        g = h // 3
        assert np.array_equal(out[h], V[0, g])
        assert lse[h] == scale * float(np.dot(q[h], K[0, g]))


def pin_equal_keys(impl):
    rng = np.random.default_rng(103)
    q, K, V, scale = small_case(rng, 4, 2, 8, 9, 0.25)
    K[:] = K[0]
    out, lse = impl.attention(q, K, V, scale)
    for h in range(4):
        g = h // 2
        np.testing.assert_allclose(out[h], V[:, g].mean(axis=0), rtol=1e-13, atol=1e-14)
        s = scale * float(np.dot(q[h], K[0, g]))
        assert abs(lse[h] - (s + math.log(9))) < 1e-12


def pin_dominant_key(impl):
    rng = np.random.default_rng(104)
    q, K, V, scale = small_case(rng, 2, 1, 4, 12, 1.0)
    q[:] = 0.0
    q[:, 0] = 1.0
    K[:, 0, 0] = rng.uniform(-1, 1, size=12)
    K[5, 0, 0] = 80.0          # logit >= others + 79
    out, _ = impl.attention(q, K, V, scale)
    np.testing.assert_allclose(out[0], V[5, 0], rtol=0, atol=1e-30 + 1e-20 * np.abs(V).max())


def pin_two_keys(impl):
    # q.k with q = (16, 0, ...) and scale 1/16 gives logits equal to k[0]:
    # logits 0 and 1, weights 1 and e.
    q = np.zeros((1, 4))
    q[0, 0] = 16.0
    K = np.zeros((2, 1, 4))
    K[1, 0, 0] = 1.0
    V = np.zeros((2, 1, 4))
    V[0, 0] = [1.0, 0.0, 2.0, -1.0]
    V[1, 0] = [0.0, 3.0, 2.0, 1.0]
    out, lse = impl.attention(q, K, V, 1.0 / 16)
    e = math.e
    np.testing.assert_allclose(out[0], (V[0, 0] + e * V[1, 0]) / (1 + e), rtol=1e-15)
    assert abs(lse[0] - math.log(1 + e)) < 1e-15


def pin_gqa_mapping(impl):
    # kv head g carries values g + 1 everywhere: query head h must read
    # h // (Hq/Hkv) + 1 exactly.
    rng = np.random.default_rng(105)
    q, K, V, scale = small_case(rng, 24, 4, 8, 5, 1.0 / 16)
    for g in range(4):
        V[:, g, :] = g + 1.0
    out, _ = impl.attention(q, K, V, scale)
    for h in range(24):
        assert np.all(np.abs(out[h] - (h // 6 + 1.0)) < 1e-13), h


def pin_bf16_decode(impl):
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x7F80, 0xFF80, 0x0001, 0x4380, 0x0000,
                     0x8000, 0x3FC0], dtype=np.uint16)
    want = [1.0, -2.0, 0.25, np.inf, -np.inf, 2.0 ** -133, 256.0, 0.0, -0.0, 1.5]
    got = impl.bf16_bits_to_f64(bits)
    for g, w in zip(got, want):
        assert g == w
    assert np.isnan(impl.bf16_bits_to_f64(np.array([0x7FC0], dtype=np.uint16))[0])


def _bf16_bits_of_small_ints(vals):
    # small integers are exact in bf16; build their bit patterns from float32
    return (np.asarray(vals, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pin_pool_layout(impl):
    n_kv, d, pt = 2, 4, 4
    row = 2 * n_kv * d
    n_phys = 6
    table = np.array([4, 1, 5, 0], dtype=np.int32)
    length = 14                                 # 3.5 pages
    # (a) value = physical page + 1
    pool = np.broadcast_to(np.arange(n_phys)[:, None, None] + 1.0,
                           (n_phys, pt, row)).copy()
    K, V = impl.request_history(_bf16_bits_of_small_ints(pool), table, length, n_kv, d, pt)
    assert K.shape == (length, n_kv, d)
    for j in range(length):
        assert np.all(K[j] == table[j // pt] + 1) and np.all(V[j] == table[j // pt] + 1)
    # (b) value = row in page + 1
    pool = np.broadcast_to(np.arange(pt)[None, :, None] + 1.0, (n_phys, pt, row)).copy()
    K, V = impl.request_history(_bf16_bits_of_small_ints(pool), table, length, n_kv, d, pt)
    for j in range(length):
        assert np.all(K[j] == j % pt + 1)
    # (c) value = column + 1: K of head g is columns [g*d, (g+1)*d), V follows all K
    pool = np.broadcast_to(np.arange(row)[None, None, :] + 1.0, (n_phys, pt, row)).copy()
    K, V = impl.request_history(_bf16_bits_of_small_ints(pool), table, length, n_kv, d, pt)
    for g in range(n_kv):
        assert np.all(K[:, g, :] == np.arange(g * d, (g + 1) * d) + 1)
        assert np.all(V[:, g, :] == n_kv * d + np.arange(g * d, (g + 1) * d) + 1)


def pin_merge_identity(impl):
    rng = np.random.default_rng(106)
    o = rng.standard_normal((1, 5, 8)).astype(np.float32).astype(np.float64)
    l = (rng.standard_normal((1, 5)) * 30).astype(np.float32).astype(np.float64)
    mo, ml = impl.lse_merge(o, l)
    assert np.array_equal(mo, o[0]) and np.array_equal(ml, l[0])


def pin_tiling_invariance(impl):
    rng = np.random.default_rng(107)
    q, K, V, scale = small_case(rng, 6, 2, 8, 40, 0.7)
    ref_o, ref_l = impl.attention(q, K, V, scale)
    for trial in range(6):
        cuts = sorted(rng.choice(np.arange(1, 40), size=rng.integers(1, 12), replace=False))
        bounds = [0] + list(cuts) + [40]
        tiles = list(zip(bounds[:-1], bounds[1:]))
        if trial % 2:
            tiles = tiles + [(0, 0), (40, 40)]          # empty tiles change nothing
        if trial == 5:
            tiles = [(j, j + 1) for j in range(40)]       # size-1 tiles
        outs, lses = impl.tile_attention(q, K, V, tiles, scale)
        mo, ml = impl.lse_merge(outs, lses)
        np.testing.assert_allclose(mo, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(ml, ref_l, rtol=0, atol=1e-12)


def pin_page_permutation(impl):
    rng = np.random.default_rng(108)
    n_kv, d, pt = 2, 8, 4
    row = 2 * n_kv * d
    length = 21
    n_pages = 6
    pool_a = rng.standard_normal((n_pages, pt, row)).astype(np.float32)
    bits_a = (pool_a.view(np.uint32) >> 16).astype(np.uint16)
    perm = rng.permutation(n_pages)
    bits_b = np.empty_like(bits_a)
    bits_b[perm] = bits_a                     # page p of A lives at perm[p] in B
    Ka, Va = impl.request_history(bits_a, np.arange(n_pages), length, n_kv, d, pt)
    Kb, Vb = impl.request_history(bits_b, perm, length, n_kv, d, pt)
    assert np.array_equal(Ka, Kb) and np.array_equal(Va, Vb)


def pin_merge_shift(impl):
    rng = np.random.default_rng(109)
    outs = rng.standard_normal((5, 3, 8))
    lses = rng.standard_normal((5, 3)) * 3
    mo, ml = impl.lse_merge(outs, lses)
    so, sl = impl.lse_merge(outs, lses + 7.25)
    np.testing.assert_allclose(so, mo, rtol=0, atol=1e-13)
    np.testing.assert_allclose(sl, ml + 7.25, rtol=0, atol=1e-12)


def pin_library_second_opinion(impl):
    rng = np.random.default_rng(110)
    q, K, V, scale = small_case(rng, 24, 4, 32, 50, 1.0 / 16)
    out, lse = impl.attention(q, K, V, scale)
    qt = torch.tensor(q)[None, :, None, :]
    kt = torch.tensor(K).permute(1, 0, 2).repeat_interleave(6, dim=0)[None]
    vt = torch.tensor(V).permute(1, 0, 2).repeat_interleave(6, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    np.testing.assert_allclose(out, ref[0, :, 0].numpy(), rtol=0, atol=1e-12)
    ref_l = torch.logsumexp(scale * (qt @ kt.transpose(-1, -2)), dim=-1)
    np.testing.assert_allclose(lse, ref_l[0, :, 0].numpy(), rtol=0, atol=1e-12)


def pin_merge_stress(impl):
    case = wl.merge_stress(seed=5, n_requests=3, n_heads=4, head_dim=8, max_parts=9,
                           max_tile=17)
    for r in range(3):
        outs, lses, t_out, t_lse = impl.merge_stress_partials(
            case.tile_logits[r], case.tile_values[r], case.tile_bias[r])
        mo, ml = impl.lse_merge(outs, lses)
        np.testing.assert_allclose(mo, t_out, rtol=0, atol=1e-12)
        np.testing.assert_allclose(ml, t_lse, rtol=0, atol=1e-11)
        # brute-force check of the target itself (shifted by the largest logit
        # so that the +-80 biases stay finite in math.exp)
        logits = np.concatenate([s + c[:, None] for s, c in
                                 zip(case.tile_logits[r], case.tile_bias[r])], axis=1)
        vals = np.concatenate(case.tile_values[r], axis=0)
        for h in range(4):
            m = max(logits[h])
            e = [math.exp(x - m) for x in logits[h]]
            z = math.fsum(e)
            want = [math.fsum(e[j] * vals[j, i] for j in range(len(e))) / z
                    for i in range(8)]
            np.testing.assert_allclose(t_out[h], want, rtol=0, atol=1e-12)
            assert abs(t_lse[h] - (m + math.log(z))) < 1e-11


def pin_empty(impl):
    rng = np.random.default_rng(111)
    q, K, V, scale = small_case(rng, 4, 2, 8, 0, 0.5)
    out, lse = impl.attention(q, K, V, scale)
    assert np.all(out == 0) and np.all(lse == -np.inf)
    mo, ml = impl.lse_merge(np.zeros((3, 4, 8)), np.full((3, 4), -np.inf))
    assert np.all(mo == 0) and np.all(ml == -np.inf)
    q, K, V, scale = small_case(rng, 4, 2, 8, 6, 0.5)
    o1, l1 = impl.attention(q, K, V, scale)
    outs = np.stack([np.zeros((4, 8)), o1])
    lses = np.stack([np.full(4, -np.inf), l1])
    mo, ml = impl.lse_merge(outs, lses)
    assert np.array_equal(mo, o1) and np.array_equal(ml, l1)


PINS = [pin_bruteforce, pin_single_key, pin_equal_keys, pin_dominant_key, pin_two_keys,
        pin_gqa_mapping, pin_bf16_decode, pin_pool_layout, pin_merge_identity,
        pin_tiling_invariance, pin_page_permutation, pin_merge_shift,
        pin_library_second_opinion, pin_merge_stress, pin_empty]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(real_impl())


def test_nan_propagates():
    rng = np.random.default_rng(112)
    q, K, V, scale = small_case(rng, 4, 2, 8, 6, 0.5)
    V[3, 0, 2] = np.nan
    out, _ = oracle.attention(q, K, V, scale)
    assert np.all(np.isnan(out[0:2, 2]))          # heads of kv group 0 see the NaN
    assert not np.any(np.isnan(out[2:4]))
    lses = np.array([[0.0, np.nan], [1.0, 2.0]])
    mo, ml = oracle.lse_merge(np.ones((2, 2, 3)), lses)
    assert np.isnan(ml[1]) and np.all(np.isnan(mo[1])) and not np.isnan(ml[0])


def test_decode_layer_new_row_and_tiles():
    """decode_layer puts the new row at position L-1 and its tiled merge equals
    the unsplit attention; checked on the tiny workload's layout."""
    w = wl.custom([150], [[(0, 64), (64, 100), (100, 150)]], n_spare=2)
    t = wl.materialize(w, "cpu")
    geo = w.geometry
    pool_bits = t["pool"][0].view(torch.int16).numpy().view(np.uint16)
    q_bits = t["q"][0, 0].view(torch.int16).numpy().view(np.uint16)
    new_bits = t["new_rows"][0, 0].view(torch.int16).numpy().view(np.uint16)
    res = oracle.decode_layer(q_bits, pool_bits, w.page_table[0], 150, w.tiles[0],
                              geo.scale, geo.n_kv_heads, geo.head_dim,
                              new_row_bits=new_bits)
    np.testing.assert_allclose(res["out"], res["unsplit_out"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(res["lse"], res["unsplit_lse"], rtol=0, atol=1e-12)
    assert np.all(np.isfinite(res["out"]))        # the NaN canaries were never read
    # the new row decides the attention when its key dominates
    new = t["new_rows"][0, 0].clone()
    new[: geo.n_kv_heads * geo.head_dim] = 0
    new[0] = 2000.0                                 # k[0] of kv head 0 huge
    qn = t["q"][0, 0].clone()
    qn[:, 0] = 1.0
    res = oracle.decode_layer(qn.view(torch.int16).numpy().view(np.uint16), pool_bits,
                              w.page_table[0], 150, w.tiles[0], geo.scale,
                              geo.n_kv_heads, geo.head_dim,
                              new_row_bits=new.view(torch.int16).numpy().view(np.uint16))
    v0 = new[geo.n_kv_heads * geo.head_dim: geo.n_kv_heads * geo.head_dim + geo.head_dim]
    np.testing.assert_allclose(res["out"][0], v0.double().numpy(), rtol=0, atol=1e-9)


# ---------------------------------------------------------------------------
# mutation tests: planted mistakes in copies of the oracle must fail a pin
# ---------------------------------------------------------------------------

def _mut_attention(kind):
    def att(q, K, V, scale):
        q = np.asarray(q, dtype=np.float64)
        n_q, d = q.shape
        n_keys, n_kv, _ = K.shape
        group = n_q // n_kv
        out = np.zeros((n_q, d))
        lse = np.full(n_q, -np.inf)
        if n_keys == 0:
            return out, lse
        for h in range(n_q):
            g = (h % n_kv) if kind == "gqa_modulo" else h // group
            sc = 1.0 if kind == "no_scale" else scale
            s = sc * (K[:, g, :] @ q[h])
            m = np.max(s)
            w = np.exp(s - m)
            z = np.sum(w)
            if kind == "no_normalise":
                out[h] = w @ V[:, g, :]
            elif kind == "k_as_v":
                out[h] = (w @ K[:, g, :]) / z
            else:
                out[h] = (w @ V[:, g, :]) / z
            if kind == "lse_without_max":
                lse[h] = np.log(z)
            elif kind == "lse_log2":
                lse[h] = m + np.log2(z)
            else:
                lse[h] = m + np.log(z)
        return out, lse
    return att


def _mut_merge(kind):
    def merge(outs, lses):
        outs = np.asarray(outs, dtype=np.float64)
        lses = np.asarray(lses, dtype=np.float64)
        n_parts, n_heads = lses.shape
        d = outs.shape[2]
        out = np.zeros((n_heads, d))
        lse = np.full(n_heads, -np.inf)
        if n_parts == 0:
            return out, lse
        for h in range(n_heads):
            col = lses[:, h]
            m = np.max(col)
            if m == -np.inf:
                continue
            if kind == "average_outputs":
                out[h] = outs[:, h].mean(axis=0)
                lse[h] = m + math.log(np.sum(np.exp(col - m)))
                continue
            with np.errstate(over="ignore", invalid="ignore"):
                w = np.exp(col) if kind == "no_max_shift" else np.exp(col - m)
                if kind == "no_max_shift":
                    out[h] = (w @ outs[:, h]) / np.sum(w)
                    lse[h] = math.log(np.sum(w)) if np.isfinite(np.sum(w)) else np.inf
                    continue
            if kind == "weights_not_normalised":
                out[h] = w @ outs[:, h]
            else:
                out[h] = (w @ outs[:, h]) / np.sum(w)
            if kind == "lse_plus_sum":
                lse[h] = m + np.sum(w)
            else:
                lse[h] = m + math.log(np.sum(w))
        return out, lse
    return merge


def _mut_history(kind):
    def hist(pool_bits, page_table_row, length, n_kv_heads, head_dim, page_tokens=64):
        pool_bits = np.asarray(pool_bits, dtype=np.uint16)
        n = -(-int(length) // page_tokens)
        pages = (np.arange(n) if kind == "ignore_page_table"
                 else np.asarray(page_table_row[:n], dtype=np.int64))
        rows = pool_bits[pages].reshape(n * page_tokens, -1)[: int(length)]
        vals = oa.bf16_bits_to_f64(rows)
        if kind == "heads_interleaved":
            kv = vals.reshape(int(length), 2, head_dim, n_kv_heads).transpose(0, 1, 3, 2)
        elif kind == "kv_swapped":
            kv = vals.reshape(int(length), 2, n_kv_heads, head_dim)[:, ::-1]
        else:
            kv = vals.reshape(int(length), 2, n_kv_heads, head_dim)
        return kv[:, 0], kv[:, 1]
    return hist


def _mut_bf16(bits):
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(15)).view(np.float32).astype(np.float64)


MUTANTS = {
    "gqa_modulo": dict(attention=_mut_attention("gqa_modulo")),
    "no_scale": dict(attention=_mut_attention("no_scale")),
    "no_normalise": dict(attention=_mut_attention("no_normalise")),
    "k_as_v": dict(attention=_mut_attention("k_as_v")),
    "lse_without_max": dict(attention=_mut_attention("lse_without_max")),
    "lse_log2": dict(attention=_mut_attention("lse_log2")),
    "merge_average_outputs": dict(lse_merge=_mut_merge("average_outputs")),
    "merge_no_max_shift": dict(lse_merge=_mut_merge("no_max_shift")),
    "merge_weights_not_normalised": dict(lse_merge=_mut_merge("weights_not_normalised")),
    "merge_lse_plus_sum": dict(lse_merge=_mut_merge("lse_plus_sum")),
    "history_ignores_page_table": dict(request_history=_mut_history("ignore_page_table")),
    "history_heads_interleaved": dict(request_history=_mut_history("heads_interleaved")),
    "history_kv_swapped": dict(request_history=_mut_history("kv_swapped")),
    "bf16_wrong_shift": dict(bf16_bits_to_f64=_mut_bf16),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    impl = impl_with(**MUTANTS[name])
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except (AssertionError, ValueError, FloatingPointError, OverflowError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
