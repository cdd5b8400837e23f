"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

* hand-worked fixtures in tests/golden/ (each cites what it follows);
* closed forms (one key returns its value; a zero query averages; a dominant key selects);
* invariants (physical page placement does not matter; splitting the keys and merging by
  log-sum-exp gives the whole; the last row of a chunk is the decode of the full sequence);
* brute force with pure-Python loops and with scipy's softmax / logsumexp on tiny inputs;
* planted mistakes: plausible bugs planted into the oracle on the CPU must fail a pin.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


_LN = math.log     # bound once, so a planted mistake in a log function cannot reach the fixtures


def _val(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"ln": _LN, "inf": math.inf, "nan": math.nan}))


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------------------------
# Golden fixtures
# ----------------------------------------------------------------------------------------------
def golden_decode_inputs():
    g = _load("decode_worked.json")
    Hq, Hkv, D, P = g["num_q_heads"], g["num_kv_heads"], g["head_dim"], g["page_size"]
    k = np.full((g["num_pages"], P, Hkv, D), np.nan)
    v = np.full_like(k, np.nan)
    slot_of = {}
    for t, page, slot in g["placement_token_page_slot"]:
        k[page, slot] = 0.0
        v[page, slot] = 0.0
        slot_of[t] = (page, slot)
    for kvh, t, d, e in g["k"]:
        k[slot_of[t] + (kvh, d)] = _val(e)
    for kvh, t, d, e in g["v"]:
        v[slot_of[t] + (kvh, d)] = _val(e)
    q = np.zeros((1, Hq, D))
    for h, d, e in g["q"]:
        q[0, h, d] = _val(e)
    bt = np.array(g["block_table"], dtype=np.int32)
    return g, q, k, v, bt, np.array([g["seq_len"]]), _val(g["scale"])


def check_golden_decode():
    g, q, k, v, bt, L, scale = golden_decode_inputs()
    o, lse = oracle.decode(q, k, v, bt, L, scale)
    exp_o = np.zeros_like(o)
    for h, d, e in g["expected_o"]:
        exp_o[0, h, d] = _val(e)
    exp_lse = np.array([[_val(e) for _, e in sorted(g["expected_lse"])]])
    return np.allclose(o, exp_o, rtol=1e-12, atol=1e-12) and np.allclose(lse, exp_lse, rtol=1e-12)


def golden_prefill_inputs():
    g = _load("prefill_worked.json")
    Hq, Hkv, D, P = g["num_q_heads"], g["num_kv_heads"], g["head_dim"], g["page_size"]
    k = np.full((g["num_pages"], P, Hkv, D), np.nan)
    v = np.full_like(k, np.nan)
    slot_of = {}
    for b, t, page, slot in g["placement_seq_token_page_slot"]:
        k[page, slot] = 0.0
        v[page, slot] = 0.0
        slot_of[(b, t)] = (page, slot)
    for b, t, d, e in g["k"]:
        k[slot_of[(b, t)] + (0, d)] = _val(e)
    for b, t, d, e in g["v"]:
        v[slot_of[(b, t)] + (0, d)] = _val(e)
    Tq = g["cu_q_lens"][-1]
    q = np.zeros((Tq, Hq, D))
    for r, h, d, e in g["q"]:
        q[r, h, d] = _val(e)
    return (g, q, np.array(g["cu_q_lens"]), k, v, np.array(g["block_table"], dtype=np.int32),
            np.array(g["seq_lens"]), _val(g["scale"]))


def check_golden_prefill():
    g, q, cu, k, v, bt, L, scale = golden_prefill_inputs()
    o, lse = oracle.prefill(q, cu, k, v, bt, L, scale)
    exp_o = np.zeros_like(o)
    for r, h, d, e in g["expected_o"]:
        exp_o[r, h, d] = _val(e)
    exp_lse = np.zeros_like(lse)
    for r, h, e in g["expected_lse"]:
        exp_lse[r, h] = _val(e)
    return np.allclose(o, exp_o, rtol=1e-12, atol=1e-12) and np.allclose(lse, exp_lse, rtol=1e-12)


def check_golden_merge():
    g = _load("merge_worked.json")
    S, R, H, D = g["parts"], g["rows"], g["heads"], g["head_dim"]
    o_parts = np.zeros((S, R, H, D))
    lse_parts = np.zeros((S, R, H))
    for s, r, h, e in g["lse_parts"]:
        lse_parts[s, r, h] = _val(e)
    for s, r, h, d, e in g["o_parts"]:
        o_parts[s, r, h, d] = _val(e)
    o, lse = oracle.merge_lse(o_parts, lse_parts)
    exp_o = np.zeros((R, H, D))
    for r, h, d, e in g["expected_o"]:
        exp_o[r, h, d] = _val(e)
    exp_lse = np.zeros((R, H))
    for r, h, e in g["expected_lse"]:
        exp_lse[r, h] = _val(e)
    same_inf = np.array_equal(np.isneginf(lse), np.isneginf(exp_lse))
    fin = np.isfinite(exp_lse)
    return (same_inf and np.allclose(lse[fin], exp_lse[fin], rtol=1e-13)
            and np.allclose(o, exp_o, rtol=1e-12, atol=1e-12))


def check_golden_append():
    g = _load("kv_append_worked.json")
    P, NP, Hkv, D = g["page_size"], g["num_pages"], g["num_kv_heads"], g["head_dim"]
    T = g["cu_new_lens"][-1]
    rng = np.random.default_rng(5)
    k_new = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    v_new = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    k_pool = rng.integers(0, 1 << 16, size=(NP, P, Hkv, D), dtype=np.uint16)
    v_pool = rng.integers(0, 1 << 16, size=(NP, P, Hkv, D), dtype=np.uint16)
    k2, v2 = oracle.kv_append(k_new, v_new, g["cu_new_lens"], g["start_pos"],
                              np.array(g["block_table"]), k_pool, v_pool)
    ek, ev = k_pool.copy(), v_pool.copy()
    for row, page, slot in g["expected_row_page_slot"]:
        ek[page, slot] = k_new[row]
        ev[page, slot] = v_new[row]
    return np.array_equal(k2, ek) and np.array_equal(v2, ev)


def test_golden_decode():
    assert check_golden_decode()


def test_golden_prefill():
    assert check_golden_prefill()


def test_golden_merge():
    assert check_golden_merge()


def test_golden_kv_append():
    assert check_golden_append()


# ----------------------------------------------------------------------------------------------
# Closed forms and invariants at the production head shape (16/8 heads, d 128, pages of 16).
# Inputs are built logically (contiguous tokens) and scattered into pages here, so the
# expected values never use the oracle's gather.
# ----------------------------------------------------------------------------------------------
HQ, HKV, D, P = 16, 8, 128, 16


def scatter(K_logical, page_list, num_pages):
    """Contiguous per-sequence tokens [L, Hkv, D] -> a NaN pool with pages page_list."""
    L = K_logical.shape[0]
    pool = np.full((num_pages, P, K_logical.shape[1], K_logical.shape[2]), np.nan)
    padded = np.full((len(page_list) * P,) + K_logical.shape[1:], np.nan)
    padded[:L] = K_logical
    pool[np.asarray(page_list)] = padded.reshape(len(page_list), P, *K_logical.shape[1:])
    return pool


def random_seq(rng, L, num_pages=None):
    n = -(-L // P)
    num_pages = num_pages or n + 3
    pages = rng.permutation(num_pages)[:n]
    K = rng.standard_normal((L, HKV, D))
    V = rng.standard_normal((L, HKV, D))
    bt = np.zeros((1, max(n, 1)), dtype=np.int32)
    bt[0, :n] = pages
    return K, V, scatter(K, pages, num_pages), scatter(V, pages, num_pages), bt


@pytest.mark.parametrize("L", [1, 15, 16, 17, 33, 257])
def test_zero_query_is_mean_of_values(L):
    rng = np.random.default_rng(L)
    K, V, kp, vp, bt = random_seq(rng, L)
    q = np.zeros((1, HQ, D))
    o, lse = oracle.decode(q, kp, vp, bt, [L], 0.1)
    for h in range(HQ):
        np.testing.assert_allclose(o[0, h], V[:, h // 2].mean(axis=0), rtol=1e-12, atol=1e-13)
        assert abs(lse[0, h] - math.log(L)) < 1e-12


def test_single_key_returns_its_value_exactly():
    rng = np.random.default_rng(1)
    K, V, kp, vp, bt = random_seq(rng, 1)
    q = rng.standard_normal((1, HQ, D))
    o, lse = oracle.decode(q, kp, vp, bt, [1], 0.25)
    for h in range(HQ):
        assert np.array_equal(o[0, h], V[0, h // 2])
        assert abs(lse[0, h] - 0.25 * math.fsum(q[0, h] * K[0, h // 2])) < 1e-12


def test_empty_sequence():
    kp = np.full((2, P, HKV, D), np.nan)
    o, lse = oracle.decode(np.ones((1, HQ, D)), kp, kp, np.zeros((1, 1), np.int32), [0], 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("t_star", [0, 15, 16, 31, 200, 299])
def test_dominant_key_selects_its_value(t_star):
    """A key whose score beats every other by more than 800 takes all the weight."""
    rng = np.random.default_rng(t_star)
    L = 300
    K, V, kp, vp, bt = random_seq(rng, L)
    q = rng.standard_normal((1, HQ, D))
    for g in range(HKV):
        # key t_star aligned with both queries of group g, huge norm
        K[t_star, g] = 1e3 * (q[0, 2 * g] + q[0, 2 * g + 1])
    n = -(-L // P)
    kp = scatter(K, bt[0, :n], kp.shape[0])
    o, lse = oracle.decode(q, kp, vp, bt, [L], 1.0)
    for h in range(HQ):
        assert np.array_equal(o[0, h], V[t_star, h // 2])
        assert np.isfinite(lse[0, h])


def test_page_permutation_is_bit_invariant():
    rng = np.random.default_rng(7)
    L = 100
    K, V, kp, vp, bt = random_seq(rng, L, num_pages=20)
    q = rng.standard_normal((1, HQ, D))
    o1, l1 = oracle.decode(q, kp, vp, bt, [L], 0.3)
    pages2 = rng.permutation(20)[: bt.shape[1]]
    bt2 = pages2[None, :].astype(np.int32)
    o2, l2 = oracle.decode(q, scatter(K, pages2, 20), scatter(V, pages2, 20), bt2, [L], 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("split", [16, 64, 160])
def test_split_and_merge_equals_whole(split):
    rng = np.random.default_rng(split)
    L = 200
    K, V, kp, vp, bt = random_seq(rng, L)
    q = rng.standard_normal((1, HQ, D))
    o, lse = oracle.decode(q, kp, vp, bt, [L], 0.2)
    o_a, l_a = oracle.decode(q, kp, vp, bt, [split], 0.2)
    o_b, l_b = oracle.decode(q, kp, vp, bt[:, split // P:], [L - split], 0.2)
    om, lm = oracle.merge_lse(np.stack([o_a, o_b]), np.stack([l_a, l_b]))
    np.testing.assert_allclose(om, o, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lm, lse, rtol=1e-13)


def test_merge_of_identical_parts():
    rng = np.random.default_rng(3)
    o1 = rng.standard_normal((5, 4, D))
    l1 = rng.standard_normal((5, 4))
    om, lm = oracle.merge_lse(np.stack([o1] * 3), np.stack([l1] * 3))
    np.testing.assert_allclose(om, o1, rtol=1e-13)
    np.testing.assert_allclose(lm, l1 + math.log(3), rtol=1e-13)


@pytest.mark.parametrize("q_len", [1, 15, 16, 17, 129])
def test_prefill_rows_equal_decode_of_their_prefix(q_len):
    """Row i of a chunk is the decode of the sequence truncated after position o + i."""
    rng = np.random.default_rng(q_len)
    L = 150 + q_len
    K, V, kp, vp, bt = random_seq(rng, L)
    q = rng.standard_normal((q_len, HQ, D))
    o, lse = oracle.prefill(q, [0, q_len], kp, vp, bt, [L], 0.15)
    for i in sorted({0, q_len // 2, q_len - 1}):
        od, ld = oracle.decode(q[i][None], kp, vp, bt, [L - q_len + i + 1], 0.15)
        np.testing.assert_allclose(o[i], od[0], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[i], ld[0], rtol=1e-13)


def test_zero_query_chunk_closed_form():
    """q = 0: row i averages V over keys 0..o+i and its lse is ln(o+i+1)."""
    rng = np.random.default_rng(11)
    o_off, q_len = 37, 20
    L = o_off + q_len
    K, V, kp, vp, bt = random_seq(rng, L)
    out, lse = oracle.prefill(np.zeros((q_len, HQ, D)), [0, q_len], kp, vp, bt, [L], 1.0)
    for i in range(q_len):
        for h in range(HQ):
            np.testing.assert_allclose(out[i, h], V[: o_off + i + 1, h // 2].mean(axis=0),
                                       rtol=1e-12, atol=1e-13)
            assert abs(lse[i, h] - math.log(o_off + i + 1)) < 1e-12


def test_large_scores_stay_finite():
    rng = np.random.default_rng(12)
    L = 64
    K, V, kp, vp, bt = random_seq(rng, L)
    q = 300.0 * rng.standard_normal((1, HQ, D))
    o, lse = oracle.decode(q, kp, vp, bt, [L], 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    assert np.all(np.abs(o) <= np.abs(V).max() + 1e-9)


def test_bruteforce_python_loops():
    """Tiny case against nested Python loops (math.exp, no numpy arithmetic)."""
    rng = np.random.default_rng(13)
    Hq, Hkv, d, page, L, NP = 4, 2, 8, 4, 11, 6
    K = rng.standard_normal((L, Hkv, d))
    V = rng.standard_normal((L, Hkv, d))
    pages = [4, 1, 3]
    kp = np.full((NP, page, Hkv, d), np.nan)
    vp = np.full((NP, page, Hkv, d), np.nan)
    for t in range(L):
        kp[pages[t // page], t % page] = K[t]
        vp[pages[t // page], t % page] = V[t]
    q = rng.standard_normal((1, Hq, d))
    scale = 0.37
    o, lse = oracle.decode(q, kp, vp, np.array([pages], np.int32), [L], scale)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = [scale * sum(q[0, h, j] * K[t, g, j] for j in range(d)) for t in range(L)]
        w = [math.exp(x) for x in s]
        tot = sum(w)
        for j in range(d):
            ref = sum(w[t] * V[t, g, j] for t in range(L)) / tot
            assert abs(o[0, h, j] - ref) < 1e-12
        assert abs(lse[0, h] - math.log(tot)) < 1e-12


def test_against_scipy_softmax_and_logsumexp():
    sp = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(14)
    L, q_len = 90, 9
    K, V, kp, vp, bt = random_seq(rng, L)
    q = rng.standard_normal((q_len, HQ, D))
    o, lse = oracle.prefill(q, [0, q_len], kp, vp, bt, [L], 0.09)
    for i in range(q_len):
        n = L - q_len + i + 1
        for h in range(HQ):
            s = 0.09 * np.einsum("d,td->t", q[i, h], K[:n, h // 2])
            np.testing.assert_allclose(lse[i, h], sp.logsumexp(s), rtol=1e-13)
            np.testing.assert_allclose(o[i, h], sp.softmax(s) @ V[:n, h // 2], rtol=1e-11, atol=1e-13)


def test_kv_append_then_gather_is_concatenation():
    rng = np.random.default_rng(15)
    L0, T = 29, 9
    n = -(-(L0 + T) // P)
    pages = rng.permutation(10)[:n]
    k_pool = rng.integers(0, 1 << 16, size=(10, P, HKV, D), dtype=np.uint16)
    v_pool = k_pool[::-1].copy()
    k_new = rng.integers(0, 1 << 16, size=(T, HKV, D), dtype=np.uint16)
    v_new = rng.integers(0, 1 << 16, size=(T, HKV, D), dtype=np.uint16)
    bt = pages[None, :].astype(np.int32)
    k2, v2 = oracle.kv_append(k_new, v_new, [0, T], [L0], bt, k_pool, v_pool)
    before = k_pool[pages].reshape(-1, HKV, D)[:L0]
    after = k2[pages].reshape(-1, HKV, D)
    assert np.array_equal(after[:L0], before)
    assert np.array_equal(after[L0:L0 + T], k_new)
    assert np.array_equal(after[L0 + T:], k_pool[pages].reshape(-1, HKV, D)[L0 + T:])
    untouched = np.setdiff1d(np.arange(10), pages)
    assert np.array_equal(k2[untouched], k_pool[untouched])
    assert np.array_equal(v2[untouched], v_pool[untouched])


def test_bf16_widening_is_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x7F80, 0xFF80], dtype=np.uint16)
    got = oracle.as_f64(bits)
    assert got[0] == 1.0 and got[1] == -1.0
    assert got[2] == 3.140625                     # 0x4049 = 1.5703125 * 2
    assert got[3] == 2.0 ** -133                  # smallest bf16 subnormal
    assert got[4] == (2 - 2 ** -7) * 2.0 ** 127   # largest finite bf16
    assert got[5] == math.inf and got[6] == -math.inf


# ----------------------------------------------------------------------------------------------
# Planted mistakes: each plausible bug, planted into the oracle on the CPU, must fail a pin.
# ----------------------------------------------------------------------------------------------
def _all_golden_pass():
    return (check_golden_decode() and check_golden_prefill() and check_golden_merge()
            and check_golden_append())


MUTANTS = {
    "gqa_map_modulo": lambda m: m.setattr(oracle, "kv_head_of", lambda h, hq, hkv: h % hkv),
    "causal_top_left": lambda m: m.setattr(oracle, "visible_key_count", lambda i, ql, sl: i + 1),
    "causal_off_by_one": lambda m: m.setattr(oracle, "visible_key_count", lambda i, ql, sl: sl - ql + i),
    "scale_dropped": lambda m: m.setattr(
        oracle, "attend_rows", (lambda f: lambda Q, K, V, c, s: f(Q, K, V, c, 1.0))(oracle.attend_rows)),
    "scale_squared": lambda m: m.setattr(
        oracle, "attend_rows", (lambda f: lambda Q, K, V, c, s: f(Q, K, V, c, s * s))(oracle.attend_rows)),
    "lse_log2": lambda m: m.setattr(oracle.np, "log", np.log2),
    "softmax_exp2": lambda m: m.setattr(oracle.np, "exp", np.exp2),
    "page_identity": lambda m: m.setattr(
        oracle, "gather_keys",
        (lambda f: lambda pool, row, L, g: f(pool, np.arange(len(row)), L, g))(oracle.gather_keys)),
    "merge_plain_mean": lambda m: m.setattr(
        oracle, "merge_lse", lambda o, l: (np.mean(o, axis=0), np.max(l, axis=0))),
}


def _mutant_append(slot_shift=0, ignore_start=False, identity_pages=False, swap_kv=False):
    """The oracle's kv_append with one step changed (for the planted-mistake test only)."""
    def kv_append(k_new, v_new, cu_new_lens, start_pos, block_table, k_pool, v_pool):
        k_out, v_out = np.array(k_pool, copy=True), np.array(v_pool, copy=True)
        P = k_pool.shape[1]
        cu = [int(c) for c in cu_new_lens]
        for b in range(len(cu) - 1):
            for j in range(cu[b + 1] - cu[b]):
                pos = (0 if ignore_start else int(start_pos[b])) + j + slot_shift
                page = pos // P if identity_pages else int(block_table[b, pos // P])
                src_k, src_v = (v_new, k_new) if swap_kv else (k_new, v_new)
                k_out[page, pos % P] = src_k[cu[b] + j]
                v_out[page, pos % P] = src_v[cu[b] + j]
        return k_out, v_out
    return kv_append


MUTANTS.update({
    "append_slot_off_by_one": lambda m: m.setattr(oracle, "kv_append", _mutant_append(slot_shift=1)),
    "append_start_ignored": lambda m: m.setattr(oracle, "kv_append", _mutant_append(ignore_start=True)),
    "append_block_table_bypassed": lambda m: m.setattr(oracle, "kv_append", _mutant_append(identity_pages=True)),
    "append_k_v_swapped": lambda m: m.setattr(oracle, "kv_append", _mutant_append(swap_kv=True)),
})


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    assert _all_golden_pass()
    with monkeypatch.context() as m:
        MUTANTS[name](m)
        with np.errstate(all="ignore"):
            try:
                caught = not _all_golden_pass()
            except (AssertionError, IndexError, ValueError):
                caught = True
    assert caught, f"planted mistake {name} passed every golden pin"
