"""Pins of the fp64 CPU oracle to facts that do not come from the oracle itself.

Each test fixes the oracle against something the pages or the mathematics
determine: the printed packing example, closed forms of special cases, the
row-sum invariant of softmax, isolation and causality invariants, chunked ==
one-shot, and an independent library routine (PyTorch's float64
scaled_dot_product_attention).  A plausible slip in the oracle (a dropped
visible key, a wrong sign or scale, the wrong KV head, a key read from the
wrong token, a transposed operand) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from prefill_phase_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run_oracle(oracle_mod, wl, cache_k, cache_v, inp, rows=None, causal=None, window=0,
               block_table=None, block_size=0, rope_theta=0.0):
    cap = wl.max_cache_len if block_table is None else block_table.shape[1] * block_size
    return oracle_mod.prefill_attention(
        W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
        inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(), inp["cache_offsets"].numpy(),
        W.bf16_bits(cache_k), W.bf16_bits(cache_v),
        n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim,
        max_cache_len=cap, scale=wl.scale,
        causal=wl.causal if causal is None else causal, window=window, rows=rows,
        block_table=None if block_table is None else np.asarray(block_table, np.int32), block_size=block_size,
        rope_theta=rope_theta)


def f64(t):
    return t.to(torch.float64).numpy()


def _custom(name, H, Hk, d, lens, pref, cap=None, seed=7, causal=True):
    cap = cap or max(p + n for p, n in zip(pref, lens))
    return W.Workload(name, H, Hk, d, cap, [W.Step(list(lens), list(pref))], list(pref),
                      seed=seed, causal=causal)


# ---------------------------------------------------------------- packing ---

def test_packing_example_from_page():
    g = json.load(open(os.path.join(GOLDEN, "varlen_packing_nxmr.json")))
    step = W.Step(g["lengths"], [0, 0, 0])
    assert step.cu_seqlens_q() == g["cu_seqlens"]
    assert step.total_q == g["total_tokens"]
    longest = max(g["lengths"])
    waste = [(longest - n) / longest for n in g["lengths"]]
    assert np.allclose(waste, g["padded_waste"])
    ex = g["second_example"]["lengths"]
    sec = g["second_example"]
    assert 1 - sum(ex) / (len(ex) * max(ex)) == pytest.approx(sec["batch_waste_approx"], abs=sec["abs_tol"])
    wl = W.get("tiny_packed")
    assert wl.steps[0].cu_seqlens_q() == g["cu_seqlens"]


def test_packed_equals_each_sequence_alone(oracle_mod):
    """Bitwise: the oracle does the same per-row arithmetic packed or alone."""
    wl = W.get("tiny_packed")
    ck, cv, (inp,) = W.make_inputs(wl)
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    cu = inp["cu_seqlens_q"].tolist()
    for b in range(wl.num_seqs):
        n = cu[b + 1] - cu[b]
        sl = slice(cu[b], cu[b + 1])
        one = _custom("one", wl.n_heads, wl.n_kv_heads, wl.head_dim, [n], [0], cap=wl.max_cache_len)
        sub = dict(q=inp["q"][sl], k=inp["k"][sl], v=inp["v"][sl],
                   cu_seqlens_q=torch.tensor([0, n], dtype=torch.int32),
                   cu_seqlens_k=torch.tensor([0, n], dtype=torch.int32),
                   cache_offsets=torch.tensor([0], dtype=torch.int32))
        o1, l1, _, _ = run_oracle(oracle_mod, one, ck[b:b + 1], cv[b:b + 1], sub)
        assert np.array_equal(o1, out[sl]) and np.array_equal(l1, lse[sl])


# ----------------------------------------------------------- closed forms ---

def test_length_one_returns_v_and_score(oracle_mod):
    """One key: the weight is exactly 1, so out = v and lse = scale * q.k."""
    wl = _custom("len1", 4, 2, 64, [1, 1, 1], [0, 0, 0])
    ck, cv, (inp,) = W.make_inputs(wl)
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    G = wl.n_heads // wl.n_kv_heads
    for t in range(3):
        for h in range(wl.n_heads):
            assert np.array_equal(out[t, h], f64(inp["v"][t, h // G]))
            s = wl.scale * float(np.dot(f64(inp["q"][t, h]), f64(inp["k"][t, h // G])))
            assert lse[t, h] == pytest.approx(s, abs=1e-13)


def test_two_keys_is_a_logistic_blend(oracle_mod):
    """One cached key plus the token itself: w1 = 1 / (1 + exp(s0 - s1))."""
    wl = _custom("two", 2, 1, 32, [1], [1])
    ck, cv, (inp,) = W.make_inputs(wl)
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    k0, v0 = f64(ck[0, 0, 0]), f64(cv[0, 0, 0])
    k1, v1 = f64(inp["k"][0, 0]), f64(inp["v"][0, 0])
    for h in range(2):
        q = f64(inp["q"][0, h])
        s0, s1 = wl.scale * q @ k0, wl.scale * q @ k1
        w1 = 1.0 / (1.0 + math.exp(s0 - s1))
        assert np.allclose(out[0, h], (1 - w1) * v0 + w1 * v1, rtol=0, atol=1e-13)
        assert lse[0, h] == pytest.approx(max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1))), abs=1e-13)


def test_causal_rows_sum_to_one(oracle_mod):
    """With every V row equal to 1 the output is the row sum of the weights."""
    wl = W.random_workload(11, head_dim=64, group=4, n_kv_heads=2, max_prefix=60, max_len=70)
    ck, cv, (inp,) = W.make_inputs(wl)
    ones = torch.ones_like(inp["v"])
    inp = dict(inp, v=ones)
    cv = torch.ones_like(cv)
    out, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    assert np.all(np.abs(out - 1.0) <= 1e-15)


def test_equal_keys_give_prefix_mean(oracle_mod):
    """All keys equal: uniform weights over the P+i+1 visible keys."""
    wl = _custom("eq", 4, 2, 32, [9, 5], [6, 0], cap=20)
    ck, cv, (inp,) = W.make_inputs(wl)
    key = inp["k"][0, 0].clone()
    inp = dict(inp, k=key.expand_as(inp["k"]).contiguous())
    ck = key.expand_as(ck).contiguous()
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    G = wl.n_heads // wl.n_kv_heads
    cu = inp["cu_seqlens_q"].tolist()
    for b, P in enumerate([6, 0]):
        for i in range(cu[b + 1] - cu[b]):
            t = cu[b] + i
            for h in range(wl.n_heads):
                kvh = h // G
                vals = np.concatenate([f64(cv[b, kvh, :P]), f64(inp["v"][cu[b]:t + 1, kvh])])
                assert vals.shape[0] == P + i + 1
                assert np.allclose(out[t, h], vals.mean(axis=0), rtol=0, atol=1e-14)
                s = wl.scale * float(f64(inp["q"][t, h]) @ f64(key))
                assert lse[t, h] == pytest.approx(s + math.log(P + i + 1), abs=1e-13)


def test_gqa_contiguous_head_groups(oracle_mod):
    """KV head j holds constant V = j+1: q head h must return h // G + 1."""
    wl = _custom("gqa", 8, 2, 32, [7, 3], [4, 2], cap=12)
    ck, cv, (inp,) = W.make_inputs(wl)
    v = torch.empty_like(inp["v"])
    for j in range(2):
        v[:, j] = float(j + 1)
        cv[:, j] = float(j + 1)
    out, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, dict(inp, v=v))
    for h in range(8):
        assert np.allclose(out[:, h], h // 4 + 1, rtol=0, atol=1e-14)


# ------------------------------------------------------------- invariants ---

def test_sequences_are_isolated(oracle_mod):
    wl = W.get("tiny_packed")
    ck, cv, (inp,) = W.make_inputs(wl)
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    k2, v2 = inp["k"].clone(), inp["v"].clone()
    k2[5:7] = -k2[5:7] * 3
    v2[5:7] = v2[5:7] + 1
    out2, lse2, _, _ = run_oracle(oracle_mod, wl, ck, cv, dict(inp, k=k2, v=v2))
    keep = np.r_[0:5, 7:10]
    assert np.array_equal(out[keep], out2[keep]) and np.array_equal(lse[keep], lse2[keep])
    assert not np.allclose(out[5:7], out2[5:7])


def test_causality(oracle_mod):
    """Changing key/value of new token i leaves rows < i untouched and moves row i."""
    wl = _custom("causal", 2, 2, 32, [12], [5], cap=17)
    ck, cv, (inp,) = W.make_inputs(wl)
    out, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    i = 6
    k2, v2 = inp["k"].clone(), inp["v"].clone()
    k2[i] = k2[i] * -2
    v2[i] = v2[i] + 3
    out2, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, dict(inp, k=k2, v=v2))
    assert np.array_equal(out[:i], out2[:i])
    assert not np.allclose(out[i:], out2[i:])
    # non-causal: every row sees every key, so the last row is the same either way
    outn, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, causal=False)
    assert np.array_equal(outn[-1], out[-1])
    assert not np.allclose(outn[0], out[0])


def test_chunked_equals_one_shot(oracle_mod):
    """A prompt in 4 chunks over the cache == one launch: outputs and cache, bitwise."""
    H, Hk, d, n, c = 4, 2, 32, 384, 96
    one = _custom("one", H, Hk, d, [n], [0], cap=n)
    ck, cv, (inp,) = W.make_inputs(one)
    out1, lse1, ck1, cv1 = run_oracle(oracle_mod, one, ck, cv, inp)
    cur_k, cur_v = W.bf16_bits(ck), W.bf16_bits(cv)
    outs, lses = [], []
    for s in range(n // c):
        sl = slice(s * c, (s + 1) * c)
        o, l, cur_k, cur_v = oracle_mod.prefill_attention(
            W.bf16_bits(inp["q"][sl]), W.bf16_bits(inp["k"][sl]), W.bf16_bits(inp["v"][sl]),
            np.array([0, c], np.int32), np.array([0, s * c + c], np.int32), np.array([s * c], np.int32),
            cur_k, cur_v, n_heads=H, n_kv_heads=Hk, head_dim=d, max_cache_len=n, scale=one.scale)
        outs.append(o)
        lses.append(l)
    assert np.array_equal(np.concatenate(outs), out1)
    assert np.array_equal(np.concatenate(lses), lse1)
    assert np.array_equal(cur_k, ck1) and np.array_equal(cur_v, cv1)


def test_row_subset_matches_full_run(oracle_mod):
    wl = W.random_workload(5, head_dim=32, group=2)
    ck, cv, (inp,) = W.make_inputs(wl)
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    rows = np.arange(0, wl.steps[0].total_q * wl.n_heads, 7, dtype=np.int64)
    o2, l2, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, rows=rows)
    t, h = rows // wl.n_heads, rows % wl.n_heads
    assert np.array_equal(o2[t, h], out[t, h]) and np.array_equal(l2[t, h], lse[t, h])


def test_cache_write_closed_form(oracle_mod):
    wl = _custom("cache", 4, 2, 32, [3, 0, 5], [2, 4, 0], cap=9)
    ck, cv, (inp,) = W.make_inputs(wl)
    _, _, ck2, cv2 = run_oracle(oracle_mod, wl, ck, cv, inp)
    exp_k, exp_v = W.bf16_bits(ck).copy(), W.bf16_bits(cv).copy()
    cu = inp["cu_seqlens_q"].tolist()
    for b, P in enumerate([2, 4, 0]):
        for i in range(cu[b + 1] - cu[b]):
            exp_k[b, :, P + i] = W.bf16_bits(inp["k"][cu[b] + i])
            exp_v[b, :, P + i] = W.bf16_bits(inp["v"][cu[b] + i])
    assert np.array_equal(ck2, exp_k) and np.array_equal(cv2, exp_v)
    # entries past each sequence's end still hold the sentinel
    assert np.all(ck2[0, :, 5:] == W.CACHE_SENTINEL_BITS)
    assert np.all(cv2[2, :, 5:] == W.CACHE_SENTINEL_BITS)


def test_bad_metadata_is_rejected(oracle_mod):
    wl = _custom("bad", 2, 2, 32, [3, 2], [1, 0], cap=4)
    ck, cv, (inp,) = W.make_inputs(wl)
    bad_k = inp["cu_seqlens_k"].clone()
    bad_k[1] += 1
    with pytest.raises(ValueError, match="cu_seqlens_k"):
        run_oracle(oracle_mod, wl, ck, cv, dict(inp, cu_seqlens_k=bad_k))
    with pytest.raises(ValueError, match="slot"):
        run_oracle(oracle_mod, wl, ck, cv, dict(inp, cache_offsets=torch.tensor([2, 0], dtype=torch.int32),
                                                cu_seqlens_k=torch.tensor([0, 5, 7], dtype=torch.int32)))


# ------------------------------------------------ toy shapes from the page ---

def test_toy_shapes_and_decode_append(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "toy_cache_shapes_yfxerp.json")))
    H, d, T = g["num_heads"], g["head_dim"], g["tokens"]
    assert H * d == g["hidden_size"]
    wl = _custom("toy", H, H, d, [T], [0], cap=T + 1)
    ck, cv, (inp,) = W.make_inputs(wl)
    key = inp["k"][0].clone()
    inp = dict(inp, k=key.expand_as(inp["k"]).contiguous())
    out, lse, ck1, cv1 = run_oracle(oracle_mod, wl, ck, cv, inp)
    assert list(ck1[0, :, :T].shape) == g["cache_shape_after_prefill"]
    assert list(out[T - 1, 0][None].shape) == g["head_output_shape"]
    # equal keys: lse - score = ln(#visible keys) -> the last prompt row scores 3 keys
    s = wl.scale * float(f64(inp["q"][T - 1, 0]) @ f64(key[0]))
    assert math.exp(lse[T - 1, 0] - s) == pytest.approx(g["last_prompt_row_scores"], rel=1e-12)
    # decode step: one new token over the 3 cached ones; the cache grows to 4
    q1 = torch.randn(1, H, d, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    o, l, ck2, _ = oracle_mod.prefill_attention(
        W.bf16_bits(q1), W.bf16_bits(key[None]), W.bf16_bits(inp["v"][:1]),
        np.array([0, 1], np.int32), np.array([0, T + 1], np.int32), np.array([T], np.int32),
        ck1, cv1, n_heads=H, n_kv_heads=H, head_dim=d, max_cache_len=T + 1, scale=wl.scale)
    assert np.array_equal(ck2[0, :, :T + 1][:, -1], W.bf16_bits(key))
    assert ck2[0, :, :T + 1].shape[1] == g["cache_len_after_append"]
    s = wl.scale * float(f64(q1[0, 0]) @ f64(key[0]))
    assert math.exp(l[0, 0] - s) == pytest.approx(g["decode_row_scores"], rel=1e-12)


def test_flop_and_kv_accounting_matches_pages():
    g = json.load(open(os.path.join(GOLDEN, "flop_and_kv_accounting.json")))
    a = g["attention_flops"]
    for c in a["cases"]:
        # the pages count full (unmasked) T x T attention: 4 * T^2 * hidden per layer
        step = W.Step([c["T"]], [0])
        flops = 4 * step.visible_pairs(causal=False) * a["d"] * a["layers"]
        assert flops == pytest.approx(c["flops"], rel=c["rel_tol"])
        # the causal count keeps the lower triangle only (diagonal included)
        assert step.visible_pairs(causal=True) == c["T"] * (c["T"] + 1) // 2
    kv = g["kv_bytes_per_token"]
    for c in kv["cases"]:
        assert 2 * c["n_kv_heads"] * kv["head_dim"] * kv["bytes_per_elem"] * kv["layers"] == c["bytes"]
    pl = g["kv_bytes_per_layer"]
    assert 2 * pl["n_kv_heads"] * pl["tokens"] * pl["head_dim"] * 2 == pl["bytes"]


# ------------------------------------------- independent library routine ---

def _sdpa_reference(wl, ck, cv, inp, causal, window=0):
    """PyTorch float64 SDPA per (sequence, head) with an explicit bottom-right mask."""
    import torch.nn.functional as F
    T = inp["q"].shape[0]
    out = torch.full((T, wl.n_heads, wl.head_dim), float("nan"), dtype=torch.float64)
    cu = inp["cu_seqlens_q"].tolist()
    off = inp["cache_offsets"].tolist()
    G = wl.n_heads // wl.n_kv_heads
    for b in range(len(off)):
        n, P = cu[b + 1] - cu[b], off[b]
        if n == 0:
            continue
        K = torch.cat([ck[b, :, :P].permute(1, 0, 2), inp["k"][cu[b]:cu[b + 1]]], 0).double()
        V = torch.cat([cv[b, :, :P].permute(1, 0, 2), inp["v"][cu[b]:cu[b + 1]]], 0).double()
        Q = inp["q"][cu[b]:cu[b + 1]].double()
        mask = torch.ones(n, P + n, dtype=torch.bool)
        if causal:
            key, qpos = torch.arange(P + n)[None, :], (P + torch.arange(n))[:, None]
            mask = key <= qpos
            if window > 0:
                mask &= key > qpos - window
        for h in range(wl.n_heads):
            o = F.scaled_dot_product_attention(Q[None, :, h], K[None, :, h // G], V[None, :, h // G],
                                               attn_mask=mask[None], scale=wl.scale)
            out[cu[b]:cu[b + 1], h] = o[0]
    return out.numpy()


@pytest.mark.parametrize("case", ["tiny_packed", "layer512", "r1", "r2", "r3", "r4"])
@pytest.mark.parametrize("causal", [True, False])
def test_matches_torch_sdpa_float64(oracle_mod, case, causal):
    if case in ("tiny_packed", "layer512"):  # the 3-prompt packing and the 7B-layer configs
        wl = W.get(case)
    else:
        i = int(case[1:])
        wl = W.random_workload(40 + i, head_dim=[32, 64, 128, 32][i - 1], group=[1, 2, 4, 8][i - 1],
                               max_len=80, max_prefix=90)
    ck, cv, (inp,) = W.make_inputs(wl)
    ck = ck.nan_to_num(0.0)
    cv = cv.nan_to_num(0.0)
    out, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, causal=causal)
    ref = _sdpa_reference(wl, ck, cv, inp, causal)
    assert np.nanmax(np.abs(out - ref)) < 1e-12
    assert np.array_equal(np.isnan(out), np.isnan(ref))


# ------------------------------------------------------------ sliding window ---
# [yfxerp] §4.3: with sliding_window = W the model attends over the last W
# tokens; read as: the query at absolute position p sees keys p - W + 1 .. p.

def test_window_closed_forms(oracle_mod):
    wl = _custom("win", 4, 2, 32, [9, 6], [7, 0], cap=20)
    ck, cv, (inp,) = W.make_inputs(wl)
    # a window longer than every sequence changes nothing (bitwise)
    full, lfull, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp)
    big, lbig, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, window=100)
    assert np.array_equal(full, big) and np.array_equal(lfull, lbig)
    # window 1: every row sees only itself -> out = v, lse = scale * q.k
    one, lone, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, window=1)
    G = wl.n_heads // wl.n_kv_heads
    for t in range(inp["q"].shape[0]):
        for h in range(wl.n_heads):
            assert np.array_equal(one[t, h], f64(inp["v"][t, h // G]))
            s_ = wl.scale * float(f64(inp["q"][t, h]) @ f64(inp["k"][t, h // G]))
            assert lone[t, h] == pytest.approx(s_, abs=1e-13)
    # equal keys, window 4: uniform weights over the last min(4, P+i+1) positions
    key = inp["k"][0, 0].clone()
    inp_eq = dict(inp, k=key.expand_as(inp["k"]).contiguous())
    ck_eq = key.expand_as(ck).contiguous()
    out, lse, _, _ = run_oracle(oracle_mod, wl, ck_eq, cv, inp_eq, window=4)
    cu = inp["cu_seqlens_q"].tolist()
    for b, P in enumerate([7, 0]):
        for i in range(cu[b + 1] - cu[b]):
            t = cu[b] + i
            lo = max(0, P + i - 3)
            for h in range(wl.n_heads):
                kvh = h // G
                allv = np.concatenate([f64(cv[b, kvh, :P]), f64(inp["v"][cu[b]:cu[b + 1], kvh])])
                vals = allv[lo:P + i + 1]
                assert np.allclose(out[t, h], vals.mean(axis=0), rtol=0, atol=1e-14)
                s_ = wl.scale * float(f64(inp["q"][t, h]) @ f64(key))
                assert lse[t, h] == pytest.approx(s_ + math.log(P + i + 1 - lo), abs=1e-13)
    # rows of the windowed softmax sum to one
    ones, _, _, _ = run_oracle(oracle_mod, wl, ck, torch.ones_like(cv), dict(inp, v=torch.ones_like(inp["v"])), window=5)
    assert np.all(np.abs(ones - 1.0) <= 1e-15)


def test_window_needs_causal(oracle_mod):
    wl = _custom("winnc", 2, 2, 32, [3], [0], cap=4)
    ck, cv, (inp,) = W.make_inputs(wl)
    with pytest.raises(ValueError, match="causal"):
        run_oracle(oracle_mod, wl, ck, cv, inp, causal=False, window=2)


@pytest.mark.parametrize("window", [1, 37, 200])
def test_window_matches_torch_sdpa_float64(oracle_mod, window):
    wl = W.random_workload(77, head_dim=64, group=2, max_len=120, max_prefix=150)
    ck, cv, (inp,) = W.make_inputs(wl)
    ck, cv = ck.nan_to_num(0.0), cv.nan_to_num(0.0)
    out, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, window=window)
    ref = _sdpa_reference(wl, ck, cv, inp, True, window=window)
    assert np.nanmax(np.abs(out - ref)) < 1e-12
    assert np.array_equal(np.isnan(out), np.isnan(ref))


def test_window_pair_count_matches_brute_force():
    """The bench's FLOP accounting under a window equals a direct count."""
    for lens, pref, win in (([9, 1, 30], [0, 5, 40], 7), ([300], [0], 64), ([5, 2, 3], [0, 0, 0], 0)):
        step = W.Step(lens, pref)
        brute = 0
        for n, P in zip(lens, pref):
            for i in range(n):
                brute += (P + i + 1) if win == 0 else min(P + i + 1, win)
        assert step.visible_pairs(True, win) == brute


# ---------------------------------------------------------------- paged cache ---
# [zskr] §4.2, [yfxerp] §4.1, [zwxr] §3.4: the cache is a pool of fixed-size
# blocks and a per-sequence block table maps logical block L (positions
# [L bs, (L + 1) bs)) to a physical block; the layout of one block is
# [kv_heads][block_size][head_dim] (the page's 16 x 16 x 128 block).

def _scatter_to_pool(cache_bits, table, bs, num_blocks):
    """Logical cache [B, Hk, cap, d] (uint16) -> pool [num_blocks, Hk, bs, d] by the table."""
    B, Hk, cap, d = cache_bits.shape
    pool = np.full((num_blocks, Hk, bs, d), W.CACHE_SENTINEL_BITS, np.uint16)
    for b in range(B):
        for pos in range(cap):
            pool[table[b][pos // bs], :, pos % bs] = cache_bits[b, :, pos]
    return pool


def _gather_from_pool(pool, table, bs, cap):
    B = len(table)
    out = np.empty((B, pool.shape[1], cap, pool.shape[3]), np.uint16)
    for b in range(B):
        for pos in range(cap):
            out[b, :, pos] = pool[table[b][pos // bs], :, pos % bs]
    return out


def _paged_case(oracle_mod, wl, bs, seed, extra=4):
    """Runs wl contiguous and paged (random physical blocks); returns both results."""
    ck, cv, (inp,) = W.make_inputs(wl)
    rng = np.random.default_rng(seed)
    maxb = -(-wl.max_cache_len // bs)
    cap = maxb * bs
    # pad the logical cache to whole blocks with the sentinel
    pad = lambda c: np.concatenate([W.bf16_bits(c), np.full(c.shape[:2] + (cap - c.shape[2], c.shape[3]),
                                                            W.CACHE_SENTINEL_BITS, np.uint16)], axis=2)
    ckb, cvb = pad(ck), pad(cv)
    nb = wl.num_seqs * maxb + extra
    table = rng.permutation(nb)[: wl.num_seqs * maxb].reshape(wl.num_seqs, maxb).astype(np.int32)
    pk, pv = _scatter_to_pool(ckb, table, bs, nb), _scatter_to_pool(cvb, table, bs, nb)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    cont = oracle_mod.prefill_attention(
        W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
        inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(), inp["cache_offsets"].numpy(), ckb, cvb,
        n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, head_dim=wl.head_dim, max_cache_len=cap,
        scale=wl.scale, causal=wl.causal)
    paged = run_oracle(oracle_mod, wl, as_bf16(pk), as_bf16(pv), inp, block_table=table, block_size=bs)
    return cont, paged, table, (pk, pv), cap


@pytest.mark.parametrize("bs,seed", [(16, 1), (5, 2), (1, 3), (64, 4)])
def test_paged_equals_contiguous(oracle_mod, bs, seed):
    """Any placement of the blocks gives the contiguous result bit for bit, and
    the new tokens land in the rows the table names (and nowhere else)."""
    wl = W.random_workload(60 + seed, head_dim=32, group=2, max_len=70, max_prefix=90)
    (o1, l1, ck1, cv1), (o2, l2, pk2, pv2), table, (pk, pv), cap = _paged_case(oracle_mod, wl, bs, seed)
    assert np.array_equal(o1, o2, equal_nan=True) and np.array_equal(l1, l2, equal_nan=True)
    assert np.array_equal(_gather_from_pool(pk2, table, bs, cap), ck1)
    assert np.array_equal(_gather_from_pool(pv2, table, bs, cap), cv1)
    unused = np.setdiff1d(np.arange(pk.shape[0]), table.ravel())
    assert np.array_equal(pk2[unused], pk[unused]) and np.array_equal(pv2[unused], pv[unused])


def test_paged_matches_torch_sdpa_float64(oracle_mod):
    """Paged read path against the library routine on the gathered logical cache."""
    wl = W.random_workload(71, head_dim=64, group=4, max_len=60, max_prefix=100)
    ck, cv, (inp,) = W.make_inputs(wl, sentinel=False)
    bs = 8
    g = torch.Generator().manual_seed(5)
    table, pk, pv = W.make_paged_cache(wl, bs, g, sentinel=False)
    out, _, _, _ = run_oracle(oracle_mod, wl, pk, pv, inp, block_table=table.numpy(), block_size=bs)
    cap = table.shape[1] * bs
    tb = table.numpy()
    lk = torch.from_numpy(_gather_from_pool(W.bf16_bits(pk), tb, bs, cap).view(np.int16)).view(torch.bfloat16)
    lv = torch.from_numpy(_gather_from_pool(W.bf16_bits(pv), tb, bs, cap).view(np.int16)).view(torch.bfloat16)
    ref = _sdpa_reference(wl, lk, lv, inp, True)
    assert np.nanmax(np.abs(out - ref)) < 1e-12


def test_paged_shared_prefix_blocks(oracle_mod):
    """Two requests with the same 2-block prefix may map it to the same physical
    blocks (prefix caching, [zwxr] §3.4): same result as private copies."""
    bs, H, Hk, d = 16, 4, 2, 32
    wl = _custom("shared", H, Hk, d, [20, 9], [32, 32], cap=64)
    ck, cv, (inp,) = W.make_inputs(wl)
    ck[1, :, :32] = ck[0, :, :32]
    cv[1, :, :32] = cv[0, :, :32]
    private = np.array([[0, 1, 2, 3], [4, 5, 6, 7]], np.int32)
    shared = np.array([[0, 1, 2, 3], [0, 1, 6, 7]], np.int32)
    nb = 8
    pk = _scatter_to_pool(W.bf16_bits(ck), private, bs, nb)
    pv = _scatter_to_pool(W.bf16_bits(cv), private, bs, nb)
    as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    o1, l1, pk1, _ = run_oracle(oracle_mod, wl, as_bf16(pk), as_bf16(pv), inp, block_table=private, block_size=bs)
    pk_s, pv_s = pk.copy(), pv.copy()
    pk_s[4:6] = W.CACHE_SENTINEL_BITS  # the private copies are not read any more
    pv_s[4:6] = W.CACHE_SENTINEL_BITS
    o2, l2, pk2, _ = run_oracle(oracle_mod, wl, as_bf16(pk_s), as_bf16(pv_s), inp, block_table=shared, block_size=bs)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.array_equal(pk2[[0, 1, 2, 3, 6, 7]], pk1[[0, 1, 2, 3, 6, 7]])


def test_paged_bad_block_table_is_rejected(oracle_mod):
    bs = 4
    wl = _custom("badpaged", 2, 2, 32, [3, 2], [5, 0], cap=8)
    ck, cv, (inp,) = W.make_inputs(wl)
    g = torch.Generator().manual_seed(0)
    table, pk, pv = W.make_paged_cache(wl, bs, g)
    for bad in (-1, pk.shape[0]):
        t = table.numpy().copy()
        t[0, 1] = bad
        with pytest.raises(ValueError, match="block table"):
            run_oracle(oracle_mod, wl, pk, pv, inp, block_table=t, block_size=bs)
    # entries past the blocks a sequence uses are not looked at
    t = table.numpy().copy()
    t[1, 1] = -1
    run_oracle(oracle_mod, wl, pk, pv, inp, block_table=t, block_size=bs)
    # max_cache_len must be max_blocks * block_size
    with pytest.raises(ValueError, match="block table"):
        oracle_mod.prefill_attention(
            W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
            inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(), inp["cache_offsets"].numpy(),
            W.bf16_bits(pk), W.bf16_bits(pv), n_heads=2, n_kv_heads=2, head_dim=32, max_cache_len=9,
            scale=wl.scale, block_table=table.numpy(), block_size=bs)


# ---------------------------------------------------------------- rotary (RoPE) ---
# [mhpn] §5.1: the token at position m has its Q/K rotated by theta_m = m * inv_freq,
# inv_freq = 1 / 10000^(arange(0, d, 2) / d), for the Llama models (rotate-half
# pairing: dimension i with i + d/2).

def test_rope_position_zero_is_identity(oracle_mod):
    """A lone token sits at position 0: no rotation, so the cache gets k bit for
    bit, out = v exactly and lse = scale * q.k."""
    wl = _custom("rope0", 4, 2, 64, [1, 1], [0, 0], cap=4)
    ck, cv, (inp,) = W.make_inputs(wl)
    out, lse, ck1, _ = run_oracle(oracle_mod, wl, ck, cv, inp, rope_theta=10000.0)
    for b in range(2):
        assert np.array_equal(ck1[b, :, 0], W.bf16_bits(inp["k"][b]))
        assert np.array_equal(out[b], f64(inp["v"][b]).repeat(2, axis=0))
        qk = (f64(inp["q"][b]).reshape(2, 2, 64) * f64(inp["k"][b])[:, None]).sum(-1).ravel()
        assert np.allclose(lse[b], wl.scale * qk, rtol=0, atol=1e-12)


@pytest.mark.parametrize("m", [1, 7, 300, 4095])
def test_rope_closed_form_rotations(oracle_mod, m):
    """Frequency 0 has inv_freq = 1 (angle m) and frequency d/4 has inv_freq =
    10000^-1/2 = 0.01 (angle m / 100): a unit key along dimension i lands on
    (cos, sin) at dimensions (i, i + d/2) of the cached, rotated key."""
    d = 32
    wl = _custom("ropecf", 2, 2, d, [m + 1], [0], cap=m + 1)
    ck, cv, (inp,) = W.make_inputs(wl)
    k = inp["k"].clone()
    k[m] = 0
    k[m, 0, 0] = 1.0          # head 0: e_0
    k[m, 1, d // 4] = 1.0     # head 1: e_{d/4}
    _, _, ck1, _ = run_oracle(oracle_mod, wl, ck, cv, dict(inp, k=k), rope_theta=10000.0)
    got = ck1[0, :, m].view(np.int16)
    got = torch.from_numpy(got.copy()).view(torch.bfloat16).double().numpy()
    a0 = float(np.float32(m))                          # fp32 angle of frequency 0
    a1 = float(np.float32(np.float32(m) * np.float32(0.01)))
    exp0 = np.zeros(d); exp0[0], exp0[d // 2] = math.cos(a0), math.sin(a0)
    exp1 = np.zeros(d); exp1[d // 4], exp1[d // 4 + d // 2] = math.cos(a1), math.sin(a1)
    bf = lambda x: torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).double().numpy()
    # frequency d/4's inv_freq is 0.01 up to fp32 rounding of the page's formula
    assert np.array_equal(got[0], bf(exp0))
    assert np.allclose(got[1], exp1, atol=2 ** -8 * 1.01 + m * 1e-8)


def test_rope_relative_position_invariance(oracle_mod):
    """With a window of 2 the second of two new tokens sees exactly those two:
    its scores then depend on positions only through their difference, so moving
    both tokens from positions 0, 1 to 777, 778 leaves its output unchanged
    (up to the bf16 rounding of the rotated vectors)."""
    H, Hk, d = 4, 2, 64
    outs = []
    for P in (0, 777):
        wl = _custom("roperel", H, Hk, d, [2], [P], cap=P + 2)
        ck, cv, (inp,) = W.make_inputs(_custom("roperel", H, Hk, d, [2], [0], cap=P + 2, seed=11))
        inp = dict(inp, cu_seqlens_k=torch.tensor([0, P + 2], dtype=torch.int32),
                   cache_offsets=torch.tensor([P], dtype=torch.int32))
        out, lse, _, _ = run_oracle(oracle_mod, wl, ck.nan_to_num(0.0), cv.nan_to_num(0.0), inp,
                                    window=2, rope_theta=10000.0)
        outs.append((out[1], lse[1]))
    # the rotated q and k are rounded to bf16 at each position (|ds| <= scale *
    # 2^-8 * |q| |k| ~ 2e-2 here): equal up to that rounding
    assert np.allclose(outs[0][0], outs[1][0], atol=1e-2)
    assert np.allclose(outs[0][1], outs[1][1], atol=1e-2)
    # and the rotation matters: without it the two positions are not equivalent to
    # a plain (unrotated) run
    wl0 = _custom("roperel", H, Hk, d, [2], [0], cap=2)
    ck, cv, (inp,) = W.make_inputs(_custom("roperel", H, Hk, d, [2], [0], cap=779, seed=11))
    plain, _, _, _ = run_oracle(oracle_mod, wl0, ck[:, :, :2].contiguous(), cv[:, :, :2].contiguous(), inp, window=2)
    assert np.abs(plain[1] - outs[0][0]).max() > 5e-2


def test_rope_chunked_equals_one_shot(oracle_mod):
    """Chunks read the earlier chunks' rotated keys back from the cache: the same
    bf16 tensors one launch attends to, so the results are identical, bit for bit."""
    H, Hk, d, n, c = 4, 2, 64, 240, 80
    one = _custom("ropeone", H, Hk, d, [n], [0], cap=n)
    ck, cv, (inp,) = W.make_inputs(one)
    out1, _, ck1, _ = run_oracle(oracle_mod, one, ck, cv, inp, rope_theta=10000.0)
    cur_k, cur_v = W.bf16_bits(ck), W.bf16_bits(cv)
    outs = []
    for s_ in range(n // c):
        sl = slice(s_ * c, (s_ + 1) * c)
        o, _, cur_k, cur_v = oracle_mod.prefill_attention(
            W.bf16_bits(inp["q"][sl]), W.bf16_bits(inp["k"][sl]), W.bf16_bits(inp["v"][sl]),
            np.array([0, c], np.int32), np.array([0, s_ * c + c], np.int32), np.array([s_ * c], np.int32),
            cur_k, cur_v, n_heads=H, n_kv_heads=Hk, head_dim=d, max_cache_len=n, scale=one.scale,
            rope_theta=10000.0)
        outs.append(o)
    assert np.array_equal(np.concatenate(outs), out1)
    assert np.array_equal(cur_k, ck1)  # the same rotated keys, rounded the same way


def test_rope_matches_complex_rotation_and_sdpa(oracle_mod):
    """Independent restatement: RoPE as multiplication of (x_i + j x_{i+d/2}) by
    exp(j * angle), then PyTorch float64 SDPA, against the oracle."""
    wl = W.random_workload(81, head_dim=64, group=2, max_len=50, max_prefix=60)
    ck, cv, (inp,) = W.make_inputs(wl, sentinel=False)
    theta = 500000.0
    out, _, _, _ = run_oracle(oracle_mod, wl, ck, cv, inp, rope_theta=theta)
    d, half = wl.head_dim, wl.head_dim // 2
    inv = (np.float32(1.0) / np.power(np.float32(theta), np.arange(0, d, 2, dtype=np.float32) / np.float32(d))
           ).astype(np.float32)
    cu = inp["cu_seqlens_q"].tolist()
    off = inp["cache_offsets"].tolist()
    pos = np.concatenate([off[b] + np.arange(cu[b + 1] - cu[b]) for b in range(len(off))]).astype(np.float32)
    ang = (pos[:, None] * inv[None, :]).astype(np.float32).astype(np.float64)  # fp32 angles
    rot = np.exp(1j * ang)[:, None, :]

    def apply(x):  # rotate, then round to the model dtype (bf16)
        x = f64(x)
        z = (x[..., :half] + 1j * x[..., half:]) * rot
        return torch.from_numpy(np.concatenate([z.real, z.imag], -1)).to(torch.bfloat16).double()
    qr, kr = apply(inp["q"]), apply(inp["k"])
    ref = _sdpa_reference_f64(wl, ck, cv, qr, kr, f64(inp["v"]), inp)
    # numpy's fp32 power and the C library's powf may differ in the last bit of
    # inv_freq, which moves an angle at position m by about m * 6e-8 and can flip
    # the bf16 rounding of a rotated element next to a tie
    err = np.abs(out - ref)
    assert np.nanmax(err) < 2e-3 and np.nanmean(err) < 1e-5


def _sdpa_reference_f64(wl, ck, cv, q, k, v, inp):
    """SDPA per (sequence, head) on already-float64 new q/k/v (rotated)."""
    import torch.nn.functional as F
    T = q.shape[0]
    out = torch.full((T, wl.n_heads, wl.head_dim), float("nan"), dtype=torch.float64)
    cu = inp["cu_seqlens_q"].tolist()
    off = inp["cache_offsets"].tolist()
    G = wl.n_heads // wl.n_kv_heads
    v = torch.as_tensor(v)
    for b in range(len(off)):
        n, P = cu[b + 1] - cu[b], off[b]
        if n == 0:
            continue
        K = torch.cat([ck[b, :, :P].permute(1, 0, 2).double(), k[cu[b]:cu[b + 1]]], 0)
        V = torch.cat([cv[b, :, :P].permute(1, 0, 2).double(), v[cu[b]:cu[b + 1]]], 0)
        Q = q[cu[b]:cu[b + 1]]
        key, qpos = torch.arange(P + n)[None, :], (P + torch.arange(n))[:, None]
        mask = key <= qpos
        for h in range(wl.n_heads):
            o = F.scaled_dot_product_attention(Q[None, :, h], K[None, :, h // G], V[None, :, h // G],
                                               attn_mask=mask[None], scale=wl.scale)
            out[cu[b]:cu[b + 1], h] = o[0]
    return out.numpy()


# ------------------------------------------------------------ int8 cache ---
# [zskr] §4.3: INT8 keys and values, queries at full precision, per-token
# granularity among the page's options.  Reading taken: symmetric, one fp32
# scale per (token, KV head) row, scale = max|x| / 127, code = nearest integer
# (ties to even) of x / scale, value = code * scale.

def _q8_case(oracle_mod, wl, inp, ck8=None, cs=None, **kw):
    B, Hk, cap, d = wl.num_seqs, wl.n_kv_heads, wl.max_cache_len, wl.head_dim
    if ck8 is None:
        ck8 = (np.zeros((B, Hk, cap, d), np.int8), np.zeros((B, Hk, cap, d), np.int8))
        cs = (np.zeros((B, Hk, cap), np.float32), np.zeros((B, Hk, cap), np.float32))
    return oracle_mod.prefill_attention(
        W.bf16_bits(inp["q"]), W.bf16_bits(inp["k"]), W.bf16_bits(inp["v"]),
        inp["cu_seqlens_q"].numpy(), inp["cu_seqlens_k"].numpy(), inp["cache_offsets"].numpy(),
        ck8[0], ck8[1], n_heads=wl.n_heads, n_kv_heads=wl.n_kv_heads, head_dim=d, max_cache_len=cap,
        scale=wl.scale, causal=wl.causal, kv_quant=1, cache_k_scale=cs[0], cache_v_scale=cs[1], **kw)


def test_quant_codes_closed_form(oracle_mod):
    """A key row whose largest magnitude is 127 has scale 1 exactly, so its codes
    are the values rounded to the nearest integer, ties to even: 2.5 -> 2,
    3.5 -> 4, -2.5 -> -2, 0.5 -> 0, 1.5 -> 2; a value row scaled by 2^-3 keeps
    the same codes with scale 2^-3; an all-zero row is scale 0, codes 0."""
    d = 32
    wl = _custom("q8cf", 2, 2, d, [1], [0], cap=2)
    _, _, (inp,) = W.make_inputs(wl)
    vals = torch.zeros(d)
    vals[:7] = torch.tensor([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -127.0])
    k = torch.zeros(1, 2, d, dtype=torch.bfloat16)
    k[0, 0] = vals
    v = torch.zeros(1, 2, d, dtype=torch.bfloat16)
    v[0, 0] = vals / 8
    _, _, (ck, sk), (cv, sv) = _q8_case(oracle_mod, wl, dict(inp, k=k, v=v))
    exp = np.zeros(d, np.int8)
    exp[:7] = [127, 2, 4, -2, 0, 2, -127]
    assert np.array_equal(ck[0, 0, 0], exp) and sk[0, 0, 0] == 1.0
    assert np.array_equal(cv[0, 0, 0], exp) and sv[0, 0, 0] == np.float32(1 / 8)
    assert not ck[0, 1, 0].any() and sk[0, 1, 0] == 0.0       # zero row
    assert not ck[0, :, 1].any() and sk[0, 0, 1] == 0.0       # untouched row


def test_quant_rounding_bound_and_extremes(oracle_mod):
    """Every stored row: |x - code * scale| <= scale / 2 (nearest rounding), the
    largest |x| maps to a code of magnitude 127, and |code| <= 127."""
    wl = W.random_workload(90, head_dim=64, group=2, max_len=40, max_prefix=0)
    _, _, (inp,) = W.make_inputs(wl)
    _, _, (ck, sk), (cv, sv) = _q8_case(oracle_mod, wl, inp)
    cu = inp["cu_seqlens_q"].tolist()
    for b in range(wl.num_seqs):
        for i in range(cu[b + 1] - cu[b]):
            for codes, scales, src in ((ck, sk, inp["k"]), (cv, sv, inp["v"])):
                x = src[cu[b] + i].double().numpy()  # [Hk, d]
                c, sc = codes[b, :, i].astype(np.float64), scales[b, :, i].astype(np.float64)
                # x / scale is an fp32 quotient (relative error 2^-24 on values up to 127)
                assert (np.abs(x - c * sc[:, None]) <= sc[:, None] * (0.5 + 127 * 2.0 ** -23)).all()
                assert (np.abs(c).max(axis=1) == 127).all()
                assert np.allclose(sc, np.abs(x).max(axis=1) / 127, rtol=1e-7)


def test_quant_prefix_read_matches_sdpa_on_dequantised_cache(oracle_mod):
    """A chunk over an int8 prefix: SDPA (float64) on the cache written out as
    code * scale, with the chunk's own keys/values at full precision."""
    wl = W.random_workload(91, head_dim=64, group=4, max_len=40, max_prefix=80, allow_empty=False)
    _, _, (inp,) = W.make_inputs(wl)
    rng = np.random.default_rng(3)
    shape = (wl.num_seqs, wl.n_kv_heads, wl.max_cache_len, wl.head_dim)
    codes = (rng.integers(-127, 128, size=shape).astype(np.int8), rng.integers(-127, 128, size=shape).astype(np.int8))
    scales = (rng.uniform(0.001, 0.03, size=shape[:-1]).astype(np.float32),
              rng.uniform(0.001, 0.03, size=shape[:-1]).astype(np.float32))
    out, _, _, _ = _q8_case(oracle_mod, wl, inp, codes, scales)
    deq = [torch.from_numpy(c.astype(np.float64) * s.astype(np.float64)[..., None]) for c, s in zip(codes, scales)]
    ref = _sdpa_reference_f64(wl, deq[0], deq[1], torch.from_numpy(f64(inp["q"])),
                              torch.from_numpy(f64(inp["k"])), f64(inp["v"]), inp)
    assert np.nanmax(np.abs(out - ref)) < 1e-12


def test_quant_zero_cache_rows_read_as_zero(oracle_mod):
    """Prefix rows with scale 0 are zero keys: every such score is 0."""
    wl = _custom("q8z", 2, 2, 32, [1], [5], cap=6)
    _, _, (inp,) = W.make_inputs(wl)
    out, lse, _, _ = _q8_case(oracle_mod, wl, inp)  # all-zero codes and scales
    s_new = wl.scale * float((inp["q"][0].double() * inp["k"][0].double()).sum(-1)[0])
    # 5 zero scores and one score s_new: lse = ln(5 + e^s_new); out = e^s_new v / (5 + e^s_new)
    assert lse[0, 0] == pytest.approx(math.log(5 + math.exp(s_new)), abs=1e-12)
    w = math.exp(s_new) / (5 + math.exp(s_new))
    assert np.allclose(out[0, 0], w * f64(inp["v"][0, 0]), atol=1e-12)


# ------------------------------------------------- rotation before rounding ---

def _libm_inv_freq(theta, d):
    """inv_freq[i] = 1 / theta^(2i/d) in fp32 through the C library's powf (the
    same routine the oracle's C code calls), so the angles agree bit for bit."""
    import ctypes
    import ctypes.util
    libm = ctypes.CDLL(ctypes.util.find_library("m"))
    libm.powf.restype = ctypes.c_float
    libm.powf.argtypes = [ctypes.c_float, ctypes.c_float]
    return np.array([np.float32(1.0) / np.float32(libm.powf(np.float32(theta), np.float32(2 * i) / np.float32(d)))
                     for i in range(d // 2)], dtype=np.float32)


@pytest.mark.parametrize("d,theta", [(32, 10000.0), (64, 500000.0), (128, 10000.0)])
def test_rope_rotation_before_rounding_matches_complex_exponential(oracle_mod, d, theta):
    """[mhpn] §5.1 restated independently: the pair (x_i, x_{i+d/2}) is the
    complex number x_i + j x_{i+d/2}, turned by exp(j m inv_freq[i]).  The
    oracle's fp64 rotation, before its bf16 rounding, equals it to 1e-12 at
    positions up to 40000 (angles taken in fp32 as the page's formula does)."""
    rng = np.random.default_rng(d)
    n = 300
    x = torch.randn(n, d, generator=torch.Generator().manual_seed(d)).to(torch.bfloat16)
    pos = np.concatenate([[0, 1, 2, 127, 128, 4095, 32767, 40000],
                          rng.integers(0, 40001, size=n - 8)]).astype(np.int32)
    got = oracle_mod.rope_rotate(W.bf16_bits(x), pos, rope_theta=theta, max_pos=40001)
    inv = _libm_inv_freq(theta, d)
    ang = (pos.astype(np.float32)[:, None] * inv[None, :]).astype(np.float32).astype(np.float64)
    xf = x.double().numpy()
    z = (xf[:, : d // 2] + 1j * xf[:, d // 2:]) * np.exp(1j * ang)
    ref = np.concatenate([z.real, z.imag], axis=1)
    assert np.abs(got - ref).max() < 1e-12
    # position 0 is the identity, exactly
    assert np.array_equal(got[0], xf[0])
    # and a rotation keeps every pair's length
    assert np.allclose(np.hypot(got[:, : d // 2], got[:, d // 2:]), np.hypot(xf[:, : d // 2], xf[:, d // 2:]),
                       rtol=0, atol=1e-12)


@pytest.mark.parametrize("m", [3, 100, 1000, 9999])
def test_quant_of_rotated_unit_key_closed_form(oracle_mod, m):
    """int8 x RoPE: a unit key e_i at position m is rotated onto (cos a, sin a)
    at dimensions (i, i + d/2), a = m * inv_freq[i], then rounded to bf16 (the
    model dtype, [mhpn] §5.1) and quantised per row ([zskr] §4.3): the larger of
    the two magnitudes becomes code +-127 with scale = that magnitude / 127, the
    other code is 127 times the ratio rounded to the nearest integer, and every
    other code is 0."""
    d = 32
    wl = _custom("q8rope", 2, 2, d, [m + 1], [0], cap=m + 1)
    _, _, (inp,) = W.make_inputs(wl)
    k = inp["k"].clone()
    k[m] = 0
    k[m, 0, 0] = 1.0          # head 0: e_0, inv_freq 1
    k[m, 1, d // 4] = 1.0     # head 1: e_{d/4}, inv_freq 1/100
    _, _, (ck, sk), _ = _q8_case(oracle_mod, wl, dict(inp, k=k), rope_theta=10000.0)
    inv = _libm_inv_freq(10000.0, d)
    bf = lambda x: float(torch.tensor(x, dtype=torch.float64).to(torch.bfloat16).double())
    for h, i in ((0, 0), (1, d // 4)):
        a = float(np.float32(np.float32(m) * inv[i]))
        x, y = bf(math.cos(a)), bf(math.sin(a))
        big = max(abs(x), abs(y))
        exp_codes = np.zeros(d, np.int64)
        for e, val in ((i, x), (i + d // 2, y)):
            r = 127 * abs(val) / big
            assert abs(r - math.floor(r) - 0.5) > 1e-4, "a tie would make the closed form ambiguous"
            exp_codes[e] = int(math.copysign(round(r), val))
        assert np.array_equal(ck[0, h, m].astype(np.int64), exp_codes), (h, ck[0, h, m], exp_codes)
        assert sk[0, h, m] == np.float32(np.float32(big) / np.float32(127.0))
